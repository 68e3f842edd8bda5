"""CPU oracle of the DFlash/DSpark drafter decode-step hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library (``context_kv_update_gb300``) never imports, links or calls it,
and this package imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, double accumulation); this
module compiles it with gcc and wraps each entry point with numpy marshalling.
bf16 tensors travel as ``uint16`` arrays holding the bf16 bit patterns.

Pins (tests/test_oracle_*.py): brute-force dense attention on tiny inputs,
split-count invariance of the split-KV form, RMSNorm / RoPE closed forms,
numpy float64 matmul for the projection, a hand-worked bookkeeping case
(tests/golden/bookkeeping_tiny.json) and bookkeeping invariants; the split
update against the fused one; the query RMSNorm + RoPE against numpy RMSNorm
and RoPE's position-difference and length invariants; strict acceptance by
hand cases and brute force; the embedding lookup as a one-hot product; the
prefill context store against the pinned decode update (one request as one
all-accepted block), request independence and the RoPE position shift.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MASK_CAUSAL_TAIL = 0
MASK_BLOCK_BIDIR = 1

ST_BAD_NACCEPTED = 1
ST_BAD_CTX_LEN = 2
ST_CTX_OUTRUN = 4
ST_BAD_PAGE = 8


def build(out_path: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile oracle.c into a shared library (gcc, OpenMP, -O2)."""
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", *extra_flags,
           _SRC, "-o", out_path, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            build()
        _lib = ctypes.CDLL(_LIB_PATH)
        return _lib


def load_variant(path: str):
    """Load a separately built copy of the oracle (used by mutation tests)."""
    return ctypes.CDLL(path)


def _p(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(ctypes.c_int(n))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ----------------------------------------------------------------- bf16


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round to bf16 through the oracle's own rounding routine (elementwise)."""
    lib = _load()
    lib.oracle_double_to_bf16.restype = ctypes.c_uint16
    lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat = x.reshape(-1)
    of = out.reshape(-1)
    for k in range(flat.size):
        of[k] = lib.oracle_double_to_bf16(float(flat[k]))
    return out


# ----------------------------------------------------------- primitives


def rmsnorm(x, g=None, eps=1e-6):
    lib = _load()
    x = _c(x, np.float64)
    out = np.empty_like(x)
    gg = None if g is None else _c(g, np.float64)
    lib.oracle_rmsnorm(_p(x), _p(gg), ctypes.c_int(x.size), ctypes.c_double(eps), _p(out))
    return out


def rope_neox(x, pos, theta):
    lib = _load()
    x = _c(x, np.float64)
    out = np.empty_like(x)
    lib.oracle_rope_neox(_p(x), ctypes.c_int(x.size), ctypes.c_double(float(pos)),
                         ctypes.c_double(theta), _p(out))
    return out


def matvec_bf16(W_bits, x):
    lib = _load()
    W_bits = _c(W_bits, np.uint16)
    x = _c(x, np.float64)
    out = np.empty(W_bits.shape[0], dtype=np.float64)
    lib.oracle_matvec_bf16(_p(W_bits), ctypes.c_int(W_bits.shape[0]), ctypes.c_int(W_bits.shape[1]),
                           _p(x), _p(out))
    return out


# ---------------------------------------------------------- bookkeeping


def bookkeeping(off, acc, n_acc, ctx_pos_pre, valid, *, M, T, P, off_div, max_ctx, mask_id):
    """Returns (dict of outputs, status).  ``off`` is a [B, >=M] int32 base array
    whose first M columns are the raw offsets (its row stride is its width);
    ``acc`` is a [B, >=T] base array of accepted tokens likewise."""
    lib = _load()
    off_c = _c(off, np.int32)
    acc_c = _c(acc, np.int32)
    B = int(np.asarray(n_acc).shape[0])
    os_ = off_c.shape[1]
    as_ = acc_c.shape[1]
    assert os_ >= M and as_ >= T
    n_acc = _c(n_acc, np.int32)
    ctx_pre = _c(ctx_pos_pre, np.int32)
    valid_c = None if valid is None else _c(valid, np.uint8)
    o = {
        "n_pages": np.empty(B, np.int32), "block_table": np.empty((B, M), np.int32),
        "alloc_limit": np.empty(B, np.int32), "bonus": np.empty(B, np.int32),
        "emb_ids": np.empty((B, T), np.int32), "ctx_pos": np.empty((B, T), np.int32),
        "q_pos": np.empty((B, T), np.int32), "ctx_dst_page": np.empty((B, T), np.int32),
        "ctx_dst_slot": np.empty((B, T), np.int32), "ctx_wmask": np.empty((B, T), np.uint8),
        "blk_page": np.empty((B, T), np.int32), "blk_slot": np.empty((B, T), np.int32),
        "blk_mask": np.empty((B, T), np.uint8), "ctx_len_new": np.empty(B, np.int32),
        "seq_lens": np.empty(B, np.int32),
    }
    st = lib.oracle_bookkeeping(
        ctypes.c_int(B), ctypes.c_int(T), ctypes.c_int(M), ctypes.c_int(P), ctypes.c_int(off_div),
        ctypes.c_int(max_ctx), ctypes.c_int(mask_id), _p(off_c), ctypes.c_int64(os_), _p(acc_c),
        ctypes.c_int64(as_), _p(n_acc), _p(ctx_pre), _p(valid_c), _p(o["n_pages"]),
        _p(o["block_table"]), _p(o["alloc_limit"]), _p(o["bonus"]), _p(o["emb_ids"]),
        _p(o["ctx_pos"]), _p(o["q_pos"]), _p(o["ctx_dst_page"]), _p(o["ctx_dst_slot"]),
        _p(o["ctx_wmask"]), _p(o["blk_page"]), _p(o["blk_slot"]), _p(o["blk_mask"]),
        _p(o["ctx_len_new"]), _p(o["seq_lens"]))
    return o, int(st)


# ------------------------------------------------------------ ctx update


def fc_hidden_norm(hidden, w_fc, g_h, eps_h):
    lib = _load()
    is_f32 = hidden.dtype == np.float32
    hid = _c(hidden, np.float32 if is_f32 else np.uint16)
    rows = int(np.prod(hid.shape[:-1]))
    D_in = hid.shape[-1]
    D = w_fc.shape[0]
    out = np.empty((rows, D), np.uint16)
    lib.oracle_fc_hidden_norm(ctypes.c_int(rows), _p(hid), ctypes.c_int(int(is_f32)),
                              ctypes.c_int(D_in), ctypes.c_int(D), _p(_c(w_fc, np.uint16)),
                              _p(_c(g_h, np.uint16)), ctypes.c_double(eps_h), _p(out))
    return out


def ctx_kv_update_gqa(g, hidden, n_acc, ctx_in, alloc_limit, tbl, valid, w_fc, g_h, w_kv, g_k,
                      pool):
    """In-place update of ``pool`` (uint16, [L][NP][2][nkv][P][hd]); returns ctx_out."""
    lib = _load()
    B, T = hidden.shape[0], hidden.shape[1]
    is_f32 = hidden.dtype == np.float32
    hid = _c(hidden, np.float32 if is_f32 else np.uint16)
    assert pool.dtype == np.uint16 and pool.flags.c_contiguous
    ctx_out = np.empty(B, np.int32)
    tbl = _c(tbl, np.int32)
    rc = lib.oracle_ctx_kv_update_gqa(
        ctypes.c_int(B), ctypes.c_int(T), ctypes.c_int(g["L"]), ctypes.c_int(g["D_in"]),
        ctypes.c_int(g["D"]), ctypes.c_int(g["nkv"]), ctypes.c_int(g["hd"]), ctypes.c_int(g["P"]),
        ctypes.c_int(tbl.shape[1]), ctypes.c_int(g["num_pool_pages"]),
        ctypes.c_double(g["rope_theta"]), ctypes.c_double(g["eps_h"]), ctypes.c_double(g["eps_k"]),
        _p(hid), ctypes.c_int(int(is_f32)), _p(_c(n_acc, np.int32)), _p(_c(ctx_in, np.int32)),
        _p(ctx_out), _p(_c(alloc_limit, np.int32)), _p(tbl),
        _p(None if valid is None else _c(valid, np.uint8)), _p(_c(w_fc, np.uint16)),
        _p(_c(g_h, np.uint16)), _p(_c(w_kv, np.uint16)), _p(_c(g_k, np.uint16)), _p(pool))
    assert rc == 0
    return ctx_out


def ctx_kv_update_mla(g, hidden, n_acc, ctx_in, alloc_limit, tbl, valid, w_fc, g_h, w_dkv, g_kv,
                      pool):
    lib = _load()
    B, T = hidden.shape[0], hidden.shape[1]
    is_f32 = hidden.dtype == np.float32
    hid = _c(hidden, np.float32 if is_f32 else np.uint16)
    assert pool.dtype == np.uint16 and pool.flags.c_contiguous
    ctx_out = np.empty(B, np.int32)
    tbl = _c(tbl, np.int32)
    rc = lib.oracle_ctx_kv_update_mla(
        ctypes.c_int(B), ctypes.c_int(T), ctypes.c_int(g["L"]), ctypes.c_int(g["D_in"]),
        ctypes.c_int(g["D"]), ctypes.c_int(g["latent"]), ctypes.c_int(g["rope_dim"]),
        ctypes.c_int(g["P"]), ctypes.c_int(tbl.shape[1]), ctypes.c_int(g["num_pool_pages"]),
        ctypes.c_double(g["rope_theta"]), ctypes.c_double(g["eps_h"]), ctypes.c_double(g["eps_k"]),
        _p(hid), ctypes.c_int(int(is_f32)), _p(_c(n_acc, np.int32)), _p(_c(ctx_in, np.int32)),
        _p(ctx_out), _p(_c(alloc_limit, np.int32)), _p(tbl),
        _p(None if valid is None else _c(valid, np.uint8)), _p(_c(w_fc, np.uint16)),
        _p(_c(g_h, np.uint16)), _p(_c(w_dkv, np.uint16)), _p(_c(g_kv, np.uint16)), _p(pool))
    assert rc == 0
    return ctx_out


# ------------------------------------------------ prefill context store


def ctx_kv_prefill(g, hidden, cu_rows, ctx_in, alloc_limit, tbl, valid, w_fc, g_h, w_kv, g_k,
                   pool):
    """Prefill context store: hidden [N, D_in] (rows of all requests, request r
    at cu_rows[r]..cu_rows[r+1]-1), written in place into ``pool`` at
    positions ctx_in[r] + i; returns ctx_out."""
    lib = _load()
    is_f32 = hidden.dtype == np.float32
    hid = _c(hidden, np.float32 if is_f32 else np.uint16)
    cu = _c(cu_rows, np.int32)
    B = cu.shape[0] - 1
    assert pool.dtype == np.uint16 and pool.flags.c_contiguous
    gqa = g["kind"] == "gqa"
    tbl = _c(tbl, np.int32)
    ctx_out = np.empty(B, np.int32)
    rc = lib.oracle_ctx_kv_prefill(
        ctypes.c_int(0 if gqa else 1), ctypes.c_int(B), ctypes.c_int(g["L"]),
        ctypes.c_int(g["D_in"]), ctypes.c_int(g["D"]), ctypes.c_int(g["nkv"] if gqa else 1),
        ctypes.c_int(g["hd"] if gqa else 0), ctypes.c_int(g.get("latent", 512)),
        ctypes.c_int(g.get("rope_dim", 64)), ctypes.c_int(g["P"]), ctypes.c_int(tbl.shape[1]),
        ctypes.c_int(g["num_pool_pages"]), ctypes.c_double(g["rope_theta"]),
        ctypes.c_double(g["eps_h"]), ctypes.c_double(g["eps_k"]), _p(hid),
        ctypes.c_int(int(is_f32)), _p(cu), _p(_c(ctx_in, np.int32)), _p(ctx_out),
        _p(_c(alloc_limit, np.int32)), _p(tbl), _p(None if valid is None else _c(valid, np.uint8)),
        _p(_c(w_fc, np.uint16)), _p(_c(g_h, np.uint16)), _p(_c(w_kv, np.uint16)),
        _p(_c(g_k, np.uint16)), _p(pool))
    assert rc == 0
    return ctx_out


# ------------------------------------------------- split context update


def ctx_kv_project(g, hidden, ctx_in, w_fc, g_h, w_kv, g_k):
    """Projection half of the split update (every row, RoPE at c + i).
    Returns (staged_c int32 [B], staged uint16 [B * T, W]) with W the
    per-row width: GQA L * 2 * nkv * hd ([L][K|V][nkv][hd]), MLA L * 576."""
    lib = _load()
    B, T = hidden.shape[0], hidden.shape[1]
    is_f32 = hidden.dtype == np.float32
    hid = _c(hidden, np.float32 if is_f32 else np.uint16)
    gqa = g["kind"] == "gqa"
    W = g["L"] * (2 * g["nkv"] * g["hd"] if gqa else g["latent"] + g["rope_dim"])
    staged_c = np.empty(B, np.int32)
    staged = np.empty((B * T, W), np.uint16)
    common = [ctypes.c_int(B), ctypes.c_int(T), ctypes.c_int(g["L"]), ctypes.c_int(g["D_in"]),
              ctypes.c_int(g["D"])]
    dims = ([ctypes.c_int(g["nkv"]), ctypes.c_int(g["hd"])] if gqa else
            [ctypes.c_int(g["latent"]), ctypes.c_int(g["rope_dim"])])
    fn = lib.oracle_ctx_kv_project_gqa if gqa else lib.oracle_ctx_kv_project_mla
    rc = fn(*common, *dims, ctypes.c_double(g["rope_theta"]), ctypes.c_double(g["eps_h"]),
            ctypes.c_double(g["eps_k"]), _p(hid), ctypes.c_int(int(is_f32)),
            _p(_c(ctx_in, np.int32)), _p(_c(w_fc, np.uint16)), _p(_c(g_h, np.uint16)),
            _p(_c(w_kv, np.uint16)), _p(_c(g_k, np.uint16)), _p(staged_c), _p(staged))
    assert rc == 0
    return staged_c, staged


def ctx_kv_commit(g, staged_c, staged, n_acc, alloc_limit, tbl, valid, pool):
    """Store half of the split update: in-place masked store into ``pool``;
    returns ctx_out."""
    lib = _load()
    B = staged_c.shape[0]
    assert pool.dtype == np.uint16 and pool.flags.c_contiguous
    gqa = g["kind"] == "gqa"
    tbl = _c(tbl, np.int32)
    ctx_out = np.empty(B, np.int32)
    rc = lib.oracle_ctx_kv_commit(
        ctypes.c_int(0 if gqa else 1), ctypes.c_int(B), ctypes.c_int(g["T"]), ctypes.c_int(g["L"]),
        ctypes.c_int(g["nkv"] if gqa else 1), ctypes.c_int(g["hd"] if gqa else 0),
        ctypes.c_int(0 if gqa else g["latent"] + g["rope_dim"]), ctypes.c_int(g["P"]),
        ctypes.c_int(tbl.shape[1]), ctypes.c_int(g["num_pool_pages"]),
        _p(_c(staged_c, np.int32)), _p(_c(staged, np.uint16)), _p(_c(n_acc, np.int32)),
        _p(ctx_out), _p(_c(alloc_limit, np.int32)), _p(tbl),
        _p(None if valid is None else _c(valid, np.uint8)), _p(pool))
    assert rc == 0
    return ctx_out


# ------------------------------------------------ either side of the path


def strict_accept(draft, target):
    """draft int32 [B, K], target int32 [B, K + 1] -> (n_acc [B], accepted
    [B, K + 1] with -1 past n_acc)."""
    lib = _load()
    d = _c(draft, np.int32)
    t = _c(target, np.int32)
    B, K = d.shape
    assert t.shape == (B, K + 1)
    n_acc = np.empty(B, np.int32)
    acc = np.empty((B, K + 1), np.int32)
    assert lib.oracle_strict_accept(ctypes.c_int(B), ctypes.c_int(K), _p(d), _p(t), _p(n_acc),
                                    _p(acc)) == 0
    return n_acc, acc


def embedding_gather(ids, table):
    """ids int32 [...], table uint16 [V, D] -> (uint16 [..., D], any id out of range)."""
    lib = _load()
    i = _c(ids, np.int32)
    tb = _c(table, np.uint16)
    V, D = tb.shape
    out = np.empty(i.shape + (D,), np.uint16)
    bad = lib.oracle_embedding_gather(ctypes.c_int(i.size), ctypes.c_int(V), ctypes.c_int(D),
                                      _p(i), _p(tb), _p(out))
    return out, bool(bad)


# ------------------------------------------------------------ query side


def q_norm_rope(q_in, gamma, pos, theta, eps):
    """q_in uint16 [..., heads, dim] (rows = leading dims), gamma uint16 [dim]
    or None (rotation only), pos int32 [rows].  Returns uint16 like q_in."""
    lib = _load()
    q = _c(q_in, np.uint16)
    dim, heads = q.shape[-1], q.shape[-2]
    rows = q.size // (dim * heads)
    pos = _c(np.asarray(pos).reshape(rows), np.int32)
    out = np.empty_like(q)
    rc = lib.oracle_q_norm_rope(ctypes.c_int(rows), ctypes.c_int(heads), ctypes.c_int(dim),
                                ctypes.c_int(0 if gamma is None else 1), ctypes.c_double(theta),
                                ctypes.c_double(eps), _p(q),
                                _p(None if gamma is None else _c(gamma, np.uint16)), _p(pos),
                                _p(out))
    assert rc == 0
    return out


# ----------------------------------------------------------- scatter


def block_kv_scatter_gqa(g, layer, blk_k, blk_v, blk_page, blk_slot, blk_mask, pool):
    lib = _load()
    B, T = blk_k.shape[0], blk_k.shape[1]
    rc = lib.oracle_block_kv_scatter_gqa(
        ctypes.c_int(B), ctypes.c_int(T), ctypes.c_int(g["nkv"]), ctypes.c_int(g["hd"]),
        ctypes.c_int(g["P"]), ctypes.c_int(g["num_pool_pages"]), ctypes.c_int(layer),
        _p(_c(blk_k, np.uint16)), _p(_c(blk_v, np.uint16)), _p(_c(blk_page, np.int32)),
        _p(_c(blk_slot, np.int32)), _p(_c(blk_mask, np.uint8)), _p(pool))
    assert rc == 0


def block_latent_scatter_mla(g, layer, blk_lat, blk_page, blk_slot, blk_mask, pool):
    lib = _load()
    B, T, W = blk_lat.shape
    rc = lib.oracle_block_latent_scatter_mla(
        ctypes.c_int(B), ctypes.c_int(T), ctypes.c_int(W), ctypes.c_int(g["P"]),
        ctypes.c_int(g["num_pool_pages"]), ctypes.c_int(layer), _p(_c(blk_lat, np.uint16)),
        _p(_c(blk_page, np.int32)), _p(_c(blk_slot, np.int32)), _p(_c(blk_mask, np.uint8)),
        _p(pool))
    assert rc == 0


# ----------------------------------------------------------- attention


def attention_gqa(g, layer, q, pool, tbl, kv_len, *, window=0, sinks=None, scale=None,
                  mask_mode=MASK_CAUSAL_TAIL, num_segments=None):
    """Direct definition (num_segments=None) or the split-KV form."""
    lib = _load()
    B, Tq, hq, hd = q.shape
    scale = (1.0 / np.sqrt(hd)) if scale is None else scale
    out = np.empty((B, Tq, hq, hd), np.float64)
    tbl = _c(tbl, np.int32)
    args = [ctypes.c_int(B), ctypes.c_int(Tq), ctypes.c_int(hq), ctypes.c_int(g["nkv"]),
            ctypes.c_int(hd), ctypes.c_int(g["P"]), ctypes.c_int(tbl.shape[1]),
            ctypes.c_int(g["num_pool_pages"]), ctypes.c_int(layer), _p(_c(q, np.uint16)),
            _p(pool), _p(tbl), _p(_c(kv_len, np.int32)), ctypes.c_int(window),
            _p(None if sinks is None else _c(sinks, np.float32)), ctypes.c_double(scale),
            ctypes.c_int(mask_mode)]
    if num_segments is None:
        rc = lib.oracle_attention_gqa(*args, _p(out))
    else:
        rc = lib.oracle_attention_gqa_split(*args, ctypes.c_int(num_segments), _p(out))
    if rc != 0:
        raise ValueError("oracle attention: key mapped outside the pool or kv_len > M*P")
    return out


def attention_mla(g, layer, q_lat, q_rope, pool, tbl, kv_len, *, window=0, sinks=None,
                  scale=None, mask_mode=MASK_CAUSAL_TAIL):
    lib = _load()
    B, Tq, hq, lat = q_lat.shape
    rope = q_rope.shape[-1]
    scale = (1.0 / np.sqrt(128 + 64)) if scale is None else scale
    out = np.empty((B, Tq, hq, lat), np.float64)
    tbl = _c(tbl, np.int32)
    rc = lib.oracle_attention_mla(
        ctypes.c_int(B), ctypes.c_int(Tq), ctypes.c_int(hq), ctypes.c_int(lat), ctypes.c_int(rope),
        ctypes.c_int(g["P"]), ctypes.c_int(tbl.shape[1]), ctypes.c_int(g["num_pool_pages"]),
        ctypes.c_int(layer), _p(_c(q_lat, np.uint16)), _p(_c(q_rope, np.uint16)), _p(pool),
        _p(tbl), _p(_c(kv_len, np.int32)), ctypes.c_int(window),
        _p(None if sinks is None else _c(sinks, np.float32)), ctypes.c_double(scale),
        ctypes.c_int(mask_mode), _p(out))
    if rc != 0:
        raise ValueError("oracle attention: key mapped outside the pool or kv_len > M*P")
    return out
