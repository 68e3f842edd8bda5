"""ctypes binding of ``libdflash.so`` (include/dflash.h).

Argument marshalling only: every function here validates nothing beyond what
ctypes needs, converts torch tensors to device pointers and the current torch
stream to a ``cudaStream_t``, calls the C entry point of the same name and
raises ``DflashError`` on a non-zero status.  All arithmetic runs in the CUDA
kernels of the library; there is no CPU or PyTorch fallback.  Loading fails
loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdflash.so")

DFLASH_OK = 0
DFLASH_ERR_INVALID_ARG = 1
DFLASH_ERR_UNSUPPORTED_GEOM = 2
DFLASH_ERR_WORKSPACE_TOO_SMALL = 3
DFLASH_ERR_CUDA = 4

DEV_BAD_NACCEPTED = 1
DEV_BAD_CTX_LEN = 2
DEV_CTX_OUTRUN = 4
DEV_BAD_PAGE = 8
DEV_KV_LEN_RANGE = 16
DEV_WAIT_TIMEOUT = 32
DEV_BAD_TOKEN = 64

KIND_GQA = 0
KIND_MLA = 1
MASK_CAUSAL_TAIL = 0
MASK_BLOCK_BIDIR = 1
DTYPE_BF16 = 0
DTYPE_F32 = 1

EXPORTS = ("dflash_step_bookkeeping", "dflash_ctx_workspace_bytes", "dflash_ctx_kv_update",
           "dflash_block_kv_scatter", "dflash_attention_num_segments",
           "dflash_attention_workspace_bytes", "dflash_block_attention", "dflash_status_string",
           "dflash_abi_version", "dflash_block_attention_noalloc",
           "dflash_block_attention_noalloc_max_scratch_bytes", "dflash_ctx_staged_bytes",
           "dflash_ctx_kv_project", "dflash_ctx_kv_commit", "dflash_q_norm_rope",
           "dflash_packed_kv_bytes", "dflash_packed_gamma_bytes", "dflash_pack_weights",
           "dflash_strict_accept", "dflash_embedding_gather", "dflash_ctx_prefill_workspace_bytes",
           "dflash_ctx_kv_prefill", "dflash_test_attention_skip_tile",
           "dflash_block_scatter_attention")


class DflashError(RuntimeError):
    def __init__(self, fn, code, lib):
        self.code = code
        msg = lib.dflash_status_string(code).decode() if lib is not None else str(code)
        super().__init__(f"{fn} failed: {msg} ({code})")


class Geom(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("d_in", ctypes.c_int32), ("d_model", ctypes.c_int32), ("hq", ctypes.c_int32),
                ("nkv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("latent_dim", ctypes.c_int32), ("rope_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("num_pool_pages", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("reserved0", ctypes.c_int32), ("rope_theta", ctypes.c_double),
                ("eps_hidden", ctypes.c_double), ("eps_k", ctypes.c_double)]


class Weights(ctypes.Structure):
    _fields_ = [("w_fc", ctypes.c_void_p), ("gamma_h", ctypes.c_void_p),
                ("w_kv", ctypes.c_void_p), ("gamma_k", ctypes.c_void_p)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("w_k", ctypes.c_void_p), ("w_v", ctypes.c_void_p), ("k_norm", ctypes.c_void_p)]


class StepOutputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "n_pages", "block_table", "alloc_limit", "bonus", "emb_ids", "ctx_pos", "q_pos",
        "ctx_dst_page", "ctx_dst_slot", "ctx_wmask", "blk_page", "blk_slot", "blk_mask",
        "ctx_len_new", "seq_lens")]


STEP_OUTPUT_FIELDS = [f[0] for f in StepOutputs._fields_]

_lib = None


def load():
    """Load libdflash.so (raises when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m context_kv_update_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    G = ctypes.POINTER(Geom)
    lib.dflash_step_bookkeeping.argtypes = [G, ctypes.c_int, vp, i64, i32, vp, i64, vp, vp, vp,
                                            i32, i32, ctypes.POINTER(StepOutputs), vp, vp]
    lib.dflash_ctx_workspace_bytes.argtypes = [G, ctypes.c_int]
    lib.dflash_ctx_workspace_bytes.restype = sz
    lib.dflash_ctx_kv_update.argtypes = [G, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp, vp, vp,
                                         ctypes.POINTER(Weights), vp, vp, sz, vp, vp]
    lib.dflash_ctx_staged_bytes.argtypes = [G, ctypes.c_int]
    lib.dflash_ctx_staged_bytes.restype = sz
    lib.dflash_ctx_kv_project.argtypes = [G, ctypes.c_int, vp, ctypes.c_int, vp,
                                          ctypes.POINTER(Weights), vp, sz, vp, sz, vp, vp]
    lib.dflash_ctx_kv_commit.argtypes = [G, ctypes.c_int, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.dflash_q_norm_rope.argtypes = [G, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, vp]
    lib.dflash_block_kv_scatter.argtypes = [G, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, vp,
                                            vp, vp]
    lib.dflash_attention_num_segments.argtypes = [G, ctypes.c_int, ctypes.c_int]
    lib.dflash_attention_workspace_bytes.argtypes = [G, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.dflash_attention_workspace_bytes.restype = sz
    lib.dflash_block_attention.argtypes = [G, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                           vp, vp, i32, vp, ctypes.c_float, ctypes.c_int,
                                           ctypes.c_int, vp, sz, vp, vp, vp]
    lib.dflash_block_scatter_attention.argtypes = [G, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp,
                                                   ctypes.c_float, ctypes.c_int, ctypes.c_int, vp,
                                                   sz, vp, vp, vp]
    lib.dflash_block_attention_noalloc.argtypes = [G, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp,
                                                   vp, vp, vp, vp, i32, vp, ctypes.c_float,
                                                   ctypes.c_int, ctypes.c_int, vp, vp, vp]
    lib.dflash_block_attention_noalloc.restype = ctypes.c_int
    lib.dflash_block_attention_noalloc_max_scratch_bytes.argtypes = []
    lib.dflash_block_attention_noalloc_max_scratch_bytes.restype = sz
    lib.dflash_ctx_prefill_workspace_bytes.argtypes = [G, ctypes.c_int, ctypes.c_int]
    lib.dflash_ctx_prefill_workspace_bytes.restype = sz
    lib.dflash_ctx_kv_prefill.argtypes = [G, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, vp, vp,
                                          vp, vp, vp, ctypes.POINTER(Weights), vp, vp, sz, vp, vp]
    lib.dflash_test_attention_skip_tile.argtypes = [ctypes.c_int]
    lib.dflash_test_attention_skip_tile.restype = None
    lib.dflash_packed_kv_bytes.argtypes = [G]
    lib.dflash_packed_kv_bytes.restype = sz
    lib.dflash_packed_gamma_bytes.argtypes = [G]
    lib.dflash_packed_gamma_bytes.restype = sz
    lib.dflash_pack_weights.argtypes = [G, ctypes.POINTER(LayerWeights), vp, vp, vp]
    lib.dflash_strict_accept.argtypes = [ctypes.c_int, ctypes.c_int, vp, i64, vp, i64, vp, vp, vp]
    lib.dflash_embedding_gather.argtypes = [ctypes.c_int, vp, vp, ctypes.c_int, ctypes.c_int, vp,
                                            vp, vp]
    lib.dflash_status_string.argtypes = [ctypes.c_int]
    lib.dflash_status_string.restype = ctypes.c_char_p
    lib.dflash_abi_version.argtypes = []
    for name in ("dflash_step_bookkeeping", "dflash_ctx_kv_update", "dflash_block_kv_scatter",
                 "dflash_block_attention", "dflash_attention_num_segments", "dflash_abi_version",
                 "dflash_ctx_kv_project", "dflash_ctx_kv_commit", "dflash_q_norm_rope",
                 "dflash_pack_weights", "dflash_strict_accept", "dflash_embedding_gather",
                 "dflash_ctx_kv_prefill", "dflash_block_scatter_attention"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


# ---------------------------------------------------------------- helpers


def make_geom(g: dict) -> Geom:
    """Geom from the dict form used by context_kv_update_gb300.inputs."""
    return Geom(kind=KIND_GQA if g["kind"] == "gqa" else KIND_MLA, num_layers=g["L"],
                d_in=g["D_in"], d_model=g["D"], hq=g["hq"],
                nkv=g["nkv"] if g["kind"] == "gqa" else 1,
                head_dim=g["hd"] if g["kind"] == "gqa" else 0,
                latent_dim=g.get("latent", 512), rope_dim=g.get("rope_dim", 64),
                page_size=g["P"], max_pages=g["max_pages"], num_pool_pages=g["num_pool_pages"],
                block_size=g["T"], reserved0=0, rope_theta=g["rope_theta"],
                eps_hidden=g["eps_h"], eps_k=g["eps_k"])


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn, code):
    if code != DFLASH_OK:
        raise DflashError(fn, code, _lib)


# ------------------------------------------------------------ entry points


def dflash_step_bookkeeping(geom, raw_offsets, off_div, accepted_tokens, n_accepted, ctx_len_pre,
                            valid, max_ctx, mask_token_id, out: dict, dev_status=None,
                            stream=None):
    """raw_offsets [B, >=M] / accepted_tokens [B, >=T] int32 CUDA tensors (row
    strided views allowed, unit column stride); out: dict of the
    dflash_step_outputs fields -> preallocated CUDA tensors."""
    lib = load()
    assert raw_offsets.stride(1) == 1 and accepted_tokens.stride(1) == 1
    o = StepOutputs(**{k: out[k].data_ptr() for k in STEP_OUTPUT_FIELDS})
    B = int(n_accepted.shape[0])
    _check("dflash_step_bookkeeping", lib.dflash_step_bookkeeping(
        ctypes.byref(geom), B, _ptr(raw_offsets), raw_offsets.stride(0), off_div,
        _ptr(accepted_tokens), accepted_tokens.stride(0), _ptr(n_accepted), _ptr(ctx_len_pre),
        _ptr(valid), max_ctx, mask_token_id, ctypes.byref(o), _ptr(dev_status), _stream(stream)))


def dflash_ctx_workspace_bytes(geom, B) -> int:
    return int(load().dflash_ctx_workspace_bytes(ctypes.byref(geom), B))


def dflash_ctx_kv_update(geom, hidden, n_accepted, ctx_len, alloc_limit, block_table, valid,
                         weights: dict, kv_pool, workspace, dev_status=None, stream=None):
    import torch
    lib = load()
    w = _weights(weights)
    dt = DTYPE_F32 if hidden.dtype == torch.float32 else DTYPE_BF16
    B = int(n_accepted.shape[0])
    _check("dflash_ctx_kv_update", lib.dflash_ctx_kv_update(
        ctypes.byref(geom), B, _ptr(hidden), dt, _ptr(n_accepted), _ptr(ctx_len),
        _ptr(alloc_limit), _ptr(block_table), _ptr(valid), ctypes.byref(w), _ptr(kv_pool),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_status),
        _stream(stream)))


def _weights(weights: dict):
    return Weights(w_fc=weights["w_fc"].data_ptr(), gamma_h=weights["g_h"].data_ptr(),
                   w_kv=weights["w_kv"].data_ptr(), gamma_k=weights["g_k"].data_ptr())


def dflash_ctx_staged_bytes(geom, B) -> int:
    return int(load().dflash_ctx_staged_bytes(ctypes.byref(geom), B))


def dflash_ctx_kv_project(geom, hidden, ctx_len, weights: dict, staged, workspace,
                          dev_status=None, stream=None):
    """Projection half of the split update: every row's stored values into
    `staged` (uint8 CUDA tensor of dflash_ctx_staged_bytes bytes)."""
    import torch
    lib = load()
    w = _weights(weights)
    dt = DTYPE_F32 if hidden.dtype == torch.float32 else DTYPE_BF16
    B = int(ctx_len.shape[0])
    _check("dflash_ctx_kv_project", lib.dflash_ctx_kv_project(
        ctypes.byref(geom), B, _ptr(hidden), dt, _ptr(ctx_len), ctypes.byref(w), _ptr(staged),
        staged.numel() * staged.element_size(), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)))


def dflash_ctx_kv_commit(geom, staged, n_accepted, ctx_len, alloc_limit, block_table, valid,
                         kv_pool, dev_status=None, stream=None):
    """Store half of the split update: masked paged store of the staged rows
    and the ctx_len advance."""
    lib = load()
    B = int(n_accepted.shape[0])
    _check("dflash_ctx_kv_commit", lib.dflash_ctx_kv_commit(
        ctypes.byref(geom), B, _ptr(staged), staged.numel() * staged.element_size(),
        _ptr(n_accepted), _ptr(ctx_len), _ptr(alloc_limit), _ptr(block_table), _ptr(valid),
        _ptr(kv_pool), _ptr(dev_status), _stream(stream)))


def dflash_q_norm_rope(geom, q_in, gamma_q, q_pos, q_out, dev_status=None, stream=None):
    """q_in / q_out bf16 CUDA tensors [B, Tq, hq, dim] (may be the same tensor),
    gamma_q [head_dim] (GQA) or None (MLA rope part), q_pos int32 [B, Tq]."""
    lib = load()
    B, Tq = int(q_pos.shape[0]), int(q_pos.shape[1])
    _check("dflash_q_norm_rope", lib.dflash_q_norm_rope(
        ctypes.byref(geom), B, Tq, _ptr(q_in), _ptr(gamma_q), _ptr(q_pos), _ptr(q_out),
        _ptr(dev_status), _stream(stream)))


def dflash_block_kv_scatter(geom, layer, blk_k, blk_v, blk_page, blk_slot, blk_mask, kv_pool,
                            dev_status=None, stream=None):
    lib = load()
    B = int(blk_page.shape[0])
    _check("dflash_block_kv_scatter", lib.dflash_block_kv_scatter(
        ctypes.byref(geom), B, layer, _ptr(blk_k), _ptr(blk_v), _ptr(blk_page), _ptr(blk_slot),
        _ptr(blk_mask), _ptr(kv_pool), _ptr(dev_status), _stream(stream)))


def dflash_attention_num_segments(geom, B, Tq) -> int:
    return int(load().dflash_attention_num_segments(ctypes.byref(geom), B, Tq))


def dflash_attention_workspace_bytes(geom, B, Tq, num_segments=0) -> int:
    return int(load().dflash_attention_workspace_bytes(ctypes.byref(geom), B, Tq, num_segments))


def dflash_block_attention(geom, layer, q, kv_pool, block_table, kv_len, out, workspace, *,
                           q_rope=None, window=0, sinks=None, scale=None,
                           mask_mode=MASK_CAUSAL_TAIL, num_segments=0, dev_status=None,
                           stream=None):
    lib = load()
    B, Tq = int(q.shape[0]), int(q.shape[1])
    scale = 0.0 if scale is None else scale  # 0 = the library's default scale
    _check("dflash_block_attention", lib.dflash_block_attention(
        ctypes.byref(geom), B, layer, Tq, _ptr(q), _ptr(q_rope), _ptr(kv_pool), _ptr(block_table),
        _ptr(kv_len), int(window), _ptr(sinks), float(scale), int(mask_mode), int(num_segments),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
        _ptr(dev_status), _stream(stream)))


def dflash_block_scatter_attention(geom, layer, blk_k, blk_v, blk_page, blk_slot, blk_mask, q,
                                   kv_pool, block_table, kv_len, out, workspace, *, q_rope=None,
                                   window=0, sinks=None, scale=None, mask_mode=MASK_CAUSAL_TAIL,
                                   num_segments=0, dev_status=None, stream=None):
    lib = load()
    B, Tq = int(q.shape[0]), int(q.shape[1])
    scale = 0.0 if scale is None else scale  # 0 = the library's default scale
    _check("dflash_block_scatter_attention", lib.dflash_block_scatter_attention(
        ctypes.byref(geom), B, layer, Tq, _ptr(blk_k), _ptr(blk_v), _ptr(blk_page),
        _ptr(blk_slot), _ptr(blk_mask), _ptr(q), _ptr(q_rope), _ptr(kv_pool), _ptr(block_table),
        _ptr(kv_len), int(window), _ptr(sinks), float(scale), int(mask_mode), int(num_segments),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
        _ptr(dev_status), _stream(stream)))


def dflash_block_attention_noalloc_max_scratch_bytes() -> int:
    return int(load().dflash_block_attention_noalloc_max_scratch_bytes())


def dflash_block_attention_noalloc(geom, layer, q, kv_pool, block_table, kv_len, out, *,
                                   q_rope=None, window=0, sinks=None, scale=None,
                                   mask_mode=MASK_CAUSAL_TAIL, num_segments=0, dev_status=None,
                                   stream=None):
    """dflash_block_attention with the library's fixed scratch (no workspace
    argument, nothing allocated)."""
    lib = load()
    B, Tq = int(q.shape[0]), int(q.shape[1])
    scale = 0.0 if scale is None else scale  # 0 = the library's default scale
    _check("dflash_block_attention_noalloc", lib.dflash_block_attention_noalloc(
        ctypes.byref(geom), B, layer, Tq, _ptr(q), _ptr(q_rope), _ptr(kv_pool), _ptr(block_table),
        _ptr(kv_len), int(window), _ptr(sinks), float(scale), int(mask_mode), int(num_segments),
        _ptr(out), _ptr(dev_status), _stream(stream)))


def dflash_packed_kv_bytes(geom) -> int:
    return int(load().dflash_packed_kv_bytes(ctypes.byref(geom)))


def dflash_packed_gamma_bytes(geom) -> int:
    return int(load().dflash_packed_gamma_bytes(ctypes.byref(geom)))


def dflash_pack_weights(geom, layers, w_kv, gamma_k, stream=None):
    """layers: one (w_k, w_v or None, k_norm) tuple of bf16 CUDA tensors per
    drafter layer; w_kv / gamma_k: preallocated CUDA outputs of
    dflash_packed_kv_bytes / dflash_packed_gamma_bytes bytes."""
    lib = load()
    arr = (LayerWeights * len(layers))(*[
        LayerWeights(w_k=wk.data_ptr(), w_v=None if wv is None else wv.data_ptr(),
                     k_norm=kn.data_ptr()) for wk, wv, kn in layers])
    _check("dflash_pack_weights", lib.dflash_pack_weights(
        ctypes.byref(geom), arr, _ptr(w_kv), _ptr(gamma_k), _stream(stream)))


def dflash_strict_accept(draft, target, n_accepted, accepted, stream=None):
    """draft int32 [B, K] / target int32 [B, K + 1] CUDA tensors (row-strided
    views allowed, unit column stride); n_accepted [B], accepted [B, K + 1]
    preallocated."""
    lib = load()
    B, K = int(target.shape[0]), int(target.shape[1]) - 1
    assert target.stride(1) == 1 and (K == 0 or draft.stride(1) == 1)
    _check("dflash_strict_accept", lib.dflash_strict_accept(
        B, K, _ptr(draft), draft.stride(0) if K > 0 else 0, _ptr(target), target.stride(0),
        _ptr(n_accepted), _ptr(accepted), _stream(stream)))


def dflash_embedding_gather(ids, table, out, dev_status=None, stream=None):
    """ids int32 CUDA tensor (any shape, contiguous), table bf16 [vocab, dim],
    out bf16 [ids.numel(), dim] (or ids.shape + (dim,))."""
    lib = load()
    vocab, dim = int(table.shape[0]), int(table.shape[1])
    _check("dflash_embedding_gather", lib.dflash_embedding_gather(
        int(ids.numel()), _ptr(ids), _ptr(table), vocab, dim, _ptr(out), _ptr(dev_status),
        _stream(stream)))


def dflash_ctx_prefill_workspace_bytes(geom, B, n_rows) -> int:
    return int(load().dflash_ctx_prefill_workspace_bytes(ctypes.byref(geom), B, n_rows))


def dflash_ctx_kv_prefill(geom, hidden, cu_rows, ctx_len, alloc_limit, block_table, valid,
                          weights: dict, kv_pool, workspace, dev_status=None, stream=None):
    """hidden [n_rows, d_in] CUDA tensor (bf16 or fp32), cu_rows int32 [B + 1]
    (request r = rows cu_rows[r]..cu_rows[r+1]-1), ctx_len int32 [B] (in:
    start positions, out: advanced)."""
    import torch
    lib = load()
    w = _weights(weights)
    dt = DTYPE_F32 if hidden.dtype == torch.float32 else DTYPE_BF16
    B = int(ctx_len.shape[0])
    _check("dflash_ctx_kv_prefill", lib.dflash_ctx_kv_prefill(
        ctypes.byref(geom), B, int(hidden.shape[0]), _ptr(hidden), dt, _ptr(cu_rows),
        _ptr(ctx_len), _ptr(alloc_limit), _ptr(block_table), _ptr(valid), ctypes.byref(w),
        _ptr(kv_pool), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _stream(stream)))


def dflash_test_attention_skip_tile(tile: int) -> None:
    """Tests of the bounded-wait path only (see include/dflash.h)."""
    load().dflash_test_attention_skip_tile(int(tile))
