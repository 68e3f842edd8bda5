"""Seeded synthetic inputs for the drafter decode-step hot path.

This module holds data generation only -- shapes, distributions and page
allocations -- and none of the method's arithmetic.  It is the one module
shared by the CUDA path's tests / benchmark and by the CPU oracle; it imports
neither of them.

Recipe (every draw from ``numpy.random.default_rng`` over
``SeedSequence(seed).spawn(N_STREAMS)``, one stream per tensor, in the fixed
order of ``_STREAMS``):

* weights ~ N(0, 0.02) rounded to bf16; norm gains 1 + N(0, 0.02) in bf16;
* target hidden rows ~ N(0, 1) (fp32 for the tiny workload, bf16 otherwise);
* KV pool pre-filled with N(0, 1) bf16; q ~ N(0, 1) bf16; sinks ~ N(0, 1) fp32;
* physical pages: a random permutation of the pool handed out to requests in
  order; raw offsets are page * off_div for allocated entries, -1 elsewhere.

bf16 tensors are numpy ``uint16`` arrays of bf16 bit patterns.
"""
from __future__ import annotations

import math

import numpy as np

_STREAMS = ("hidden", "w_fc", "g_h", "w_kv", "g_k", "n_acc", "ctx_len", "pages", "pool", "q",
            "sinks", "blk", "acc", "misc")
N_STREAMS = len(_STREAMS)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 data to bf16 (nearest-even) and return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rngs(seed: int) -> dict:
    ss = np.random.SeedSequence(seed).spawn(N_STREAMS)
    return {name: np.random.default_rng(s) for name, s in zip(_STREAMS, ss)}


def _normal_bf16(rng, shape, std=1.0, mean=0.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return f32_to_bf16_bits(x)


# ------------------------------------------------------------- workloads
#
# Geometry keys: kind ("gqa" | "mla"), L, D_in, D, hq, nkv, hd, latent,
# rope_dim, P (page size), T (block size), rope_theta, eps_h, eps_k.

TINY = dict(kind="gqa", B=1, L=1, D_in=256, D=256, hidden_dtype="f32", hq=4, nkv=2, hd=64,
            T=4, P=16, rope_theta=1e4, eps_h=1e-6, eps_k=1e-6, ctx=[100], n_acc=[3],
            alloc_pages=[10], pool_pages=16, max_pages=16, max_ctx=1 << 30)

QWEN3_8B = dict(kind="gqa", B=1, L=5, D_in=4096, D=4096, hidden_dtype="bf16", hq=32, nkv=8,
                hd=128, T=16, P=64, rope_theta=1e6, eps_h=1e-6, eps_k=1e-6, ctx=[32768],
                n_acc=None, alloc_pages=None, pool_pages=None, max_pages=None,
                max_ctx=1 << 30)

SLIDING_WINDOW = dict(kind="gqa", B=1, L=1, D_in=4096, D=4096, hidden_dtype="bf16", hq=32,
                      nkv=2, hd=128, T=3, P=64, rope_theta=1e6, eps_h=1e-6, eps_k=1e-6,
                      ctx=[131072 - 3], n_acc=[3], alloc_pages=None, pool_pages=None,
                      max_pages=None, max_ctx=1 << 30, window=1024, sinks=True)

MLA = dict(kind="mla", B=1, L=3, D_in=4096, D=4096, hidden_dtype="bf16", hq=64, nkv=1,
           hd=576, latent=512, rope_dim=64, T=8, P=64, rope_theta=1e6, eps_h=1e-6,
           eps_k=1e-6, ctx=[32768], n_acc=None, alloc_pages=None, pool_pages=None,
           max_pages=None, max_ctx=1 << 30)

WORKLOADS = {"tiny": TINY, "qwen3_8b": QWEN3_8B, "sliding_window": SLIDING_WINDOW, "mla": MLA}


def batch_sweep(B: int) -> dict:
    """Qwen3-8B geometry with B requests, ctx ~ U[1K, 8K], n ~ U{1..8}, 10% at
    the allocation ceiling (those get A = c + floor(n / 2))."""
    return dict(QWEN3_8B, B=B, ctx=None, n_acc=None, sweep=True)


def workload(name: str, **over) -> dict:
    if name.startswith("batch_sweep_"):
        cfg = batch_sweep(int(name.rsplit("_", 1)[1]))
    else:
        cfg = dict(WORKLOADS[name])
    cfg.update(over)
    cfg["name"] = name
    return cfg


# ---------------------------------------------------------------- problem


def make_problem(cfg: dict, seed: int = 0, *, with_weights: bool = True,
                 with_pool: bool = True, off_div: int = 1) -> dict:
    """Build every input of one decode step for workload ``cfg``.

    Returns a dict with the geometry under ``"g"`` and numpy arrays:
    hidden, n_acc, ctx_len (pre-step), acc (accepted tokens), raw_offsets,
    pages (physical page ids, -1 unallocated), valid, weights, pool, q (per
    layer), sinks, blk_k / blk_v (or blk_lat) per layer.
    """
    R = _rngs(seed)
    B, T, P, L = cfg["B"], cfg["T"], cfg["P"], cfg["L"]
    kind = cfg["kind"]

    # per-request step scalars
    if cfg.get("n_acc") is not None:
        n_acc = np.asarray(cfg["n_acc"], np.int32)
    else:
        hi = 8 if cfg.get("sweep") else T
        n_acc = R["n_acc"].integers(1, hi + 1, size=B).astype(np.int32)
    ceiling = np.zeros(B, bool)
    if cfg.get("ctx") is not None:
        ctx = np.asarray(cfg["ctx"], np.int32)
        if ctx.size == 1 and B > 1:
            ctx = np.full(B, ctx[0], np.int32)
    else:
        ctx = R["ctx_len"].integers(1024, 8192 + 1, size=B).astype(np.int32)
        if cfg.get("sweep"):
            k = max(1, int(round(0.1 * B))) if B >= 2 else 0
            ceiling[R["misc"].permutation(B)[:k]] = True

    # pages each request owns: enough for c + 2T (rounded up to a page)
    if cfg.get("alloc_pages") is not None:
        alloc_pages = np.asarray(cfg["alloc_pages"], np.int64)
    else:
        alloc_pages = -(-(ctx.astype(np.int64) + 2 * T) // P)
    alloc_lim = alloc_pages * P
    for r in np.nonzero(ceiling)[0]:
        # make A_r = c_r + floor(n_r / 2) fall inside this step's accepted rows
        a = int(alloc_pages[r]) * P
        ctx[r] = a - int(n_acc[r]) // 2
        alloc_lim[r] = a
    max_pages = cfg.get("max_pages") or int(alloc_pages.max()) + 2
    pool_pages = cfg.get("pool_pages") or int(alloc_pages.sum()) + 4
    perm = R["pages"].permutation(pool_pages).astype(np.int32)
    pages = np.full((B, max_pages), -1, np.int32)
    pos = 0
    for r in range(B):
        n = int(alloc_pages[r])
        pages[r, :n] = perm[pos:pos + n]
        pos += n
    assert pos <= pool_pages
    raw_offsets = np.where(pages >= 0, pages * off_div, -1).astype(np.int32)

    g = dict(kind=kind, L=L, D_in=cfg["D_in"], D=cfg["D"], hq=cfg["hq"], nkv=cfg["nkv"],
             hd=cfg["hd"], latent=cfg.get("latent", 512), rope_dim=cfg.get("rope_dim", 64),
             P=P, T=T, max_pages=max_pages, num_pool_pages=pool_pages,
             rope_theta=float(cfg["rope_theta"]), eps_h=float(cfg["eps_h"]),
             eps_k=float(cfg["eps_k"]))

    prob = dict(cfg=cfg, g=g, B=B, n_acc=n_acc, ctx_len=ctx.astype(np.int32),
                alloc_limit=np.minimum(alloc_lim, cfg["max_ctx"]).astype(np.int32),
                pages=pages, raw_offsets=raw_offsets, off_div=off_div,
                valid=np.ones(B, np.uint8), max_ctx=int(cfg["max_ctx"]), mask_id=151669)
    prob["acc"] = R["acc"].integers(0, 151936, size=(B, T)).astype(np.int32)

    D_in, D = cfg["D_in"], cfg["D"]
    if cfg.get("hidden_dtype") == "f32":
        prob["hidden"] = R["hidden"].standard_normal(size=(B, T, D_in), dtype=np.float32)
    else:
        prob["hidden"] = _normal_bf16(R["hidden"], (B, T, D_in))

    if with_weights:
        prob["w_fc"] = _normal_bf16(R["w_fc"], (D, D_in), std=0.02)
        prob["g_h"] = _normal_bf16(R["g_h"], (D,), std=0.02, mean=1.0)
        if kind == "gqa":
            nkv, hd = cfg["nkv"], cfg["hd"]
            prob["w_kv"] = _normal_bf16(R["w_kv"], (L, 2, nkv, hd, D), std=0.02)
            prob["g_k"] = _normal_bf16(R["g_k"], (L, hd), std=0.02, mean=1.0)
        else:
            lat, rope = cfg["latent"], cfg["rope_dim"]
            prob["w_kv"] = _normal_bf16(R["w_kv"], (L, lat + rope, D), std=0.02)
            prob["g_k"] = _normal_bf16(R["g_k"], (L, lat), std=0.02, mean=1.0)

    if with_pool:
        if kind == "gqa":
            shape = (L, pool_pages, 2, cfg["nkv"], P, cfg["hd"])
        else:
            shape = (L, pool_pages, P, cfg["latent"] + cfg["rope_dim"])
        prob["pool"] = _normal_bf16(R["pool"], shape)

    # per-layer drafter queries / block K/V (inputs of the attention stage)
    hq = cfg["hq"]
    if kind == "gqa":
        prob["q"] = _normal_bf16(R["q"], (L, B, T, hq, cfg["hd"]))
        prob["blk_k"] = _normal_bf16(R["blk"], (L, B, T, cfg["nkv"], cfg["hd"]))
        prob["blk_v"] = _normal_bf16(R["blk"], (L, B, T, cfg["nkv"], cfg["hd"]))
    else:
        lat, rope = cfg["latent"], cfg["rope_dim"]
        prob["q_lat"] = _normal_bf16(R["q"], (L, B, T, hq, lat))
        prob["q_rope"] = _normal_bf16(R["q"], (L, B, T, hq, rope))
        prob["blk_lat"] = _normal_bf16(R["blk"], (L, B, T, lat + rope))
    prob["sinks"] = R["sinks"].standard_normal(size=(L, hq), dtype=np.float32)
    prob["window"] = int(cfg.get("window", 0))
    prob["use_sinks"] = bool(cfg.get("sinks", False))
    return prob


def attention_scale(g: dict) -> float:
    """Softmax scale the workloads use: 1/sqrt(hd) (GQA), 1/sqrt(128 + 64) (MLA)."""
    if g["kind"] == "gqa":
        return 1.0 / math.sqrt(g["hd"])
    return 1.0 / math.sqrt(128 + 64)
