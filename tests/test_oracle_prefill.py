"""Pins of the oracle's prefill context store (TensorRT-LLM PR #20550,
Description, TLLM_DFLASH_FUSED_PROLOGUE: the single-latent
_store_context_kv_paged scatter used by prefill):

- one request's prompt rows are exactly one decode-update block with every
  row accepted (the decode update is pinned on its own, tests/test_oracle_pins.py);
- requests are independent: one varlen call equals one call per request;
- a row one position later is the same key rotated by one RoPE step (the
  2x2 rotation of each dimension pair, written here from the definition);
- rows past the allocation limit or on an unmapped page are not stored, and
  nothing but the destinations changes."""
import numpy as np
import pytest

import oracle
from context_kv_update_gb300 import inputs


def _geom(kind):
    if kind == "gqa":
        return dict(kind="gqa", L=2, D_in=64, D=64, hq=4, nkv=2, hd=16, P=8, T=0,
                    num_pool_pages=12, rope_theta=1e4, eps_h=1e-6, eps_k=1e-6)
    return dict(kind="mla", L=2, D_in=64, D=64, hq=4, nkv=1, hd=0, latent=32, rope_dim=16, P=8,
                T=0, num_pool_pages=12, rope_theta=1e4, eps_h=1e-6, eps_k=1e-6)


def _weights(g, rng):
    bf = lambda a: inputs.f32_to_bf16_bits(a.astype(np.float32))  # noqa: E731
    D, D_in, L = g["D"], g["D_in"], g["L"]
    w_fc = bf(rng.standard_normal((D, D_in)) * 0.1)
    g_h = bf(1 + 0.02 * rng.standard_normal(D))
    if g["kind"] == "gqa":
        w_kv = bf(rng.standard_normal((L, 2, g["nkv"], g["hd"], D)) * 0.1)
        g_k = bf(1 + 0.02 * rng.standard_normal((L, g["hd"])))
    else:
        w_kv = bf(rng.standard_normal((L, g["latent"] + g["rope_dim"], D)) * 0.1)
        g_k = bf(1 + 0.02 * rng.standard_normal((L, g["latent"])))
    return w_fc, g_h, w_kv, g_k


def _pool(g, rng):
    if g["kind"] == "gqa":
        shape = (g["L"], g["num_pool_pages"], 2, g["nkv"], g["P"], g["hd"])
    else:
        shape = (g["L"], g["num_pool_pages"], g["P"], g["latent"] + g["rope_dim"])
    return rng.integers(1, 65535, size=shape).astype(np.uint16)


@pytest.mark.parametrize("kind", ["gqa", "mla"])
def test_prefill_of_one_request_is_one_all_accepted_update_block(kind):
    rng = np.random.default_rng(1)
    g = _geom(kind)
    w = _weights(g, rng)
    n, c = 11, 5
    M = 6
    tbl = rng.permutation(g["num_pool_pages"])[:M].astype(np.int32)[None]
    hidden = inputs.f32_to_bf16_bits(rng.standard_normal((n, g["D_in"])).astype(np.float32))
    alloc = np.array([M * g["P"]], np.int32)
    pool0 = _pool(g, rng)
    pa = pool0.copy()
    ca = oracle.ctx_kv_prefill(g, hidden, np.array([0, n], np.int32), np.array([c], np.int32),
                               alloc, tbl, None, *w, pa)
    pb = pool0.copy()
    upd = oracle.ctx_kv_update_gqa if kind == "gqa" else oracle.ctx_kv_update_mla
    cb = upd(dict(g, T=n), hidden[None], np.array([n], np.int32), np.array([c], np.int32), alloc,
             tbl, None, *w, pb)
    np.testing.assert_array_equal(pa, pb)
    np.testing.assert_array_equal(ca, cb)
    assert ca[0] == c + n
    assert (pa != pool0).any()


@pytest.mark.parametrize("kind", ["gqa", "mla"])
def test_prefill_requests_are_independent(kind):
    rng = np.random.default_rng(2)
    g = _geom(kind)
    w = _weights(g, rng)
    M = 4
    n_r = [5, 0, 7, 3, 4]
    c_r = [2, 3, 9, -1, 0]
    valid = np.array([1, 1, 1, 1, 0], np.uint8)
    B = len(n_r)
    cu = np.concatenate([[0], np.cumsum(n_r)]).astype(np.int32)
    perm = rng.permutation(g["num_pool_pages"]).astype(np.int32)
    tbl = np.full((B, M), -1, np.int32)
    tbl[0, :2], tbl[1, :1], tbl[2, :3], tbl[3, :1], tbl[4, :1] = (
        perm[0:2], perm[2:3], perm[3:6], perm[6:7], perm[7:8])
    tbl[2, 1] = -1                       # an unmapped page in the middle
    alloc = np.array([16, 8, 14, 8, 8], np.int32)  # request 2 runs into its ceiling
    hidden = inputs.f32_to_bf16_bits(rng.standard_normal((cu[-1], g["D_in"])).astype(np.float32))
    pool0 = _pool(g, rng)
    pa = pool0.copy()
    ca = oracle.ctx_kv_prefill(g, hidden, cu, np.array(c_r, np.int32), alloc, tbl, valid, *w, pa)
    pb = pool0.copy()
    cb = []
    for r in range(B):
        cb.append(oracle.ctx_kv_prefill(
            g, np.ascontiguousarray(hidden[cu[r]:cu[r + 1]]), np.array([0, n_r[r]], np.int32),
            np.array([c_r[r]], np.int32), alloc[r:r + 1], tbl[r:r + 1], valid[r:r + 1], *w,
            pb)[0])
    np.testing.assert_array_equal(pa, pb)
    np.testing.assert_array_equal(ca, np.array(cb))
    # advance: live rows clamp at the ceiling; the dummy (c < 0) and the
    # invalid slot report 0
    assert ca.tolist() == [7, 3, 14, 0, 0]


def _rotate(x, pos, theta):
    """Rotate-half RoPE written from its definition: dimension j pairs with
    j + d/2 and turns by pos * theta^(-2j/d)."""
    d = x.shape[-1]
    j = np.arange(d // 2)
    a = pos * theta ** (-2.0 * j / d)
    lo, hi = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([lo * np.cos(a) - hi * np.sin(a), hi * np.cos(a) + lo * np.sin(a)],
                          axis=-1)


def test_prefill_position_shift_is_one_rope_step():
    rng = np.random.default_rng(3)
    g = _geom("gqa")
    w = _weights(g, rng)
    row = inputs.f32_to_bf16_bits(rng.standard_normal((1, g["D_in"])).astype(np.float32))
    hidden = np.concatenate([row, row])
    cu = np.array([0, 1, 2], np.int32)
    c = np.array([20, 21], np.int32)
    perm = rng.permutation(g["num_pool_pages"]).astype(np.int32)
    tbl = np.stack([perm[:4], perm[4:8]]).astype(np.int32)
    pool = _pool(g, rng)
    oracle.ctx_kv_prefill(g, hidden, cu, c, np.array([32, 32], np.int32), tbl, None, *w, pool)
    P = g["P"]
    k0 = oracle.bf16_to_f64(pool[:, tbl[0, 20 // P], 0, :, 20 % P])
    k1 = oracle.bf16_to_f64(pool[:, tbl[1, 21 // P], 0, :, 21 % P])
    v0 = pool[:, tbl[0, 20 // P], 1, :, 20 % P]
    v1 = pool[:, tbl[1, 21 // P], 1, :, 21 % P]
    np.testing.assert_array_equal(v0, v1)  # V carries no position
    # k1 = R(21) n, k0 = R(20) n  =>  R(-20) k0 == R(-21) k1 up to the bf16 stores
    np.testing.assert_allclose(_rotate(k0, -20.0, g["rope_theta"]),
                               _rotate(k1, -21.0, g["rope_theta"]), atol=2e-2, rtol=2e-2)
    assert not np.allclose(k0, k1, atol=1e-3)


def test_prefill_changes_only_its_destinations():
    rng = np.random.default_rng(4)
    g = _geom("mla")
    w = _weights(g, rng)
    n, c = 9, 3
    tbl = np.array([[4, -1, 7, 2]], np.int32)      # page 1 unmapped
    alloc = np.array([10], np.int32)             # positions 3..9 of 3..11 stored
    hidden = inputs.f32_to_bf16_bits(rng.standard_normal((n, g["D_in"])).astype(np.float32))
    pool0 = _pool(g, rng)
    pool = pool0.copy()
    ctx = oracle.ctx_kv_prefill(g, hidden, np.array([0, n], np.int32), np.array([c], np.int32),
                                alloc, tbl, None, *w, pool)
    assert ctx.tolist() == [10]
    P = g["P"]
    expect = {(int(tbl[0, p // P]), p % P) for p in range(c, 10) if tbl[0, p // P] >= 0}
    changed = {(int(a), int(b)) for a, b in np.argwhere((pool != pool0).any(axis=-1).any(axis=0))}
    assert changed == expect
    # the stored latent is RMS-normalised (gain ~1): unit RMS within bf16
    lat = g["latent"]
    pg, sl = next(iter(expect))
    x = oracle.bf16_to_f64(pool[0, pg, sl, :lat]) / oracle.bf16_to_f64(w[3][0])
    assert abs(np.sqrt(np.mean(x ** 2)) - 1.0) < 1e-2
