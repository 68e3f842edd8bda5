"""The oracle's split context update (projection before acceptance, store
after the join; TensorRT-LLM PR #20550, Description, overlapped context
projection) against the oracle's fused update, which the pins of
test_oracle_pins.py tie to the pages: projection + commit must leave the pool
and ctx_len bit-identical, for live, dummy, masked, ceiling and bad-page rows.
"""
import numpy as np
import pytest

import oracle
from context_kv_update_gb300 import inputs


def _fused(prob, valid, tbl, alloc):
    g = prob["g"]
    pool = prob["pool"].copy()
    upd = oracle.ctx_kv_update_gqa if g["kind"] == "gqa" else oracle.ctx_kv_update_mla
    ctx = upd(g, prob["hidden"], prob["n_acc"], prob["ctx_len"], alloc, tbl, valid,
              prob["w_fc"], prob["g_h"], prob["w_kv"], prob["g_k"], pool)
    return pool, ctx


def _split(prob, valid, tbl, alloc):
    g = prob["g"]
    staged_c, staged = oracle.ctx_kv_project(g, prob["hidden"], prob["ctx_len"], prob["w_fc"],
                                             prob["g_h"], prob["w_kv"], prob["g_k"])
    pool = prob["pool"].copy()
    ctx = oracle.ctx_kv_commit(g, staged_c, staged, prob["n_acc"], alloc, tbl, valid, pool)
    return pool, ctx, staged_c, staged


def _cases():
    small = dict(D_in=128, D=192)
    return [
        ("tiny", {}),
        ("tiny", dict(small, B=3, L=2, T=8, nkv=2, hq=4, hd=64, hidden_dtype="bf16",
                      ctx=[10, 40, 75], n_acc=[8, 3, 5], alloc_pages=[6, 6, 6], pool_pages=24,
                      max_pages=8)),
        ("mla", dict(small, ctx=[300], n_acc=[6])),
    ]


@pytest.mark.parametrize("name,over", _cases())
def test_split_update_equals_fused(name, over):
    prob = inputs.make_problem(inputs.workload(name, **over), seed=3)
    B = prob["B"]
    tbl = prob["pages"].copy()
    alloc = prob["alloc_limit"].copy()
    valid = np.ones(B, np.uint8)
    if B >= 3:
        valid[1] = 0                                    # a dummy slot
        alloc[2] = int(prob["ctx_len"][2]) + 2          # ceiling after two rows
        c0 = int(prob["ctx_len"][0])
        tbl[0, (c0 + 5) // prob["g"]["P"]] = -1          # an unmapped page
    pool_f, ctx_f = _fused(prob, valid, tbl, alloc)
    pool_s, ctx_s, staged_c, staged = _split(prob, valid, tbl, alloc)
    np.testing.assert_array_equal(staged_c, prob["ctx_len"])
    np.testing.assert_array_equal(ctx_s, ctx_f)
    np.testing.assert_array_equal(pool_s, pool_f)
    assert (pool_f != prob["pool"]).any()


def test_projection_ignores_the_mask_inputs():
    """The projection reads only the hidden rows, the weights and the
    pre-step ctx_len: rows past n_accepted are projected too, and their staged
    values are the ones a longer acceptance would store."""
    prob = inputs.make_problem(inputs.workload("tiny"), seed=4)
    g = prob["g"]
    _, staged = oracle.ctx_kv_project(g, prob["hidden"], prob["ctx_len"], prob["w_fc"],
                                      prob["g_h"], prob["w_kv"], prob["g_k"])
    full = dict(prob)
    full["n_acc"] = np.full(prob["B"], g["T"], np.int32)
    pool_f, _ = _fused(full, None, prob["pages"], np.full(prob["B"], 1 << 30, np.int32))
    # every row of the block landed in the pool of the fully accepted step
    c = int(prob["ctx_len"][0])
    P, nkv, hd = g["P"], g["nkv"], g["hd"]
    for i in range(g["T"]):
        page, slot = prob["pages"][0, (c + i) // P], (c + i) % P
        for kv in range(2):
            for h in range(nkv):
                got = staged[i].reshape(g["L"], 2, nkv, hd)[0, kv, h]
                np.testing.assert_array_equal(got, pool_f[0, page, kv, h, slot])
