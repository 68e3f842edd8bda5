"""dflash_block_attention_noalloc: the block attention for callers that cannot
allocate device memory where they run it (a plugin whose framework owns all
device buffers and hands it no allocator, an allocation-free real-time loop).
Its scratch is a fixed array inside the library, so the test calls it through
the C ABI with no workspace and checks its output against
dflash_block_attention's (which takes a caller workspace) and against the CPU
oracle, within the parity tolerance, on two calls in a row with different
problems (the second call finds the first one's partials in the shared array).

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process."""
import numpy as np
import pytest

import oracle
from context_kv_update_gb300 import inputs
from tests.gpu_helpers import assert_close, bf16_f64, bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_kv_update_gb300 import build
    build.build()
    import context_kv_update_gb300 as dl
    dl.load()
    return dl


def _case(seed, ctx, Tq, window, use_sinks):
    prob = inputs.make_problem(inputs.workload("qwen3_8b", ctx=[ctx], T=Tq, L=2), seed=seed,
                               with_weights=False)
    return prob, prob["g"], window, (prob["sinks"][1] if use_sinks else None)


def _both(dl, prob, g, window, sinks):
    import torch
    geom = dl.make_geom(g)
    B, T, hq, hd = prob["B"], g["T"], g["hq"], g["hd"]
    q = to_dev(prob["q"][1])
    pool = to_dev(prob["pool"])
    tbl = to_dev(prob["pages"])
    kv_len = to_dev(np.array([int(prob["ctx_len"][0]) + T], np.int32))
    s = None if sinks is None else to_dev(sinks)
    ws = torch.empty(dl.dflash_attention_workspace_bytes(geom, B, T, 0), dtype=torch.uint8,
                     device="cuda")
    ref = torch.empty((B, T, hq, hd), dtype=torch.bfloat16, device="cuda")
    dl.dflash_block_attention(geom, 1, q, pool, tbl, kv_len, ref, ws, window=window, sinks=s)
    out = torch.full((B, T, hq, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dflash_block_attention_noalloc(geom, 1, q, pool, tbl, kv_len, out, window=window, sinks=s,
                                      dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return bf16_f64(bits(ref)), bf16_f64(bits(out))


def test_noalloc_matches_workspace_entry_point_and_oracle_twice(dl):
    # first call: 4K context, 16 queries, sinks; second: 9K context, 3 queries, window
    for seed, ctx, Tq, window, use_sinks in ((1, 4096, 16, 0, True), (2, 9000, 3, 700, False)):
        prob, g, window, sinks = _case(seed, ctx, Tq, window, use_sinks)
        ref, out = _both(dl, prob, g, window, sinks)
        assert_close(out, ref, f"noalloc vs workspace entry point ctx={ctx} Tq={Tq}")
        kv_len = np.array([int(prob["ctx_len"][0]) + g["T"]], np.int32)
        want = oracle.attention_gqa(g, 1, prob["q"][1], prob["pool"], prob["pages"], kv_len,
                                    window=window, sinks=sinks)
        assert_close(out, want, f"noalloc vs oracle ctx={ctx} Tq={Tq}")


def test_noalloc_rejects_problems_beyond_its_scratch(dl):
    import ctypes
    from context_kv_update_gb300 import _lib
    prob = inputs.make_problem(inputs.workload("qwen3_8b", ctx=[2048]), seed=0, with_weights=False,
                               with_pool=False)
    geom = dl.make_geom(prob["g"])
    cap = dl.dflash_block_attention_noalloc_max_scratch_bytes()
    assert cap == 32 << 20
    # many requests and segments: the split-KV scratch would exceed the fixed array
    B, Tq, S = 64, 16, 64
    assert dl.dflash_attention_workspace_bytes(geom, B, Tq, S) > cap
    # every buffer is NULL: the size limit is checked before the pointers, so a
    # library that lost the limit stops at the NULL check and launches nothing
    lib = _lib.load()
    rc = lib.dflash_block_attention_noalloc(ctypes.byref(geom), B, 0, Tq, None, None, None, None,
                                            None, 0, None, 0.0, 0, S, None, None, None)
    assert rc == _lib.DFLASH_ERR_WORKSPACE_TOO_SMALL
    # argument errors come first, as for dflash_block_attention
    rc = lib.dflash_block_attention_noalloc(ctypes.byref(geom), B, 0, Tq, None, None, None, None,
                                            None, 0, None, 0.0, 9, S, None, None, None)
    assert rc == _lib.DFLASH_ERR_INVALID_ARG
