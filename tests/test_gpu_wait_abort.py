"""The bounded-wait path of the attention kernels, exercised without any
fault: a test-only hook makes the producer leave one key tile (MLA: one
64-key half-tile) unloaded, so the MMA issuer's wait for it runs out (about
2 s).  Every role then winds down
(the softmax warps and the PV issuer see the shared abort flag, each MMA
issuer waits for its own MMAs, the producer waits a bounded time for copies
in flight, TMEM is freed), the kernel returns, DFLASH_DEV_WAIT_TIMEOUT is set
in the device status, and the context stays usable: the next call, with the
hook off, matches the oracle.  Tiny case, one segment per KV head."""
import time

import numpy as np
import pytest

import oracle
from tests.gpu_helpers import assert_close, bf16_f64, bits, to_dev
from tests.test_gpu_attention import _gqa_case, _mla_case

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


def test_unloaded_tile_times_out_cleanly_and_the_context_survives(dl):
    import torch
    kv_lens = [1000]  # 8 tiles of 128 keys, all in one segment
    g, pool, tbl, q, sinks = _gqa_case(31, kv_lens, hq=4, nkv=2, hd=64, P=16, Tq=2)
    geom = dl.make_geom(g)
    B, Tq, hq, hd = q.shape
    q_d, pool_d, tbl_d = to_dev(q), to_dev(pool), to_dev(tbl)
    kv_d = to_dev(np.asarray(kv_lens, np.int32))
    ws = torch.empty(dl.dflash_attention_workspace_bytes(geom, B, Tq, 1), dtype=torch.uint8,
                     device="cuda")
    out = torch.zeros((B, Tq, hq, hd), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dflash_test_attention_skip_tile(2)
    try:
        t0 = time.time()
        dl.dflash_block_attention(geom, 0, q_d, pool_d, tbl_d, kv_d, out, ws, num_segments=1,
                                  dev_status=st)
        torch.cuda.synchronize()
        took = time.time() - t0
    finally:
        dl.dflash_test_attention_skip_tile(-1)
    assert int(st.item()) & dl._lib.DEV_WAIT_TIMEOUT
    assert took < 30.0
    # the context is intact: the same call without the hook matches the oracle
    st.zero_()
    dl.dflash_block_attention(geom, 0, q_d, pool_d, tbl_d, kv_d, out, ws, num_segments=1,
                              dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.attention_gqa(g, 0, q, pool, tbl, np.asarray(kv_lens))
    assert_close(bf16_f64(bits(out)), ref, "after the timed-out call")


def test_mla_unloaded_half_tile_times_out_cleanly_and_the_context_survives(dl):
    """The MLA kernel's wind-down: the issuers' readiness loop runs out of
    time on the missing half-tile, the softmax's wait too, the producer waits
    only for the copies it issued, TMEM is freed, and the next call matches
    the oracle."""
    import torch
    kv_lens = [1000]  # 8 tiles of 128 keys (16 half-tiles), all in one segment
    g, pool, tbl, ql, qr, sinks = _mla_case(32, kv_lens, hq=16, P=64, Tq=2)
    geom = dl.make_geom(g)
    B, Tq, hq, lat = ql.shape
    ql_d, qr_d, pool_d, tbl_d = to_dev(ql), to_dev(qr), to_dev(pool), to_dev(tbl)
    kv_d = to_dev(np.asarray(kv_lens, np.int32))
    ws = torch.empty(dl.dflash_attention_workspace_bytes(geom, B, Tq, 1), dtype=torch.uint8,
                     device="cuda")
    out = torch.zeros((B, Tq, hq, lat), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dflash_test_attention_skip_tile(3)
    try:
        t0 = time.time()
        dl.dflash_block_attention(geom, 0, ql_d, pool_d, tbl_d, kv_d, out, ws, q_rope=qr_d,
                                  num_segments=1, dev_status=st)
        torch.cuda.synchronize()
        took = time.time() - t0
    finally:
        dl.dflash_test_attention_skip_tile(-1)
    assert int(st.item()) & dl._lib.DEV_WAIT_TIMEOUT
    assert took < 30.0
    st.zero_()
    dl.dflash_block_attention(geom, 0, ql_d, pool_d, tbl_d, kv_d, out, ws, q_rope=qr_d,
                              num_segments=1, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.attention_mla(g, 0, ql, qr, pool, tbl, np.asarray(kv_lens))
    assert_close(bf16_f64(bits(out)), ref, "after the timed-out call")
