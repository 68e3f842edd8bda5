"""GPU parity of the split context update (dflash_ctx_kv_project before
acceptance, dflash_ctx_kv_commit after the join; TensorRT-LLM PR #20550,
Description, overlapped context projection):

- project + commit leave the pool and ctx_len bit-identical to the fused
  dflash_ctx_kv_update on the same inputs;
- the staged rows match the oracle's projection within tolerance, and the
  recorded pre-step lengths exactly;
- commit of the GPU's own staged rows matches the oracle's commit of the same
  rows bit for bit (it is a masked copy).
"""
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


def _dev_inputs(prob):
    import torch
    hid = prob["hidden"]
    hid_d = to_dev(hid) if hid.dtype == np.uint16 else torch.from_numpy(hid).cuda()
    w = {k: to_dev(prob[k]) for k in ("w_fc", "g_h", "w_kv", "g_k")}
    return hid_d, w


def _staged_views(staged, B, N, W):
    """(c int32 [B], rows uint16 [N, W]) of a staged buffer."""
    raw = staged.cpu().numpy()
    off = (4 * B + 255) // 256 * 256
    return raw[:4 * B].view(np.int32), raw[off:off + N * W * 2].view(np.uint16).reshape(N, W)


def _run(dl, prob, valid, tbl, alloc):
    import torch
    g = prob["g"]
    geom = dl.make_geom(g)
    B, T = prob["B"], g["T"]
    hid_d, w = _dev_inputs(prob)
    ws = torch.empty(dl.dflash_ctx_workspace_bytes(geom, B), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    valid_d = None if valid is None else to_dev(valid)
    # fused
    pool_f = to_dev(prob["pool"])
    ctx_f = to_dev(prob["ctx_len"])
    dl.dflash_ctx_kv_update(geom, hid_d, to_dev(prob["n_acc"]), ctx_f, to_dev(alloc), to_dev(tbl),
                            valid_d, w, pool_f, ws, st)
    # split
    staged = torch.empty(dl.dflash_ctx_staged_bytes(geom, B), dtype=torch.uint8, device="cuda")
    staged.fill_(0xFF)  # NaN-poisoned: every row the commit reads must have been written
    pool_s = to_dev(prob["pool"])
    ctx_s = to_dev(prob["ctx_len"])
    dl.dflash_ctx_kv_project(geom, hid_d, ctx_s, w, staged, ws, st)
    dl.dflash_ctx_kv_commit(geom, staged, to_dev(prob["n_acc"]), ctx_s, to_dev(alloc), to_dev(tbl),
                            valid_d, pool_s, st)
    torch.cuda.synchronize()
    return (bits(pool_f), ctx_f.cpu().numpy(), bits(pool_s), ctx_s.cpu().numpy(), staged,
            int(st.item()))


def _cases():
    return [
        ("tiny", {}),                                   # fp32 hidden, 2 KV heads of 64
        ("qwen3_8b", dict(ctx=[2048])),
        ("batch_sweep_8", {}),
        ("mla", dict(ctx=[2048])),
    ]


@pytest.mark.parametrize("name,over", _cases())
def test_split_update(dl, name, over):
    prob = inputs.make_problem(inputs.workload(name, **over), seed=12)
    g = prob["g"]
    B, T = prob["B"], g["T"]
    tbl = prob["pages"].copy()
    alloc = prob["alloc_limit"].copy()
    valid = None
    if B >= 4:
        valid = np.ones(B, np.uint8)
        valid[1] = 0
        alloc[2] = int(prob["ctx_len"][2]) + 1
        c3 = int(prob["ctx_len"][3])
        tbl[3, c3 // g["P"]] = g["num_pool_pages"] + 3    # out of the pool: masked + flagged
    pool_f, ctx_f, pool_s, ctx_s, staged, st = _run(dl, prob, valid, tbl, alloc)
    # bit-identical to the fused call
    np.testing.assert_array_equal(ctx_s, ctx_f)
    np.testing.assert_array_equal(pool_s, pool_f)
    assert (pool_s != prob["pool"]).any()
    # the staged rows against the oracle's projection
    gqa = g["kind"] == "gqa"
    W = g["L"] * (2 * g["nkv"] * g["hd"] if gqa else g["latent"] + g["rope_dim"])
    c_gpu, rows_gpu = _staged_views(staged, B, B * T, W)
    c_ref, rows_ref = oracle.ctx_kv_project(g, prob["hidden"], prob["ctx_len"], prob["w_fc"],
                                            prob["g_h"], prob["w_kv"], prob["g_k"])
    np.testing.assert_array_equal(c_gpu, c_ref)
    assert_close(bf16_f64(rows_gpu), bf16_f64(rows_ref), "staged rows")
    # commit = the oracle's masked copy of the GPU's staged rows
    pool_ref = prob["pool"].copy()
    ctx_ref = oracle.ctx_kv_commit(g, c_gpu, rows_gpu, prob["n_acc"], alloc, tbl, valid, pool_ref)
    np.testing.assert_array_equal(pool_s, pool_ref)
    np.testing.assert_array_equal(ctx_s, ctx_ref)
    if B >= 4:
        assert st & 8  # DFLASH_DEV_BAD_PAGE
