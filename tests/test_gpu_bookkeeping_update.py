"""GPU parity: bookkeeping (bit-exact), context-KV update (tolerance on written
rows, bit-exact elsewhere, bit-exact ctx_len) and block scatter (bit-exact),
each through the C ABI against the CPU oracle on the same seeded inputs."""
import json
import os

import numpy as np
import pytest

import oracle
from context_kv_update_gb300 import inputs
from tests.gpu_helpers import assert_close, bf16_f64, bits, to_dev

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


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


# ------------------------------------------------------------ bookkeeping


def _run_bk_gpu(dl, geom, off, acc, n_acc, ctx, valid, M, T, off_div, max_ctx, mask_id):
    import torch
    B = len(n_acc)
    out = {}
    for k in dl.STEP_OUTPUT_FIELDS:
        shape = (B, M) if k == "block_table" else (B, T) if k in (
            "emb_ids", "ctx_pos", "q_pos", "ctx_dst_page", "ctx_dst_slot", "ctx_wmask", "blk_page",
            "blk_slot", "blk_mask") else (B,)
        dt = torch.uint8 if k in ("ctx_wmask", "blk_mask") else torch.int32
        out[k] = torch.full(shape, 77, dtype=dt, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    off_d = to_dev(off)
    acc_d = to_dev(acc)
    dl.dflash_step_bookkeeping(geom, off_d[:, :M], off_div, acc_d[:, :T], to_dev(n_acc),
                               to_dev(ctx), None if valid is None else to_dev(valid), max_ctx,
                               mask_id, out, st)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}, int(st.item())


def _geom_for(dl, M, T, P):
    g = inputs.make_problem(inputs.workload("tiny", T=T, P=P), seed=0, with_pool=False,
                            with_weights=False)["g"]
    g = dict(g, max_pages=M, P=P, T=T)
    return dl.make_geom(g)


def test_bookkeeping_golden(dl):
    gold = json.load(open(os.path.join(GOLDEN, "bookkeeping_tiny.json")))
    cm = gold["common"]
    geom = _geom_for(dl, cm["M"], cm["T"], cm["P"])
    for case in gold["cases"]:
        out, st = _run_bk_gpu(dl, geom, np.array([case["off"]], np.int32),
                              np.array([case["acc"]], np.int32),
                              np.array([case["n_acc"]], np.int32), np.array([case["ctx"]], np.int32),
                              np.array([case["valid"]], np.uint8), cm["M"], cm["T"],
                              case["off_div"], cm["max_ctx"], cm["mask_id"])
        for key, val in case["expect"].items():
            if key == "status":
                assert st == val, case["name"]
            else:
                assert out[key].reshape(-1).tolist() == np.asarray(val).reshape(-1).tolist(), \
                    (case["name"], key)


@pytest.mark.parametrize("B,M,T,P,div", [(1, 16, 4, 16, 1), (7, 9, 4, 8, 2), (64, 600, 16, 64, 1),
                                         (33, 129, 8, 64, 3)])
def test_bookkeeping_random_vs_oracle(dl, B, M, T, P, div):
    rng = np.random.default_rng(B * 1000 + M)
    geom = _geom_for(dl, M, T, P)
    for trial in range(4):
        off = np.full((B, M + 5), -1, np.int32)  # wider base: strided rows
        for r in range(B):
            n = int(rng.integers(0, M + 1))
            off[r, :n] = rng.permutation(8 * M)[:n] * div
            holes = rng.random(M) < (0.5 if trial == 3 else 0.05)
            off[r, :M][holes] = rng.choice([-1, 0, -9], size=int(holes.sum()))
        if trial == 1:
            off[0, :M] = -1          # all-negative row
            off[min(1, B - 1), :M] = 0  # all-zero row
        acc = rng.integers(0, 150000, size=(B, T + 3)).astype(np.int32)
        n_acc = rng.integers(0, T + 2, size=B).astype(np.int32)
        ctx = rng.integers(-2, M * P + 2 * P, size=B).astype(np.int32)
        valid = (rng.random(B) < 0.8).astype(np.uint8)
        max_ctx = int(rng.integers(P, M * P + 1))
        ref, st_ref = oracle.bookkeeping(off, acc, n_acc, ctx, valid, M=M, T=T, P=P, off_div=div,
                                         max_ctx=max_ctx, mask_id=151669)
        got, st = _run_bk_gpu(dl, geom, off, acc, n_acc, ctx, valid, M, T, div, max_ctx, 151669)
        for k in ref:
            np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
        assert st == st_ref


def test_bookkeeping_all_live_valid_null(dl):
    prob = inputs.make_problem(inputs.workload("batch_sweep_16"), seed=3, with_pool=False,
                               with_weights=False)
    g = prob["g"]
    geom = dl.make_geom(g)
    ref, st_ref = oracle.bookkeeping(prob["raw_offsets"], prob["acc"], prob["n_acc"],
                                     prob["ctx_len"], None, M=g["max_pages"], T=g["T"], P=g["P"],
                                     off_div=1, max_ctx=prob["max_ctx"], mask_id=prob["mask_id"])
    got, st = _run_bk_gpu(dl, geom, prob["raw_offsets"], prob["acc"], prob["n_acc"],
                          prob["ctx_len"], None, g["max_pages"], g["T"], 1, prob["max_ctx"],
                          prob["mask_id"])
    for k in ref:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    assert st == st_ref


# ------------------------------------------------------------ ctx update


def _weights_dev(prob):
    return {k: to_dev(prob[k]) for k in ("w_fc", "g_h", "w_kv", "g_k")}


def _update_both(dl, prob, valid=None, tbl=None, alloc=None):
    import torch
    g = prob["g"]
    geom = dl.make_geom(g)
    tbl = prob["pages"] if tbl is None else tbl
    alloc = prob["alloc_limit"] if alloc is None else alloc
    pool_ref = prob["pool"].copy()
    upd = oracle.ctx_kv_update_gqa if g["kind"] == "gqa" else oracle.ctx_kv_update_mla
    ctx_ref = upd(g, prob["hidden"], prob["n_acc"], prob["ctx_len"], alloc, tbl, valid,
                  prob["w_fc"], prob["g_h"], prob["w_kv"], prob["g_k"], pool_ref)
    B = prob["B"]
    pool_d = to_dev(prob["pool"])
    hid = prob["hidden"]
    hid_d = to_dev(hid) if hid.dtype == np.uint16 else torch.from_numpy(hid).cuda()
    ctx_d = to_dev(prob["ctx_len"])
    ws = torch.empty(dl.dflash_ctx_workspace_bytes(geom, B), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)  # NaN-poisoned scratch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dflash_ctx_kv_update(geom, hid_d, to_dev(prob["n_acc"]), ctx_d, to_dev(alloc), to_dev(tbl),
                            None if valid is None else to_dev(valid), _weights_dev(prob), pool_d,
                            ws, st)
    torch.cuda.synchronize()
    return pool_ref, ctx_ref, bits(pool_d), ctx_d.cpu().numpy(), int(st.item())


def _check_pool(prob, pool_ref, pool_gpu):
    pool0 = prob["pool"]
    changed = pool_ref != pool0
    # rows the oracle wrote: compare those rows (whole rows) within tolerance
    g = prob["g"]
    if g["kind"] == "gqa":
        row_changed = changed.any(axis=-1)  # [L, NP, 2, nkv, P]
    else:
        row_changed = changed.any(axis=-1)  # [L, NP, P]
    untouched = ~np.broadcast_to(row_changed[..., None], pool0.shape)
    np.testing.assert_array_equal(pool_gpu[untouched], pool0[untouched])
    assert_close(bf16_f64(pool_gpu[~untouched]), bf16_f64(pool_ref[~untouched]), "written rows")
    return int(row_changed.sum())


def test_update_tiny_fp32_hidden(dl):
    prob = inputs.make_problem(inputs.workload("tiny"), seed=0)
    pool_ref, ctx_ref, pool_gpu, ctx_gpu, st = _update_both(dl, prob)
    n = _check_pool(prob, pool_ref, pool_gpu)
    assert n == 3 * 2 * 2  # 3 rows x (K, V) x 2 heads
    np.testing.assert_array_equal(ctx_gpu, ctx_ref)
    assert st == 0


@pytest.mark.parametrize("name,over", [
    ("qwen3_8b", dict(ctx=[2048])),
    ("qwen3_8b", dict(ctx=[32768], n_acc=[16])),
    ("batch_sweep_8", {}),
    ("batch_sweep_32", {}),
])
def test_update_qwen_shapes(dl, name, over):
    prob = inputs.make_problem(inputs.workload(name, **over), seed=1)
    pool_ref, ctx_ref, pool_gpu, ctx_gpu, st = _update_both(dl, prob)
    n = _check_pool(prob, pool_ref, pool_gpu)
    assert n > 0
    np.testing.assert_array_equal(ctx_gpu, ctx_ref)


@pytest.mark.parametrize("D_in,D,nkv,hd,L,B,hidden", [
    (1024, 2560, 4, 64, 2, 2, "bf16"),   # hidden norm: 5-CTA clusters of 512 columns
    (2048, 6144, 2, 128, 1, 1, "f32"),   # 8 CTAs of 768 columns (6 of 8 slots a thread)
    (512, 8192, 1, 128, 1, 3, "bf16"),   # 8 CTAs of 1024 columns; fc has 8 K blocks
    (4096, 576, 2, 64, 1, 2, "f32"),     # 2 CTAs of 288 columns: tiles straddle CTAs
    (64, 64, 1, 64, 1, 1, "bf16"),       # one 64-column CTA, one K block
    (1024, 2560, 4, 64, 2, 20, "bf16"),  # 320 rows: the many-row norm (80 of 96 threads)
    (512, 1536, 2, 32, 1, 17, "f32"),    # 272 rows, head rows of 4 lanes
])
def test_update_odd_widths(dl, D_in, D, nkv, hd, L, B, hidden):
    """d_model / d_in / stacked K/V widths off the benchmark shapes: every
    cluster layout of the hidden RMSNorm and GEMMs whose tiles are shared by
    few or many CTAs, checked against the oracle."""
    n_acc = [16 - (3 * b) % 16 for b in range(B)]
    over = dict(D_in=D_in, D=D, nkv=nkv, hq=2 * nkv, hd=hd, L=L, B=B, T=16, hidden_dtype=hidden,
                ctx=[100 + 7 * (b % 8) for b in range(B)], n_acc=n_acc,
                alloc_pages=[12] * B, pool_pages=16 * B, max_pages=16)
    prob = inputs.make_problem(inputs.workload("tiny", **over), seed=11)
    pool_ref, ctx_ref, pool_gpu, ctx_gpu, st = _update_both(dl, prob)
    n = _check_pool(prob, pool_ref, pool_gpu)
    assert n == sum(n_acc) * 2 * nkv * L
    np.testing.assert_array_equal(ctx_gpu, ctx_ref)
    assert st == 0


@pytest.mark.parametrize("name", ["batch_sweep_8", "batch_sweep_32"])
def test_update_dummies_bad_pages_and_ceiling(dl, name):
    # batch 32 = 512 rows: the many-row norm resolves the destinations
    prob = inputs.make_problem(inputs.workload(name), seed=5)
    valid = np.ones(prob["B"], np.uint8)
    valid[[1, 4]] = 0
    tbl = prob["pages"].copy()
    # request 2: its next page points outside the pool -> rows there masked + flag
    c2 = int(prob["ctx_len"][2])
    tbl[2, c2 // prob["g"]["P"]] = prob["g"]["num_pool_pages"] + 5
    alloc = prob["alloc_limit"].copy()
    alloc[3] = int(prob["ctx_len"][3]) + 1  # ceiling after one row
    # the oracle masks out-of-pool pages without touching them as well
    pool_ref, ctx_ref, pool_gpu, ctx_gpu, st = _update_both(dl, prob, valid=valid, tbl=tbl,
                                                            alloc=alloc)
    _check_pool(prob, pool_ref, pool_gpu)
    np.testing.assert_array_equal(ctx_gpu, ctx_ref)
    assert st & 8  # DFLASH_DEV_BAD_PAGE


@pytest.mark.parametrize("ctx", [2048, 32768, 131072 + 5])
def test_update_mla(dl, ctx):
    """MLA latent update; the long contexts put the rope part's angles at
    positions past 32K and 128K."""
    prob = inputs.make_problem(inputs.workload("mla", ctx=[ctx], n_acc=[8]), seed=2)
    pool_ref, ctx_ref, pool_gpu, ctx_gpu, st = _update_both(dl, prob)
    n = _check_pool(prob, pool_ref, pool_gpu)
    assert n == prob["g"]["L"] * int(prob["n_acc"][0])
    np.testing.assert_array_equal(ctx_gpu, ctx_ref)


def test_update_ctx_len_agrees_with_bookkeeping(dl):
    prob = inputs.make_problem(inputs.workload("batch_sweep_16"), seed=9)
    g = prob["g"]
    ref, _ = oracle.bookkeeping(prob["raw_offsets"], prob["acc"], prob["n_acc"], prob["ctx_len"],
                                None, M=g["max_pages"], T=g["T"], P=g["P"], off_div=1,
                                max_ctx=prob["max_ctx"], mask_id=prob["mask_id"])
    geom = dl.make_geom(g)
    got, _ = _run_bk_gpu(dl, geom, prob["raw_offsets"], prob["acc"], prob["n_acc"],
                         prob["ctx_len"], None, g["max_pages"], g["T"], 1, prob["max_ctx"],
                         prob["mask_id"])
    _, ctx_ref, _, ctx_gpu, _ = _update_both(dl, prob, alloc=got["alloc_limit"],
                                             tbl=got["block_table"])
    np.testing.assert_array_equal(ctx_gpu, got["ctx_len_new"])
    np.testing.assert_array_equal(ctx_gpu, ref["ctx_len_new"])


# ------------------------------------------------------------ scatter


@pytest.mark.parametrize("kind", ["gqa", "mla"])
def test_block_scatter_bit_exact(dl, kind):
    import torch
    name = "batch_sweep_4" if kind == "gqa" else "mla"
    prob = inputs.make_problem(inputs.workload(name, **({} if kind == "gqa" else {"ctx": [300]})),
                               seed=4, with_weights=False)
    g = prob["g"]
    geom = dl.make_geom(g)
    bk, _ = oracle.bookkeeping(prob["raw_offsets"], prob["acc"], prob["n_acc"], prob["ctx_len"],
                               None, M=g["max_pages"], T=g["T"], P=g["P"], off_div=1,
                               max_ctx=prob["max_ctx"], mask_id=prob["mask_id"])
    pool_ref = prob["pool"].copy()
    pool_d = to_dev(prob["pool"])
    for layer in range(g["L"]):
        if kind == "gqa":
            oracle.block_kv_scatter_gqa(g, layer, prob["blk_k"][layer], prob["blk_v"][layer],
                                        bk["blk_page"], bk["blk_slot"], bk["blk_mask"], pool_ref)
            dl.dflash_block_kv_scatter(geom, layer, to_dev(prob["blk_k"][layer]),
                                       to_dev(prob["blk_v"][layer]), to_dev(bk["blk_page"]),
                                       to_dev(bk["blk_slot"]), to_dev(bk["blk_mask"]), pool_d)
        else:
            oracle.block_latent_scatter_mla(g, layer, prob["blk_lat"][layer], bk["blk_page"],
                                            bk["blk_slot"], bk["blk_mask"], pool_ref)
            dl.dflash_block_kv_scatter(geom, layer, to_dev(prob["blk_lat"][layer]), None,
                                       to_dev(bk["blk_page"]), to_dev(bk["blk_slot"]),
                                       to_dev(bk["blk_mask"]), pool_d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(pool_d), pool_ref)
    assert (pool_ref != prob["pool"]).any()


def test_block_scatter_wide_rows(dl):
    """64 KV heads x 128 dims: 2048 16-byte vectors a block row, more than the
    scatter keeps in registers (the rest go through its tail loop)."""
    import torch
    over = dict(nkv=64, hq=64, hd=128, L=2, B=2, T=8, ctx=[40, 90], n_acc=[5, 8],
                alloc_pages=[12, 12], pool_pages=32, max_pages=16)
    prob = inputs.make_problem(inputs.workload("tiny", **over), seed=6, with_weights=False)
    g = prob["g"]
    geom = dl.make_geom(g)
    bk, _ = oracle.bookkeeping(prob["raw_offsets"], prob["acc"], prob["n_acc"], prob["ctx_len"],
                               None, M=g["max_pages"], T=g["T"], P=g["P"], off_div=1,
                               max_ctx=prob["max_ctx"], mask_id=prob["mask_id"])
    pool_ref = prob["pool"].copy()
    pool_d = to_dev(prob["pool"])
    for layer in range(g["L"]):
        oracle.block_kv_scatter_gqa(g, layer, prob["blk_k"][layer], prob["blk_v"][layer],
                                    bk["blk_page"], bk["blk_slot"], bk["blk_mask"], pool_ref)
        dl.dflash_block_kv_scatter(geom, layer, to_dev(prob["blk_k"][layer]),
                                   to_dev(prob["blk_v"][layer]), to_dev(bk["blk_page"]),
                                   to_dev(bk["blk_slot"]), to_dev(bk["blk_mask"]), pool_d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(pool_d), pool_ref)
    assert (pool_ref != prob["pool"]).sum() > 0
