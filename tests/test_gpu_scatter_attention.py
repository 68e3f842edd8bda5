"""GPU parity of the fused block scatter + attention call
(dflash_block_scatter_attention) through the C ABI: the pool bit-identical to
the oracle's scatter, the output within the attention tolerance of the oracle's
attention over that pool, and both bit-identical to the two separate GPU calls
(dflash_block_kv_scatter, then dflash_block_attention).  The pool slots the
block is placed at start as NaN, so a copy of those keys issued before the
block's rows were written shows up as a non-finite or mismatching output."""
import numpy as np
import pytest

import oracle
from context_kv_update_gb300 import inputs
from tests.gpu_helpers import assert_close, bf16_f64, bits, to_dev

pytestmark = pytest.mark.gpu

NAN_BF16 = np.uint16(0x7FC0)


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


def _problem(name, seed, **over):
    prob = inputs.make_problem(inputs.workload(name, **over), seed=seed, with_weights=False)
    g = prob["g"]
    bk, _ = oracle.bookkeeping(prob["raw_offsets"], prob["acc"], prob["n_acc"], prob["ctx_len"],
                               None, M=g["max_pages"], T=g["T"], P=g["P"], off_div=1,
                               max_ctx=prob["max_ctx"], mask_id=prob["mask_id"])
    return prob, g, bk


def _poison_block_slots(g, pool, bk):
    """NaN into every slot the block is placed at, in every layer."""
    for k in np.flatnonzero(bk["blk_mask"].reshape(-1)):
        pg, sl = int(bk["blk_page"].reshape(-1)[k]), int(bk["blk_slot"].reshape(-1)[k])
        if g["kind"] == "gqa":
            pool[:, pg, :, :, sl, :] = NAN_BF16
        else:
            pool[:, pg, sl, :] = NAN_BF16


def _layer_inputs(prob, g, layer):
    if g["kind"] == "gqa":
        return dict(blk_k=prob["blk_k"][layer], blk_v=prob["blk_v"][layer], q=prob["q"][layer],
                    q_rope=None)
    return dict(blk_k=prob["blk_lat"][layer], blk_v=None, q=prob["q_lat"][layer],
                q_rope=prob["q_rope"][layer])


def _oracle_layer(g, layer, li, bk, pool_ref, tbl, kv_len, *, window, sinks, mode):
    """Oracle: the scatter into pool_ref (in place), then attention over it."""
    scale = inputs.attention_scale(g)
    if g["kind"] == "gqa":
        oracle.block_kv_scatter_gqa(g, layer, li["blk_k"], li["blk_v"], bk["blk_page"],
                                    bk["blk_slot"], bk["blk_mask"], pool_ref)
        return oracle.attention_gqa(g, layer, li["q"], pool_ref, tbl, kv_len, window=window,
                                    sinks=sinks, scale=scale, mask_mode=mode)
    oracle.block_latent_scatter_mla(g, layer, li["blk_k"], bk["blk_page"], bk["blk_slot"],
                                    bk["blk_mask"], pool_ref)
    return oracle.attention_mla(g, layer, li["q"], li["q_rope"], pool_ref, tbl, kv_len,
                                window=window, sinks=sinks, scale=scale, mask_mode=mode)


def _gpu_layer(dl, g, layer, li, bk, pool_d, tbl_d, kv_len_d, *, fused, window, sinks, mode, S):
    """One layer on the GPU: the fused call, or the two separate calls."""
    import torch
    geom = dl.make_geom(g)
    B, Tq, hq = li["q"].shape[:3]
    dv = g["hd"] if g["kind"] == "gqa" else g["latent"]
    ws = torch.empty(dl.dflash_attention_workspace_bytes(geom, B, Tq, S), dtype=torch.uint8,
                     device="cuda")
    ws.fill_(0xFF)
    out = torch.full((B, Tq, hq, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    blk_k = to_dev(li["blk_k"])
    blk_v = None if li["blk_v"] is None else to_dev(li["blk_v"])
    page, slot, mask = (to_dev(bk["blk_page"]), to_dev(bk["blk_slot"]), to_dev(bk["blk_mask"]))
    q = to_dev(li["q"])
    q_rope = None if li["q_rope"] is None else to_dev(li["q_rope"])
    sk = None if sinks is None else to_dev(sinks)
    scale = inputs.attention_scale(g)
    if fused:
        dl.dflash_block_scatter_attention(geom, layer, blk_k, blk_v, page, slot, mask, q, pool_d,
                                          tbl_d, kv_len_d, out, ws, q_rope=q_rope, window=window,
                                          sinks=sk, scale=scale, mask_mode=mode, num_segments=S,
                                          dev_status=st)
    else:
        dl.dflash_block_kv_scatter(geom, layer, blk_k, blk_v, page, slot, mask, pool_d,
                                   dev_status=st)
        dl.dflash_block_attention(geom, layer, q, pool_d, tbl_d, kv_len_d, out, ws,
                                  q_rope=q_rope, window=window, sinks=sk, scale=scale,
                                  mask_mode=mode, num_segments=S, dev_status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


def _run_case(dl, prob, g, bk, *, window=0, sinks=False, mode=0, S=0, kv_len=None, layers=None):
    import torch
    pool = prob["pool"].copy()
    _poison_block_slots(g, pool, bk)
    pool_ref = pool.copy()
    pool_f = to_dev(pool)
    pool_s = to_dev(pool)
    tbl = bk["block_table"]
    kv = bk["seq_lens"] if kv_len is None else np.asarray(kv_len, np.int32)
    tbl_d, kv_d = to_dev(tbl), to_dev(kv)
    for layer in (range(g["L"]) if layers is None else layers):
        li = _layer_inputs(prob, g, layer)
        sk = prob["sinks"][layer] if sinks else None
        ref = _oracle_layer(g, layer, li, bk, pool_ref, tbl, kv, window=window, sinks=sk,
                            mode=mode)
        out_f, st_f = _gpu_layer(dl, g, layer, li, bk, pool_f, tbl_d, kv_d, fused=True,
                                 window=window, sinks=sk, mode=mode, S=S)
        out_s, st_s = _gpu_layer(dl, g, layer, li, bk, pool_s, tbl_d, kv_d, fused=False,
                                 window=window, sinks=sk, mode=mode, S=S)
        assert st_f == 0 and st_s == 0, (st_f, st_s)
        np.testing.assert_array_equal(bits(out_f), bits(out_s))
        assert_close(bf16_f64(bits(out_f)), ref, f"{g['kind']} layer {layer} S={S}")
        assert torch.equal(pool_f.view(torch.int16), pool_s.view(torch.int16))
    np.testing.assert_array_equal(bits(pool_f), pool_ref)
    assert not np.isnan(bf16_f64(pool_ref)).any()  # every poisoned slot was written


# 16-row blocks (ctx + n .. + 15) starting at 120 mod 128 (the rows straddle two
# key tiles, so with one tile per segment two CTAs write them), on a tile
# boundary, and near the start of the cache; pages for ctx + 2T per request
_CTX = dict(ctx=[115, 1000, 250, 3], n_acc=[5, 16, 6, 1], alloc_pages=None, pool_pages=None,
            max_pages=None)
# 8-row MLA blocks across a half-tile boundary (188..195), a tile boundary
# (1020..1027), at a tile start and near the start of the cache
_CTX_MLA = dict(ctx=[185, 1016, 250, 3], n_acc=[3, 4, 6, 1], alloc_pages=None, pool_pages=None,
                max_pages=None)


@pytest.mark.parametrize("S", [0, 1, 3, 1000])
def test_fused_scatter_attention_gqa_segments(dl, S):
    prob, g, bk = _problem("tiny", 21 + S, B=4, L=2, hq=32, nkv=8, hd=128, T=16, P=64, **_CTX)
    _run_case(dl, prob, g, bk, S=S)


@pytest.mark.parametrize("hq,nkv,hd,P,mode,window,sinks", [
    (32, 2, 128, 64, 0, 0, True),    # 256 query rows per KV head: two row tiles write
    (8, 2, 64, 16, 1, 40, False),    # head_dim 64, 16-key pages, a window
    (12, 1, 128, 32, 0, 5, True),    # one KV head, a window narrower than the block
])
def test_fused_scatter_attention_gqa_geometries(dl, hq, nkv, hd, P, mode, window, sinks):
    prob, g, bk = _problem("tiny", hq + P, B=4, L=2, hq=hq, nkv=nkv, hd=hd, T=16, P=P, **_CTX)
    _run_case(dl, prob, g, bk, mode=mode, window=window, sinks=sinks, S=1000)


@pytest.mark.parametrize("S,mode,window", [(0, 0, 0), (1000, 1, 0), (2, 0, 300)])
def test_fused_scatter_attention_mla(dl, S, mode, window):
    prob, g, bk = _problem("mla", 40 + S, B=4, L=2, **_CTX_MLA)
    _run_case(dl, prob, g, bk, S=S, mode=mode, window=window, sinks=mode == 1)


def test_fused_scatter_rows_no_segment_reads(dl):
    """kv_len below the block (0 and 5 with a 16-row block): the rows at
    negative positions belong to no segment and are still written."""
    prob, g, bk = _problem("tiny", 5, B=4, L=1, hq=8, nkv=2, hd=64, T=16, P=16, **_CTX)
    kv = bk["seq_lens"].copy()
    kv[0], kv[1] = 0, 5
    _run_case(dl, prob, g, bk, kv_len=kv)


def test_fused_scatter_bad_page_flags_like_the_scatter(dl):
    import torch
    prob, g, bk = _problem("tiny", 9, B=2, L=1, hq=8, nkv=2, hd=64, T=4, P=16, ctx=[40, 90],
                           n_acc=[2, 4], alloc_pages=None, pool_pages=None, max_pages=None)
    bk = dict(bk)
    bk["blk_page"] = bk["blk_page"].copy()
    k = int(np.flatnonzero(bk["blk_mask"].reshape(-1))[0])
    bk["blk_page"].reshape(-1)[k] = g["num_pool_pages"] + 3
    li = _layer_inputs(prob, g, 0)
    outs = []
    for fused in (True, False):
        pool_d = to_dev(prob["pool"])
        out, st = _gpu_layer(dl, g, 0, li, bk, pool_d, to_dev(bk["block_table"]),
                             to_dev(bk["seq_lens"]), fused=fused, window=0, sinks=None, mode=0,
                             S=0)
        assert st & dl._lib.DEV_BAD_PAGE
        outs.append((bits(out), bits(pool_d)))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


def test_fused_scatter_attention_qwen_32k_one_layer(dl):
    """The 32K Qwen3-8B-shaped step's layer in the launch configuration the
    benchmark times: fused and separate calls bit-identical (output and pool),
    the block's slots written with its rows."""
    import torch
    prob, g, bk = _problem("qwen3_8b", 32, L=1)
    pool = prob["pool"]
    _poison_block_slots(g, pool, bk)
    li = _layer_inputs(prob, g, 0)
    tbl_d, kv_d = to_dev(bk["block_table"]), to_dev(bk["seq_lens"])
    pool_f = to_dev(pool)
    pool_s = pool_f.clone()
    out_f, st_f = _gpu_layer(dl, g, 0, li, bk, pool_f, tbl_d, kv_d, fused=True, window=0,
                             sinks=None, mode=0, S=0)
    out_s, st_s = _gpu_layer(dl, g, 0, li, bk, pool_s, tbl_d, kv_d, fused=False, window=0,
                             sinks=None, mode=0, S=0)
    assert st_f == 0 and st_s == 0
    assert torch.isfinite(out_f.float()).all()
    assert torch.equal(out_f.view(torch.int16), out_s.view(torch.int16))
    assert torch.equal(pool_f.view(torch.int16), pool_s.view(torch.int16))
    T = g["T"]
    for i in range(T):
        pg, sl = int(bk["blk_page"][0, i]), int(bk["blk_slot"][0, i])
        assert bk["blk_mask"][0, i]
        got_k = bits(pool_f[0, pg, 0, :, sl, :])
        got_v = bits(pool_f[0, pg, 1, :, sl, :])
        np.testing.assert_array_equal(got_k, li["blk_k"][0, i])
        np.testing.assert_array_equal(got_v, li["blk_v"][0, i])
