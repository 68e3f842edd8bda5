"""GPU parity of the calls around the path, all bit-exact:

- dflash_pack_weights: per-layer k/v (or latent) projections and norm gains ->
  the stacked layout the context update reads, equal to the stacking the
  seeded inputs use, and an update run on the packed weights equals one run
  on the reference stacking bit for bit;
- dflash_strict_accept against the oracle's strict acceptance (hand cases,
  random drafts, K = 0, K past one warp), feeding dflash_step_bookkeeping
  directly (bonus = the target's token at n - 1);
- dflash_embedding_gather against the oracle's lookup, fed by the GPU
  bookkeeping's emb_ids, with out-of-range ids flagged and zeroed."""
import numpy as np
import pytest

import oracle
from context_kv_update_gb300 import inputs
from tests.gpu_helpers import bits, to_dev

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


def _per_layer(prob):
    """The per-layer tensors a model would hold, as separate device buffers."""
    g = prob["g"]
    layers = []
    for l in range(g["L"]):
        if g["kind"] == "gqa":
            nkv, hd, D = g["nkv"], g["hd"], g["D"]
            wk = to_dev(np.ascontiguousarray(prob["w_kv"][l, 0].reshape(nkv * hd, D)))
            wv = to_dev(np.ascontiguousarray(prob["w_kv"][l, 1].reshape(nkv * hd, D)))
        else:
            wk = to_dev(np.ascontiguousarray(prob["w_kv"][l]))
            wv = None
        layers.append((wk, wv, to_dev(np.ascontiguousarray(prob["g_k"][l]))))
    return layers


@pytest.mark.parametrize("name,over", [("tiny", {}), ("qwen3_8b", {"ctx": [2048]}),
                                       ("mla", {"ctx": [2048]})])
def test_pack_weights_is_the_reference_stacking(dl, name, over):
    import torch
    prob = inputs.make_problem(inputs.workload(name, **over), seed=3, with_pool=False)
    g = prob["g"]
    geom = dl.make_geom(g)
    w_kv = torch.full((dl.dflash_packed_kv_bytes(geom),), 0xAB, dtype=torch.uint8, device="cuda")
    gam = torch.full((dl.dflash_packed_gamma_bytes(geom),), 0xAB, dtype=torch.uint8,
                     device="cuda")
    dl.dflash_pack_weights(geom, _per_layer(prob), w_kv, gam)
    torch.cuda.synchronize()
    got = w_kv.cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(got, prob["w_kv"].reshape(-1))
    np.testing.assert_array_equal(gam.cpu().numpy().view(np.uint16), prob["g_k"].reshape(-1))


def test_update_on_packed_weights_equals_reference_stacking(dl):
    import torch
    prob = inputs.make_problem(inputs.workload("qwen3_8b", ctx=[2048]), seed=4)
    g = prob["g"]
    geom = dl.make_geom(g)
    B = prob["B"]
    w_kv = torch.empty(dl.dflash_packed_kv_bytes(geom), dtype=torch.uint8, device="cuda")
    gam = torch.empty(dl.dflash_packed_gamma_bytes(geom), dtype=torch.uint8, device="cuda")
    dl.dflash_pack_weights(geom, _per_layer(prob), w_kv, gam)
    pools = []
    for wk, gk in ((to_dev(prob["w_kv"]), to_dev(prob["g_k"])),
                   (w_kv.view(torch.bfloat16), gam.view(torch.bfloat16))):
        pool = to_dev(prob["pool"])
        ctx = to_dev(prob["ctx_len"])
        ws = torch.empty(dl.dflash_ctx_workspace_bytes(geom, B), dtype=torch.uint8, device="cuda")
        w = {"w_fc": to_dev(prob["w_fc"]), "g_h": to_dev(prob["g_h"]), "w_kv": wk, "g_k": gk}
        dl.dflash_ctx_kv_update(geom, to_dev(prob["hidden"]), to_dev(prob["n_acc"]), ctx,
                                to_dev(prob["alloc_limit"]), to_dev(prob["pages"]),
                                None, w, pool, ws)
        torch.cuda.synchronize()
        pools.append(bits(pool))
    np.testing.assert_array_equal(pools[0], pools[1])


def _accept_case(rng, B, K, p_match=0.8, vocab=6):
    target = rng.integers(0, vocab, size=(B, K + 1)).astype(np.int32)
    draft = np.where(rng.random((B, K)) < p_match, target[:, :K],
                     rng.integers(0, vocab, size=(B, K))).astype(np.int32)
    return draft, target


@pytest.mark.parametrize("B,K", [(4, 3), (64, 15), (7, 0), (33, 40), (1, 31), (3, 32)])
def test_strict_accept_matches_oracle(dl, B, K):
    import torch
    rng = np.random.default_rng(B * 100 + K)
    draft, target = _accept_case(rng, B, K)
    if B >= 4:  # every draft accepted in row 0, none in row 1
        draft[0] = target[0, :K]
        if K > 0:
            draft[1, 0] = target[1, 0] + 1
    n_ref, acc_ref = oracle.strict_accept(draft, target)
    n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
    dl.dflash_strict_accept(to_dev(draft) if K > 0 else torch.empty((B, 0), dtype=torch.int32,
                                                                    device="cuda"),
                            to_dev(target), n, acc)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(n.cpu().numpy(), n_ref)
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)


def test_strict_accept_strided_views(dl):
    import torch
    rng = np.random.default_rng(9)
    B, K = 10, 7
    draft, target = _accept_case(rng, B, K)
    # rows embedded in wider buffers (row strides 12 and 11)
    dbig = torch.zeros((B, 12), dtype=torch.int32, device="cuda")
    tbig = torch.zeros((B, 11), dtype=torch.int32, device="cuda")
    dbig[:, :K] = to_dev(draft)
    tbig[:, :K + 1] = to_dev(target)
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    acc = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    dl.dflash_strict_accept(dbig[:, :K], tbig[:, :K + 1], n, acc)
    torch.cuda.synchronize()
    n_ref, acc_ref = oracle.strict_accept(draft, target)
    np.testing.assert_array_equal(n.cpu().numpy(), n_ref)
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)


def test_accept_feeds_bookkeeping_and_lookup(dl):
    """strict acceptance -> bookkeeping -> embedding lookup, all on the GPU:
    the bonus is the target's token at n - 1 and the lookup's rows are the
    table rows of [bonus, mask_id, ...]."""
    import torch
    cfg = inputs.workload("batch_sweep_8")
    prob = inputs.make_problem(cfg, seed=5, with_weights=False, with_pool=False)
    g = prob["g"]
    geom = dl.make_geom(g)
    B, T, M = prob["B"], g["T"], g["max_pages"]
    rng = np.random.default_rng(6)
    vocab = 151936
    draft, target = _accept_case(rng, B, T - 1, p_match=0.7, vocab=vocab)
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    acc = torch.empty((B, T), dtype=torch.int32, device="cuda")
    dl.dflash_strict_accept(to_dev(draft), to_dev(target), n, acc)
    outs = {}
    for k in dl.STEP_OUTPUT_FIELDS:
        shape = (B, M) if k == "block_table" else (B, T) if k in (
            "emb_ids", "ctx_pos", "q_pos", "ctx_dst_page", "ctx_dst_slot", "ctx_wmask", "blk_page",
            "blk_slot", "blk_mask") else (B,)
        outs[k] = torch.zeros(shape, dtype=torch.uint8 if k in ("ctx_wmask", "blk_mask")
                              else torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dflash_step_bookkeeping(geom, to_dev(prob["raw_offsets"]), 1, acc, n,
                               to_dev(prob["ctx_len"]), None, prob["max_ctx"], prob["mask_id"],
                               outs, st)
    D = 256
    table_np = inputs.f32_to_bf16_bits(rng.standard_normal((vocab, D), dtype=np.float32))
    table = to_dev(table_np)
    rows = torch.empty((B * T, D), dtype=torch.bfloat16, device="cuda")
    dl.dflash_embedding_gather(outs["emb_ids"], table, rows, dev_status=st)
    torch.cuda.synchronize()
    n_ref, acc_ref = oracle.strict_accept(draft, target)
    np.testing.assert_array_equal(n.cpu().numpy(), n_ref)
    bk, _ = oracle.bookkeeping(prob["raw_offsets"], acc_ref, n_ref, prob["ctx_len"], None, M=M,
                               T=T, P=g["P"], off_div=1, max_ctx=prob["max_ctx"],
                               mask_id=prob["mask_id"])
    for k in bk:
        np.testing.assert_array_equal(outs[k].cpu().numpy(), bk[k], err_msg=k)
    np.testing.assert_array_equal(bk["bonus"], target[np.arange(B), n_ref - 1])
    want, bad = oracle.embedding_gather(bk["emb_ids"], table_np)
    assert not bad
    np.testing.assert_array_equal(bits(rows), want.reshape(B * T, D))
    assert int(st.item()) == 0


def test_embedding_gather_out_of_range_ids(dl):
    import torch
    rng = np.random.default_rng(7)
    V, D = 300, 24 * 8
    table_np = inputs.f32_to_bf16_bits(rng.standard_normal((V, D), dtype=np.float32))
    ids = rng.integers(0, V, size=37).astype(np.int32)
    ids[[3, 10, 36]] = [-1, V, 1 << 30]
    out = torch.full((37, D), 1.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dflash_embedding_gather(to_dev(ids), to_dev(table_np), out, dev_status=st)
    torch.cuda.synchronize()
    want, bad = oracle.embedding_gather(ids, table_np)
    assert bad
    np.testing.assert_array_equal(bits(out), want)
    assert int(st.item()) & 64
