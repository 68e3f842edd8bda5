"""GPU parity of the prefill context store (row f3) against the oracle:
written rows within the update tolerance, every other pool entry
bit-identical, ctx_len bit-exact -- with variable rows per request, chunk
starts, an allocation ceiling inside the chunk, an unmapped page, an empty and
an invalid request, fp32 and bf16 hidden rows, GQA and the single-latent MLA
pool, and row counts that span several GEMM row tiles."""
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


def _case(name, n_r, c_r, seed, *, f32=False, ceiling=None, hole=None, valid=None, over=None):
    """Weights of workload `name`; a pool holding every request's pages (a
    random permutation), seeded hidden rows, allocation ceilings."""
    cfg = inputs.workload(name, **(over or {}))
    prob = inputs.make_problem(cfg, seed=seed, with_pool=False)
    g = dict(prob["g"])
    rng = np.random.default_rng(seed + 100)
    P = g["P"]
    B = len(n_r)
    pages = [-(-(c + n + 1) // P) for c, n in zip(c_r, n_r)]
    M = max(pages) + 1
    NP = sum(pages) + 3
    g.update(max_pages=M, num_pool_pages=NP)
    perm = rng.permutation(NP).astype(np.int32)
    tbl = np.full((B, M), -1, np.int32)
    pos = 0
    for r, k in enumerate(pages):
        tbl[r, :k] = perm[pos:pos + k]
        pos += k
    if hole is not None:
        tbl[hole[0], hole[1]] = -1
    alloc = np.array([k * P for k in pages], np.int32)
    if ceiling is not None:
        alloc[ceiling[0]] = ceiling[1]
    cu = np.concatenate([[0], np.cumsum(n_r)]).astype(np.int32)
    N = int(cu[-1])
    if f32:
        hidden = rng.standard_normal((N, g["D_in"]), dtype=np.float32)
    else:
        hidden = inputs.f32_to_bf16_bits(rng.standard_normal((N, g["D_in"]), dtype=np.float32))
    if g["kind"] == "gqa":
        shape = (g["L"], NP, 2, g["nkv"], P, g["hd"])
    else:
        shape = (g["L"], NP, P, g["latent"] + g["rope_dim"])
    pool = inputs.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
    w = {k: prob[k] for k in ("w_fc", "g_h", "w_kv", "g_k")}
    return g, hidden, cu, np.array(c_r, np.int32), alloc, tbl, pool, w, valid


def _run(dl, g, hidden, cu, ctx, alloc, tbl, pool, w, valid):
    import torch
    geom = dl.make_geom(g)
    B = len(ctx)
    pool_ref = pool.copy()
    ctx_ref = oracle.ctx_kv_prefill(g, hidden, cu, ctx, alloc, tbl, valid, w["w_fc"], w["g_h"],
                                    w["w_kv"], w["g_k"], pool_ref)
    pool_d = to_dev(pool)
    hid_d = to_dev(hidden) if hidden.dtype == np.uint16 else torch.from_numpy(hidden).cuda()
    ctx_d = to_dev(ctx)
    ws = torch.empty(dl.dflash_ctx_prefill_workspace_bytes(geom, B, hidden.shape[0]),
                     dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dflash_ctx_kv_prefill(geom, hid_d, to_dev(cu), ctx_d, to_dev(alloc), to_dev(tbl),
                             None if valid is None else to_dev(valid),
                             {k: to_dev(v) for k, v in w.items()}, pool_d, ws, st)
    torch.cuda.synchronize()
    got = bits(pool_d)
    changed = (pool_ref != pool).any(axis=-1)
    untouched = ~np.broadcast_to(changed[..., None], pool.shape)
    np.testing.assert_array_equal(got[untouched], pool[untouched])
    assert_close(bf16_f64(got[~untouched]), bf16_f64(pool_ref[~untouched]), "written rows")
    np.testing.assert_array_equal(ctx_d.cpu().numpy(), ctx_ref)
    return int(changed.sum()), ctx_ref, int(st.item())


def test_prefill_tiny_varlen_fp32(dl):
    # three requests: a fresh prompt, an empty one, a chunk starting at 20 whose
    # allocation ends inside the chunk; one page of request 0 unmapped
    g, *rest = _case("tiny", [37, 0, 150], [0, 5, 20], 1, f32=True, ceiling=(2, 100), hole=(0, 1))
    n, ctx, st = _run(dl, g, *rest)
    assert ctx.tolist() == [37, 5, 100]
    assert n == (37 - 16 + 80) * 2 * g["nkv"] * g["L"]  # page 1 of request 0 (16 rows) unmapped
    assert st == 0


def test_prefill_qwen_shape_multi_row_tiles(dl):
    # 701 rows: the projection GEMMs run three 256-row tiles, the last ragged;
    # the many-row epilogue pairs rows, and the odd last row has no partner
    g, *rest = _case("qwen3_8b", [301, 400], [0, 4096], 2, over={"ctx": [2048]})
    n, ctx, _ = _run(dl, g, *rest)
    assert ctx.tolist() == [301, 4496]
    assert n == 701 * 2 * g["nkv"] * g["L"]


def test_prefill_mla_single_latent_pool(dl):
    valid = np.array([1, 0, 1], np.uint8)
    g, *rest = _case("mla", [512, 64, 425], [0, 0, 128], 3, over={"ctx": [2048]},
                     ceiling=(2, 500), valid=valid)
    rest[-1] = valid
    n, ctx, _ = _run(dl, g, *rest)
    assert ctx.tolist() == [512, 0, 500]
    assert n == (512 + (500 - 128)) * g["L"]
