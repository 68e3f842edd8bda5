"""GPU parity of the query-side RMSNorm + RoPE (dflash_q_norm_rope; TensorRT-LLM
PR #13995, commits "use fused qk-norm+rope on non-YaRN draft" and "match RoPE
between context and query") against the oracle on the same seeded inputs,
with positions up to the 393K context; in place equals out of place."""
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


@pytest.mark.parametrize("kind,hq,dim", [("gqa", 32, 128), ("gqa", 8, 64), ("mla", 16, 64)])
def test_q_norm_rope(dl, kind, hq, dim):
    import torch
    rng = np.random.default_rng(21)
    B, Tq = 3, 5
    if kind == "gqa":
        g = inputs.workload("tiny", hq=hq, nkv=hq // 4, hd=dim, rope_theta=1e6)
    else:
        g = inputs.workload("mla", hq=hq, rope_dim=dim, ctx=[300])
    prob = inputs.make_problem(g, seed=1, with_weights=False)
    geom = dl.make_geom(prob["g"])
    q = oracle.f64_to_bf16(rng.standard_normal((B, Tq, hq, dim)))
    gamma = oracle.f64_to_bf16(1 + 0.1 * rng.standard_normal(dim)) if kind == "gqa" else None
    pos = np.array([[0, 1, 2, 3, 4], [32768, 32769, 32770, 32771, 32772],
                    [393211, 393212, 393213, 393214, 393215]], np.int32)
    ref = oracle.q_norm_rope(q, gamma, pos, prob["g"]["rope_theta"], prob["g"]["eps_k"])
    q_d = to_dev(q)
    out_d = torch.empty_like(q_d)
    gamma_d = None if gamma is None else to_dev(gamma)
    pos_d = to_dev(pos)
    dl.dflash_q_norm_rope(geom, q_d, gamma_d, pos_d, out_d)
    torch.cuda.synchronize()
    out = bits(out_d)
    assert_close(bf16_f64(out), bf16_f64(ref), "rotated queries")
    # in place gives the same bits
    dl.dflash_q_norm_rope(geom, q_d, gamma_d, pos_d, q_d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(q_d), out)
