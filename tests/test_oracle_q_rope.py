"""Pins of the oracle's query-side RMSNorm + RoPE (TensorRT-LLM PR #13995,
commits "use fused qk-norm+rope on non-YaRN draft" and "match RoPE between
context and query") against facts that do not come from the oracle:

- at position 0 the rotation is the identity, so the output is the textbook
  RMSNorm, computed here in numpy float64;
- rotate-half RoPE makes q . k depend only on the position difference;
- the rotation keeps the length of every (j, j + dim/2) pair.
"""
import numpy as np

import oracle


def _bf16(rng, shape, scale=1.0):
    return oracle.f64_to_bf16(rng.standard_normal(shape) * scale)


def test_position_zero_is_plain_rmsnorm():
    rng = np.random.default_rng(0)
    q = _bf16(rng, (3, 4, 128))
    gamma = oracle.f64_to_bf16(1 + 0.1 * rng.standard_normal(128))
    out = oracle.q_norm_rope(q, gamma, np.zeros(3, np.int32), 1e6, 1e-6)
    x = oracle.bf16_to_f64(q)
    g = oracle.bf16_to_f64(gamma)
    ref = x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + 1e-6) * g
    got = oracle.bf16_to_f64(out)
    # one bf16 rounding of the same real number: within half an ulp of it
    np.testing.assert_allclose(got, ref, rtol=2 ** -8, atol=1e-30)


def test_scores_depend_only_on_the_position_difference():
    rng = np.random.default_rng(1)
    dim, theta = 64, 1e4
    q = _bf16(rng, (1, 1, dim))
    k = _bf16(rng, (1, 1, dim))
    def score(pq, pk):
        a = oracle.bf16_to_f64(oracle.q_norm_rope(q, None, [pq], theta, 0.0))
        b = oracle.bf16_to_f64(oracle.q_norm_rope(k, None, [pk], theta, 0.0))
        return float((a * b).sum())
    base = score(37, 5)
    for shift in (1, 100, 4096, 300000):
        assert abs(score(37 + shift, 5 + shift) - base) < 0.05 * (1 + abs(base))
    assert abs(score(37, 5) - score(5, 37)) > 1e-3  # the sign of the difference matters


def test_rotation_keeps_pair_lengths():
    rng = np.random.default_rng(2)
    dim = 128
    q = _bf16(rng, (5, 2, dim))
    pos = np.array([0, 1, 777, 32768, 393215], np.int32)
    out = oracle.bf16_to_f64(oracle.q_norm_rope(q, None, pos, 1e6, 0.0))
    x = oracle.bf16_to_f64(q)
    h = dim // 2
    np.testing.assert_allclose(np.hypot(out[..., :h], out[..., h:]),
                               np.hypot(x[..., :h], x[..., h:]), rtol=2 ** -7)
