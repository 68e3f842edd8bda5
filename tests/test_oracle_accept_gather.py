"""Pins of the oracle's strict acceptance (TensorRT-LLM PR #20550, follow-up
commit "spec_tail_kernels.py") and the noise-block embedding lookup
(TensorRT-LLM PR #13995, "fuse query-input build ... + fused embedding
lookup"): hand-worked cases, a brute-force restatement over random drafts,
the link to the bookkeeping's bonus token, and the lookup as a one-hot
matrix product."""
import numpy as np

import oracle


def test_strict_accept_hand_cases():
    draft = np.array([[5, 6, 7], [5, 6, 7], [9, 6, 7], [5, 0, 7]], np.int32)
    target = np.array([[5, 6, 7, 8],     # every draft matches: 3 + the bonus 8
                       [5, 6, 1, 8],     # third draft rejected: the target's 1 is the bonus
                       [4, 6, 7, 8],     # first draft rejected: only the bonus 4
                       [5, 6, 7, 8]], np.int32)
    n, acc = oracle.strict_accept(draft, target)
    assert n.tolist() == [4, 3, 1, 2]
    assert acc.tolist() == [[5, 6, 7, 8], [5, 6, 1, -1], [4, -1, -1, -1], [5, 6, -1, -1]]


def test_strict_accept_matches_its_definition_on_random_drafts():
    rng = np.random.default_rng(0)
    B, K = 64, 15
    target = rng.integers(0, 4, size=(B, K + 1)).astype(np.int32)
    draft = np.where(rng.random((B, K)) < 0.8, target[:, :K],
                     rng.integers(0, 4, size=(B, K))).astype(np.int32)
    n, acc = oracle.strict_accept(draft, target)
    for r in range(B):
        m = 0
        for j in range(K):
            if draft[r, j] != target[r, j]:
                break
            m += 1
        assert n[r] == m + 1
        assert (acc[r, :m + 1] == target[r, :m + 1]).all() and (acc[r, m + 1:] == -1).all()
        # the accepted drafts are the draft's own prefix; the last accepted
        # token (the bookkeeping's bonus, accepted[n - 1]) is the target's
        assert (acc[r, :m] == draft[r, :m]).all()
        assert acc[r, n[r] - 1] == target[r, n[r] - 1]


def test_embedding_gather_is_a_one_hot_product():
    rng = np.random.default_rng(1)
    V, D = 50, 24
    table = oracle.f64_to_bf16(rng.standard_normal((V, D)))
    bonus = np.array([3, 17, 49], np.int32)
    mask_id = 7
    ids = np.full((3, 4), mask_id, np.int32)
    ids[:, 0] = bonus                      # [bonus, mask_id, mask_id, mask_id]
    out, bad = oracle.embedding_gather(ids, table)
    assert not bad
    onehot = np.eye(V)[ids]                # [3, 4, V]
    np.testing.assert_array_equal(oracle.bf16_to_f64(out), onehot @ oracle.bf16_to_f64(table))
    _, bad = oracle.embedding_gather(np.array([V], np.int32), table)
    assert bad
