"""Pins of the CPU oracle against facts fixed outside it (CPU only).

Each test ties an oracle function to something other than its own formula:
hand-worked bookkeeping values, closed forms of RMSNorm and RoPE, numpy's
float64 matmul, a brute-force dense attention with an explicit mask matrix,
invariants (split-count independence, masked entries untouched) and special
cases that reduce to known answers.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from context_kv_update_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ bf16


def test_bf16_rounding_known_values():
    # 1.0 -> 0x3F80; 1 + 2^-8 is a tie between 0x3F80 and 0x3F81 -> even 0x3F80;
    # 1 + 3*2^-8 ties between 0x3F81 and 0x3F82 -> even 0x3F82; -2.5 -> 0xC020.
    vals = [1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 0.0, 65280.0]
    want = [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000, 0x477F]
    assert list(oracle.f64_to_bf16(vals)) == want
    assert list(oracle.bf16_to_f64(np.array(want, np.uint16))) == [1.0, 1.0, 1.0 + 2 ** -6, -2.5,
                                                                   0.0, 65280.0]


# -------------------------------------------------------------- RMSNorm


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(128)
    y = oracle.rmsnorm(x, None, eps=0.0)
    assert abs(np.sqrt(np.mean(y * y)) - 1.0) < 1e-14
    for alpha in (1e-3, 0.5, 7.0, 1e4):
        np.testing.assert_allclose(oracle.rmsnorm(alpha * x, None, eps=0.0), y, rtol=1e-13)
    # the gain multiplies elementwise
    g = rng.standard_normal(128)
    np.testing.assert_allclose(oracle.rmsnorm(x, g, eps=0.0), y * g, rtol=1e-13)


def test_rmsnorm_constant_vector_with_eps():
    # x = c * ones -> c / sqrt(c^2 + eps) in every entry
    for c, eps in ((0.3, 1e-6), (-2.0, 1e-6), (1e-3, 1e-6), (5.0, 0.25)):
        y = oracle.rmsnorm(np.full(64, c), None, eps=eps)
        np.testing.assert_allclose(y, c / math.sqrt(c * c + eps), rtol=1e-14)


# ----------------------------------------------------------------- RoPE


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(2).standard_normal(128)
    np.testing.assert_array_equal(oracle.rope_neox(x, 0, 1e6), x)


def test_rope_two_dims_is_plain_rotation():
    # n = 2: one pair (x0, x1), frequency theta^0 = 1, angle = pos
    for pos in (1, 2, 100, 393216):
        y = oracle.rope_neox(np.array([1.0, 0.0]), pos, 1e4)
        np.testing.assert_allclose(y, [math.cos(pos), math.sin(pos)], atol=1e-12)
        y = oracle.rope_neox(np.array([0.0, 1.0]), pos, 1e4)
        np.testing.assert_allclose(y, [-math.sin(pos), math.cos(pos)], atol=1e-12)


def test_rope_known_frequency_quarter_turn():
    # n = 4, theta = 1e4: pair j = 1 couples dims 1 and 3 with f = 1e4^(-1/2) = 0.01.
    # At pos = 50*pi the angle is pi/2: (x1, x3) = (1, 0) -> (0, 1).
    x = np.array([0.0, 1.0, 0.0, 0.0])
    y = oracle.rope_neox(x, 50 * math.pi, 1e4)
    np.testing.assert_allclose(y[[1, 3]], [0.0, 1.0], atol=1e-12)
    # pair j = 0 (dims 0 and 2) turns by the position itself
    y0 = oracle.rope_neox(np.array([1.0, 0.0, 0.0, 0.0]), 0.5, 1e4)
    np.testing.assert_allclose(y0, [math.cos(0.5), 0.0, math.sin(0.5), 0.0], atol=1e-15)


def test_rope_preserves_pair_norms_and_composes():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(64)
    h = 32
    for p1, p2 in ((3, 5), (1000, 24000), (131071, 262145)):
        y1 = oracle.rope_neox(x, p1, 1e6)
        np.testing.assert_allclose(y1[:h] ** 2 + y1[h:] ** 2, x[:h] ** 2 + x[h:] ** 2, rtol=1e-12)
        y12 = oracle.rope_neox(y1, p2, 1e6)
        np.testing.assert_allclose(y12, oracle.rope_neox(x, p1 + p2, 1e6), atol=1e-9)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    base = np.dot(oracle.rope_neox(q, 40, 1e6), oracle.rope_neox(k, 7, 1e6))
    for shift in (1, 1000, 300000):
        s = np.dot(oracle.rope_neox(q, 40 + shift, 1e6), oracle.rope_neox(k, 7 + shift, 1e6))
        assert abs(s - base) < 1e-8


# ------------------------------------------------------------ projection


def test_matvec_matches_numpy_float64():
    rng = np.random.default_rng(5)
    W = inputs.f32_to_bf16_bits(rng.standard_normal((96, 256), dtype=np.float32) * 0.02)
    x = rng.standard_normal(256)
    ref = inputs.bf16_bits_to_f32(W).astype(np.float64) @ x
    np.testing.assert_allclose(oracle.matvec_bf16(W, x), ref, rtol=1e-12, atol=1e-14)


def test_fc_hidden_norm_properties():
    prob = inputs.make_problem(inputs.workload("tiny"), seed=0, with_pool=False)
    hid = prob["hidden"].reshape(-1, 256)
    one = np.full(256, 0x3F80, np.uint16)  # gain 1.0
    hn = oracle.bf16_to_f64(oracle.fc_hidden_norm(hid, prob["w_fc"], one, 1e-6))
    # unit RMS per row, up to bf16 rounding
    np.testing.assert_allclose(np.sqrt(np.mean(hn * hn, axis=1)), 1.0, atol=4e-3)
    # doubling W_fc (exact in bf16) leaves the normalised rows unchanged but for
    # bf16 ties of h, which move an entry by at most one ulp
    w2 = inputs.f32_to_bf16_bits(inputs.bf16_bits_to_f32(prob["w_fc"]) * 2)
    hn2 = oracle.bf16_to_f64(oracle.fc_hidden_norm(hid, w2, one, 1e-6))
    assert np.max(np.abs(hn2 - hn)) <= 2 ** -7 * np.max(np.abs(hn))
    # h itself: the sign pattern of hn equals that of the fc product
    x = inputs.bf16_bits_to_f32(inputs.f32_to_bf16_bits(hid)).astype(np.float64)
    h = x @ inputs.bf16_bits_to_f32(prob["w_fc"]).astype(np.float64).T
    big = np.abs(h) > 1e-2
    assert np.all(np.sign(hn[big]) == np.sign(h[big]))


# ----------------------------------------------------- context-KV update


def _tiny_update(seed=0, **over):
    prob = inputs.make_problem(inputs.workload("tiny", **over), seed=seed)
    g = prob["g"]
    pool0 = prob["pool"].copy()
    pool = prob["pool"].copy()
    ctx_out = oracle.ctx_kv_update_gqa(g, prob["hidden"], prob["n_acc"], prob["ctx_len"],
                                       prob["alloc_limit"], prob["pages"], prob["valid"],
                                       prob["w_fc"], prob["g_h"], prob["w_kv"], prob["g_k"], pool)
    return prob, pool0, pool, ctx_out


def test_update_writes_only_destinations():
    prob, pool0, pool, ctx_out = _tiny_update()
    # tiny workload: c=100, n=3, P=16 -> rows at positions 100..102 on logical page 6
    page = prob["pages"][0, 6]
    changed = np.argwhere(pool != pool0)
    touched = {(int(c[1]), int(c[4])) for c in changed}  # (page, slot)
    assert touched == {(page, 4), (page, 5), (page, 6)}
    assert ctx_out.tolist() == [103]


def test_update_v_is_plain_projection_and_k_is_normed_rotation():
    prob, pool0, pool, _ = _tiny_update()
    g = prob["g"]
    hid = prob["hidden"].reshape(-1, 256)
    hn = oracle.bf16_to_f64(oracle.fc_hidden_norm(hid, prob["w_fc"], prob["g_h"], 1e-6))
    Wkv = inputs.bf16_bits_to_f32(prob["w_kv"]).astype(np.float64)  # [L, 2, nkv, hd, D]
    page = prob["pages"][0, 6]
    gk = oracle.bf16_to_f64(prob["g_k"][0])
    for i in range(3):
        for h in range(g["nkv"]):
            v_ref = Wkv[0, 1, h] @ hn[i]
            v = oracle.bf16_to_f64(pool[0, page, 1, h, 4 + i])
            np.testing.assert_allclose(v, v_ref, rtol=2 ** -8, atol=1e-6)
            # K: undo the gain and the rotation; what is left must be a positive
            # multiple of W_k hn (the norm is one scalar per head), with RMS 1.
            k = oracle.bf16_to_f64(pool[0, page, 0, h, 4 + i])
            k_unrot = oracle.rope_neox(k, -(100 + i), g["rope_theta"]) / gk
            t = Wkv[0, 0, h] @ hn[i]
            ratio = k_unrot / t
            big = np.abs(t) > 0.2 * np.max(np.abs(t))
            assert np.std(ratio[big]) < 2e-2 * np.mean(ratio[big])
            assert abs(np.sqrt(np.mean(k_unrot ** 2)) - 1.0) < 1e-2


def test_update_relative_rotation_between_rows():
    # duplicate hidden row 0 into row 1: stored K(row1) = R(+1) K(row0) up to bf16
    prob = inputs.make_problem(inputs.workload("tiny"), seed=0)
    prob["hidden"][0, 1] = prob["hidden"][0, 0]
    g = prob["g"]
    pool = prob["pool"].copy()
    oracle.ctx_kv_update_gqa(g, prob["hidden"], prob["n_acc"], prob["ctx_len"],
                             prob["alloc_limit"], prob["pages"], prob["valid"], prob["w_fc"],
                             prob["g_h"], prob["w_kv"], prob["g_k"], pool)
    page = prob["pages"][0, 6]
    for h in range(g["nkv"]):
        k0 = oracle.bf16_to_f64(pool[0, page, 0, h, 4])
        k1 = oracle.bf16_to_f64(pool[0, page, 0, h, 5])
        np.testing.assert_allclose(oracle.rope_neox(k0, 1, g["rope_theta"]), k1, atol=3e-2)
        np.testing.assert_array_equal(pool[0, page, 1, h, 4], pool[0, page, 1, h, 5])


def test_update_dummy_and_ceiling_rows():
    prob = inputs.make_problem(inputs.workload("tiny"), seed=0)
    g = prob["g"]
    pool = prob["pool"].copy()
    valid = np.zeros(1, np.uint8)
    ctx_out = oracle.ctx_kv_update_gqa(g, prob["hidden"], prob["n_acc"], prob["ctx_len"],
                                       prob["alloc_limit"], prob["pages"], valid, prob["w_fc"],
                                       prob["g_h"], prob["w_kv"], prob["g_k"], pool)
    assert ctx_out.tolist() == [0]
    np.testing.assert_array_equal(pool, prob["pool"])
    # ceiling: A = 101 -> only position 100 is written, c' = 101
    pool = prob["pool"].copy()
    ctx_out = oracle.ctx_kv_update_gqa(g, prob["hidden"], prob["n_acc"], prob["ctx_len"],
                                       np.array([101], np.int32), prob["pages"], None,
                                       prob["w_fc"], prob["g_h"], prob["w_kv"], prob["g_k"], pool)
    assert ctx_out.tolist() == [101]
    slots = {int(c[4]) for c in np.argwhere(pool != prob["pool"])}
    assert slots == {4}


def test_update_mla_latent_row():
    cfg = inputs.workload("mla", B=1, L=1, D_in=256, D=256, ctx=[70], n_acc=[2], T=4, P=16)
    prob = inputs.make_problem(cfg, seed=0)
    g = prob["g"]
    pool = prob["pool"].copy()
    ctx_out = oracle.ctx_kv_update_mla(g, prob["hidden"], prob["n_acc"], prob["ctx_len"],
                                       prob["alloc_limit"], prob["pages"], None, prob["w_fc"],
                                       prob["g_h"], prob["w_kv"], prob["g_k"], pool)
    assert ctx_out.tolist() == [72]
    page = prob["pages"][0, 70 // 16]
    changed = {(int(c[1]), int(c[2])) for c in np.argwhere(pool != prob["pool"])}
    assert changed == {(page, 70 % 16), (page, 71 % 16)}
    hn = oracle.bf16_to_f64(oracle.fc_hidden_norm(prob["hidden"].reshape(-1, 256), prob["w_fc"],
                                                  prob["g_h"], 1e-6))
    W = inputs.bf16_bits_to_f32(prob["w_kv"][0]).astype(np.float64)
    for i in range(2):
        row = oracle.bf16_to_f64(pool[0, page, (70 + i) % 16])
        c = W @ hn[i]
        lat = row[:512] / oracle.bf16_to_f64(prob["g_k"][0])
        assert abs(np.sqrt(np.mean(lat ** 2)) - 1.0) < 1e-2
        ratio = lat / c[:512]
        big = np.abs(c[:512]) > 0.2 * np.max(np.abs(c[:512]))
        assert np.std(ratio[big]) < 2e-2 * np.mean(ratio[big])
        rope = oracle.rope_neox(row[512:], -(70 + i), g["rope_theta"])
        np.testing.assert_allclose(rope, c[512:], rtol=2e-2, atol=2e-3)


# ----------------------------------------------------------- bookkeeping


def test_bookkeeping_hand_worked_cases():
    with open(os.path.join(GOLDEN, "bookkeeping_tiny.json")) as f:
        gold = json.load(f)
    cm = gold["common"]
    for case in gold["cases"]:
        off = np.array([case["off"]], np.int32)
        acc = np.array([case["acc"]], np.int32)
        out, st = oracle.bookkeeping(off, acc, np.array([case["n_acc"]]), np.array([case["ctx"]]),
                                     np.array([case["valid"]], np.uint8), M=cm["M"], T=cm["T"],
                                     P=cm["P"], off_div=case["off_div"], max_ctx=cm["max_ctx"],
                                     mask_id=cm["mask_id"])
        exp = case["expect"]
        assert st == exp["status"], case["name"]
        for key, val in exp.items():
            if key == "status":
                continue
            assert np.asarray(out[key]).reshape(-1).tolist() == np.asarray(val).reshape(-1).tolist(), \
                (case["name"], key)


def _random_bk(rng, B, T, P, M, div):
    off = np.full((B, M + 3), -1, np.int32)  # 3 extra columns: a strided view
    for r in range(B):
        n = rng.integers(0, M + 1)
        off[r, :n] = rng.permutation(4 * M)[:n] * div
        # sprinkle holes and zeros
        holes = rng.random(M) < 0.1
        off[r, :M][holes] = rng.choice([-1, 0, -7], size=holes.sum())
    acc = rng.integers(0, 1000, size=(B, T + 2)).astype(np.int32)
    n_acc = rng.integers(0, T + 2, size=B).astype(np.int32)
    ctx = rng.integers(-1, M * P + 8, size=B).astype(np.int32)
    valid = (rng.random(B) < 0.85).astype(np.uint8)
    return off, acc, n_acc, ctx, valid


@pytest.mark.parametrize("div", [1, 2, 3])
def test_bookkeeping_invariants(div):
    rng = np.random.default_rng(10 + div)
    T, P, M, max_ctx, mask = 4, 8, 6, 40, 99999
    for _ in range(40):
        B = 16
        off, acc, n_acc, ctx, valid = _random_bk(rng, B, T, P, M, div)
        out, st = oracle.bookkeeping(off, acc, n_acc, ctx, valid, M=M, T=T, P=P, off_div=div,
                                     max_ctx=max_ctx, mask_id=mask)
        for r in range(B):
            live = valid[r] and 1 <= n_acc[r] <= T and ctx[r] >= 0
            row = off[r, :M]
            tbl = out["block_table"][r]
            assert np.all(tbl >= 0) and np.all(tbl == np.maximum(row, 0) // div)
            if not live:
                assert out["ctx_len_new"][r] == 0 and out["seq_lens"][r] == 0
                assert out["ctx_wmask"][r].sum() == 0 and out["blk_mask"][r].sum() == 0
                assert np.all(out["emb_ids"][r] == mask)
                continue
            n, c = int(n_acc[r]), int(ctx[r])
            A = out["alloc_limit"][r]
            assert A == min(max_ctx, int((row >= 0).sum()) * P)
            assert out["bonus"][r] == acc[r, n - 1]
            assert out["emb_ids"][r, 0] == acc[r, n - 1] and np.all(out["emb_ids"][r, 1:] == mask)
            assert out["ctx_pos"][r].tolist() == list(range(c, c + T))
            cn = out["ctx_len_new"][r]
            assert cn <= A and (cn == c + n or cn == A)
            assert out["q_pos"][r].tolist() == list(range(cn, cn + T))
            assert out["seq_lens"][r] == cn + T
            # every written row is accepted, below A, on a mapped page, at its slot
            dst = set()
            for i in range(T):
                w = out["ctx_wmask"][r, i]
                p = c + i
                if w:
                    assert i < n and p < A and row[p // P] >= 0
                    assert out["ctx_dst_page"][r, i] == row[p // P] // div
                    assert out["ctx_dst_slot"][r, i] == p % P
                    dst.add((out["ctx_dst_page"][r, i], out["ctx_dst_slot"][r, i]))
                else:
                    assert out["ctx_dst_page"][r, i] == -1 and out["ctx_dst_slot"][r, i] == -1
                    assert i >= n or p >= A or row[p // P] < 0
            assert len(dst) == out["ctx_wmask"][r].sum()  # no two rows share a slot
            for i in range(T):
                p = cn + i
                if out["blk_mask"][r, i]:
                    assert out["blk_page"][r, i] == row[p // P] // div
                    assert out["blk_slot"][r, i] == p % P
        if np.any(valid.astype(bool) & ((n_acc < 1) | (n_acc > T))):
            assert st & oracle.ST_BAD_NACCEPTED


def test_bookkeeping_strided_views_equal_dense():
    rng = np.random.default_rng(7)
    T, P, M = 4, 8, 6
    off, acc, n_acc, ctx, valid = _random_bk(rng, 8, T, P, M, 1)
    a, _ = oracle.bookkeeping(off, acc, n_acc, ctx, valid, M=M, T=T, P=P, off_div=1, max_ctx=10 ** 6,
                              mask_id=5)
    b, _ = oracle.bookkeeping(off[:, :M].copy(), acc[:, :T].copy(), n_acc, ctx, valid, M=M, T=T, P=P,
                              off_div=1, max_ctx=10 ** 6, mask_id=5)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


# ------------------------------------------------------------- attention


def _dense_attention(q, Kd, Vd, mask, sink, scale):
    """Brute force: explicit [Tq, kv] mask matrix, numpy softmax, sink as an
    extra logit column carrying a zero value."""
    s = scale * (q @ Kd.T)
    s = np.where(mask, s, -np.inf)
    if sink is not None:
        s = np.concatenate([s, np.full((s.shape[0], 1), sink)], axis=1)
        Vd = np.concatenate([Vd, np.zeros((1, Vd.shape[1]))], axis=0)
    out = np.zeros((s.shape[0], Vd.shape[1]))
    for i in range(s.shape[0]):
        if np.all(np.isinf(s[i])):
            continue
        e = np.exp(s[i] - np.max(s[i]))
        out[i] = (e / e.sum()) @ Vd
    return out


def _mask_matrix(kv_len, Tq, window, mode):
    j = np.arange(kv_len)[None, :]
    p = (kv_len - Tq + np.arange(Tq))[:, None]
    m = np.ones((Tq, kv_len), bool)
    if mode == oracle.MASK_CAUSAL_TAIL:
        m &= j <= p
    if window > 0:
        m &= (p - j) < window
    return m


def _small_gqa(seed, kv_lens, hq=6, nkv=2, hd=16, P=8, Tq=3):
    rng = np.random.default_rng(seed)
    B = len(kv_lens)
    M = max(-(-k // P) for k in kv_lens) + 1
    NP = B * M + 3
    perm = rng.permutation(NP)
    tbl = np.full((B, M), -1, np.int32)
    pos = 0
    for r, k in enumerate(kv_lens):
        n = -(-k // P)
        tbl[r, :n] = perm[pos:pos + n]
        pos += n
    g = dict(nkv=nkv, P=P, num_pool_pages=NP)
    pool = inputs.f32_to_bf16_bits(rng.standard_normal((2, NP, 2, nkv, P, hd), dtype=np.float32))
    q = inputs.f32_to_bf16_bits(rng.standard_normal((B, Tq, hq, hd), dtype=np.float32))
    sinks = rng.standard_normal(hq).astype(np.float32)
    return g, pool, tbl, q, sinks


def _gather(pool, tbl, r, kv_len, layer, kv, kvh, P):
    rows = [pool[layer, tbl[r, j // P], kv, kvh, j % P] for j in range(kv_len)]
    return oracle.bf16_to_f64(np.array(rows).reshape(kv_len, -1))


@pytest.mark.parametrize("mode", [oracle.MASK_CAUSAL_TAIL, oracle.MASK_BLOCK_BIDIR])
@pytest.mark.parametrize("window", [0, 5, 1000])
@pytest.mark.parametrize("with_sink", [False, True])
def test_attention_matches_brute_force(mode, window, with_sink):
    kv_lens = [1, 2, 19, 40]
    g, pool, tbl, q, sinks = _small_gqa(20, kv_lens)
    out = oracle.attention_gqa(g, 1, q, pool, tbl, np.array(kv_lens), window=window,
                               sinks=sinks if with_sink else None, mask_mode=mode)
    hd, hq, Tq, G = q.shape[3], q.shape[2], q.shape[1], q.shape[2] // g["nkv"]
    for r, kl in enumerate(kv_lens):
        m = _mask_matrix(kl, Tq, window, mode)
        for h in range(hq):
            Kd = _gather(pool, tbl, r, kl, 1, 0, h // G, g["P"])
            Vd = _gather(pool, tbl, r, kl, 1, 1, h // G, g["P"])
            ref = _dense_attention(oracle.bf16_to_f64(q[r, :, h]), Kd, Vd, m,
                                   float(sinks[h]) if with_sink else None, 1 / math.sqrt(hd))
            np.testing.assert_allclose(out[r, :, h], ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("mode", [oracle.MASK_CAUSAL_TAIL, oracle.MASK_BLOCK_BIDIR])
@pytest.mark.parametrize("window", [0, 7])
def test_attention_split_count_invariance(mode, window):
    kv_lens = [3, 33, 57]
    g, pool, tbl, q, sinks = _small_gqa(21, kv_lens, Tq=4)
    ref = oracle.attention_gqa(g, 0, q, pool, tbl, np.array(kv_lens), window=window, sinks=sinks,
                               mask_mode=mode)
    for S in (1, 2, 3, 7, 16, 64, 100):
        out = oracle.attention_gqa(g, 0, q, pool, tbl, np.array(kv_lens), window=window,
                                   sinks=sinks, mask_mode=mode, num_segments=S)
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_attention_special_cases():
    g, pool, tbl, q, sinks = _small_gqa(22, [1, 25])
    hd, G = q.shape[3], q.shape[2] // g["nkv"]
    # one visible key (kv_len 1, query 2 of 3 at p = 0... causal tail: only the
    # last query sees key 0) -> out = v_0
    out = oracle.attention_gqa(g, 0, q, pool, tbl, np.array([1, 25]))
    for h in range(q.shape[2]):
        v0 = oracle.bf16_to_f64(pool[0, tbl[0, 0], 1, h // G, 0])
        np.testing.assert_allclose(out[0, 2, h], v0, rtol=1e-14)
        assert np.all(out[0, :2, h] == 0.0)  # empty key sets give 0
    # q = 0 -> equal scores -> mean of the visible values
    qz = np.zeros_like(q)
    out = oracle.attention_gqa(g, 0, qz, pool, tbl, np.array([1, 25]), mask_mode=1)
    for h in range(q.shape[2]):
        Vd = _gather(pool, tbl, 1, 25, 0, 1, h // G, g["P"])
        np.testing.assert_allclose(out[1, 0, h], Vd.mean(axis=0), rtol=1e-12)
    # a sink at -1e30 is no sink; a window >= kv_len is no window
    a = oracle.attention_gqa(g, 0, q, pool, tbl, np.array([1, 25]))
    b = oracle.attention_gqa(g, 0, q, pool, tbl, np.array([1, 25]),
                             sinks=np.full(q.shape[2], -1e30, np.float32))
    np.testing.assert_allclose(a, b, rtol=1e-14)
    c = oracle.attention_gqa(g, 0, q, pool, tbl, np.array([1, 25]), window=25)
    np.testing.assert_array_equal(a, c)
    # a sink equal to the only score halves the output of a single-key query
    qv = oracle.bf16_to_f64(q[0, 2, 0])
    k0 = oracle.bf16_to_f64(pool[0, tbl[0, 0], 0, 0, 0])
    s0 = np.float32(np.dot(qv, k0) / math.sqrt(hd))
    sk = np.full(q.shape[2], s0, np.float32)
    d = oracle.attention_gqa(g, 0, q, pool, tbl, np.array([1, 25]), sinks=sk)
    v0 = oracle.bf16_to_f64(pool[0, tbl[0, 0], 1, 0, 0])
    np.testing.assert_allclose(d[0, 2, 0], v0 / (1 + math.exp(float(s0) - np.dot(qv, k0) / math.sqrt(hd))),
                               rtol=1e-6)


def test_mla_attention_matches_brute_force():
    rng = np.random.default_rng(23)
    B, Tq, hq, lat, rope, P = 2, 3, 4, 32, 8, 8
    kv_lens = [9, 30]
    M = 5
    NP = 12
    perm = rng.permutation(NP)
    tbl = np.full((B, M), -1, np.int32)
    tbl[0, :2] = perm[:2]
    tbl[1, :4] = perm[2:6]
    pool = inputs.f32_to_bf16_bits(rng.standard_normal((1, NP, P, lat + rope), dtype=np.float32))
    ql = inputs.f32_to_bf16_bits(rng.standard_normal((B, Tq, hq, lat), dtype=np.float32))
    qr = inputs.f32_to_bf16_bits(rng.standard_normal((B, Tq, hq, rope), dtype=np.float32))
    sinks = rng.standard_normal(hq).astype(np.float32)
    g = dict(P=P, num_pool_pages=NP)
    for mode in (0, 1):
        out = oracle.attention_mla(g, 0, ql, qr, pool, tbl, np.array(kv_lens), window=6,
                                   sinks=sinks, scale=0.1, mask_mode=mode)
        for r, kl in enumerate(kv_lens):
            rows = oracle.bf16_to_f64(np.array([pool[0, tbl[r, j // P], j % P] for j in range(kl)]))
            m = _mask_matrix(kl, Tq, 6, mode)
            for h in range(hq):
                qq = np.concatenate([oracle.bf16_to_f64(ql[r, :, h]), oracle.bf16_to_f64(qr[r, :, h])],
                                    axis=1)
                ref = _dense_attention(qq, rows, rows[:, :lat], m, float(sinks[h]), 0.1)
                np.testing.assert_allclose(out[r, :, h], ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- scatter


def test_block_scatter_places_rows():
    rng = np.random.default_rng(30)
    B, T, nkv, hd, P, NP = 2, 3, 2, 8, 4, 6
    g = dict(nkv=nkv, hd=hd, P=P, num_pool_pages=NP)
    pool0 = rng.integers(0, 65535, size=(2, NP, 2, nkv, P, hd)).astype(np.uint16)
    bk = rng.integers(0, 65535, size=(B, T, nkv, hd)).astype(np.uint16)
    bv = rng.integers(0, 65535, size=(B, T, nkv, hd)).astype(np.uint16)
    page = np.array([[1, 1, 4], [5, 0, -1]], np.int32)
    slot = np.array([[2, 3, 0], [1, 3, -1]], np.int32)
    mask = np.array([[1, 1, 1], [1, 0, 0]], np.uint8)
    pool = pool0.copy()
    oracle.block_kv_scatter_gqa(g, 1, bk, bv, page, slot, mask, pool)
    exp = pool0.copy()
    for r in range(B):
        for i in range(T):
            if mask[r, i]:
                exp[1, page[r, i], 0, :, slot[r, i]] = bk[r, i]
                exp[1, page[r, i], 1, :, slot[r, i]] = bv[r, i]
    np.testing.assert_array_equal(pool, exp)


def test_block_latent_scatter_places_rows():
    # MLA block scatter: each placed row's whole latent (latent + rope part)
    # lands at (layer, page, slot); masked and unplaced rows, every other
    # slot and every other layer plane keep their nonzero contents.
    rng = np.random.default_rng(31)
    B, T, W, P, NP, L = 3, 4, 24, 4, 7, 3
    g = dict(P=P, num_pool_pages=NP)
    pool0 = rng.integers(1, 65535, size=(L, NP, P, W)).astype(np.uint16)
    blk = rng.integers(1, 65535, size=(B, T, W)).astype(np.uint16)
    page = np.array([[2, 2, 6, 0], [3, 3, 3, -1], [5, 1, -1, -1]], np.int32)
    slot = np.array([[0, 3, 1, 2], [1, 2, 0, -1], [3, 0, -1, -1]], np.int32)
    mask = np.array([[1, 1, 1, 0], [1, 1, 1, 0], [1, 1, 0, 0]], np.uint8)
    for layer in (0, L - 1):
        pool = pool0.copy()
        oracle.block_latent_scatter_mla(g, layer, blk, page, slot, mask, pool)
        exp = pool0.copy()
        for r in range(B):
            for i in range(T):
                if mask[r, i]:
                    exp[layer, page[r, i], slot[r, i]] = blk[r, i]
        np.testing.assert_array_equal(pool, exp)
        # exactly the placed rows changed, and only in this layer's plane
        changed = np.argwhere(np.any(pool != pool0, axis=-1))
        assert len(changed) == int(mask.sum())
        assert set(changed[:, 0].tolist()) == {layer}
