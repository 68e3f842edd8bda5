"""Planted-mistake checks: each mutation of a copy of oracle.c must make at
least one pin fail.  The mutated copy is built in a temporary directory and
swapped in for the duration of one test; the committed oracle is untouched."""
import os
import subprocess

import pytest

import oracle
import tests.test_oracle_accept_gather as accept_pins
import tests.test_oracle_pins as pins
import tests.test_oracle_prefill as prefill_pins
import tests.test_oracle_q_rope as q_pins
import tests.test_oracle_split_update as split_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = [
    # (id, original text, replacement, pin functions that must catch it)
    ("rope_sign", "out[j] = x0 * c - x1 * s;", "out[j] = x0 * c + x1 * s;",
     [pins.test_rope_two_dims_is_plain_rotation]),
    ("rope_freq", "pow(theta, -2.0 * (double)j / (double)n)", "pow(theta, -1.0 * (double)j / (double)n)",
     [pins.test_rope_known_frequency_quarter_turn]),
    ("rms_divisor", "ss / (double)n + eps", "ss / (double)(n - 1) + eps",
     [pins.test_rmsnorm_unit_rms_and_scale_invariance]),
    ("window_off_by_one", "int w0 = p - window + 1;", "int w0 = p - window;",
     [lambda: pins.test_attention_matches_brute_force(oracle.MASK_CAUSAL_TAIL, 5, False)]),
    ("causal_off_by_one", "(mask_mode == OR_MASK_CAUSAL_TAIL) ? p : kv_len - 1",
     "(mask_mode == OR_MASK_CAUSAL_TAIL) ? p - 1 : kv_len - 1",
     [lambda: pins.test_attention_matches_brute_force(oracle.MASK_CAUSAL_TAIL, 0, False)]),
    ("merge_weight", "den += w * ls[sI];", "den += ls[sI];",
     [lambda: pins.test_attention_split_count_invariance(oracle.MASK_BLOCK_BIDIR, 0)]),
    ("advance_unclamped", "cn = (int)(s < A ? s : A);", "cn = (int)s;",
     [pins.test_bookkeeping_hand_worked_cases]),
    ("table_no_clamp", "tbl[(int64_t)r * M + j] = (v > 0 ? v : 0) / off_div;",
     "tbl[(int64_t)r * M + j] = v / off_div;", [pins.test_bookkeeping_hand_worked_cases]),
    ("kv_head_swap", "oracle_matvec_bf16(W, hd, D, hn, t);",
     "oracle_matvec_bf16(W + (kv == 0 ? (size_t)nkv * hd * D : 0), hd, D, hn, t);",
     [pins.test_update_v_is_plain_projection_and_k_is_normed_rotation]),
    # the next rows' functions
    ("accept_off_by_one", "n_acc[r] = m + 1;", "n_acc[r] = m;",
     [accept_pins.test_strict_accept_hand_cases]),
    ("q_norm_dropped", "oracle_rmsnorm(x, g, dim, eps, n);", "memcpy(n, x, sizeof(double) * dim);",
     [q_pins.test_position_zero_is_plain_rmsnorm]),
    ("commit_kv_swap", "memcpy(dst, src + (((size_t)l * 2 + kv) * nkv + hh) * hd, sizeof(uint16_t) * hd);",
     "memcpy(dst, src + (((size_t)l * 2 + (1 - kv)) * nkv + hh) * hd, sizeof(uint16_t) * hd);",
     [lambda: split_pins.test_split_update_equals_fused(*split_pins._cases()[1])]),
    ("latent_scatter_layer_stride",
     "memcpy(pool + (((size_t)layer * num_pool_pages + pg) * P + sl) * (size_t)W,",
     "memcpy(pool + (((size_t)num_pool_pages + pg) * P + sl) * (size_t)W,",
     [pins.test_block_latent_scatter_places_rows]),
    ("latent_scatter_row_stride",
     "blk_lat + (size_t)k * W, sizeof(uint16_t) * W);",
     "blk_lat + (size_t)i * W, sizeof(uint16_t) * W);",
     [pins.test_block_latent_scatter_places_rows]),
    # prefill context store
    ("prefill_position_off_by_one", "int i = n - cu_rows[r];", "int i = n - cu_rows[r] + 1;",
     [lambda: prefill_pins.test_prefill_of_one_request_is_one_all_accepted_update_block("gqa")]),
    ("prefill_request_lookup", "while (cu_rows[r + 1] <= n) ++r;", "while (cu_rows[r + 1] < n) ++r;",
     [lambda: prefill_pins.test_prefill_requests_are_independent("mla")]),
    ("prefill_advance", "long long s = (long long)c + (cu_rows[r + 1] - cu_rows[r]);",
     "long long s = (long long)c + (cu_rows[r + 1] - cu_rows[r]) - 1;",
     [lambda: prefill_pins.test_prefill_of_one_request_is_one_all_accepted_update_block("mla")]),
]


@pytest.mark.parametrize("mid,old,new,catchers", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(tmp_path, monkeypatch, mid, old, new, catchers):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {mid} not unique"
    mut = tmp_path / "oracle_mut.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-std=c11", "-O1", "-fPIC", "-shared", "-fopenmp", str(mut), "-o",
                    str(so), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.load_variant(str(so)))
    caught = False
    for fn in catchers:
        try:
            fn()
        except (AssertionError, ValueError):
            caught = True
    assert caught, f"mutation {mid} survived its pins"
