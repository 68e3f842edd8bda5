"""Host-side arithmetic of bench.py that the roofline and launch-count fields
rest on: the workload selection, each configuration's algorithmic bytes and
FLOPs per attention call (checked against the counts written out by hand),
and the kernel launches per step."""
import argparse

import numpy as np

import bench
from context_kv_update_gb300 import inputs


def _args(**kw):
    a = argparse.Namespace(workload=None, ctx=None, window=None)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _prob(**kw):
    tag, cfg = bench.workload_config(_args(**kw))
    return tag, inputs.make_problem(cfg, seed=0, with_weights=False, with_pool=False)


def test_headline_bytes_per_call():
    tag, prob = _prob()
    assert tag == bench.WORKLOAD_TAG
    nbytes, flops, kv = bench.attention_work(prob)
    g = prob["g"]
    # B = 1: every visible key once, K and V, 8 heads x 128 dims x 2 B
    assert prob["B"] == 1 and kv == int(prob["ctx_len"][0]) + int(prob["n_acc"][0]) + g["T"]
    assert nbytes == kv * 8 * 128 * 2 * 2
    # QK and PV: 2 FLOPs per multiply-add, 16 tokens x 32 heads, 128 dims each
    assert flops == 2 * 2 * kv * (16 * 32) * 128
    # per layer the fused scatter + attention call: main kernel + merge
    assert bench.kernel_launches_per_step(g) == 1 + 4 + 5 * 2
    assert bench.kernel_launches_per_step(g, fused_layer=False) == 1 + 4 + 5 * 3
    # beyond 256 update rows the many-row epilogue adds its row set-up launch
    assert bench.kernel_launches_per_step(g, B=16) == 1 + 4 + 5 * 2
    assert bench.kernel_launches_per_step(g, B=17) == 1 + 4 + 1 + 5 * 2
    # the block scatter: 16 rows x K, V of 8 heads x 128 dims, read and written
    assert bench.block_scatter_bytes(prob) == 2 * 16 * 2 * 8 * 128 * 2


def test_fused_layer_rule():
    """The caller-side choice of the fused scatter + attention call: the 32K
    headline (one wave of 152 CTAs, the block in a 5-tile tail segment of
    14-tile segments) fuses; a 2K context (one-tile segments), the batch
    sweeps past one wave and the MLA drafter do not."""
    _, prob = _prob()
    assert bench.fused_layer_pays(prob, 19, 152)
    assert not bench.fused_layer_pays(prob, 19, 100)  # more CTAs than SMs
    _, p2k = _prob(ctx=2048)
    assert not bench.fused_layer_pays(p2k, 19, 152)
    _, pb4 = _prob(workload="batch_sweep_4")
    assert not bench.fused_layer_pays(pb4, 7, 152)
    _, pm = _prob(workload="mla", ctx=32768)
    assert not bench.fused_layer_pays(pm, 19, 152)
    # a block in a full-length segment: kv_len = 34040 fills 266 = 19 x 14
    # tiles, so the block's rows land in the last of 19 equal segments
    prob_full = dict(prob, ctx_len=np.array([34040 - 1 - 16], np.int32),
                     n_acc=np.array([1], np.int32), alloc_limit=np.array([1 << 20], np.int32))
    assert not bench.fused_layer_pays(prob_full, 19, 152)


def test_sliding_window_reads_only_the_window():
    _, prob = _prob(workload="sliding_window")
    nbytes, _, _ = bench.attention_work(prob)
    # the union of the rows' windows: (W + Tq - 1) keys x 2 heads x 128 x 2 x 2 B
    assert nbytes == (1024 + 3 - 1) * 2 * 128 * 2 * 2
    tag, prob0 = _prob(workload="sliding_window", window=0)
    assert tag == "sliding_window_window0"
    full, _, kv = bench.attention_work(prob0)
    assert full == kv * 2 * 128 * 2 * 2


def test_mla_intensity():
    tag, prob = _prob(workload="mla", ctx=32768)
    assert tag == "mla_ctx32768"
    nbytes, flops, kv = bench.attention_work(prob)
    assert nbytes == kv * 576 * 2
    rows = 8 * 64
    assert flops == 2 * kv * rows * (576 + 512)
    assert round(flops / nbytes) == 967
    assert bench.block_scatter_bytes(prob) == 2 * 8 * 576 * 2


def test_batch_sweep_counts_every_request():
    tag, prob = _prob(workload="batch_sweep_8")
    assert tag == "batch_sweep_8"
    nbytes, _, _ = bench.attention_work(prob)
    kv = np.minimum(prob["ctx_len"].astype(np.int64) + prob["n_acc"], prob["alloc_limit"]) + 16
    assert nbytes == int(kv.sum()) * 8 * 128 * 2 * 2


def test_launch_counts_of_the_variants():
    _, prob = _prob(workload="tiny")
    g = prob["g"]
    assert prob["hidden"].dtype == np.float32
    assert bench.kernel_launches_per_step(g, True) == 1 + 4 + 1 + 1 * 2
    assert bench.kernel_launches_per_step(g, True, True) == 1 + 4 + 1 + 1 + 1 * 2
    assert bench.kernel_launches_per_step(g, True, True, 1, False) == 1 + 4 + 1 + 1 + 1 * 3
