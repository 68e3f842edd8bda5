"""The C-ABI library loads and exports every symbol include/dflash.h declares;
host-side validation rejects bad arguments before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from context_kv_update_gb300 import build, _lib
    build.build()
    return _lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "dflash.h")).read()
    return re.findall(r"DFLASH_API\s+[\w\s\*]+?\b(dflash_\w+)\s*\(", src)


def test_header_declares_the_entry_points():
    names = set(_declared())
    for n in ("dflash_step_bookkeeping", "dflash_ctx_kv_update", "dflash_block_kv_scatter",
              "dflash_block_attention", "dflash_ctx_workspace_bytes",
              "dflash_attention_workspace_bytes", "dflash_attention_num_segments",
              "dflash_ctx_kv_project", "dflash_ctx_kv_commit", "dflash_ctx_staged_bytes",
              "dflash_q_norm_rope", "dflash_pack_weights", "dflash_packed_kv_bytes",
              "dflash_packed_gamma_bytes", "dflash_strict_accept", "dflash_embedding_gather",
              "dflash_ctx_kv_prefill", "dflash_ctx_prefill_workspace_bytes",
              "dflash_block_scatter_attention"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from context_kv_update_gb300 import _lib
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) == set(_lib.EXPORTS)
    # nothing else leaks out of the shared object
    out = os.popen(f"nm -D --defined-only {_lib.LIB_PATH}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(_declared())


def test_struct_sizes_match_header(lib):
    from context_kv_update_gb300 import _lib
    assert ctypes.sizeof(_lib.Geom) == 14 * 4 + 3 * 8
    assert ctypes.sizeof(_lib.Weights) == 4 * 8
    assert ctypes.sizeof(_lib.StepOutputs) == 15 * 8
    assert ctypes.sizeof(_lib.LayerWeights) == 3 * 8


def _geom():
    from context_kv_update_gb300 import inputs, make_geom
    prob = inputs.make_problem(inputs.workload("tiny"), seed=0, with_pool=False, with_weights=False)
    return make_geom(prob["g"])


def test_validation_rejects_without_launching(lib):
    from context_kv_update_gb300 import _lib
    g = _geom()
    G = ctypes.byref(g)
    null = None
    # null geometry / negative batch / bad layer / bad mask mode
    assert lib.dflash_block_attention(None, 1, 0, 4, null, null, null, null, null, 0, null, 1.0, 0,
                                      0, null, 0, null, null, null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_block_attention(G, -1, 0, 4, null, null, null, null, null, 0, null, 1.0, 0,
                                      0, null, 0, null, null, null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_block_attention(G, 1, 5, 4, null, null, null, null, null, 0, null, 1.0, 0,
                                      0, null, 0, null, null, null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_block_attention(G, 1, 0, 4, null, null, null, null, null, 0, null, 1.0, 7,
                                      0, null, 0, null, null, null) == _lib.DFLASH_ERR_INVALID_ARG
    # null buffers
    assert lib.dflash_block_attention(G, 1, 0, 4, null, null, null, null, null, 0, null, 1.0, 0,
                                      0, null, 0, null, null, null) == _lib.DFLASH_ERR_INVALID_ARG
    # B == 0 is a no-op
    assert lib.dflash_block_attention(G, 0, 0, 4, null, null, null, null, null, 0, null, 1.0, 0,
                                      0, null, 0, null, null, null) == _lib.DFLASH_OK
    # misaligned q
    p = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1002)
    assert lib.dflash_block_attention(G, 1, 0, 4, odd, null, p, p, p, 0, null, 1.0, 0, 1, p,
                                      1 << 30, p, null, null) == _lib.DFLASH_ERR_INVALID_ARG
    # workspace too small
    assert lib.dflash_block_attention(G, 1, 0, 4, p, null, p, p, p, 0, null, 1.0, 0, 1, p, 16, p,
                                      null, null) == _lib.DFLASH_ERR_WORKSPACE_TOO_SMALL
    # unsupported head dim
    g2 = _geom()
    g2.head_dim = 96
    assert lib.dflash_block_attention(ctypes.byref(g2), 1, 0, 4, p, null, p, p, p, 0, null, 1.0,
                                      0, 1, p, 1 << 30, p, null,
                                      null) == _lib.DFLASH_ERR_UNSUPPORTED_GEOM
    # MLA requires q_rope; GQA forbids it
    assert lib.dflash_block_attention(G, 1, 0, 4, p, p, p, p, p, 0, null, 1.0, 0, 1, p, 1 << 30, p,
                                      null, null) == _lib.DFLASH_ERR_INVALID_ARG
    # ctx update: bad dtype, workspace too small, missing weights
    w = _lib.Weights(0x1000, 0x1000, 0x1000, 0x1000)
    assert lib.dflash_ctx_kv_update(G, 1, p, 9, p, p, p, p, null, ctypes.byref(w), p, p, 1 << 30,
                                    null, null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_ctx_kv_update(G, 1, p, 0, p, p, p, p, null, ctypes.byref(w), p, p, 64, null,
                                    null) == _lib.DFLASH_ERR_WORKSPACE_TOO_SMALL
    w0 = _lib.Weights(0x1000, None, 0x1000, 0x1000)
    assert lib.dflash_ctx_kv_update(G, 1, p, 0, p, p, p, p, null, ctypes.byref(w0), p, p, 1 << 30,
                                    null, null) == _lib.DFLASH_ERR_INVALID_ARG
    # split update: staged bytes cover c [B] + rows; short or misaligned staged
    # buffers, bad dtype and missing arguments are rejected before any launch
    T, L, nkv, hd = g.block_size, g.num_layers, g.nkv, g.head_dim
    assert lib.dflash_ctx_staged_bytes(G, 3) == 256 + 3 * T * L * 2 * nkv * hd * 2
    assert lib.dflash_ctx_staged_bytes(None, 3) == 0
    assert lib.dflash_ctx_kv_project(G, 1, p, 9, p, ctypes.byref(w), p, 1 << 30, p, 1 << 30,
                                     null, null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_ctx_kv_project(G, 1, p, 0, p, ctypes.byref(w), p, 16, p, 1 << 30,
                                     null, null) == _lib.DFLASH_ERR_WORKSPACE_TOO_SMALL
    assert lib.dflash_ctx_kv_project(G, 1, p, 0, p, ctypes.byref(w), odd, 1 << 30, p, 1 << 30,
                                     null, null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_ctx_kv_project(G, 1, p, 0, null, ctypes.byref(w), p, 1 << 30, p, 1 << 30,
                                     null, null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_ctx_kv_project(G, 0, null, 0, null, ctypes.byref(w), null, 0, null, 0,
                                     null, null) == _lib.DFLASH_OK
    assert lib.dflash_ctx_kv_commit(G, 1, p, 16, p, p, p, p, null, p, null,
                                    null) == _lib.DFLASH_ERR_WORKSPACE_TOO_SMALL
    assert lib.dflash_ctx_kv_commit(G, 1, odd, 1 << 30, p, p, p, p, null, p, null,
                                    null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_ctx_kv_commit(G, 1, p, 1 << 30, null, p, p, p, null, p, null,
                                    null) == _lib.DFLASH_ERR_INVALID_ARG
    # query norm + RoPE (every case here is rejected before any launch): GQA
    # without the gain, Tq < 1, a pointer off the 2-byte grid; B == 0 is a no-op
    odd1 = ctypes.c_void_p(0x1001)
    assert lib.dflash_q_norm_rope(G, 1, 4, p, null, p, p, null, null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_q_norm_rope(G, 1, 0, p, p, p, p, null, null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_q_norm_rope(G, 1, 4, odd1, p, p, p, null,
                                  null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_q_norm_rope(G, 1, 4, p, p, null, p, null,
                                  null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_q_norm_rope(G, 0, 4, null, p, null, null, null, null) == _lib.DFLASH_OK
    # bookkeeping: off_div < 1, stride below the row width
    outs = _lib.StepOutputs(*([0x1000] * 15))
    assert lib.dflash_step_bookkeeping(G, 1, p, 16, 0, p, 4, p, p, null, 100, 7,
                                       ctypes.byref(outs), null, null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_step_bookkeeping(G, 1, p, 3, 1, p, 4, p, p, null, 100, 7,
                                       ctypes.byref(outs), null, null) == _lib.DFLASH_ERR_INVALID_ARG
    # scatter: MLA-only NULL blk_v rule, bad layer
    assert lib.dflash_block_kv_scatter(G, 1, 0, p, null, p, p, p, p, null,
                                       null) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_block_kv_scatter(G, 1, 3, p, p, p, p, p, p, null,
                                       null) == _lib.DFLASH_ERR_INVALID_ARG


def test_fused_scatter_attention_validation(lib):
    """The fused scatter + attention call checks the block width against the
    geometry's block_size, before the B == 0 no-op (every pointer stays null:
    nothing can launch)."""
    from context_kv_update_gb300 import _lib
    g = _geom()  # block_size 4
    G = ctypes.byref(g)
    null = None

    def call(Tq, B=1, blk_k=null, blk_v=null, page=null, slot=null, mask=null):
        return lib.dflash_block_scatter_attention(G, B, 0, Tq, blk_k, blk_v, page, slot, mask,
                                                  null, null, null, null, null, 0, null, 1.0, 0,
                                                  0, null, 0, null, null, null)
    assert call(5) == _lib.DFLASH_ERR_INVALID_ARG          # Tq != block_size
    assert call(5, B=0) == _lib.DFLASH_ERR_INVALID_ARG     # checked before the B == 0 no-op
    assert call(4, B=0) == _lib.DFLASH_OK
    assert call(4) == _lib.DFLASH_ERR_INVALID_ARG          # null buffers


def test_workspace_queries(lib):
    from context_kv_update_gb300 import _lib
    g = _geom()
    assert lib.dflash_ctx_workspace_bytes(ctypes.byref(g), 1) > 0
    assert lib.dflash_attention_workspace_bytes(ctypes.byref(g), 1, 4, 3) >= 3 * 4 * 4 * (64 + 2) * 4
    assert lib.dflash_attention_workspace_bytes(None, 1, 4, 3) == 0
    assert lib.dflash_status_string(3) == b"workspace too small"


def test_attention_scale_default_and_argument_order(lib):
    """scale <= 0 selects the library's default (accepted: the call reaches the
    workspace check); a non-finite scale is an argument error.  The
    allocation-free call checks its arguments first, then its size limit, then
    the buffer pointers (so NULL buffers on an oversized problem report the
    size, and a bad mode reports the mode)."""
    from context_kv_update_gb300 import _lib
    g = _geom()
    G = ctypes.byref(g)
    p = ctypes.c_void_p(0x1000)
    for scale in (0.0, -1.0):
        assert lib.dflash_block_attention(G, 1, 0, 4, p, None, p, p, p, 0, None, scale, 0, 1, p, 16,
                                          p, None, None) == _lib.DFLASH_ERR_WORKSPACE_TOO_SMALL
    for scale in (float("nan"), float("inf")):
        assert lib.dflash_block_attention(G, 1, 0, 4, p, None, p, p, p, 0, None, scale, 0, 1, p,
                                          1 << 30, p, None, None) == _lib.DFLASH_ERR_INVALID_ARG
    big_B, S = 4096, 64
    assert lib.dflash_block_attention_noalloc(G, big_B, 0, 4, None, None, None, None, None, 0, None,
                                              0.0, 0, S, None, None,
                                              None) == _lib.DFLASH_ERR_WORKSPACE_TOO_SMALL
    assert lib.dflash_block_attention_noalloc(G, big_B, 0, 4, None, None, None, None, None, 0, None,
                                              0.0, 5, S, None, None,
                                              None) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_block_attention_noalloc(G, big_B, 9, 4, None, None, None, None, None, 0, None,
                                              0.0, 0, S, None, None,
                                              None) == _lib.DFLASH_ERR_INVALID_ARG
    # a small problem with NULL buffers stops at the pointer check
    assert lib.dflash_block_attention_noalloc(G, 1, 0, 4, None, None, None, None, None, 0, None,
                                              0.0, 0, 1, None, None,
                                              None) == _lib.DFLASH_ERR_INVALID_ARG
    # B == 0 with a bad argument is still an error
    assert lib.dflash_block_attention_noalloc(G, 0, 0, 4, None, None, None, None, None, -1, None,
                                              0.0, 0, 0, None, None,
                                              None) == _lib.DFLASH_ERR_INVALID_ARG


def test_pack_accept_gather_validation(lib):
    from context_kv_update_gb300 import _lib
    g = _geom()
    G = ctypes.byref(g)
    p = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1008)
    L, nkv, hd, D = g.num_layers, g.nkv, g.head_dim, g.d_model
    assert lib.dflash_packed_kv_bytes(G) == L * 2 * nkv * hd * D * 2
    assert lib.dflash_packed_gamma_bytes(G) == L * hd * 2
    assert lib.dflash_packed_kv_bytes(None) == 0
    ok = (_lib.LayerWeights * L)(*[_lib.LayerWeights(0x1000, 0x2000, 0x3000)] * L)
    no_v = (_lib.LayerWeights * L)(*[_lib.LayerWeights(0x1000, None, 0x3000)] * L)
    bad_al = (_lib.LayerWeights * L)(*[_lib.LayerWeights(0x1008, 0x2000, 0x3000)] * L)
    assert lib.dflash_pack_weights(G, no_v, p, p, None) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_pack_weights(G, bad_al, p, p, None) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_pack_weights(G, ok, odd, p, None) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_pack_weights(G, None, p, p, None) == _lib.DFLASH_ERR_INVALID_ARG
    g65 = _geom()
    g65.num_layers = 65
    assert lib.dflash_pack_weights(ctypes.byref(g65), ok, p, p,
                                   None) == _lib.DFLASH_ERR_UNSUPPORTED_GEOM
    # strict acceptance: negative sizes, short strides, missing outputs; B == 0
    assert lib.dflash_strict_accept(-1, 3, p, 3, p, 4, p, p, None) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_strict_accept(2, 3, p, 2, p, 4, p, p, None) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_strict_accept(2, 3, p, 3, p, 3, p, p, None) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_strict_accept(2, 3, p, 3, p, 4, None, p, None) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_strict_accept(0, 3, None, 3, None, 4, None, None, None) == _lib.DFLASH_OK
    # embedding lookup: dim not a multiple of 8, misaligned table, n == 0
    assert lib.dflash_embedding_gather(4, p, p, 100, 12, p, None,
                                       None) == _lib.DFLASH_ERR_UNSUPPORTED_GEOM
    assert lib.dflash_embedding_gather(4, p, odd, 100, 16, p, None,
                                       None) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_embedding_gather(4, p, p, 0, 16, p, None,
                                       None) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_embedding_gather(0, None, None, 100, 16, None, None, None) == _lib.DFLASH_OK


def test_prefill_validation(lib):
    from context_kv_update_gb300 import _lib
    g = _geom()
    G = ctypes.byref(g)
    p = ctypes.c_void_p(0x1000)
    w = _lib.Weights(0x1000, 0x1000, 0x1000, 0x1000)
    W = ctypes.byref(w)
    assert lib.dflash_ctx_prefill_workspace_bytes(G, 2, 100) > lib.dflash_ctx_prefill_workspace_bytes(G, 2, 10)
    assert lib.dflash_ctx_prefill_workspace_bytes(G, 2, 70000) == 0
    # more rows than one call takes, bad dtype, missing cu_rows, short workspace
    assert lib.dflash_ctx_kv_prefill(G, 1, 70000, p, 0, p, p, p, p, None, W, p, p, 1 << 40, None,
                                     None) == _lib.DFLASH_ERR_UNSUPPORTED_GEOM
    assert lib.dflash_ctx_kv_prefill(G, 1, 10, p, 7, p, p, p, p, None, W, p, p, 1 << 40, None,
                                     None) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_ctx_kv_prefill(G, 1, 10, p, 0, None, p, p, p, None, W, p, p, 1 << 40, None,
                                     None) == _lib.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_ctx_kv_prefill(G, 1, 10, p, 0, p, p, p, p, None, W, p, p, 64, None,
                                     None) == _lib.DFLASH_ERR_WORKSPACE_TOO_SMALL
    assert lib.dflash_ctx_kv_prefill(G, 0, 0, None, 0, None, None, None, None, None, W, None, None,
                                     0, None, None) == _lib.DFLASH_OK
