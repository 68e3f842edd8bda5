"""GB300 (sm_103a) library for the data-parallel hot path of a DFlash / DSpark
block drafter's decode step: bookkeeping, context-KV update, block-KV scatter
and split-KV block attention, behind the C ABI of include/dflash.h.

The Python names below are the C entry points of the same names (ctypes
marshalling only).  ``inputs`` holds the seeded synthetic workloads.
"""
from ._lib import (DflashError, Geom, LayerWeights, StepOutputs, Weights,  # noqa: F401
                   STEP_OUTPUT_FIELDS, dflash_embedding_gather, dflash_pack_weights,
                   dflash_packed_gamma_bytes, dflash_packed_kv_bytes, dflash_strict_accept,
                   dflash_attention_num_segments, dflash_attention_workspace_bytes,
                   dflash_block_attention, dflash_block_attention_noalloc,
                   dflash_block_attention_noalloc_max_scratch_bytes, dflash_block_kv_scatter,
                   dflash_block_scatter_attention,
                   dflash_ctx_kv_commit, dflash_ctx_kv_prefill, dflash_ctx_kv_project,
                   dflash_ctx_kv_update, dflash_ctx_prefill_workspace_bytes,
                   dflash_ctx_staged_bytes, dflash_ctx_workspace_bytes, dflash_q_norm_rope,
                   dflash_step_bookkeeping, dflash_test_attention_skip_tile, load, make_geom,
                   KIND_GQA, KIND_MLA, MASK_CAUSAL_TAIL, MASK_BLOCK_BIDIR)
