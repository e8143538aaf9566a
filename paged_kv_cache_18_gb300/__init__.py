"""GB300-native paged KV-cache decode attention.

The compute path is ``libpkv.so`` (hand-written CUDA for sm_103a behind the C
ABI in ``include/pkv.h``); this package is its thin Python binding plus the
seeded workload generator and byte accounting used by the tests and the
benchmark.  Build the library with ``paged_kv_cache_18_gb300.build.build()``.
"""
from .binding import (PKV_KERNEL_AUTO, PKV_KERNEL_MMA, PKV_KERNEL_SIMT,  # noqa: F401
                      PKV_KERNEL_TC, BlockManager, PkvError, append_attention,
                      append_attention_host, bm_hash, copy_blocks, host_step_staging_size,
                      kv_append, kv_append_fp8, mla_append, mla_decode_attention,
                      mla_plan, mla_workspace_size, paged_attention_fp8, paged_decode_attention,
                      paged_prefill_attention, plan, plan_for, read_error_word,
                      spec_verify_attention, tree_verify_attention, version, workspace_size)
