"""The allocation-free decode entry point, pkv_paged_decode_attention_noalloc.

It exists for callers that cannot allocate device memory per call (a plugin
whose host framework owns every device allocation, or a latency-critical loop
that must not call cudaMalloc/cudaFree), so it keeps the split-K partials in
a fixed scratch array inside the library instead of a caller workspace.

This file is collected last on purpose, so that a failure here cannot stop a
``-x`` run before every other test has run.  The checks call the C ABI
directly and compare the new entry point with pkv_paged_decode_attention on
the same inputs, twice in a row (the scratch array keeps the previous call's
contents between calls).
"""
import ctypes

import pytest
import torch

from paged_kv_cache_18_gb300 import binding
from paged_kv_cache_18_gb300 import workloads as W
from tests.gpu_util import DeviceBatch, assert_close, host_f64, oracle_after_append

pytestmark = pytest.mark.gpu

SCRATCH = 8 << 20  # PKV_NOALLOC_SCRATCH_BYTES


def _call_noalloc(d, out, split_blocks, merge=0):
    b, wl = d.b, d.b.wl
    L = binding.lib()
    opts = binding.Options(0, split_blocks, 0, 0, merge)
    return L.pkv_paged_decode_attention_noalloc(
        out.data_ptr(), d.q[:, 0].data_ptr(), d.k_cache.data_ptr(), d.v_cache.data_ptr(),
        d.table.data_ptr(), d.table.shape[1], d.lens.data_ptr(), b.max_context_len, wl.batch,
        wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, b.num_blocks,
        wl.softmax_scale, 1, ctypes.byref(opts), d.err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("split_blocks", [0, 3])
def test_noalloc_matches_workspace_entry_point_twice(split_blocks):
    wl = W.Workload("noalloc", 4, 32, 8, 128, "bf16", context_lens=[70, 900, 2500, 4096],
                    seed=41 + split_blocks)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    need = binding.workspace_size(wl.batch, 1, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                  b.max_context_len, torch.bfloat16, split_blocks=split_blocks)
    assert 0 < need <= SCRATCH  # the case really uses the scratch array
    ref = d.attend(split_blocks=split_blocks)[:, 0].clone()
    oracle = oracle_after_append(b)[:, 0]
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _call_noalloc(d, out, split_blocks) == 0
        torch.cuda.synchronize()
        assert int(d.err.item()) == 0
        assert_close(host_f64(out, "bf16"), host_f64(ref, "bf16"), "bf16", "noalloc vs workspace")
        assert_close(host_f64(out, "bf16"), oracle, "bf16", "noalloc vs oracle")


def test_noalloc_rejects_partials_beyond_the_scratch():
    wl = W.Workload("noalloc big", 64, 32, 8, 128, "bf16", context_lens=[40000], seed=43)
    need = binding.workspace_size(wl.batch, 1, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                  40000, torch.bfloat16, split_blocks=16)
    assert need > SCRATCH
    L = binding.lib()
    opts = binding.Options(0, 16)
    # rejected before anything is enqueued.  The device pointers are null, so
    # that should the size check ever regress, the attention call's own
    # argument check refuses the call (PKV_ERR_INVALID_ARG) instead of
    # launching kernels on made-up addresses.
    st = L.pkv_paged_decode_attention_noalloc(None, None, None, None, None, 2500, None, 40000,
                                              64, 32, 8, 128, 16, 100000, 0.1, 1,
                                              ctypes.byref(opts), None, None)
    assert st == 3  # PKV_ERR_WORKSPACE


def test_noalloc_varied_shapes_with_the_last_cta_merge():
    """Calls of different shapes in turn share the scratch array; with the
    last-CTA merge forced, each call's arrival counters land on what the
    previous call left there (partials or counters) and must still start
    from zero."""
    cases = [(W.Workload("na a", 6, 32, 8, 128, "bf16", len_range=(500, 4000), seed=44), 16),
             (W.Workload("na b", 3, 16, 4, 128, "bf16", len_range=(100, 2500), seed=45), 8),
             (W.Workload("na c", 9, 8, 8, 64, "bf16", len_range=(300, 3000), seed=46), 12),
             (W.Workload("na d", 2, 32, 8, 128, "bf16", context_lens=[6000, 9000], seed=47),
              20)]
    batches = []
    for wl, sb in cases:
        b = W.make_batch(wl)
        d = DeviceBatch(b)
        d.append()
        pl = binding.plan(wl.batch, 1, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                          b.max_context_len, torch.bfloat16, split_blocks=sb)
        assert 1 < pl["num_splits"] <= 32 and 0 < pl["workspace_bytes"] <= SCRATCH
        batches.append((d, sb, oracle_after_append(b)[:, 0]))
    for rep in range(2):
        for d, sb, ref in batches:
            out = torch.full_like(d.q[:, 0], float("nan"))
            assert _call_noalloc(d, out, sb, merge=1) == 0
            torch.cuda.synchronize()
            assert int(d.err.item()) == 0
            assert_close(host_f64(out, "bf16"), ref, "bf16", f"{d.b.wl.name} rep {rep}")
