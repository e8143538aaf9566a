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


def _call_noalloc(d, out, split_blocks):
    b, wl = d.b, d.b.wl
    L = binding.lib()
    opts = binding.Options(0, split_blocks)
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
    # rejected before anything is enqueued: no pointer is touched
    st = L.pkv_paged_decode_attention_noalloc(16, 16, 16, 16, 16, 2500, 16, 40000, 64, 32, 8,
                                              128, 16, 100000, 0.1, 1, ctypes.byref(opts), None,
                                              None)
    assert st == 3  # PKV_ERR_WORKSPACE
