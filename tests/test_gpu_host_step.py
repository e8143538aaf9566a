"""The host-buffer step (pkv_append_attention_host): inputs and output in
host memory.  Page-locked (pinned, mapped) buffers are read and written by
the kernels in place; pageable ones are copied in and out around the fused
append + attention on the caller's stream.  Either way the output must
equal the oracle within tolerance, the cache writes must be bit-exact, and
the result must be exactly what the same launch gives on device copies of
the inputs."""
import numpy as np
import pytest
import torch

import paged_kv_cache_18_gb300 as pkv
from paged_kv_cache_18_gb300 import workloads as W
from tests.gpu_util import DeviceBatch, assert_close, cache_bits, host_f64, oracle_after_append

pytestmark = pytest.mark.gpu


def pinned(t: torch.Tensor) -> torch.Tensor:
    return t.cpu().pin_memory()


def host_inputs(d: DeviceBatch, Q: int):
    """Pinned host copies of the step's inputs, in the fused call's layouts."""
    wl = d.b.wl
    B, Hkv, D = wl.batch, wl.num_kv_heads, wl.head_dim
    q = d.q if Q > 1 else d.q[:, 0]
    return dict(q=pinned(q), k_new=pinned(d.k_new.view(B, Q, Hkv, D)),
                v_new=pinned(d.v_new.view(B, Q, Hkv, D)), table=pinned(d.table),
                lens=pinned(d.lens))


def staging_for(b: W.PagedBatch, Q: int, split_blocks=0, kernel=0) -> torch.Tensor:
    wl = b.wl
    n = pkv.host_step_staging_size(wl.batch, Q, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                   b.block_table.shape[1], b.max_context_len,
                                   {"bf16": torch.bfloat16, "f16": torch.float16,
                                    "f32": torch.float32}[wl.dtype],
                                   kernel=kernel, split_blocks=split_blocks)
    return torch.empty(n, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("dtype,kernel", [("bf16", 0), ("f16", 0), ("f32", 0), ("bf16", 1)])
@pytest.mark.parametrize("Q,Hq,Hkv", [(1, 8, 2), (1, 40, 40), (5, 32, 8)])
@pytest.mark.parametrize("split_blocks", [0, 3])
def test_host_step_matches_oracle_and_device_call(dtype, kernel, Q, Hq, Hkv, split_blocks):
    lens = [max(1, Q - 1), Q, 16, 17, 33, 250, 1000]
    D = 128 if dtype != "f32" else 64
    wl = W.Workload(f"host step {dtype} Q{Q} {Hq}/{Hkv}", len(lens), Hq, Hkv, D, dtype,
                    context_lens=lens, num_queries=Q, seed=900 + Q + Hq + split_blocks)
    b = W.make_batch(wl)
    d_host, d_dev = DeviceBatch(b), DeviceBatch(b)
    h = host_inputs(d_host, Q)
    out = torch.full_like(h["q"], float("nan")).pin_memory()
    staging = staging_for(b, Q, split_blocks, kernel)
    pkv.append_attention_host(h["q"], h["k_new"], h["v_new"], d_host.k_cache, d_host.v_cache,
                              h["table"], h["lens"], out, staging, b.max_context_len,
                              scale=wl.softmax_scale, kernel=kernel, split_blocks=split_blocks,
                              error_word=d_host.err)
    torch.cuda.current_stream().synchronize()
    assert int(d_host.err.item()) == 0
    # the same launch on device-resident inputs
    B = wl.batch
    ref_dev = pkv.append_attention(d_dev.q if Q > 1 else d_dev.q[:, 0],
                                   d_dev.k_new.view(B, Q, Hkv, D),
                                   d_dev.v_new.view(B, Q, Hkv, D), d_dev.k_cache, d_dev.v_cache,
                                   d_dev.table, d_dev.lens, scale=wl.softmax_scale,
                                   max_context_len=b.max_context_len, kernel=kernel,
                                   split_blocks=split_blocks)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_dev.cpu())
    for a, c in ((d_host.k_cache, d_dev.k_cache), (d_host.v_cache, d_dev.v_cache)):
        np.testing.assert_array_equal(cache_bits(a), cache_bits(c))
    # and against the oracle
    ref = oracle_after_append(b)
    bits = cache_bits(d_host.k_cache)
    np.testing.assert_array_equal(bits, b.k_cache.view(bits.dtype))
    got = host_f64(out if Q > 1 else out[:, None], dtype)
    assert_close(got, ref, dtype, wl.name)


def test_host_steps_in_sequence_reuse_one_staging_buffer():
    """Two steps back to back on one stream and one staging buffer: the second
    step's copies wait for the first step's launch (stream order), so both
    outputs are right."""
    wl = W.Workload("host steps", 6, 32, 8, 128, "bf16", len_range=(40, 900), seed=931)
    b1 = W.make_batch(wl)
    wl2 = W.Workload("host steps 2", 6, 32, 8, 128, "bf16", len_range=(40, 900), seed=932)
    b2 = W.make_batch(wl2)
    outs = []
    d1, d2 = DeviceBatch(b1), DeviceBatch(b2)
    staging = max((staging_for(b1, 1), staging_for(b2, 1)), key=lambda t: t.numel())
    for d, b in ((d1, b1), (d2, b2)):
        h = host_inputs(d, 1)
        out = torch.empty_like(h["q"]).pin_memory()
        pkv.append_attention_host(h["q"], h["k_new"], h["v_new"], d.k_cache, d.v_cache,
                                  h["table"], h["lens"], out, staging, b.max_context_len,
                                  scale=b.wl.softmax_scale)
        outs.append((out, b))
    torch.cuda.current_stream().synchronize()
    for out, b in outs:
        assert_close(host_f64(out[:, None], "bf16"), oracle_after_append(b), "bf16", b.wl.name)


def test_host_step_small_staging_is_rejected_before_any_copy():
    wl = W.Workload("host step small", 4, 32, 8, 128, "bf16", len_range=(40, 300), seed=933)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    h = host_inputs(d, 1)
    out = torch.full_like(h["q"], 7.0).pin_memory()
    staging = staging_for(b, 1)
    small = staging[: staging.numel() - 256]
    before = cache_bits(d.k_cache).copy()
    with pytest.raises(pkv.PkvError) as e:
        pkv.append_attention_host(h["q"], h["k_new"], h["v_new"], d.k_cache, d.v_cache,
                                  h["table"], h["lens"], out, small, b.max_context_len)
    assert e.value.status == 3  # PKV_ERR_WORKSPACE
    # head_dim the kernels do not build: rejected before any copy as well
    with pytest.raises(pkv.PkvError):
        pkv.binding._check("pkv_append_attention_host", pkv.binding.lib().pkv_append_attention_host(
            out.data_ptr(), h["q"].data_ptr(), h["k_new"].data_ptr(), h["v_new"].data_ptr(),
            d.k_cache.data_ptr(), d.v_cache.data_ptr(), h["table"].data_ptr(),
            h["table"].shape[1], h["lens"].data_ptr(), b.max_context_len, 4, 1, 32, 8, 96, 16,
            d.k_cache.shape[0], 0.1, 1, staging.data_ptr(), staging.numel(), None, None,
            pkv.binding._stream(d.k_cache)))
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    np.testing.assert_array_equal(cache_bits(d.k_cache), before)


@pytest.mark.parametrize("pinned_mask", [0b000000, 0b101010, 0b010101, 0b111110])
def test_host_step_pageable_and_mixed_buffers(pinned_mask):
    """Bit k of pinned_mask: buffer k of (q, k_new, v_new, table, lens, out)
    is page-locked (read or written in place), else pageable (staged)."""
    Q = 5
    wl = W.Workload("host step mixed", 5, 32, 8, 128, "bf16", context_lens=[5, 17, 90, 700, 3000],
                    num_queries=Q, seed=940 + pinned_mask)
    b = W.make_batch(wl)
    d_host, d_dev = DeviceBatch(b), DeviceBatch(b)
    h = host_inputs(d_host, Q)
    names = ["q", "k_new", "v_new", "table", "lens"]
    for k, n in enumerate(names):
        if not (pinned_mask >> k) & 1:
            h[n] = h[n].clone()           # a pageable copy
            assert not h[n].is_pinned()
    out = torch.full_like(h["q"], float("nan"))
    if (pinned_mask >> 5) & 1:
        out = out.pin_memory()
    staging = staging_for(b, Q)
    pkv.append_attention_host(h["q"], h["k_new"], h["v_new"], d_host.k_cache, d_host.v_cache,
                              h["table"], h["lens"], out, staging, b.max_context_len,
                              error_word=d_host.err)
    torch.cuda.current_stream().synchronize()
    assert int(d_host.err.item()) == 0
    ref_dev = pkv.append_attention(d_dev.q, d_dev.k_new.view(5, Q, 8, 128),
                                   d_dev.v_new.view(5, Q, 8, 128), d_dev.k_cache, d_dev.v_cache,
                                   d_dev.table, d_dev.lens, max_context_len=b.max_context_len)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_dev.cpu())
    for a, c in ((d_host.k_cache, d_dev.k_cache), (d_host.v_cache, d_dev.v_cache)):
        np.testing.assert_array_equal(cache_bits(a), cache_bits(c))
    assert_close(host_f64(out, "bf16"), oracle_after_append(b), "bf16", wl.name)
