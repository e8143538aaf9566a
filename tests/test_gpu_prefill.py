"""Chunked prefill on the GPU (pkv_paged_prefill_attention) against the
float64 oracle: each sequence's chunk rows are appended with kv_append, then
every query row attends to its cache up to itself.  The oracle runs per
sequence as causal verification with Q = the chunk length, the definition
the pins tie to PyTorch's float64 causal attention."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_18_gb300 as pkv
from paged_kv_cache_18_gb300 import binding
from paged_kv_cache_18_gb300 import workloads as W
from tests.gpu_util import assert_close, dev_tensor, host_f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


class DevicePrefill:
    def __init__(self, b: W.PrefillBatch):
        dt = b.wl.dtype
        self.b = b
        self.k = dev_tensor(b.k_cache, dt, DEV)
        self.v = dev_tensor(b.v_cache, dt, DEV)
        self.k_new = dev_tensor(b.k_new, dt, DEV)
        self.v_new = dev_tensor(b.v_new, dt, DEV)
        self.q = dev_tensor(b.q, dt, DEV)
        self.slots = torch.from_numpy(b.slot_mapping).to(DEV)
        self.table = torch.from_numpy(b.block_table).to(DEV)
        self.lens = torch.from_numpy(b.context_lens).to(DEV)
        self.qs = torch.from_numpy(b.query_start).to(DEV)
        self.err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def run(self, stages=0, expect_err=0):
        if self.slots.numel():
            pkv.kv_append(self.k_new, self.v_new, self.k, self.v, self.slots, error_word=self.err)
        out = pkv.paged_prefill_attention(self.q, self.k, self.v, self.table, self.lens, self.qs,
                                          max_query_len=self.b.max_query_len,
                                          scale=self.b.wl.softmax_scale, stages=stages,
                                          error_word=self.err)
        assert binding.read_error_word(self.err) == expect_err
        return host_f64(out, self.b.wl.dtype)


def oracle_prefill(b: W.PrefillBatch, rows_per_seq=None, seed=0):
    """Float64 output [total_q, Hq, D] (NaN where not computed)."""
    if not getattr(b, "_appended", False):
        if b.slot_mapping.size:
            oracle.kv_append(b.k_cache, b.v_cache, b.k_new, b.v_new, b.slot_mapping, b.wl.dtype)
        b._appended = True
    Hq, D = b.wl.num_heads, b.wl.head_dim
    out = np.full((b.total_q, Hq, D), np.nan)
    rng = np.random.default_rng(seed)
    for s in range(b.wl.batch):
        q0, q1 = int(b.query_start[s]), int(b.query_start[s + 1])
        if q1 == q0:
            continue
        rows = None
        if rows_per_seq is not None and (q1 - q0) * Hq > rows_per_seq:
            # always the last row's heads (the most keys) and the first row
            pick = set(rng.choice((q1 - q0) * Hq, rows_per_seq, replace=False).tolist())
            pick |= set(range((q1 - q0 - 1) * Hq, (q1 - q0) * Hq)) | set(range(Hq))
            rows = np.array(sorted(pick), dtype=np.int64)
        o = oracle.paged_attention(b.q[q0:q1][None], b.k_cache, b.v_cache,
                                   b.block_table[s:s + 1], b.context_lens[s:s + 1],
                                   b.wl.softmax_scale, b.wl.dtype, rows=rows)
        out[q0:q1] = o[0]
    return out


def check(b, stages=0, rows_per_seq=None, what=""):
    d = DevicePrefill(b)
    got = d.run(stages)
    ref = oracle_prefill(b, rows_per_seq)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    return assert_close(got, ref, b.wl.dtype, what)


RAGGED = dict(chunk_lens=[1, 37, 128, 300], prefix_lens=[0, 17, 200, 5])


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("heads", [(8, 2), (4, 4), (8, 1), (16, 2)])
def test_prefill_ragged(dtype, D, heads):
    wl = W.PrefillWorkload("ragged", 4, heads[0], heads[1], D, dtype, seed=11, **RAGGED)
    check(W.make_prefill_batch(wl), what=f"{dtype} D{D} {heads}")


@pytest.mark.parametrize("chunk", [1, 15, 16, 17, 127, 128, 129, 255, 256, 257, 640])
def test_prefill_from_empty_cache_is_causal_attention(chunk):
    wl = W.PrefillWorkload("causal", 2, 8, 2, 128, "bf16", chunk_lens=[chunk],
                           prefix_lens=[0], seed=12)
    check(W.make_prefill_batch(wl), what=f"chunk {chunk}")


@pytest.mark.parametrize("prefix", [1, 16, 100, 127, 128, 129, 1000, 4000])
def test_prefill_after_a_cached_prefix(prefix):
    wl = W.PrefillWorkload("prefix", 2, 32, 8, 128, "bf16", chunk_lens=[96, 200],
                           prefix_lens=[prefix, prefix + 7], seed=13)
    check(W.make_prefill_batch(wl), rows_per_seq=512, what=f"prefix {prefix}")


@pytest.mark.parametrize("D,stages", [(128, 3), (128, 4), (128, 5), (128, 6), (128, 8), (64, 4),
                                      (64, 8), (64, 12), (64, 16)])
def test_prefill_ring_depths(D, stages):
    wl = W.PrefillWorkload("stages", 3, 8, 2, D, "bf16", chunk_lens=[64, 300, 513],
                           prefix_lens=[700, 0, 260], seed=14)
    check(W.make_prefill_batch(wl), stages=stages, what=f"D{D} stages {stages}")


@pytest.mark.parametrize("group", [1, 2, 4, 8, 16, 32, 64, 128])
def test_prefill_group_sizes(group):
    wl = W.PrefillWorkload("group", 2, group, 1, 64, "bf16", chunk_lens=[33, 70],
                           prefix_lens=[150, 3], seed=15)
    check(W.make_prefill_batch(wl), what=f"group {group}")


def test_prefill_scores_that_keep_growing():
    # keys scaled up along the sequence: the running maximum rises chunk after
    # chunk, so the lazy reference is raised (and O rescaled) many times
    wl = W.PrefillWorkload("growing", 2, 8, 2, 128, "bf16", chunk_lens=[200, 64],
                           prefix_lens=[1500, 900], seed=16)
    b = W.make_prefill_batch(wl)
    bs = wl.block_size
    for s in range(wl.batch):
        for i in range(int(b.context_lens[s]) - int(b.query_start[s + 1] - b.query_start[s])):
            phys, off = int(b.block_table[s, i // bs]), i % bs
            row = W.storage_to_f64(b.k_cache[phys, :, off, :], "bf16") * (1 + i / 60.0)
            b.k_cache[phys, :, off, :] = W.to_storage(row.astype(np.float32), "bf16")
    q = W.storage_to_f64(b.q, "bf16") * 3.0
    b.q[...] = W.to_storage(q.astype(np.float32), "bf16")
    check(b, rows_per_seq=400, what="growing scores")


def test_prefill_chunks_of_uniform_length_match_spec_verify():
    wl = W.PrefillWorkload("uniform", 4, 32, 8, 128, "bf16", chunk_lens=[5],
                           prefix_range=(100, 900), seed=17)
    b = W.make_prefill_batch(wl)
    got = DevicePrefill(b).run()
    ref = oracle_prefill(b)
    assert_close(got, ref, "bf16", "prefill Q=5")
    # the same call through the verification entry point
    d = DevicePrefill(b)
    q4 = d.q.view(wl.batch, 5, wl.num_heads, wl.head_dim)
    out = pkv.spec_verify_attention(q4, d.k, d.v, d.table, d.lens, scale=wl.softmax_scale)
    verify = host_f64(out, "bf16").reshape(got.shape)
    assert_close(verify, ref, "bf16", "verify Q=5")


def test_prefill_skips_and_records_an_inconsistent_sequence():
    wl = W.PrefillWorkload("bad", 3, 8, 2, 128, "bf16", chunk_lens=[40, 50, 60],
                           prefix_lens=[10, 20, 30], seed=18)
    b = W.make_prefill_batch(wl)
    d = DevicePrefill(b)
    pkv.kv_append(d.k_new, d.v_new, d.k, d.v, d.slots)
    d.lens[1] = 10                        # fewer cached rows than the chunk's 50
    out = torch.full_like(d.q, float("nan"))
    pkv.paged_prefill_attention(d.q, d.k, d.v, d.table, d.lens, d.qs, max_query_len=60,
                                scale=wl.softmax_scale, out=out, error_word=d.err)
    assert binding.read_error_word(d.err) == 3          # PKV_DEVERR_CONTEXT_LEN
    got = host_f64(out, "bf16")
    ref = oracle_prefill(b)
    q0, q1 = int(b.query_start[1]), int(b.query_start[2])
    assert np.isnan(got[q0:q1]).all()                   # not written
    keep = np.r_[0:q0, q1:b.total_q]
    assert_close(got[keep], ref[keep], "bf16", "other sequences")


def test_prefill_records_a_bad_block_and_stays_finite():
    wl = W.PrefillWorkload("badblock", 2, 8, 2, 128, "bf16", chunk_lens=[40, 60],
                           prefix_lens=[300, 20], seed=19)
    b = W.make_prefill_batch(wl)
    d = DevicePrefill(b)
    pkv.kv_append(d.k_new, d.v_new, d.k, d.v, d.slots)
    d.table[0, 3] = b.num_blocks + 5      # a prefix block of sequence 0
    out = pkv.paged_prefill_attention(d.q, d.k, d.v, d.table, d.lens, d.qs, max_query_len=60,
                                      scale=wl.softmax_scale, error_word=d.err)
    assert binding.read_error_word(d.err) == 2          # PKV_DEVERR_BLOCK_ID
    got = host_f64(out, "bf16")
    assert np.isfinite(got).all()
    ref = oracle_prefill(b)
    q0 = int(b.query_start[1])
    assert_close(got[q0:], ref[q0:], "bf16", "the other sequence")


def test_prefill_empty_calls_and_zero_length_chunks():
    wl = W.PrefillWorkload("zeros", 3, 8, 2, 128, "bf16", chunk_lens=[0, 20, 0],
                           prefix_lens=[50, 5, 0], seed=20)
    check(W.make_prefill_batch(wl), what="zero-length chunks")
    d = DevicePrefill(W.make_prefill_batch(wl))
    empty_q = d.q[:0]
    pkv.paged_prefill_attention(empty_q, d.k, d.v, d.table, d.lens, torch.zeros_like(d.qs),
                                max_query_len=0)


def test_prefill_rejects_what_it_does_not_run():
    wl = W.PrefillWorkload("rej", 1, 6, 2, 128, "bf16", chunk_lens=[8], prefix_lens=[0])
    d = DevicePrefill(W.make_prefill_batch(wl))   # group 3 does not divide 128
    with pytest.raises(binding.PkvError):
        pkv.paged_prefill_attention(d.q, d.k, d.v, d.table, d.lens, d.qs, max_query_len=8)
    wl = W.PrefillWorkload("rej", 1, 8, 2, 128, "bf16", chunk_lens=[8], prefix_lens=[0])
    d = DevicePrefill(W.make_prefill_batch(wl))   # the scale must be finite
    for bad in (float("nan"), float("inf")):
        with pytest.raises(binding.PkvError):
            pkv.paged_prefill_attention(d.q, d.k, d.v, d.table, d.lens, d.qs, max_query_len=8,
                                        scale=bad)
    # zero or below: the library's default 1/sqrt(head_dim), bitwise
    pkv.kv_append(d.k_new, d.v_new, d.k, d.v, d.slots)
    outs = [pkv.paged_prefill_attention(d.q, d.k, d.v, d.table, d.lens, d.qs, max_query_len=8,
                                        scale=s).clone()
            for s in (float(np.float32(1 / np.sqrt(128))), 0.0, -0.1)]
    assert torch.isfinite(outs[0].float()).all()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    wl = W.PrefillWorkload("rej", 1, 8, 2, 256, "bf16", chunk_lens=[8], prefix_lens=[0])
    d = DevicePrefill(W.make_prefill_batch(wl))   # head_dim 256
    with pytest.raises(binding.PkvError):
        pkv.paged_prefill_attention(d.q, d.k, d.v, d.table, d.lens, d.qs, max_query_len=8)


def test_prefill_full_size_workload():
    wl = W.PREFILL_WORKLOADS["prefill_llama3_8b"]
    check(W.make_prefill_batch(wl), what=wl.name)   # every (position, head) row


def test_prefill_step_replays_from_a_cuda_graph():
    # the append and the prefill call capture into one graph (no host sync,
    # no allocation inside the calls) and replay to the same result
    wl = W.PrefillWorkload("graph", 3, 32, 8, 128, "bf16", chunk_lens=[64, 300, 17],
                           prefix_lens=[500, 40, 1200], seed=21)
    b = W.make_prefill_batch(wl)
    d = DevicePrefill(b)
    out = torch.empty_like(d.q)

    def step():
        pkv.kv_append(d.k_new, d.v_new, d.k, d.v, d.slots, error_word=d.err)
        pkv.paged_prefill_attention(d.q, d.k, d.v, d.table, d.lens, d.qs,
                                    max_query_len=b.max_query_len, scale=wl.softmax_scale,
                                    out=out, error_word=d.err)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up: kernel attributes are set outside the capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    ref = oracle_prefill(b, rows_per_seq=256)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_close(host_f64(out, "bf16"), ref, "bf16", "graph replay")
    assert binding.read_error_word(d.err) == 0
