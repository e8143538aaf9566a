"""GPU parity of MLA decode (pkv_mla_append + pkv_mla_decode_attention)
against the float64 MLA oracle (``oracle/mla.py``).  Appends are compared bit
for bit; outputs within the bf16 / f16 tolerances.  Unused cache rows and
blocks are NaN-filled, so a read outside a context shows up as a non-finite
output."""
import numpy as np
import pytest
import torch

import paged_kv_cache_18_gb300 as pkv
from oracle import mla as oracle_mla
from paged_kv_cache_18_gb300 import workloads as W
from tests.gpu_util import assert_close, cache_bits, dev_tensor, host_f64

pytestmark = pytest.mark.gpu

EDGE_LENS = [1, 15, 16, 17, 31, 33, 100, 1000]


class MlaDevice:
    def __init__(self, b: W.MlaBatch, device="cuda:0"):
        dt = b.wl.dtype
        self.b = b
        self.cache = dev_tensor(b.ckv_cache, dt, device)
        self.new = dev_tensor(b.ckv_new, dt, device)
        self.q = dev_tensor(b.q, dt, device)
        self.slots = torch.from_numpy(b.slot_mapping).to(device)
        self.table = torch.from_numpy(b.block_table).to(device)
        self.lens = torch.from_numpy(b.context_lens).to(device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def step(self, **kw):
        pkv.mla_append(self.new, self.cache, self.slots, error_word=self.err)
        return pkv.mla_decode_attention(self.q, self.cache, self.table, self.lens,
                                        self.b.wl.softmax_scale,
                                        max_context_len=self.b.max_context_len,
                                        error_word=self.err, **kw)


def oracle_after_append(b: W.MlaBatch) -> np.ndarray:
    cache = b.ckv_cache.copy()
    bs = b.wl.block_size
    for t, s in enumerate(b.slot_mapping):
        if s >= 0:
            cache[s // bs, s % bs] = b.ckv_new[t]
    return cache, oracle_mla.mla_decode(b.q, cache, b.block_table, b.context_lens,
                                        b.wl.latent_dim, b.wl.softmax_scale, b.wl.dtype)


def run(wl, **kw):
    b = W.make_mla_batch(wl)
    d = MlaDevice(b)
    out = d.step(**kw)
    torch.cuda.synchronize()
    cache_ref, ref = oracle_after_append(b)
    np.testing.assert_array_equal(cache_bits(d.cache), cache_ref)   # the append, bit for bit
    assert int(d.err.item()) == 0
    got = host_f64(out, wl.dtype)
    assert np.isfinite(got).all()
    return assert_close(got, ref, wl.dtype, wl.name)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("rope", [0, 64])
@pytest.mark.parametrize("heads", [16, 32, 128])
def test_mla_edge_lengths(dtype, rope, heads):
    wl = W.MlaWorkload(f"mla {dtype} r{rope} h{heads}", len(EDGE_LENS), heads, rope, dtype,
                       context_lens=EDGE_LENS, seed=1100 + rope + heads)
    run(wl)


@pytest.mark.parametrize("split_blocks", [1, 3, 7, 40])
@pytest.mark.parametrize("rope", [0, 64])
def test_mla_forced_splits(split_blocks, rope):
    wl = W.MlaWorkload(f"mla split {split_blocks}", 5, 16, rope, "bf16",
                       context_lens=[1, 40, 300, 777, 2049], seed=1200 + split_blocks)
    run(wl, split_blocks=split_blocks)


@pytest.mark.parametrize("stages", [3, 4, 5])
def test_mla_ring_depths(stages):
    wl = W.MlaWorkload(f"mla stages {stages}", 6, 32, 64, "bf16", len_range=(1, 1500),
                       seed=1300 + stages)
    run(wl, stages=stages)
    run(wl, stages=stages, split_blocks=5)


def test_mla_scores_growing_along_the_keys():
    """Positive queries and rows whose values rise with the position: every
    few blocks a score passes the lazy reference maximum, forcing rescales."""
    wl = W.MlaWorkload("mla growing", 3, 16, 64, "bf16", context_lens=[64, 500, 1600], seed=1400)
    b = W.make_mla_batch(wl)
    rng = np.random.default_rng(1401)
    q = np.abs(rng.standard_normal(b.q.shape, dtype=np.float32))
    b.q = W.to_storage(q, "bf16")
    for bi, L in enumerate(b.context_lens):
        for i in range(int(L)):
            phys, off = int(b.block_table[bi, i // 16]), i % 16
            row = np.abs(rng.standard_normal(wl.width, dtype=np.float32)) * 0.1 + 0.002 * i
            stored = W.to_storage(row, "bf16")
            if i == L - 1:
                b.ckv_new[bi] = stored      # appended by the step
            else:
                b.ckv_cache[phys, off] = stored
    d = MlaDevice(b)
    out = d.step()
    torch.cuda.synchronize()
    _, ref = oracle_after_append(b)
    assert_close(host_f64(out, "bf16"), ref, "bf16", wl.name)


def test_mla_bad_block_is_recorded_and_ignored():
    wl = W.MlaWorkload("mla bad block", 3, 16, 64, "bf16", context_lens=[40, 100, 70], seed=1500)
    b = W.make_mla_batch(wl)
    d = MlaDevice(b)
    table = d.table.clone()
    table[1, 2] = b.num_blocks + 5          # a block id past the cache
    pkv.mla_append(d.new, d.cache, d.slots)
    out = pkv.mla_decode_attention(d.q, d.cache, table, d.lens, wl.softmax_scale,
                                   max_context_len=b.max_context_len, error_word=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 2           # PKV_DEVERR_BLOCK_ID
    got = host_f64(out, "bf16")
    assert np.isfinite(got).all()
    # the other sequences are exact
    _, ref = oracle_after_append(b)
    assert_close(got[[0, 2]], ref[[0, 2]], "bf16", "others")


def test_mla_empty_sequence_and_empty_batch():
    wl = W.MlaWorkload("mla empty", 3, 16, 0, "bf16", context_lens=[0, 17, 1], seed=1600)
    b = W.make_mla_batch(wl)
    d = MlaDevice(b)
    out = d.step()
    torch.cuda.synchronize()
    got = host_f64(out, "bf16")
    assert not got[0].any()
    _, ref = oracle_after_append(b)
    assert_close(got, ref, "bf16", wl.name)
    e = pkv.mla_decode_attention(d.q[:0], d.cache, d.table[:0], d.lens[:0], 0.1,
                                 max_context_len=0)
    assert e.shape == (0, 16, 512)


def test_mla_rejects_what_it_does_not_build():
    wl = W.MlaWorkload("mla rejects", 2, 16, 64, "bf16", context_lens=[5, 9], seed=1700)
    d = MlaDevice(W.make_mla_batch(wl))
    with pytest.raises(pkv.PkvError):   # 8 heads: not a multiple of 16
        pkv.mla_decode_attention(d.q[:, :8].contiguous(), d.cache, d.table, d.lens, 0.1)
    with pytest.raises(pkv.PkvError):   # ring depth 2 is not built
        pkv.mla_decode_attention(d.q, d.cache, d.table, d.lens, 0.1, stages=2)


def test_mla_step_replays_from_a_cuda_graph():
    wl = W.MlaWorkload("mla graph", 8, 32, 64, "bf16", len_range=(50, 3000), seed=1800)
    b = W.make_mla_batch(wl)
    d = MlaDevice(b)
    ws = torch.empty(max(16, pkv.mla_workspace_size(8, 32, 64, b.max_context_len,
                                                    torch.bfloat16)),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty(8, 32, 512, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d.step(out=out, workspace=ws)       # warm-up (plans, attributes)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        d.step(out=out, workspace=ws)
    _, ref = oracle_after_append(b)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_close(host_f64(out, "bf16"), ref, "bf16", "graph")


def test_mla_full_workload_in_the_bench_configuration():
    wl = W.MLA_WORKLOADS["mla_deepseek_v2"]
    b = W.make_mla_batch(wl)
    d = MlaDevice(b)
    out = d.step()
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    _, ref = oracle_after_append(b)
    max_abs, rel = assert_close(host_f64(out, "bf16"), ref, "bf16", wl.name)
    print(f"{wl.name}: max-abs {max_abs:.3e} rel-L2 {rel:.3e}")
