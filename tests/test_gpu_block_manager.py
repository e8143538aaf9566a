"""Copy-on-write and prefix sharing on the GPU.

``copy_blocks`` is checked byte for byte against a host copy.  Then the
native block manager drives whole decode loops: its slots feed ``kv_append``,
its copy pairs feed ``copy_blocks``, and its block tables feed the attention
calls, whose output must match the float64 oracle run on each sequence's
logical rows laid out contiguously (a table the manager never saw).  Every
K/V row is a function of the token prefix it belongs to, as a model's would
be, so a block shared through a fork or a prefix-cache hit holds the right
rows only if the bookkeeping is right; unwritten cache rows are NaN.
"""
import math

import numpy as np
import pytest
import torch

from oracle import twin
import paged_kv_cache_18_gb300 as pkv
from paged_kv_cache_18_gb300 import binding
from paged_kv_cache_18_gb300 import workloads as W
from tests.gpu_util import assert_close, dev_tensor, host_f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


# --- copy_blocks ------------------------------------------------------------------
@pytest.mark.parametrize("dtype,Hkv,D", [(torch.bfloat16, 2, 128), (torch.float16, 1, 64),
                                         (torch.float32, 4, 128), (torch.uint8, 1, 64),
                                         (torch.uint8, 8, 256)])
def test_copy_blocks_is_a_byte_copy(dtype, Hkv, D):
    NB, bs = 96, 16
    rng = np.random.default_rng(7)
    esize = torch.tensor([], dtype=dtype).element_size()
    shape = (NB, Hkv, bs, D)
    kb = rng.integers(0, 256, NB * Hkv * bs * D * esize, dtype=np.uint8)
    vb = rng.integers(0, 256, kb.size, dtype=np.uint8)
    k = torch.from_numpy(kb.copy()).to(DEV).view(dtype).view(shape)
    v = torch.from_numpy(vb.copy()).to(DEV).view(dtype).view(shape)
    src = rng.choice(48, 37, replace=True).astype(np.int32)
    dst = (48 + rng.permutation(48)[:37]).astype(np.int32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.copy_blocks(k, v, src, dst, error_word=err)
    blk = kb.size // NB
    ek, ev = kb.reshape(NB, blk).copy(), vb.reshape(NB, blk).copy()
    ek[dst], ev[dst] = ek[src], ev[src]
    assert np.array_equal(k.view(torch.uint8).cpu().numpy().reshape(NB, blk), ek)
    assert np.array_equal(v.view(torch.uint8).cpu().numpy().reshape(NB, blk), ev)
    assert binding.read_error_word(err) == 0


def test_copy_blocks_skips_and_records_out_of_range_ids():
    NB, bs, Hkv, D = 8, 16, 2, 64
    k = torch.randn(NB, Hkv, bs, D, device=DEV).to(torch.bfloat16)
    v = torch.randn(NB, Hkv, bs, D, device=DEV).to(torch.bfloat16)
    k0, v0 = k.clone(), v.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.copy_blocks(k, v, [0, 99, 3, -1], [1, 2, NB, 4], error_word=err)
    assert binding.read_error_word(err) == 2          # PKV_DEVERR_BLOCK_ID
    assert torch.equal(k[1], k0[0]) and torch.equal(v[1], v0[0])
    for b in (0, 2, 3, 4, 5, 6, 7):
        assert torch.equal(k[b], k0[b]) and torch.equal(v[b], v0[b])


def test_copy_blocks_of_nothing_is_a_no_op():
    k = torch.zeros(4, 1, 16, 64, dtype=torch.bfloat16, device=DEV)
    pkv.copy_blocks(k, k.clone(), [], [])


# --- the manager driving decode -----------------------------------------------------
class Engine:
    """A toy serving loop over one paged cache, driven by the native manager."""

    def __init__(self, num_blocks, Hq=8, Hkv=2, D=128, bs=16):
        self.bs, self.Hq, self.Hkv, self.D = bs, Hq, Hkv, D
        self.mgr = pkv.BlockManager(num_blocks, bs)
        shape = (num_blocks, Hkv, bs, D)
        self.k = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=DEV)
        self.v = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=DEV)
        self.err = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.tokens = {}
        self._rows = {}
        self.rng = np.random.default_rng(11)

    def rows(self, prefix):
        """(k, v) bf16 bit patterns [Hkv, D] of the last token of `prefix`."""
        key = tuple(prefix)
        if key not in self._rows:
            g = np.random.default_rng(list(key))
            kv = g.standard_normal((2, self.Hkv, self.D), dtype=np.float32)
            self._rows[key] = W.to_storage(kv, "bf16")
        return self._rows[key]

    def _write(self, sid, first, slots):
        toks = self.tokens[sid]
        kb = np.stack([self.rows(toks[:p + 1])[0] for p in range(first, len(toks))])
        vb = np.stack([self.rows(toks[:p + 1])[1] for p in range(first, len(toks))])
        assert len(slots) == len(kb)
        pkv.kv_append(dev_tensor(kb, "bf16", DEV), dev_tensor(vb, "bf16", DEV), self.k, self.v,
                      torch.from_numpy(np.asarray(slots, dtype=np.int64)).to(DEV),
                      error_word=self.err)

    def add(self, sid, prompt):
        cached, slots = self.mgr.add_sequence(sid, prompt)
        self.tokens[sid] = list(prompt)
        if len(slots):
            self._write(sid, cached, slots)
        return cached

    def append(self, sid, new):
        slots, copies = self.mgr.append(sid, new)
        for src, dst in copies:
            pkv.copy_blocks(self.k, self.v, [src], [dst], error_word=self.err)
        first = len(self.tokens[sid])
        self.tokens[sid] += list(new)
        self._write(sid, first, slots)
        return copies

    def fork(self, parent, child):
        self.mgr.fork(parent, child)
        self.tokens[child] = list(self.tokens[parent])

    def free(self, sid):
        self.mgr.free(sid)
        del self.tokens[sid]

    def check_attention(self, sids, num_queries=1):
        table, lens = self.mgr.block_table(sids)
        assert lens.tolist() == [len(self.tokens[s]) for s in sids]
        B, D = len(sids), self.D
        qbits = W.to_storage(self.rng.standard_normal((B, num_queries, self.Hq, D),
                                                      dtype=np.float32), "bf16")
        q = dev_tensor(qbits, "bf16", DEV)
        tab = torch.from_numpy(table).to(DEV)
        ln = torch.from_numpy(lens).to(DEV)
        scale = 1.0 / math.sqrt(D)
        if num_queries == 1:
            out = pkv.paged_decode_attention(q[:, 0], self.k, self.v, tab, ln, scale=scale,
                                             max_context_len=int(lens.max()),
                                             error_word=self.err)[:, None]
        else:
            out = pkv.spec_verify_attention(q, self.k, self.v, tab, ln, scale=scale,
                                            max_context_len=int(lens.max()),
                                            error_word=self.err)
        assert binding.read_error_word(self.err) == 0
        assert_close(host_f64(out, "bf16"), self.reference(sids, qbits), "bf16",
                     f"sequences {sids}")

    def reference(self, sids, qbits):
        """The oracle over each sequence's rows, laid out block after block."""
        bs = self.bs
        blocks_k, blocks_v, table, lens = [], [], [], []
        width = max(-(-len(self.tokens[s]) // bs) for s in sids)
        for s in sids:
            toks = self.tokens[s]
            rows = [self.rows(toks[:p + 1]) for p in range(len(toks))]
            nb = -(-len(toks) // bs)
            pad = [np.zeros((2, self.Hkv, self.D), np.uint16)] * (nb * bs - len(toks))
            dense = np.stack(rows + pad).reshape(nb, bs, 2, self.Hkv, self.D)
            first = len(blocks_k)
            blocks_k += list(dense[:, :, 0].transpose(0, 2, 1, 3))
            blocks_v += list(dense[:, :, 1].transpose(0, 2, 1, 3))
            table.append(list(range(first, first + nb)) + [0] * (width - nb))
            lens.append(len(toks))
        return twin.contiguous_attention(qbits, np.stack(blocks_k), np.stack(blocks_v),
                                         np.asarray(table, np.int32), np.asarray(lens, np.int32),
                                         1.0 / math.sqrt(self.D), "bf16")


def test_parallel_sampling_with_copy_on_write():
    e = Engine(64)
    prompt = e.rng.integers(0, 1000, 40).tolist()
    assert e.add(0, prompt) == 0
    for child in (1, 2, 3):
        e.fork(0, child)
    e.free(0)
    copies = 0
    for step in range(20):
        for s in (1, 2, 3):
            copies += len(e.append(s, [int(e.rng.integers(0, 1000))]))
        if step % 4 == 0 or step == 19:
            e.check_attention([1, 2, 3])
    assert copies == 2            # two samples copied the shared tail; the last wrote in place
    # the two full prompt blocks are still shared by all three samples
    assert [e.mgr.block_info(b)[0] for b in e.mgr.sequence(1)[0][:2]] == [3, 3]


def test_prefix_cache_hit_serves_the_shared_rows():
    e = Engine(64)
    a = e.rng.integers(0, 1000, 50).tolist()
    e.add(0, a)
    e.check_attention([0])
    e.free(0)                                          # its blocks stay cached
    b = a[:48] + e.rng.integers(0, 1000, 7).tolist()
    assert e.add(1, b) == 48                           # three full blocks reused
    c = a[:16] + e.rng.integers(0, 1000, 30).tolist()
    assert e.add(2, c) == 16
    for _ in range(5):
        for s in (1, 2):
            e.append(s, [int(e.rng.integers(0, 1000))])
    e.check_attention([1, 2])
    # speculative verification of four tokens through the manager's table
    e.append(1, e.rng.integers(0, 1000, 4).tolist())
    e.append(2, e.rng.integers(0, 1000, 4).tolist())
    e.check_attention([1, 2], num_queries=4)


def test_eviction_under_memory_pressure_keeps_live_rows_intact():
    e = Engine(12, Hq=4, Hkv=1, D=64)
    rng = np.random.default_rng(5)
    live = []
    for sid in range(12):
        prompt = rng.integers(0, 3, int(rng.integers(1, 40))).tolist()
        try:
            e.add(sid, prompt)
            live.append(sid)
        except binding.PkvError:
            pass                                       # the pool is full: nothing changed
        if len(live) > 2:
            e.free(live.pop(0))
        for s in live:
            try:
                e.append(s, [int(rng.integers(0, 3))])
            except binding.PkvError:
                pass
        if live:
            e.check_attention(live)


def test_copy_on_write_and_decode_replay_from_a_cuda_graph():
    # a decode step whose slots and copy pairs came from the manager: the
    # block copy, the append and the attention capture into one graph
    e = Engine(32)
    prompt = e.rng.integers(0, 1000, 24).tolist()
    e.add(0, prompt)
    e.fork(0, 1)
    token = 7
    slots, copies = e.mgr.append(1, [token])
    assert len(copies) == 1
    e.tokens[1] = e.tokens[1] + [token]
    toks = e.tokens[1]
    kb, vb = e.rows(toks)
    k_new = dev_tensor(kb[None], "bf16", DEV)
    v_new = dev_tensor(vb[None], "bf16", DEV)
    slot_t = torch.from_numpy(np.asarray(slots, dtype=np.int64)).to(DEV)
    src = torch.tensor([copies[0][0]], dtype=torch.int32, device=DEV)
    dst = torch.tensor([copies[0][1]], dtype=torch.int32, device=DEV)
    table, lens = e.mgr.block_table([0, 1])
    tab, ln = torch.from_numpy(table).to(DEV), torch.from_numpy(lens).to(DEV)
    q = dev_tensor(W.to_storage(e.rng.standard_normal((2, 1, e.Hq, e.D), dtype=np.float32),
                                "bf16"), "bf16", DEV)
    out = torch.empty(2, e.Hq, e.D, dtype=torch.bfloat16, device=DEV)

    def step():
        pkv.copy_blocks(e.k, e.v, src, dst, error_word=e.err)
        pkv.kv_append(k_new, v_new, e.k, e.v, slot_t, error_word=e.err)
        pkv.paged_decode_attention(q[:, 0], e.k, e.v, tab, ln, scale=1.0 / math.sqrt(e.D),
                                   max_context_len=int(lens.max()), out=out,
                                   error_word=e.err)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    qbits = q.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = e.reference([0, 1], qbits)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_close(host_f64(out, "bf16")[:, None], ref, "bf16", "graph replay")
    assert binding.read_error_word(e.err) == 0
