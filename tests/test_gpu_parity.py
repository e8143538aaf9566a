"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Appends are compared bit for bit over the whole cache; attention outputs
within the tolerances of ``gpu_util.TOL``.  Unused cache rows and blocks are
NaN-filled by the workload generator, so any read outside a context shows up
as a non-finite output.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_18_gb300 import workloads as W
from tests.gpu_util import (DeviceBatch, assert_close, cache_bits, errors, host_f64, tuning,
                            oracle_after_append)

pytestmark = pytest.mark.gpu

EDGE_LENS = [1, 15, 16, 17, 31, 32, 33, 100]


def run_case(wl, kernel=0, split_blocks=0, stages=0, warp_tiles=0, blocks_per_iter=0):
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    with tuning(warp_tiles=warp_tiles, blocks_per_iter=blocks_per_iter):
        out = d.attend(kernel=kernel, split_blocks=split_blocks, stages=stages)
    torch.cuda.synchronize()
    ref = oracle_after_append(b)
    # the append is bit-exact over the whole cache
    np.testing.assert_array_equal(cache_bits(d.k_cache), b.k_cache.view(cache_bits(d.k_cache).dtype))
    np.testing.assert_array_equal(cache_bits(d.v_cache), b.v_cache.view(cache_bits(d.v_cache).dtype))
    got = host_f64(out, wl.dtype)
    assert int(d.err.item()) == 0
    return assert_close(got, ref, wl.dtype, wl.name)


KERNELS = {"simt": 1, "mma": 2}


@pytest.mark.parametrize("dtype,kernel", [("f32", "simt"), ("bf16", "simt"), ("bf16", "mma"),
                                          ("f16", "simt"), ("f16", "mma")])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (8, 1), (16, 2)])
def test_decode_edge_lengths(dtype, kernel, D, Hq, Hkv):
    wl = W.Workload(f"decode {dtype} {kernel} D{D} {Hq}/{Hkv}", len(EDGE_LENS), Hq, Hkv, D,
                    dtype, context_lens=EDGE_LENS, seed=100 + D + Hq + Hkv)
    run_case(wl, kernel=KERNELS[kernel])


@pytest.mark.parametrize("dtype,kernel", [("f32", "simt"), ("bf16", "simt"), ("bf16", "mma"),
                                          ("f16", "mma")])
@pytest.mark.parametrize("Q,Hq,Hkv", [(5, 32, 8), (3, 4, 4), (8, 16, 2), (2, 8, 1)])
@pytest.mark.parametrize("D", [64, 128])
def test_spec_verify_edge_lengths(dtype, kernel, Q, Hq, Hkv, D):
    lens = [Q, Q + 1, 15, 16, 17, 33, 64, 131]
    wl = W.Workload(f"verify {dtype} {kernel} Q{Q} {Hq}/{Hkv} D{D}", len(lens), Hq, Hkv, D,
                    dtype, context_lens=lens, num_queries=Q, seed=200 + Q + Hq + D)
    run_case(wl, kernel=KERNELS[kernel])


@pytest.mark.parametrize("kernel", ["simt", "mma"])
@pytest.mark.parametrize("split_blocks", [1, 2, 3, 7, 64])
def test_forced_splits(kernel, split_blocks):
    wl = W.Workload(f"split {split_blocks}", 5, 16, 4, 128, "bf16",
                    context_lens=[1, 40, 300, 777, 1024], seed=300 + split_blocks)
    run_case(wl, kernel=KERNELS[kernel], split_blocks=split_blocks)


@pytest.mark.parametrize("split_blocks", [1, 5])
def test_forced_splits_verify(split_blocks):
    wl = W.Workload("split verify", 4, 32, 8, 128, "bf16", context_lens=[5, 17, 21, 500],
                    num_queries=5, seed=320 + split_blocks)
    run_case(wl, kernel=2, split_blocks=split_blocks)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Q,Hq,Hkv", [(1, 32, 8), (5, 32, 8), (1, 8, 1), (2, 8, 1)])
def test_mma_stage_depths(D, Q, Hq, Hkv):
    import paged_kv_cache_18_gb300 as pkv
    lens = [Q, 16, 17, 50, 257, 1000]
    accepted = []
    for stages in (1, 2, 3, 4, 6):
        try:
            pkv.plan(len(lens), Q, Hq, Hkv, D, max(lens), torch.bfloat16, kernel=2, stages=stages)
        except pkv.PkvError:
            continue
        accepted.append(stages)
        wl = W.Workload(f"stages {stages} D{D} Q{Q}", len(lens), Hq, Hkv, D, "bf16",
                        context_lens=lens, num_queries=Q, seed=400 + D + stages + Q)
        run_case(wl, kernel=2, stages=stages)
    assert len(accepted) == 2, accepted  # a shallow and a deep ring per tile shape


def test_zero_and_short_contexts_give_zero_rows():
    wl = W.Workload("zero", 3, 8, 2, 128, "bf16", context_lens=[0, 2, 40], num_queries=3, seed=7)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    for kernel in (1, 2):
        got = host_f64(d.attend(kernel=kernel), "bf16")
        assert (got[0] == 0).all() and (got[1, 0] == 0).all()
        assert_close(got, oracle_after_append(b), "bf16", "zero")


def test_split_invariance_and_determinism():
    wl = W.Workload("inv", 4, 32, 8, 128, "bf16", context_lens=[100, 900, 2000, 33], seed=8)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    ref = oracle_after_append(b)
    outs = {}
    for sb in (0, 1, 4, 1000):
        o1 = d.attend(split_blocks=sb).clone()
        o2 = d.attend(split_blocks=sb)
        assert torch.equal(o1, o2), "same inputs, same plan: bitwise identical"
        outs[sb] = host_f64(o1, "bf16")
        assert_close(outs[sb], ref, "bf16", f"split {sb}")
    # different partitions agree to within the output rounding
    for sb in (1, 4, 1000):
        assert np.abs(outs[sb] - outs[0]).max() <= 2 ** -7


def test_spec_rows_match_decode_on_prefixes():
    wl = W.Workload("prefix", 3, 32, 8, 128, "bf16", context_lens=[20, 300, 1111],
                    num_queries=5, seed=9)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    spec = host_f64(d.attend(), "bf16")
    for j in range(5):
        lens = (d.lens - 5 + 1 + j).contiguous()
        import paged_kv_cache_18_gb300 as pkv
        dec = pkv.paged_decode_attention(d.q[:, j].contiguous(), d.k_cache, d.v_cache, d.table,
                                         lens, max_context_len=b.max_context_len)
        got = host_f64(dec, "bf16")
        assert np.abs(got - spec[:, j]).max() <= 2 ** -7


def test_error_word_bad_block_and_long_context():
    wl = W.Workload("bad", 2, 8, 2, 64, "bf16", context_lens=[40, 50], seed=10)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    for kernel in (1, 2):
        d.err.zero_()
        d.table[0, 1] = b.num_blocks + 5   # out of range: skipped and reported
        out = d.attend(kernel=kernel)
        torch.cuda.synchronize()
        assert int(d.err.item()) == 2
        assert torch.isfinite(out.float()).all()
        d.table[0, 1] = int(b.block_table[0, 1])
        d.err.zero_()
        d.lens[1] = 60                      # beyond max_context_len = 50: clamped, reported
        out = d.attend(kernel=kernel)
        torch.cuda.synchronize()
        assert int(d.err.item()) == 3
        d.lens[1] = 50
    d.err.zero_()
    d.attend()
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0


def test_kv_append_skips_padding_and_reports_bad_slots():
    wl = W.Workload("slots", 4, 4, 4, 128, "bf16", context_lens=[3, 20, 16, 1], seed=11)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    before = cache_bits(d.k_cache).copy()
    d.slots[1] = -1
    d.slots[2] = b.num_blocks * 16 + 3
    d.append()
    torch.cuda.synchronize()
    assert int(d.err.item()) == 1
    after = cache_bits(d.k_cache)
    for t in (1, 2):
        s = int(b.slot_mapping[t])
        np.testing.assert_array_equal(after[s // 16, :, s % 16], before[s // 16, :, s % 16])
    for t in (0, 3):
        s = int(b.slot_mapping[t])
        np.testing.assert_array_equal(after[s // 16, :, s % 16], b.k_new[t])


@pytest.mark.parametrize("merge", [0, 1, 2])
def test_cuda_graph_replay(merge):
    """Capture and replay; merge 1 is the last CTA's in-kernel merge, 2 the
    merge kernel launched as a programmatic dependent of the attention."""
    wl = W.Workload("graph", 8, 32, 8, 128, "bf16", len_range=(100, 3000), seed=12)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    import paged_kv_cache_18_gb300 as pkv
    with tuning(merge=merge):
        ws_bytes = pkv.workspace_size(8, 1, 32, 8, 128, b.max_context_len, torch.bfloat16)
        assert pkv.plan(8, 1, 32, 8, 128, b.max_context_len, torch.bfloat16)["num_splits"] > 1
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
        out = torch.empty(8, 1, 32, 128, dtype=torch.bfloat16, device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            d.append()
            d.attend(out=out[:, 0], workspace=ws)   # warm-up (plans, attributes)
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            d.append()
            d.attend(out=out[:, 0], workspace=ws)
    ref = oracle_after_append(b)
    for _ in range(3):  # replays reuse the captured call's merge counters
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_close(host_f64(out, "bf16"), ref, "bf16", "graph")


# ---- the five named workloads at full size, in the bench's launch config --
# Every output row is compared with the oracle (all sequences, queries and
# heads), not a sample.
@pytest.mark.slow
@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_named_workload_full_size(name):
    wl = W.WORKLOADS[name]
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    out = d.attend()
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    ref = oracle_after_append(b)
    # bit-exact append over the whole cache
    k_bits = cache_bits(d.k_cache)
    assert np.array_equal(k_bits, b.k_cache.view(k_bits.dtype))
    del k_bits
    v_bits = cache_bits(d.v_cache)
    assert np.array_equal(v_bits, b.v_cache.view(v_bits.dtype))
    del v_bits
    got = host_f64(out, wl.dtype)
    max_abs, rel = assert_close(got, ref, wl.dtype, name)
    # every output row is finite (no NaN-filled row was read)
    assert np.isfinite(got).all()
    print(f"{name}: max-abs {max_abs:.3e} rel-L2 {rel:.3e}")


@pytest.mark.slow
def test_tree_workload_full_size():
    """The Medusa-tree bench workload, in the bench's launch configuration."""
    import oracle
    import paged_kv_cache_18_gb300 as pkv
    wl = W.TREE_WORKLOADS["medusa_tree"]
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    masks = W.tree_mask_bits(wl.tree_parents)
    out = pkv.tree_verify_attention(d.q, d.k_cache, d.v_cache, d.table, d.lens,
                                    torch.from_numpy(masks.view(np.int64)).cuda(),
                                    scale=wl.softmax_scale, max_context_len=b.max_context_len,
                                    error_word=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    oracle.kv_append(b.k_cache, b.v_cache, b.k_new, b.v_new, b.slot_mapping, wl.dtype)
    ref = oracle.tree_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                                wl.softmax_scale, wl.dtype, masks)
    got = host_f64(out, wl.dtype)
    assert np.isfinite(got).all()
    max_abs, rel = assert_close(got, ref, wl.dtype, wl.name)
    print(f"medusa_tree: max-abs {max_abs:.3e} rel-L2 {rel:.3e}")


# ---- fused append + attention (one launch) --------------------------------
@pytest.mark.parametrize("dtype,kernel", [("f32", "simt"), ("bf16", "simt"), ("bf16", "mma"),
                                          ("f16", "mma")])
@pytest.mark.parametrize("Q,Hq,Hkv", [(1, 8, 2), (1, 4, 4), (5, 32, 8), (3, 8, 1), (8, 32, 8),
                                     (10, 16, 4), (13, 8, 2)])
@pytest.mark.parametrize("split_blocks", [0, 1, 3])
def test_fused_append_attention(dtype, kernel, Q, Hq, Hkv, split_blocks):
    import paged_kv_cache_18_gb300 as pkv
    lens = [max(1, Q - 1), Q, Q + 1, 16, 17, 31, 33, 100, 250]
    D = 128 if dtype != "f32" else 64
    wl = W.Workload(f"fused {dtype} {kernel} Q{Q}", len(lens), Hq, Hkv, D, dtype,
                    context_lens=lens, num_queries=Q, seed=500 + Q + Hq + split_blocks)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    B = wl.batch
    kn = d.k_new.view(B, Q, Hkv, D)
    vn = d.v_new.view(B, Q, Hkv, D)
    q = d.q if Q > 1 else d.q[:, 0]
    out = pkv.append_attention(q, kn, vn, d.k_cache, d.v_cache, d.table, d.lens,
                               scale=wl.softmax_scale, max_context_len=b.max_context_len,
                               kernel=KERNELS[kernel], split_blocks=split_blocks,
                               error_word=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    ref = oracle_after_append(b)
    bits = cache_bits(d.k_cache)
    np.testing.assert_array_equal(bits, b.k_cache.view(bits.dtype))
    bits = cache_bits(d.v_cache)
    np.testing.assert_array_equal(bits, b.v_cache.view(bits.dtype))
    got = host_f64(out if Q > 1 else out[:, None], dtype)
    assert_close(got, ref, dtype, wl.name)


def test_fused_matches_two_calls_bitwise():
    """Same plan, same arithmetic: the fused launch and append-then-attend
    give bit-identical outputs."""
    import paged_kv_cache_18_gb300 as pkv
    wl = W.Workload("fused bitwise", 6, 32, 8, 128, "bf16", len_range=(20, 3000), seed=77)
    for Q in (1, 5):
        wl.num_queries = Q
        b = W.make_batch(wl)
        d1, d2 = DeviceBatch(b), DeviceBatch(b)
        d1.append()
        o1 = d1.attend()
        kn = d2.k_new.view(wl.batch, Q, 8, 128)
        vn = d2.v_new.view(wl.batch, Q, 8, 128)
        o2 = pkv.append_attention(d2.q if Q > 1 else d2.q[:, 0], kn, vn, d2.k_cache,
                                  d2.v_cache, d2.table, d2.lens,
                                  max_context_len=b.max_context_len)
        o2 = o2 if Q > 1 else o2[:, None]
        assert torch.equal(o1, o2)
        for a, c in ((d1.k_cache, d2.k_cache), (d1.v_cache, d2.v_cache)):
            assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def _workspace_filled(pattern: str, nbytes: int, ns: int) -> torch.Tensor:
    """A workspace of nbytes whose prior contents follow `pattern`."""
    n32 = (nbytes + 3) // 4
    if pattern == "ramp":       # int32 1, 2, 3, ...: what a block table or token ids leave
        w = torch.arange(1, n32 + 1, dtype=torch.int32, device="cuda")
    elif pattern == "near":     # every 32-bit word one arrival short of a sequence's count
        w = torch.full((n32,), ns - 1, dtype=torch.int32, device="cuda")
    elif pattern == "ones":     # all bits set
        w = torch.full((n32,), -1, dtype=torch.int32, device="cuda")
    else:                       # uniform random bytes
        g = torch.Generator(device="cuda").manual_seed(5)
        w = torch.randint(-2 ** 31, 2 ** 31 - 1, (n32,), dtype=torch.int32, device="cuda",
                          generator=g)
    return w.view(torch.uint8)[:nbytes]


@pytest.mark.parametrize("pattern", ["ramp", "near", "ones", "random"])
def test_split_counters_need_no_prior_state(pattern):
    """The split-K workspace may hold anything before a call (block tables,
    token ids, another call's partials): the arrival counters of the
    last-CTA merge start from zero in every call, so each sequence's splits
    are merged exactly once, after all of them have arrived (the
    Flash-Decoding reduction sees every chunk once)."""
    import paged_kv_cache_18_gb300 as pkv
    wl = W.Workload("stale", 6, 32, 8, 128, "bf16", len_range=(500, 4000), seed=13)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    ref = oracle_after_append(b)
    with tuning(merge=1):       # force the last-CTA merge (the one with counters)
        for sb in (16, 40, 0):
            pl = pkv.plan(6, 1, 32, 8, 128, b.max_context_len, torch.bfloat16, split_blocks=sb)
            assert pl["num_splits"] > 1 and pl["merge_kernel"] == 0, pl
            need = pkv.workspace_size(6, 1, 32, 8, 128, b.max_context_len, torch.bfloat16,
                                      split_blocks=sb)
            ws = _workspace_filled(pattern, need, pl["num_splits"])
            for _ in range(2):  # and again on what the first call left
                out = d.attend(split_blocks=sb, workspace=ws)
                torch.cuda.synchronize()
                assert_close(host_f64(out, "bf16"), ref, "bf16", f"{pattern} ws sb={sb}")
                ws.copy_(_workspace_filled(pattern, need, pl["num_splits"]))


def test_shared_workspace_across_shapes():
    """One workspace serves calls of different shapes in turn, each landing
    its counters on what the previous call left (partials, other counters)."""
    import paged_kv_cache_18_gb300 as pkv
    cases = [W.Workload("ws a", 6, 32, 8, 128, "bf16", len_range=(500, 4000), seed=14),
             W.Workload("ws b", 3, 16, 4, 128, "bf16", len_range=(100, 2500), seed=15,
                        num_queries=2),
             W.Workload("ws c", 9, 8, 8, 64, "bf16", len_range=(300, 3000), seed=16)]
    ws = _workspace_filled("ramp", 64 << 20, 1)
    with tuning(merge=1):
        for rep in range(2):
            for wl in cases:
                b = W.make_batch(wl)
                d = DeviceBatch(b)
                d.append()
                for sb in (16, 24):
                    pl = pkv.plan(wl.batch, wl.num_queries, wl.num_heads, wl.num_kv_heads,
                                  wl.head_dim, b.max_context_len, torch.bfloat16,
                                  split_blocks=sb)
                    assert pl["num_splits"] > 1 and pl["merge_kernel"] == 0, pl
                    assert pl["workspace_bytes"] <= ws.numel()
                    out = d.attend(split_blocks=sb, workspace=ws)
                    torch.cuda.synchronize()
                    assert_close(host_f64(out, "bf16"), oracle_after_append(b), "bf16",
                                 f"{wl.name} sb={sb} rep {rep}")


@pytest.mark.parametrize("Q", [1, 5])
def test_default_scale_is_one_over_sqrt_head_dim(Q):
    """A scale of zero or below selects 1/sqrt(head_dim) in the library
    (bitwise the same launch as that scale passed explicitly)."""
    import paged_kv_cache_18_gb300 as pkv
    wl = W.Workload("scale", 4, 16, 4, 128, "bf16", context_lens=[5, 90, 700, 1500],
                    num_queries=Q, seed=17)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    fn = pkv.spec_verify_attention if Q > 1 else pkv.paged_decode_attention
    q = d.q if Q > 1 else d.q[:, 0]
    outs = [fn(q, d.k_cache, d.v_cache, d.table, d.lens, scale=s,
               max_context_len=b.max_context_len).clone()
            for s in (float(np.float32(1 / np.sqrt(128))), 0.0, -3.0, None)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    with pytest.raises(pkv.PkvError):
        fn(q, d.k_cache, d.v_cache, d.table, d.lens, scale=float("nan"),
           max_context_len=b.max_context_len)


@pytest.mark.parametrize("rows_per_cta,merge", [(0, 2), (16, 0), (8, 1), (3, 2)])
def test_row_caps_and_merge_modes(rows_per_cta, merge):
    from paged_kv_cache_18_gb300 import binding
    wl = W.Workload("caps", 5, 32, 8, 128, "bf16", context_lens=[5, 40, 700, 1500, 2222],
                    num_queries=5, seed=600 + rows_per_cta + merge)
    binding.TUNING.update(rows_per_cta=rows_per_cta, merge=merge)
    try:
        for sb in (0, 8):
            run_case(wl, kernel=2, split_blocks=sb)
        run_case(wl, kernel=1, split_blocks=8)
    finally:
        binding.TUNING.clear()


# ---- tree verification (Medusa tree attention) ----------------------------
def _tree_masks(Q, n, rng):
    from tests.toy_decoder import ancestor_masks
    out = []
    for _ in range(n):
        parents = [-1] + [int(rng.integers(0, j)) for j in range(1, Q)]
        out.append(ancestor_masks(parents))
    return np.stack(out)


@pytest.mark.parametrize("dtype,kernel", [("f32", 1), ("bf16", 1), ("bf16", 2)])
@pytest.mark.parametrize("Q,Hq,Hkv,shared", [(2, 8, 2, True), (5, 32, 8, False),
                                             (16, 8, 1, False), (33, 4, 4, True),
                                             (64, 8, 2, False)])
@pytest.mark.parametrize("split_blocks", [0, 2])
def test_tree_verify(dtype, kernel, Q, Hq, Hkv, shared, split_blocks):
    import oracle
    import paged_kv_cache_18_gb300 as pkv
    rng = np.random.default_rng(Q * 7 + split_blocks)
    lens = [Q, Q + 3, Q + 40, Q + 300]
    D = 64 if dtype == "f32" else 128
    wl = W.Workload(f"tree {dtype} k{kernel} Q{Q}", len(lens), Hq, Hkv, D, dtype,
                    context_lens=lens, num_queries=Q, seed=700 + Q + split_blocks)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    masks = _tree_masks(Q, 1 if shared else wl.batch, rng)
    masks = masks[0] if shared else masks
    tm = torch.from_numpy(np.ascontiguousarray(masks).view(np.int64)).cuda()
    out = pkv.tree_verify_attention(d.q, d.k_cache, d.v_cache, d.table, d.lens, tm,
                                    scale=wl.softmax_scale, max_context_len=b.max_context_len,
                                    kernel=kernel, split_blocks=split_blocks, error_word=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    oracle.kv_append(b.k_cache, b.v_cache, b.k_new, b.v_new, b.slot_mapping, dtype)
    ref = oracle.tree_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                                wl.softmax_scale, dtype, masks)
    assert_close(host_f64(out, dtype), ref, dtype, wl.name)


@pytest.mark.parametrize("kernel", [1, 2])
def test_chain_tree_equals_spec_verify_bitwise(kernel):
    import paged_kv_cache_18_gb300 as pkv
    wl = W.Workload("chain", 4, 32, 8, 128, "bf16", context_lens=[5, 50, 700, 2000],
                    num_queries=5, seed=720)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    chain = torch.tensor([(2 << j) - 1 for j in range(5)], dtype=torch.int64, device="cuda")
    t = pkv.tree_verify_attention(d.q, d.k_cache, d.v_cache, d.table, d.lens, chain,
                                  max_context_len=b.max_context_len, kernel=kernel)
    s = d.attend(kernel=kernel)
    assert torch.equal(t, s)


# Several 8-column query tiles in one warp (K / V fragments read once for
# all of them): every tile count each head dim takes, ragged lengths,
# partial last tiles and splits.
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D,warp_tiles,Q,Hq,Hkv", [
    (128, 2, 3, 16, 4), (128, 2, 1, 16, 1), (128, 3, 5, 32, 8), (128, 3, 3, 24, 3),
    (128, 3, 1, 24, 1), (64, 2, 2, 8, 1), (64, 3, 5, 16, 4), (64, 4, 4, 64, 8),
    (64, 4, 7, 36, 9)])
@pytest.mark.parametrize("split_blocks", [0, 3])
def test_mma_multi_tile_warps(dtype, D, warp_tiles, Q, Hq, Hkv, split_blocks):
    lens = [Q, 15, 16, 33, 250, 700]
    wl = W.Workload(f"{dtype} D{D} nt{warp_tiles} Q{Q} {Hq}/{Hkv} sb{split_blocks}", len(lens),
                    Hq, Hkv, D, dtype, context_lens=lens, num_queries=Q,
                    seed=1300 + D + 7 * warp_tiles + Q + Hq + split_blocks)
    assert -(-Q * (Hq // Hkv) // 8) == warp_tiles  # one column group of warp_tiles tiles
    run_case(wl, kernel=2, split_blocks=split_blocks, warp_tiles=warp_tiles)


# Four and five column groups: 25 to 40 query rows per KV head in one CTA,
# each staged block read once for all of them.  Full and partial last
# tiles, both rings, splits.
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D,Q,Hq,Hkv,cg", [
    (128, 4, 32, 4, 4), (128, 5, 32, 4, 5), (128, 9, 12, 3, 5), (128, 33, 1, 1, 5),
    (64, 10, 16, 4, 5), (64, 26, 1, 1, 4)])
@pytest.mark.parametrize("split_blocks", [0, 3])
def test_mma_wide_column_groups(dtype, D, Q, Hq, Hkv, cg, split_blocks):
    import paged_kv_cache_18_gb300 as pkv
    lens = [Q, Q + 1, Q + 15, Q + 33, 250, 700]
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    accepted = []
    for stages in (1, 2, 3, 4, 6):
        try:
            p = pkv.plan(len(lens), Q, Hq, Hkv, D, max(lens), tdt, kernel=2, stages=stages)
        except pkv.PkvError:
            continue
        accepted.append(stages)
        assert p["row_chunks"] == 1 and -(-p["rows_per_cta"] // 8) == cg
        assert p["threads_per_cta"] == 32 * cg
        wl = W.Workload(f"{dtype} D{D} cg{cg} Q{Q} {Hq}/{Hkv} st{stages} sb{split_blocks}",
                        len(lens), Hq, Hkv, D, dtype, context_lens=lens, num_queries=Q,
                        seed=1400 + D + 11 * Q + Hq + stages + split_blocks)
        run_case(wl, kernel=2, split_blocks=split_blocks, stages=stages)
    assert accepted == [4, 6], accepted


def test_mma_multi_tile_rejects_oversize():
    import paged_kv_cache_18_gb300 as pkv
    with tuning(warp_tiles=2), pytest.raises(pkv.PkvError):
        # two 8-column tiles of a 256-dim head per warp
        pkv.plan(2, 3, 16, 4, 256, 100, torch.bfloat16, kernel=2)


# Two KV blocks per warp iteration (their chains interleave): every ring of
# four or more stages, odd block counts (a last iteration with one block),
# splits, the fused append and tree masks.
TWO_BLOCK_CASES = [  # D, Q, Hq, Hkv, stages
    (128, 5, 32, 8, 0), (128, 5, 32, 8, 6), (128, 3, 16, 4, 4), (64, 4, 64, 8, 0),
    (64, 3, 40, 5, 0), (128, 7, 24, 8, 0)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D,Q,Hq,Hkv,stages", TWO_BLOCK_CASES)
@pytest.mark.parametrize("split_blocks", [0, 3, 5])
def test_mma_two_blocks_per_iteration(dtype, D, Q, Hq, Hkv, stages, split_blocks):
    lens = [Q, 15, 16, 17, 33, 48, 250, 701]
    wl = W.Workload(f"{dtype} kb2 D{D} Q{Q} {Hq}/{Hkv} st{stages} sb{split_blocks}", len(lens),
                    Hq, Hkv, D, dtype, context_lens=lens, num_queries=Q,
                    seed=1400 + D + Q + Hq + stages + split_blocks)
    run_case(wl, kernel=2, split_blocks=split_blocks, stages=stages, blocks_per_iter=2)


@pytest.mark.parametrize("D,Q,Hq,Hkv", [(128, 1, 8, 8), (128, 2, 8, 2), (256, 1, 8, 2),
                                        (128, 1, 16, 1)])
def test_two_blocks_need_four_stages(D, Q, Hq, Hkv):
    import paged_kv_cache_18_gb300 as pkv
    # one-tile rings of 2 / 3 stages (and 1 / 2 at head_dim 256) cannot
    # keep a pair in flight: refused, not run
    with tuning(blocks_per_iter=2), pytest.raises(pkv.PkvError):
        pkv.plan(2, Q, Hq, Hkv, D, 100, torch.bfloat16, kernel=2)


@pytest.mark.parametrize("split_blocks", [0, 3])
def test_two_blocks_fused_append(split_blocks):
    import paged_kv_cache_18_gb300 as pkv
    Q, Hq, Hkv, D = 5, 32, 8, 128
    lens = [Q - 1, Q, Q + 1, 16, 17, 31, 33, 100, 250]
    wl = W.Workload(f"kb2 fused sb{split_blocks}", len(lens), Hq, Hkv, D, "bf16",
                    context_lens=lens, num_queries=Q, seed=1450 + split_blocks)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    kn = d.k_new.view(wl.batch, Q, Hkv, D)
    vn = d.v_new.view(wl.batch, Q, Hkv, D)
    with tuning(blocks_per_iter=2):
        out = pkv.append_attention(d.q, kn, vn, d.k_cache, d.v_cache, d.table, d.lens,
                                   scale=wl.softmax_scale, max_context_len=b.max_context_len,
                                   kernel=2, split_blocks=split_blocks, error_word=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    ref = oracle_after_append(b)
    for cache, host in ((d.k_cache, b.k_cache), (d.v_cache, b.v_cache)):
        bits = cache_bits(cache)
        np.testing.assert_array_equal(bits, host.view(bits.dtype))
    assert_close(host_f64(out, "bf16"), ref, "bf16", wl.name)


@pytest.mark.parametrize("Q,Hq,Hkv", [(5, 32, 8), (16, 8, 1), (9, 16, 8)])
def test_two_blocks_tree_verify(Q, Hq, Hkv):
    import oracle
    import paged_kv_cache_18_gb300 as pkv
    rng = np.random.default_rng(Q + 31)
    lens = [Q, Q + 3, Q + 40, Q + 301]
    wl = W.Workload(f"kb2 tree Q{Q}", len(lens), Hq, Hkv, 128, "bf16", context_lens=lens,
                    num_queries=Q, seed=1460 + Q)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    masks = _tree_masks(Q, wl.batch, rng)
    tm = torch.from_numpy(np.ascontiguousarray(masks).view(np.int64)).cuda()
    with tuning(blocks_per_iter=2):
        out = pkv.tree_verify_attention(d.q, d.k_cache, d.v_cache, d.table, d.lens, tm,
                                        scale=wl.softmax_scale,
                                        max_context_len=b.max_context_len, kernel=2,
                                        error_word=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    oracle.kv_append(b.k_cache, b.v_cache, b.k_new, b.v_new, b.slot_mapping, "bf16")
    ref = oracle.tree_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                                wl.softmax_scale, "bf16", masks)
    assert_close(host_f64(out, "bf16"), ref, "bf16", wl.name)


# ---- tcgen05 kernel (TMEM accumulators, 128-key chunks) -------------------
TC_CASES = [  # Q, Hq, Hkv: 20, 9, 16, 16, 32, 32, 28, 15, 4 and 1 query rows per KV head
    (5, 32, 8), (3, 24, 8), (2, 32, 4), (1, 16, 1), (4, 32, 4), (8, 16, 4), (7, 36, 9),
    (3, 40, 8), (1, 32, 8), (1, 8, 8)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("Q,Hq,Hkv", TC_CASES)
@pytest.mark.parametrize("split_blocks", [0, 3, 8, 9])
def test_tc_kernel(dtype, Q, Hq, Hkv, split_blocks):
    lens = [Q, 15, 16, 17, 127, 128, 129, 300, 1000]
    wl = W.Workload(f"tc {dtype} Q{Q} {Hq}/{Hkv} sb{split_blocks}", len(lens), Hq, Hkv, 128,
                    dtype, context_lens=lens, num_queries=Q,
                    seed=1600 + Q + Hq + Hkv + split_blocks)
    run_case(wl, kernel=3, split_blocks=split_blocks)


def test_tc_kernel_long_and_ragged():
    wl = W.Workload("tc long", 6, 32, 8, 128, "bf16", len_range=(1, 9000), num_queries=5,
                    seed=1650)
    run_case(wl, kernel=3)
    run_case(wl, kernel=3, split_blocks=40)


@pytest.mark.parametrize("Q,Hq,Hkv", [(5, 32, 8), (16, 8, 4), (9, 16, 8)])
def test_tc_tree_verify(Q, Hq, Hkv):
    import oracle
    import paged_kv_cache_18_gb300 as pkv
    rng = np.random.default_rng(Q + 77)
    lens = [Q, Q + 3, Q + 140, Q + 301]
    wl = W.Workload(f"tc tree Q{Q}", len(lens), Hq, Hkv, 128, "bf16", context_lens=lens,
                    num_queries=Q, seed=1660 + Q)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    masks = _tree_masks(Q, wl.batch, rng)
    tm = torch.from_numpy(np.ascontiguousarray(masks).view(np.int64)).cuda()
    out = pkv.tree_verify_attention(d.q, d.k_cache, d.v_cache, d.table, d.lens, tm,
                                    scale=wl.softmax_scale, max_context_len=b.max_context_len,
                                    kernel=3, error_word=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    oracle.kv_append(b.k_cache, b.v_cache, b.k_new, b.v_new, b.slot_mapping, "bf16")
    ref = oracle.tree_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                                wl.softmax_scale, "bf16", masks)
    assert_close(host_f64(out, "bf16"), ref, "bf16", wl.name)


def test_tc_refuses_what_it_does_not_build():
    import paged_kv_cache_18_gb300 as pkv
    for args in [(2, 1, 8, 8, 64, 100, torch.bfloat16),    # head_dim 64
                 (2, 1, 8, 8, 128, 100, torch.float32)]:   # float32
        with pytest.raises(pkv.PkvError):
            pkv.plan(*args, kernel=3)
    # up to 64 rows per KV head in one CTA (the 64-column tile); more are
    # split over row chunks of <= 64
    p = pkv.plan(2, 9, 32, 8, 128, 100, torch.bfloat16, kernel=3)
    assert p["rows_per_cta"] == 36 and p["row_chunks"] == 1
    p = pkv.plan(2, 18, 32, 8, 128, 100, torch.bfloat16, kernel=3)
    assert p["rows_per_cta"] == 36 and p["row_chunks"] == 2
    with pytest.raises(pkv.PkvError):   # three V stages do not fit beside the wide tile
        pkv.plan(2, 9, 32, 8, 128, 100, torch.bfloat16, kernel=3, stages=3)
    # FP8 caches stay on the other kernels
    with pytest.raises(pkv.PkvError):
        pkv.plan(2, 1, 8, 8, 128, 100, "fp8", kernel=3)


@pytest.mark.parametrize("stages", [1, 2, 3])
@pytest.mark.parametrize("Q,Hq,Hkv", [(5, 32, 8), (2, 32, 4), (1, 8, 8)])
@pytest.mark.parametrize("split_blocks", [0, 3, 17])
def test_tc_ring_depths(stages, Q, Hq, Hkv, split_blocks):
    lens = [Q, 16, 129, 300, 1000, 2100]
    wl = W.Workload(f"tc st{stages} Q{Q} {Hq}/{Hkv} sb{split_blocks}", len(lens), Hq, Hkv, 128,
                    "bf16", context_lens=lens, num_queries=Q,
                    seed=1700 + 10 * stages + Q + Hq + split_blocks)
    run_case(wl, kernel=3, stages=stages, split_blocks=split_blocks)


@pytest.mark.parametrize("persistent", [1, 2])
@pytest.mark.parametrize("stages", [1, 2, 3])
@pytest.mark.parametrize("split_blocks", [8, 13, 56])
def test_tc_many_items_per_cta(persistent, stages, split_blocks):
    # enough (split, KV head, sequence) items that every CTA walking them
    # (persistent 1) takes several, reusing its Q^T and O^T buffers across
    # items; persistent 2: one CTA per item
    with tuning(persistent=persistent):
        wl = W.Workload(f"tc items p{persistent} st{stages} sb{split_blocks}", 16, 32, 8, 128,
                        "bf16", len_range=(1, 6000), num_queries=5,
                        seed=1800 + stages + split_blocks)
        run_case(wl, kernel=3, stages=stages, split_blocks=split_blocks)
        wl = W.Workload(f"tc items gqa p{persistent} st{stages} sb{split_blocks}", 64, 32, 8,
                        128, "bf16", len_range=(1, 3000), num_queries=3,
                        seed=1850 + stages + split_blocks)
        run_case(wl, kernel=3, stages=stages, split_blocks=split_blocks)


# ---- split-K partition made on the device from the real lengths -----------
DEVICE_LENS = [
    [32768, 65536],                                  # long contexts, unequal
    [1, 15, 16, 17, 300, 2000, 0, 5000],             # ragged, with an empty sequence
    [700] * 32,                                      # the most sequences it takes
    [40, 40],                                        # fewer items than CTAs
]


@pytest.mark.parametrize("lens_i", range(len(DEVICE_LENS)))
@pytest.mark.parametrize("Q,Hq,Hkv", [(1, 32, 8), (5, 32, 8), (1, 8, 8), (3, 16, 2)])
@pytest.mark.parametrize("kernel,waves", [(2, 1), (2, 3), (1, 1)])
def test_device_split_partition(lens_i, Q, Hq, Hkv, kernel, waves):
    """The partition the kernels derive on the device (split length from the
    batch's block counts, flat grid of work items, one partial per item and
    CTA column) gives the oracle's result; the merge kernel finds every
    item of every row."""
    import paged_kv_cache_18_gb300 as pkv
    lens = DEVICE_LENS[lens_i]
    if Q > 1:
        lens = [max(L, Q) for L in lens]
    D = 128
    dtype = "bf16"
    wl = W.Workload(f"device split {lens_i} Q{Q} {Hq}/{Hkv} k{kernel} w{waves}", len(lens), Hq,
                    Hkv, D, dtype, context_lens=lens, num_queries=Q,
                    seed=800 + lens_i * 7 + Q + Hq + kernel + waves)
    b = W.make_batch(wl)
    with tuning(split_waves=waves):
        pl = pkv.plan(wl.batch, Q, Hq, Hkv, D, b.max_context_len, torch.bfloat16, kernel=kernel)
        assert pl["split_target"] > 0
        run_case(wl, kernel=kernel)


def test_device_split_partition_equals_host_partition():
    """Same inputs through both partitions: the same answer to within the
    output rounding (each equals the oracle), and the device one is
    deterministic."""
    import paged_kv_cache_18_gb300 as pkv
    wl = W.Workload("dev vs host", 12, 32, 8, 128, "bf16", len_range=(100, 9000), seed=830,
                    num_queries=5)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    ref = oracle_after_append(b)
    outs = {}
    for waves in (-1, 1, 2):
        with tuning(split_waves=waves):
            pl = pkv.plan(wl.batch, 5, 32, 8, 128, b.max_context_len, torch.bfloat16)
            assert (pl["split_target"] > 0) == (waves > 0)
            o1 = d.attend().clone()
            o2 = d.attend()
        assert torch.equal(o1, o2)
        outs[waves] = host_f64(o1, "bf16")
        assert_close(outs[waves], ref, "bf16", f"waves {waves}")
    assert np.abs(outs[1] - outs[-1]).max() <= 2 ** -7


def test_device_split_partition_fused_append_tree_fp8_and_graph():
    """The fused append, tree verification and FP8 caches take the same
    partition; a captured graph replays it."""
    import oracle
    import paged_kv_cache_18_gb300 as pkv
    from tests.gpu_util import assert_close_fp8
    lens = [37, 4000, 900, 16, 12000, 9]   # every row below L holds data (L >= 7 tree nodes)
    # fused append + verify
    wl = W.Workload("dev fused", len(lens), 32, 8, 128, "bf16", context_lens=lens, num_queries=5,
                    seed=840)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    pkv.binding.TUNING["split_waves"] = 1
    try:
        _device_split_calls(wl, b, d)
    finally:
        pkv.binding.TUNING.pop("split_waves", None)


def _device_split_calls(wl, b, d):
    import oracle
    import paged_kv_cache_18_gb300 as pkv
    from tests.gpu_util import assert_close_fp8
    lens = list(wl.context_lens)
    pl = pkv.plan(wl.batch, 5, 32, 8, 128, b.max_context_len, torch.bfloat16)
    assert pl["split_target"] > 0
    kn, vn = d.k_new.view(wl.batch, 5, 8, 128), d.v_new.view(wl.batch, 5, 8, 128)
    out = pkv.append_attention(d.q, kn, vn, d.k_cache, d.v_cache, d.table, d.lens,
                               max_context_len=b.max_context_len, error_word=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    assert_close(host_f64(out, "bf16"), oracle_after_append(b), "bf16", "fused device split")
    # tree verification over the same cache
    masks = W.tree_mask_bits(W.medusa_parents((2, 2)))
    q7 = torch.randn(wl.batch, len(masks), 32, 128, device="cuda").to(torch.bfloat16)
    lens7 = d.lens
    t = pkv.tree_verify_attention(q7, d.k_cache, d.v_cache, d.table, lens7,
                                  torch.from_numpy(masks.view(np.int64)).cuda(),
                                  max_context_len=b.max_context_len)
    from tests.gpu_util import cache_bits
    kbits, vbits = cache_bits(d.k_cache), cache_bits(d.v_cache)
    q7h = q7.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.tree_attention(q7h, kbits, vbits, b.block_table, lens7.cpu().numpy(),
                                1 / np.sqrt(128), "bf16", masks)
    assert_close(host_f64(t, "bf16"), ref, "bf16", "tree device split")
    # FP8 cache
    kc8, vc8 = W.fp8_caches(b, 0.0123, 0.0171)
    k8, v8 = torch.from_numpy(kc8).cuda(), torch.from_numpy(vc8).cuda()
    o8 = pkv.paged_attention_fp8(d.q, k8, v8, d.table, d.lens, 0.0123, 0.0171,
                                 max_context_len=b.max_context_len)
    ref8 = oracle.paged_attention_fp8(b.q, kc8, vc8, b.block_table, b.context_lens,
                                      1 / np.sqrt(128), "bf16", 0.0123, 0.0171)
    assert_close_fp8(host_f64(o8, "bf16"), ref8, "bf16", "fp8 device split")
    # graph replay
    ws = torch.empty(pl["workspace_bytes"], dtype=torch.uint8, device="cuda")
    o = torch.empty_like(d.q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d.attend(out=o, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        d.attend(out=o, workspace=ws)
    for _ in range(2):
        o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_close(host_f64(o, "bf16"), oracle_after_append(b), "bf16", "graph device split")


def test_device_split_reports_long_context_once():
    """A context above max_context_len is clamped and recorded, as in the
    host partition."""
    wl = W.Workload("dev err", 3, 32, 8, 128, "bf16", context_lens=[3000, 50, 800], seed=850)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    d.lens[1] = 5000   # beyond max_context_len = 3000
    with tuning(split_waves=1):
        out = d.attend()
    torch.cuda.synchronize()
    assert int(d.err.item()) == 3
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("lens_i", range(len(DEVICE_LENS)))
@pytest.mark.parametrize("Q,Hq,Hkv", [(5, 32, 8), (1, 32, 8), (3, 36, 9)])
@pytest.mark.parametrize("waves,persistent", [(0, 0), (2, 0), (3, 1)])
def test_tc_device_partition(lens_i, Q, Hq, Hkv, waves, persistent):
    """The tcgen05 kernel takes the device partition by default (items of
    nearly equal length, one wave of SMs): one CTA per item, or CTAs walking
    several items (persistent 1)."""
    import paged_kv_cache_18_gb300 as pkv
    lens = [max(L, Q) for L in DEVICE_LENS[lens_i]]
    wl = W.Workload(f"tc dev {lens_i} Q{Q} w{waves} p{persistent}", len(lens), Hq, Hkv, 128,
                    "bf16", context_lens=lens, num_queries=Q,
                    seed=1900 + lens_i * 11 + Q + waves + persistent)
    with tuning(split_waves=waves, persistent=persistent):
        b_max = max(lens)
        pl = pkv.plan(len(lens), Q, Hq, Hkv, 128, b_max, torch.bfloat16, kernel=3)
        assert pl["split_target"] > 0
        run_case(wl, kernel=3)


# ---- balanced partition of the tcgen05 kernel (its default) ------------------
STREAM_K_LENS = [
    [0, 1, 15, 16, 17, 300, 2000, 5000],         # ragged, with an empty sequence
    [700] * 32,                                  # the most sequences it takes
    [40, 40],                                    # fewer blocks than CTAs
    [65536, 1, 32768],                           # long contexts beside a tiny one
    [8192, 512] * 8,                             # the verify shape's extremes
]


@pytest.mark.parametrize("lens_i", range(len(STREAM_K_LENS)))
@pytest.mark.parametrize("Q,Hq,Hkv", [(1, 32, 8), (5, 32, 8), (3, 36, 9), (2, 32, 4)])
@pytest.mark.parametrize("stages", [0, 1, 3])
def test_tc_stream_k(lens_i, Q, Hq, Hkv, stages):
    """Every CTA takes an equal share of the batch's (unit, block) list; a
    unit is split wherever a CTA boundary falls in it and the merge finds its
    splits from its first and last block.  Empty sequences (decode) give
    zeros."""
    import paged_kv_cache_18_gb300 as pkv
    lens = STREAM_K_LENS[lens_i]
    if Q > 1:
        lens = [max(L, Q) for L in lens]
    wl = W.Workload(f"tc stream-k {lens_i} Q{Q} {Hq}/{Hkv} st{stages}", len(lens), Hq, Hkv, 128,
                    "bf16", context_lens=lens, num_queries=Q,
                    seed=2100 + lens_i * 13 + Q + Hq + stages)
    pl = pkv.plan(len(lens), Q, Hq, Hkv, 128, max(lens), torch.bfloat16, kernel=3,
                  stages=stages)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert pl["stream_k"] == 1 and pl["split_target"] == pl["grid_x"] == sms * pl["ctas_per_sm"]
    run_case(wl, kernel=3, stages=stages)


def test_tc_stream_k_workspace_graph_and_errors():
    """The balanced partition ignores what the workspace held, replays from a
    graph, is deterministic, and records a context above max_context_len
    (clamped) like the other partitions."""
    import paged_kv_cache_18_gb300 as pkv
    wl = W.Workload("tc stream-k ws", 16, 32, 8, 128, "bf16", len_range=(512, 8192),
                    num_queries=5, seed=2200)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    ref = oracle_after_append(b)
    pl = pkv.plan(wl.batch, 5, 32, 8, 128, b.max_context_len, torch.bfloat16, kernel=3)
    assert pl["stream_k"] == 1
    ws = torch.full((pl["workspace_bytes"],), 0xFF, dtype=torch.uint8, device="cuda")  # NaN floats
    o = torch.empty_like(d.q)
    d.attend(kernel=3, out=o, workspace=ws)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    first = o.clone()
    assert_close(host_f64(o, "bf16"), ref, "bf16", "stream-k, NaN-filled workspace")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d.attend(kernel=3, out=o, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        d.attend(kernel=3, out=o, workspace=ws)
    for _ in range(2):
        o.zero_()
        ws.fill_(0xFF)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, first)
    # a length beyond max_context_len: clamped and recorded
    wl2 = W.Workload("tc stream-k err", 3, 32, 8, 128, "bf16", context_lens=[3000, 50, 800],
                     seed=2210)
    b2 = W.make_batch(wl2)
    d2 = DeviceBatch(b2)
    d2.append()
    d2.lens[1] = 5000
    out = d2.attend(kernel=3)
    torch.cuda.synchronize()
    assert int(d2.err.item()) == 3
    assert torch.isfinite(out.float()).all()


def test_tc_stream_k_tree_masks():
    """Tree verification (7-node tree over 4 query heads per KV head: 28 rows)
    through the tcgen05 kernel's balanced partition."""
    import oracle
    import paged_kv_cache_18_gb300 as pkv
    from tests.gpu_util import cache_bits
    lens = [37, 4000, 900, 16, 12000, 9]
    wl = W.Workload("tc stream-k tree", len(lens), 32, 8, 128, "bf16", context_lens=lens,
                    seed=2220)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    masks = W.tree_mask_bits(W.medusa_parents((2, 2)))
    q7 = torch.randn(wl.batch, len(masks), 32, 128, device="cuda").to(torch.bfloat16)
    t = pkv.tree_verify_attention(q7, d.k_cache, d.v_cache, d.table, d.lens,
                                  torch.from_numpy(masks.view(np.int64)).cuda(),
                                  max_context_len=b.max_context_len, kernel=3,
                                  error_word=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    oracle_after_append(b)
    q7h = q7.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.tree_attention(q7h, cache_bits(d.k_cache), cache_bits(d.v_cache),
                                b.block_table, d.lens.cpu().numpy(), 1 / np.sqrt(128), "bf16",
                                masks)
    assert_close(host_f64(t, "bf16"), ref, "bf16", "tc stream-k tree")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("Q,Hq,Hkv", [(1, 8, 2), (1, 4, 4), (5, 32, 8), (3, 8, 1), (8, 32, 8),
                                     (16, 8, 4), (2, 32, 8), (9, 32, 8)])
@pytest.mark.parametrize("split_blocks", [0, 1, 3, 9])
def test_tc_fused_append_attention(dtype, Q, Hq, Hkv, split_blocks):
    """The tcgen05 kernel's fused append: the producers fill the blocks that
    hold new rows themselves (older rows from the cache, new rows from k_new /
    v_new) and row chunk 0 writes the new rows into the cache, bit for bit
    (36 rows per KV head: two row chunks reading the same blocks); with the
    balanced partition (split_blocks 0) and the host's."""
    import paged_kv_cache_18_gb300 as pkv
    lens = [max(1, Q - 1), Q, Q + 1, 16, 17, 31, 33, 100, 250, 129, 4000]
    D = 128
    wl = W.Workload(f"tc fused {dtype} Q{Q} {Hq}/{Hkv} sb{split_blocks}", len(lens), Hq, Hkv, D,
                    dtype, context_lens=lens, num_queries=Q,
                    seed=2300 + Q + Hq + split_blocks)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    B = wl.batch
    kn = d.k_new.view(B, Q, Hkv, D)
    vn = d.v_new.view(B, Q, Hkv, D)
    q = d.q if Q > 1 else d.q[:, 0]
    out = pkv.append_attention(q, kn, vn, d.k_cache, d.v_cache, d.table, d.lens,
                               scale=wl.softmax_scale, max_context_len=b.max_context_len,
                               kernel=3, split_blocks=split_blocks, error_word=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    ref = oracle_after_append(b)
    for cache, host in ((d.k_cache, b.k_cache), (d.v_cache, b.v_cache)):
        bits = cache_bits(cache)
        np.testing.assert_array_equal(bits, host.view(bits.dtype))
    got = host_f64(out if Q > 1 else out[:, None], dtype)
    assert_close(got, ref, dtype, wl.name)


def test_tc_fused_matches_two_calls_bitwise():
    """The tcgen05 kernel: the fused launch and append-then-attend give
    bit-identical outputs and caches (the same plan, the same arithmetic)."""
    import paged_kv_cache_18_gb300 as pkv
    wl = W.Workload("tc fused bitwise", 16, 32, 8, 128, "bf16", len_range=(20, 8192), seed=2350)
    for Q in (1, 5):
        wl.num_queries = Q
        b = W.make_batch(wl)
        d1, d2 = DeviceBatch(b), DeviceBatch(b)
        d1.append()
        o1 = d1.attend(kernel=3)
        kn = d2.k_new.view(wl.batch, Q, 8, 128)
        vn = d2.v_new.view(wl.batch, Q, 8, 128)
        o2 = pkv.append_attention(d2.q if Q > 1 else d2.q[:, 0], kn, vn, d2.k_cache,
                                  d2.v_cache, d2.table, d2.lens,
                                  max_context_len=b.max_context_len, kernel=3)
        o2 = o2 if Q > 1 else o2[:, None]
        assert torch.equal(o1, o2)
        for a, c in ((d1.k_cache, d2.k_cache), (d1.v_cache, d2.v_cache)):
            assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_merge_rows_kernel_many_splits():
    """The warp-per-row merge (from 1024 output rows, device partitions) over
    rows with more than 32 splits: the log-sum-exps are taken 32 at a time."""
    import paged_kv_cache_18_gb300 as pkv
    from paged_kv_cache_18_gb300 import accounting
    lens = [16384, 12000]
    Q, Hq, Hkv = 16, 32, 8
    wl = W.Workload("merge rows", len(lens), Hq, Hkv, 128, "bf16", context_lens=lens,
                    num_queries=Q, seed=2400)
    assert wl.batch * Q * Hq >= 1024
    with tuning(split_waves=16):
        pl = pkv.plan(wl.batch, Q, Hq, Hkv, 128, max(lens), torch.bfloat16, kernel=2)
        ns = accounting.device_split_counts(lens, 16, Hkv * pl["row_chunks"], pl["split_target"],
                                            max(lens), -(-max(lens) // 16))
        assert max(ns) > 32
        run_case(wl, kernel=2)


@pytest.mark.parametrize("stages", [1, 2])
@pytest.mark.parametrize("Q,Hq,Hkv", [(9, 32, 8), (16, 32, 8), (5, 64, 8), (17, 16, 4)])
@pytest.mark.parametrize("split_blocks", [0, 3, 17])
def test_tc_wide_tile(stages, Q, Hq, Hkv, split_blocks):
    """The tcgen05 kernel's 64-column tile (33..64 query rows per KV head: one
    Q^T and one P^T buffer, 512 TMEM columns), with the balanced partition
    and the host's; 68 rows take two row chunks."""
    lens = [Q, 16, 129, 300, 1000, 2100, 5000]
    wl = W.Workload(f"tc wide st{stages} Q{Q} {Hq}/{Hkv} sb{split_blocks}", len(lens), Hq, Hkv,
                    128, "bf16", context_lens=lens, num_queries=Q,
                    seed=2500 + 10 * stages + Q + Hq + split_blocks)
    run_case(wl, kernel=3, stages=stages, split_blocks=split_blocks)


@pytest.mark.parametrize("branching", [(3, 2), (4, 3), (2, 2, 2)])
def test_tc_wide_tile_tree(branching):
    """Medusa-style trees over four query heads per KV head (40, 68 and 60
    rows) through the tcgen05 kernel: per-node ancestor masks."""
    import oracle
    import paged_kv_cache_18_gb300 as pkv
    from tests.gpu_util import cache_bits
    parents = W.medusa_parents(branching)
    n = len(parents)
    lens = [n, n + 3, 600, 4000, 9000, 130]
    wl = W.Workload(f"tc tree {branching}", len(lens), 32, 8, 128, "bf16", context_lens=lens,
                    num_queries=n, seed=2600 + n)
    b = W.make_batch(wl)
    d = DeviceBatch(b)
    d.append()
    masks = W.tree_mask_bits(parents)
    out = pkv.tree_verify_attention(d.q, d.k_cache, d.v_cache, d.table, d.lens,
                                    torch.from_numpy(masks.view(np.int64)).cuda(),
                                    scale=wl.softmax_scale, max_context_len=b.max_context_len,
                                    kernel=3, error_word=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    oracle_after_append(b)
    ref = oracle.tree_attention(b.q, cache_bits(d.k_cache), cache_bits(d.v_cache),
                                b.block_table, b.context_lens, wl.softmax_scale, "bf16", masks)
    assert_close(host_f64(out, "bf16"), ref, "bf16", wl.name)
