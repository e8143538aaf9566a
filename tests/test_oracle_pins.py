"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each test ties the oracle to something other than itself: the independent
NumPy twin, a closed form, a library routine (PyTorch's
scaled_dot_product_attention in float64 on the CPU), a brute-force pure-Python
evaluation, or numbers the pages print.  ``test_oracle_mutations.py`` plants
plausible mistakes in a copy of the C oracle and checks that these pins fail.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import twin
from paged_kv_cache_18_gb300 import workloads as W


def appended(wl, poison=True):
    """Batch of ``wl`` with the new rows written by the oracle's append."""
    b = W.make_batch(wl, poison=poison)
    oracle.kv_append(b.k_cache, b.v_cache, b.k_new, b.v_new, b.slot_mapping,
                     wl.dtype)
    return b


def run(b, scale=None, rows=None, orc=None):
    orc = orc or oracle.default()
    return orc.paged_attention(b.q, b.k_cache, b.v_cache, b.block_table,
                               b.context_lens,
                               b.wl.softmax_scale if scale is None else scale,
                               b.wl.dtype, rows=rows)


CASES = [
    W.Workload("mha f32", 4, 6, 6, 64, "f32", context_lens=[17, 64, 100, 256], seed=11),
    W.Workload("gqa bf16", 3, 8, 2, 128, "bf16", context_lens=[1, 16, 33], seed=12),
    W.Workload("mqa f16", 2, 4, 1, 64, "f16", context_lens=[40, 7], seed=13),
    W.Workload("spec bf16", 3, 8, 2, 64, "bf16", context_lens=[5, 21, 48],
               num_queries=5, seed=14),
    W.Workload("spec short", 2, 4, 4, 64, "f32", context_lens=[3, 1], num_queries=4,
               seed=15),
]


# 1. Paged == contiguous: the row-by-row table walk (C) equals dense attention
#    on gathered rows (NumPy), for shuffled physical blocks
#    ("Inference part 1", PagedAttention; "Efficient Inference", block table).
@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_paged_equals_contiguous(wl):
    b = appended(wl)
    o1 = run(b)
    o2 = twin.contiguous_attention(b.q, b.k_cache, b.v_cache, b.block_table,
                                   b.context_lens, wl.softmax_scale, wl.dtype)
    assert not np.isnan(o1).any()
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_block_permutation_invariance():
    """Any relabelling of the physical blocks gives the identical result."""
    wl = W.Workload("perm", 2, 4, 2, 64, "bf16", context_lens=[70, 33], seed=21)
    b = appended(wl)
    ref = run(b)
    rng = np.random.default_rng(0)
    perm = rng.permutation(b.num_blocks)
    inv = np.argsort(perm)  # new id of old block o is inv[o]
    b.k_cache = np.ascontiguousarray(b.k_cache[perm])
    b.v_cache = np.ascontiguousarray(b.v_cache[perm])
    owned = b.block_table >= 0
    b.block_table = np.where(owned, inv[np.maximum(b.block_table, 0)], -1).astype(np.int32)
    np.testing.assert_array_equal(run(b), ref)


# 2. A context of one row returns its V row exactly.
def test_single_row_returns_v0():
    wl = W.Workload("L1", 3, 4, 2, 64, "bf16", context_lens=[1, 1, 1], seed=31)
    b = appended(wl)
    out = run(b)
    for bi in range(3):
        phys = b.block_table[bi, 0]
        for h in range(4):
            v0 = twin.widen(b.v_cache[phys, h // 2, 0], "bf16")
            np.testing.assert_array_equal(out[bi, 0, h], v0)


# 3. Identical keys (or scale 0) give uniform weights: the mean of V.
def test_identical_keys_mean_of_v():
    wl = W.Workload("same k", 2, 2, 1, 64, "f32", context_lens=[37, 16], seed=41)
    b = appended(wl)
    for bi in range(2):
        L = int(b.context_lens[bi])
        for i in range(L):
            phys = b.block_table[bi, i // 16]
            b.k_cache[phys, 0, i % 16] = b.k_cache[b.block_table[bi, 0], 0, 0]
    out = run(b)
    for bi in range(2):
        L = int(b.context_lens[bi])
        v = twin.widen(twin.gather_sequence(b.v_cache, b.block_table[bi], L), "f32")
        for h in range(2):
            np.testing.assert_allclose(out[bi, 0, h], v[:, 0].mean(axis=0), rtol=0, atol=1e-14)


def test_zero_scale_mean_of_v():
    wl = W.Workload("scale0", 2, 4, 2, 64, "bf16", context_lens=[50, 9], seed=42)
    b = appended(wl)
    out = run(b, scale=0.0)
    for bi in range(2):
        L = int(b.context_lens[bi])
        v = twin.widen(twin.gather_sequence(b.v_cache, b.block_table[bi], L), "bf16")
        for h in range(4):
            np.testing.assert_allclose(out[bi, 0, h], v[:, h // 2].mean(axis=0),
                                       rtol=0, atol=1e-14)


# 4. Shift invariance: adding one vector to every key adds scale*<q, c> to
#    every score of a row, which the softmax removes (the key-smoothing
#    identity of SageAttention, "Inference part 1", quantized attention).
def test_key_shift_invariance():
    wl = W.Workload("shift", 2, 4, 2, 64, "f32", context_lens=[45, 20], seed=51)
    b = appended(wl)
    # dyadic values so that k + c is exact in float32
    rng = np.random.default_rng(5)
    b.k_cache[:] = (rng.integers(-16, 17, b.k_cache.shape) / 8).astype(np.float32)
    b.q[:] = (rng.integers(-16, 17, b.q.shape) / 8).astype(np.float32)
    ref = run(b)
    c = (rng.integers(-16, 17, (2, 64)) / 4).astype(np.float32)
    b.k_cache += c[None, :, None, :]
    np.testing.assert_allclose(run(b), ref, rtol=0, atol=1e-12)


# 5. MQA/GQA reductions: the head map h -> h // G ("Inference part 1",
#    MultiHeadAttention_GQA, repeat_interleave; "Efficient Inference").
def test_repeat_interleaved_cache_identical():
    wl = W.Workload("gqa", 2, 8, 2, 64, "bf16", context_lens=[30, 64], seed=61)
    b = appended(wl)
    ref = run(b)
    rep_k = np.ascontiguousarray(np.repeat(b.k_cache, 4, axis=1))
    rep_v = np.ascontiguousarray(np.repeat(b.v_cache, 4, axis=1))
    out = oracle.paged_attention(b.q, rep_k, rep_v, b.block_table, b.context_lens,
                                 wl.softmax_scale, "bf16")
    np.testing.assert_array_equal(out, ref)


def test_mha_is_per_head_single_head():
    wl = W.Workload("mha", 2, 3, 3, 64, "f32", context_lens=[19, 40], seed=62)
    b = appended(wl)
    ref = run(b)
    for h in range(3):
        kh = np.ascontiguousarray(b.k_cache[:, h:h + 1])
        vh = np.ascontiguousarray(b.v_cache[:, h:h + 1])
        qh = np.ascontiguousarray(b.q[:, :, h:h + 1])
        out = oracle.paged_attention(qh, kh, vh, b.block_table, b.context_lens,
                                     wl.softmax_scale, "f32")
        np.testing.assert_array_equal(out[:, :, 0], ref[:, :, h])


# 6. Append then decode == the last rows of a full causal prefill over the
#    sequence, computed by PyTorch's float64 SDPA with is_causal and
#    enable_gqa ("Inference part 1", KV cache: the new tokens attend to the
#    cached ones and to themselves; "Efficient Inference", generate_kv).
@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_matches_causal_prefill_sdpa(wl):
    b = appended(wl)
    out = run(b)
    Q, Hq, Hkv = wl.num_queries, wl.num_heads, wl.num_kv_heads
    for bi in range(wl.batch):
        L = int(b.context_lens[bi])
        k = torch.from_numpy(twin.widen(twin.gather_sequence(b.k_cache, b.block_table[bi], L), wl.dtype))
        v = torch.from_numpy(twin.widen(twin.gather_sequence(b.v_cache, b.block_table[bi], L), wl.dtype))
        qn = torch.from_numpy(twin.widen(b.q[bi], wl.dtype))  # [Q, Hq, D]
        # Prefill queries: only the last Q rows are real queries here; the
        # earlier rows get arbitrary queries and are discarded.
        qfull = torch.zeros(L, Hq, wl.head_dim, dtype=torch.float64)
        first = max(0, L - Q)
        qfull[first:] = qn[Q - (L - first):]
        o = torch.nn.functional.scaled_dot_product_attention(
            qfull.transpose(0, 1)[None], k.transpose(0, 1)[None],
            v.transpose(0, 1)[None], is_causal=True, scale=wl.softmax_scale,
            enable_gqa=(Hq != Hkv))[0].transpose(0, 1)  # [L, Hq, D]
        for j in range(Q):
            i = L - Q + j
            if i < 0:
                np.testing.assert_array_equal(out[bi, j], 0.0)
            else:
                np.testing.assert_allclose(out[bi, j], o[i].numpy(), rtol=0, atol=1e-12)


# 7. A speculative-verify row j equals plain decode over the prefix of
#    L - Q + 1 + j rows ("Inference part 2", generate_speculative: the
#    target scores every draft position in one pass).
def test_spec_rows_equal_decode_on_prefixes():
    wl = W.Workload("spec", 3, 8, 2, 64, "bf16", context_lens=[9, 40, 77],
                    num_queries=5, seed=71)
    b = appended(wl)
    spec = run(b)
    for j in range(5):
        lens = (b.context_lens - 5 + 1 + j).astype(np.int32)
        dec = oracle.paged_attention(np.ascontiguousarray(b.q[:, j]), b.k_cache,
                                     b.v_cache, b.block_table, lens,
                                     wl.softmax_scale, "bf16")
        np.testing.assert_array_equal(spec[:, j], dec[:, 0])


def test_no_visible_row_returns_zero():
    wl = W.Workload("empty", 3, 2, 2, 64, "f32", context_lens=[0, 2, 5],
                    num_queries=3, seed=72)
    b = appended(wl)
    out = run(b)
    assert (out[0] == 0).all()           # L = 0: nothing visible
    assert (out[1, 0] == 0).all()        # L - Q + 0 < 0
    assert not (out[1, 1] == 0).all()    # sees row 0
    assert not np.isnan(out).any()


# 10. Brute force on tiny inputs: pure-Python loops, exp without max
#     subtraction, exactly summed with math.fsum.
def test_brute_force_tiny():
    wl = W.Workload("tiny", 2, 2, 1, 64, "f32", context_lens=[5, 18],
                    num_queries=2, seed=81)
    b = appended(wl)
    out = run(b)
    s = wl.softmax_scale
    for bi in range(2):
        L = int(b.context_lens[bi])
        for j in range(2):
            for h in range(2):
                q = [float(x) for x in b.q[bi, j, h]]
                ws, vs = [], []
                for i in range(L - 2 + 1 + j):
                    phys = int(b.block_table[bi, i // 16])
                    k = [float(x) for x in b.k_cache[phys, 0, i % 16]]
                    ws.append(math.exp(s * math.fsum(a * c for a, c in zip(q, k))))
                    vs.append([float(x) for x in b.v_cache[phys, 0, i % 16]])
                den = math.fsum(ws)
                want = [math.fsum(w * v[d] for w, v in zip(ws, vs)) / den for d in range(64)]
                np.testing.assert_allclose(out[bi, j, h], want, rtol=0, atol=1e-13)


# 11. Online softmax == standard: the blockwise recurrence of the pages
#     ("KV cache, prefill va decode", section 07, online softmax; "Inference
#     part 1", FlashAttention equations) restated in float64 agrees with the
#     two-pass oracle to rounding.
def test_online_recurrence_equals_two_pass():
    wl = W.Workload("online", 2, 4, 2, 64, "bf16", context_lens=[300, 97], seed=91)
    b = appended(wl)
    ref = run(b)
    s = wl.softmax_scale
    for bi in range(2):
        L = int(b.context_lens[bi])
        k = twin.widen(twin.gather_sequence(b.k_cache, b.block_table[bi], L), "bf16")
        v = twin.widen(twin.gather_sequence(b.v_cache, b.block_table[bi], L), "bf16")
        for h in range(4):
            q = twin.widen(b.q[bi, 0, h], "bf16")
            m, l, o = -np.inf, 0.0, np.zeros(64)
            for t in range(0, L, 37):
                sc = k[t:t + 37, h // 2] @ q * s
                m_new = max(m, sc.max())
                p = np.exp(sc - m_new)
                corr = math.exp(m - m_new)
                l = l * corr + p.sum()
                o = o * corr + p @ v[t:t + 37, h // 2]
                m = m_new
            np.testing.assert_allclose(o / l, ref[bi, 0, h], rtol=0, atol=1e-14)


# The pages print the float32-vs-float64 error of causal attention on
# randn(8, 2048, 128) (golden file).  The oracle, run as the float64
# reference of that experiment, must show float32 errors of the same size:
# a wrong mask, scale or operand would make them O(1).
def test_fp32_error_scale_matches_printed_experiment():
    golden = {}
    with open("tests/golden/online_softmax_fp32.txt") as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, val = line.split()
                golden[name] = float(val)
    torch.manual_seed(0)
    H, N, D = 8, 2048, 128
    q, k, v = (torch.randn(H, N, D) for _ in range(3))
    # the oracle in its paged form: one sequence of N rows, N query rows
    to_cache = lambda t: np.ascontiguousarray(
        t.numpy().reshape(H, N // 16, 16, D).transpose(1, 0, 2, 3))
    kc, vc = to_cache(k), to_cache(v)
    table = np.arange(N // 16, dtype=np.int32)[None]
    qp = np.ascontiguousarray(q.numpy().transpose(1, 0, 2)[None])  # [1, N, H, D]
    ref = oracle.paged_attention(qp, kc, vc, table, np.array([N], np.int32),
                                 1 / math.sqrt(D), "f32")[0].transpose(1, 0, 2)
    s = q @ k.transpose(-1, -2) / D ** 0.5
    mask = torch.ones(N, N, dtype=torch.bool).triu(1)
    std = torch.softmax(s.masked_fill(mask, float("-inf")), dim=-1) @ v
    err = float(np.abs(std.double().numpy() - ref).max())
    printed = golden["standard_fp32"]
    # same experiment, same seed: the error reproduces the printed value
    # (8.70e-07) up to the BLAS's summation order
    assert abs(err - printed) < 0.05 * printed, (err, printed)


# 8. Greedy speculative verification reproduces plain greedy decoding
#    ("Inference part 2", section "Speculative decoding": "the output is
#    identical to greedy decoding with the target alone").
def test_greedy_speculative_equals_greedy():
    from tests.toy_decoder import ToyDecoder, greedy, speculative
    prompt = [3, 17, 5, 9, 30, 2, 11]
    n = 40
    ref = greedy(ToyDecoder(seed=3), prompt, n)
    rng = np.random.default_rng(1)

    def propose(tokens, k):
        # the true continuation with ~30 % of the drafts corrupted
        pos = len(tokens)
        out = []
        for i in range(k):
            t = ref[pos + i] if pos + i < len(ref) else 0
            out.append(int(rng.integers(48)) if rng.random() < 0.3 else t)
        return out

    got, passes, acc = speculative(ToyDecoder(seed=3), prompt, n, propose, 4)
    assert got == ref
    assert passes < n and acc > 0  # drafts were actually accepted


# ---- tree verification (Medusa tree attention, "Inference part 2") -------
def random_tree(Q, rng):
    parents = [-1] + [int(rng.integers(0, j)) for j in range(1, Q)]
    from tests.toy_decoder import ancestor_masks
    return parents, ancestor_masks(parents)


def test_tree_chain_mask_is_causal_verify():
    wl = W.Workload("tree chain", 3, 8, 2, 64, "bf16", context_lens=[9, 40, 77],
                    num_queries=6, seed=101)
    b = appended(wl)
    chain = np.array([(2 << j) - 1 for j in range(6)], dtype=np.uint64)
    np.testing.assert_array_equal(
        oracle.tree_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                              wl.softmax_scale, "bf16", chain), run(b))


@pytest.mark.parametrize("Q", [2, 7, 33, 64])
def test_tree_paged_equals_dense_twin(Q):
    rng = np.random.default_rng(Q)
    wl = W.Workload("tree", 3, 8, 2, 64, "f32", context_lens=[Q, Q + 5, Q + 100],
                    num_queries=Q, seed=102 + Q)
    b = appended(wl)
    masks = np.stack([random_tree(Q, rng)[1] for _ in range(3)])
    o1 = oracle.tree_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                               wl.softmax_scale, "f32", masks)
    o2 = twin.tree_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                             wl.softmax_scale, "f32", masks)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_tree_node_equals_decode_on_its_path():
    """Node j of a tree sees exactly the cache and its ancestors: moving its
    path's rows in front of it and decoding gives the same output."""
    rng = np.random.default_rng(5)
    Q = 9
    parents, masks = random_tree(Q, rng)
    wl = W.Workload("tree path", 1, 4, 2, 64, "f32", context_lens=[50], num_queries=Q,
                    seed=103)
    b = appended(wl)
    tree = oracle.tree_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                                 wl.softmax_scale, "f32", masks)
    L, base = 50, 50 - Q
    k = twin.gather_sequence(b.k_cache, b.block_table[0], L)
    v = twin.gather_sequence(b.v_cache, b.block_table[0], L)
    for j in range(Q):
        path = [kk for kk in range(Q) if (int(masks[j]) >> kk) & 1]
        rows = list(range(base)) + [base + kk for kk in path]
        n = len(rows)
        nb = -(-n // 16)
        kc = np.full((nb, 2, 16, 64), np.nan, np.float32)
        vc = np.full_like(kc, np.nan)
        for r, src in enumerate(rows):
            kc[r // 16, :, r % 16] = k[src]
            vc[r // 16, :, r % 16] = v[src]
        dec = oracle.paged_attention(np.ascontiguousarray(b.q[:, j]), kc, vc,
                                     np.arange(nb, dtype=np.int32)[None],
                                     np.array([n], np.int32), wl.softmax_scale, "f32")
        np.testing.assert_allclose(tree[0, j], dec[0, 0], rtol=0, atol=1e-13)


def test_tree_speculative_equals_greedy():
    """Verifying a candidate tree and keeping the longest accepted path
    reproduces plain greedy decoding ("Inference part 2", Medusa)."""
    from tests.toy_decoder import ToyDecoder, greedy, tree_speculative
    prompt = [3, 17, 5, 9, 30, 2, 11]
    n = 40
    ref = greedy(ToyDecoder(seed=3), prompt, n)
    rng = np.random.default_rng(2)

    def propose_tree(tokens):
        # two candidates per level, one of them the true continuation half
        # of the time; level d's nodes hang off the first node of level d-1
        pos = len(tokens)
        toks, pars = [], []
        prev = 0
        for d in range(3):
            truth = ref[pos + d] if pos + d < len(ref) else 0
            first = len(toks) + 1
            for c in range(2):
                good = c == 0 and rng.random() < 0.7
                toks.append(truth if good else int(rng.integers(48)))
                pars.append(prev)
            prev = first
        return toks, pars

    got, passes = tree_speculative(ToyDecoder(seed=3), prompt, n, propose_tree)
    assert got == ref
    assert passes < n
