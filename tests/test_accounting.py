"""Byte accounting pinned to the KV-sizing numbers the pages print
(golden file ``tests/golden/kv_sizing.txt``)."""
import os

import pytest

from paged_kv_cache_18_gb300 import accounting

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_sizing.txt")


def _rows():
    per_token, per_seq = [], []
    for line in open(GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        f = line.split()
        if f[0] == "SEQ":
            per_seq.append((f[1], *map(int, f[2:7]), float(f[7])))
        else:
            per_token.append((f[0], f[1], *map(int, f[2:6]), float(f[6]), float(f[7])))
    return per_token, per_seq


@pytest.mark.parametrize("row", _rows()[0], ids=lambda r: r[0])
def test_kib_per_token_matches_printed_table(row):
    name, kind, layers, kv_heads, head_dim, bpv, kib, gib128k = row
    got = accounting.kv_bytes_per_token(layers, kv_heads, head_dim, bpv,
                                        latent=(kind == "MLA"))
    assert round(got / 1024, 1) == kib
    assert round(got * 131072 / 1024 ** 3, 2) == gib128k


@pytest.mark.parametrize("row", _rows()[1], ids=lambda r: r[0])
def test_sequence_bytes_match_printed(row):
    name, layers, heads, head_dim, bpv, seq, gb = row
    got = accounting.kv_bytes_per_token(layers, heads, head_dim, bpv) * seq
    assert round(got / 1e9, 2) == gb


def test_attention_bytes_llama2_13b_layer():
    # one layer of the Llama-2-13B-shaped batch: 32 sequences x 2048 rows
    b = accounting.attention_bytes([2048] * 32, 1, 40, 40, 128, 16, 2)
    assert b["kv"] == 32 * 2048 * 40 * 128 * 2 * 2 == 1342177280
    # the per-layer KV of one sequence x 40 layers is the printed 1.68 GB
    assert round(b["kv"] / 32 * 40 / 1e9, 2) == 1.68


# --- the chunked-prefill workload ---------------------------------------------------
def test_prefill_flops_equal_a_brute_force_count_of_visible_pairs():
    from paged_kv_cache_18_gb300 import workloads as W
    wl = W.PrefillWorkload("tiny", 3, 4, 2, 64, "bf16", chunk_lens=[1, 7, 20],
                           prefix_lens=[0, 5, 33], seed=3)
    pairs = 0
    for P, C in zip(wl.prefixes().tolist(), wl.chunks().tolist()):
        L = P + C
        for j in range(C):              # row j sees keys 0 .. L - C + j
            pairs += sum(1 for i in range(L) if i <= L - C + j)
    # two products (QK and PV), a multiply and an add each, per head dim and head
    assert wl.flops() == 4 * wl.num_heads * wl.head_dim * pairs


def test_prefill_batch_layout():
    import numpy as np
    from paged_kv_cache_18_gb300 import workloads as W
    wl = W.PrefillWorkload("tiny", 3, 4, 2, 64, "bf16", chunk_lens=[1, 17, 40],
                           prefix_lens=[15, 0, 33], seed=4)
    b = W.make_prefill_batch(wl)
    assert b.query_start.tolist() == [0, 1, 18, 58]
    assert b.context_lens.tolist() == [16, 17, 73]
    assert b.q.shape == (58, 4, 64) and b.k_new.shape == (58, 2, 64)
    bs = wl.block_size
    for s in range(3):
        C = int(b.query_start[s + 1] - b.query_start[s])
        P = int(b.context_lens[s]) - C
        for j in range(C):
            slot = int(b.slot_mapping[b.query_start[s] + j])
            # the chunk's row j is logical row P + j of sequence s
            assert slot == int(b.block_table[s, (P + j) // bs]) * bs + (P + j) % bs
            # and its slot waits, NaN-filled, for the append
            assert np.isnan(W.storage_to_f64(b.k_cache[slot // bs, :, slot % bs, :],
                                             "bf16")).all()
    # every physical block belongs to at most one sequence
    used = b.block_table[b.block_table >= 0]
    assert len(set(used.tolist())) == used.size
