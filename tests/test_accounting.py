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
