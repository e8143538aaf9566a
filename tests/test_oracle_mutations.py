"""Planted mistakes in the C oracle must be caught by its pins.

Each mutation below is a plausible slip in ``oracle/pkv_oracle.c`` (a wrong
index, a dropped term, a flipped sign, a transposed operand).  The test
compiles a mutated copy into a temporary library, runs a battery of pins on
it, and requires at least one pin to fail, while the unmutated oracle passes
all of them.  Every mutation keeps memory accesses in bounds.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import twin
from paged_kv_cache_18_gb300 import workloads as W

MUTATIONS = {
    "block index i%bs": ("block_table[(int64_t)b * max_blocks + i / bs]",
                         "block_table[(int64_t)b * max_blocks + i % bs]"),
    "row in block off by one": ("+ i % bs) * D;", "+ (i + 1) % bs) * D;"),
    "gqa map h%Hkv": ("const int g = h / (Hq / Hkv);", "const int g = h % Hkv;"),
    "mask off by one": ("(int64_t)L - Q + 1 + j;", "(int64_t)L - Q + j;"),
    "dropped scale": ("scores[i] = scale * dot;", "scores[i] = dot;"),
    "flipped exp sign": ("exp(scores[i] - m)", "exp(m - scores[i])"),
    "no normalisation": ("out_row[d] /= denom;", "out_row[d] /= 1.0;"),
    "K used as V": ("widen(v_cache, v_base + d, dtype)", "widen(k_cache, v_base + d, dtype)"),
    "query row ignored": ("(((int64_t)b * Q + j) * Hq + h) * D;",
                          "(((int64_t)b * Q + 0) * Hq + h) * D;"),
    "append slot offset": ("offset = slot % bs;", "offset = (slot + 1) % bs;"),
}

PIN_CASES = [
    W.Workload("gqa spec", 3, 8, 2, 64, "bf16", context_lens=[5, 21, 48],
               num_queries=3, seed=14),
    W.Workload("mha f32", 2, 3, 3, 64, "f32", context_lens=[1, 37], seed=15),
]


def _battery(orc) -> list:
    """Names of the pins ``orc`` fails."""
    failed = []
    for wl in PIN_CASES:
        b = W.make_batch(wl)
        truth = W.make_batch(wl, poison=False)
        orc.kv_append(b.k_cache, b.v_cache, b.k_new, b.v_new, b.slot_mapping, wl.dtype)
        # append pin: every owned slot now holds the unpoisoned value
        for bi in range(wl.batch):
            L = int(b.context_lens[bi])
            got = twin.gather_sequence(b.k_cache, b.block_table[bi], L)
            want = twin.gather_sequence(truth.k_cache, truth.block_table[bi], L)
            if not np.array_equal(got.view(np.uint8), want.view(np.uint8)):
                failed.append(f"append {wl.name}")
                break
        try:
            out = orc.paged_attention(b.q, b.k_cache, b.v_cache, b.block_table,
                                      b.context_lens, wl.softmax_scale, wl.dtype)
        except ValueError:
            failed.append(f"error {wl.name}")
            continue
        # paged == contiguous twin
        o2 = twin.contiguous_attention(b.q, b.k_cache, b.v_cache, b.block_table,
                                       b.context_lens, wl.softmax_scale, wl.dtype)
        if not np.allclose(out, o2, rtol=0, atol=1e-12):
            failed.append(f"twin {wl.name}")
        # causal prefill by the library routine
        for bi in range(wl.batch):
            L, Q = int(b.context_lens[bi]), wl.num_queries
            k = torch.from_numpy(twin.widen(twin.gather_sequence(b.k_cache, b.block_table[bi], L), wl.dtype))
            v = torch.from_numpy(twin.widen(twin.gather_sequence(b.v_cache, b.block_table[bi], L), wl.dtype))
            qf = torch.zeros(L, wl.num_heads, wl.head_dim, dtype=torch.float64)
            first = max(0, L - Q)
            qf[first:] = torch.from_numpy(twin.widen(b.q[bi], wl.dtype))[Q - (L - first):]
            o = torch.nn.functional.scaled_dot_product_attention(
                qf.transpose(0, 1)[None], k.transpose(0, 1)[None], v.transpose(0, 1)[None],
                is_causal=True, scale=wl.softmax_scale,
                enable_gqa=wl.num_heads != wl.num_kv_heads)[0].transpose(0, 1)
            rows = [j for j in range(Q) if L - Q + j >= 0]
            want = np.stack([o[L - Q + j].numpy() for j in rows])
            if not np.allclose(out[bi, rows], want, rtol=0, atol=1e-12):
                failed.append(f"sdpa {wl.name}")
                break
    return failed


def test_unmutated_oracle_passes_battery():
    assert _battery(oracle.default()) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(oracle.SOURCE).read()
    assert old in src, f"mutation anchor for {name!r} not found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(mutated), str(tmp_path / "libmutant.so"))
    failed = _battery(oracle.Oracle(lib))
    assert failed, f"planted mistake {name!r} passed every pin"


# ---- tree verification --------------------------------------------------
TREE_MUTATIONS = {
    "tree bit off by one": ("((mask >> (i - base)) & 1u)", "((mask >> (i - base + 1)) & 1u)"),
    "tree drops a cached row": ("seen[i] = (i < base) ||", "seen[i] = (i + 1 < base) ||"),
    "tree ignores mask": ("seen[i] = (i < base) || ((mask >> (i - base)) & 1u);",
                          "seen[i] = 1;"),
}


def _tree_battery(orc) -> list:
    from tests.toy_decoder import ancestor_masks
    failed = []
    rng = np.random.default_rng(9)
    wl = W.Workload("tree m", 3, 8, 2, 64, "f32", context_lens=[9, 40, 77], num_queries=6,
                    seed=120)
    b = W.make_batch(wl)
    orc.kv_append(b.k_cache, b.v_cache, b.k_new, b.v_new, b.slot_mapping, "f32")
    chain = np.array([(2 << j) - 1 for j in range(6)], dtype=np.uint64)
    causal = orc.paged_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                                 wl.softmax_scale, "f32")
    try:
        got = orc.tree_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                                 wl.softmax_scale, "f32", chain)
        if not np.array_equal(got, causal):
            failed.append("chain == causal")
        parents = [-1] + [int(rng.integers(0, j)) for j in range(1, 6)]
        masks = ancestor_masks(parents)
        got = orc.tree_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                                 wl.softmax_scale, "f32", masks)
        want = twin.tree_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                                   wl.softmax_scale, "f32", masks)
        if not np.allclose(got, want, rtol=0, atol=1e-12):
            failed.append("twin")
    except ValueError:
        failed.append("error")
    return failed


def test_unmutated_tree_oracle_passes_battery():
    assert _tree_battery(oracle.default()) == []


@pytest.mark.parametrize("name", sorted(TREE_MUTATIONS))
def test_tree_mutation_is_caught(name, tmp_path):
    old, new = TREE_MUTATIONS[name]
    src = open(oracle.SOURCE).read()
    assert old in src, f"mutation anchor for {name!r} not found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(mutated), str(tmp_path / "libmutant.so"))
    assert _tree_battery(oracle.Oracle(lib)), f"planted mistake {name!r} passed every pin"


# ---- FP8 E4M3 cache -------------------------------------------------------
FP8_MUTATIONS = {
    "e4m3 exponent bias": ("v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 11);"),
    "e4m3 subnormal scale": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "ties to odd": ("(err == best_err && (c & 1u) == 0u)", "(err == best_err && (c & 1u) == 1u)"),
    "overflow to NaN": ("if (a > 448.0) return sign | 0x7eu;", "if (a > 448.0) return sign | 0x7fu;"),
    "k scale dropped": ("* (oracle_e4m3_value(k_cache[kb + d]) * k_scale)",
                        "* (oracle_e4m3_value(k_cache[kb + d]))"),
}


def _fp8_battery(orc) -> list:
    failed = []
    vals = np.array([orc.e4m3_value(c) for c in range(256)])
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    if not np.array_equal(vals, lib, equal_nan=True):
        failed.append("decode vs library")
    x = np.array([1.0625, 1.1875, -3.25, 500.0, 1e-3, 0.3], dtype=np.float32)
    ours = [orc.e4m3_encode(v) for v in x]
    want = [0x38, 0x3A, torch.tensor([-3.25]).to(torch.float8_e4m3fn).view(torch.uint8).item(),
            0x7E, torch.tensor([1e-3]).to(torch.float8_e4m3fn).view(torch.uint8).item(),
            torch.tensor([0.3]).to(torch.float8_e4m3fn).view(torch.uint8).item()]
    if ours != want:
        failed.append("encode")
    wl = W.Workload("fp8 m", 2, 4, 2, 64, "bf16", context_lens=[17, 40], seed=44)
    b = W.make_batch(wl, poison=False)
    NB, Hkv, bs, D = b.k_cache.shape
    kc = (np.arange(NB * Hkv * bs * D) * 37 % 126).astype(np.uint8).reshape(NB, Hkv, bs, D)
    vc = (np.arange(NB * Hkv * bs * D) * 53 % 126).astype(np.uint8).reshape(NB, Hkv, bs, D)
    got = orc.paged_attention_fp8(b.q, kc, vc, b.block_table, b.context_lens, wl.softmax_scale,
                                  "bf16", 0.03, 0.02)
    want = twin.contiguous_attention_fp8(b.q, kc, vc, b.block_table, b.context_lens,
                                         wl.softmax_scale, "bf16", 0.03, 0.02)
    if not np.allclose(got, want, rtol=0, atol=1e-12):
        failed.append("attention vs twin")
    return failed


def test_unmutated_fp8_oracle_passes_battery():
    assert _fp8_battery(oracle.default()) == []


@pytest.mark.parametrize("name", sorted(FP8_MUTATIONS))
def test_fp8_mutation_is_caught(name, tmp_path):
    old, new = FP8_MUTATIONS[name]
    src = open(oracle.SOURCE).read()
    assert old in src, f"mutation anchor for {name!r} not found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(mutated), str(tmp_path / "libmutant.so"))
    assert _fp8_battery(oracle.Oracle(lib)), f"planted mistake {name!r} passed every pin"
