"""Pins of the MLA decode oracle (``oracle/mla.py``), none of which re-types
its formula:

* absorbed attention equals attention with every head's keys and values
  recomputed from the latents through random up-projections (the identity
  behind the absorption in "Inference part 1", section "Smaller KV caches:
  MQA, GQA and MLA", whose code checks the same equality);
* without a rotary part it is multi-query attention with K = V = the latents,
  i.e. the C oracle (O1) with one KV head;
* one cached row returns that row's latent exactly; equal latents return
  that latent whatever the rotary keys (the rotary part reaches the scores,
  never the output);
* two rows against the closed form of a two-way softmax;
* the physical block order is irrelevant (paging is an indirection);
* planted mistakes in a copy of the oracle's source are caught.
"""
import math
import pathlib

import numpy as np
import pytest

import oracle
from oracle import mla

BS = 16


def paged(rows_per_seq, width, rng, dtype=np.float64, shuffle=True, extra_blocks=3):
    """A [NB, BS, width] cache holding each sequence's rows in shuffled
    blocks, its block table and lengths."""
    lens = [r.shape[0] for r in rows_per_seq]
    nblk = [-(-L // BS) for L in lens]
    NB = sum(nblk) + extra_blocks
    perm = rng.permutation(NB) if shuffle else np.arange(NB)
    cache = rng.standard_normal((NB, BS, width)).astype(dtype)
    table = np.zeros((len(lens), max(nblk)), dtype=np.int32)
    at = 0
    for b, rows in enumerate(rows_per_seq):
        for n in range(nblk[b]):
            phys = perm[at]
            at += 1
            table[b, n] = phys
            chunk = rows[n * BS:(n + 1) * BS]
            cache[phys, :chunk.shape[0]] = chunk
    return cache, table, np.asarray(lens, dtype=np.int32)


def test_absorbed_attention_equals_recomputed_keys_and_values():
    rng = np.random.default_rng(0)
    H, dh, dv, d_c, d_r = 4, 16, 12, 32, 8
    w_uk = rng.standard_normal((H, dh, d_c)) / math.sqrt(d_c)
    w_uv = rng.standard_normal((H, dv, d_c)) / math.sqrt(d_c)
    scale = 1.0 / math.sqrt(dh + d_r)
    seqs, expect, qs = [], [], []
    for L in (1, 15, 16, 37, 70):
        c = rng.standard_normal((L, d_c))
        k_rope = rng.standard_normal((L, d_r))
        q_nope = rng.standard_normal((H, dh))
        q_rope = rng.standard_normal((H, d_r))
        seqs.append(np.concatenate([c, k_rope], axis=1))
        qs.append(mla.absorb_query(q_nope, q_rope, w_uk))
        expect.append(mla.attention_recomputed(q_nope, q_rope, c, k_rope, w_uk, w_uv, scale))
    cache, table, lens = paged(seqs, d_c + d_r, rng)
    out = mla.mla_decode(np.stack(qs), cache, table, lens, d_c, scale, "f64")
    for b in range(len(seqs)):
        got = mla.expand_output(out[b], w_uv)
        np.testing.assert_allclose(got, expect[b], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_without_a_rotary_part_it_is_mqa_over_the_latents(dtype):
    """d_r = 0: one KV head whose keys and values are both the latents,
    computed by the C oracle from the same storage."""
    rng = np.random.default_rng(1)
    H, d_c = 8, 64
    lens = [1, 17, 40, 100]
    seqs = [rng.standard_normal((L, d_c)).astype(np.float32) for L in lens]
    cache32, table, lens_a = paged(seqs, d_c, rng, dtype=np.float32)
    q32 = rng.standard_normal((len(lens), H, d_c)).astype(np.float32)
    if dtype == "bf16":
        # storage: the upper 16 bits (truncation keeps the values exact in both)
        cache = (cache32.view(np.uint32) >> 16).astype(np.uint16)
        q = (q32.view(np.uint32) >> 16).astype(np.uint16)
    else:
        cache, q = cache32, q32
    scale = 0.125
    got = mla.mla_decode(q, cache, table, lens_a, d_c, scale, dtype)
    kv = np.ascontiguousarray(cache[:, None])  # [NB, 1, BS, d_c]
    ref = oracle.paged_attention(q, kv, kv, table, lens_a, scale, dtype)[:, 0]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_one_row_returns_its_latent_and_equal_latents_ignore_the_rotary_keys():
    rng = np.random.default_rng(2)
    H, d_c, d_r = 5, 24, 8
    row = rng.standard_normal((1, d_c + d_r))
    c_bar = rng.standard_normal(d_c)
    same = np.concatenate([np.tile(c_bar, (45, 1)), rng.standard_normal((45, d_r)) * 3], axis=1)
    cache, table, lens = paged([row, same], d_c + d_r, rng)
    q = rng.standard_normal((2, H, d_c + d_r)) * 2
    out = mla.mla_decode(q, cache, table, lens, d_c, 0.3, "f64")
    np.testing.assert_array_equal(out[0], np.tile(row[0, :d_c], (H, 1)))
    np.testing.assert_allclose(out[1], np.tile(c_bar, (H, 1)), rtol=1e-14, atol=1e-14)


def test_two_rows_closed_form():
    """softmax over two scores s0, s1: weight of row 1 = 1 / (1 + e^(s0 - s1))."""
    rng = np.random.default_rng(3)
    d_c, d_r = 6, 2
    rows = rng.standard_normal((2, d_c + d_r))
    q = rng.standard_normal((1, 1, d_c + d_r))
    scale = 0.7
    s0 = scale * sum(q[0, 0, k] * rows[0, k] for k in range(d_c + d_r))
    s1 = scale * sum(q[0, 0, k] * rows[1, k] for k in range(d_c + d_r))
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    want = (1 - w1) * rows[0, :d_c] + w1 * rows[1, :d_c]
    cache, table, lens = paged([rows], d_c + d_r, rng)
    got = mla.mla_decode(q, cache, table, lens, d_c, scale, "f64")[0, 0]
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-15)


def test_block_order_is_irrelevant():
    rng = np.random.default_rng(4)
    d_c, d_r, H = 32, 8, 3
    seqs = [rng.standard_normal((L, d_c + d_r)) for L in (33, 64, 5)]
    q = rng.standard_normal((3, H, d_c + d_r))
    a = mla.mla_decode(q, *paged(seqs, d_c + d_r, np.random.default_rng(10), shuffle=False),
                       d_c, 0.2, "f64")
    b = mla.mla_decode(q, *paged(seqs, d_c + d_r, np.random.default_rng(11), shuffle=True),
                       d_c, 0.2, "f64")
    np.testing.assert_array_equal(a, b)


def test_empty_sequence_gives_zeros():
    rng = np.random.default_rng(5)
    cache, table, lens = paged([rng.standard_normal((3, 10))], 10, rng)
    lens[0] = 0
    out = mla.mla_decode(rng.standard_normal((1, 2, 10)), cache, table, lens, 8, 1.0, "f64")
    assert not out.any()


# ---- planted mistakes ----------------------------------------------------------
MUTATIONS = {
    "scale dropped": ("s = (qb @ rows.T) * scale", "s = (qb @ rows.T)"),
    "rotary part left out of the scores": ("s = (qb @ rows.T) * scale",
                                           "s = (qb[:, :d_c] @ rows[:, :d_c].T) * scale"),
    "value slice taken from the end": ("out[b] = w @ rows[:, :d_c]",
                                       "out[b] = w @ rows[:, -d_c:]"),
    "block table ignored": ("cache[np.asarray(table_row[:n_blocks], dtype=np.int64)]",
                            "cache[np.arange(n_blocks)]"),
    "softmax over heads": ("w /= w.sum(axis=1, keepdims=True)", "w /= w.sum(axis=0, keepdims=True)"),
    "last row dropped": ("gather_latents(ckv_cache, block_table[b], L)",
                         "gather_latents(ckv_cache, block_table[b], max(L - 1, 1))"),
}

PINS = [test_absorbed_attention_equals_recomputed_keys_and_values,
        lambda: test_without_a_rotary_part_it_is_mqa_over_the_latents("f32"),
        test_one_row_returns_its_latent_and_equal_latents_ignore_the_rotary_keys,
        test_two_rows_closed_form, test_block_order_is_irrelevant]


def _mutant(old, new):
    src = pathlib.Path(mla.__file__).read_text()
    assert src.count(old) == 1, old
    src = src.replace(old, new).replace("from .twin import widen", "")
    ns = {"widen": oracle.twin.widen, "__name__": "mla_mutant"}
    exec(compile(src, "mla_mutant", "exec"), ns)
    return ns


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    ns = _mutant(*MUTATIONS[name])
    for fn in ("gather_latents", "mla_decode"):
        monkeypatch.setattr(mla, fn, ns[fn])
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, f"no pin caught: {name}"
