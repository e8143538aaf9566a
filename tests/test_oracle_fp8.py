"""Pins of the FP8 E4M3 KV-cache oracle ("Inference part 2", sections
"Number formats" and "KV cache quantization"; one float32 scale per cache
tensor, round to nearest even with saturation at +-448)."""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import twin
from paged_kv_cache_18_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "number_formats.txt")


def _formats():
    rows = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            name, bits, s, e, m, largest = line.split()
            rows[name] = (int(bits), int(s), int(e), int(m), float(largest))
    return rows


def test_e4m3_matches_printed_format_table():
    bits, s, e, m, largest = _formats()["FP8_E4M3"]
    assert (bits, s, e, m) == (8, 1, 4, 3)
    o = oracle.default()
    values = np.array([o.e4m3_value(c) for c in range(256)])
    finite = values[np.isfinite(values)]
    assert finite.max() == largest and finite.min() == -largest
    assert np.isnan(values).sum() == 2          # S.1111.111, no infinity
    assert len(set(finite.tolist())) == 253     # +0 and -0 compare equal


def test_e4m3_decode_matches_library_cast():
    o = oracle.default()
    ours = np.array([o.e4m3_value(c) for c in range(256)])
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(ours, lib)
    np.testing.assert_array_equal(ours, twin.e4m3_values())


def test_e4m3_encode_rounding_and_saturation():
    o = oracle.default()
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * s
                        for s in (1e-3, 0.1, 1, 30, 300)])
    inr = np.abs(x) <= 448
    ours = np.array([o.e4m3_encode(v) for v in x[inr]])
    lib = torch.from_numpy(x[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, lib)
    # saturation, NaN, signed zero
    assert o.e4m3_encode(1e6) == 0x7E and o.e4m3_encode(-449.0) == 0xFE
    assert o.e4m3_encode(float("nan")) == 0x7F
    assert o.e4m3_encode(0.0) == 0x00 and o.e4m3_encode(-0.0) == 0x80
    # ties go to the even code: 1 + 1/16 lies halfway between codes 0x38 (1.0)
    # and 0x39 (1.125); 1 + 3/16 between 0x39 and 0x3A
    assert o.e4m3_encode(1.0625) == 0x38 and o.e4m3_encode(1.1875) == 0x3A


def _fp8_batch(wl, k_scale, v_scale):
    """Seeded batch whose cache is quantised to e4m3 codes by the oracle's
    append of every row (new rows appended separately)."""
    b = W.make_batch(wl, poison=False)
    NB, Hkv, bs, D = b.k_cache.shape
    kc = np.zeros((NB, Hkv, bs, D), np.uint8)
    vc = np.zeros_like(kc)
    # every slot of every block: quantise the whole float cache in one append
    all_slots = np.arange(NB * bs, dtype=np.int64)
    kf = np.ascontiguousarray(b.k_cache.transpose(0, 2, 1, 3).reshape(NB * bs, Hkv, D))
    vf = np.ascontiguousarray(b.v_cache.transpose(0, 2, 1, 3).reshape(NB * bs, Hkv, D))
    oracle.kv_append_fp8(kc, vc, kf, vf, all_slots, wl.dtype, k_scale, v_scale)
    return b, kc, vc


def test_fp8_append_is_elementwise_quantisation():
    wl = W.Workload("fp8 append", 3, 4, 2, 64, "bf16", context_lens=[5, 20, 33], seed=31)
    b = W.make_batch(wl)
    NB, Hkv, bs, D = b.k_cache.shape
    kc = np.zeros((NB, Hkv, bs, D), np.uint8)
    vc = np.zeros_like(kc)
    oracle.kv_append_fp8(kc, vc, b.k_new, b.v_new, b.slot_mapping, "bf16", 0.0123, 0.02)
    o = oracle.default()
    kn = twin.widen(b.k_new, "bf16").astype(np.float32)
    for t, slot in enumerate(b.slot_mapping):
        for h in range(Hkv):
            got = kc[slot // bs, h, slot % bs]
            want = [o.e4m3_encode(np.float32(x) / np.float32(0.0123)) for x in kn[t, h]]
            np.testing.assert_array_equal(got, want)
            # round trip within half a code step (relative 2^-4)
            back = twin.e4m3_values()[got] * 0.0123
            assert np.all(np.abs(back - kn[t, h]) <= np.abs(kn[t, h]) * 2.0 ** -4 + 2.0 ** -10 * 0.0123)


@pytest.mark.parametrize("Q,q_dtype", [(1, "bf16"), (5, "bf16"), (1, "f32"), (3, "f16")])
def test_fp8_attention_equals_dense_twin(Q, q_dtype):
    wl = W.Workload("fp8 attn", 3, 8, 2, 128, q_dtype, context_lens=[Q, 40, 300],
                    num_queries=Q, seed=32 + Q)
    b, kc, vc = _fp8_batch(wl, 0.0123, 0.017)
    o1 = oracle.default().paged_attention_fp8(b.q, kc, vc, b.block_table, b.context_lens,
                                              wl.softmax_scale, q_dtype, 0.0123, 0.017)
    o2 = twin.contiguous_attention_fp8(b.q, kc, vc, b.block_table, b.context_lens,
                                       wl.softmax_scale, q_dtype, 0.0123, 0.017)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_fp8_attention_with_power_of_two_scale_equals_bf16_oracle():
    """A power-of-two scale makes every dequantised value exact in bf16: the
    fp8 oracle must then equal the bf16 oracle bit for bit on that cache."""
    wl = W.Workload("fp8 pow2", 2, 8, 2, 64, "bf16", context_lens=[17, 90], num_queries=2,
                    seed=33)
    b, kc, vc = _fp8_batch(wl, 2.0 ** -6, 2.0 ** -5)
    vals = twin.e4m3_values()
    kb = W.round_f32_to_bf16_bits((vals[kc] * 2.0 ** -6).astype(np.float32))
    vb = W.round_f32_to_bf16_bits((vals[vc] * 2.0 ** -5).astype(np.float32))
    fp8 = oracle.default().paged_attention_fp8(b.q, kc, vc, b.block_table, b.context_lens,
                                               wl.softmax_scale, "bf16", 2.0 ** -6, 2.0 ** -5)
    bf = oracle.paged_attention(b.q, kb, vb, b.block_table, b.context_lens, wl.softmax_scale,
                                "bf16")
    np.testing.assert_array_equal(fp8, bf)
