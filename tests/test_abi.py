"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, validates arguments synchronously (nothing reaches CUDA on bad
input), and its launch planner is self-consistent."""
import contextlib
import ctypes
import os
import re

import pytest
import torch

from paged_kv_cache_18_gb300 import binding, build


@contextlib.contextmanager
def tuning(**kw):
    """Extra pkv_options fields for every binding call inside the block."""
    saved = dict(binding.TUNING)
    binding.TUNING.update(kw)
    try:
        yield
    finally:
        binding.TUNING.clear()
        binding.TUNING.update(saved)

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "pkv.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PKV_API[^;(]*?\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_binding_list():
    assert declared_functions() == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_only_the_c_abi_is_exported(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    ours = [l.split()[-1] for l in out.splitlines() if " T " in l and "pkv" in l]
    assert sorted(ours) == declared_functions()


def test_version_and_status_strings(L):
    assert "sm_103a" in binding.version()
    names = [L.pkv_status_string(i).decode() for i in range(8)]
    assert names[0] == "ok" and len(set(names)) == 8
    assert names[6] == "host memory allocation failed" and names[7] == "unknown status"


# --- argument validation (returns before any CUDA call) -------------------
def decode(L, **kw):
    a = dict(out=16, q=16, k=16, v=16, table=16, max_blocks=8, lens=16, max_ctx=100, B=2,
             Hq=8, Hkv=2, D=128, bs=16, NB=10, scale=0.1, dtype=1, ws=None, ws_bytes=0,
             opt=None, err=None, stream=None)
    a.update(kw)
    return L.pkv_paged_decode_attention(a["out"], a["q"], a["k"], a["v"], a["table"],
                                        a["max_blocks"], a["lens"], a["max_ctx"], a["B"],
                                        a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"], a["scale"],
                                        a["dtype"], a["ws"], a["ws_bytes"], a["opt"], a["err"],
                                        a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(out=None), 1), (dict(table=None), 1), (dict(lens=None), 1),
    (dict(Hq=7), 1), (dict(Hkv=0), 1), (dict(D=96), 2), (dict(bs=32), 2), (dict(dtype=9), 1),
    (dict(max_ctx=-1), 1), (dict(max_ctx=8 * 16 + 1), 1), (dict(NB=0), 1),
    (dict(scale=float("nan")), 1), (dict(q=8), 5), (dict(k=24), 5), (dict(B=70000), 2),
])
def test_attention_argument_errors(L, kw, status):
    assert decode(L, **kw) == status


def test_empty_batch_is_a_no_op(L):
    assert decode(L, B=0, q=None, out=None) == 0


def test_spec_verify_argument_errors(L):
    f = L.pkv_spec_verify_attention
    # num_queries = 0 is invalid
    assert f(16, 16, 16, 16, 16, 8, 16, 100, 2, 0, 8, 2, 128, 16, 10, 0.1, 1, None, 0, None,
             None, None) == 1


def test_kv_append_argument_errors(L):
    f = L.pkv_kv_append
    assert f(16, 16, 16, 16, 16, 0, 2, 128, 16, 10, 1, None, None) == 0   # no tokens
    assert f(None, 16, 16, 16, 16, 4, 2, 128, 16, 10, 1, None, None) == 1
    assert f(16, 16, 16, 16, 16, 4, 2, 128, 16, 10, 7, None, None) == 1   # dtype
    assert f(16, 16, 16, 16, 16, 4, 2, 4, 16, 10, 1, None, None) == 2     # 8-byte rows
    assert f(16, 16, 16, 16, 12, 4, 2, 128, 16, 10, 1, None, None) == 5   # slot align
    assert f(16, 16, 16, 24, 16, 4, 2, 128, 16, 10, 1, None, None) == 5


# --- planner (no GPU: explicit SM count) -----------------------------------
def test_plan_kernel_choice():
    p = binding.plan_for(4, 1, 6, 6, 64, 256, torch.float32, num_sms=152)
    assert p["kernel"] == binding.PKV_KERNEL_SIMT
    p = binding.plan_for(32, 1, 40, 40, 128, 2048, torch.bfloat16, num_sms=152)
    assert p["kernel"] == binding.PKV_KERNEL_MMA and p["rows_per_cta"] == 1
    p = binding.plan_for(128, 1, 32, 8, 128, 4096, torch.bfloat16, num_sms=152)
    assert p["kernel"] == binding.PKV_KERNEL_MMA and p["rows_per_cta"] == 4
    # a 10-node tree over four query heads per KV head: 40 rows, one CTA of
    # five column-group warps per (sequence, KV head)
    p = binding.plan_for(16, 10, 32, 8, 128, 8192, torch.bfloat16, num_sms=152)
    assert (p["rows_per_cta"], p["row_chunks"], p["threads_per_cta"]) == (40, 1, 160)
    p = binding.plan_for(16, 11, 32, 8, 128, 8192, torch.bfloat16, num_sms=152)
    assert (p["rows_per_cta"], p["row_chunks"]) == (22, 2)
    with pytest.raises(binding.PkvError):
        binding.plan_for(1, 1, 8, 8, 64, 16, torch.float32, num_sms=152,
                         kernel=binding.PKV_KERNEL_MMA)


@pytest.mark.parametrize("B,Q,Hq,Hkv,D,ctx,dt", [
    (4, 1, 6, 6, 64, 256, torch.float32), (32, 1, 40, 40, 128, 2048, torch.bfloat16),
    (128, 1, 32, 8, 128, 4096, torch.bfloat16), (2, 1, 32, 8, 128, 65536, torch.bfloat16),
    (16, 5, 32, 8, 128, 8192, torch.bfloat16), (3, 7, 64, 2, 64, 1000, torch.float16),
    (1, 1, 128, 1, 256, 300, torch.bfloat16), (5, 3, 16, 2, 256, 70, torch.float32),
    (16, 10, 32, 8, 128, 8192, torch.bfloat16), (3, 9, 12, 3, 128, 500, torch.float16),
    (2, 13, 8, 2, 128, 3000, torch.bfloat16), (4, 33, 8, 8, 64, 900, torch.float16),
])
@pytest.mark.parametrize("kernel", [0, 1])
def test_plan_invariants(B, Q, Hq, Hkv, D, ctx, dt, kernel):
    p = binding.plan_for(B, Q, Hq, Hkv, D, ctx, dt, num_sms=152, kernel=kernel)
    rows = Hq // Hkv * Q
    assert p["rows_per_cta"] * p["row_chunks"] >= rows
    assert (p["rows_per_cta"] - 1) * p["row_chunks"] < rows
    max_blocks = -(-ctx // 16)
    if p["split_target"] > 0:
        # partition from the real lengths, on the device: a flat grid of at
        # most split_target work items, whole waves of resident CTAs, one
        # partial per (item, CTA column), merged by the merge kernel
        T, U = p["split_target"], Hkv * p["row_chunks"]
        assert B <= 32 and p["split_blocks"] == 0 and p["merge_kernel"] == 1
        assert T % (152 * p["ctas_per_sm"]) == 0 and T >= B * U
        assert (p["grid_x"], p["grid_y"], p["grid_z"]) == (T, 1, 1)
        assert p["num_splits"] == max(1, T // U)
        parts = T * p["rows_per_cta"]
        assert p["workspace_bytes"] == (-(-parts * D * 4 // 256) * 256 + -(-parts * 4 // 256) * 256
                                        + -(-(2 * B + 2) * 4 // 256) * 256)
        assert p["smem_bytes"] <= 227 * 1024
        return
    assert p["num_splits"] * p["split_blocks"] >= max_blocks
    assert (p["num_splits"] - 1) * p["split_blocks"] < max(max_blocks, 1)
    assert (p["grid_x"], p["grid_y"], p["grid_z"]) == (p["num_splits"], Hkv * p["row_chunks"], B)
    if p["num_splits"] == 1:
        assert p["workspace_bytes"] == 0
    else:
        o = B * Q * Hq * p["num_splits"] * D * 4
        lse = B * Q * Hq * p["num_splits"] * 4
        fused = p["num_splits"] <= 32 and p["rows_per_cta"] * p["num_splits"] <= 64
        ctr = B * Hkv * p["row_chunks"] * 4 if fused else 0   # 32-bit arrival counters
        assert p["workspace_bytes"] == (-(-o // 256) * 256 + -(-lse // 256) * 256
                                        + -(-ctr // 256) * 256)
        assert p["merge_kernel"] == (0 if fused else 1)
    assert p["smem_bytes"] <= 227 * 1024


def test_plan_splits_long_contexts_and_honours_override():
    # 16 (sequence, KV head) pairs cannot fill 152 SMs: split, at most 32
    # ways, the split length from max_context_len
    p = binding.plan_for(2, 1, 32, 8, 128, 65536, torch.bfloat16, num_sms=152)
    assert p["split_target"] == 0 and 16 <= p["num_splits"] <= 32
    # on request, the partition from the real lengths, made on the device
    for waves in (1, 2):
        with tuning(split_waves=waves):
            p = binding.plan_for(2, 1, 32, 8, 128, 65536, torch.bfloat16, num_sms=152)
        assert p["split_target"] == waves * 152 * p["ctas_per_sm"]
        assert p["grid_x"] == p["split_target"]
    with tuning(split_waves=1):   # not for more than 32 sequences
        p = binding.plan_for(33, 1, 32, 8, 128, 65536, torch.bfloat16, num_sms=152)
    assert p["split_target"] == 0 and p["num_splits"] > 1
    p = binding.plan_for(2, 1, 32, 8, 128, 65536, torch.bfloat16, num_sms=152, split_blocks=7)
    assert p["split_blocks"] == 7 and p["num_splits"] == -(-4096 // 7)
    p = binding.plan_for(2, 1, 32, 8, 128, 100, torch.bfloat16, num_sms=152, split_blocks=1000)
    assert p["num_splits"] == 1


def test_plan_does_not_split_when_waves_gain_nothing():
    # 1280 equal units of 128 blocks on 152 SMs x 3 CTAs: 3 waves whole, and
    # 6 waves of 64-block halves: no split
    p = binding.plan_for(32, 1, 40, 40, 128, 2048, torch.bfloat16, num_sms=152, ctas_per_sm=3)
    assert p["num_splits"] == 1 and p["split_target"] == 0
    # 1024 units of up to 256 blocks: 3 waves of 256 against 9 of 64: split
    p = binding.plan_for(128, 1, 32, 8, 128, 4096, torch.bfloat16, num_sms=152, ctas_per_sm=3)
    assert p["num_splits"] == 4 and p["split_blocks"] == 64


def test_plan_caps_split_length_in_bytes():
    # the same KV bytes per split for a one-byte cache: twice the blocks
    p16 = binding.plan_for(128, 1, 32, 8, 128, 4096, torch.bfloat16, num_sms=152, ctas_per_sm=3)
    p8 = binding.plan_for(128, 1, 32, 8, 128, 4096, "fp8", num_sms=152, ctas_per_sm=3)
    assert p8["split_blocks"] == 2 * p16["split_blocks"]


def test_bounded_wait_check_validates_its_arguments(L):
    assert L.pkv_check_bounded_wait(None, 100, None, None) == 1
    assert L.pkv_check_bounded_wait(16, 0, None, None) == 1
    assert L.pkv_check_bounded_wait(16, 10**8, None, None) == 1
    assert L.pkv_check_bounded_wait(18, 100, None, None) == 5   # misaligned error word


def host_step(L, **kw):
    a = dict(out=16, q=16, kn=16, vn=16, k=256, v=256, table=16, max_blocks=8, lens=16,
             max_ctx=100, B=2, Q=1, Hq=8, Hkv=2, D=128, bs=16, NB=10, scale=0.1, dtype=1,
             staging=256, staging_bytes=1 << 20, opt=None, err=None, stream=None)
    a.update(kw)
    return L.pkv_append_attention_host(
        a["out"], a["q"], a["kn"], a["vn"], a["k"], a["v"], a["table"], a["max_blocks"],
        a["lens"], a["max_ctx"], a["B"], a["Q"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"],
        a["scale"], a["dtype"], a["staging"], a["staging_bytes"], a["opt"], a["err"],
        a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(B=0, q=None, out=None, staging=None), 0),        # nothing to do
    (dict(q=None), 1), (dict(out=None), 1), (dict(kn=None), 1), (dict(table=None), 1),
    (dict(lens=None), 1), (dict(Q=0), 1), (dict(B=-1), 1), (dict(max_blocks=0), 1),
    (dict(dtype=3), 1),                                    # FP8 caches: not this call
    (dict(staging=None), 3), (dict(staging=16), 3),        # staging missing / misaligned
])
def test_host_step_argument_errors(L, kw, status):
    assert host_step(L, **kw) == status


def test_host_step_staging_size_argument_errors(L):
    f = L.pkv_host_step_staging_size
    n = ctypes.c_size_t(0)
    assert f(2, 1, 8, 2, 128, 16, 8, 100, 1, None, None) == 1             # no result pointer
    assert f(2, 1, 8, 2, 128, 16, 8, 100, 3, None, ctypes.byref(n)) == 1  # FP8
    assert f(2, 1, 8, 2, 128, 16, 0, 100, 1, None, ctypes.byref(n)) == 1  # no table width


def mla_decode(L, **kw):
    a = dict(out=16, q=16, c=256, table=16, max_blocks=8, lens=16, max_ctx=100, B=2, H=16,
             latent=512, rope=64, bs=16, NB=10, scale=0.1, dtype=1, ws=None, ws_bytes=0,
             opt=None, err=None, stream=None)
    a.update(kw)
    return L.pkv_mla_decode_attention(
        a["out"], a["q"], a["c"], a["table"], a["max_blocks"], a["lens"], a["max_ctx"], a["B"],
        a["H"], a["latent"], a["rope"], a["bs"], a["NB"], a["scale"], a["dtype"], a["ws"],
        a["ws_bytes"], a["opt"], a["err"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(B=0, q=None, out=None), 0),                      # nothing to do
    (dict(q=None), 1), (dict(c=None), 1), (dict(table=None), 1), (dict(lens=None), 1),
    (dict(dtype=9), 1), (dict(NB=0), 1), (dict(max_ctx=8 * 16 + 1), 1),
    (dict(scale=float("nan")), 1), (dict(q=8), 5), (dict(c=24), 5),
    (dict(H=8), 2), (dict(latent=256), 2), (dict(rope=32), 2), (dict(dtype=0), 2),  # f32
    (dict(bs=32), 2),
])
def test_mla_argument_errors(L, kw, status):
    assert mla_decode(L, **kw) == status


def test_mla_append_and_workspace_argument_errors(L):
    f = L.pkv_mla_append
    assert f(16, 16, 16, 0, 576, 16, 10, 1, None, None) == 0      # no tokens
    assert f(None, 16, 16, 4, 576, 16, 10, 1, None, None) == 1
    assert f(16, 16, 16, 4, 4, 16, 10, 1, None, None) == 2        # 8-byte rows
    assert f(16, 24, 16, 4, 576, 16, 10, 1, None, None) == 5      # cache misaligned
    n = ctypes.c_size_t(0)
    g = L.pkv_mla_workspace_size
    assert g(2, 16, 512, 64, 16, 100, 1, None, None) == 1            # no result pointer
    assert g(2, 8, 512, 64, 16, 100, 1, None, ctypes.byref(n)) == 2  # heads
    opt = binding.Options(2, 0, 0, 0, 0, 0, 0, 0)                   # a kernel choice
    assert g(2, 16, 512, 64, 16, 100, 1, ctypes.byref(opt), ctypes.byref(n)) == 2


@pytest.mark.parametrize("B,Q,Hq,Hkv,ctx", [(16, 5, 32, 8, 8192), (1, 1, 32, 8, 100),
                                            (32, 1, 32, 8, 4096), (3, 3, 36, 9, 65536)])
def test_tc_plan_balanced_partition(B, Q, Hq, Hkv, ctx):
    """The tcgen05 kernel's default plan: the balanced partition over one CTA
    per SM, with slots for every CTA plus every unit (a split in slot c + U)."""
    p = binding.plan_for(B, Q, Hq, Hkv, 128, ctx, torch.bfloat16, num_sms=152, kernel=3)
    assert p["kernel"] == 3 and p["stream_k"] == 1 and p["ctas_per_sm"] == 1
    G = 152
    assert p["split_target"] == p["grid_x"] == G and (p["grid_y"], p["grid_z"]) == (1, 1)
    assert p["split_blocks"] == 0 and p["merge_kernel"] == 1
    assert p["num_splits"] == min(G, -(-ctx // 16))
    slots = (G + B * Hkv * p["row_chunks"]) * p["rows_per_cta"]
    assert p["workspace_bytes"] == (-(-slots * 128 * 4 // 256) * 256 + -(-slots * 4 // 256) * 256
                                    + -(-(2 * B + 2) * 4 // 256) * 256)
    # more than 32 sequences, or an explicit split length: the host plan
    p = binding.plan_for(33, Q, Hq, Hkv, 128, ctx, torch.bfloat16, num_sms=152, kernel=3)
    assert p["stream_k"] == 0 and p["split_target"] == 0
    p = binding.plan_for(B, Q, Hq, Hkv, 128, ctx, torch.bfloat16, num_sms=152, kernel=3,
                         split_blocks=64)
    assert p["stream_k"] == 0 and p["split_blocks"] == min(64, -(-ctx // 16))
    with tuning(split_waves=2):   # on request, the whole-item device partition
        p = binding.plan_for(B, Q, Hq, Hkv, 128, ctx, torch.bfloat16, num_sms=152, kernel=3)
    assert p["stream_k"] == 0 and p["split_target"] >= 2 * 152


def _stream_k_pieces_brute(lens, units, ctas, weight):
    """(unit, CTAs whose ranges hold some of its blocks), by walking every
    place of the list: a unit with n blocks is `weight` places of no block,
    then its n blocks."""
    nb = [-(-L // 16) for L in lens]
    T = units * sum(n + weight for n in nb if n > 0)
    owner = []
    for c in range(ctas):
        owner += [c] * (T * (c + 1) // ctas - T * c // ctas)
    assert len(owner) == T
    pieces, x = [], 0
    for b, n in enumerate(nb):
        for u in range(units):
            if n == 0:
                pieces.append((b * units + u, [], x))
                continue
            cs = sorted(set(owner[x + weight:x + weight + n]))
            pieces.append((b * units + u, cs, x + weight))
            x += n + weight
    return pieces, T


@pytest.mark.parametrize("weight", [0, 24])
@pytest.mark.parametrize("lens,units,ctas", [([0, 1, 15, 16, 17, 300, 2000, 5000], 8, 152),
                                             ([40, 40], 8, 152), ([700] * 32, 8, 152),
                                             ([65536, 1, 32768], 9, 152), ([3, 5], 1, 7)])
def test_stream_k_partition_mirror(lens, units, ctas, weight):
    """The balanced partition's arithmetic (the CTA of a place, the slot of a
    split), checked against a place-by-place walk: each unit's splits are the
    CTAs between those of its first and last block whose ranges are not
    empty, the slots c + U are distinct and fit in ctas + units, and the
    splits per unit the byte accounting uses agree."""
    from paged_kv_cache_18_gb300 import accounting
    pieces, T = _stream_k_pieces_brute(lens, units, ctas, weight)
    seen = set()
    for U, cs, first in pieces:
        if not cs:
            continue
        # the CTAs between the first block's and the last's, less those whose
        # range is empty (fewer places than CTAs)
        assert cs == [c for c in range(cs[0], cs[-1] + 1) if T * (c + 1) // ctas > T * c // ctas]
        n = -(-lens[U // units] // 16)
        assert cs[0] == ((first + 1) * ctas - 1) // T and cs[-1] == ((first + n) * ctas - 1) // T
        for c in cs:
            slot = c + U
            assert slot not in seen and slot < ctas + units * len(lens)
            seen.add(slot)
    got = accounting.stream_k_splits(lens, 16, units, ctas, max(lens), 10 ** 6, weight=weight)
    for b in range(len(lens)):
        want = sum(len(cs) for U, cs, _ in pieces if U // units == b) / units
        assert got[b] == want


def test_tc_plan_wide_tile():
    """The tcgen05 kernel serves up to 64 query rows per KV head in one CTA
    (its 64-column tile: one Q^T and one P^T buffer, at most two V stages);
    more rows are cut into row chunks of at most 64."""
    for Q, rows in ((9, 36), (16, 64)):
        p = binding.plan_for(4, Q, 32, 8, 128, 4096, torch.bfloat16, num_sms=152, kernel=3)
        assert (p["rows_per_cta"], p["row_chunks"]) == (rows, 1)
        assert p["smem_bytes"] <= 227 * 1024 and p["warp_tiles"] == 8
    p = binding.plan_for(4, 17, 32, 8, 128, 4096, torch.bfloat16, num_sms=152, kernel=3)
    assert (p["rows_per_cta"], p["row_chunks"]) == (34, 2)
    for st in (1, 2):
        p = binding.plan_for(4, 9, 32, 8, 128, 4096, torch.bfloat16, num_sms=152, kernel=3,
                             stages=st)
        assert p["stages"] == st
    with pytest.raises(binding.PkvError):   # a third V stage does not fit beside it
        binding.plan_for(4, 9, 32, 8, 128, 4096, torch.bfloat16, num_sms=152, kernel=3,
                         stages=3)
