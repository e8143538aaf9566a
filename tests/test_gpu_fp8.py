"""GPU parity of the FP8 E4M3 KV cache: the quantising append bit for bit
against the oracle's, and attention over the code caches against the
float64 oracle (keys and values dequantised as code * tensor scale)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_18_gb300 as pkv
from paged_kv_cache_18_gb300 import workloads as W
from tests.gpu_util import TORCH_DT, assert_close_fp8, dev_tensor, host_f64, tuning

pytestmark = pytest.mark.gpu

K_SCALE, V_SCALE = 0.0123, 0.0171


def run_fp8(wl, split_blocks=0, k_scale=K_SCALE, v_scale=V_SCALE, kernel=0, stages=0,
            q_gain=None):
    b = W.make_batch(wl)
    if q_gain is not None:
        # rescale each query row by its own gain (exactly representable range
        # tests of the per-row power-of-two shift into f16)
        qf = W.storage_to_f64(b.q, wl.dtype).astype(np.float32)
        qf = qf * np.asarray(q_gain, dtype=np.float32).reshape(1, 1, -1, 1)
        b.q = W.to_storage(qf, wl.dtype).reshape(b.q.shape)
    kc, vc = W.fp8_caches(b, k_scale, v_scale)
    dev = "cuda"
    dkc, dvc = torch.from_numpy(kc).to(dev), torch.from_numpy(vc).to(dev)
    kn, vn = dev_tensor(b.k_new, wl.dtype, dev), dev_tensor(b.v_new, wl.dtype, dev)
    slots = torch.from_numpy(b.slot_mapping).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.kv_append_fp8(kn, vn, dkc, dvc, slots, k_scale, v_scale, error_word=err)
    q = dev_tensor(b.q, wl.dtype, dev)
    if wl.num_queries == 1:
        q = q[:, 0].contiguous()
    out = pkv.paged_attention_fp8(q, dkc, dvc, torch.from_numpy(b.block_table).to(dev),
                                  torch.from_numpy(b.context_lens).to(dev), k_scale, v_scale,
                                  scale=wl.softmax_scale, max_context_len=b.max_context_len,
                                  split_blocks=split_blocks, error_word=err, kernel=kernel,
                                  stages=stages)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the quantising append, bit for bit
    oracle.kv_append_fp8(kc, vc, b.k_new, b.v_new, b.slot_mapping, wl.dtype, k_scale, v_scale)
    np.testing.assert_array_equal(dkc.cpu().numpy(), kc)
    np.testing.assert_array_equal(dvc.cpu().numpy(), vc)
    ref = oracle.paged_attention_fp8(b.q, kc, vc, b.block_table, b.context_lens,
                                     wl.softmax_scale, wl.dtype, k_scale, v_scale)
    got = host_f64(out if wl.num_queries > 1 else out[:, None], wl.dtype)
    return assert_close_fp8(got, ref, wl.dtype, wl.name)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("Q,Hq,Hkv", [(1, 8, 8), (1, 8, 2), (5, 8, 2), (2, 4, 1)])
def test_fp8_append_and_attention(dtype, D, Q, Hq, Hkv):
    lens = [max(Q, 1), 16, 17, 33, 250, 1000]
    wl = W.Workload(f"fp8 {dtype} D{D} Q{Q} {Hq}/{Hkv}", len(lens), Hq, Hkv, D, dtype,
                    context_lens=lens, num_queries=Q, seed=800 + D + Q + Hq)
    run_fp8(wl)


# The tensor-core kernel (16-bit q) and the CUDA-core kernel, explicitly.
@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D,Q,Hq,Hkv", [(128, 1, 8, 8), (128, 1, 32, 8), (128, 5, 32, 8),
                                        (128, 3, 40, 40), (256, 1, 8, 2), (256, 4, 4, 2),
                                        (128, 7, 12, 2)])
def test_fp8_kernels(kernel, dtype, D, Q, Hq, Hkv):
    lens = [Q, 15, 16, 47, 129, 700, 2100]
    wl = W.Workload(f"fp8 k{kernel} {dtype} D{D} Q{Q} {Hq}/{Hkv}", len(lens), Hq, Hkv, D, dtype,
                    context_lens=lens, num_queries=Q, seed=860 + D + 3 * Q + Hq + kernel)
    run_fp8(wl, kernel=kernel)


# Four and five column groups over FP8 codes (25 to 40 query rows per KV
# head in one CTA), with and without splits.
@pytest.mark.parametrize("Q,Hq,Hkv,cg", [(4, 32, 4, 4), (5, 32, 4, 5), (9, 12, 3, 5)])
@pytest.mark.parametrize("split_blocks", [0, 3])
def test_fp8_wide_column_groups(Q, Hq, Hkv, cg, split_blocks):
    lens = [Q, Q + 1, Q + 15, Q + 33, 250, 700]
    p = pkv.plan(len(lens), Q, Hq, Hkv, 128, max(lens), "fp8", kernel=2)
    assert p["row_chunks"] == 1 and p["threads_per_cta"] == 32 * cg
    wl = W.Workload(f"fp8 cg{cg} Q{Q} {Hq}/{Hkv} sb{split_blocks}", len(lens), Hq, Hkv, 128,
                    "bf16", context_lens=lens, num_queries=Q, seed=1500 + Q + Hq + split_blocks)
    run_fp8(wl, kernel=2, split_blocks=split_blocks)


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("split_blocks", [1, 3, 16])
def test_fp8_splits(kernel, split_blocks):
    wl = W.Workload("fp8 split", 4, 32, 8, 128, "bf16", context_lens=[1, 200, 1500, 3000],
                    seed=830 + split_blocks)
    run_fp8(wl, split_blocks=split_blocks, kernel=kernel)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("Q,Hq,Hkv", [(1, 8, 8), (3, 32, 8), (5, 32, 8), (2, 8, 1)])
def test_fp8_mma_stage_depths(D, Q, Hq, Hkv):
    lens = [Q, 16, 17, 50, 257, 1000]
    accepted = []
    for stages in range(1, 13):
        try:
            pkv.plan(len(lens), Q, Hq, Hkv, D, max(lens), "fp8", kernel=2, stages=stages)
        except pkv.PkvError:
            continue
        accepted.append(stages)
        wl = W.Workload(f"fp8 stages {stages} D{D} Q{Q}", len(lens), Hq, Hkv, D, "bf16",
                        context_lens=lens, num_queries=Q, seed=900 + D + stages + Q)
        run_fp8(wl, kernel=2, stages=stages)
    assert len(accepted) == 2, accepted  # a shallow and a deep ring per tile shape


@pytest.mark.parametrize("kernel", [1, 2])
def test_fp8_query_range(kernel):
    # rows of very large and very small queries: the tensor-core kernel
    # shifts each row by its own power of two into f16 range
    gains = [3.0e4, 1.0e-6, 1.0, 2.0 ** 40, 2.0 ** -60, 0.0, 7.5, 1.0e8]
    wl = W.Workload("fp8 q range", 3, 8, 2, 128, "bf16", context_lens=[5, 64, 517],
                    seed=890)
    run_fp8(wl, kernel=kernel, q_gain=gains)


def test_fp8_mma_rejects_f32_queries():
    wl = W.Workload("fp8 f32 mma", 2, 8, 2, 128, "f32", context_lens=[20, 40], seed=891)
    with pytest.raises(pkv.PkvError):
        run_fp8(wl, kernel=2)


def test_fp8_auto_picks_tensor_cores():
    assert pkv.plan(4, 1, 32, 8, 128, 2048, "fp8")["kernel"] == 2


def test_fp8_saturation_and_scales():
    # a small scale pushes x / scale past 448: codes saturate, results still match
    wl = W.Workload("fp8 sat", 3, 8, 2, 128, "bf16", context_lens=[10, 90, 300], seed=840)
    run_fp8(wl, k_scale=0.002, v_scale=1.0)


def test_fp8_rejected_by_16bit_entry_points():
    wl = W.Workload("fp8 rej", 1, 4, 4, 128, "bf16", context_lens=[20], seed=841)
    b = W.make_batch(wl)
    kc, vc = W.fp8_caches(b, 1.0, 1.0)
    L = pkv.binding.lib()
    st = L.pkv_paged_decode_attention(16, 16, 16, 16, 16, 2, 16, 20, 1, 4, 4, 128, 16, 10, 0.1,
                                      3, None, 0, None, None, None)
    assert st == 1


# Two KV blocks per warp iteration over FP8 caches (rings of 4 / 6 stages
# for one column group, 8 / 12 for three).
@pytest.mark.parametrize("D,Q,Hq,Hkv,stages", [(128, 1, 8, 8, 0), (128, 1, 32, 8, 6),
                                               (128, 5, 32, 8, 0), (256, 1, 8, 8, 4),
                                               (128, 3, 16, 4, 0)])
@pytest.mark.parametrize("split_blocks", [0, 3])
def test_fp8_two_blocks_per_iteration(D, Q, Hq, Hkv, stages, split_blocks):
    lens = [Q, 15, 16, 17, 47, 129, 701]
    wl = W.Workload(f"fp8 kb2 D{D} Q{Q} {Hq}/{Hkv}", len(lens), Hq, Hkv, D, "bf16",
                    context_lens=lens, num_queries=Q, seed=1500 + D + Q + Hq + split_blocks)
    with tuning(blocks_per_iter=2):
        run_fp8(wl, kernel=2, stages=stages, split_blocks=split_blocks)
