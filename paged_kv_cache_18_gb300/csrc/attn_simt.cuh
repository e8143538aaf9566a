// attn_simt.cuh -- paged decode / speculative-verify attention with CUDA-core
// dot products: the kernel template, shared by the translation units that
// instantiate it (float32 / bfloat16 / float16 caches in attn_simt.cu, FP8
// E4M3 caches in attn_simt_fp8.cu).
//
// Same work split as the tensor-core kernel: one CTA per (sequence, KV head,
// row chunk, split) serving the R query rows that share the KV head, each
// warp owning every W-th block of the split with its own ring of NS stages.
// A block's K tile and V tile (each one contiguous run of 16 rows) arrive by
// one 1-D bulk copy each (cp.async.bulk, completion on an mbarrier), from the
// physical block the table names ("Inference part 1", section
// "PagedAttention").
//
// Lane layout: the 32 lanes form 4 row groups of 8 lanes; a row group takes
// rows g, g + 4, g + 8, g + 12 of the block, and each of its 8 lanes holds
// every 8th 16-byte vector of the row (128 contiguous bytes per quarter warp:
// no bank conflicts).  Scores are reduced over the 8 lanes with shuffles; the
// online softmax ("Inference part 1", section "FlashAttention", m / l / O
// recurrence, in log2 units) runs per row group over 4 rows at a time, and
// the 4 row groups and W warps are merged at the end like chunks of
// Flash-Decoding.  Rows past the context are skipped entirely, so NaN-filled
// unused rows never reach the output.
#pragma once

#include <cuda_fp8.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace simt {

template <typename T> __device__ __forceinline__ void vec_to_float(const uint4 &v, float *f);
template <> __device__ __forceinline__ void vec_to_float<float>(const uint4 &v, float *f) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
template <> __device__ __forceinline__ void vec_to_float<__nv_bfloat16>(const uint4 &v, float *f) {
  unpack2<__nv_bfloat16>(v.x, f[0], f[1]);
  unpack2<__nv_bfloat16>(v.y, f[2], f[3]);
  unpack2<__nv_bfloat16>(v.z, f[4], f[5]);
  unpack2<__nv_bfloat16>(v.w, f[6], f[7]);
}
template <> __device__ __forceinline__ void vec_to_float<__half>(const uint4 &v, float *f) {
  unpack2<__half>(v.x, f[0], f[1]);
  unpack2<__half>(v.y, f[2], f[3]);
  unpack2<__half>(v.z, f[4], f[5]);
  unpack2<__half>(v.w, f[6], f[7]);
}
// 16 e4m3 codes -> their values (exact through half precision).
__device__ __forceinline__ void e4m3x4_to_float(uint32_t w, float *f) {
  const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu),
                                                    __NV_E4M3);
  const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16),
                                                    __NV_E4M3);
  const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
  f[0] = a.x;
  f[1] = a.y;
  f[2] = b.x;
  f[3] = b.y;
}
template <> __device__ __forceinline__ void vec_to_float<E4M3>(const uint4 &v, float *f) {
  e4m3x4_to_float(v.x, f);
  e4m3x4_to_float(v.y, f + 4);
  e4m3x4_to_float(v.z, f + 8);
  e4m3x4_to_float(v.w, f + 12);
}

template <typename T> __device__ __forceinline__ float load_float(const T *p);
template <> __device__ __forceinline__ float load_float<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float load_float<__nv_bfloat16>(const __nv_bfloat16 *p) {
  return __bfloat162float(*p);
}
template <> __device__ __forceinline__ float load_float<__half>(const __half *p) {
  return __half2float(*p);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// TQ: element type of q and out; TC: element type of the caches.
template <typename TQ, typename TC, int D, int R, int W, int NS>
__global__ void __launch_bounds__(W * 32) attn_simt_kernel(const AttnParams p) {
  // The next kernel of the stream (the merge kernel, or the next call's
  // attention) may be scheduled now; it waits for this grid.  This kernel is
  // itself launched as a programmatic dependent of the one before it, so
  // before touching global memory it waits for that one to complete.
  pdl_launch_dependents();
  pdl_wait();
  constexpr int ELT = Elt<TC>::bytes;
  constexpr int RB = D * ELT;             // bytes of one row
  constexpr int TILE = kBlockSize * RB;   // bytes of one (block, kv head) tile
  constexpr int STAGE = 2 * TILE;
  constexpr int VPL = RB / 128;           // 16-byte vectors per lane per row
  constexpr int EV = 16 / ELT;            // elements per vector
  constexpr int EPL = VPL * EV;           // elements per lane per row (= D / 8)
  static_assert(RB % 128 == 0, "row must be a multiple of 128 bytes");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_base + W * NS * STAGE;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = lane >> 3, t = lane & 7;
  const CtaWork wk = cta_work(p);
  if (!wk.active) return;  // a split past its sequence's end (the whole CTA agrees)
  const int kvh = wk.kvh, chunk = wk.chunk, b = wk.b;
  const SeqExtent ext = wk.ext;
  const int L = ext.L;
  const int blk_begin = wk.blk_begin;
  const int nspan = max(wk.blk_end - blk_begin, 0);
  const int n_my = nspan > warp ? (nspan - warp + W - 1) / W : 0;

  // Query rows in registers (this lane's slice of the head dim).
  float qv[R][EPL];
  int lim[R];
  unsigned long long tm[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t row = cta_row_index(p, b, kvh, chunk, r);
    lim[r] = row < 0 ? -1 : cta_row_limit(p, L, chunk, r);
    tm[r] = cta_row_tree_mask(p, b, chunk, r);
    const TQ *qrow = reinterpret_cast<const TQ *>(p.q) + (row < 0 ? 0 : row) * D;
#pragma unroll
    for (int cv = 0; cv < VPL; ++cv)
#pragma unroll
      for (int e = 0; e < EV; ++e)
        qv[r][cv * EV + e] = row < 0 ? 0.f : load_float<TQ>(qrow + (t + 8 * cv) * EV + e);
  }

  float acc[R][EPL];
  float m[R], l[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[r][e] = 0.f;
  }

  const uint32_t my_bars = bar_base + warp * NS * 8;
  const uint32_t my_stages = smem_base + warp * NS * STAGE;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(my_bars + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int32_t *table = p.block_table + static_cast<int64_t>(b) * p.max_blocks_per_seq +
                         blk_begin + warp;
  auto load_entries = [&](int chunk32) -> int {
    const int i = chunk32 * 32 + lane;
    return i < n_my ? ld_keep(table + static_cast<int64_t>(i) * W) : -1;
  };
  int tab_cur = load_entries(0);
  int tab_next = load_entries(1);
  uint32_t bad_mask = 0;
  const uint8_t *kbase = reinterpret_cast<const uint8_t *>(p.k_cache);
  const uint8_t *vbase = reinterpret_cast<const uint8_t *>(p.v_cache);

  auto issue = [&](int i) {
    if ((i & 31) == 0 && i > 0) {
      tab_cur = tab_next;
      tab_next = load_entries((i >> 5) + 1);
    }
    const int v = __shfl_sync(kFull, tab_cur, i & 31);
    const bool bad = v < 0 || static_cast<int64_t>(v) >= p.num_blocks;
    bad_mask = bad ? (bad_mask | (1u << (i & 31))) : (bad_mask & ~(1u << (i & 31)));
    if (lane == 0) {
      if (bad) record_error(p.err, PKV_DEVERR_BLOCK_ID);
      const int64_t phys = bad ? 0 : v;
      const int64_t off = (phys * p.num_kv_heads + kvh) * static_cast<int64_t>(TILE);
      const int s = i % NS;
      const uint32_t bar = my_bars + 8 * s;
      const uint32_t st = my_stages + s * STAGE;
      mbar_arrive_expect_tx(bar, STAGE);
      bulk_g2s(st, kbase + off, TILE, bar);
      bulk_g2s(st + TILE, vbase + off, TILE, bar);
    }
  };

  const int npre = min(NS, n_my);
  for (int i = 0; i < npre; ++i) issue(i);
  int issued = npre;

  bool timed_out = false;
  int landed = 0;
  for (int i = 0; i < n_my; ++i) {
    const int s = i % NS;
    if (!mbar_wait_bounded(my_bars + 8 * s, (i / NS) & 1)) {
      timed_out = true;
      landed = i;
      break;
    }
    const uint32_t ktile = my_stages + s * STAGE;
    const uint32_t vtile = ktile + TILE;
    const int key0 = (blk_begin + warp + i * W) * kBlockSize;
    const bool bad = (bad_mask >> (i & 31)) & 1u;
    if (p.k_new != nullptr && !bad && key0 + kBlockSize > L - p.num_queries) {
      const int64_t phys = __ldg(table + static_cast<int64_t>(i) * W);
      patch_new_rows<D, ELT>(p, ktile, vtile, b, kvh, key0, L, phys, chunk == 0,
                             [](int r, int vec) { return static_cast<uint32_t>(r * RB + vec * 16); });
    }

    // Scores of rows rg, rg+4, rg+8, rg+12 for every query row.
    float sc[4][R];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int row = rg + 4 * k;
      float kf[EPL];
#pragma unroll
      for (int cv = 0; cv < VPL; ++cv)
        vec_to_float<TC>(lds128(ktile + row * RB + (t + 8 * cv) * 16), &kf[cv * EV]);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) d = fmaf(qv[r][e], kf[e], d);
        d += __shfl_xor_sync(kFull, d, 1);
        d += __shfl_xor_sync(kFull, d, 2);
        d += __shfl_xor_sync(kFull, d, 4);
        const bool vis = lim[r] >= 0 && key_visible(p, key0 + row, L, bad, lim[r], tm[r]);
        sc[k][r] = vis ? d * p.scale_log2 : -INFINITY;
      }
    }
    // Online softmax over these 4 rows.
    float pw[4][R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float mx = fmaxf(fmaxf(sc[0][r], sc[1][r]), fmaxf(sc[2][r], sc[3][r]));
      const float m_new = fmaxf(m[r], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = ex2(m[r] - m_use);
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pw[k][r] = ex2(sc[k][r] - m_use);
        sum += pw[k][r];
      }
      l[r] = l[r] * corr + sum;
      m[r] = m_new;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[r][e] *= corr;
    }
    // P V over the rows that exist.
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int row = rg + 4 * k;
      if (!bad && key0 + row < L) {
        float vf[EPL];
#pragma unroll
        for (int cv = 0; cv < VPL; ++cv)
          vec_to_float<TC>(lds128(vtile + row * RB + (t + 8 * cv) * 16), &vf[cv * EV]);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[r][e] = fmaf(pw[k][r], vf[e], acc[r][e]);
      }
    }
    __syncwarp();
    if (i + NS < n_my) {
      issue(i + NS);
      ++issued;
    }
  }
  if (timed_out) {
    if (lane == 0) record_error(p.err, PKV_DEVERR_TIMEOUT);
    for (int k = landed; k < issued; ++k) mbar_wait_bounded(my_bars + 8 * (k % NS), (k / NS) & 1);
  }

  // Merge the 4 row groups of the warp (lanes t, t+8, t+16, t+24).
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float M = fmaxf(m[r], __shfl_xor_sync(kFull, m[r], 8));
    M = fmaxf(M, __shfl_xor_sync(kFull, M, 16));
    const float s = ex2(m[r] - ((M == -INFINITY) ? 0.f : M));
    float lv = l[r] * s;
    lv += __shfl_xor_sync(kFull, lv, 8);
    lv += __shfl_xor_sync(kFull, lv, 16);
    l[r] = lv;
    m[r] = M;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      float a = acc[r][e] * s;
      a += __shfl_xor_sync(kFull, a, 8);
      a += __shfl_xor_sync(kFull, a, 16);
      acc[r][e] = a;
    }
  }

  __syncthreads();
  constexpr int NC = R;
  constexpr int DP = D + 4;
  float *red_o = reinterpret_cast<float *>(smem);
  float *red_m = red_o + W * NC * DP;
  float *red_l = red_m + W * NC;
  float *wscale = red_l + W * NC;
  if (rg == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int cv = 0; cv < VPL; ++cv)
#pragma unroll
        for (int e = 0; e < EV; ++e)
          red_o[(warp * NC + r) * DP + (t + 8 * cv) * EV + e] = acc[r][cv * EV + e];
      if (t == 0) {
        red_m[warp * NC + r] = m[r];
        red_l[warp * NC + r] = l[r];
      }
    }
  }
  __syncthreads();
  cta_epilogue<TQ, D, NC, W, W * 32>(p, red_m, red_l, red_o, wscale, wk);
}

constexpr int kSimtWarps = 4;

using SimtLaunch = cudaError_t (*)(const AttnParams &, dim3, cudaStream_t);

// Stages per warp: about 32 KB of K/V tiles per warp, between 1 and 3.
template <typename TC, int D>
constexpr int simt_stages() {
  constexpr int stage = 2 * kBlockSize * D * Elt<TC>::bytes;
  return (32768 / stage) < 1 ? 1 : ((32768 / stage) > 3 ? 3 : (32768 / stage));
}

template <typename TC, int D, int R>
constexpr size_t simt_smem_bytes() {
  constexpr int kSimtStages = simt_stages<TC, D>();
  constexpr size_t stages = size_t(kSimtWarps) * kSimtStages * 2 * kBlockSize * D * Elt<TC>::bytes;
  constexpr size_t red = (size_t(kSimtWarps) * R * (D + 4) + size_t(3 * kSimtWarps + 2) * R) * 4;
  static_assert(red <= stages, "epilogue scratch must fit in the stage memory");
  return stages + size_t(kSimtWarps) * kSimtStages * 8 + 128;
}

template <typename TQ, typename TC, int D, int R>
KernelInfo simt_info_t() {
  KernelInfo k;
  k.func = reinterpret_cast<const void *>(
      &attn_simt_kernel<TQ, TC, D, R, kSimtWarps, simt_stages<TC, D>()>);
  k.threads = kSimtWarps * 32;
  k.smem = simt_smem_bytes<TC, D, R>();
  k.warps = kSimtWarps;
  k.stages = simt_stages<TC, D>();
  return k;
}

template <typename TQ, typename TC, int D, int R>
cudaError_t simt_launch_t(const AttnParams &p, dim3 grid, cudaStream_t stream) {
  const KernelInfo k = simt_info_t<TQ, TC, D, R>();
  // a programmatic dependent of the kernel before it (with split-K counters,
  // the kernel that zeroes them)
  return launch_kernel(true,
                       attn_simt_kernel<TQ, TC, D, R, kSimtWarps, simt_stages<TC, D>()>, grid,
                       k.threads, k.smem, stream, p);
}

// Query rows per CTA: R * D / 8 registers of query and of accumulator per
// lane, kept <= 64 each.
template <typename TQ, typename TC, int D>
bool simt_pick(int r, KernelInfo *info, SimtLaunch *launch) {
  switch (r) {
    case 1: *info = simt_info_t<TQ, TC, D, 1>(); *launch = &simt_launch_t<TQ, TC, D, 1>; return true;
    case 2: *info = simt_info_t<TQ, TC, D, 2>(); *launch = &simt_launch_t<TQ, TC, D, 2>; return true;
    case 4:
      if (D > 128) return false;
      *info = simt_info_t<TQ, TC, D, (D > 128 ? 1 : 4)>();
      *launch = &simt_launch_t<TQ, TC, D, (D > 128 ? 1 : 4)>;
      return true;
    case 8:
      if (D > 64) return false;
      *info = simt_info_t<TQ, TC, D, (D > 64 ? 1 : 8)>();
      *launch = &simt_launch_t<TQ, TC, D, (D > 64 ? 1 : 8)>;
      return true;
    default: return false;
  }
}

}  // namespace simt
}  // namespace pkv
