// attn_mla.cu -- multi-head latent attention (MLA) decode over a paged latent
// cache, on the tensor cores (mma.sync).
//
// What it computes ("Inference part 1", section "Smaller KV caches: MQA, GQA
// and MLA": the cached latent vectors act as both keys and values once the
// up-projections are absorbed, multi-query attention with one large shared
// head; "KV cache, prefill va decode", section 04: d_c = 512 latent values
// plus d_h^R = 64 rotary key values per token).  A cache row is
// [c (512) ; k_rope (DR = 0 or 64)], rows paged through the block table.
// For query head h (q_h = [q_c ; q_r], absorbed and rotated by the caller):
//   score_{h,i} = scale q_h . row_i             (over all 512 + DR values)
//   out_h       = sum_i softmax_i(score_h) c_i  (the 512 latent values)
// so each row is read from HBM once and used as key and as value.
//
// One CTA per (sequence, 16 query heads, split); 9 warps:
//   warps 0-7  compute: column group cg = warp / 4 holds heads 8 cg .. 8 cg + 7
//              (the MMA's N = 8), quarter qw = warp % 4 owns value dims
//              128 qw .. 128 qw + 127;
//   warp 8     TMA producer: each block's 16 rows (DR = 64: 9 panels of
//              128 bytes, 128-byte swizzle) into a ring of NS stages.
// Per block, in the transposed orientation of the decode kernels (keys on M):
//   partial S^T[16 x 8] = K[16 x W/4] . Q^T[W/4 x 8] over the warp's quarter
//   of the W = 512 + DR score dims (16-value steps qw, qw + 4, ...: one per
//   128-byte panel, at the same swizzled offset); the four quarters of a column group meet
//   in shared memory and are summed in a fixed order, so all four warps hold
//   the same scores, maxima and weights;
//   online softmax with a lazy reference maximum, in log2 units ("Inference
//   part 1", section "FlashAttention");
//   O^T[128 x 8] += V^T[128 x 16] . P^T[16 x 8] over the warp's value dims,
//   V being the first 512 values of the same staged rows (P as high part and
//   remainder, two MMAs, so that rounding P costs no accuracy).
// Rows past the context get -inf scores and their V^T fragments are zeroed;
// a bad block id is recorded and its rows masked.  Every wait is bounded.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace mla {

constexpr int kLatent = 512;                         // d_c
constexpr int kHeads = 16;                           // query heads per CTA
constexpr int kGroups = 2;                           // column groups of 8 heads
constexpr int kQuarters = 4;                         // warps per column group
constexpr int kComputeWarps = kGroups * kQuarters;
constexpr int kProducerWarp = kComputeWarps;
constexpr int kThreads = (kComputeWarps + 1) * 32;   // 288
constexpr int kVTiles = kLatent / kQuarters / 16;    // 8 value m-tiles per warp
constexpr float kRescaleSlack = 8.f;                 // weights stay below 2^8

template <int DR, int NS> struct Geom {
  static constexpr int kWidth = kLatent + DR;                 // values per cache row
  static constexpr int kPanels = kWidth / 64;                 // 128-byte panels
  static constexpr int kPanelBytes = kBlockSize * 128;
  static constexpr int kTileBytes = kPanels * kPanelBytes;    // one block
  static constexpr int kSteps = kWidth / 16;                  // score k-steps
  static constexpr int kQSteps = kSteps / kQuarters;          // a warp's share: 8 or 9
  static constexpr int kChains = kQSteps % 3 == 0 ? 3 : 4;    // accumulator chains
  static constexpr int kXOff = NS * kTileBytes;               // score partials
  static constexpr int kXBytes = 2 * kGroups * kQuarters * 32 * 16;
  static constexpr int kOutStride = kLatent + 4;              // staged output row (floats)
  static constexpr int kBytes = kXOff + kXBytes;
  static_assert(kSteps % kQuarters == 0, "score steps split evenly");
  static_assert(kHeads * kOutStride * 4 <= kXOff, "the output stage fits in the ring");
};

// Byte offset of 16-bit element (row, d), d a multiple of 8, in a block
// copied panel by panel with the 128-byte swizzle (chunk k of a 128-byte
// line sits at k ^ (line & 7)).
__device__ __forceinline__ uint32_t tile_off(int row, int d) {
  const int bo = 2 * d;
  return (bo >> 7) * (kBlockSize * 128) + row * 128 + ((((bo & 127) >> 4) ^ (row & 7)) << 4);
}

// Named barrier of one column group's four warps (ids 1 and 2).
__device__ __forceinline__ void group_sync(int cg) {
  if (cg == 0)
    asm volatile("bar.sync 1, 128;" ::: "memory");
  else
    asm volatile("bar.sync 2, 128;" ::: "memory");
}

template <typename T, int DR, int NS>
__global__ void __launch_bounds__(kThreads, 2)
    attn_mla_kernel(const __grid_constant__ CUtensorMap cmap, const AttnParams p) {
  using G = Geom<DR, NS>;
  // The next kernel of the stream (the merge kernel, or the next call's
  // attention) may be scheduled now; it waits for this grid.  This kernel is
  // itself launched as a programmatic dependent of the one before it, so
  // before touching global memory it waits for that one to complete.
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  __shared__ uint64_t full[NS], empty[NS];
  __shared__ volatile int s_abort;
  __shared__ float s_lse[kHeads];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int split = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const SeqExtent ext = seq_extent(p, b, split == 0 && hg == 0 && threadIdx.x == 0);
  const int L = ext.L;
  const int blk_begin = split * p.split_blocks;
  if (split > 0 && blk_begin >= ext.nblk) return;  // this sequence has fewer splits
  const int n_my = max(min(blk_begin + p.split_blocks, ext.nblk) - blk_begin, 0);
  const int32_t *table =
      p.block_table + static_cast<int64_t>(b) * p.max_blocks_per_seq + blk_begin;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kComputeWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // Online-softmax state of this thread's two columns (heads 8 cg + 2c, +1)
  // and its O^T fragments (value dims 128 qw + 16 mt + g, + 8).
  float o[kVTiles][4];
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
#pragma unroll
  for (int mt = 0; mt < kVTiles; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  const int cg = warp >> 2, qw = warp & 3;

  if (warp == kProducerWarp) {
    // ---- TMA producer ----------------------------------------------------------
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      int next = n_my > 0 ? ld_keep(table) : 0;  // each entry loaded one block ahead
      for (int i = 0; i < n_my; ++i) {
        const int s = i % NS;
        const int v = next;
        if (i + 1 < n_my) next = ld_keep(table + i + 1);
        if (i >= NS && !mbar_wait_bounded(smem_u32(&empty[s]), ((i / NS) - 1) & 1)) ok = false;
        if (!ok || s_abort) break;
        const bool bad = v < 0 || static_cast<int64_t>(v) >= p.num_blocks;
        if (bad) record_error(p.err, PKV_DEVERR_BLOCK_ID);
        const uint32_t bar = smem_u32(&full[s]);
        mbar_arrive_expect_tx(bar, G::kTileBytes);
        if (p.tile_box) {  // the block's 16 latent rows in one copy
          tma_load_5d(sbase + s * G::kTileBytes, &cmap, bar, 0, 0, 0, 0, bad ? 0 : v);
        } else {
#pragma unroll
          for (int pn = 0; pn < G::kPanels; ++pn)
            tma_load_4d(sbase + s * G::kTileBytes + pn * G::kPanelBytes, &cmap, bar, pn * 64, 0,
                        0, bad ? 0 : v);
        }
        issued = i + 1;
      }
      if (!ok) {
        s_abort = 1;
        record_error(p.err, PKV_DEVERR_TIMEOUT);
      }
      if (s_abort) {  // copies in flight when the CTA gave up: a bounded chance to land
        for (int k = max(0, issued - NS); k < issued; ++k)
          mbar_wait_bounded(smem_u32(&full[k % NS]), (k / NS) & 1);
      }
    }
  } else {
    // ---- compute warps ----------------------------------------------------------
    // Q^T fragments of this warp's score steps (B operand: k = row value, n = head).
    const int64_t qrow = static_cast<int64_t>(b) * p.num_heads + hg * kHeads + cg * 8 + g;
    const T *qp = reinterpret_cast<const T *>(p.q) + qrow * G::kWidth;
    uint32_t qf[G::kQSteps][2];
#pragma unroll
    for (int kk = 0; kk < G::kQSteps; ++kk) {
      const int d = (kk * kQuarters + qw) * 16 + 2 * c;  // score step 4 kk + qw
      qf[kk][0] = *reinterpret_cast<const uint32_t *>(qp + d);
      qf[kk][1] = *reinterpret_cast<const uint32_t *>(qp + d + 8);
    }
    float4 *xs = reinterpret_cast<float4 *>(smem + G::kXOff);
    // table entries of blocks 32 j .. 32 j + 31, one per lane (bad-block flags)
    auto entries = [&](int j) {
      const int i = 32 * j + lane;
      return i < n_my ? ld_keep(table + i) : 0;
    };
    int tab = entries(0);
    bool aborted = false;
    for (int i = 0; i < n_my; ++i) {
      const int s = i % NS;
      const uint32_t tile = sbase + s * G::kTileBytes;
      const int key0 = (blk_begin + i) * kBlockSize;
      if (i > 0 && (i & 31) == 0) tab = entries(i >> 5);
      const int v = __shfl_sync(kFull, tab, i & 31);
      const bool bad = v < 0 || static_cast<int64_t>(v) >= p.num_blocks;
      // once any warp or the producer has given up, no warp waits again
      aborted = __any_sync(kFull, aborted || s_abort != 0);
      if (!aborted && !__all_sync(kFull, mbar_wait_bounded(smem_u32(&full[s]), (i / NS) & 1))) {
        aborted = true;
        s_abort = 1;
        if (lane == 0) record_error(p.err, PKV_DEVERR_TIMEOUT);
      }
      // partial scores over this warp's quarter of the row (steps qw, qw + 4, ...)
      const uint32_t kbase = tile + tile_off(lane & 15, qw * 16 + (lane >> 4) * 8);
      // V^T fragments: rows (lane & 7) + 8 (lane >> 4), value dims 128 qw + 16 mt
      // + 8 h (h = bit 3 of the lane), in panel 2 qw + mt / 4; their 16-byte chunk
      // 2 (mt % 4) + h sits at (2 (mt % 4)) ^ h ^ (row & 7), 2 (mt % 4) being even
      const int vrow = (lane & 7) + ((lane >> 4) << 3);
      const uint32_t vbase = tile + 2 * qw * G::kPanelBytes + vrow * 128;
      const uint32_t vx = static_cast<uint32_t>((((lane >> 3) & 1) ^ (vrow & 7)) << 4);
      float part[4] = {0.f, 0.f, 0.f, 0.f};
      if (!aborted) {
        float acc[G::kChains][4];
#pragma unroll
        for (int ch = 0; ch < G::kChains; ++ch) acc[ch][0] = acc[ch][1] = acc[ch][2] = acc[ch][3] = 0.f;
        // step 4 kk + qw covers values 64 kk + 16 qw ..: panel kk, the same
        // swizzled 16-byte chunk in every panel
#pragma unroll
        for (int kk = 0; kk < G::kQSteps; ++kk) {
          uint32_t a[4];
          ldsm_x4(a, kbase + kk * G::kPanelBytes);
          Mma<T>::run(acc[kk % G::kChains], a, qf[kk][0], qf[kk][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float t = acc[0][e];
#pragma unroll
          for (int ch = 1; ch < G::kChains; ++ch) t += acc[ch][e];
          part[e] = t;
        }
      }
      // the four quarters meet (every warp of the group passes here each block)
      float4 *xg = xs + ((i & 1) * kGroups + cg) * kQuarters * 32;
      xg[qw * 32 + lane] = make_float4(part[0], part[1], part[2], part[3]);
      group_sync(cg);
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < kQuarters; ++w) {
        const float4 x = xg[w * 32 + lane];
        sc[0] += x.x;
        sc[1] += x.y;
        sc[2] += x.z;
        sc[3] += x.w;
      }
      const bool live = !aborted;
      if (live) {
        // scaled scores; rows past the context or in a bad block: -inf
        const bool need_mask = bad || key0 + kBlockSize > L;
        bool above = false;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float t = sc[e] * p.scale_log2;
          if (need_mask && (bad || key0 + g + ((e >> 1) << 3) >= L)) t = -INFINITY;
          sc[e] = t;
          above |= t > m[e & 1] + kRescaleSlack;
        }
        // lazy reference maximum: raised (rescaling l and O) only when a
        // score passes it by more than the slack; O / l does not depend on it
        if (__any_sync(kFull, above)) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float mx = fmaxf(sc[e], sc[e + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
            const float m_new = fmaxf(m[e], mx);
            const float corr = ex2(m[e] - (m_new == -INFINITY ? 0.f : m_new));
            l[e] *= corr;
            m[e] = m_new;
#pragma unroll
            for (int mt = 0; mt < kVTiles; ++mt) {
              o[mt][e] *= corr;
              o[mt][e + 2] *= corr;
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float mu = m[e] == -INFINITY ? 0.f : m[e];
          const float p0 = ex2(sc[e] - mu), p1 = ex2(sc[e + 2] - mu);
          l[e] += p0 + p1;
          sc[e] = p0;
          sc[e + 2] = p1;
        }
        // P^T operand fragments: high part and rounding remainder
        const uint32_t h01 = Mma<T>::pack(sc[0], sc[1]), h23 = Mma<T>::pack(sc[2], sc[3]);
        float r0, r1, r2, r3;
        Mma<T>::unpack(h01, r0, r1);
        Mma<T>::unpack(h23, r2, r3);
        const uint32_t ph0 = movm_t(h01), ph1 = movm_t(h23);
        const uint32_t pl0 = movm_t(Mma<T>::pack(sc[0] - r0, sc[1] - r1));
        const uint32_t pl1 = movm_t(Mma<T>::pack(sc[2] - r2, sc[3] - r3));
        // V^T columns (keys) past the context: zeroed, so that NaN-filled
        // rows never enter an MMA
        const int nv = bad ? 0 : L - key0;
        const uint32_t km0 = (2 * c < nv ? 0x0000ffffu : 0u) | (2 * c + 1 < nv ? 0xffff0000u : 0u);
        const uint32_t km8 =
            (2 * c + 8 < nv ? 0x0000ffffu : 0u) | (2 * c + 9 < nv ? 0xffff0000u : 0u);
        // value tiles four at a time: the high parts, then the remainders, so
        // that no MMA waits on the one just issued to its accumulator
#pragma unroll
        for (int m0 = 0; m0 < kVTiles; m0 += 4) {
          uint32_t a[4][4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int mt = m0 + w;
            ldsm_x4_t(a[w], vbase + (mt >> 2) * G::kPanelBytes + ((32 * (mt & 3)) ^ vx));
            a[w][0] &= km0;
            a[w][1] &= km0;
            a[w][2] &= km8;
            a[w][3] &= km8;
          }
#pragma unroll
          for (int w = 0; w < 4; ++w) Mma<T>::run(o[m0 + w], a[w], ph0, ph1);
#pragma unroll
          for (int w = 0; w < 4; ++w) Mma<T>::run(o[m0 + w], a[w], pl0, pl1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));  // this warp is done with the stage
    }
    // row sums over the 8 lanes of a column
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float t = l[e];
      t += __shfl_xor_sync(kFull, t, 4);
      t += __shfl_xor_sync(kFull, t, 8);
      t += __shfl_xor_sync(kFull, t, 16);
      l[e] = t;
    }
  }

  // ---- epilogue: O / l staged per head in shared memory, then written out ----
  __syncthreads();  // every stage consumed: the ring becomes the output stage
  float *ost = reinterpret_cast<float *>(smem);
  if (warp < kComputeWarps) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int col = cg * 8 + 2 * c + (e & 1);
      const float inv = l[e & 1] > 0.f ? 1.f / l[e & 1] : 0.f;
#pragma unroll
      for (int mt = 0; mt < kVTiles; ++mt)
        ost[col * G::kOutStride + qw * 128 + mt * 16 + g + ((e >> 1) << 3)] = o[mt][e] * inv;
    }
    if (qw == 0 && g == 0) {
#pragma unroll
      for (int e = 0; e < 2; ++e)
        s_lse[cg * 8 + 2 * c + e] = l[e] > 0.f ? m[e] + __log2f(l[e]) : -INFINITY;
    }
  }
  __syncthreads();
  const bool direct = p.num_splits == 1;
  const int64_t row0 = static_cast<int64_t>(b) * p.num_heads + hg * kHeads;
  for (int idx = threadIdx.x; idx < kHeads * (kLatent / 4); idx += kThreads) {
    const int h = idx / (kLatent / 4), d0 = (idx - h * (kLatent / 4)) * 4;
    const float4 x = *reinterpret_cast<const float4 *>(&ost[h * G::kOutStride + d0]);
    const int64_t row = row0 + h;
    if (direct) {
      T *dst = reinterpret_cast<T *>(p.out) + row * kLatent + d0;
      dst[0] = from_float<T>(x.x * p.out_scale);
      dst[1] = from_float<T>(x.y * p.out_scale);
      dst[2] = from_float<T>(x.z * p.out_scale);
      dst[3] = from_float<T>(x.w * p.out_scale);
    } else {
      *reinterpret_cast<float4 *>(&p.part_o[(row * p.num_splits + split) * kLatent + d0]) = x;
      if (d0 == 0) p.part_lse[row * p.num_splits + split] = s_lse[h];
    }
  }
}

// ---- host side -----------------------------------------------------------------
using MlaLaunch = cudaError_t (*)(const CUtensorMap &, const AttnParams &, dim3, cudaStream_t);

template <typename T, int DR, int NS>
cudaError_t launch_t(const CUtensorMap &cmap, const AttnParams &p, dim3 grid,
                     cudaStream_t stream) {
  // a programmatic dependent of the kernel before it (see the kernel's entry)
  return launch_kernel(true, attn_mla_kernel<T, DR, NS>, grid, kThreads,
                       Geom<DR, NS>::kBytes + 1024, stream, cmap, p);
}

template <typename T, int DR, int NS> bool info_t(KernelInfo *info, MlaLaunch *launch) {
  info->func = reinterpret_cast<const void *>(&attn_mla_kernel<T, DR, NS>);
  info->threads = kThreads;
  info->warps = kThreads / 32;
  info->stages = NS;
  info->smem = Geom<DR, NS>::kBytes + 1024;  // + alignment slack
  *launch = &launch_t<T, DR, NS>;
  return true;
}

// `stages`: ring depth 3, 4 or 5 blocks (0: 4, two CTAs per SM with 18 KB rows).
template <typename T, int DR> bool pick_stages(int stages, KernelInfo *info, MlaLaunch *launch) {
  switch (stages == 0 ? 4 : stages) {
    case 3: return info_t<T, DR, 3>(info, launch);
    case 4: return info_t<T, DR, 4>(info, launch);
    case 5: return info_t<T, DR, 5>(info, launch);
    default: return false;
  }
}

bool pick(pkv_dtype dtype, int rope_dim, int stages, KernelInfo *info, MlaLaunch *launch) {
  if (dtype == PKV_BF16) {
    if (rope_dim == 64) return pick_stages<__nv_bfloat16, 64>(stages, info, launch);
    if (rope_dim == 0) return pick_stages<__nv_bfloat16, 0>(stages, info, launch);
  } else if (dtype == PKV_F16) {
    if (rope_dim == 64) return pick_stages<__half, 64>(stages, info, launch);
    if (rope_dim == 0) return pick_stages<__half, 0>(stages, info, launch);
  }
  return false;
}

// ---- split-K merge of the 512-wide latent outputs -----------------------------
// The Flash-Decoding reduction ("Inference part 1", section "FlashDecoding")
// of the partials this kernel leaves per (row, split), [row][split]: split s
// holds O_s / l_s and lse_s = m_s + log2(l_s); with M = max_s lse_s,
//   out = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M).
// One CTA per output row (a (sequence, head) pair), warp w taking head dims
// 128 w .. 128 w + 127 (four a lane): every warp reads the row's log-sum-exps
// (lane s the split s, 32 at a time), takes their maximum and weights by
// shuffles, and accumulates its dims with eight splits' vectors in flight --
// no block barrier, and the 1,024 rows of the DeepSeek-V2-shaped step in one
// wave.  (A CTA per row with its warps sharing the splits and meeting in
// shared memory took 11.5 us cold there; a warp per row, 12.4 us.)  A
// programmatic dependent of the attention kernel: nothing is read before
// pdl_wait.
constexpr int kMergeWarps = kMlaLatent / 128;  // 4
template <typename T>
__global__ void __launch_bounds__(kMergeWarps * 32) mla_merge_kernel(const AttnParams p) {
  constexpr int D = kMlaLatent;  // 512
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  const int b = static_cast<int>(row / p.num_heads);
  const SeqExtent ext = seq_extent(p, b, false);
  int ns = (ext.nblk + p.split_blocks - 1) / p.split_blocks;
  ns = ns < 1 ? 1 : (ns > p.num_splits ? p.num_splits : ns);
  const int64_t first = row * p.num_splits;
  auto lse_of = [&](int s) -> float { return s < ns ? __ldcg(p.part_lse + first + s) : -INFINITY; };
  const float l0 = lse_of(lane);
  float M = l0;
  for (int s0 = 32; s0 < ns; s0 += 32) M = fmaxf(M, lse_of(s0 + lane));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  const int dim = 128 * warp + 4 * lane;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < ns; s0 += 32) {
      const float w_mine = ex2((s0 == 0 ? l0 : lse_of(s0 + lane)) - M);  // 0 for -inf
      wsum += w_mine;
      const int n = min(32, ns - s0);
      for (int t0 = 0; t0 < n; t0 += 8) {
        float4 v[8];
        float w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          w[u] = __shfl_sync(kFull, w_mine, (t0 + u) & 31);
          if (t0 + u >= n) w[u] = 0.f;
          v[u] = w[u] > 0.f ? __ldcg(reinterpret_cast<const float4 *>(
                                  p.part_o + (first + s0 + t0 + u) * D + dim))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          acc.x = fmaf(w[u], v[u].x, acc.x);
          acc.y = fmaf(w[u], v[u].y, acc.y);
          acc.z = fmaf(w[u], v[u].z, acc.z);
          acc.w = fmaf(w[u], v[u].w, acc.w);
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(kFull, wsum, o);
  const float inv = wsum > 0.f ? p.out_scale / wsum : 0.f;
  T *dst = reinterpret_cast<T *>(p.out) + row * D + dim;
  dst[0] = from_float<T>(acc.x * inv);
  dst[1] = from_float<T>(acc.y * inv);
  dst[2] = from_float<T>(acc.z * inv);
  dst[3] = from_float<T>(acc.w * inv);
}

}  // namespace mla

cudaError_t mla_merge_launch(pkv_dtype dtype, const AttnParams &p, cudaStream_t stream) {
  const int64_t nrows = static_cast<int64_t>(p.batch) * p.num_heads;
  if (nrows == 0) return cudaSuccess;
  if (nrows > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(nrows));
  switch (dtype) {
    case PKV_BF16:
      return launch_kernel(true, mla::mla_merge_kernel<__nv_bfloat16>, grid,
                           mla::kMergeWarps * 32, 0, stream, p);
    case PKV_F16:
      return launch_kernel(true, mla::mla_merge_kernel<__half>, grid, mla::kMergeWarps * 32, 0,
                           stream, p);
    default: return cudaErrorInvalidValue;
  }
}

bool mla_kernel_info(pkv_dtype dtype, int rope_dim, int stages, KernelInfo *info) {
  mla::MlaLaunch launch = nullptr;
  return mla::pick(dtype, rope_dim, stages, info, &launch);
}

cudaError_t mla_launch(pkv_dtype dtype, int rope_dim, int stages, const CUtensorMap &cmap,
                       const AttnParams &p, dim3 grid, cudaStream_t stream) {
  KernelInfo info;
  mla::MlaLaunch launch = nullptr;
  if (!mla::pick(dtype, rope_dim, stages, &info, &launch)) return cudaErrorInvalidValue;
  return launch(cmap, p, grid, stream);
}

}  // namespace pkv
