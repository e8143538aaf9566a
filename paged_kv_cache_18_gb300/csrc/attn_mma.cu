// attn_mma.cu -- paged decode / speculative-verify attention on tensor cores
// (bf16 and fp16 caches).
//
// One CTA serves one (sequence b, KV head, row chunk, split): the NC query
// rows that share the KV head (the group of query heads of grouped-query
// attention x the verified queries), so every K/V byte of a block is read
// from HBM once for all of them ("Inference part 1", section "Smaller KV
// caches: MQA, GQA and MLA": consecutive query heads share one KV head).
//
// Data movement.  Each warp owns the blocks w, w + W, w + 2W, ... of the
// split and a private ring of NS shared-memory stages.  One lane issues, per
// block, tiled TMA copies (cp.async.bulk.tensor) of the block's K and V tiles
// straight from the physical block named by the block table ("Inference part
// 1", section "PagedAttention": the kernel reads the blocks through the
// table), with the 128-byte swizzle so that the ldmatrix reads below are
// bank-conflict free.  Completion is counted on one mbarrier per stage.
//
// Math, per 16-row block, in the transposed orientation (keys on the MMA's
// M side so that a handful of query rows only pad N up to 8):
//   S^T[16 x NC] = K[16 x D] . Q^T[D x NC]          (mma.sync m16n8k16)
//   online softmax over the keys of each column ("Inference part 1",
//   section "FlashAttention", the m / l / O recurrence; "KV cache, prefill
//   va decode", section 07, online softmax), in log2 units;
//   O^T[D x NC] += V^T[D x 16] . P^T[16 x NC]       (P split into a bf16/fp16
//   high and low part, two MMAs, so that rounding P costs no accuracy)
// P^T's operand layout is obtained from S^T's accumulator layout with
// movmatrix.trans.  Rows past the context and masked (verify) entries get
// -inf scores; the V^T fragments of rows past the context are zeroed, so
// NaN-filled unused rows never reach the output.
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// Largest excess (log2 units) of a score over its column's reference max
// before the reference is raised: block weights stay below 2^8.
constexpr float kRescaleSlack = 8.f;

template <int D> struct MmaGeom {
  static constexpr int kParts = D / 64;                 // 128-byte panels per row
  static constexpr int kPanelBytes = kBlockSize * 128;  // 2 KB
  static constexpr int kTileBytes = kParts * kPanelBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;    // K tile + V tile
  static constexpr int kSteps = D / 16;
};

// Byte offset of element (row, d) (d a multiple of 8) in a swizzled tile.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int d) {
  const int part = d >> 6;
  const int chunk = (d & 63) >> 3;
  return part * MmaGeom<D>::kPanelBytes + row * 128 + ((chunk ^ (row & 7)) << 4);
}

// Named barrier over the `count` warps of one block lane (id 1 + lane).
__device__ __forceinline__ void lane_sync(int id, int count) {
  if (count == 1) {
    __syncwarp();
  } else {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count * 32) : "memory");
  }
}

// BL block lanes x CG column groups = BL * CG warps.  Block lane bl owns the
// blocks bl, bl + BL, ... of the split and a ring of NS stages; the CG warps
// of a lane share each staged block, warp cg computing query columns
// 8 cg .. 8 cg + 7.  The lane's first warp issues the copies.
template <typename T, int D, int CG, int BL, int NS>
__global__ void __launch_bounds__(BL * CG * 32)
    attn_mma_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const AttnParams p) {
  using G = MmaGeom<D>;
  constexpr int NC = CG * 8;  // query columns of this CTA (padded)
  constexpr int KS = G::kSteps;
  constexpr int NW = BL * CG;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);
  __shared__ uint64_t bars[BL * NS];  // the stage's copies landed
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bl = warp / CG, cg = warp - (warp / CG) * CG;
  const bool leader = cg == 0;
  const int g = lane >> 2, c = lane & 3;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / p.row_chunks;
  const int chunk = blockIdx.y - kvh * p.row_chunks;
  const int b = blockIdx.z;

  const SeqExtent ext = seq_extent(p, b, split == 0 && chunk == 0 && kvh == 0 &&
                                             threadIdx.x == 0);
  const int L = ext.L;
  const int blk_begin = split * p.split_blocks;
  if (split > 0 && blk_begin >= ext.nblk) return;  // this sequence has fewer splits
  const int blk_end = min(blk_begin + p.split_blocks, ext.nblk);
  const int ns_b = max(1, min(p.num_splits, (ext.nblk + p.split_blocks - 1) / p.split_blocks));
  const int nspan = max(blk_end - blk_begin, 0);
  const int n_my = nspan > bl ? (nspan - bl + BL - 1) / BL : 0;
  const int col0 = cg * 8;

  // Q^T operand fragments of this warp's 8 columns (B operand: k = head dim).
  uint32_t qf[KS][2];
  {
    const int64_t row = cta_row_index(p, b, kvh, chunk, col0 + g);
    const T *qrow = reinterpret_cast<const T *>(p.q) + (row < 0 ? 0 : row) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qf[ks][0] = row < 0 ? 0u : *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 2 * c);
      qf[ks][1] = row < 0 ? 0u : *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + 2 * c);
    }
  }
  // Visible-row limit of the two columns this thread holds.
  int lim[2];
  unsigned long long tm[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    lim[e] = cta_row_limit(p, L, chunk, col0 + 2 * c + e);
    tm[e] = cta_row_tree_mask(p, b, chunk, col0 + 2 * c + e);
  }
  const int mask_from = L - p.num_queries;  // first row some column may not see

  // Online-softmax state.
  float o[KS][4];
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;

  // The lane's ring.
  const uint32_t my_bars = smem_u32(&bars[bl * NS]);
  const uint32_t my_stages = smem_base + bl * NS * G::kStageBytes;
  if (threadIdx.x == 0) s_abort = 0;
  if (leader && lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(my_bars + 8 * s, 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int32_t *table = p.block_table + static_cast<int64_t>(b) * p.max_blocks_per_seq +
                         blk_begin + bl;
  auto load_entries = [&](int chunk32) -> int {
    const int i = chunk32 * 32 + lane;
    return i < n_my ? __ldg(table + static_cast<int64_t>(i) * BL) : -1;
  };
  int tab_cur = load_entries(0);
  int tab_next = load_entries(1);
  uint32_t bad_mask = 0;

  // Track block i's table entry (every warp of the lane), and have the
  // lane's leader issue its copies into stage i % NS.
  auto issue = [&](int i) {
    if ((i & 31) == 0 && i > 0) {
      tab_cur = tab_next;
      tab_next = load_entries((i >> 5) + 1);
    }
    const int v = __shfl_sync(kFull, tab_cur, i & 31);
    const bool bad = v < 0 || static_cast<int64_t>(v) >= p.num_blocks;
    bad_mask = bad ? (bad_mask | (1u << (i & 31))) : (bad_mask & ~(1u << (i & 31)));
    if (leader && lane == 0) {
      if (bad) record_error(p.err, PKV_DEVERR_BLOCK_ID);
      const int phys = bad ? 0 : v;
      const int s = i % NS;
      const uint32_t bar = my_bars + 8 * s;
      const uint32_t st = my_stages + s * G::kStageBytes;
      mbar_arrive_expect_tx(bar, G::kStageBytes);
#pragma unroll
      for (int part = 0; part < G::kParts; ++part)
        tma_load_4d(st + part * G::kPanelBytes, &kmap, bar, part * 64, 0, kvh, phys);
#pragma unroll
      for (int part = 0; part < G::kParts; ++part)
        tma_load_4d(st + G::kTileBytes + part * G::kPanelBytes, &vmap, bar, part * 64, 0, kvh,
                    phys);
    }
  };

  const int npre = min(NS, n_my);
  for (int i = 0; i < npre; ++i) issue(i);
  int issued = npre;

  int consumed = 0;
  bool aborted = false;
  for (int i = 0; i < n_my; ++i) {
    const int s = i % NS;
    // A copy that never lands aborts the CTA (with column groups, through a
    // shared flag): from then on no warp waits or computes, but every warp
    // still takes part in each lane_sync.
    if (!aborted && !mbar_wait_bounded(my_bars + 8 * s, (i / NS) & 1)) {
      aborted = true;
      if (CG > 1) s_abort = 1;
      if (lane == 0) record_error(p.err, PKV_DEVERR_TIMEOUT);
    }
    if (CG > 1 && !aborted) aborted = s_abort != 0;
    const bool live = !aborted;
    if (live) consumed = i + 1;
    const uint32_t ktile = my_stages + s * G::kStageBytes;
    const uint32_t vtile = ktile + G::kTileBytes;
    const int key0 = (blk_begin + bl + i * BL) * kBlockSize;
    const bool bad = (bad_mask >> (i & 31)) & 1u;
    if (p.k_new != nullptr && !bad && key0 + kBlockSize > L - p.num_queries) {
      if (leader && live) {
        const int64_t phys = __ldg(table + static_cast<int64_t>(i) * BL);
        patch_new_rows<D, 2>(p, ktile, vtile, b, kvh, key0, L, phys, chunk == 0,
                             [](int r, int vec) { return swz<D>(r, vec * 8); });
      }
      lane_sync(1 + bl, CG);
    }

    if (live) {
      // S^T = K Q^T, the head-dim steps spread over four accumulator chains.
      constexpr int NCH = KS < 4 ? KS : 4;
      float acc[NCH][4];
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) acc[ch][0] = acc[ch][1] = acc[ch][2] = acc[ch][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, ktile + swz<D>(lane & 15, ks * 16 + (lane >> 4) * 8));
        Mma<T>::run(acc[ks % NCH], a, qf[ks][0], qf[ks][1]);
      }
      float sc[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float t = acc[0][e];
#pragma unroll
        for (int ch = 1; ch < NCH; ++ch) t += acc[ch][e];
        sc[e] = t;
      }
      const bool need_mask = bad || key0 + kBlockSize > mask_from;
      bool above = false;  // some score exceeds its column's reference by > the slack
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = sc[e] * p.scale_log2;
        if (need_mask && !key_visible(p, key0 + g + ((e >> 1) << 3), L, bad, lim[e & 1], tm[e & 1]))
          v = -INFINITY;
        sc[e] = v;
        above |= v > m[e & 1] + kRescaleSlack;
      }
      // Online softmax.  The exponentials use a per-column reference m that
      // is raised (to the exact running max, rescaling l and O by
      // 2^(m_old - m)) only when a score exceeds it by more than
      // kRescaleSlack; otherwise the block's weights 2^(s - m) stay below
      // 2^kRescaleSlack and no cross-lane max, correction or rescale is
      // needed.  The result O / l does not depend on the reference.
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
          for (int mt = 0; mt < KS; ++mt) {
            o[mt][e] *= corr;
            o[mt][e + 2] *= corr;
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float m_use = m[e] == -INFINITY ? 0.f : m[e];
        const float p0 = ex2(sc[e] - m_use);
        const float p1 = ex2(sc[e + 2] - m_use);
        l[e] += p0 + p1;
        sc[e] = p0;
        sc[e + 2] = p1;
      }
      // P^T operand fragments: high part and rounding remainder.
      const uint32_t h01 = Mma<T>::pack(sc[0], sc[1]);
      const uint32_t h23 = Mma<T>::pack(sc[2], sc[3]);
      float r0, r1, r2, r3;
      Mma<T>::unpack(h01, r0, r1);
      Mma<T>::unpack(h23, r2, r3);
      const uint32_t ph0 = movm_t(h01), ph1 = movm_t(h23);
      const uint32_t pl0 = movm_t(Mma<T>::pack(sc[0] - r0, sc[1] - r1));
      const uint32_t pl1 = movm_t(Mma<T>::pack(sc[2] - r2, sc[3] - r3));
      // O^T += V^T P^T.  In a block that ends past the context, zero the V^T
      // columns (keys) past it so that NaN-filled rows never enter an MMA.
      const int nvalid = bad ? 0 : L - key0;
      auto pv = [&](auto partial) {
        uint32_t km0 = 0xffffffffu, km8 = 0xffffffffu;
        if (decltype(partial)::value) {
          km0 = (2 * c < nvalid ? 0x0000ffffu : 0u) | (2 * c + 1 < nvalid ? 0xffff0000u : 0u);
          km8 = (2 * c + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * c + 9 < nvalid ? 0xffff0000u : 0u);
        }
        // Four head-dim tiles at a time: their high-part MMAs first, then the
        // low parts, so that no MMA waits on the one just issued.
        constexpr int GRP = KS < 4 ? KS : 4;
#pragma unroll
        for (int m0 = 0; m0 < KS; m0 += GRP) {
          uint32_t a[GRP][4];
#pragma unroll
          for (int u = 0; u < GRP; ++u) {
            ldsm_x4_t(a[u], vtile + swz<D>((lane & 7) + ((lane >> 4) << 3),
                                           (m0 + u) * 16 + ((lane >> 3) & 1) * 8));
            if (decltype(partial)::value) {
              a[u][0] &= km0;
              a[u][1] &= km0;
              a[u][2] &= km8;
              a[u][3] &= km8;
            }
          }
#pragma unroll
          for (int u = 0; u < GRP; ++u) Mma<T>::run(o[m0 + u], a[u], ph0, ph1);
#pragma unroll
          for (int u = 0; u < GRP; ++u) Mma<T>::run(o[m0 + u], a[u], pl0, pl1);
        }
      };
      if (nvalid < kBlockSize)
        pv(std::true_type{});
      else
        pv(std::false_type{});
    }
    lane_sync(1 + bl, CG);  // every warp of the lane is done with stage s
    if (i + NS < n_my) {
      if (!aborted) issue(i + NS);
      ++issued;
    }
  }
  if (aborted && leader && lane == 0) {
    // Give the copies still in flight a bounded chance to land before the
    // shared memory is reused.
    for (int k = consumed; k < issued; ++k)
      mbar_wait_bounded(my_bars + 8 * (k % NS), (k / NS) & 1);
  }

  // Row sums: reduce the per-thread partial sums over the 8 lanes of a column.
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float v = l[e];
    v += __shfl_xor_sync(kFull, v, 4);
    v += __shfl_xor_sync(kFull, v, 8);
    v += __shfl_xor_sync(kFull, v, 16);
    l[e] = v;
  }

  // Hand the per-warp states to the CTA epilogue (reusing the stage memory):
  // one state per (block lane, column).
  __syncthreads();
  constexpr int DP = D + 4;
  float *red_o = reinterpret_cast<float *>(smem);
  float *red_m = red_o + BL * NC * DP;
  float *red_l = red_m + BL * NC;
  float *wscale = red_l + BL * NC;
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int col = col0 + 2 * c + (e & 1);
      const int d = mt * 16 + g + ((e >> 1) << 3);
      red_o[(bl * NC + col) * DP + d] = o[mt][e];
    }
  if (g == 0) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      red_m[bl * NC + col0 + 2 * c + e] = m[e];
      red_l[bl * NC + col0 + 2 * c + e] = l[e];
    }
  }
  __syncthreads();
  cta_epilogue<T, D, NC, BL, NW * 32>(p, red_m, red_l, red_o, wscale, b, kvh, chunk, split,
                                      ns_b);
}

// Block lanes for CG column groups: about four warps per CTA.
template <int CG> constexpr int mma_lanes() { return CG >= 3 ? 1 : 4 / CG; }

// Stages per block lane, shallow and deep.  Fewer lanes per CTA take deeper
// rings so that every CTA keeps about the same bytes in flight: 2 / 3 stages
// for four lanes (single column group), 3 / 4 for two, 4 / 6 for one (1 / 2
// at head_dim 256).
template <int D, int CG, bool DEEP> constexpr int mma_stages() {
  return D >= 256 ? (DEEP ? 2 : 1)
                  : (CG >= 3 ? (DEEP ? 6 : 4) : (CG == 2 ? (DEEP ? 4 : 3) : (DEEP ? 3 : 2)));
}

template <typename T, int D, int CG, bool DEEP>
constexpr size_t mma_smem_bytes() {
  constexpr int BL = mma_lanes<CG>();
  constexpr int NS = mma_stages<D, CG, DEEP>();
  constexpr int NC = CG * 8;
  constexpr size_t stages = size_t(BL) * NS * MmaGeom<D>::kStageBytes;
  constexpr size_t red = (size_t(BL) * NC * (D + 4) + size_t(3 * BL + 2) * NC) * 4;
  constexpr size_t merge = (size_t(NC) * kMaxFusedSplits + NC) * 4;
  constexpr size_t need = red > merge ? red : merge;
  constexpr size_t scratch = need > stages ? need : stages;
  return scratch + 1024;
}

using MmaLaunch = cudaError_t (*)(const CUtensorMap &, const CUtensorMap &, const AttnParams &,
                                  dim3, cudaStream_t);

template <typename T, int D, int CG, bool DEEP>
KernelInfo mma_info_t() {
  constexpr int BL = mma_lanes<CG>();
  KernelInfo k;
  k.func = reinterpret_cast<const void *>(
      &attn_mma_kernel<T, D, CG, BL, mma_stages<D, CG, DEEP>()>);
  k.threads = BL * CG * 32;
  k.smem = mma_smem_bytes<T, D, CG, DEEP>();
  k.warps = BL * CG;
  k.stages = mma_stages<D, CG, DEEP>();
  return k;
}

template <typename T, int D, int CG, bool DEEP>
cudaError_t launch_t(const CUtensorMap &km, const CUtensorMap &vm, const AttnParams &p, dim3 grid,
                     cudaStream_t stream) {
  const KernelInfo k = mma_info_t<T, D, CG, DEEP>();
  attn_mma_kernel<T, D, CG, mma_lanes<CG>(), mma_stages<D, CG, DEEP>()>
      <<<grid, k.threads, k.smem, stream>>>(km, vm, p);
  return cudaGetLastError();
}

// Default ring: the shallow one (for one column group at head_dim <= 128,
// 3 CTAs per SM; the 8-row GQA tile measured 0.949 of the HBM peak against
// 0.932 with the deep ring).
template <typename T, int D, int CG>
bool mma_pick_stages(int stages, KernelInfo *info, MmaLaunch *launch) {
  if (stages == 0) stages = mma_stages<D, CG, false>();
  if (stages == mma_stages<D, CG, true>()) {
    *info = mma_info_t<T, D, CG, true>();
    *launch = &launch_t<T, D, CG, true>;
    return true;
  }
  if (stages == mma_stages<D, CG, false>()) {
    *info = mma_info_t<T, D, CG, false>();
    *launch = &launch_t<T, D, CG, false>;
    return true;
  }
  return false;
}

// Column groups x head dim within the budget (CG * D <= 384).
template <typename T, int D>
bool mma_pick(int cg, int stages, KernelInfo *info, MmaLaunch *launch) {
  switch (cg) {
    case 1: return mma_pick_stages<T, D, 1>(stages, info, launch);
    case 2: return D <= 128 && mma_pick_stages<T, D, (D <= 128 ? 2 : 1)>(stages, info, launch);
    case 3: return D <= 128 && mma_pick_stages<T, D, (D <= 128 ? 3 : 1)>(stages, info, launch);
    case 4: return D <= 64 && mma_pick_stages<T, D, (D <= 64 ? 4 : 1)>(stages, info, launch);
    default: return false;
  }
}

template <typename T>
bool mma_pick_d(int D, int cg, int stages, KernelInfo *info, MmaLaunch *launch) {
  switch (D) {
    case 64: return mma_pick<T, 64>(cg, stages, info, launch);
    case 128: return mma_pick<T, 128>(cg, stages, info, launch);
    case 256: return mma_pick<T, 256>(cg, stages, info, launch);
    default: return false;
  }
}

bool mma_pick_any(pkv_dtype dtype, int D, int cg, int stages, KernelInfo *info,
                  MmaLaunch *launch) {
  if (dtype == PKV_BF16) return mma_pick_d<__nv_bfloat16>(D, cg, stages, info, launch);
  if (dtype == PKV_F16) return mma_pick_d<__half>(D, cg, stages, info, launch);
  return false;
}

}  // namespace

int mma_max_tiles(int head_dim) { return head_dim <= 64 ? 4 : (head_dim <= 128 ? 3 : 1); }

bool mma_kernel_info(pkv_dtype dtype, int head_dim, int n_tiles, int stages, KernelInfo *info) {
  MmaLaunch launch = nullptr;
  return mma_pick_any(dtype, head_dim, n_tiles, stages, info, &launch);
}

cudaError_t mma_launch(pkv_dtype dtype, int head_dim, int n_tiles, int stages,
                       const CUtensorMap &kmap, const CUtensorMap &vmap, const AttnParams &p,
                       dim3 grid, cudaStream_t stream) {
  KernelInfo info;
  MmaLaunch launch = nullptr;
  if (!mma_pick_any(dtype, head_dim, n_tiles, stages, &info, &launch))
    return cudaErrorInvalidValue;
  return launch(kmap, vmap, p, grid, stream);
}

}  // namespace pkv
