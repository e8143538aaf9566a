// attn_mma.cuh -- paged decode / speculative-verify attention on tensor cores:
// the kernel template, instantiated for bf16 / fp16 caches in attn_mma.cu and
// for FP8 E4M3 caches (bf16 / fp16 queries) in attn_mma_fp8.cu.
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
#pragma once

#include <cuda_fp8.h>

#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace mma {

// Largest excess (log2 units) of a score over its column's reference max
// before the reference is raised: block weights stay below 2^8.
constexpr float kRescaleSlack = 8.f;

// Tile geometry for a head dim D of ELT-byte cache elements: each row is cut
// into 128-byte panels (one TMA box each), 16 rows per panel.
template <int D, int ELT> struct MmaGeom {
  static constexpr int kRowBytes = D * ELT;
  static constexpr int kParts = kRowBytes / 128;        // 128-byte panels per row
  static constexpr int kPanelElems = 128 / ELT;
  static constexpr int kPanelBytes = kBlockSize * 128;  // 2 KB
  static constexpr int kTileBytes = kParts * kPanelBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;    // K tile + V tile
  static constexpr int kSteps = D / 16;                 // MMA k-steps over the head dim
};

// Byte offset of row `row`, byte `bo` (a multiple of 16 for whole chunks) in a
// tile copied with the 128-byte swizzle: chunk c of a 128-byte line sits at
// c ^ (line & 7).
__device__ __forceinline__ uint32_t swzb(int row, int bo) {
  const int part = bo >> 7;
  const int chunk = (bo & 127) >> 4;
  return part * (kBlockSize * 128) + row * 128 + ((chunk ^ (row & 7)) << 4) + (bo & 15);
}

// The same for 16-bit elements: element (row, d), d a multiple of 8.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int d) {
  return swzb(row, 2 * d);
}

// Element type of the MMA for a cache type: the cache's own 16-bit type, or
// f16 for FP8 codes (widened exactly to f16).
template <typename T, typename TC> struct MmaType { using type = T; };
template <typename T> struct MmaType<T, E4M3> { using type = __half; };

// Four e4m3 codes (bytes 0..3 of `four`) -> the f16 values of bytes 0, 1
// (packed in `lo`) and of bytes 2, 3 (in `hi`); exact, e4m3 being a subset
// of f16.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t four, uint32_t &lo, uint32_t &hi) {
  asm("{\n\t.reg .b16 c01, c23;\n\t"
      "mov.b32 {c01, c23}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, c01;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, c23;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(four));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Head-dim index of O^T accumulator element e (0..3) of m-tile mt for lane
// group g.  16-bit caches: the MMA's natural rows (d = 16 mt + g, + 8).
// FP8 caches: row g of m-tile mt is d = 16 mt + 2g and row g + 8 is
// 16 mt + 2g + 1, the order in which a transposed ldmatrix of byte pairs
// delivers the V^T fragments.
template <bool FP8>
__device__ __forceinline__ int o_dim(int mt, int g, int e) {
  if (FP8) return mt * 16 + 2 * g + (e >> 1);
  return mt * 16 + g + ((e >> 1) << 3);
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
// of a lane share each staged block, warp cg computing the NT 8-column tiles
// of query columns 8 NT cg .. 8 NT (cg + 1) - 1 (a warp with several tiles
// reads each K / V fragment once for all of them).  The lane's first warp
// issues the copies.
//
// T: element type of q and out (bf16 / f16); TC: cache element (T, or E4M3:
// one-byte codes, widened to f16 for f16 MMAs; q then enters as f16 after a
// per-row power-of-two shift that keeps it in f16 range, undone in the score
// scale).
// Resident CTAs a kernel is compiled for: the three-warp tile fits six per
// SM in shared memory, which its registers must then allow (<= 112 each);
// the four- and five-warp tiles five and four (<= 102 each).
template <int CG, int NT> constexpr int mma_min_ctas() {
  return NT != 1 ? 1 : (CG == 3 ? 6 : (CG == 4 ? 5 : (CG == 5 ? 4 : 1)));
}

template <typename T, typename TC, int D, int CG, int NT, int KB, int BL, int NS>
__global__ void __launch_bounds__(BL * CG * 32, (mma_min_ctas<CG, NT>()))
    attn_mma_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const AttnParams p) {
  static_assert(NS >= KB, "an iteration's blocks must all be in flight at once");
  // The next kernel of the stream (the merge kernel, or the next call's
  // attention) may be scheduled now; it waits for this grid.  This kernel is
  // itself launched as a programmatic dependent of the one before it, so
  // before touching global memory it waits for that one to complete.
  pdl_launch_dependents();
  pdl_wait();
  constexpr bool FP8 = std::is_same<TC, E4M3>::value;
  using TM = typename MmaType<T, TC>::type;
  using G = MmaGeom<D, Elt<TC>::bytes>;
  constexpr int NC = CG * NT * 8;  // query columns of this CTA (padded)
  constexpr int KS = G::kSteps;
  constexpr int NW = BL * CG;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);
  __shared__ uint64_t bars[BL * NS];  // the stage's copies landed
  __shared__ volatile int s_abort;
  __shared__ int s_lim[NC];                  // causal visible-row limit per column
  __shared__ unsigned long long s_tm[NC];    // tree mask per column

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bl = warp / CG, cg = warp - (warp / CG) * CG;
  const bool leader = cg == 0;
  const int g = lane >> 2, c = lane & 3;
  const CtaWork wk = cta_work(p);
  if (!wk.active) return;  // a split past its sequence's end (the whole CTA agrees)
  const int kvh = wk.kvh, chunk = wk.chunk, b = wk.b;
  const SeqExtent ext = wk.ext;
  const int L = ext.L;
  const int blk_begin = wk.blk_begin;
  const int nspan = max(wk.blk_end - blk_begin, 0);
  const int n_my = nspan > bl ? (nspan - bl + BL - 1) / BL : 0;
  const int col0 = cg * NT * 8;

  const int mask_from = L - p.num_queries;  // first row some column may not see

  // Online-softmax state.
  float o[KS][NT][4];
  float m[NT][2], l[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt][0] = m[nt][1] = -INFINITY;
    l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
  }

  // The lane's ring; per-column visibility.
  const uint32_t my_bars = smem_u32(&bars[bl * NS]);
  const uint32_t my_stages = smem_base + bl * NS * G::kStageBytes;
  if (threadIdx.x == 0) s_abort = 0;
  for (int col = threadIdx.x; col < NC; col += NW * 32) {
    s_lim[col] = cta_row_limit(p, L, chunk, col);
    s_tm[col] = cta_row_tree_mask(p, b, chunk, col);
  }
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
    return i < n_my ? ld_keep(table + static_cast<int64_t>(i) * BL) : -1;
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
      if (p.tile_box) {  // one copy per tile
        tma_load_5d(st, &kmap, bar, 0, 0, 0, kvh, phys);
        tma_load_5d(st + G::kTileBytes, &vmap, bar, 0, 0, 0, kvh, phys);
      } else {           // one copy per 128-byte column panel
#pragma unroll
        for (int part = 0; part < G::kParts; ++part)
          tma_load_4d(st + part * G::kPanelBytes, &kmap, bar, part * G::kPanelElems, 0, kvh,
                      phys);
#pragma unroll
        for (int part = 0; part < G::kParts; ++part)
          tma_load_4d(st + G::kTileBytes + part * G::kPanelBytes, &vmap, bar,
                      part * G::kPanelElems, 0, kvh, phys);
      }
    }
  };

  const int npre = min(NS, n_my);
  for (int i = 0; i < npre; ++i) issue(i);
  int issued = npre;

  // q is loaded once the first copies are in flight, so that its latency
  // (a round trip to wherever q lives) overlaps theirs.
  // Q^T operand fragments of this warp's columns (B operand: k = head dim).
  // 16-bit caches: the natural k order.  FP8 caches: k-step ks covers head
  // dims 16 ks .. 16 ks + 15 with lane c holding 16 ks + 4c .. 4c + 3 (the
  // order the K fragments arrive in), shifted by 2^qshift into f16 range.
  uint32_t qf[KS][NT][2];
  float colfac[NT][2];  // score scale of my two columns of each tile
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int64_t row = cta_row_index(p, b, kvh, chunk, col0 + nt * 8 + g);
    const T *qrow = reinterpret_cast<const T *>(p.q) + (row < 0 ? 0 : row) * D;
    colfac[nt][0] = colfac[nt][1] = p.scale_log2;
    if constexpr (!FP8) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qf[ks][nt][0] =
            row < 0 ? 0u : *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 2 * c);
        qf[ks][nt][1] =
            row < 0 ? 0u : *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + 2 * c);
      }
    } else {
      float qv[KS][4];
      float amax = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t w0 = 0u, w1 = 0u;
        if (row >= 0) {
          const uint2 w = *reinterpret_cast<const uint2 *>(qrow + ks * 16 + 4 * c);
          w0 = w.x;
          w1 = w.y;
        }
        Mma<T>::unpack(w0, qv[ks][0], qv[ks][1]);
        Mma<T>::unpack(w1, qv[ks][2], qv[ks][3]);
#pragma unroll
        for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(qv[ks][e]));
      }
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
      // amax in [2^(ex-1), 2^ex): scaling by 2^(15 - ex) puts the row's
      // largest magnitude in [2^14, 2^15), inside f16 range.
      const int ex = amax > 0.f ? ((__float_as_int(amax) >> 23) & 0xff) - 126 : 15;
      const int qshift = max(-120, min(120, 15 - ex));
      const float up = exp2f(static_cast<float>(qshift));
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qf[ks][nt][0] = Mma<__half>::pack(qv[ks][0] * up, qv[ks][1] * up);
        qf[ks][nt][1] = Mma<__half>::pack(qv[ks][2] * up, qv[ks][3] * up);
      }
      // my score columns 2c, 2c+1 were shifted by the lanes of groups 2c, 2c+1
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int sh = __shfl_sync(kFull, qshift, 4 * (2 * c + e));
        colfac[nt][e] = p.scale_log2 * exp2f(static_cast<float>(-sh));
      }
    }
  }

  int consumed = 0;
  bool aborted = false;
  for (int i0 = 0; i0 < n_my; i0 += KB) {
    // This iteration's KB blocks (the last may hold fewer).  A copy that
    // never lands aborts the CTA (with column groups, through a shared
    // flag): from then on no warp waits or computes, but every warp still
    // takes part in each lane_sync.
    bool has[KB], bad[KB];
    int key0[KB];
    uint32_t ktile[KB], vtile[KB];
#pragma unroll
    for (int u = 0; u < KB; ++u) {
      const int i = i0 + u;
      const int s = i % NS;
      has[u] = KB == 1 || i < n_my;
      if (has[u] && !aborted) {
        // one decision per warp: its lanes then agree on every later shuffle
        if (__all_sync(kFull, mbar_wait_bounded(my_bars + 8 * s, (i / NS) & 1))) {
          consumed = i + 1;
        } else {
          aborted = true;
          if (CG > 1) s_abort = 1;
          if (lane == 0) record_error(p.err, PKV_DEVERR_TIMEOUT);
        }
      }
      ktile[u] = my_stages + s * G::kStageBytes;
      vtile[u] = ktile[u] + G::kTileBytes;
      key0[u] = (blk_begin + bl + i * BL) * kBlockSize;
      bad[u] = !has[u] || ((bad_mask >> (i & 31)) & 1u);
    }
    if (CG > 1 && !aborted) aborted = s_abort != 0;
    const bool live = !aborted;
    if constexpr (!FP8) {  // the fused append (16-bit caches only)
      if (p.k_new != nullptr) {
        bool any = false;
#pragma unroll
        for (int u = 0; u < KB; ++u) {
          if (bad[u] || key0[u] + kBlockSize <= L - p.num_queries) continue;
          any = true;
          if (leader && live) {
            const int64_t phys = __ldg(table + static_cast<int64_t>(i0 + u) * BL);
            patch_new_rows<D, 2>(p, ktile[u], vtile[u], b, kvh, key0[u], L, phys, chunk == 0,
                                 [](int r, int vec) { return swz<D>(r, vec * 8); });
          }
        }
        if (any) lane_sync(1 + bl, CG);
      }
    }

    if (live) {
      // S^T = K Q^T per block.  One tile of one block: the head-dim steps
      // spread over four accumulator chains; otherwise the tiles' and
      // blocks' MMAs interleave.  (A block past the sequence's end, in the
      // last iteration, is computed on whatever its stage holds and masked
      // out entirely.)
      constexpr int NCH = (NT * KB) == 1 ? (KS < 4 ? KS : 4) : ((NT * KB) == 2 ? 2 : 1);
      float sc[KB][NT][4];
      bool above = false;  // some score exceeds its column's reference by > the slack
#pragma unroll
      for (int u = 0; u < KB; ++u) {
        float acc[NCH][NT][4];
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            acc[ch][nt][0] = acc[ch][nt][1] = acc[ch][nt][2] = acc[ch][nt][3] = 0.f;
        if constexpr (!FP8) {
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            uint32_t a[4];
            ldsm_x4(a, ktile[u] + swz<D>(lane & 15, ks * 16 + (lane >> 4) * 8));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              Mma<TM>::run(acc[ks % NCH][nt], a, qf[ks][nt][0], qf[ks][nt][1]);
          }
        } else {
          // One ldmatrix brings 16 keys x 32 head dims of codes: lane (g, c)
          // gets 4 consecutive codes of keys g and g + 8 from each 16-byte
          // half.
#pragma unroll
          for (int pr = 0; pr < KS / 2; ++pr) {
            uint32_t r[4];
            ldsm_x4(r, ktile[u] + swzb(lane & 15, pr * 32 + (lane >> 4) * 16));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t a[4];
              e4m3x4_to_f16(r[2 * h], a[0], a[2]);      // key g: dims 4c, 4c+1 | 4c+2, 4c+3
              e4m3x4_to_f16(r[2 * h + 1], a[1], a[3]);  // key g + 8
              const int ks = 2 * pr + h;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                Mma<TM>::run(acc[ks % NCH][nt], a, qf[ks][nt][0], qf[ks][nt][1]);
            }
          }
        }
        const bool need_mask = bad[u] || key0[u] + kBlockSize > mask_from;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float t = acc[0][nt][e];
#pragma unroll
            for (int ch = 1; ch < NCH; ++ch) t += acc[ch][nt][e];
            float v = t * colfac[nt][e & 1];
            if (need_mask) {
              const int col = col0 + nt * 8 + 2 * c + (e & 1);
              if (!key_visible(p, key0[u] + g + ((e >> 1) << 3), L, bad[u], s_lim[col],
                               s_tm[col]))
                v = -INFINITY;
            }
            sc[u][nt][e] = v;
            above |= v > m[nt][e & 1] + kRescaleSlack;
          }
        }
      }
      // Online softmax.  The exponentials use a per-column reference m that
      // is raised (to the exact running max, rescaling l and O by
      // 2^(m_old - m)) only when a score exceeds it by more than
      // kRescaleSlack; otherwise the weights 2^(s - m) stay below
      // 2^kRescaleSlack and no cross-lane max, correction or rescale is
      // needed.  The result O / l does not depend on the reference.
      if (__any_sync(kFull, above)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float mx = fmaxf(sc[0][nt][e], sc[0][nt][e + 2]);
#pragma unroll
            for (int u = 1; u < KB; ++u) mx = fmaxf(mx, fmaxf(sc[u][nt][e], sc[u][nt][e + 2]));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
            const float m_new = fmaxf(m[nt][e], mx);
            const float corr = ex2(m[nt][e] - (m_new == -INFINITY ? 0.f : m_new));
            l[nt][e] *= corr;
            m[nt][e] = m_new;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
              o[mt][nt][e] *= corr;
              o[mt][nt][e + 2] *= corr;
            }
          }
      }
      // Weights, and the P^T operand fragments.  bf16 / f16 MMAs on 16-bit
      // caches: high part and rounding remainder (a single bf16 P would add
      // about 1.6e-3 of relative error).  FP8 caches: one f16 P (weights
      // <= 2^8; 2^-11 relative rounding).
      uint32_t ph[KB][NT][2], pl[KB][NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float m_use = m[nt][e] == -INFINITY ? 0.f : m[nt][e];
#pragma unroll
          for (int u = 0; u < KB; ++u) {
            const float p0 = ex2(sc[u][nt][e] - m_use);
            const float p1 = ex2(sc[u][nt][e + 2] - m_use);
            l[nt][e] += p0 + p1;
            sc[u][nt][e] = p0;
            sc[u][nt][e + 2] = p1;
          }
        }
#pragma unroll
      for (int u = 0; u < KB; ++u)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint32_t h01 = Mma<TM>::pack(sc[u][nt][0], sc[u][nt][1]);
          const uint32_t h23 = Mma<TM>::pack(sc[u][nt][2], sc[u][nt][3]);
          ph[u][nt][0] = movm_t(h01);
          ph[u][nt][1] = movm_t(h23);
          pl[u][nt][0] = pl[u][nt][1] = 0u;
          if constexpr (!FP8) {
            float r0, r1, r2, r3;
            Mma<TM>::unpack(h01, r0, r1);
            Mma<TM>::unpack(h23, r2, r3);
            pl[u][nt][0] = movm_t(Mma<TM>::pack(sc[u][nt][0] - r0, sc[u][nt][1] - r1));
            pl[u][nt][1] = movm_t(Mma<TM>::pack(sc[u][nt][2] - r2, sc[u][nt][3] - r3));
          }
        }
      // O^T += V^T P^T.  In a block that ends past the context, zero the V^T
      // columns (keys) past it so that NaN-filled rows never enter an MMA.
      int nvalid[KB];
      bool full = true;
#pragma unroll
      for (int u = 0; u < KB; ++u) {
        nvalid[u] = bad[u] ? 0 : L - key0[u];
        full = full && nvalid[u] >= kBlockSize;
      }
      auto pv = [&](auto partial) {
        uint32_t km0[KB], km8[KB];
#pragma unroll
        for (int u = 0; u < KB; ++u) {
          km0[u] = km8[u] = 0xffffffffu;
          if (decltype(partial)::value) {
            const int nv = nvalid[u];
            km0[u] = (2 * c < nv ? 0x0000ffffu : 0u) | (2 * c + 1 < nv ? 0xffff0000u : 0u);
            km8[u] = (2 * c + 8 < nv ? 0x0000ffffu : 0u) | (2 * c + 9 < nv ? 0xffff0000u : 0u);
          }
        }
        if constexpr (!FP8) {
          // Head-dim tiles a group at a time: the high-part MMAs of every
          // block first, then the low parts, so that no MMA waits on the
          // one just issued.
          constexpr int GRP = (NT * KB) > 1 ? 2 : (KS < 4 ? KS : 4);
#pragma unroll
          for (int m0 = 0; m0 < KS; m0 += GRP) {
            uint32_t a[KB][GRP][4];
#pragma unroll
            for (int u = 0; u < KB; ++u)
#pragma unroll
              for (int w = 0; w < GRP; ++w) {
                ldsm_x4_t(a[u][w], vtile[u] + swz<D>((lane & 7) + ((lane >> 4) << 3),
                                                     (m0 + w) * 16 + ((lane >> 3) & 1) * 8));
                if (decltype(partial)::value) {
                  a[u][w][0] &= km0[u];
                  a[u][w][1] &= km0[u];
                  a[u][w][2] &= km8[u];
                  a[u][w][3] &= km8[u];
                }
              }
#pragma unroll
            for (int u = 0; u < KB; ++u)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int w = 0; w < GRP; ++w)
                  Mma<TM>::run(o[m0 + w][nt], a[u][w], ph[u][nt][0], ph[u][nt][1]);
#pragma unroll
            for (int u = 0; u < KB; ++u)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int w = 0; w < GRP; ++w)
                  Mma<TM>::run(o[m0 + w][nt], a[u][w], pl[u][nt][0], pl[u][nt][1]);
          }
        } else {
          // V^T fragments from codes: one transposed ldmatrix of byte pairs
          // per 32 head dims gives lane (g, c), for keys 2c, 2c+1 (and
          // 2c+8, 2c+9), the codes of dims 2g, 2g+1 of each 16-dim tile; a
          // byte permute pairs the two keys of each dim (see o_dim).
#pragma unroll
          for (int pr = 0; pr < KS / 2; ++pr) {
#pragma unroll
            for (int u = 0; u < KB; ++u) {
              uint32_t r[4];
              ldsm_x4_t(r, vtile[u] + swzb(lane & 15, pr * 32 + (lane >> 4) * 16));
              uint32_t a[2][4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                // r[j]: keys (2c | 2c+8) and (2c+1 | 2c+9), dims 2g, 2g+1
                uint32_t lo, hi;
                e4m3x4_to_f16(prmt(r[j], 0u, 0x3120), lo, hi);
                a[j >> 1][(j & 1) * 2] = lo;       // dim 2g
                a[j >> 1][(j & 1) * 2 + 1] = hi;   // dim 2g + 1
              }
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                if (decltype(partial)::value) {
                  a[h][0] &= km0[u];
                  a[h][1] &= km0[u];
                  a[h][2] &= km8[u];
                  a[h][3] &= km8[u];
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  Mma<TM>::run(o[2 * pr + h][nt], a[h], ph[u][nt][0], ph[u][nt][1]);
              }
            }
          }
        }
      };
      if (full)
        pv(std::false_type{});
      else
        pv(std::true_type{});
    }
    lane_sync(1 + bl, CG);  // every warp of the lane is done with these stages
#pragma unroll
    for (int u = 0; u < KB; ++u) {
      if (i0 + u + NS < n_my && !aborted) {
        issue(i0 + u + NS);
        ++issued;
      }
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
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = l[nt][e];
      v += __shfl_xor_sync(kFull, v, 4);
      v += __shfl_xor_sync(kFull, v, 8);
      v += __shfl_xor_sync(kFull, v, 16);
      l[nt][e] = v;
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
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = col0 + nt * 8 + 2 * c + (e & 1);
        red_o[(bl * NC + col) * DP + o_dim<FP8>(mt, g, e)] = o[mt][nt][e];
      }
  if (g == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        red_m[bl * NC + col0 + nt * 8 + 2 * c + e] = m[nt][e];
        red_l[bl * NC + col0 + nt * 8 + 2 * c + e] = l[nt][e];
      }
  }
  __syncthreads();
  cta_epilogue<T, D, NC, BL, NW * 32>(p, red_m, red_l, red_o, wscale, wk);
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

// FP8 tiles are half the bytes: twice the stages for the same bytes in flight.
template <typename TC, int D, int CG, bool DEEP> constexpr int mma_stages_t() {
  return mma_stages<D, CG, DEEP>() * (std::is_same<TC, E4M3>::value ? 2 : 1);
}

template <typename T, typename TC, int D, int CG, int NT, bool DEEP>
constexpr size_t mma_smem_bytes() {
  constexpr int BL = mma_lanes<CG>();
  constexpr int NS = mma_stages_t<TC, D, CG, DEEP>();
  constexpr int NC = CG * NT * 8;
  constexpr size_t stages = size_t(BL) * NS * MmaGeom<D, Elt<TC>::bytes>::kStageBytes;
  constexpr size_t red = (size_t(BL) * NC * (D + 4) + size_t(3 * BL + 2) * NC) * 4;
  constexpr size_t merge = (size_t(NC) * kMaxFusedSplits + NC) * 4;
  constexpr size_t need = red > merge ? red : merge;
  constexpr size_t scratch = need > stages ? need : stages;
  return scratch + 1024;
}

using MmaLaunch = cudaError_t (*)(const CUtensorMap &, const CUtensorMap &, const AttnParams &,
                                  dim3, cudaStream_t);

template <typename T, typename TC, int D, int CG, int NT, int KB, bool DEEP>
KernelInfo mma_info_t() {
  constexpr int BL = mma_lanes<CG>();
  KernelInfo k;
  k.func = reinterpret_cast<const void *>(
      &attn_mma_kernel<T, TC, D, CG, NT, KB, BL, mma_stages_t<TC, D, CG, DEEP>()>);
  k.threads = BL * CG * 32;
  k.smem = mma_smem_bytes<T, TC, D, CG, NT, DEEP>();
  k.warps = BL * CG;
  k.stages = mma_stages_t<TC, D, CG, DEEP>();
  k.warp_tiles = NT;
  k.blocks_per_iter = KB;
  return k;
}

template <typename T, typename TC, int D, int CG, int NT, int KB, bool DEEP>
cudaError_t launch_t(const CUtensorMap &km, const CUtensorMap &vm, const AttnParams &p, dim3 grid,
                     cudaStream_t stream) {
  const KernelInfo k = mma_info_t<T, TC, D, CG, NT, KB, DEEP>();
  // a programmatic dependent of the kernel before it (with split-K counters,
  // the kernel that zeroes them)
  return launch_kernel(true,
                       attn_mma_kernel<T, TC, D, CG, NT, KB, mma_lanes<CG>(),
                                       mma_stages_t<TC, D, CG, DEEP>()>,
                       grid, k.threads, k.smem, stream, km, vm, p);
}

// Default ring: the shallow one (for one column group at head_dim <= 128,
// 3 CTAs per SM; the 8-row GQA tile measured 0.949 of the HBM peak against
// 0.932 with the deep ring).
//
// A warp waits for the KB blocks of an iteration before it issues the next
// ones, so KB blocks per iteration need a ring of at least KB stages (else
// the wait could never end); rings of fewer than 2 KB stages are not built
// either (no pair in flight while a pair is computed).
template <typename T, typename TC, int D, int CG, int NT, int KB, bool DEEP>
bool mma_pick_ring(KernelInfo *info, MmaLaunch *launch) {
  if constexpr (KB > 1 && mma_stages_t<TC, D, CG, DEEP>() < 2 * KB) {
    return false;
  } else {
    *info = mma_info_t<T, TC, D, CG, NT, KB, DEEP>();
    *launch = &launch_t<T, TC, D, CG, NT, KB, DEEP>;
    return true;
  }
}

template <typename T, typename TC, int D, int CG, int NT, int KB>
bool mma_pick_stages(int stages, KernelInfo *info, MmaLaunch *launch) {
  if (stages == 0) stages = mma_stages_t<TC, D, CG, false>();
  if (stages == mma_stages_t<TC, D, CG, true>())
    return mma_pick_ring<T, TC, D, CG, NT, KB, true>(info, launch);
  if (stages == mma_stages_t<TC, D, CG, false>())
    return mma_pick_ring<T, TC, D, CG, NT, KB, false>(info, launch);
  return false;
}

// Blocks per iteration: one or two for single-tile warps (two need rings of
// four stages or more to keep a pair in flight), one for multi-tile warps.
template <typename T, typename TC, int D, int CG>
bool mma_pick_kb(int kb, int stages, KernelInfo *info, MmaLaunch *launch) {
  if (kb == 2) return mma_pick_stages<T, TC, D, CG, 1, 2>(stages, info, launch);
  return kb == 1 && mma_pick_stages<T, TC, D, CG, 1, 1>(stages, info, launch);
}

// Column groups x tiles per warp x head dim within the register and shared
// memory budgets: cg warps of nt 8-column tiles each.  One tile per warp: up
// to five column groups (40 query rows, e.g. a 10-node tree over four query
// heads per KV head, read from one staged copy of each block) at head_dim
// <= 128, one at 256.  Several tiles in one warp (its O^T accumulators hold
// nt * D / 4 floats per thread): nt * D <= 384, one column group.
template <typename T, typename TC, int D>
bool mma_pick(int cg, int nt, int kb, int stages, KernelInfo *info, MmaLaunch *launch) {
  if (nt == 1) {
    switch (cg) {
      case 1: return mma_pick_kb<T, TC, D, 1>(kb, stages, info, launch);
      case 2: return D <= 128 && mma_pick_kb<T, TC, D, (D <= 128 ? 2 : 1)>(kb, stages, info, launch);
      case 3: return D <= 128 && mma_pick_kb<T, TC, D, (D <= 128 ? 3 : 1)>(kb, stages, info, launch);
      case 4: return D <= 128 && mma_pick_kb<T, TC, D, (D <= 128 ? 4 : 1)>(kb, stages, info, launch);
      case 5: return D <= 128 && mma_pick_kb<T, TC, D, (D <= 128 ? 5 : 1)>(kb, stages, info, launch);
      default: return false;
    }
  }
  if (cg != 1 || kb != 1) return false;
  switch (nt) {
    case 2:
      return D <= 128 && mma_pick_stages<T, TC, D, 1, (D <= 128 ? 2 : 1), 1>(stages, info, launch);
    case 3:
      return D <= 128 && mma_pick_stages<T, TC, D, 1, (D <= 128 ? 3 : 1), 1>(stages, info, launch);
    case 4:
      return D <= 64 && mma_pick_stages<T, TC, D, 1, (D <= 64 ? 4 : 1), 1>(stages, info, launch);
    default: return false;
  }
}

}  // namespace mma
}  // namespace pkv
