// attn_prefill.cu -- chunked prefill attention over the paged KV cache on the
// fifth-generation tensor cores (tcgen05), accumulators in tensor memory.
//
// What it computes: sequence b brings q_len new query rows (one prefill
// chunk) whose keys and values have already been appended to its cache,
// which now holds L rows, the chunk's own rows last.  Query row j attends to
// cache rows i <= L - q_len + j: everything before the chunk and the chunk's
// rows up to itself ("Inference part 1", section "KV cache": new tokens
// attend to the cached ones and to the new ones up to themselves; section
// "Chunked prefill": a long prompt is processed chunk by chunk).  The
// arithmetic is FlashAttention's ("Inference part 1", section
// "FlashAttention"): tiles of query rows, keys streamed through on-chip memory
// in chunks, a running maximum and sum per row, the output divided by the
// sum at the end.  Prefill is a dense contraction (many query rows per key),
// so both products run on the tensor cores.
//
// One CTA per 256 query rows of one (sequence, KV head).  A row is a (query
// position, head of the KV head's group) pair, so each K/V chunk streamed
// once serves every query head that shares the KV head.  320 threads:
//   warps 0-3 / 4-7  softmax and epilogue of query tile 0 / 1 (128 rows each,
//                    one row per thread: TMEM lane = row);
//   warp 8           TMA producer: the Q tiles, then K and V chunks of 128
//                    keys (8 blocks through the block table) into a ring of
//                    NS stages, K and V alternating;
//   warp 9           MMA issuer (one lane) and TMEM owner.
// Per 128-key chunk c and tile t:
//   S_t[128 x 128] = Q_t[128 x D] . K_c^T                  (TMEM, fp32)
//   softmax per row, thread-local: masked scores in log2 units, a lazy
//   reference max m (raised, with l and O rescaled, only when a score exceeds
//   it by more than 2^8), P = 2^(s - m) written back over S_t in the 16-bit
//   input type: for bf16 as a high part (columns 0..63) and the remainder
//   P - high (columns 64..127), since one bf16 rounding of P alone costs
//   about 1.6e-3 of relative L2 error, as much as the output's own rounding;
//   f16 (11 significant bits) needs no remainder
//   O_t[128 x D]  += P_t[128 x 128] . V_c[128 x D]         (A read from TMEM;
//                    bf16: a second product with the remainder)
// The issuer interleaves the tiles (P.V of tile 0 then the next S of tile 0,
// then the same for tile 1), so one tile's MMAs run while the other's softmax
// does.  TMEM: S_0, S_1 (128 columns each) and O_0, O_1 (D columns each),
// 512 columns: one CTA per SM.
// Operands: Q and K K-major with the 128-byte swizzle (as the TMA writes
// them), V MN-major with the 128-byte swizzle (its own layout), P from TMEM.
// Keys past the context or in a bad block never reach an MMA as NaN: their
// scores are masked to -inf (P = 0), and the producer zeroes their V rows in
// shared memory before releasing the chunk (0 x NaN would be NaN).
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "tc_ptx.cuh"

namespace pkv {
namespace prefill {

constexpr int kTileRows = 128;                     // query rows per MMA tile (M)
constexpr int kTiles = 2;                          // tiles per CTA
constexpr int kCtaRows = kTiles * kTileRows;
constexpr int kChunkKeys = 128;                    // keys per chunk
constexpr int kChunkBlocks = kChunkKeys / kBlockSize;
constexpr int kSoftmaxWarps = 4 * kTiles;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kIssuerWarp = kSoftmaxWarps + 1;
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
constexpr float kRescaleSlack = 8.f;

template <int D, int NS> struct Geom {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int kPanels = D / 64;                      // 128-byte column panels
  static constexpr int kPanelBytes = 128 * 128;               // 128 rows x 128 B
  static constexpr int kStageBytes = kPanels * kPanelBytes;   // a Q tile, or one K / V chunk
  static constexpr int kRingOff = kTiles * kStageBytes;
  static constexpr int kBytes = kRingOff + NS * kStageBytes;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kOCol = kTiles * kChunkKeys;           // O_t at kOCol + D t
  static_assert(kOCol + kTiles * D <= 512, "TMEM columns");
};

// P is split into a high part and a remainder for bf16 (see above).
template <typename T> constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;

template <typename T> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// One CTA's share of the work, the same in every thread.
struct Work {
  int b, kvh, row0;   // rows row0 .. row0 + rows - 1 of the sequence's (position, head) rows
  int rows, q0, qlen, L;
  int tiles;          // 1 or 2
  int chunks[kTiles]; // 128-key chunks each tile reads
  int nblk;           // cache blocks the CTA reads
};

__device__ __forceinline__ Work make_work(const PrefillParams &p) {
  Work w;
  w.kvh = blockIdx.x;
  w.b = blockIdx.y;
  // the sequence's last rows (the most keys) are launched first
  w.row0 = (p.pairs - 1 - static_cast<int>(blockIdx.z)) * kCtaRows;
  const int q0 = __ldg(p.query_start + w.b), q1 = __ldg(p.query_start + w.b + 1);
  const int L = __ldg(p.context_lens + w.b);
  const bool sane = q0 >= 0 && q1 >= q0 && q1 <= p.total_q && q1 - q0 <= p.max_query_len &&
                    L >= q1 - q0 &&
                    static_cast<int64_t>(L) <=
                        static_cast<int64_t>(p.max_blocks_per_seq) * kBlockSize;
  if (!sane && blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0)
    record_error(p.err, PKV_DEVERR_CONTEXT_LEN);
  w.q0 = q0;
  w.qlen = sane ? q1 - q0 : 0;
  w.L = L;
  w.rows = min(kCtaRows, w.qlen * p.group - w.row0);
  w.tiles = w.rows > kTileRows ? 2 : 1;
  int lim = 0;
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
    const int last = w.row0 + min(t * kTileRows + kTileRows, w.rows) - 1;
    lim = w.L - w.qlen + last / p.group;  // the last key tile t's rows see
    w.chunks[t] = t < w.tiles ? lim / kChunkKeys + 1 : 0;
    if (t == w.tiles - 1) w.nblk = lim / kBlockSize + 1;
  }
  return w;
}

template <typename T, int D, int NS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  using G = Geom<D, NS>;
  const Work w = make_work(p);
  if (w.rows <= 0) return;  // the whole CTA, before any barrier or TMEM use

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  __shared__ uint64_t full[NS], empty[NS], q_full, landed, s_full[kTiles], p_full[kTiles],
      pv_done[kTiles], mma_idle;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&landed), 1);
    mbar_init(smem_u32(&mma_idle), 1);
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(smem_u32(&s_full[t]), 1);
      mbar_init(smem_u32(&p_full[t]), 4);
      mbar_init(smem_u32(&pv_done[t]), 1);
    }
    fence_mbar_init();
  }
  if (warp == kIssuerWarp) tc::tmem_alloc(smem_u32(&tmem_base_s), G::kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_base_s;
  const int32_t *table = p.block_table + static_cast<int64_t>(w.b) * p.max_blocks_per_seq;
  const int n_chunks = w.chunks[w.tiles - 1];
  auto abort_all = [&]() {
    s_abort = 1;
    record_error(p.err, PKV_DEVERR_TIMEOUT);
  };

  if (warp == kProducerWarp) {
    // ---- TMA producer ----------------------------------------------------------
    bool ok = true;
    int issued = 0;
    uint32_t nfix = 0;
    if (lane == 0) mbar_arrive_expect_tx(smem_u32(&q_full), w.tiles * G::kStageBytes);
    __syncwarp();
    if (lane < w.tiles * G::kPanels) {
      // a Q tile: 128 / group positions x the group's heads, one 128-byte
      // panel per box; rows past the query tensor read as zero
      const int t = lane / G::kPanels, pn = lane % G::kPanels;
      tma_load_3d(sbase + t * G::kStageBytes + pn * G::kPanelBytes, &qmap, smem_u32(&q_full),
                  pn * 64, w.kvh * p.group, w.q0 + (w.row0 + t * kTileRows) / p.group);
    }
    for (int c = 0; c < n_chunks && ok; ++c) {
      const int nb = min(kChunkBlocks, w.nblk - c * kChunkBlocks);
      const int entry = lane < nb ? __ldg(table + c * kChunkBlocks + lane) : 0;
      const bool bad = lane < nb && (entry < 0 || static_cast<int64_t>(entry) >= p.num_blocks);
      const uint32_t bad_mask = __ballot_sync(kFull, bad);
      const int n_load = nb - __popc(bad_mask);
      // V rows from this one (chunk-local) on are past the context or past
      // the blocks read
      const int zfrom = min(w.L, (c * kChunkBlocks + nb) * kBlockSize) - c * kChunkKeys;
      for (int kv = 0; kv < 2; ++kv) {
        const int idx = 2 * c + kv, s = idx % NS;
        bool wt = !s_abort;
        if (wt && idx >= NS) wt = mbar_wait_bounded(smem_u32(&empty[s]), ((idx / NS) - 1) & 1);
        if (!__all_sync(kFull, wt)) {
          ok = false;
          break;
        }
        // V chunks with rows to zero land on their own barrier first
        const bool fix = kv == 1 && (bad_mask != 0 || zfrom < kChunkKeys);
        const uint32_t bar = smem_u32(fix ? &landed : &full[s]);
        if (lane == 0) {
          if (kv == 0 && bad_mask) record_error(p.err, PKV_DEVERR_BLOCK_ID);
          mbar_arrive_expect_tx(bar, n_load * G::kPanels * kBlockSize * 128);
        }
        __syncwarp();
        const uint32_t dst = sbase + G::kRingOff + s * G::kStageBytes;
        if (lane < nb && !bad) {
#pragma unroll
          for (int pn = 0; pn < G::kPanels; ++pn)
            tma_load_4d(dst + pn * G::kPanelBytes + lane * kBlockSize * 128, kv ? &vmap : &kmap,
                        bar, pn * 64, 0, w.kvh, entry);
        }
        issued = idx + 1;
        if (fix) {
          bool got = lane == 0 ? mbar_wait_bounded(smem_u32(&landed), nfix & 1) : true;
          ++nfix;
          if (!__shfl_sync(kFull, got, 0)) {
            ok = false;
            break;
          }
          // whole 128-byte rows: the swizzle only permutes a row's own pieces
          for (int e = lane; e < kChunkKeys * G::kPanels * 8; e += 32) {
            const int row = e / (G::kPanels * 8), pn = (e / 8) % G::kPanels, piece = e % 8;
            if (row >= zfrom || ((bad_mask >> (row / kBlockSize)) & 1u))
              tc::st_shared_v4(dst + pn * G::kPanelBytes + row * 128 + piece * 16, 0u, 0u, 0u, 0u);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(smem_u32(&full[s]));
        }
      }
    }
    if (!ok && lane == 0) abort_all();
    // Copies issued but perhaps never consumed (an aborted CTA): give them a
    // bounded chance to land before the CTA exits.
    if (lane == 0 && s_abort) {
      mbar_wait_bounded(smem_u32(&q_full), 0);
      if (nfix > 0) mbar_wait_bounded(smem_u32(&landed), (nfix - 1) & 1);
      for (int i = max(0, issued - NS); i < issued; ++i)
        mbar_wait_bounded(smem_u32(&full[i % NS]), (i / NS) & 1);
    }
  } else if (warp == kIssuerWarp) {
    // ---- MMA issuer ---------------------------------------------------------------
    if (lane == 0) {
      const uint32_t id_s = tc::instr_desc<T>(kTileRows, kChunkKeys, 0, 0);
      const uint32_t id_o = tc::instr_desc<T>(kTileRows, D, 0, 1);
      // descriptors differ only in their start address (bits 0..13: addr >> 4)
      const uint64_t dk = tc::smem_desc(0, 16, 1024, tc::kSwizzle128);
      const uint64_t dv = tc::smem_desc(0, G::kPanelBytes, 1024, tc::kSwizzle128);
      auto ring = [&](int idx) { return sbase + G::kRingOff + (idx % NS) * G::kStageBytes; };
      auto issue_s = [&](int c, int t) {
        const uint32_t qa = sbase + t * G::kStageBytes, ka = ring(2 * c);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * G::kPanelBytes + (ks & 3) * 32;
          tc::mma(tmem + t * kChunkKeys, dk | ((qa + off) >> 4), dk | ((ka + off) >> 4), id_s,
                  ks > 0);
        }
        tc::commit(smem_u32(&s_full[t]));
      };
      auto issue_o = [&](int c, int t) {
        const uint32_t va = ring(2 * c + 1);
#pragma unroll
        for (int ks = 0; ks < kChunkKeys / 16; ++ks) {
          const uint64_t vb = dv | ((va + ks * 16 * 128) >> 4);
          tc::mma_ts(tmem + G::kOCol + t * D, tmem + t * kChunkKeys + ks * 8, vb, id_o,
                     c > 0 || ks > 0);
          if constexpr (kSplitP<T>)
            tc::mma_ts(tmem + G::kOCol + t * D, tmem + t * kChunkKeys + 64 + ks * 8, vb, id_o,
                       true);
        }
        tc::commit(smem_u32(&pv_done[t]));
      };
      auto full_wait = [&](int idx) {
        return mbar_wait_bounded(smem_u32(&full[idx % NS]), (idx / NS) & 1);
      };
      bool ok = mbar_wait_bounded(smem_u32(&q_full), 0) && full_wait(0);
      if (ok) {
        tc::fence_after();
        for (int t = 0; t < w.tiles; ++t) issue_s(0, t);
        tc::commit(smem_u32(&empty[0]));
      }
      for (int c = 0; ok && c < n_chunks; ++c) {
        if (!full_wait(2 * c + 1)) {
          ok = false;
          break;
        }
        bool next_k = false;
        for (int t = 0; t < w.tiles && ok; ++t) {
          if (c >= w.chunks[t]) continue;
          if (!mbar_wait_bounded(smem_u32(&p_full[t]), c & 1)) {
            ok = false;
            break;
          }
          tc::fence_after();
          issue_o(c, t);
          if (c + 1 < w.chunks[t]) {
            // S_{c+1} overwrites the columns P_c is read from: after P.V
            if ((!next_k && !full_wait(2 * c + 2)) ||
                !mbar_wait_bounded(smem_u32(&pv_done[t]), c & 1)) {
              ok = false;
              break;
            }
            next_k = true;
            tc::fence_after();
            issue_s(c + 1, t);
          }
        }
        if (!ok) break;
        tc::commit(smem_u32(&empty[(2 * c + 1) % NS]));
        if (next_k) tc::commit(smem_u32(&empty[(2 * c + 2) % NS]));
      }
      if (!ok) abort_all();
      // every MMA issued has completed before TMEM is released
      tc::commit(smem_u32(&mma_idle));
      mbar_wait_bounded(smem_u32(&mma_idle), 0);
    }
    __syncwarp();
  } else {
    // ---- softmax and epilogue: one query row per thread ----------------------------
    const int t = warp / 4, quad = warp % 4;
    if (t < w.tiles) {
      const int r = w.row0 + t * kTileRows + quad * 32 + lane;
      const bool valid = r < w.row0 + w.rows;
      const int j = r / p.group, h = r - j * p.group;
      const int lim = valid ? w.L - w.qlen + j : -1;  // the last key this row sees
      const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
      const uint32_t s_addr = tmem + lane_base + t * kChunkKeys;
      const uint32_t o_addr = tmem + lane_base + G::kOCol + t * D;
      const int nch = w.chunks[t];
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      for (int c = 0; c < nch; ++c) {
        const int nb = min(kChunkBlocks, w.nblk - c * kChunkBlocks);
        const int entry = lane < nb ? __ldg(table + c * kChunkBlocks + lane) : 0;
        const uint32_t bad_mask = __ballot_sync(
            kFull, lane < nb && (entry < 0 || static_cast<int64_t>(entry) >= p.num_blocks));
        const bool wt = mbar_wait_bounded(smem_u32(&s_full[t]), c & 1);
        if (!__all_sync(kFull, wt && !s_abort)) {
          ok = false;
          break;
        }
        tc::fence_after();
        uint32_t sr[kChunkKeys / 32][32];
#pragma unroll
        for (int q = 0; q < kChunkKeys / 32; ++q) tc::tmem_ld32(s_addr + 32 * q, sr[q]);
        tc::tmem_wait_ld();
        const int key0 = c * kChunkKeys;
        const bool need_mask = key0 + kChunkKeys - 1 > lim || bad_mask != 0;
        float mc = -INFINITY;
#pragma unroll
        for (int k = 0; k < kChunkKeys; ++k) {
          float x = __uint_as_float(sr[k / 32][k % 32]) * p.scale_log2;
          if (need_mask && (key0 + k > lim || ((bad_mask >> (k / kBlockSize)) & 1u)))
            x = -INFINITY;
          sr[k / 32][k % 32] = __float_as_uint(x);
          mc = fmaxf(mc, x);
        }
        const bool raise = mc > m_ref + kRescaleSlack;
        const float m_new = raise ? mc : m_ref;
        const float alpha = !raise ? 1.f : (m_ref == -INFINITY ? 0.f : ex2(m_ref - m_new));
        l *= alpha;
        if (c > 0 && __any_sync(kFull, raise)) {
          // P.V of chunk c - 1 has completed: S_c was computed after it
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            tc::tmem_ld32(o_addr + 32 * q, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::tmem_st32(o_addr + 32 * q, o);
          }
        }
        m_ref = m_new;
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        float rs = 0.f;
        if constexpr (kSplitP<T>) {
          // the 64 columns of P's high part, then the 64 of its remainder
          // (S_t has been read in full into registers)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int k = 64 * q + 2 * e;
              const float a = ex2(__uint_as_float(sr[k / 32][k % 32]) - m_use);
              const float b = ex2(__uint_as_float(sr[k / 32][k % 32 + 1]) - m_use);
              rs += a + b;
              const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
              hi[e] = *reinterpret_cast<const uint32_t *>(&h);
              lo[e] = pack2<T>(a - __low2float(h), b - __high2float(h));
            }
            tc::tmem_st32(s_addr + 32 * q, hi);
            tc::tmem_st32(s_addr + 64 + 32 * q, lo);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int k = 64 * q + 2 * e;
              const float a = ex2(__uint_as_float(sr[k / 32][k % 32]) - m_use);
              const float b = ex2(__uint_as_float(sr[k / 32][k % 32 + 1]) - m_use);
              rs += a + b;
              pk[e] = pack2<T>(a, b);
            }
            tc::tmem_st32(s_addr + 32 * q, pk);
          }
        }
        l += rs;
        tc::tmem_wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(smem_u32(&p_full[t]));
      }
      if (ok) {
        const bool wt = mbar_wait_bounded(smem_u32(&pv_done[t]), (nch - 1) & 1);
        ok = __all_sync(kFull, wt && !s_abort);
      }
      if (ok) {
        tc::fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        T *orow = reinterpret_cast<T *>(p.out) +
                  (static_cast<int64_t>(w.q0 + j) * p.num_heads + w.kvh * p.group + h) * D;
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tc::tmem_ld32(o_addr + 32 * q, o);
          tc::tmem_wait_ld();
          if (valid) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack2<T>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
            uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * q);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
        }
      }
      if (!ok && lane == 0) abort_all();
    }
  }

  tc::fence_before();
  __syncthreads();
  if (warp == kIssuerWarp) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, G::kTmemCols);
  }
}

// ---- host side -----------------------------------------------------------------
constexpr int kDefaultStages128 = 4, kDefaultStages64 = 8;

template <typename T, int D, int NS>
cudaError_t launch_t(const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                     const PrefillParams &p, cudaStream_t stream) {
  using G = Geom<D, NS>;
  const size_t smem = G::kBytes + 1024;  // + alignment slack
  const cudaError_t e = cudaFuncSetAttribute(
      prefill_kernel<T, D, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid(p.num_kv_heads, p.batch, p.pairs);
  prefill_kernel<T, D, NS><<<grid, kThreads, smem, stream>>>(qmap, kmap, vmap, p);
  return cudaGetLastError();
}

using LaunchFn = cudaError_t (*)(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                 const PrefillParams &, cudaStream_t);

template <typename T> LaunchFn pick_t(int D, int stages) {
  if (D == 128) {
    switch (stages == 0 ? kDefaultStages128 : stages) {
      case 3: return launch_t<T, 128, 3>;
      case 4: return launch_t<T, 128, 4>;
      case 5: return launch_t<T, 128, 5>;
      default: return nullptr;
    }
  }
  if (D == 64) {
    switch (stages == 0 ? kDefaultStages64 : stages) {
      case 4: return launch_t<T, 64, 4>;
      case 6: return launch_t<T, 64, 6>;
      case 8: return launch_t<T, 64, 8>;
      default: return nullptr;
    }
  }
  return nullptr;
}

LaunchFn pick(pkv_dtype dtype, int D, int stages) {
  if (dtype == PKV_BF16) return pick_t<__nv_bfloat16>(D, stages);
  if (dtype == PKV_F16) return pick_t<__half>(D, stages);
  return nullptr;
}

}  // namespace prefill

bool prefill_supported(pkv_dtype dtype, int head_dim, int group, int stages) {
  return group >= 1 && group <= prefill::kTileRows && prefill::kTileRows % group == 0 &&
         prefill::pick(dtype, head_dim, stages) != nullptr;
}

int prefill_rows_per_cta() { return prefill::kCtaRows; }

cudaError_t prefill_launch(pkv_dtype dtype, int head_dim, int stages, const CUtensorMap &qmap,
                           const CUtensorMap &kmap, const CUtensorMap &vmap,
                           const PrefillParams &p, cudaStream_t stream) {
  const prefill::LaunchFn fn = prefill::pick(dtype, head_dim, stages);
  if (!fn) return cudaErrorInvalidValue;
  return fn(qmap, kmap, vmap, p, stream);
}

}  // namespace pkv
