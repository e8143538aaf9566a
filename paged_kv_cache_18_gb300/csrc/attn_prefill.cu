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
// One CTA per 256 query rows of one (sequence, KV head), longest first.  A row is a (query
// position, head of the KV head's group) pair, so each K/V chunk streamed
// once serves every query head that shares the KV head.  352 threads:
//   warps 0-3 / 4-7  softmax and epilogue of query tile 0 / 1 (128 rows
//                    each, one row per thread: TMEM lane = row); the two
//                    tiles' softmaxes take turns chunk by chunk;
//   warp 8           TMA producer: the Q tiles, then K and V chunks of CK
//                    keys (CK / 16 blocks through the block table) into a
//                    ring of NS stages, K and V alternating;
//   warps 9 / 10     MMA issuer of tile 0 / 1 (one lane each); warp 9 owns
//                    the TMEM allocation.
// Per chunk c of CK keys (64, or 128) and tile t:
//   S[128 x CK] = Q_t[128 x D] . K_c^T    (TMEM, fp32; 64-key chunks: buffer
//                                          c & 1 of the tile, so S_{c+1} is
//                                          computed while the softmax works
//                                          on S_c; 128-key chunks: one buffer)
//   softmax per row, thread-local: masked scores in log2 units, a lazy
//   reference max m (raised, with l and O rescaled, only when a score exceeds
//   it by more than 2^8), P = 2^(s - m) written back over the S buffer in the
//   16-bit input type, each 32-key group over its own 32 columns: for bf16 a
//   high part (16 columns) and the remainder P - high (16), since one bf16
//   rounding of P alone costs about 1.6e-3 of relative L2 error, as much as
//   the output's own rounding; f16 (11 significant bits) needs no remainder
//   O_t[128 x D] += P[128 x CK] . V_c[CK x D]   (A read from TMEM; bf16: a
//                                               second product with the
//                                               remainder)
// TMEM: 128 S columns (two buffers of 64, or one of 128) and O (D columns)
// per tile, 512 columns: one CTA per SM.  (With 128-key chunks each tile's
// softmax waits for its own P.V and next S; the 64-key default does not.)
// While one tile's softmax runs, the tensor cores run the other tile's P.V
// and next S: the two tiles' work interleaves.
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
constexpr int kCostKeys = 64;                      // keys per unit of the work order's cost
constexpr int kSoftmaxWarps = 4 * kTiles;          // one per TMEM lane quadrant per tile
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kIssuerWarp = kSoftmaxWarps + 1;     // tile t's MMAs: warp kIssuerWarp + t
constexpr int kThreads = (kSoftmaxWarps + 1 + kTiles) * 32;
constexpr float kRescaleSlack = 8.f;
// Named barrier 1 + t: tile t's softmax hands over to the other tile's.

// CK keys per chunk (the N of S): 128 with one S buffer per tile, or 64 with
// two (S of the next chunk computed during the softmax of this one).
template <int D, int NS, int CK> struct Geom {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int kPanels = D / 64;                        // 128-byte column panels
  static constexpr int kQPanelBytes = kTileRows * 128;          // 128 rows x 128 B
  static constexpr int kQBytes = kPanels * kQPanelBytes;        // one Q tile
  static constexpr int kKVPanelBytes = CK * 128;                // CK rows x 128 B
  static constexpr int kStageBytes = kPanels * kKVPanelBytes;   // one K or V chunk
  static constexpr int kRingOff = kTiles * kQBytes;
  static constexpr int kBytes = kRingOff + NS * kStageBytes;
  static constexpr uint32_t kTmemCols = 512;
  // tile t: S (and P over it) of chunk c at column 128 t + CK (c % kBufs);
  // O_t at kOCol + D t
  static constexpr int kBufs = 128 / CK;
  static constexpr int kOCol = kTiles * 128;
  static_assert(kOCol + kTiles * D <= 512, "TMEM columns");
};

// Packed pairs of floats (the f32x2 arithmetic of sm_100 and later: one
// instruction for both halves).
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2unpack(uint64_t r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

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
  int chunks0, chunks1;  // chunks tile 0 / tile 1 reads
  int nblk;           // cache blocks the CTA reads
  __device__ __forceinline__ int chunks(int t) const { return t == 0 ? chunks0 : chunks1; }
};

// A sequence's extent: its chunk rows, cached rows and CTA row pairs (256
// (position, head) rows each); a sequence whose query_start / context_lens
// break the rules has no pairs.
struct SeqShape {
  int q0, qlen, L, pairs;
};
__device__ __forceinline__ SeqShape seq_shape(const PrefillParams &p, int b) {
  SeqShape q;
  const int q0 = __ldg(p.query_start + b), q1 = __ldg(p.query_start + b + 1);
  q.L = __ldg(p.context_lens + b);
  q.q0 = q0;
  const bool sane = q0 >= 0 && q1 >= q0 && q1 <= p.total_q && q1 - q0 <= p.max_query_len &&
                    q.L >= q1 - q0 &&
                    static_cast<int64_t>(q.L) <=
                        static_cast<int64_t>(p.max_blocks_per_seq) * kBlockSize;
  q.qlen = sane ? q1 - q0 : 0;
  q.pairs = (q.qlen * p.group + kCtaRows - 1) / kCtaRows;
  return q;
}
// Chunks the CTA of row pair `pair` runs (those of its last row): the cost
// that orders the work.  Non-decreasing in `pair`.
__device__ __forceinline__ int pair_cost(const SeqShape &q, int group, int pair) {
  const int last = min(pair * kCtaRows + kCtaRows, q.qlen * group) - 1;
  return (q.L - q.qlen + last / group) / kCostKeys + 1;
}
// First pair of the sequence whose cost is at least v (q.pairs if none).
__device__ __forceinline__ int first_pair_at_least(const SeqShape &q, int group, int v) {
  int lo = 0, hi = q.pairs;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (pair_cost(q, group, mid) >= v)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo;
}

// CTAs take the (sequence, row pair) units longest first: the hardware starts
// CTAs in index order as SMs free up, so this is a longest-first list
// schedule (the costs differ by up to the ratio of the longest context to
// the shortest).  Unit rank r (descending cost; ties by sequence, then pair)
// is found by each warp on its own: a binary search over the cost value of
// the count of units at or above it (per sequence a binary search over its
// pairs), then a walk over the sequences within that cost.  Returns
// false when rank r has no unit.
__device__ __forceinline__ bool locate_unit(const PrefillParams &p, int r, int *b_out,
                                            int *pair_out) {
  const int lane = threadIdx.x & 31;
  auto count_ge = [&](int v) {
    int n = 0;
    for (int b = lane; b < p.batch; b += 32) {
      const SeqShape q = seq_shape(p, b);
      n += q.pairs - first_pair_at_least(q, p.group, v);
    }
    return __reduce_add_sync(kFull, n);
  };
  int vmax = 0;
  for (int b = lane; b < p.batch; b += 32) {
    const SeqShape q = seq_shape(p, b);
    if (q.pairs > 0) vmax = max(vmax, pair_cost(q, p.group, q.pairs - 1));
  }
  vmax = __reduce_max_sync(kFull, vmax);
  if (vmax == 0 || count_ge(1) <= r) return false;
  int lo = 1, hi = vmax;  // the largest v with count_ge(v) > r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (count_ge(mid) > r)
      lo = mid;
    else
      hi = mid - 1;
  }
  int skip = r - (lo < vmax ? count_ge(lo + 1) : 0);  // units of cost lo before rank r
  for (int b0 = 0; b0 < p.batch; b0 += 32) {
    const int b = b0 + lane;
    int f = 0, m = 0;
    if (b < p.batch) {
      const SeqShape q = seq_shape(p, b);
      f = first_pair_at_least(q, p.group, lo);
      m = first_pair_at_least(q, p.group, lo + 1) - f;
    }
    int incl = m;  // inclusive prefix sum over the lanes
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, d);
      if (lane >= d) incl += y;
    }
    const int total = __shfl_sync(kFull, incl, 31);
    if (skip < total) {
      const int src = __ffs(__ballot_sync(kFull, incl > skip)) - 1;
      const int before = __shfl_sync(kFull, incl - m, src);
      *b_out = b0 + src;
      *pair_out = __shfl_sync(kFull, f, src) + (skip - before);
      return true;
    }
    skip -= total;
  }
  return false;  // (not reached when the counts agree)
}

template <int CK> __device__ __forceinline__ Work make_work(const PrefillParams &p) {
  Work w;
  w.kvh = static_cast<int>(blockIdx.x % p.num_kv_heads);
  int pair = 0;
  if (!locate_unit(p, static_cast<int>(blockIdx.x / p.num_kv_heads), &w.b, &pair)) {
    w.rows = 0;
    return w;
  }
  const SeqShape q = seq_shape(p, w.b);
  w.q0 = q.q0;
  w.qlen = q.qlen;
  w.L = q.L;
  w.row0 = pair * kCtaRows;
  w.rows = min(kCtaRows, w.qlen * p.group - w.row0);
  w.tiles = w.rows > kTileRows ? 2 : 1;
  // the last key each tile's rows see
  const int lim0 = w.L - w.qlen + (w.row0 + min(kTileRows, w.rows) - 1) / p.group;
  const int lim1 = w.L - w.qlen + (w.row0 + w.rows - 1) / p.group;
  w.chunks0 = lim0 / CK + 1;
  w.chunks1 = w.tiles == 2 ? lim1 / CK + 1 : 0;
  w.nblk = (w.tiles == 2 ? lim1 : lim0) / kBlockSize + 1;
  return w;
}

// Sequences that break the rules are recorded once (by the first CTA).
__device__ __forceinline__ void check_sequences(const PrefillParams &p) {
  if (blockIdx.x != 0 || threadIdx.x >= 32) return;
  bool bad = false;
  for (int b = threadIdx.x; b < p.batch; b += 32) {
    const int q0 = __ldg(p.query_start + b), q1 = __ldg(p.query_start + b + 1);
    bad |= seq_shape(p, b).qlen == 0 && q1 != q0;
  }
  if (__any_sync(kFull, bad) && threadIdx.x == 0) record_error(p.err, PKV_DEVERR_CONTEXT_LEN);
}

template <typename T, int D, int NS, int CK>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  using G = Geom<D, NS, CK>;
  constexpr int kChunkKeys = CK, kChunkBlocks = CK / kBlockSize, kBufs = G::kBufs;
  constexpr int kHalves = CK / 64;  // 64-key halves of a chunk in the softmax
  check_sequences(p);
  const Work w = make_work<CK>(p);
  if (w.rows <= 0) return;  // the whole CTA, before any barrier or TMEM use

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  // per tile and S buffer u (chunk c uses u = c % kBufs)
  __shared__ uint64_t full[NS], empty[NS], q_full, landed, s_full[kTiles][2], p_full[kTiles][2],
      pv_done[kTiles][2], mma_idle[kTiles];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kTiles);  // one release per tile's issuer
    }
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&landed), 1);
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(smem_u32(&mma_idle[t]), 1);
      for (int u = 0; u < 2; ++u) {
        mbar_init(smem_u32(&s_full[t][u]), 1);
        mbar_init(smem_u32(&p_full[t][u]), 4);
        mbar_init(smem_u32(&pv_done[t][u]), 1);
      }
    }
    fence_mbar_init();
  }
  if (warp == kIssuerWarp) tc::tmem_alloc(smem_u32(&tmem_base_s), G::kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_base_s;
  const int32_t *table = p.block_table + static_cast<int64_t>(w.b) * p.max_blocks_per_seq;
  const int n_chunks = w.chunks(w.tiles - 1);
  auto abort_all = [&]() {
    s_abort = 1;
    record_error(p.err, PKV_DEVERR_TIMEOUT);
  };

  if (warp == kProducerWarp) {
    // ---- TMA producer ----------------------------------------------------------
    bool ok = true;
    int issued = 0;
    uint32_t nfix = 0;
    if (lane == 0) mbar_arrive_expect_tx(smem_u32(&q_full), w.tiles * G::kQBytes);
    __syncwarp();
    if (lane < w.tiles * G::kPanels) {
      // a Q tile: 128 / group positions x the group's heads, one 128-byte
      // panel per box; rows past the query tensor read as zero
      const int t = lane / G::kPanels, pn = lane % G::kPanels;
      tma_load_3d(sbase + t * G::kQBytes + pn * G::kQPanelBytes, &qmap, smem_u32(&q_full),
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
            tma_load_4d(dst + pn * G::kKVPanelBytes + lane * kBlockSize * 128,
                        kv ? &vmap : &kmap, bar, pn * 64, 0, w.kvh, entry);
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
              tc::st_shared_v4(dst + pn * G::kKVPanelBytes + row * 128 + piece * 16, 0u, 0u, 0u,
                               0u);
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
  } else if (warp >= kIssuerWarp) {
    // ---- MMA issuers: one thread per tile ----------------------------------------
    // Chunk c: S_c into the tile's buffer c % kBufs (64-key chunks: two
    // chunks ahead, so S_{c+1} is there when the softmax finishes chunk c),
    // then P_c . V_c once the softmax has written P_c over S_c.  Each tile
    // has its own issuing thread, so one tile's waits never hold up the
    // other's MMAs; every K / V stage is released by both (a tile that is
    // done, or absent, releases the stages it no longer reads as they arrive).  The issuers poll their barriers
    // (no suspension): their wake-up is on the critical path.
    const int t = warp - kIssuerWarp;
    if (lane == 0) {
      const uint32_t id_s = tc::instr_desc<T>(kTileRows, kChunkKeys, 0, 0);
      const uint32_t id_o = tc::instr_desc<T>(kTileRows, D, 0, 1);
      // descriptors differ only in their start address (bits 0..13: addr >> 4)
      const uint64_t dk = tc::smem_desc(0, 16, 1024, tc::kSwizzle128);
      const uint64_t dv = tc::smem_desc(0, G::kKVPanelBytes, 1024, tc::kSwizzle128);
      const int mine = t < w.tiles ? w.chunks(t) : 0;
      auto ring = [&](int idx) { return sbase + G::kRingOff + (idx % NS) * G::kStageBytes; };
      auto sbuf = [&](int c) { return tmem + t * 128 + (c % kBufs) * kChunkKeys; };
      auto issue_s = [&](int c) {
        const uint32_t qa = sbase + t * G::kQBytes, ka = ring(2 * c);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t offq = (ks >> 2) * G::kQPanelBytes + (ks & 3) * 32;
          const uint32_t offk = (ks >> 2) * G::kKVPanelBytes + (ks & 3) * 32;
          tc::mma(sbuf(c), dk | ((qa + offq) >> 4), dk | ((ka + offk) >> 4), id_s, ks > 0);
        }
        tc::commit(smem_u32(&s_full[t][c % kBufs]));
      };
      auto issue_o = [&](int c) {
        const uint32_t va = ring(2 * c + 1);
#pragma unroll
        for (int ks = 0; ks < kChunkKeys / 16; ++ks) {
          // keys 16 ks .. 16 ks + 15: P columns of 32-key group ks / 2
          const uint64_t vb = dv | ((va + ks * 16 * 128) >> 4);
          const uint32_t pc = sbuf(c) + 32 * (ks >> 1) + 8 * (ks & 1);
          tc::mma_ts(tmem + G::kOCol + t * D, pc, vb, id_o, c > 0 || ks > 0);
          if constexpr (kSplitP<T>) tc::mma_ts(tmem + G::kOCol + t * D, pc + 16, vb, id_o, true);
        }
        tc::commit(smem_u32(&pv_done[t][c % kBufs]));
      };
      auto spin = [&](uint64_t &bar, uint32_t parity) {
        return tc::mbar_spin_bounded(smem_u32(&bar), parity);
      };
      auto full_wait = [&](int idx) { return spin(full[idx % NS], (idx / NS) & 1); };
      // release a stage: when this thread's MMAs reading it complete, or now
      auto release = [&](int idx, bool read) {
        if (read)
          tc::commit(smem_u32(&empty[idx % NS]));
        else
          tc::mbar_arrive(smem_u32(&empty[idx % NS]));
      };
      bool ok = spin(q_full, 0);
      for (int c = 0; ok && c < kBufs && c < n_chunks; ++c) {
        if (!full_wait(2 * c)) {
          ok = false;
          break;
        }
        if (c < mine) {
          tc::fence_after();
          issue_s(c);
        }
        release(2 * c, c < mine);
      }
      for (int c = 0; ok && c < n_chunks; ++c) {
        if (!full_wait(2 * c + 1)) {
          ok = false;
          break;
        }
        if (c < mine) {
          if (!spin(p_full[t][c % kBufs], (c / kBufs) & 1)) {
            ok = false;
            break;
          }
          tc::fence_after();
          issue_o(c);
        }
        release(2 * c + 1, c < mine);
        if (c + kBufs < n_chunks) {
          if (!full_wait(2 * (c + kBufs))) {
            ok = false;
            break;
          }
          if (c + kBufs < mine) {
            // S_{c+kBufs} overwrites the buffer P_c is read from: after P_c . V_c
            if (!spin(pv_done[t][c % kBufs], (c / kBufs) & 1)) {
              ok = false;
              break;
            }
            tc::fence_after();
            issue_s(c + kBufs);
          }
          release(2 * (c + kBufs), c + kBufs < mine);
        }
      }
      if (!ok) abort_all();
      // every MMA this thread issued has completed before TMEM is released
      tc::commit(smem_u32(&mma_idle[t]));
      spin(mma_idle[t], 0);
    }
    __syncwarp();
  } else {
    // ---- softmax and epilogue: one query row per thread ----------------------------
    // Warp w: tile t = w / 4, TMEM lane quadrant w % 4.  The two tiles'
    // softmaxes take turns (tile 0's chunk c, tile 1's chunk c, tile 0's
    // chunk c + 1, ...), so each has the SM's issue slots and exp2 units to
    // itself while the tensor cores work on the other tile.  The hand-over is
    // a pair of named barriers (one tile's 128 threads arrive, the other's
    // wait); a warp that has given up keeps executing the same sequence of
    // them, so no warp is ever left waiting at one.
    const int t = warp / 4, quad = warp % 4;
    if (t < w.tiles) {
      const int r = w.row0 + t * kTileRows + quad * 32 + lane;
      const bool valid = r < w.row0 + w.rows;
      const int j = r / p.group, h = r - j * p.group;
      const int lim = valid ? w.L - w.qlen + j : -1;  // the last key this row sees
      const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
      const uint32_t o_addr = tmem + lane_base + G::kOCol + t * D;
      const int nch = w.chunks(t);
      const bool turns = w.tiles == 2;
      const int n_other = turns ? w.chunks(1 - t) : 0;
      // The barriers order memory, not arithmetic: the exp2 work is pure
      // register arithmetic, which the compiler may move across them.  So the
      // wait hands out, from the same asm statement, a value the exp2 loop
      // consumes (it cannot start before the wait), and the hand-over takes
      // the loop's row sums as inputs (it cannot leave before the loop ends).
      // (Immediate barrier ids: a bar.arrive / bar.sync pair naming its
      // barrier through a register measured as not waiting on this GPU.)
      auto turn_wait = [&](int c, float dep) -> float {  // before chunk c's exp2
        const int oc = t == 0 ? c - 1 : c;
        if (turns && oc >= 0 && oc < n_other) {
          if (t == 0)  // tile 1's hand-over
            asm volatile("bar.sync 2, 256;\n\tmov.b32 %0, %0;" : "+f"(dep) : : "memory");
          else         // tile 0's hand-over
            asm volatile("bar.sync 1, 256;\n\tmov.b32 %0, %0;" : "+f"(dep) : : "memory");
        }
        return dep;
      };
      auto turn_pass = [&](int c, uint64_t dep0, uint64_t dep1) {  // after chunk c's exp2
        const int oc = t == 0 ? c : c + 1;  // its chunk that waits for this one
        if (turns && oc < n_other) {
          if (t == 0)
            asm volatile("bar.arrive 1, 256;" ::"l"(dep0), "l"(dep1) : "memory");
          else
            asm volatile("bar.arrive 2, 256;" ::"l"(dep0), "l"(dep1) : "memory");
        }
      };
      const float sl = p.scale_log2;
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      // A warp whose 32 rows are all past the tile's last row (a short
      // chunk) has no softmax to do: it only keeps pace with the chunks
      // (waits for S so that it never arrives for a chunk two ahead) and
      // releases P; the P.V rows it leaves are never stored.
      const bool idle = w.row0 + t * kTileRows + quad * 32 >= w.row0 + w.rows;
      // block-table entries of a chunk (lanes 0..3), loaded one chunk ahead
      auto table_entry = [&](int c) {
        const int nb = min(kChunkBlocks, w.nblk - c * kChunkBlocks);
        return lane < nb ? __ldg(table + c * kChunkBlocks + lane) : 0;
      };
      int entry_next = idle ? 0 : table_entry(0);
      for (int c = 0; c < nch; ++c) {
        const uint32_t s_addr = tmem + lane_base + t * 128 + (c % kBufs) * kChunkKeys;
        const int key0 = c * kChunkKeys;
        uint32_t va[32], vb[32];
        uint32_t bad_mask = 0;
        if (idle) {
          if (ok) {
            const bool wt = mbar_wait_bounded(smem_u32(&s_full[t][c % kBufs]), (c / kBufs) & 1);
            ok = __all_sync(kFull, wt && !s_abort);
          }
          turn_wait(c, 0.f);
          if (ok && lane == 0) tc::mbar_arrive(smem_u32(&p_full[t][c % kBufs]));
          turn_pass(c, 0ull, 0ull);
          continue;
        }
        if (ok) {
          const int nb = min(kChunkBlocks, w.nblk - c * kChunkBlocks);
          const int entry = entry_next;
          if (c + 1 < nch) entry_next = table_entry(c + 1);
          bad_mask = __ballot_sync(
              kFull, lane < nb && (entry < 0 || static_cast<int64_t>(entry) >= p.num_blocks));
          const bool wt = mbar_wait_bounded(smem_u32(&s_full[t][c % kBufs]), (c / kBufs) & 1);
          ok = __all_sync(kFull, wt && !s_abort);
          if (ok) {
            tc::fence_after();
            tc::tmem_ld32(s_addr, va);
            tc::tmem_ld32(s_addr + 32, vb);
          }
        }
        if (!ok) {
          turn_wait(c, 0.f);
          turn_pass(c, 0ull, 0ull);
          continue;
        }
        // keys this row may not see (past its last key, or in a bad block):
        // score -inf (g: the chunk's 32-key group)
        auto mask32 = [&](uint32_t(&v)[32], int g) {
          if (key0 + 32 * g + 31 > lim || ((bad_mask >> (2 * g)) & 3u) != 0) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int k = 32 * g + e;
              if (key0 + k > lim || ((bad_mask >> (k / kBlockSize)) & 1u))
                v[e] = __float_as_uint(-INFINITY);
            }
          }
        };
        // one 64-key half of the chunk's scores into va / vb, masked
        auto load_half = [&](int hh) {
          tc::tmem_ld32(s_addr + 64 * hh, va);
          tc::tmem_ld32(s_addr + 64 * hh + 32, vb);
          tc::tmem_wait_ld_regs(va);
          tc::tmem_wait_ld_regs(vb);
          mask32(va, 2 * hh);
          mask32(vb, 2 * hh + 1);
        };
        // the chunk's largest raw score (the scale is positive, so scaling
        // after the maximum is the same); a 128-key chunk is read in two
        // halves, the second staying in registers for the exp2 pass
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        auto max_half = [&]() {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            mx[0] = fmaxf(mx[0], __uint_as_float(va[e]));
            mx[1] = fmaxf(mx[1], __uint_as_float(va[e + 1]));
            mx[2] = fmaxf(mx[2], __uint_as_float(vb[e]));
            mx[3] = fmaxf(mx[3], __uint_as_float(vb[e + 1]));
          }
        };
        tc::tmem_wait_ld_regs(va);
        tc::tmem_wait_ld_regs(vb);
        mask32(va, 0);
        mask32(vb, 1);
        max_half();
#pragma unroll 1
        for (int hh = 1; hh < kHalves; ++hh) {
          load_half(hh);
          max_half();
        }
        const float mc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl;
        const bool raise = mc > m_ref + kRescaleSlack;
        const float m_new = raise ? mc : m_ref;
        const float alpha = !raise ? 1.f : (m_ref == -INFINITY ? 0.f : ex2(m_ref - m_new));
        l *= alpha;
        if (c > 0 && __any_sync(kFull, raise)) {
          // O holds P_{c-1} . V_{c-1} once that product has completed
          const bool pw =
              mbar_wait_bounded(smem_u32(&pv_done[t][(c - 1) % kBufs]), ((c - 1) / kBufs) & 1);
          if (!__all_sync(kFull, pw && !s_abort)) {
            ok = false;
            turn_wait(c, 0.f);
            turn_pass(c, 0ull, 0ull);
            continue;
          }
          tc::fence_after();
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            tc::tmem_ld32(o_addr + 32 * q, o);
            tc::tmem_wait_ld_regs(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::tmem_st32(o_addr + 32 * q, o);
          }
        }
        m_ref = m_new;
        // P = 2^(s scale_log2 - m) written over each 32-key group's own S
        // columns: the high part in its first 16, the remainder in the other
        // 16 (f16: P alone in the first 16)
        // (pairs of scores in f32x2 arithmetic: the scale-and-shift, the
        // row-sum accumulation and the remainder of the bf16 split)
        // the exp2 phase is the part the tiles take turns at: the other
        // tile's loads, maximum and rescale test overlap it
        const float neg_m = turn_wait(c, m_ref == -INFINITY ? 0.f : -m_ref);
        const uint64_t sl2 = f2pack(sl, sl), nm2 = f2pack(neg_m, neg_m);
        uint64_t rs2[2] = {0ull, 0ull};  // (+0.0f, +0.0f)
#pragma unroll 1
        for (int hh = kHalves - 1; hh >= 0; --hh) {
          if (hh < kHalves - 1) load_half(hh);  // (the last half read is still in va / vb)
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const uint32_t(&v)[32] = g ? vb : va;
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const uint64_t t2 =
                  ffma2(f2pack(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sl2, nm2);
              const float2 t = f2unpack(t2);
              const float x = ex2(t.x), y = ex2(t.y);
              const uint64_t pxy = f2pack(x, y);
              rs2[e & 1] = fadd2(rs2[e & 1], pxy);
              if constexpr (kSplitP<T>) {
                const __nv_bfloat162 hv = __floats2bfloat162_rn(x, y);
                const uint32_t hb = *reinterpret_cast<const uint32_t *>(&hv);
                hi[e] = hb;
                const float2 r = f2unpack(fsub2(
                    pxy, f2pack(__uint_as_float(hb << 16), __uint_as_float(hb & 0xffff0000u))));
                lo[e] = pack2<T>(r.x, r.y);
              } else {
                hi[e] = pack2<T>(x, y);
              }
            }
            tc::tmem_st16u(s_addr + 64 * hh + 32 * g, hi);
            if constexpr (kSplitP<T>) tc::tmem_st16u(s_addr + 64 * hh + 32 * g + 16, lo);
          }
        }
        turn_pass(c, rs2[0], rs2[1]);
        const float2 ra = f2unpack(rs2[0]), rb = f2unpack(rs2[1]);
        l += (ra.x + ra.y) + (rb.x + rb.y);
        tc::tmem_wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(smem_u32(&p_full[t][c % kBufs]));
      }
      if (ok && !idle) {
        const bool wt =
            mbar_wait_bounded(smem_u32(&pv_done[t][(nch - 1) % kBufs]), ((nch - 1) / kBufs) & 1);
        ok = __all_sync(kFull, wt && !s_abort);
      }
      if (ok && !idle) {
        tc::fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        T *orow = reinterpret_cast<T *>(p.out) +
                  (static_cast<int64_t>(w.q0 + j) * p.num_heads + w.kvh * p.group + h) * D;
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tc::tmem_ld32(o_addr + 32 * q, o);
          tc::tmem_wait_ld_regs(o);
          if (valid) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack2<T>(__uint_as_float(o[2 * e]) * inv,
                               __uint_as_float(o[2 * e + 1]) * inv);
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
// `stages` is the K / V ring depth in chunks; it also chooses the chunk:
// head_dim 128: 3-5 stages of 128-key chunks, 6 or 8 of 64-key ones;
// head_dim 64: 4-8 stages of 128-key chunks, 12 or 16 of 64-key ones.
// 64-key chunks are the default: with 128-key ones each tile's softmax also
// waits for its own P.V and next S (one S buffer), and the Llama-3-8B-shaped
// prefill (head_dim 128) ran at 521-537 TFLOP/s against 603-617.
constexpr int kDefaultStages128 = 8, kDefaultStages64 = 12;

template <typename T, int D, int NS, int CK>
cudaError_t launch_t(const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                     const PrefillParams &p, cudaStream_t stream) {
  using G = Geom<D, NS, CK>;
  const size_t smem = G::kBytes + 1024;  // + alignment slack
  const cudaError_t e = cudaFuncSetAttribute(prefill_kernel<T, D, NS, CK>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // one CTA per (sequence, row pair, KV head) unit, longest units first
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(p.pairs) * p.batch * p.num_kv_heads));
  prefill_kernel<T, D, NS, CK><<<grid, kThreads, smem, stream>>>(qmap, kmap, vmap, p);
  return cudaGetLastError();
}

using LaunchFn = cudaError_t (*)(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                 const PrefillParams &, cudaStream_t);

template <typename T> LaunchFn pick_t(int D, int stages) {
  if (D == 128) {
    switch (stages == 0 ? kDefaultStages128 : stages) {
      case 3: return launch_t<T, 128, 3, 128>;
      case 4: return launch_t<T, 128, 4, 128>;
      case 5: return launch_t<T, 128, 5, 128>;
      case 6: return launch_t<T, 128, 6, 64>;
      case 8: return launch_t<T, 128, 8, 64>;
      default: return nullptr;
    }
  }
  if (D == 64) {
    switch (stages == 0 ? kDefaultStages64 : stages) {
      case 4: return launch_t<T, 64, 4, 128>;
      case 6: return launch_t<T, 64, 6, 128>;
      case 8: return launch_t<T, 64, 8, 128>;
      case 12: return launch_t<T, 64, 12, 64>;
      case 16: return launch_t<T, 64, 16, 64>;
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
