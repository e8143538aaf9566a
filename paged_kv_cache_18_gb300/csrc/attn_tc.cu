// attn_tc.cu -- paged decode / verification attention on the fifth-generation
// tensor cores (tcgen05), accumulators in tensor memory (TMEM).
//
// Same arithmetic as attn_mma.cuh ("Inference part 1", sections "PagedAttention",
// "FlashAttention" and "FlashDecoding"), organised for tcgen05: one thread
// issues asynchronous 128-row MMAs over eight cache blocks at a time, and the
// softmax runs on values read from TMEM.  It serves tiles of up to 64 query
// rows (NC = 16, 32 or 64 columns): the verification tile of K+1 drafts (or a
// tree's nodes) x the query heads of one KV head, where the mma.sync kernel
// spends its time repeating a per-block chain once per 8-column tile.
//
// One CTA per (split, KV head x row chunk, sequence), 320 threads:
//   warps 0-7  softmax and epilogue; warp w reads TMEM lanes 32 (w % 4) ..
//              32 (w % 4) + 31 -- keys of the current 128-key chunk in S^T,
//              head dims in O^T -- for half w / 4 of the query columns (two
//              warps per lane quadrant keep each warp's chain short);
//   warp 8     TMA producer: K and V tiles of each block, through the block
//              table, into a ring of NS chunk stages;
//   warp 9     MMA issuer (one lane) and TMEM owner.
// Per chunk c of 128 keys (8 blocks):
//   S^T[128 keys x NC] = K_c[128 x D] . Q^T[D x NC]          (TMEM, 2 buffers)
//   softmax over keys per column, lazy per-column reference max m (raised,
//   with l and O rescaled, only when a score exceeds it by more than 2^8:
//   a CTA-wide vote per chunk, a cross-thread max only then)
//   P^T (bf16/f16 high part + remainder) -> shared memory
//   O^T[D x 2 NC] += V_c^T[D x 128] . [P_hi^T P_lo^T][128 x 2 NC]  (TMEM;
//   the two halves are summed at the end)
// Operands: K and Q^T K-major with the 128-byte swizzle (as the TMA writes
// K), V^T MN-major with the 128-byte swizzle (V's own layout), P^T MN-major
// without swizzle.  Keys that no column may see (past the context, past the
// split, bad blocks) get -inf scores and their V rows are zeroed in shared
// memory, so NaN-filled rows never enter an MMA (0 x NaN would be NaN).
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "tc_ptx.cuh"

namespace pkv {
namespace tc {

constexpr int kChunkBlocks = 8;                    // blocks per 128-key chunk
constexpr int kChunkKeys = kChunkBlocks * kBlockSize;
constexpr int kSoftmaxWarps = 8;  // two per TMEM lane quadrant
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kKProducerWarp = kSoftmaxWarps;
constexpr int kIssuerWarp = kSoftmaxWarps + 1;
constexpr int kVProducerWarp = kSoftmaxWarps + 2;
constexpr int kThreads = kSoftmaxThreads + 96;
constexpr float kRescaleSlack = 8.f;

// CTA-wide OR over the 256 softmax threads (named barrier 1).
__device__ __forceinline__ bool softmax_any(bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, 256, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"(v ? 1u : 0u)
      : "memory");
  return out != 0;
}
// CTA-wide AND over the 256 softmax threads (named barrier 1): every wait's
// outcome is decided once for the eight warps, so none of them leaves the
// loop while the others wait at a named barrier.
__device__ __forceinline__ bool softmax_all(bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 1, 256, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"(v ? 1u : 0u)
      : "memory");
  return out != 0;
}
__device__ __forceinline__ void softmax_sync() {
  asm volatile("bar.sync 2, 256;" ::: "memory");
}

// ---- geometry ----------------------------------------------------------------
// Two rings, NS stages for K and NV for V: a stage is one chunk's K (or V)
// tile, two 64-dim panels of 128 rows x 128 B (block j of the chunk at rows
// 16 j .. 16 j + 15).  K is free again as soon as S^T is computed, V only
// after P.V, so V's ring is the one that bounds the copies in flight.
template <int D, int NC, int NS, int NV, int PB, int QB> struct TcGeom {
  static_assert(D == 128, "head_dim 128");
  static constexpr int kPanelBytes = kChunkKeys * 128;      // 16 KB
  static constexpr int kTileBytes = 2 * kPanelBytes;        // 32 KB: one stage
  static constexpr int kVOff = NS * kTileBytes;             // the V ring
  static constexpr int kQtPanelBytes = NC * 128;            // Q^T: NC rows per panel
  static constexpr int kQtOff = (NS + NV) * kTileBytes;     // QB Q^T buffers of 2 panels
  static constexpr int kPOff = kQtOff + QB * 2 * kQtPanelBytes;  // P^T: (high, low) x PB
  static constexpr int kPBytes = kChunkKeys * NC * 2;
  // an item's partial outputs, [column][head dim] fp32, for one bulk store
  static constexpr int kStgOff = kPOff + PB * 2 * kPBytes;
  static constexpr int kBytes = kStgOff + NC * D * 4;
  // S^T (two buffers of NC) and two O^T buffers (items alternate) of 2 NC
  // (NC columns for the high part of P, NC for the remainder, summed at
  // the end)
  static constexpr int kTmemCols = 6 * NC <= 128 ? 128 : (6 * NC <= 256 ? 256 : 512);
};

// Per-stage facts the producer hands to the consumers (published before its
// mbarrier arrive, which orders them).
struct StageInfo {
  int nb;             // blocks present (1..8)
  uint32_t bad_mask;  // bit j: block j's table entry was out of range
};

// --------------------------------------------------------------------------------
//
// NS K stages and NV V stages; PB = 1 or 2 P^T buffers (with one, chunk c's
// softmax writes P^T only after chunk c - 1's P.V has read it); QB = 1 or 2
// Q^T buffers (with one, an item's Q^T is stored once the last S^T of the
// item before has been computed).
// A work item: one split of one (sequence, KV head, row chunk).  Items are
// numbered split-fastest; the persistent CTA g takes items g, g + G, ...,
// every role enumerating the same sequence.
//
// With the device partition (split_target > 0), items are the flat list of
// cta_work in pkv_device.cuh: the kernel's prologue leaves, per sequence b,
// its split count, first item and block count in shared memory (`dev`),
// and item i is found there; its partials go to [item][CTA column].
struct Item {
  int b, kvh, chunk_row, split, L, blk_begin, nspan, n_chunks, ns_b, idx;
  bool valid;
};
struct DevSplits {
  int ns[32], first[32], nb[32], L[32];
  // balanced partition: first[b] = the flat block where sequence b's units
  // start, nb[b] = n_b, L[b] its length; this CTA's blocks [lo, hi) span
  // n_local units from unit u0 on
  int u0, n_local;
  long long lo, hi;
};
__device__ __forceinline__ Item decode_item(const AttnParams &p, int i, bool report,
                                            const DevSplits *dev) {
  Item it;
  it.idx = i;
  if (p.stream_k) {
    // item i: the part of this CTA's range in its i-th unit
    const int units = p.num_kv_heads * p.row_chunks;
    const int U = dev->u0 + i;
    const int b = U / units, u = U - b * units;
    it.b = b;
    it.kvh = u / p.row_chunks;
    it.chunk_row = u - it.kvh * p.row_chunks;
    const int nb = dev->nb[b];
    // the unit's blocks: places s_u .. s_u + nb - 1 of the list
    const long long s_u = static_cast<long long>(dev->first[b]) +
                          static_cast<long long>(u) * (nb + p.sk_weight) + p.sk_weight;
    const long long lo = max(dev->lo, s_u), hi = min(dev->hi, s_u + nb);
    it.valid = hi > lo;
    it.blk_begin = it.valid ? static_cast<int>(lo - s_u) : 0;
    it.nspan = it.valid ? static_cast<int>(hi - lo) : 0;
    it.n_chunks = (it.nspan + kChunkBlocks - 1) / kChunkBlocks;
    it.L = dev->L[b];
    it.split = 0;
    it.ns_b = 0;
    it.idx = static_cast<int>(blockIdx.x) + U;  // the split's slot
    return it;
  }
  if (p.split_target > 0) {
    const int units = p.num_kv_heads * p.row_chunks;
    int b = -1;
    for (int bb = 0; bb < p.batch; ++bb)
      if (i < dev->first[bb] + dev->ns[bb] * units) {
        b = bb;
        break;
      }
    it.valid = b >= 0;
    it.b = b < 0 ? 0 : b;
    const int ns = b < 0 ? 1 : dev->ns[b];
    const int r = b < 0 ? 0 : i - dev->first[b];
    const int u = r / ns;
    it.split = r - u * ns;
    it.kvh = u / p.row_chunks;
    it.chunk_row = u - it.kvh * p.row_chunks;
    const SeqExtent ext = seq_extent(p, it.b, report && it.valid && r == 0);
    it.L = ext.L;
    const int nb = b < 0 ? 0 : dev->nb[b];
    it.blk_begin = static_cast<int>(static_cast<int64_t>(it.split) * nb / ns);
    const int blk_end = static_cast<int>(static_cast<int64_t>(it.split + 1) * nb / ns);
    it.nspan = it.valid ? max(blk_end - it.blk_begin, 0) : 0;
    it.n_chunks = (it.nspan + kChunkBlocks - 1) / kChunkBlocks;
    it.ns_b = ns;
    return it;
  }
  const int ns = p.num_splits, Y = p.num_kv_heads * p.row_chunks;
  it.split = i % ns;
  const int t = i / ns;
  const int y = t % Y;
  it.b = t / Y;
  it.kvh = y / p.row_chunks;
  it.chunk_row = y - it.kvh * p.row_chunks;
  const SeqExtent ext = seq_extent(p, it.b, report && it.split == 0 && y == 0);
  it.L = ext.L;
  it.blk_begin = it.split * p.split_blocks;
  it.valid = !(it.split > 0 && it.blk_begin >= ext.nblk);
  const int blk_end = min(it.blk_begin + p.split_blocks, ext.nblk);
  it.nspan = max(blk_end - it.blk_begin, 0);
  it.n_chunks = (it.nspan + kChunkBlocks - 1) / kChunkBlocks;
  it.ns_b = max(1, min(ns, (ext.nblk + p.split_blocks - 1) / p.split_blocks));
  return it;
}

// Fused append (p.k_new set): fill the stage rows of the chunk's blocks in
// `mixed` (bit j: block j holds some of the Q new rows of the sequence, at
// positions L - Q .. L - 1) by hand: rows before L - Q from the cache, the
// new rows from k_new (K producer) or v_new (V producer), zeros past L.  The
// item of row chunk 0 also stores the new rows into the cache for the steps
// that follow (its split is the only one holding those blocks).  The layout
// is the copy's: row r of the chunk at r * 128 in the panel of its 64
// dimensions, 16-byte piece q at (q ^ (r % 8)) * 16 (128-byte swizzle).
// Warp-collective; `entry` is lane j's table entry for block j.
template <typename T>
__device__ __forceinline__ void fill_new_rows(const AttnParams &p, const Item &it, bool is_k,
                                              uint32_t mixed, int entry, int key0c,
                                              uint32_t stage, int panel_bytes) {
  constexpr int VPR = 128 * sizeof(T) / 16;  // 16-byte pieces per row (16)
  const int lane = threadIdx.x & 31;
  const int first_new = it.L - p.num_queries;
  const uint4 *cache = reinterpret_cast<const uint4 *>(is_k ? p.k_cache : p.v_cache);
  uint4 *cache_w = reinterpret_cast<uint4 *>(const_cast<void *>(is_k ? p.k_cache : p.v_cache));
  const uint4 *src = reinterpret_cast<const uint4 *>(is_k ? p.k_new : p.v_new);
  const bool write_cache = it.chunk_row == 0;
  for (uint32_t m = mixed; m != 0u; m &= m - 1u) {
    const int j = __ffs(m) - 1;
    const int64_t phys = __shfl_sync(kFull, entry, j);
    const int64_t tile = (phys * p.num_kv_heads + it.kvh) * kBlockSize * VPR;
#pragma unroll 2
    for (int idx = lane; idx < kBlockSize * VPR; idx += 32) {
      const int r = idx / VPR, vec = idx - r * VPR;
      const int pos = key0c + j * kBlockSize + r;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (pos >= first_new && pos < it.L) {
        const int64_t k =
            (static_cast<int64_t>(it.b) * p.num_queries + (pos - first_new)) * p.num_kv_heads +
            it.kvh;
        v = __ldg(src + k * VPR + vec);
        if (write_cache) cache_w[tile + r * VPR + vec] = v;
      } else if (pos < first_new) {
        v = __ldg(cache + tile + r * VPR + vec);
      }
      const int row = j * kBlockSize + r, part = vec >> 3, q = vec & 7;
      st_shared_v4(stage + part * panel_bytes + row * 128 + ((q ^ (row & 7)) << 4), v.x, v.y,
                   v.z, v.w);
    }
  }
  // generic writes, read next by the tensor core (async proxy)
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// Index of the partial of CTA column `col` (output row `row`) of item `it`
// (device partitions: slot it.idx, one partial per CTA column).
__device__ __forceinline__ int64_t tc_partial(const AttnParams &p, const Item &it, int64_t row,
                                              int col) {
  return p.split_target == 0 ? row * p.num_splits + it.split
                             : static_cast<int64_t>(it.idx) * p.rows_per_cta + col;
}

template <typename T, int D, int NC, int NS, int NV, int PB, int QB>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const AttnParams p, int num_items) {
  using G = TcGeom<D, NC, NS, NV, PB, QB>;
  constexpr int NCW = NC / 2;  // query columns of one softmax warp
  pdl_launch_dependents();  // the merge kernel may be scheduled now; it waits for this grid
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);

  // One barrier per buffer wherever a producer may run two phases ahead of
  // a waiter otherwise (P^T is double-buffered: the softmax can write chunk
  // g + 1's P^T before the issuer has waited for chunk g's).
  __shared__ uint64_t k_full[NS], k_empty[NS], v_full[NV], v_empty[NV], s_full[2], s_free[2],
      p_full[PB], pv_done[PB], qt_full[QB], qt_empty[QB], o_free[2], mma_idle;
  // Chunk facts from the K producer, a ring of NS + 2: the slot of chunk g
  // is rewritten (for chunk g + NS + 2) only after a K stage reuse that
  // waits on the softmax having released S^T of chunk g, read after them.
  __shared__ StageInfo stage_info[NS + 2];
  __shared__ uint32_t tmem_base_s;
  __shared__ __align__(16) float red[4][NC];
  __shared__ float lse_stg[NC];  // an item's log-sum-exps (device partitions)
  __shared__ volatile int s_abort;
  __shared__ DevSplits dev;  // the device partition's per-sequence layout

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G0 = blockIdx.x, GS = gridDim.x;

  // Softmax warp w: TMEM lane quadrant quad = w % 4 (keys / head dims
  // 32 quad .. 32 quad + 31) and column half half = w / 4 (columns
  // NCW half .. NCW half + NCW - 1).
  const int quad = warp & 3, half = (warp >> 2) & 1;
  const int kl = quad * 32 + lane;
  const int col0 = half * NCW;

  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&s_free[i]), kSoftmaxWarps);
      mbar_init(smem_u32(&o_free[i]), kSoftmaxWarps);
    }
    for (int i = 0; i < QB; ++i) {
      mbar_init(smem_u32(&qt_full[i]), 1);
      mbar_init(smem_u32(&qt_empty[i]), 1);
    }
    for (int i = 0; i < PB; ++i) {
      mbar_init(smem_u32(&p_full[i]), kSoftmaxWarps);
      mbar_init(smem_u32(&pv_done[i]), 1);
    }
    mbar_init(smem_u32(&mma_idle), 1);
    fence_mbar_init();
  }
  // Everything above overlaps the previous kernel in the stream; its writes
  // (the cache rows of an append, the previous call's merge reading the
  // workspace this kernel rewrites) are complete and visible after this.
  pdl_wait();
  if (p.stream_k && warp == 0) {  // warp-collective; read by every role below
    // The balanced partition: the flat list's offsets, this CTA's range and
    // the units it meets.  CTA 0 reports bad lengths (once) and publishes the
    // layout for the merge kernel.
    const int units = p.num_kv_heads * p.row_chunks;
    const SeqExtent ext = lane < p.batch ? seq_extent(p, lane, blockIdx.x == 0) : SeqExtent{0, 0};
    const int vlen = ext.nblk > 0 ? ext.nblk + p.sk_weight : 0;  // places of each unit of b
    int incl = vlen * units;  // < 2^31 (checked by the host)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const int s_b = incl - vlen * units;
    const int total = __shfl_sync(kFull, incl, 31);
    dev.first[lane] = s_b;
    dev.nb[lane] = ext.nblk;
    dev.L[lane] = ext.L;
    dev.ns[lane] = 0;
    const long long lo = sk_begin(total, gridDim.x, blockIdx.x);
    const long long hi = sk_begin(total, gridDim.x, blockIdx.x + 1);
    // the unit holding place x (-1: none, never for 0 <= x < total)
    auto unit_of = [&](long long x) -> int {
      const unsigned m = __ballot_sync(
          kFull, lane < p.batch && vlen > 0 && x >= s_b &&
                     x < s_b + static_cast<long long>(vlen) * units);
      const int b = m ? __ffs(m) - 1 : 0;
      const int sb = __shfl_sync(kFull, s_b, b), vl = __shfl_sync(kFull, vlen, b);
      return m ? b * units + static_cast<int>((x - sb) / vl) : -1;
    };
    int u0 = 0, n = 0;
    if (lo < hi) {
      const int a = unit_of(lo), z = unit_of(hi - 1);
      if (a >= 0 && z >= a) {
        u0 = a;
        n = z - a + 1;
      }
    }
    if (lane == 0) {
      dev.u0 = u0;
      dev.n_local = n;
      dev.lo = lo;
      dev.hi = hi;
    }
    if (blockIdx.x == 0) {
      if (lane < p.batch) {
        p.split_info[2 * lane] = s_b;
        p.split_info[2 * lane + 1] = ext.nblk;
      }
      if (lane == 0) p.split_info[2 * p.batch] = total;
    }
  } else if (p.split_target > 0 && warp == 0) {
    const SeqSplits sp = device_splits(p);
    dev.ns[lane] = sp.ns;
    dev.first[lane] = sp.first_item;
    dev.nb[lane] = sp.nb;
    // the merge kernel finds each sequence's items from this (every CTA
    // computes the same layout; the first one publishes it)
    if (blockIdx.x == 0 && lane < p.batch) {
      p.split_info[2 * lane] = sp.ns;
      p.split_info[2 * lane + 1] = sp.first_item;
    }
  }
  if (warp == kIssuerWarp) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
            smem_u32(&tmem_base_s)),
        "r"(G::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tmem_s[2] = {tmem, tmem + NC};
  // This CTA's items: i = i0, i0 + di, ... below i_end (every role walks
  // the same sequence).
  const int i0 = p.stream_k ? 0 : G0, di = p.stream_k ? 1 : GS;
  const int i_end = p.stream_k ? dev.n_local : num_items;
  const uint32_t tmem_o[2] = {tmem + 2 * NC, tmem + 4 * NC};

  auto abort_all = [&]() {
    s_abort = 1;
    record_error(p.err, PKV_DEVERR_TIMEOUT);
  };
  // Items with keys (items of an empty sequence are written directly by the
  // softmax warps and take no part in the pipeline).
  auto active = [](const Item &it) { return it.valid && it.n_chunks > 0; };

  if (warp == kKProducerWarp || warp == kVProducerWarp) {
    // ---- TMA producers: one warp for K (and each item's Q^T), one for V -------
    const bool is_k = warp == kKProducerWarp;
    uint64_t *full = is_k ? k_full : v_full;
    uint64_t *empty = is_k ? k_empty : v_empty;
    const CUtensorMap *map = is_k ? &kmap : &vmap;
    const uint32_t ring = sbase + (is_k ? 0 : G::kVOff);
    const int NR = is_k ? NS : NV;  // this ring's stages
    int g = 0, na = 0, issued = 0;
    bool ok = true;
    // The producers read one step ahead of their copies, so that no global
    // load sits between a stage becoming free and its copy: the table
    // entries of the next chunk (the next item's first, at an item's last
    // chunk) and, for K, the next item's query rows (in registers until its
    // Q^T buffer is free, stored after that item's first K copy is issued).
    constexpr int kPer = NC * (D / 8) / 32;  // 16-byte query pieces per lane
    uint4 qv[kPer];
    auto load_q = [&](const Item &x) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int e = lane + 32 * k, col = e / (D / 8), q = e - col * (D / 8);
        const int64_t row = cta_row_index(p, x.b, x.kvh, x.chunk_row, col);
        qv[k] = row >= 0 ? __ldg(reinterpret_cast<const uint4 *>(
                               reinterpret_cast<const T *>(p.q) + row * D + q * 8))
                         : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    auto entries = [&](const Item &x, int c) -> int {
      const int nb = min(kChunkBlocks, x.nspan - c * kChunkBlocks);
      return lane < nb ? ld_keep(p.block_table + static_cast<int64_t>(x.b) * p.max_blocks_per_seq +
                                 x.blk_begin + c * kChunkBlocks + lane)
                       : 0;
    };
    auto next_item = [&](int &ii, Item &out) -> bool {
      for (; ii < i_end; ii += di) {
        out = decode_item(p, ii, false, &dev);
        if (active(out)) {
          ii += di;
          return true;
        }
      }
      return false;
    };
    int i = i0;
    Item it{};
    bool have = next_item(i, it);
    int entry_nx = have ? entries(it, 0) : 0;
    if (have && is_k) load_q(it);
    while (have && ok) {
      const int qb = na % QB;
      Item nx{};
      bool have_nx = false, looked = false;
      for (int c = 0; c < it.n_chunks; ++c, ++g) {
        const int s = g % NR;
        const int entry = entry_nx;
        if (c + 1 < it.n_chunks) {
          entry_nx = entries(it, c + 1);
        } else {
          have_nx = next_item(i, nx);
          looked = true;
          entry_nx = have_nx ? entries(nx, 0) : 0;
        }
        bool w = !s_abort;
        if (w && g >= NR) w = mbar_wait_bounded(smem_u32(&empty[s]), ((g / NR) - 1) & 1);
        if (!__all_sync(kFull, w)) {
          ok = false;
          break;
        }
        const int nb = min(kChunkBlocks, it.nspan - c * kChunkBlocks);
        const bool bad = lane < nb && (entry < 0 || static_cast<int64_t>(entry) >= p.num_blocks);
        const uint32_t bad_mask = __ballot_sync(kFull, bad);
        const uint32_t bar = smem_u32(&full[s]);
        // Fused append: blocks holding new rows (positions L - Q .. L - 1)
        // are filled by this warp instead of a copy -- older rows from the
        // cache, new rows from k_new / v_new -- and the stage's barrier
        // completes only after that (its one arrival comes last).
        const int key0c = (it.blk_begin + c * kChunkBlocks) * kBlockSize;
        const uint32_t mixed =
            p.k_new == nullptr
                ? 0u
                : __ballot_sync(kFull, lane < nb && !bad &&
                                           key0c + (lane + 1) * kBlockSize > it.L - p.num_queries);
        if (lane == 0) {
          if (is_k) {
            if (bad_mask) record_error(p.err, PKV_DEVERR_BLOCK_ID);
            stage_info[g % (NS + 2)].nb = nb;
            stage_info[g % (NS + 2)].bad_mask = bad_mask;
          }
          const uint32_t bytes = (nb - __popc(mixed)) * 2 * 2048;
          if (mixed)
            mbar_expect_tx(bar, bytes);
          else
            mbar_arrive_expect_tx(bar, bytes);
        }
        __syncwarp();
        if (lane < nb && !((mixed >> lane) & 1u)) {
          const int phys = bad ? 0 : entry;
          const uint32_t st = ring + s * G::kTileBytes + lane * 2048;
#pragma unroll
          for (int part = 0; part < 2; ++part)
            tma_load_4d(st + part * G::kPanelBytes, map, bar, part * 64, 0, it.kvh, phys);
        }
        if (mixed) {
          fill_new_rows<T>(p, it, is_k, mixed, entry, key0c,
                           ring + s * G::kTileBytes, G::kPanelBytes);
          if (lane == 0) mbar_arrive(bar);
        }
        issued = g + 1;
        if (is_k && c == 0) {
          // Q^T of the item: query columns as rows of the K-major swizzled
          // operand (padding columns zero), once the Q^T buffer is free.
          const bool wq =
              na < QB || mbar_wait_bounded(smem_u32(&qt_empty[qb]), ((na / QB) - 1) & 1);
          if (!__all_sync(kFull, wq && !s_abort)) {
            ok = false;
            break;
          }
          const uint32_t qt = sbase + G::kQtOff + qb * 2 * G::kQtPanelBytes;
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            const int e = lane + 32 * k, col = e / (D / 8), q = e - col * (D / 8);
            st_shared_v4(qt + (q >> 3) * G::kQtPanelBytes + col * 128 +
                             (((q & 7) ^ (col & 7)) << 4),
                         qv[k].x, qv[k].y, qv[k].z, qv[k].w);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&qt_full[qb]));
        }
        if (is_k && looked && have_nx) load_q(nx);  // the next item's rows, in flight
      }
      if (!looked) have_nx = next_item(i, nx);  // (only after a break: ok is false)
      it = nx;
      have = have_nx;
      ++na;
    }
    if (!ok && lane == 0) abort_all();
    // Copies issued but perhaps never consumed (an aborted CTA): give them a
    // bounded chance to land before the CTA exits.
    if (lane == 0 && s_abort)
      for (int c = max(0, issued - NR); c < issued; ++c)
        mbar_wait_bounded(smem_u32(&full[c % NR]), (c / NR) & 1);
  } else if (warp == kIssuerWarp) {
    // ---- MMA issuer --------------------------------------------------------------
    if (lane == 0) {
      const uint32_t id_s = instr_desc<T>(128, NC, 0, 0);
      // P.V with the high part and the remainder of P^T side by side as one
      // operand of 2 NC columns: half the MMAs of two N = NC products
      const uint32_t id_pv = instr_desc<T>(128, 2 * NC, 1, 1);
      // Descriptors differ only in their start address (bits 0..13, address
      // >> 4): build each kind once and add the address per MMA.
      const uint64_t dk = smem_desc(0, 16, 1024, kSwizzle128);
      const uint64_t dv = smem_desc(0, G::kPanelBytes, 1024, kSwizzle128);
      const uint64_t dp = smem_desc(0, 128, kChunkKeys * 16, kSwizzleNone);
      // Cursors over the flat chunk sequence, across item boundaries: S^T
      // runs ahead of P.V as far as its two buffers allow.
      int i_s = i0, c_s = 0, na_s = 0, g_s = 0;   // next S^T: item, chunk, active index, flat
      int i_v = i0, c_v = 0, na_v = 0, g_v = 0;   // next P.V
      Item it_s{}, it_v{};
      auto next_active = [&](int &i, Item &it) {
        for (; i < i_end; i += di) {
          it = decode_item(p, i, false, &dev);
          if (active(it)) return true;
        }
        return false;
      };
      bool more_s = next_active(i_s, it_s), more_v = next_active(i_v, it_v);
      auto s_ready = [&](bool block) -> bool {
        const int s = g_s % NS, sb = g_s & 1, qb = na_s % QB;
        const uint32_t kf = smem_u32(&k_full[s]), sf = smem_u32(&s_free[sb]);
        const uint32_t qf = smem_u32(&qt_full[qb]);
        const uint32_t pk = (g_s / NS) & 1, ps = ((g_s >> 1) - 1) & 1, pq = (na_s / QB) & 1;
        if (block)
          return (c_s > 0 || mbar_wait_bounded(qf, pq)) && mbar_wait_bounded(kf, pk) &&
                 (g_s < 2 || mbar_wait_bounded(sf, ps));
        return (c_s > 0 || mbar_test(qf, pq)) && mbar_test(kf, pk) &&
               (g_s < 2 || mbar_test(sf, ps));
      };
      auto issue_s = [&]() {
        const int s = g_s % NS, sb = g_s & 1, qb = na_s % QB;
        fence_after();
        const uint64_t ka = dk | ((sbase + s * G::kTileBytes) >> 4);
        const uint64_t qa = dk | ((sbase + G::kQtOff + qb * 2 * G::kQtPanelBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * G::kPanelBytes + (ks & 3) * 32) >> 4;
          const uint32_t offq = ((ks >> 2) * G::kQtPanelBytes + (ks & 3) * 32) >> 4;
          mma(tmem_s[sb], ka + off, qa + offq, id_s, ks > 0);
        }
        commit(smem_u32(&s_full[sb]));
        commit(smem_u32(&k_empty[s]));
        ++g_s;
        if (++c_s == it_s.n_chunks) {  // the item's last S^T: its Q^T buffer is free
          commit(smem_u32(&qt_empty[qb]));
          c_s = 0;
          ++na_s;
          i_s += di;
          more_s = next_active(i_s, it_s);
        }
      };
      // P.V of the next chunk: its P^T written, its V landed and, for an
      // item's first chunk, the O^T buffer released by the item two back.
      auto pv_ready = [&]() -> bool {
        const int ob = na_v & 1;
        return mbar_test(smem_u32(&p_full[g_v % PB]), (g_v / PB) & 1) &&
               mbar_test(smem_u32(&v_full[g_v % NV]), (g_v / NV) & 1) &&
               (c_v > 0 || na_v < 2 || mbar_test(smem_u32(&o_free[ob]), ((na_v >> 1) - 1) & 1));
      };
      auto issue_pv = [&]() {
        const int ob = na_v & 1;
        fence_after();
        const uint64_t va = dv | ((sbase + G::kVOff + (g_v % NV) * G::kTileBytes) >> 4);
        const uint64_t pa = dp | ((sbase + G::kPOff + (g_v % PB) * 2 * G::kPBytes) >> 4);
#pragma unroll
        for (int j = 0; j < kChunkKeys / 16; ++j)
          mma(tmem_o[ob], va + ((j * 2048) >> 4), pa + ((j * 256) >> 4), id_pv, c_v > 0 || j > 0);
        commit(smem_u32(&v_empty[g_v % NV]));
        commit(smem_u32(&pv_done[g_v % PB]));
        ++g_v;
        if (++c_v == it_v.n_chunks) {
          c_v = 0;
          ++na_v;
          i_v += di;
          more_v = next_active(i_v, it_v);
        }
      };
      // The two MMA streams are issued as soon as each is ready, each in
      // chunk order: S^T of chunk g goes out once K has landed and the
      // softmax has read S^T of chunk g - 2 (the buffer it reuses), without
      // waiting for the P.V of chunk g - 1, whose V may land later; so the
      // softmax finds each chunk's scores ready when it finishes the last.
      // (With S^T issued only after the previous P.V, the softmax warps
      // waited ~40 % of every chunk for it.)  A stream that makes no progress
      // for the wait limit gives up.
      bool ok = true;
      unsigned long long t_last = global_ns();
      while (ok && (more_v || more_s)) {
        bool progress = false;
        if (more_s && s_ready(false)) {
          issue_s();
          progress = true;
        }
        if (more_v && g_v < g_s && pv_ready()) {
          issue_pv();
          progress = true;
        }
        if (progress) {
          t_last = global_ns();
        } else if (global_ns() - t_last > kWaitLimitNs || s_abort) {
          ok = false;
        } else {
          __nanosleep(20);  // leave the sub-partition's issue slots to the softmax warps
        }
      }
      if (!ok) abort_all();
      // every MMA this thread issued has completed before TMEM is released
      commit(smem_u32(&mma_idle));
      mbar_wait_bounded(smem_u32(&mma_idle), 0);
    }
  } else {
    // ---- softmax warps -------------------------------------------------------------
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const float colfac = p.scale_log2;
    // per item: the columns' references m (the same in every thread of the
    // column half) and this thread's partial column sums l
    float m[NCW], l[NCW];
    int g = 0, na = 0;
    bool ok = true;
    for (int i = i0; i < i_end && ok; i += di) {
      const Item it = decode_item(p, i, tid == 0 && !p.stream_k, &dev);
      if (!it.valid) continue;
      if (it.n_chunks == 0) {
        // an empty sequence: zero output rows (one split)
        for (int j = 0; j < NCW; ++j) {
          const int64_t row = cta_row_index(p, it.b, it.kvh, it.chunk_row, col0 + j);
          if (row < 0) continue;
          if (p.num_splits == 1 && p.split_target == 0) {
            reinterpret_cast<T *>(p.out)[row * D + kl] = from_float<T>(0.f);
          } else {
            const int64_t pi = tc_partial(p, it, row, col0 + j);
            p.part_o[pi * D + kl] = 0.f;
            if (quad == 0 && lane == 0) p.part_lse[pi] = -INFINITY;
          }
        }
        continue;
      }
      const int ob = na & 1;
      const int mask_from = it.L - p.num_queries;
#pragma unroll
      for (int j = 0; j < NCW; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.f;
      }
      for (int c = 0; c < it.n_chunks; ++c, ++g) {
        const int s = g % NV, sb = g & 1;  // s: the chunk's V stage
        if (!softmax_all(mbar_wait_bounded(smem_u32(&s_full[sb]), (g >> 1) & 1) && !s_abort)) {
          ok = false;
          break;
        }
        fence_after();
        // Which keys are real: the producer's block count and bad blocks (read
        // before S^T is released, see stage_info).
        const StageInfo info = stage_info[g % (NS + 2)];
        float sc[NCW];
        tmem_ld<NCW>(tmem_s[sb] + lane_base + col0, sc);
        tmem_wait_ld();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s_free[sb]));

        const int key0 = (it.blk_begin + c * kChunkBlocks) * kBlockSize;
        const int key = key0 + kl;
        const bool bad = kl >= info.nb * kBlockSize || ((info.bad_mask >> (kl >> 4)) & 1u);
        const bool need_mask = info.nb < kChunkBlocks || info.bad_mask != 0 ||
                               key0 + kChunkKeys > mask_from;
        bool above = false;
#pragma unroll
        for (int j = 0; j < NCW; ++j) sc[j] *= colfac;
        if (need_mask) {
          // (a uniform branch) column col is query row r = chunk_row *
          // rows_per_cta + col: query r / G, visible rows < L - Q + 1 + r / G;
          // walked without divisions
          const int r0 = it.chunk_row * p.rows_per_cta + col0;
          int jq = r0 / p.group, hh = r0 - jq * p.group;
#pragma unroll
          for (int j = 0; j < NCW; ++j) {
            const bool real = col0 + j < p.rows_per_cta && r0 + j < p.rows;
            const int lim = it.L - p.num_queries + 1 + (real ? jq : 0);
            const unsigned long long tm =
                (p.tree_mask != nullptr && real)
                    ? __ldg(p.tree_mask + static_cast<int64_t>(it.b) * p.mask_stride + jq)
                    : 0ull;
            if (!key_visible(p, key, it.L, bad, lim, tm)) sc[j] = -INFINITY;
            if (++hh == p.group) {
              hh = 0;
              ++jq;
            }
          }
        }
#pragma unroll
        for (int j = 0; j < NCW; ++j) above |= sc[j] > m[j] + kRescaleSlack;
        if (softmax_any(above)) {
          // Raise the references to the columns' running maxima: a max over
          // the 128 keys (shuffles, then the four quadrant warps of this
          // column half in shared memory).
          float corr[NCW];
#pragma unroll
          for (int j = 0; j < NCW; ++j) {
            float mx = sc[j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
            if (lane == 0) red[quad][col0 + j] = mx;
          }
          softmax_sync();
#pragma unroll
          for (int j = 0; j < NCW; ++j) {
            const int col = col0 + j;
            const float mx = fmaxf(fmaxf(red[0][col], red[1][col]), fmaxf(red[2][col], red[3][col]));
            const float m_new = fmaxf(m[j], mx);
            corr[j] = ex2(m[j] - (m_new == -INFINITY ? 0.f : m_new));
            m[j] = m_new;
            l[j] *= corr[j];
          }
          softmax_sync();  // red[] is reused by the next vote
          if (c > 0) {
            // O^T (head dims kl, this thread's columns) times corr, once chunk
            // g - 1's P.V, the last writer of O^T, has landed.
            if (!softmax_all(mbar_wait_bounded(smem_u32(&pv_done[(g - 1) % PB]),
                                               ((g - 1) / PB) & 1))) {
              ok = false;
              break;
            }
            fence_after();
#pragma unroll
            for (int part = 0; part < 2; ++part) {  // O^T of the high part and of the remainder
              float v[NCW];
              tmem_ld<NCW>(tmem_o[ob] + lane_base + part * NC + col0, v);
              tmem_wait_ld();
#pragma unroll
              for (int k2 = 0; k2 < NCW; ++k2) v[k2] *= corr[k2];
              tmem_st<NCW>(tmem_o[ob] + lane_base + part * NC + col0, v);
            }
            tmem_wait_st();
          }
        }
        // Weights and their 16-bit high part / remainder, column pairs packed.
        uint32_t hi[NCW / 2], lo[NCW / 2];
#pragma unroll
        for (int j = 0; j < NCW; j += 2) {
          const float m0 = m[j] == -INFINITY ? 0.f : m[j];
          const float m1 = m[j + 1] == -INFINITY ? 0.f : m[j + 1];
          const float p0 = ex2(sc[j] - m0), p1 = ex2(sc[j + 1] - m1);
          l[j] += p0;
          l[j + 1] += p1;
          const uint32_t h01 = Mma<T>::pack(p0, p1);
          float r0, r1;
          Mma<T>::unpack(h01, r0, r1);
          hi[j / 2] = h01;
          lo[j / 2] = Mma<T>::pack(p0 - r0, p1 - r1);
        }
        // P^T buffer g % PB was last read by chunk g - PB's P.V.
        if (g >= PB && !softmax_all(mbar_wait_bounded(smem_u32(&pv_done[g % PB]),
                                                       ((g / PB) - 1) & 1))) {
          ok = false;
          break;
        }
        // Keys no column sees get their V rows zeroed, once V has landed.
        // A parity wait is exact only once the barrier's previous phase has
        // completed: chunk g - NV's V.  With NV >= PB the P^T wait above
        // implies it (chunk g - PB's P.V has read its V and every earlier
        // one); with fewer V stages than P^T buffers the issuer may still be
        // waiting for chunk g - 1's V (S^T runs ahead of P.V), so wait for
        // that P.V first.
        if (NV < PB && need_mask && g >= 1 &&
            !softmax_all(mbar_wait_bounded(smem_u32(&pv_done[(g - 1) % PB]),
                                           ((g - 1) / PB) & 1))) {
          ok = false;
          break;
        }
        if (need_mask && !softmax_all(mbar_wait_bounded(smem_u32(&v_full[s]), (g / NV) & 1))) {
          ok = false;
          break;
        }
        if (half == 0 && need_mask && (bad || key >= it.L)) {
          const uint32_t vrow = sbase + G::kVOff + s * G::kTileBytes + kl * 128;
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_shared_v4(vrow + part * G::kPanelBytes + q * 16, 0u, 0u, 0u, 0u);
        }
        // P^T rows (key kl): core matrices of 8 keys x 8 columns.
        const uint32_t prow =
            sbase + G::kPOff + (g % PB) * 2 * G::kPBytes + (kl >> 3) * 128 + (kl & 7) * 16;
#pragma unroll
        for (int gg = 0; gg < NCW / 8; ++gg) {
          const int g8 = (col0 >> 3) + gg;
          st_shared_v4(prow + g8 * (kChunkKeys * 16), hi[4 * gg], hi[4 * gg + 1],
                       hi[4 * gg + 2], hi[4 * gg + 3]);
          st_shared_v4(prow + G::kPBytes + g8 * (kChunkKeys * 16), lo[4 * gg], lo[4 * gg + 1],
                       lo[4 * gg + 2], lo[4 * gg + 3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&p_full[g % PB]));
      }
      if (!ok) break;
      // The item's result: O^T once its last P.V has landed, column sums
      // over the four quadrant warps, then out (or this split's partial).
      const int gl = g - 1;
      if (!softmax_all(mbar_wait_bounded(smem_u32(&pv_done[gl % PB]), (gl / PB) & 1))) {
        ok = false;
        break;
      }
      fence_after();
      float o_hi[NCW], o_lo[NCW];
      tmem_ld<NCW>(tmem_o[ob] + lane_base + col0, o_hi);
      tmem_ld<NCW>(tmem_o[ob] + lane_base + NC + col0, o_lo);
      tmem_wait_ld();
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&o_free[ob]));
#pragma unroll
      for (int j = 0; j < NCW; ++j) {
        float v = l[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
        if (lane == 0) red[quad][col0 + j] = v;
      }
      if (p.split_target > 0 && tid == 0) bulk_wait_read();  // the staging buffer is free
      softmax_sync();
      // Every shared-memory read first (vectorised), then only stores: the
      // tensor core and the copies keep shared memory busy, and a read
      // queued behind each store would cost a round trip per column.
      float lsum[NCW];
#pragma unroll
      for (int j = 0; j < NCW; j += 4) {
        float4 a = *reinterpret_cast<const float4 *>(&red[0][col0 + j]);
#pragma unroll
        for (int q = 1; q < 4; ++q) {
          const float4 v = *reinterpret_cast<const float4 *>(&red[q][col0 + j]);
          a.x += v.x;
          a.y += v.y;
          a.z += v.z;
          a.w += v.w;
        }
        lsum[j] = a.x;
        lsum[j + 1] = a.y;
        lsum[j + 2] = a.z;
        lsum[j + 3] = a.w;
      }
      if (p.split_target > 0) {
        // Device partitions: the item's columns are consecutive partials
        // ([slot][column]).  They are staged in shared memory and one bulk
        // copy takes them out while the warps go on with the next item; the
        // warps' own global stores would queue behind the copies that keep
        // HBM busy.  (Padding columns are staged too but not copied.)
        float lse_mine = -INFINITY;  // column col0 + lane's log-sum-exp (lanes < NCW)
#pragma unroll
        for (int j = 0; j < NCW; ++j) {
          const float inv = lsum[j] > 0.f ? __fdividef(1.f, lsum[j]) : 0.f;
          st_shared_f32(sbase + G::kStgOff + ((col0 + j) * D + kl) * 4, (o_hi[j] + o_lo[j]) * inv);
          if (lane == j) lse_mine = lsum[j] > 0.f ? m[j] + __log2f(lsum[j]) : -INFINITY;
        }
        if (quad == 0 && lane < NCW) lse_stg[col0 + lane] = lse_mine;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        softmax_sync();  // (red[] and the staging are reused by the next item)
        const int n = min(p.rows_per_cta, p.rows - it.chunk_row * p.rows_per_cta);
        const int64_t slot0 = static_cast<int64_t>(it.idx) * p.rows_per_cta;
        if (tid == 0) {  // read back by bulk_wait_read at the next epilogue
          bulk_s2g(p.part_o + slot0 * D, sbase + G::kStgOff, static_cast<uint32_t>(n) * D * 4);
          bulk_commit();
        }
        if (warp == 0)  // (up to 64 columns)
          for (int c = lane; c < n; c += 32) __stcg(p.part_lse + slot0 + c, lse_stg[c]);
      } else {
        // Output rows of the columns, walked without divisions: column col is
        // query row r = chunk_row * rows_per_cta + col, query r / G, head
        // kvh * G + r % G.
        const int r0 = it.chunk_row * p.rows_per_cta + col0;
        int jq = r0 / p.group, hh = r0 - jq * p.group;
        float lse_mine = -INFINITY;  // column col0 + lane's log-sum-exp (lanes < NCW)
        int64_t row_mine = -1;
#pragma unroll
        for (int j = 0; j < NCW; ++j) {
          const int col = col0 + j;
          const bool real = col < p.rows_per_cta && r0 + j < p.rows;
          const int64_t row = (static_cast<int64_t>(it.b) * p.num_queries + jq) * p.num_heads +
                              it.kvh * p.group + hh;
          if (++hh == p.group) {
            hh = 0;
            ++jq;
          }
          if (!real) continue;
          const float inv = lsum[j] > 0.f ? __fdividef(1.f, lsum[j]) : 0.f;
          const float o = o_hi[j] + o_lo[j];
          if (p.num_splits == 1) {
            reinterpret_cast<T *>(p.out)[row * D + kl] = from_float<T>(o * inv * p.out_scale);
          } else {
            const int64_t pi = tc_partial(p, it, row, col);
            __stcg(p.part_o + pi * D + kl, o * inv);
            if (lane == j) {
              lse_mine = lsum[j] > 0.f ? m[j] + __log2f(lsum[j]) : -INFINITY;
              row_mine = pi;
            }
          }
        }
        if (quad == 0 && row_mine >= 0) __stcg(p.part_lse + row_mine, lse_mine);
        softmax_sync();  // red[] is reused by the next item
      }
      ++na;
    }
    if (!ok && tid == 0) abort_all();
    if (tid == 0) bulk_wait_all();  // the partials are written before the CTA exits
  }

  fence_before();
  __syncthreads();
  if (warp == kIssuerWarp) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(G::kTmemCols));
  }
}

}  // namespace tc
}  // namespace pkv
namespace pkv {
namespace tc {

// Rings of 32 KB stages (bf16/fp16, head_dim 128).  `stages` names the V
// ring's depth; the K ring takes min(stages, 2) (K is released as soon as
// S^T is computed, so two stages keep its copies ahead).  Up to 32 columns,
// two P^T and two Q^T buffers fit beside them in shared memory; the 64-column
// tile (up to 64 query rows, a 10-node tree over four heads) takes one of
// each (and at most two V stages).
template <int NC, int NV> struct TcConfig {
  static constexpr int NS = NV < 2 ? NV : 2;
  static constexpr int PB = NC > 32 ? 1 : 2;
  static constexpr int QB = NC > 32 ? 1 : 2;
};
constexpr int kDefaultStages = 2;

template <typename T, int NC, int NV>
KernelInfo info_t() {
  using C = TcConfig<NC, NV>;
  KernelInfo k;
  k.func = reinterpret_cast<const void *>(&attn_tc_kernel<T, 128, NC, C::NS, NV, C::PB, C::QB>);
  k.threads = kThreads;
  k.warps = kThreads / 32;
  k.stages = NV;
  k.smem = static_cast<size_t>(TcGeom<128, NC, C::NS, NV, C::PB, C::QB>::kBytes) + 1024;
  k.warp_tiles = NC / 8;
  return k;
}

template <typename T, int NC, int NV>
cudaError_t launch_t(const CUtensorMap &km, const CUtensorMap &vm, const AttnParams &p, dim3 grid,
                     cudaStream_t stream) {
  using C = TcConfig<NC, NV>;
  const KernelInfo k = info_t<T, NC, NV>();
  // persistent: grid.x CTAs walk the grid.y x grid.z x splits items (or the
  // device partition's split_target items)
  const int items = p.split_target > 0 ? p.split_target
                                       : p.num_splits * p.num_kv_heads * p.row_chunks * p.batch;
  // a programmatic dependent of the kernel before it (it waits for that
  // kernel before touching global memory)
  return launch_kernel(true, attn_tc_kernel<T, 128, NC, C::NS, NV, C::PB, C::QB>, dim3(grid.x),
                       k.threads, k.smem, stream, km, vm, p, items);
}

using Launch = cudaError_t (*)(const CUtensorMap &, const CUtensorMap &, const AttnParams &, dim3,
                               cudaStream_t);

template <typename T, int NC>
bool pick_ns(int stages, KernelInfo *info, Launch *launch) {
  switch (stages == 0 ? kDefaultStages : stages) {
    case 1: *info = info_t<T, NC, 1>(); if (launch) *launch = &launch_t<T, NC, 1>; return true;
    case 2: *info = info_t<T, NC, 2>(); if (launch) *launch = &launch_t<T, NC, 2>; return true;
    case 3:
      if constexpr (NC > 32) return false;  // shared memory
      else {
        *info = info_t<T, NC, 3>();
        if (launch) *launch = &launch_t<T, NC, 3>;
        return true;
      }
    default: return false;
  }
}

template <typename T>
bool pick_t(int rows, int stages, KernelInfo *info, Launch *launch) {
  if (rows <= 16) return pick_ns<T, 16>(stages, info, launch);
  if (rows <= 32) return pick_ns<T, 32>(stages, info, launch);
  if (rows <= 64) return pick_ns<T, 64>(stages, info, launch);
  return false;
}

bool pick(pkv_dtype dtype, int head_dim, int rows, int stages, KernelInfo *info, Launch *launch) {
  if (head_dim != 128 || rows < 1) return false;
  if (dtype == PKV_BF16) return pick_t<__nv_bfloat16>(rows, stages, info, launch);
  if (dtype == PKV_F16) return pick_t<__half>(rows, stages, info, launch);
  return false;
}

}  // namespace tc

bool tc_kernel_info(pkv_dtype dtype, int head_dim, int rows_per_cta, int stages,
                    KernelInfo *info) {
  return tc::pick(dtype, head_dim, rows_per_cta, stages, info, nullptr);
}

cudaError_t tc_launch(pkv_dtype dtype, int head_dim, int rows_per_cta, int stages,
                      const CUtensorMap &kmap, const CUtensorMap &vmap, const AttnParams &p,
                      dim3 grid, cudaStream_t stream) {
  KernelInfo info;
  tc::Launch launch = nullptr;
  if (!tc::pick(dtype, head_dim, rows_per_cta, stages, &info, &launch))
    return cudaErrorInvalidValue;
  return launch(kmap, vmap, p, grid, stream);
}

}  // namespace pkv
