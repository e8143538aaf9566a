// pkv_device.cuh -- device-side building blocks shared by the attention
// kernels: kernel parameters, inline-PTX wrappers (mbarrier, bulk and tensor
// copies, ldmatrix / movmatrix / mma), and the epilogue that merges the
// per-warp online-softmax states of one CTA and writes the output or the
// split-K partials.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

constexpr int kBlockSize = 16;   // tokens per KV block (rows of one tile)
constexpr unsigned kFull = 0xffffffffu;
// A shared-memory copy that has not landed after this long is reported as
// PKV_DEVERR_TIMEOUT instead of being waited for forever.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Parameters of one attention launch (passed by value).
struct AttnParams {
  void *out;                    // [B, Q, Hq, D] elt
  const void *q;                // [B, Q, Hq, D] elt
  const void *k_cache;          // [NB, Hkv, 16, D] elt
  const void *v_cache;
  const int32_t *block_table;   // [B, max_blocks_per_seq]
  const int32_t *context_lens;  // [B]
  const void *k_new;            // [B, Q, Hkv, D] elt: new rows appended in the same launch
  const void *v_new;            //   (nullptr: the cache already holds them)
  float *part_o;                // [B*Q*Hq, num_splits, D]   (split-K only)
  float *part_lse;              // [B*Q*Hq, num_splits]      (log2 units)
  unsigned int *counters;       // [B, Hkv, row_chunks] split arrivals, zeroed by a kernel
                                //   launched just before this one (see split_arrive);
                                //   nullptr: a separate merge kernel runs after
  const unsigned long long *tree_mask;  // [B, Q] with stride mask_stride (0: shared),
                                        //   or nullptr: causal among the Q rows
  int64_t mask_stride;
  int32_t *err;                 // optional device error word
  int64_t num_blocks;
  int batch, num_queries, num_heads, num_kv_heads, group;
  int rows;                     // group * num_queries query rows per KV head
  int rows_per_cta, row_chunks;
  int max_blocks_per_seq, max_context_len;
  int split_blocks, num_splits;
  int split_target;             // > 0: split-K partition made on the device into at most
                                //   this many work items (see cta_work); 0: host partition
  int *split_info;              // device partition: [batch][2] = (ns_b, first item of b);
                                //   balanced partition: (first flat block, n_b), then the
                                //   total; written by the attention kernel for the merge
  int stream_k;                 // with split_target = G > 0: the balanced partition
                                //   (sk_begin below), G CTAs; else split_target items
  int sk_weight;                //   its per-unit weight W, in blocks (sk_begin below)
  int tile_box;                 // the cache maps copy a whole (block, KV head) tile per box
                                //   (5-D maps); 0: one 128-byte column panel per box (4-D)
  float scale_log2;             // softmax scale * log2(e) (* key scale of an FP8 cache)
  float out_scale;              // multiplies every output (value scale of an FP8 cache; else 1)
};

// Chunked prefill: the query rows of sequence b are q[query_start[b] ..
// query_start[b + 1]) ([total_q, Hq, D]); its cache holds context_lens[b]
// rows, the chunk's own rows last.
struct PrefillParams {
  void *out;                     // [total_q, Hq, D] elt
  const int32_t *block_table;    // [B, max_blocks_per_seq]
  const int32_t *context_lens;   // [B]
  const int32_t *query_start;    // [B + 1]
  int32_t *err;                  // optional device error word
  int64_t num_blocks;
  int max_blocks_per_seq, batch, total_q, max_query_len;
  int num_heads, num_kv_heads, group, pairs;
  float scale_log2;              // softmax scale * log2(e)
};

// FP8 E4M3 cache element (one byte; value = code value * tensor scale).
struct E4M3 {};

template <typename T> struct Elt;
template <> struct Elt<E4M3> { static constexpr int bytes = 1; };
template <> struct Elt<float> { static constexpr int bytes = 4; };
template <> struct Elt<__nv_bfloat16> { static constexpr int bytes = 2; };
template <> struct Elt<__half> { static constexpr int bytes = 2; };

__device__ __forceinline__ void record_error(int32_t *err, int code) {
  if (err) atomicCAS(reinterpret_cast<int *>(err), 0, code);
}

// ---- conversions --------------------------------------------------------
__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T> __device__ __forceinline__ void unpack2(uint32_t w, float &a, float &b);
template <> __device__ __forceinline__ void unpack2<__nv_bfloat16>(uint32_t w, float &a, float &b) {
  a = lo_bf16(w);
  b = hi_bf16(w);
}
template <> __device__ __forceinline__ void unpack2<__half>(uint32_t w, float &a, float &b) {
  __half2 h = *reinterpret_cast<__half2 *>(&w);
  float2 f = __half22float2(h);
  a = f.x;
  b = f.y;
}

template <typename T> __device__ __forceinline__ T from_float(float x);
template <> __device__ __forceinline__ float from_float<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <> __device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }

// 2^x (PTX ex2.approx; ex2(-inf) = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- shared-memory addressing and mbarriers -----------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch.  A kernel that calls pdl_launch_dependents
// lets the next kernel of its stream, when that one is launched with
// programmatic stream serialisation, be scheduled before it finishes; the
// dependent kernel calls pdl_wait before it reads anything this kernel
// writes (the wait returns once this grid has completed and its memory
// operations are visible).  Both are no-ops without such a pairing.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kernel` on `stream`, as a programmatic dependent of the kernel
// enqueued just before it when `dependent` is true (then it may start while
// that kernel still runs, and must pdl_wait before it touches what that
// kernel writes).
template <typename... Params, typename... Args>
cudaError_t launch_kernel(bool dependent, void (*kernel)(Params...), dim3 grid, int threads,
                          size_t smem, cudaStream_t stream, Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = dependent ? attr : nullptr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// A load of read-only data that stays in the register it is loaded into.
// Block-table entries are loaded a chunk ahead of their use; written as a
// plain __ldg the compiler may drop the register and load again at the use
// (the load is invariant), which puts a global-memory round trip on every
// block of the loop.  An asm statement is neither duplicated nor moved.
__device__ __forceinline__ int ld_keep(const int32_t *ptr) {
  int v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(ptr));
  return v;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Expect `bytes` more of copies in the current phase, without an arrival.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of the barrier, giving up after limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded_ns(uint32_t bar, uint32_t parity,
                                                     unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  return mbar_wait_bounded_ns(bar, parity, kWaitLimitNs);
}

// ---- bulk copies (TMA engine) -------------------------------------------
// Contiguous global -> shared copy; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Tiled 3-D tensor copy (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// Tiled 4-D tensor copy (coordinates innermost first).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// Tiled 5-D tensor copy (coordinates innermost first).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(bar)
      : "memory");
}

// ---- warp-level matrix ops ----------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

template <typename T> struct Mma;
template <> struct Mma<__nv_bfloat16> {
  static __device__ __forceinline__ void run(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
  static __device__ __forceinline__ void unpack(uint32_t w, float &lo, float &hi) {
    unpack2<__nv_bfloat16>(w, lo, hi);
  }
};
template <> struct Mma<__half> {
  static __device__ __forceinline__ void run(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
  static __device__ __forceinline__ void unpack(uint32_t w, float &lo, float &hi) {
    unpack2<__half>(w, lo, hi);
  }
};

// ---- per-CTA bookkeeping ------------------------------------------------
// Where query row `col` of this CTA lives: flat output row index
// ((b * Q + j) * Hq + h), or -1 when the column is padding.
__device__ __forceinline__ int64_t cta_row_index(const AttnParams &p, int b, int kvh, int chunk,
                                                 int col) {
  if (col >= p.rows_per_cta) return -1;
  const int r = chunk * p.rows_per_cta + col;
  if (r >= p.rows) return -1;
  const int j = r / p.group;
  const int h = kvh * p.group + (r - j * p.group);
  return (static_cast<int64_t>(b) * p.num_queries + j) * p.num_heads + h;
}

// Number of key rows query row `col` may see: L - Q + 1 + j (<= 0: none).
__device__ __forceinline__ int cta_row_limit(const AttnParams &p, int L, int chunk, int col) {
  const int r = chunk * p.rows_per_cta + col;
  const int j = (col < p.rows_per_cta && r < p.rows) ? r / p.group : 0;
  return L - p.num_queries + 1 + j;
}

// Tree mask of query row `col` of this CTA (tree verification): bit k set
// when the row may see row L - Q + k.  0 for padding columns.
__device__ __forceinline__ unsigned long long cta_row_tree_mask(const AttnParams &p, int b,
                                                                int chunk, int col) {
  const int r = chunk * p.rows_per_cta + col;
  if (p.tree_mask == nullptr || col >= p.rows_per_cta || r >= p.rows) return 0ull;
  return __ldg(p.tree_mask + static_cast<int64_t>(b) * p.mask_stride + r / p.group);
}

// Whether key row `key` is visible to a query row: rows past the context and
// rows of a bad block never are; with a tree mask, cached rows (before the Q
// new ones) always are and new row k when bit k is set; otherwise the causal
// limit `lim` (rows < L - Q + 1 + j) applies.
__device__ __forceinline__ bool key_visible(const AttnParams &p, int key, int L, bool bad, int lim,
                                            unsigned long long tm) {
  if (bad || key >= L) return false;
  if (p.tree_mask == nullptr) return key < lim;
  const int t = key - (L - p.num_queries);
  return t < 0 || ((tm >> t) & 1ull);
}

// Effective context length of sequence b and its block count, with the
// precondition checks that never fault (recorded in the error word).
struct SeqExtent {
  int L, nblk;
};
__device__ __forceinline__ SeqExtent seq_extent(const AttnParams &p, int b, bool report) {
  int L = p.context_lens[b];
  if (L < 0) L = 0;
  if (L > p.max_context_len) {
    if (report) record_error(p.err, PKV_DEVERR_CONTEXT_LEN);
    L = p.max_context_len;
  }
  int nblk = (L + kBlockSize - 1) / kBlockSize;
  if (nblk > p.max_blocks_per_seq) {
    if (report) record_error(p.err, PKV_DEVERR_CONTEXT_LEN);
    nblk = p.max_blocks_per_seq;
    L = nblk * kBlockSize;
  }
  return {L, nblk};
}

// ---- split-K partition ------------------------------------------------------
// Host partition (split_target == 0): the grid is (splits, KV heads x row
// chunks, batch) and split s of a sequence covers blocks s * split_blocks ..
// s * split_blocks + split_blocks - 1 (planned from max_context_len).
//
// Device partition (split_target = T > 0, batch <= 32): the split length is
// chosen here from the batch's real block counts n_b, so that the work items
// -- (sequence, unit, split), a unit being one KV head x row chunk -- number
// at most T (the host makes T whole waves of resident CTAs):  S is the
// smallest length >= kMinDeviceSplit with  units * sum_b ns_b <= T,  where
// ns_b = max(1, ceil(n_b / S)).  Sequence b's blocks are cut into ns_b
// nearly equal runs, and the grid is flat: CTA t takes item t, items being
// numbered sequence by sequence, unit by unit, split by split.  Partials are
// stored per item: [item][rows_per_cta] vectors of head_dim floats and one
// log-sum-exp each.  Every warp that needs the partition computes it alike.
constexpr int kMinDeviceSplit = 16;

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Warp-collective: lane b < batch holds n_b (others 0); returns S.
__device__ __forceinline__ int device_split_len(const AttnParams &p, int nb, int units) {
  const int lane = threadIdx.x & 31;
  const int cap = max(p.split_target / units, 1);  // sum over sequences of ns_b
  const int total = warp_sum_i(nb);
  int lo = max(kMinDeviceSplit, (total + cap - 1) / cap);
  int hi = max(lo, warp_max_i(nb));  // one split per sequence: batch <= cap (host)
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int cnt = warp_sum_i(lane < p.batch ? max(1, (nb + mid - 1) / mid) : 0);
    if (cnt <= cap) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// Per-sequence split layout of the device partition (warp-collective):
// lane b < batch gets ns_b and the index of its first item.
struct SeqSplits {
  int nb, ns, first_item;
};
__device__ __forceinline__ SeqSplits device_splits(const AttnParams &p) {
  const int lane = threadIdx.x & 31;
  const int units = p.num_kv_heads * p.row_chunks;
  SeqSplits r;
  r.nb = lane < p.batch ? seq_extent(p, lane, false).nblk : 0;
  const int S = device_split_len(p, r.nb, units);
  r.ns = lane < p.batch ? max(1, (r.nb + S - 1) / S) : 0;
  int incl = r.ns * units;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  r.first_item = incl - r.ns * units;
  return r;
}

// Balanced partition (split_target = G > 0 with stream_k set; batch <= 32;
// the tcgen05 kernel).  The units of the batch -- (sequence, KV head, row
// chunk), every unit of sequence b holding n_b blocks -- are laid end to end
// in one list, sequence after sequence; a unit with blocks takes W + n_b
// places in it (W = sk_weight: the fixed cost of starting and finishing a
// piece of work, counted in blocks, then its n_b blocks), a unit without
// none.  CTA c of the G takes the list's places sk_begin(c) ..
// sk_begin(c + 1) - 1 of T: each CTA the same amount of work to within one
// block, however ragged the lengths, so that no CTA waits at the end for a
// long item of another.  The blocks of a CTA's range inside one unit U (U =
// its index in the list) are a split of that unit; its partials go to slot
// c + U.  Slots are distinct (a later unit in the list never meets an earlier
// CTA) and those of one unit consecutive, so G + units slots hold them all
// and the merge finds a unit's splits from its first and last block alone
// (skipping the CTAs whose range is empty, which exist when T < G: a CTA
// strictly between those two has all its places among the unit's blocks).
__device__ __forceinline__ int64_t sk_begin(int64_t T, int G, int c) { return T * c / G; }
// The CTA whose range holds flat block x (0 <= x < T): the largest c with
// sk_begin(c) <= x.
__device__ __forceinline__ int sk_cta_of(int64_t T, int G, int64_t x) {
  return static_cast<int>(((x + 1) * G - 1) / T);
}

// The work of this CTA.
struct CtaWork {
  int b, kvh, chunk, split, ns_b, blk_begin, blk_end;
  int64_t item;  // device partition: the item index (blockIdx.x); else -1
  SeqExtent ext;
  bool active;   // false: nothing to do (a split past its sequence's end)
};
__device__ __forceinline__ CtaWork cta_work(const AttnParams &p) {
  CtaWork w;
  if (p.split_target == 0) {
    w.split = blockIdx.x;
    w.kvh = blockIdx.y / p.row_chunks;
    w.chunk = blockIdx.y - w.kvh * p.row_chunks;
    w.b = blockIdx.z;
    w.ext = seq_extent(p, w.b, w.split == 0 && w.chunk == 0 && w.kvh == 0 && threadIdx.x == 0);
    w.blk_begin = w.split * p.split_blocks;
    w.active = !(w.split > 0 && w.blk_begin >= w.ext.nblk);
    w.blk_end = min(w.blk_begin + p.split_blocks, w.ext.nblk);
    w.ns_b = max(1, min(p.num_splits, (w.ext.nblk + p.split_blocks - 1) / p.split_blocks));
    w.item = -1;
    return w;
  }
  const SeqSplits sp = device_splits(p);
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const unsigned hit =
      __ballot_sync(kFull, lane < p.batch && sp.first_item + sp.ns * p.num_kv_heads *
                                                                  p.row_chunks > t);
  w.active = hit != 0u;
  const int b = w.active ? __ffs(hit) - 1 : 0;
  const int ns = __shfl_sync(kFull, sp.ns, b);
  const int first = __shfl_sync(kFull, sp.first_item, b);
  const int nb = __shfl_sync(kFull, sp.nb, b);
  w.b = b;
  w.item = t;
  if (!w.active) return w;
  const int r = t - first;
  const int u = r / ns;
  w.split = r - u * ns;
  w.kvh = u / p.row_chunks;
  w.chunk = u - w.kvh * p.row_chunks;
  w.ns_b = ns;
  w.ext = seq_extent(p, b, w.split == 0 && u == 0 && threadIdx.x == 0);
  if (r == 0 && threadIdx.x == 0) {  // the sequence's first item publishes its layout
    p.split_info[2 * b] = ns;
    p.split_info[2 * b + 1] = first;
  }
  w.blk_begin = static_cast<int>(static_cast<int64_t>(w.split) * nb / ns);
  w.blk_end = static_cast<int>(static_cast<int64_t>(w.split + 1) * nb / ns);
  return w;
}

// Index of the partial (output vector and log-sum-exp) of CTA column `col`
// of work item w, for flat output row `row`.
__device__ __forceinline__ int64_t partial_index(const AttnParams &p, const CtaWork &w,
                                                 int64_t row, int col) {
  return p.split_target == 0 ? row * p.num_splits + w.split
                             : w.item * p.rows_per_cta + col;
}

// Fused append.  The Q new rows of sequence b sit at logical positions
// L - Q .. L - 1.  A warp that has just received the tile of block `blk`
// (first row key0) overwrites the tile rows of any new position in it with
// k_new / v_new (so the attention sees them whatever the cache held there),
// and, when `write_cache` is set, also stores them into the cache at the
// physical block `phys` for the steps that follow.  `row_off(r, vec)` gives
// the byte offset of 16-byte vector `vec` of tile row r in shared memory.
template <int D, int ELT, typename RowOff>
__device__ __forceinline__ void patch_new_rows(const AttnParams &p, uint32_t ktile,
                                               uint32_t vtile, int b, int kvh, int key0, int L,
                                               int64_t phys, bool write_cache, RowOff row_off) {
  constexpr int VPR = D * ELT / 16;  // 16-byte vectors per row
  const int first = max(L - p.num_queries, key0);
  const int last = min(L, key0 + kBlockSize);  // exclusive
  const int n = (last - first) * VPR;
  const int lane = threadIdx.x & 31;
  for (int idx = lane; idx < n; idx += 32) {
    const int r = first + idx / VPR;  // logical row
    const int vec = idx - (idx / VPR) * VPR;
    const int j = r - (L - p.num_queries);
    const int64_t src = ((static_cast<int64_t>(b) * p.num_queries + j) * p.num_kv_heads + kvh) *
                            VPR + vec;
    const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(p.k_new) + src);
    const uint4 vv = __ldg(reinterpret_cast<const uint4 *>(p.v_new) + src);
    const uint32_t off = row_off(r - key0, vec);
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(ktile + off), "r"(kv.x), "r"(kv.y),
                 "r"(kv.z), "r"(kv.w)
                 : "memory");
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(vtile + off), "r"(vv.x), "r"(vv.y),
                 "r"(vv.z), "r"(vv.w)
                 : "memory");
    if (write_cache) {
      const int64_t dst = ((phys * p.num_kv_heads + kvh) * kBlockSize + (r - key0)) * VPR + vec;
      reinterpret_cast<uint4 *>(const_cast<void *>(p.k_cache))[dst] = kv;
      reinterpret_cast<uint4 *>(const_cast<void *>(p.v_cache))[dst] = vv;
    }
  }
  // The patched stage may be refilled by a bulk copy later: order these
  // generic writes before any later async-proxy write to the same memory.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// Largest split count whose merge the last-arriving CTA does itself.
constexpr int kMaxFusedSplits = 32;

// Split-K arrival: count this CTA in its (sequence, KV head, row chunk)
// counter; true for the CTA that completes the count.  The counters start at
// zero whatever the workspace held before the call: the host enqueues a
// zeroing kernel (zero_words_kernel) right before this launch, which runs as
// its programmatic dependent, and the wait below returns only once that
// kernel has completed and its writes are visible.  Everything before this
// point overlaps it.
__device__ __forceinline__ bool split_arrive(const AttnParams &p, int b, int kvh, int chunk,
                                             int ns_b) {
  unsigned int *ctr =
      p.counters + (static_cast<int64_t>(b) * p.num_kv_heads + kvh) * p.row_chunks + chunk;
  pdl_wait();
  return atomicAdd(ctr, 1u) + 1u == static_cast<unsigned int>(ns_b);
}

// CTA epilogue.  Every warp w has left, for each of the NC query columns of
// this CTA, its running max m (log2 units), its sum l and its unnormalised
// output o[0..D) in shared memory:
//   red_m[w * NC + col], red_l[w * NC + col], red_o[(w * NC + col) * DP + d].
// The states are merged exactly as the online softmax merges two chunks
// (rescale each by 2^(m_w - M)).  Then the CTA writes
//   - the normalised output, when the launch or this sequence has one split;
//   - otherwise this split's normalised output and its log-sum-exp, and, with
//     counters, the CTA that completes the sequence's splits merges them
//     (the Flash-Decoding reduction: weights 2^(lse_s - max lse)).
template <typename T, int D, int NC, int W, int NTHR>
__device__ __forceinline__ void cta_epilogue(const AttnParams &p, float *red_m, float *red_l,
                                             float *red_o, float *wscale, const CtaWork &wk) {
  const int b = wk.b, kvh = wk.kvh, chunk = wk.chunk, ns_b = wk.ns_b;
  constexpr int DP = D + 4;
  constexpr int QV = D / 4;
  const int tid = threadIdx.x;
  // 1) per column: global max, per-warp scale factors and 1 / sum.
  if (tid < NC) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, red_m[w * NC + tid]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float s = ex2(red_m[w * NC + tid] - Mu);
      wscale[w * NC + tid] = s;
      lsum += red_l[w * NC + tid] * s;
    }
    wscale[W * NC + tid] = lsum > 0.f ? 1.f / lsum : 0.f;
    wscale[(W + 1) * NC + tid] = lsum > 0.f ? M + __log2f(lsum) : -INFINITY;
  }
  __syncthreads();
  // (the device partition always leaves partials for the merge kernel)
  const bool direct =
      p.split_target == 0 && (p.num_splits == 1 || (ns_b == 1 && p.counters != nullptr));
  // 2) 4 consecutive d per thread-step.
  for (int idx = tid; idx < NC * QV; idx += NTHR) {
    const int col = idx / QV;
    const int d0 = (idx - col * QV) * 4;
    const int64_t row = cta_row_index(p, b, kvh, chunk, col);
    if (row < 0) continue;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float s = wscale[w * NC + col];
      const float4 o = *reinterpret_cast<const float4 *>(&red_o[(w * NC + col) * DP + d0]);
      acc[0] += s * o.x;
      acc[1] += s * o.y;
      acc[2] += s * o.z;
      acc[3] += s * o.w;
    }
    const float inv = wscale[W * NC + col];
    if (direct) {
      const float os = inv * p.out_scale;
      T *dst = reinterpret_cast<T *>(p.out) + row * D + d0;
#pragma unroll
      for (int e = 0; e < 4; ++e) dst[e] = from_float<T>(acc[e] * os);
    } else {
      float4 v = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
      const int64_t pi = partial_index(p, wk, row, col);
      *reinterpret_cast<float4 *>(&p.part_o[pi * D + d0]) = v;
      if (d0 == 0) p.part_lse[pi] = wscale[(W + 1) * NC + col];
    }
  }
  if (direct || p.counters == nullptr) return;

  // 3) publish the partials, count the arrival.
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = split_arrive(p, b, kvh, chunk, ns_b) ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // 4) the last CTA merges the ns_b splits of its rows.  Shared memory
  // (free now): weights[NC][kMaxFusedSplits], then 1 / sum per column.
  float *wts = red_o;
  float *winv = red_o + NC * kMaxFusedSplits;
  const int warp = tid >> 5, lane = tid & 31;
  for (int col = warp; col < NC; col += NTHR / 32) {
    const int64_t row = cta_row_index(p, b, kvh, chunk, col);
    if (row < 0) continue;
    const float lse = lane < ns_b ? __ldcg(p.part_lse + row * p.num_splits + lane) : -INFINITY;
    float M = lse;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    const float w = (M == -INFINITY) ? 0.f : ex2(lse - M);
    float sum = w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
    wts[col * kMaxFusedSplits + lane] = w;
    if (lane == 0) winv[col] = sum > 0.f ? 1.f / sum : 0.f;
  }
  __syncthreads();
  for (int idx = tid; idx < NC * QV; idx += NTHR) {
    const int col = idx / QV;
    const int d0 = (idx - col * QV) * 4;
    const int64_t row = cta_row_index(p, b, kvh, chunk, col);
    if (row < 0) continue;
    const float *po = p.part_o + row * p.num_splits * D + d0;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int sp = 0; sp < ns_b; ++sp) {
      const float w = wts[col * kMaxFusedSplits + sp];
      const float4 o = __ldcg(reinterpret_cast<const float4 *>(po + static_cast<int64_t>(sp) * D));
      acc[0] += w * o.x;
      acc[1] += w * o.y;
      acc[2] += w * o.z;
      acc[3] += w * o.w;
    }
    const float inv = winv[col] * p.out_scale;
    T *dst = reinterpret_cast<T *>(p.out) + row * D + d0;
#pragma unroll
    for (int e = 0; e < 4; ++e) dst[e] = from_float<T>(acc[e] * inv);
  }
}

}  // namespace pkv
