// pkv_api.cu -- the C ABI (include/pkv.h): argument validation, the launch
// planner, tensor-map encoding and dispatch to the kernel families.
//
// Nothing here allocates, frees or synchronises (except pkv_read_error_word,
// which documents that it does); every launch, and every host <-> device copy
// of pkv_append_attention_host, goes to the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/pkv.h"
#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMinSplitBlocks = 16;     // 4 blocks per warp: fills the pipeline
constexpr int kMaxUnitBytes = 64 * 8192;  // longest split, in K+V bytes of one KV head
                                          // (64 blocks of a 16-bit, 128-dim cache)
constexpr int kTargetWaves = 3;         // CTAs ~ this many times the resident slots
                                        // (the 20-row verify tile: 0.641 of the HBM
                                        // peak at 4 waves, 0.673 at 3)
constexpr int kMaxSplits = 32;          // per sequence: each split adds merge work
// The balanced partition's weight of a unit, in blocks: what starting and
// finishing a piece of work costs the tcgen05 kernel (its query rows, the
// first chunk's scores, the epilogue: ~5 us against ~0.2 us a block on the
// verify step).
constexpr int kStreamKWeight = 24;
constexpr size_t kUsableSmemPerSm = 228 * 1024;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elt_bytes(pkv_dtype dt) { return dt == PKV_F32 ? 4 : (dt == PKV_FP8_E4M3 ? 1 : 2); }

bool valid_dtype(int dt) { return dt == PKV_F32 || dt == PKV_BF16 || dt == PKV_F16; }

bool valid_cache_dtype(int dt) { return valid_dtype(dt) || dt == PKV_FP8_E4M3; }

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// The softmax scale of a call: a positive argument as given; zero or a
// negative value selects 1/sqrt(head_dim), the scale of standard attention.
float softmax_scale(float scale, int head_dim) {
  return scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(head_dim)));
}

struct DeviceInfo {
  std::atomic<int> sm_count{0};
};
DeviceInfo g_devices[kMaxDevices];

cudaError_t current_sm_count(int *device, int *sms) {
  cudaError_t e = cudaGetDevice(device);
  if (e != cudaSuccess) return e;
  if (*device < 0 || *device >= kMaxDevices) return cudaErrorInvalidDevice;
  int n = g_devices[*device].sm_count.load(std::memory_order_relaxed);
  if (n == 0) {
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *device);
    if (e != cudaSuccess) return e;
    g_devices[*device].sm_count.store(n, std::memory_order_relaxed);
  }
  *sms = n;
  return cudaSuccess;
}

// Once per (kernel, device): allow the kernel's dynamic shared memory and
// ask the occupancy calculator how many CTAs fit on one SM.  One slot per
// kernel instantiation a process uses (the library builds about 250).
constexpr int kMaxKernels = 1024;
struct FuncSlot {
  const void *func;
  std::atomic<int> ctas[kMaxDevices];
};
std::mutex g_func_mu;
FuncSlot g_funcs[kMaxKernels];
int g_nfuncs = 0;

cudaError_t prepare_kernel(const KernelInfo &k, int device, int *ctas_per_sm) {
  FuncSlot *slot = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_func_mu);
    for (int i = 0; i < g_nfuncs; ++i)
      if (g_funcs[i].func == k.func) slot = &g_funcs[i];
    if (!slot) {
      if (g_nfuncs >= kMaxKernels) return cudaErrorMemoryAllocation;
      slot = &g_funcs[g_nfuncs++];
      slot->func = k.func;
      for (auto &c : slot->ctas) c.store(0);
    }
  }
  int n = slot->ctas[device].load(std::memory_order_acquire);
  if (n == 0) {
    cudaError_t e = cudaFuncSetAttribute(k.func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(k.smem));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k.func, k.threads, k.smem);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    slot->ctas[device].store(n, std::memory_order_release);
  }
  *ctas_per_sm = n;
  return cudaSuccess;
}

// dtype is the cache's element type, qdtype that of q and out (equal unless
// the cache is FP8 E4M3).
struct Shape {
  int batch, num_queries, num_heads, num_kv_heads, head_dim, block_size, max_context_len;
  pkv_dtype dtype;
  pkv_dtype qdtype;
};

Shape make_shape(int batch, int num_queries, int num_heads, int num_kv_heads, int head_dim,
                 int block_size, int max_context_len, pkv_dtype dtype) {
  // Plans over an FP8 cache do not depend on q's type.
  const pkv_dtype q = dtype == PKV_FP8_E4M3 ? PKV_BF16 : dtype;
  return Shape{batch, num_queries, num_heads, num_kv_heads, head_dim, block_size,
               max_context_len, dtype, q};
}

pkv_status check_shape(const Shape &s) {
  if (s.batch < 0 || s.num_queries < 1 || s.num_heads < 1 || s.num_kv_heads < 1 ||
      s.head_dim < 1 || s.block_size < 1 || s.max_context_len < 0 ||
      !valid_cache_dtype(s.dtype) || !valid_dtype(s.qdtype))
    return PKV_ERR_INVALID_ARG;
  if (s.dtype != PKV_FP8_E4M3 && s.qdtype != s.dtype) return PKV_ERR_INVALID_ARG;
  if (s.dtype == PKV_FP8_E4M3 && s.head_dim != 128 && s.head_dim != 256)
    return PKV_ERR_UNSUPPORTED;
  if (s.num_heads % s.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (s.head_dim != 64 && s.head_dim != 128 && s.head_dim != 256) return PKV_ERR_UNSUPPORTED;
  if (s.block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (s.batch > 65535) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

// Kernel family and per-CTA row tile.  Returns false if unsupported.
bool choose_kernel(const Shape &s, const pkv_options *opt, pkv_plan *pl, KernelInfo *info) {
  const int rows = (s.num_heads / s.num_kv_heads) * s.num_queries;
  int kernel = opt ? opt->kernel : PKV_KERNEL_AUTO;
  // 16-bit and FP8 caches go to the tensor-core kernel even for one query row
  // per KV head (0.995 of the HBM peak on the 40-head, 2048-row bf16 layer,
  // against 0.974 for the CUDA-core kernel); float32 (cache or q) has no exact
  // tensor-core path.
  const bool f32 = s.dtype == PKV_F32 || s.qdtype == PKV_F32;
  if (kernel == PKV_KERNEL_AUTO) kernel = f32 ? PKV_KERNEL_SIMT : PKV_KERNEL_MMA;
  if ((kernel == PKV_KERNEL_MMA || kernel == PKV_KERNEL_TC) && f32) return false;
  if (kernel == PKV_KERNEL_TC && s.dtype != s.qdtype) return false;
  if (kernel != PKV_KERNEL_MMA && kernel != PKV_KERNEL_SIMT && kernel != PKV_KERNEL_TC)
    return false;
  int cap = kernel == PKV_KERNEL_MMA  ? 8 * mma_max_tiles(s.head_dim)
            : kernel == PKV_KERNEL_TC ? kTcMaxRows
                                      : simt_max_rows(s.head_dim);
  if (opt && opt->rows_per_cta > 0 && opt->rows_per_cta < cap) cap = opt->rows_per_cta;
  const int chunks = ceil_div(rows, cap);
  const int per_cta = ceil_div(rows, chunks);
  bool ok = false;
  const int stages = opt ? opt->stages : 0;
  if (kernel == PKV_KERNEL_MMA) {
    MmaShape m{ceil_div(per_cta, 8), opt ? opt->warp_tiles : 0,
               opt ? opt->blocks_per_iter : 0, stages};
    // Two blocks per iteration for FP8 caches with several column tiles
    // (the 20-row verify tile: 0.362 -> 0.391 of the HBM peak); one
    // otherwise (bf16 verify: 0.629 -> 0.609 with two).
    if (m.blocks_per_iter == 0 && s.dtype == PKV_FP8_E4M3 && m.n_tiles >= 2) {
      m.blocks_per_iter = 2;
      ok = mma_kernel_info(s.dtype, s.qdtype, s.head_dim, m, info);
      if (!ok) m.blocks_per_iter = 0;
    }
    if (!ok) ok = mma_kernel_info(s.dtype, s.qdtype, s.head_dim, m, info);
  } else if (kernel == PKV_KERNEL_TC) {
    ok = tc_kernel_info(s.dtype, s.head_dim, per_cta, stages, info);
  } else {
    if (stages != 0) return false;
    int r = 1;
    while (r < per_cta) r <<= 1;
    ok = simt_kernel_info(s.dtype, s.qdtype, s.head_dim, r, info);
  }
  if (!ok) return false;
  pl->kernel = kernel;
  pl->rows_per_cta = per_cta;
  pl->row_chunks = chunks;
  pl->threads_per_cta = info->threads;
  pl->stages = info->stages;
  pl->smem_bytes = info->smem;
  pl->warp_tiles = info->warp_tiles;
  pl->blocks_per_iter = info->blocks_per_iter;
  return true;
}

// Split-K workspace: float32 partial outputs, their log-sum-exps and, when
// the last CTA of a sequence merges (at most kMaxFusedSplits splits), one
// 32-bit arrival counter per (sequence, KV head, row chunk), zeroed by every
// call before its attention kernel counts in it.  Regions are 256-byte
// aligned.
struct WorkspaceLayout {
  size_t lse_off, ctr_off, total;
  bool fused_merge;
};
WorkspaceLayout workspace_layout(const Shape &s, int num_splits, int row_chunks, int rows_per_cta,
                                 int merge, int split_target = 0, int stream_k = 0) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = static_cast<size_t>(s.batch) * s.num_queries * s.num_heads;
  WorkspaceLayout w{};
  if (split_target > 0) {
    // device partitions: one partial per (work item, CTA column), merged by
    // the merge kernel; the balanced partition's slots are its CTAs plus
    // its units (a split in slot c + U)
    const size_t slots = static_cast<size_t>(split_target) +
                         (stream_k ? static_cast<size_t>(s.batch) * s.num_kv_heads * row_chunks : 0);
    const size_t parts = slots * rows_per_cta;
    w.lse_off = up(parts * s.head_dim * sizeof(float));
    w.ctr_off = w.lse_off + up(parts * sizeof(float));  // here: the layout per sequence
    w.total = w.ctr_off + up((static_cast<size_t>(s.batch) * 2 + 2) * sizeof(int));
    w.fused_merge = false;
    return w;
  }
  w.lse_off = up(rows * num_splits * s.head_dim * sizeof(float));
  w.ctr_off = w.lse_off + up(rows * num_splits * sizeof(float));
  // The completing CTA reads back rows x splits partial vectors in its tail:
  // worth it for a few (GQA, long contexts: 0.949 vs 0.936 of the HBM peak),
  // not for the 20 x 10 of speculative verification (0.567 vs 0.603).
  const bool small = static_cast<int64_t>(rows_per_cta) * num_splits <= 64;
  w.fused_merge = num_splits <= kMaxFusedSplits && (merge == 1 || (merge == 0 && small));
  w.total = w.ctr_off;
  if (w.fused_merge)
    w.total += up(static_cast<size_t>(s.batch) * s.num_kv_heads * row_chunks *
                  sizeof(unsigned int));
  return w;
}

// Split-K partition.  A sequence of n blocks is cut into chunks of
// split_blocks blocks; each chunk is one CTA.  Splitting pays when the
// unsplit grid leaves the GPU short of work (few sequences x KV heads, long
// contexts) or when long sequences would dominate the tail of a ragged batch.
void plan_splits(const Shape &s, const pkv_options *opt, int num_sms, int ctas_per_sm,
                 pkv_plan *pl) {
  const int max_blocks = ceil_div(s.max_context_len, s.block_size);
  const int64_t units =
      static_cast<int64_t>(s.batch) * s.num_kv_heads * static_cast<int64_t>(pl->row_chunks);
  const bool persistent = pl->kernel == PKV_KERNEL_TC;
  int split_blocks;
  if (opt && opt->split_blocks > 0) {
    split_blocks = opt->split_blocks;
  } else if (persistent) {
    // tcgen05 kernel: items of 256 blocks (32 chunks; the 20-row verify tile
    // measured 0.492 of the HBM peak against 0.439 at 64 and 0.489 at 128,
    // one CTA per item), or fewer when that leaves SMs idle.
    const int64_t slots = static_cast<int64_t>(num_sms) * ctas_per_sm;
    const int64_t per = (units * max_blocks + slots - 1) / slots;
    split_blocks = static_cast<int>(std::min<int64_t>(256, std::max<int64_t>(32, (per + 7) / 8 * 8)));
    if (split_blocks < ceil_div(max_blocks, kMaxSplits))
      split_blocks = (ceil_div(max_blocks, kMaxSplits) + 7) / 8 * 8;
  } else {
    const int64_t slots = static_cast<int64_t>(num_sms) * ctas_per_sm;
    const int64_t want = kTargetWaves * slots;
    const int block_bytes = 2 * s.block_size * s.head_dim * elt_bytes(s.dtype);
    const int max_unit_blocks = kMaxUnitBytes / block_bytes > 1 ? kMaxUnitBytes / block_bytes : 1;
    if (units >= want || max_blocks <= kMinSplitBlocks) {
      split_blocks = max_blocks;
    } else {
      const int64_t splits = (want + units - 1) / units;
      split_blocks = ceil_div(max_blocks, splits);
      if (split_blocks < kMinSplitBlocks) split_blocks = kMinSplitBlocks;
      if (split_blocks > max_unit_blocks && split_blocks < max_blocks) split_blocks = max_unit_blocks;
      if (split_blocks < ceil_div(max_blocks, kMaxSplits)) split_blocks = ceil_div(max_blocks, kMaxSplits);
      // Keep the split only if it shortens the schedule: with every sequence
      // at the longest length, ceil(CTAs / slots) waves of split_blocks each
      // against ceil(units / slots) waves of max_blocks.  (1280 equal
      // 128-block units on 456 slots take 3 waves whole and 6 waves of 64
      // blocks split: the same, plus the merge.)
      const int64_t ns = ceil_div(max_blocks, split_blocks);
      const int64_t whole = (units + slots - 1) / slots * max_blocks;
      const int64_t split = (units * ns + slots - 1) / slots * split_blocks;
      if (whole <= split) split_blocks = max_blocks;
    }
  }
  if (split_blocks < 1) split_blocks = 1;
  // Partition from the real lengths (read on the device, cta_work), on
  // request (split_waves = k > 0) for a batch of at most 32 sequences: k
  // waves of resident CTAs with splits of nearly equal length, whatever
  // max_context_len says.  It is not the default: measured on the long-context
  // and verify workloads it lost to the host plan (two sequences of 32768 and
  // 65536 rows: one exact wave of 456 CTAs, 0.806 of the HBM peak, against
  // 0.842 for the host's 384; speculative verify 0.588 against 0.639), the
  // kernels being bound by the bytes in flight rather than by idle slots.
  int waves = opt ? opt->split_waves : 0;
  const int64_t unit_rows = static_cast<int64_t>(s.num_kv_heads) * pl->row_chunks;
  pl->stream_k = 0;
  // The tcgen05 kernel (one CTA per SM) takes the balanced partition by
  // default: every CTA the same number of blocks, whatever the lengths.  Any
  // whole-item partition leaves SMs idle at the end: the verify step's two
  // waves of items of 13 to 19 chunks measured 0.537 of the HBM peak, the
  // host plan's 256-block items 0.512.
  if (persistent && waves == 0 && !(opt && opt->split_blocks > 0) && s.batch <= 32 &&
      max_blocks > 0 &&
      units * (max_blocks + kStreamKWeight) < (int64_t(1) << 31)) {  // int offsets on device
    const int64_t slots = static_cast<int64_t>(num_sms) * ctas_per_sm;
    pl->split_target = static_cast<int>(std::min<int64_t>(slots, 0x7fffffff));
    pl->stream_k = 1;
    pl->split_blocks = 0;
    // a unit's splits: at most one per CTA, and each holds a block
    pl->num_splits = static_cast<int>(std::min<int64_t>(slots, max_blocks));
    pl->grid_x = pl->split_target;
    pl->grid_y = pl->grid_z = 1;
    pl->ctas_per_sm = ctas_per_sm;
    const WorkspaceLayout w = workspace_layout(s, pl->num_splits, pl->row_chunks,
                                               pl->rows_per_cta, 2, pl->split_target, 1);
    pl->workspace_bytes = w.total;
    pl->merge_kernel = 1;
    return;
  }
  if (waves > 0 && !(opt && opt->split_blocks > 0) && s.batch <= 32 && max_blocks > 0 &&
      static_cast<int64_t>(max_blocks) * s.batch < (int64_t(1) << 30)) {  // int sums on device
    const int64_t slots = static_cast<int64_t>(num_sms) * ctas_per_sm;
    int64_t target = (waves > 0 ? waves : 1) * slots;
    if (target < units) target = (units + slots - 1) / slots * slots;  // one split each fits
    if (target <= 0x7fffffffLL) {
      pl->split_target = static_cast<int>(target);
      pl->split_blocks = 0;
      pl->num_splits = static_cast<int>(std::max<int64_t>(1, target / unit_rows));
      pl->grid_x = pl->split_target;
      if (persistent && opt && opt->persistent == 1)  // walk: one CTA per resident slot
        pl->grid_x = static_cast<int>(std::min<int64_t>(target, slots));
      pl->grid_y = pl->grid_z = 1;
      pl->ctas_per_sm = ctas_per_sm;
      const WorkspaceLayout w = workspace_layout(s, pl->num_splits, pl->row_chunks,
                                                 pl->rows_per_cta, 2, pl->split_target);
      pl->workspace_bytes = w.total;
      pl->merge_kernel = 1;
      return;
    }
  }
  pl->split_target = 0;
  int num_splits = max_blocks > 0 ? ceil_div(max_blocks, split_blocks) : 1;
  if (num_splits <= 1) {
    num_splits = 1;
    split_blocks = max_blocks > 0 ? max_blocks : 1;
  }
  pl->split_blocks = split_blocks;
  pl->num_splits = num_splits;
  pl->grid_x = num_splits;
  pl->grid_y = s.num_kv_heads * pl->row_chunks;
  pl->grid_z = s.batch;
  if (persistent) {
    // one CTA per resident slot walks the items (split x KV head x row chunk
    // x sequence), or (persistent = 2) one CTA per item
    const int64_t items = units * num_splits;
    const int64_t slots = static_cast<int64_t>(num_sms) * ctas_per_sm;
    // one CTA per item by default (0.492 against 0.449 walking 56-block items)
    const bool walk = opt && opt->persistent == 1;
    pl->grid_x = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>(walk ? std::min(items, slots) : items, 0x7fffffff)));
    pl->grid_y = pl->grid_z = 1;
  }
  pl->ctas_per_sm = ctas_per_sm;
  pl->workspace_bytes = 0;
  pl->merge_kernel = 0;
  if (num_splits > 1) {
    const WorkspaceLayout w = workspace_layout(s, num_splits, pl->row_chunks, pl->rows_per_cta,
                                               persistent ? 2 : (opt ? opt->merge : 0));
    pl->workspace_bytes = w.total;
    pl->merge_kernel = w.fused_merge ? 0 : 1;
  }
}

pkv_status make_plan(const Shape &s, const pkv_options *opt, int num_sms, int ctas_per_sm,
                     pkv_plan *pl, KernelInfo *info) {
  pkv_status st = check_shape(s);
  if (st != PKV_OK) return st;
  if (opt && (opt->split_blocks < 0 || opt->stages < 0 || opt->rows_per_cta < 0 ||
              opt->merge < 0 || opt->merge > 2 || opt->split_waves < -1 ||
              opt->split_waves > 64))
    return PKV_ERR_INVALID_ARG;
  if (!choose_kernel(s, opt, pl, info)) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(s.num_kv_heads) * pl->row_chunks > 65535) return PKV_ERR_UNSUPPORTED;
  if (ctas_per_sm <= 0) {
    const size_t per = info->smem + 1024;
    ctas_per_sm = static_cast<int>(kUsableSmemPerSm / per);
    if (ctas_per_sm > 2048 / info->threads) ctas_per_sm = 2048 / info->threads;
    if (ctas_per_sm < 1) ctas_per_sm = 1;
  }
  plan_splits(s, opt, num_sms, ctas_per_sm, pl);
  return PKV_OK;
}

pkv_status device_plan(const Shape &s, const pkv_options *opt, pkv_plan *pl, KernelInfo *info,
                       int *device, int *sms) {
  pkv_status st = check_shape(s);
  if (st != PKV_OK) return st;
  if (current_sm_count(device, sms) != cudaSuccess) return PKV_ERR_CUDA;
  pkv_plan tmp{};
  st = make_plan(s, opt, *sms, 1, &tmp, info);  // picks the kernel
  if (st != PKV_OK) return st;
  int ctas = 0;
  if (prepare_kernel(*info, *device, &ctas) != cudaSuccess) return PKV_ERR_CUDA;
  return make_plan(s, opt, *sms, ctas, pl, info);
}

// ---- tensor maps for the tensor-core kernel ------------------------------
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// The cache [NB, Hkv, 16, D] as a 4-D tensor (D, 16, Hkv, NB); one box is a
// 128-byte column panel (64 16-bit elements or 128 FP8 codes) of one (block,
// KV head) tile, 128-byte swizzled in shared memory.
bool encode_cache_map(CUtensorMap *map, const void *base, pkv_dtype dt, int D, int Hkv,
                      int64_t NB) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const int eb = elt_bytes(dt);
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(kBlockSize),
                              static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(NB)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * eb,
                                 static_cast<cuuint64_t>(D) * eb * kBlockSize,
                                 static_cast<cuuint64_t>(D) * eb * kBlockSize * Hkv};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / eb),
                             static_cast<cuuint32_t>(kBlockSize), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType type = dt == PKV_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : dt == PKV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return fn(map, type, 4, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same cache as a 5-D tensor (d within a panel, row, panel, KV head,
// block): one box is a whole (block, KV head) tile, all its 128-byte column
// panels, laid out in shared memory panel after panel exactly as the 4-D
// map's boxes are (so one copy instruction replaces one per panel).  The
// panel and row dimensions are listed out of address order (rows 128 * parts
// bytes apart, panels 128), which the encoder may refuse: then the caller
// keeps the 4-D map.
bool encode_cache_tile_map(CUtensorMap *map, const void *base, pkv_dtype dt, int D, int Hkv,
                           int64_t NB) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const int eb = elt_bytes(dt);
  const int parts = D * eb / 128;
  if (parts < 1 || parts * 128 != D * eb || parts > 256) return false;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(128 / eb),
                              static_cast<cuuint64_t>(kBlockSize),
                              static_cast<cuuint64_t>(parts), static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(NB)};
  const cuuint64_t row = static_cast<cuuint64_t>(D) * eb;
  const cuuint64_t strides[4] = {row, 128, row * kBlockSize, row * kBlockSize * Hkv};
  const cuuint32_t box[5] = {static_cast<cuuint32_t>(128 / eb),
                             static_cast<cuuint32_t>(kBlockSize),
                             static_cast<cuuint32_t>(parts), 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUtensorMapDataType type = dt == PKV_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : dt == PKV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return fn(map, type, 5, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

pkv_status run_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_table, int max_blocks_per_seq,
                         const int32_t *context_lens, const Shape &s, int64_t num_blocks,
                         float scale, void *workspace, size_t workspace_bytes,
                         const pkv_options *opt, int32_t *error_word, cudaStream_t stream,
                         const void *k_new = nullptr, const void *v_new = nullptr,
                         const uint64_t *tree_mask = nullptr, int64_t mask_stride = 0,
                         float k_scale = 1.f, float v_scale = 1.f, bool check_only = false) {
  pkv_status st = check_shape(s);
  if (st != PKV_OK) return st;
  if (k_new && s.dtype == PKV_FP8_E4M3) return PKV_ERR_UNSUPPORTED;
  if (s.batch == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_table || !context_lens)
    return PKV_ERR_INVALID_ARG;
  if (num_blocks < 1 || max_blocks_per_seq < 1 || !std::isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  scale = softmax_scale(scale, s.head_dim);
  if (static_cast<int64_t>(s.max_context_len) >
      static_cast<int64_t>(max_blocks_per_seq) * s.block_size)
    return PKV_ERR_INVALID_ARG;
  if (num_blocks > (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_table, 4) || !aligned(context_lens, 4) ||
      (error_word && !aligned(error_word, 4)) || !aligned(k_new, 16) || !aligned(v_new, 16))
    return PKV_ERR_ALIGNMENT;

  pkv_plan pl{};
  KernelInfo info;
  int device = 0, sms = 0;
  st = device_plan(s, opt, &pl, &info, &device, &sms);
  if (st != PKV_OK) return st;
  if (pl.workspace_bytes > 0) {
    if (!workspace || !aligned(workspace, 16) || workspace_bytes < pl.workspace_bytes)
      return PKV_ERR_WORKSPACE;
  }
  if (check_only) return PKV_OK;  // every check of a call, nothing enqueued

  AttnParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.k_new = k_new;
  p.v_new = v_new;
  p.tree_mask = reinterpret_cast<const unsigned long long *>(tree_mask);
  p.mask_stride = mask_stride;
  p.err = error_word;
  p.num_blocks = num_blocks;
  p.batch = s.batch;
  p.num_queries = s.num_queries;
  p.num_heads = s.num_heads;
  p.num_kv_heads = s.num_kv_heads;
  p.group = s.num_heads / s.num_kv_heads;
  p.rows = p.group * s.num_queries;
  p.rows_per_cta = pl.rows_per_cta;
  p.row_chunks = pl.row_chunks;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_context_len = s.max_context_len;
  p.split_blocks = pl.split_blocks;
  p.num_splits = pl.num_splits;
  p.split_target = pl.split_target;
  p.stream_k = pl.stream_k;
  p.sk_weight = pl.stream_k ? kStreamKWeight : 0;
  p.scale_log2 =
      static_cast<float>(static_cast<double>(scale) * 1.4426950408889634 * k_scale);
  p.out_scale = v_scale;
  bool merge_kernel = false;
  if (pl.num_splits > 1 || pl.split_target > 0) {
    const WorkspaceLayout w =
        workspace_layout(s, pl.num_splits, pl.row_chunks, pl.rows_per_cta,
                         pl.kernel == PKV_KERNEL_TC ? 2 : (opt ? opt->merge : 0),
                         pl.split_target, pl.stream_k);
    char *base = static_cast<char *>(workspace);
    p.part_o = reinterpret_cast<float *>(base);
    p.part_lse = reinterpret_cast<float *>(base + w.lse_off);
    if (pl.split_target > 0) p.split_info = reinterpret_cast<int *>(base + w.ctr_off);
    if (w.fused_merge) {
      p.counters = reinterpret_cast<unsigned int *>(base + w.ctr_off);
    } else {
      merge_kernel = true;
    }
  }

  const dim3 grid(pl.grid_x, pl.grid_y, pl.grid_z);
  cudaError_t e;
  if (p.counters != nullptr) {
    // whatever the workspace held: the counters start at zero
    e = zero_counters_launch(p.counters,
                             static_cast<int64_t>(s.batch) * s.num_kv_heads * pl.row_chunks,
                             stream);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
  }
  if (pl.kernel == PKV_KERNEL_MMA) {
    CUtensorMap kmap, vmap;
    p.tile_box =
        encode_cache_tile_map(&kmap, k_cache, s.dtype, s.head_dim, s.num_kv_heads, num_blocks) &&
        encode_cache_tile_map(&vmap, v_cache, s.dtype, s.head_dim, s.num_kv_heads, num_blocks);
    if (!p.tile_box &&
        (!encode_cache_map(&kmap, k_cache, s.dtype, s.head_dim, s.num_kv_heads, num_blocks) ||
         !encode_cache_map(&vmap, v_cache, s.dtype, s.head_dim, s.num_kv_heads, num_blocks)))
      return PKV_ERR_CUDA;
    const MmaShape m{ceil_div(pl.rows_per_cta, 8), pl.warp_tiles, pl.blocks_per_iter, pl.stages};
    e = mma_launch(s.dtype, s.qdtype, s.head_dim, m, kmap, vmap, p, grid, stream);
  } else if (pl.kernel == PKV_KERNEL_TC) {
    CUtensorMap kmap, vmap;
    if (!encode_cache_map(&kmap, k_cache, s.dtype, s.head_dim, s.num_kv_heads, num_blocks) ||
        !encode_cache_map(&vmap, v_cache, s.dtype, s.head_dim, s.num_kv_heads, num_blocks))
      return PKV_ERR_CUDA;
    e = tc_launch(s.dtype, s.head_dim, pl.rows_per_cta, pl.stages, kmap, vmap, p, grid, stream);
  } else {
    int r = 1;
    while (r < pl.rows_per_cta) r <<= 1;
    e = simt_launch(s.dtype, s.qdtype, s.head_dim, r, p, grid, stream);
  }
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  if (merge_kernel) {
    e = merge_launch(s.qdtype, s.head_dim, p, sms, stream);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

const char *pkv_status_string(pkv_status status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PKV_ERR_CUDA: return "CUDA runtime or launch error";
    case PKV_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case PKV_ERR_HOST_MEMORY: return "host memory allocation failed";
    default: return "unknown status";
  }
}

const char *pkv_version(void) { return "pkv 0.1.0 sm_103a"; }

pkv_status pkv_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int64_t num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int64_t num_blocks, pkv_dtype dtype,
                         int32_t *error_word, pkv_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || num_blocks < 1 ||
      !valid_dtype(dtype))
    return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
  const int64_t row_bytes = static_cast<int64_t>(head_dim) * elt_bytes(dtype);
  if (row_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(slot_mapping, 8) || (error_word && !aligned(error_word, 4)))
    return PKV_ERR_ALIGNMENT;
  int device = 0, sms = 0;
  if (current_sm_count(&device, &sms) != cudaSuccess) return PKV_ERR_CUDA;
  const cudaError_t e = append_launch(k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens,
                                      num_kv_heads, static_cast<int>(row_bytes / 16), block_size,
                                      num_blocks, error_word, sms,
                                      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_copy_blocks(void *k_cache, void *v_cache, const int32_t *src, const int32_t *dst,
                           int num_pairs, int num_kv_heads, int head_dim, int block_size,
                           int64_t num_blocks, pkv_dtype dtype, int32_t *error_word,
                           pkv_stream_t stream) {
  if (num_pairs < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || num_blocks < 1 ||
      !valid_cache_dtype(dtype))
    return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src || !dst) return PKV_ERR_INVALID_ARG;
  const int64_t block_bytes =
      static_cast<int64_t>(num_kv_heads) * block_size * head_dim * elt_bytes(dtype);
  if (block_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(src, 4) || !aligned(dst, 4) ||
      (error_word && !aligned(error_word, 4)))
    return PKV_ERR_ALIGNMENT;
  int device = 0, sms = 0;
  if (current_sm_count(&device, &sms) != cudaSuccess) return PKV_ERR_CUDA;
  const cudaError_t e = copy_blocks_launch(k_cache, v_cache, src, dst, num_pairs, block_bytes,
                                           num_blocks, error_word, sms,
                                           reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Q [total_q, Hq, D] as a 3-D tensor (D, Hq, total_q); one box is a
// 128-byte column panel of 128 rows: 128 / group positions x the group's
// heads, 128-byte swizzled.  Rows past total_q read as zero.
bool encode_query_map(CUtensorMap *map, const void *base, pkv_dtype dt, int D, int Hq,
                      int total_q, int group) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const int eb = elt_bytes(dt);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                              static_cast<cuuint64_t>(total_q)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * eb,
                                 static_cast<cuuint64_t>(D) * eb * Hq};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / eb), static_cast<cuuint32_t>(group),
                             static_cast<cuuint32_t>(128 / group)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType type =
      dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(map, type, 3, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

pkv_status pkv_paged_prefill_attention(void *out, const void *q, const void *k_cache,
                                       const void *v_cache, const int32_t *block_table,
                                       int max_blocks_per_seq, const int32_t *context_lens,
                                       const int32_t *query_start, int max_query_len, int batch,
                                       int total_q, int num_heads, int num_kv_heads, int head_dim,
                                       int block_size, int64_t num_blocks, float scale,
                                       pkv_dtype dtype, const pkv_options *options,
                                       int32_t *error_word, pkv_stream_t stream) {
  if (batch < 0 || total_q < 0 || max_query_len < 0 || num_heads < 1 || num_kv_heads < 1 ||
      num_heads % num_kv_heads != 0 || !valid_dtype(dtype))
    return PKV_ERR_INVALID_ARG;
  const int group = num_heads / num_kv_heads;
  const int stages = options ? options->stages : 0;
  if (block_size != kBlockSize || !prefill_supported(dtype, head_dim, group, stages))
    return PKV_ERR_UNSUPPORTED;
  if (batch == 0 || total_q == 0 || max_query_len == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_table || !context_lens || !query_start)
    return PKV_ERR_INVALID_ARG;
  if (num_blocks < 1 || max_blocks_per_seq < 1 || !std::isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(max_query_len) * group;
  const int64_t pairs = (rows + prefill_rows_per_cta() - 1) / prefill_rows_per_cta();
  if (pairs * batch * num_kv_heads > 0x7fffffff) return PKV_ERR_UNSUPPORTED;  // one CTA each
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_table, 4) || !aligned(context_lens, 4) || !aligned(query_start, 4) ||
      (error_word && !aligned(error_word, 4)))
    return PKV_ERR_ALIGNMENT;
  CUtensorMap qmap, kmap, vmap;
  if (!encode_query_map(&qmap, q, dtype, head_dim, num_heads, total_q, group) ||
      !encode_cache_map(&kmap, k_cache, dtype, head_dim, num_kv_heads, num_blocks) ||
      !encode_cache_map(&vmap, v_cache, dtype, head_dim, num_kv_heads, num_blocks))
    return PKV_ERR_INVALID_ARG;
  PrefillParams p{};
  p.out = out;
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.query_start = query_start;
  p.err = error_word;
  p.num_blocks = num_blocks;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.batch = batch;
  p.total_q = total_q;
  p.max_query_len = max_query_len;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = group;
  p.pairs = static_cast<int>(pairs);
  p.scale_log2 = softmax_scale(scale, head_dim) * 1.4426950408889634f;
  const cudaError_t e = prefill_launch(dtype, head_dim, stages, qmap, kmap, vmap, p,
                                       reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_check_bounded_wait(int32_t *error_word, uint32_t limit_us,
                                  uint64_t *waited_ns, pkv_stream_t stream) {
  if (!error_word || limit_us < 1 || limit_us > 10000000u) return PKV_ERR_INVALID_ARG;
  if (!aligned(error_word, 4) || (waited_ns && !aligned(waited_ns, 8))) return PKV_ERR_ALIGNMENT;
  const cudaError_t e = bounded_wait_launch(
      error_word, 1000ull * limit_us, reinterpret_cast<unsigned long long *>(waited_ns),
      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_attention_plan_for(int batch, int num_queries, int num_heads, int num_kv_heads,
                                  int head_dim, int block_size, int max_context_len,
                                  pkv_dtype dtype, const pkv_options *options, int num_sms,
                                  int ctas_per_sm, pkv_plan *plan) {
  if (!plan || num_sms < 1 || ctas_per_sm < 0) return PKV_ERR_INVALID_ARG;
  const Shape s = make_shape(batch, num_queries, num_heads, num_kv_heads, head_dim, block_size,
                max_context_len, dtype);
  pkv_plan pl{};
  KernelInfo info;
  const pkv_status st = make_plan(s, options, num_sms, ctas_per_sm, &pl, &info);
  if (st == PKV_OK) *plan = pl;
  return st;
}

pkv_status pkv_attention_plan(int batch, int num_queries, int num_heads, int num_kv_heads,
                              int head_dim, int block_size, int max_context_len, pkv_dtype dtype,
                              const pkv_options *options, pkv_plan *plan) {
  if (!plan) return PKV_ERR_INVALID_ARG;
  const Shape s = make_shape(batch, num_queries, num_heads, num_kv_heads, head_dim, block_size,
                max_context_len, dtype);
  pkv_plan pl{};
  KernelInfo info;
  int device = 0, sms = 0;
  const pkv_status st = device_plan(s, options, &pl, &info, &device, &sms);
  if (st == PKV_OK) *plan = pl;
  return st;
}

pkv_status pkv_attention_workspace_size(int batch, int num_queries, int num_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int max_context_len, pkv_dtype dtype,
                                        const pkv_options *options, size_t *bytes) {
  if (!bytes) return PKV_ERR_INVALID_ARG;
  pkv_plan pl{};
  const pkv_status st = pkv_attention_plan(batch, num_queries, num_heads, num_kv_heads, head_dim,
                                           block_size, max_context_len, dtype, options, &pl);
  if (st != PKV_OK) return st;
  *bytes = pl.workspace_bytes;
  if (dtype == PKV_FP8_E4M3 && (!options || options->kernel != PKV_KERNEL_MMA)) {
    // float32 queries over an FP8 cache take the CUDA-core kernel: report
    // enough for either plan.
    Shape s = make_shape(batch, num_queries, num_heads, num_kv_heads, head_dim, block_size,
                         max_context_len, dtype);
    s.qdtype = PKV_F32;
    pkv_plan p32{};
    KernelInfo info;
    int device = 0, sms = 0;
    if (device_plan(s, options, &p32, &info, &device, &sms) == PKV_OK &&
        p32.workspace_bytes > *bytes)
      *bytes = p32.workspace_bytes;
  }
  return PKV_OK;
}

pkv_status pkv_paged_decode_attention(void *out, const void *q, const void *k_cache,
                                      const void *v_cache, const int32_t *block_table,
                                      int max_blocks_per_seq, const int32_t *context_lens,
                                      int max_context_len, int batch, int num_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int64_t num_blocks, float scale, pkv_dtype dtype,
                                      void *workspace, size_t workspace_bytes,
                                      const pkv_options *options, int32_t *error_word,
                                      pkv_stream_t stream) {
  if (dtype == PKV_FP8_E4M3) return PKV_ERR_INVALID_ARG;  // pkv_paged_attention_fp8
  const Shape s = make_shape(batch, 1, num_heads, num_kv_heads, head_dim, block_size, max_context_len, dtype);
  return run_attention(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens, s,
                       num_blocks, scale, workspace, workspace_bytes, options, error_word,
                       reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_spec_verify_attention(void *out, const void *q, const void *k_cache,
                                     const void *v_cache, const int32_t *block_table,
                                     int max_blocks_per_seq, const int32_t *context_lens,
                                     int max_context_len, int batch, int num_queries,
                                     int num_heads, int num_kv_heads, int head_dim,
                                     int block_size, int64_t num_blocks, float scale,
                                     pkv_dtype dtype, void *workspace, size_t workspace_bytes,
                                     const pkv_options *options, int32_t *error_word,
                                     pkv_stream_t stream) {
  if (dtype == PKV_FP8_E4M3) return PKV_ERR_INVALID_ARG;  // pkv_paged_attention_fp8
  const Shape s = make_shape(batch, num_queries, num_heads, num_kv_heads, head_dim, block_size,
                max_context_len, dtype);
  return run_attention(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens, s,
                       num_blocks, scale, workspace, workspace_bytes, options, error_word,
                       reinterpret_cast<cudaStream_t>(stream));
}

pkv_status pkv_append_attention(void *out, const void *q, const void *k_new, const void *v_new,
                                void *k_cache, void *v_cache, const int32_t *block_table,
                                int max_blocks_per_seq, const int32_t *context_lens,
                                int max_context_len, int batch, int num_queries, int num_heads,
                                int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                float scale, pkv_dtype dtype, void *workspace,
                                size_t workspace_bytes, const pkv_options *options,
                                int32_t *error_word, pkv_stream_t stream) {
  if (dtype == PKV_FP8_E4M3) return PKV_ERR_INVALID_ARG;  // pkv_paged_attention_fp8
  if (batch > 0 && (!k_new || !v_new)) return PKV_ERR_INVALID_ARG;
  const Shape s = make_shape(batch, num_queries, num_heads, num_kv_heads, head_dim, block_size,
                max_context_len, dtype);
  return run_attention(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens, s,
                       num_blocks, scale, workspace, workspace_bytes, options, error_word,
                       reinterpret_cast<cudaStream_t>(stream), k_new, v_new);
}

namespace {
// The staging buffer of a host-buffer step, in this order, each piece at a
// 256-byte boundary: q, k_new, v_new, block_table, context_lens, out, then
// the attention workspace.
struct Staging {
  size_t q, k_new, v_new, table, lens, out, ws, total;
};
size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

pkv_status staging_layout(int batch, int num_queries, int num_heads, int num_kv_heads,
                          int head_dim, int block_size, int max_blocks_per_seq,
                          int max_context_len, pkv_dtype dtype, const pkv_options *options,
                          Staging *st) {
  if (!valid_dtype(dtype) || batch < 0 || num_queries < 1 || num_heads < 1 ||
      num_kv_heads < 1 || head_dim < 1 || max_blocks_per_seq < 1)
    return PKV_ERR_INVALID_ARG;
  size_t ws = 0;
  const pkv_status s = pkv_attention_workspace_size(batch, num_queries, num_heads, num_kv_heads,
                                                    head_dim, block_size, max_context_len, dtype,
                                                    options, &ws);
  if (s != PKV_OK) return s;
  const size_t rows = static_cast<size_t>(batch) * num_queries;
  const size_t q = rows * num_heads * head_dim * elt_bytes(dtype);
  const size_t kv = rows * num_kv_heads * head_dim * elt_bytes(dtype);
  size_t at = 0;
  auto take = [&](size_t n) {
    const size_t here = at;
    at += round256(n);
    return here;
  };
  st->q = take(q);
  st->k_new = take(kv);
  st->v_new = take(kv);
  st->table = take(static_cast<size_t>(batch) * max_blocks_per_seq * sizeof(int32_t));
  st->lens = take(static_cast<size_t>(batch) * sizeof(int32_t));
  st->out = take(q);
  st->ws = take(ws);
  st->total = at;
  return PKV_OK;
}
}  // namespace

pkv_status pkv_host_step_staging_size(int batch, int num_queries, int num_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int max_blocks_per_seq, int max_context_len,
                                      pkv_dtype dtype, const pkv_options *options,
                                      size_t *bytes) {
  if (!bytes) return PKV_ERR_INVALID_ARG;
  Staging st{};
  const pkv_status s = staging_layout(batch, num_queries, num_heads, num_kv_heads, head_dim,
                                      block_size, max_blocks_per_seq, max_context_len, dtype,
                                      options, &st);
  if (s == PKV_OK) *bytes = st.total;
  return s;
}

// Device address through which kernels can read or write host memory `p`
// in place (page-locked, mapped memory: on GB300 the GPU reaches it over the
// chip-to-chip link), or nullptr when they cannot (pageable memory, or a
// pointer the runtime does not know).
void *host_mapped(const void *p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();  // clear the lookup's error
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

pkv_status pkv_append_attention_host(void *out_host, const void *q_host, const void *k_new_host,
                                     const void *v_new_host, void *k_cache, void *v_cache,
                                     const int32_t *block_table_host, int max_blocks_per_seq,
                                     const int32_t *context_lens_host, int max_context_len,
                                     int batch, int num_queries, int num_heads, int num_kv_heads,
                                     int head_dim, int block_size, int64_t num_blocks,
                                     float scale, pkv_dtype dtype, void *staging,
                                     size_t staging_bytes, const pkv_options *options,
                                     int32_t *error_word, pkv_stream_t stream) {
  if (!valid_dtype(dtype) || batch < 0 || num_queries < 1 || max_blocks_per_seq < 1)
    return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (!out_host || !q_host || !k_new_host || !v_new_host || !block_table_host ||
      !context_lens_host)
    return PKV_ERR_INVALID_ARG;
  if (!staging || !aligned(staging, 256)) return PKV_ERR_WORKSPACE;
  Staging st{};
  pkv_status s = staging_layout(batch, num_queries, num_heads, num_kv_heads, head_dim,
                                block_size, max_blocks_per_seq, max_context_len, dtype, options,
                                &st);
  if (s != PKV_OK) return s;
  if (staging_bytes < st.total) return PKV_ERR_WORKSPACE;
  uint8_t *base = static_cast<uint8_t *>(staging);
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const Shape shape = make_shape(batch, num_queries, num_heads, num_kv_heads, head_dim,
                                 block_size, max_context_len, dtype);
  const size_t rows = static_cast<size_t>(batch) * num_queries;
  const size_t q_bytes = rows * num_heads * head_dim * elt_bytes(dtype);
  const size_t kv_bytes = rows * num_kv_heads * head_dim * elt_bytes(dtype);
  // Where the kernels find each input.  The block table and the lengths are
  // read at the start of every CTA, before its first copy can be issued, so
  // they are staged in device memory: pulled in by one gather kernel when
  // the GPU can address them (mapped page-locked memory; on GB300 the
  // chip-to-chip link carries the accesses).  The new K/V rows are read by
  // the kernels in place (only where a sequence ends), and so is q when the
  // plan splits a sequence at most 4 ways (each q row is read by its splits'
  // CTAs, after their first copies are in flight; with more splits the
  // repeated fetches across the link cost more than one gather: 22 splits of
  // the speculative-verify step, 0.11 ms in place against 0.095 gathered),
  // so those bytes cross the link while the cache streams from HBM.
  // An input the GPU cannot address takes one host-to-device copy into the
  // staging buffer.  The output is written straight into mapped host memory
  // (stores do not wait), else staged and copied back.
  pkv_plan plan{};
  {
    KernelInfo info;
    int device = 0, sms = 0;
    s = device_plan(shape, options, &plan, &info, &device, &sms);
    if (s != PKV_OK) return s;
  }
  const bool q_in_place = plan.num_splits <= 4 && plan.split_target == 0;
  struct In {
    size_t off;
    const void *src;
    size_t n;
    bool in_place_ok;
    const void *use;  // what the kernels read
    bool copy;        // a host-to-device copy into the staging buffer
  } in[] = {{st.q, q_host, q_bytes, q_in_place, nullptr, false},
            {st.k_new, k_new_host, kv_bytes, true, nullptr, false},
            {st.v_new, v_new_host, kv_bytes, true, nullptr, false},
            {st.table, block_table_host,
             static_cast<size_t>(batch) * max_blocks_per_seq * sizeof(int32_t), false, nullptr,
             false},
            {st.lens, context_lens_host, static_cast<size_t>(batch) * sizeof(int32_t), false,
             nullptr, false}};
  GatherList gather{};
  for (auto &c : in) {
    const void *mapped = host_mapped(c.src);
    if (mapped && c.in_place_ok && aligned(mapped, 16)) {
      c.use = mapped;
    } else if (mapped && aligned(mapped, 4)) {
      gather.item[gather.count++] = {mapped, base + c.off, static_cast<int64_t>(c.n)};
      c.use = base + c.off;
    } else {
      c.copy = true;
      c.use = base + c.off;
    }
  }
  void *out_dev = host_mapped(out_host);
  if (out_dev && !aligned(out_dev, 16)) out_dev = nullptr;
  const bool out_staged = out_dev == nullptr;
  if (out_staged) out_dev = base + st.out;
  // Every check of the launch, on the pointers it will use, before anything is enqueued.
  auto attend = [&](bool check_only) {
    return run_attention(out_dev, in[0].use, k_cache, v_cache,
                         static_cast<const int32_t *>(in[3].use), max_blocks_per_seq,
                         static_cast<const int32_t *>(in[4].use), shape, num_blocks, scale,
                         base + st.ws, staging_bytes - st.ws, options, error_word, cs, in[1].use,
                         in[2].use, nullptr, 0, 1.f, 1.f, check_only);
  };
  s = attend(true);
  if (s != PKV_OK) return s;
  for (const auto &c : in)  // host to device, one copy per input the GPU cannot address
    if (c.copy && cudaMemcpyAsync(base + c.off, c.src, c.n, cudaMemcpyHostToDevice, cs) !=
                      cudaSuccess)
      return PKV_ERR_CUDA;
  if (gather.count > 0) {
    int device = 0, sms = 0;
    if (current_sm_count(&device, &sms) != cudaSuccess ||
        gather_launch(gather, sms, cs) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  s = attend(false);
  if (s != PKV_OK) return s;
  if (out_staged &&
      cudaMemcpyAsync(out_host, base + st.out, q_bytes, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

pkv_status pkv_tree_verify_attention(void *out, const void *q, const void *k_cache,
                                     const void *v_cache, const int32_t *block_table,
                                     int max_blocks_per_seq, const int32_t *context_lens,
                                     int max_context_len, int batch, int num_queries,
                                     int num_heads, int num_kv_heads, int head_dim,
                                     int block_size, int64_t num_blocks, float scale,
                                     pkv_dtype dtype, const uint64_t *tree_mask,
                                     int64_t mask_batch_stride, void *workspace,
                                     size_t workspace_bytes, const pkv_options *options,
                                     int32_t *error_word, pkv_stream_t stream) {
  if (dtype == PKV_FP8_E4M3) return PKV_ERR_INVALID_ARG;  // pkv_paged_attention_fp8
  if (num_queries > 64 || mask_batch_stride < 0) return PKV_ERR_INVALID_ARG;
  if (batch > 0 && !tree_mask) return PKV_ERR_INVALID_ARG;
  if (!aligned(tree_mask, 8)) return PKV_ERR_ALIGNMENT;
  const Shape s = make_shape(batch, num_queries, num_heads, num_kv_heads, head_dim, block_size,
                max_context_len, dtype);
  return run_attention(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens, s,
                       num_blocks, scale, workspace, workspace_bytes, options, error_word,
                       reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr, tree_mask,
                       mask_batch_stride);
}

pkv_status pkv_kv_append_fp8(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                             const int64_t *slot_mapping, int64_t num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int64_t num_blocks,
                             pkv_dtype src_dtype, float k_scale, float v_scale,
                             int32_t *error_word, pkv_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || num_blocks < 1 ||
      !valid_dtype(src_dtype) || !(k_scale > 0.f) || !(v_scale > 0.f) ||
      !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (head_dim % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(slot_mapping, 8) || (error_word && !aligned(error_word, 4)))
    return PKV_ERR_ALIGNMENT;
  int device = 0, sms = 0;
  if (current_sm_count(&device, &sms) != cudaSuccess) return PKV_ERR_CUDA;
  const cudaError_t e = append_fp8_launch(src_dtype, k_new, v_new, k_cache, v_cache, slot_mapping,
                                          num_tokens, num_kv_heads, head_dim, block_size,
                                          num_blocks, k_scale, v_scale, error_word, sms,
                                          reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_paged_attention_fp8(void *out, const void *q, const void *k_cache,
                                   const void *v_cache, const int32_t *block_table,
                                   int max_blocks_per_seq, const int32_t *context_lens,
                                   int max_context_len, int batch, int num_queries, int num_heads,
                                   int num_kv_heads, int head_dim, int block_size,
                                   int64_t num_blocks, float scale, pkv_dtype q_dtype,
                                   float k_scale, float v_scale, void *workspace,
                                   size_t workspace_bytes, const pkv_options *options,
                                   int32_t *error_word, pkv_stream_t stream) {
  if (!valid_dtype(q_dtype) || !(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) ||
      !std::isfinite(v_scale))
    return PKV_ERR_INVALID_ARG;
  Shape s = make_shape(batch, num_queries, num_heads, num_kv_heads, head_dim, block_size,
                       max_context_len, PKV_FP8_E4M3);
  s.qdtype = q_dtype;
  return run_attention(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens, s,
                       num_blocks, scale, workspace, workspace_bytes, options, error_word,
                       reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr, 0,
                       k_scale, v_scale);
}

}  // extern "C"

namespace pkv {
namespace {

// An MLA decode call's checked sizes and launch plan: split-K over the
// latent rows with the rules of the other decode kernels (about kTargetWaves
// waves of CTAs, >= kMinSplitBlocks blocks and <= kMaxSplits splits per
// sequence), units being (sequence, 16 query heads).
struct MlaPlan {
  KernelInfo info;
  int device = 0, sms = 0, ctas_per_sm = 0;
  int split_blocks = 1, num_splits = 1;
  size_t lse_off = 0, workspace = 0;
};

pkv_status mla_plan(int batch, int num_heads, int latent_dim, int rope_dim, int block_size,
                    int max_context_len, pkv_dtype dtype, const pkv_options *opt, MlaPlan *pl) {
  if (batch < 0 || num_heads < 1 || latent_dim < 1 || rope_dim < 0 || block_size < 1 ||
      max_context_len < 0 || !valid_dtype(dtype))
    return PKV_ERR_INVALID_ARG;
  if (latent_dim != kMlaLatent || (rope_dim != 0 && rope_dim != 64) || dtype == PKV_F32 ||
      block_size != kBlockSize || num_heads % kMlaHeadsPerCta != 0 || batch > 65535 ||
      num_heads / kMlaHeadsPerCta > 65535)
    return PKV_ERR_UNSUPPORTED;
  if (opt && (opt->kernel != PKV_KERNEL_AUTO || opt->rows_per_cta != 0 || opt->merge != 0 ||
              opt->warp_tiles != 0 || opt->blocks_per_iter != 0 || opt->persistent != 0 ||
              opt->split_waves != 0))
    return PKV_ERR_UNSUPPORTED;  // only stages and split_blocks apply here
  if (!mla_kernel_info(dtype, rope_dim, opt ? opt->stages : 0, &pl->info))
    return PKV_ERR_UNSUPPORTED;
  if (current_sm_count(&pl->device, &pl->sms) != cudaSuccess) return PKV_ERR_CUDA;
  if (prepare_kernel(pl->info, pl->device, &pl->ctas_per_sm) != cudaSuccess) return PKV_ERR_CUDA;
  const int max_blocks = ceil_div(max_context_len, kBlockSize);
  const int64_t units = static_cast<int64_t>(batch) * (num_heads / kMlaHeadsPerCta);
  int sb = max_blocks;
  if (opt && opt->split_blocks > 0) {
    sb = opt->split_blocks;
  } else if (units > 0 && max_blocks > kMinSplitBlocks) {
    const int64_t slots = static_cast<int64_t>(pl->sms) * pl->ctas_per_sm;
    const int64_t want = kTargetWaves * slots;
    if (units < want) {
      const int64_t splits = (want + units - 1) / units;
      sb = std::max(kMinSplitBlocks, ceil_div(max_blocks, splits));
      sb = std::max(sb, ceil_div(max_blocks, kMaxSplits));
      // keep the split only if it shortens the wave-quantised schedule
      const int64_t ns = ceil_div(max_blocks, sb);
      const int64_t whole = (units + slots - 1) / slots * max_blocks;
      const int64_t split = (units * ns + slots - 1) / slots * sb;
      if (whole <= split) sb = max_blocks;
    }
  }
  if (sb < 1) sb = 1;
  int ns = max_blocks > 0 ? ceil_div(max_blocks, sb) : 1;
  if (ns <= 1) {
    ns = 1;
    sb = max_blocks > 0 ? max_blocks : 1;
  }
  if (ns > 65535) return PKV_ERR_UNSUPPORTED;
  pl->split_blocks = sb;
  pl->num_splits = ns;
  if (ns > 1) {
    const size_t rows = static_cast<size_t>(batch) * num_heads * ns;
    pl->lse_off = (rows * kMlaLatent * sizeof(float) + 255) & ~static_cast<size_t>(255);
    pl->workspace = pl->lse_off + rows * sizeof(float);
  }
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_mla_plan(int batch, int num_heads, int latent_dim, int rope_dim, int block_size,
                        int max_context_len, pkv_dtype dtype, const pkv_options *options,
                        pkv_plan *plan) {
  if (!plan) return PKV_ERR_INVALID_ARG;
  MlaPlan pl;
  const pkv_status st = mla_plan(batch, num_heads, latent_dim, rope_dim, block_size,
                                 max_context_len, dtype, options, &pl);
  if (st != PKV_OK) return st;
  *plan = pkv_plan{};
  plan->kernel = PKV_KERNEL_MMA;
  plan->rows_per_cta = kMlaHeadsPerCta;
  plan->row_chunks = num_heads / kMlaHeadsPerCta;
  plan->split_blocks = pl.split_blocks;
  plan->num_splits = pl.num_splits;
  plan->grid_x = pl.num_splits;
  plan->grid_y = num_heads / kMlaHeadsPerCta;
  plan->grid_z = batch;
  plan->threads_per_cta = pl.info.threads;
  plan->stages = pl.info.stages;
  plan->ctas_per_sm = pl.ctas_per_sm;
  plan->smem_bytes = pl.info.smem;
  plan->workspace_bytes = pl.workspace;
  plan->merge_kernel = pl.num_splits > 1 ? 1 : 0;
  plan->warp_tiles = 1;
  plan->blocks_per_iter = 1;
  return PKV_OK;
}

pkv_status pkv_mla_workspace_size(int batch, int num_heads, int latent_dim, int rope_dim,
                                  int block_size, int max_context_len, pkv_dtype dtype,
                                  const pkv_options *options, size_t *bytes) {
  if (!bytes) return PKV_ERR_INVALID_ARG;
  MlaPlan pl;
  const pkv_status st = mla_plan(batch, num_heads, latent_dim, rope_dim, block_size,
                                 max_context_len, dtype, options, &pl);
  if (st == PKV_OK) *bytes = pl.workspace;
  return st;
}

pkv_status pkv_mla_decode_attention(void *out, const void *q, const void *ckv_cache,
                                    const int32_t *block_table, int max_blocks_per_seq,
                                    const int32_t *context_lens, int max_context_len, int batch,
                                    int num_heads, int latent_dim, int rope_dim, int block_size,
                                    int64_t num_blocks, float scale, pkv_dtype dtype,
                                    void *workspace, size_t workspace_bytes,
                                    const pkv_options *options, int32_t *error_word,
                                    pkv_stream_t stream) {
  // argument checks that need no device come first
  if (batch < 0 || num_heads < 1 || max_context_len < 0 || !valid_dtype(dtype))
    return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (!out || !q || !ckv_cache || !block_table || !context_lens) return PKV_ERR_INVALID_ARG;
  if (num_blocks < 1 || max_blocks_per_seq < 1 || !std::isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * kBlockSize)
    return PKV_ERR_INVALID_ARG;
  if (num_blocks > (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(ckv_cache, 16) ||
      !aligned(block_table, 4) || !aligned(context_lens, 4) ||
      (error_word && !aligned(error_word, 4)))
    return PKV_ERR_ALIGNMENT;
  MlaPlan pl;
  pkv_status st = mla_plan(batch, num_heads, latent_dim, rope_dim, block_size, max_context_len,
                           dtype, options, &pl);
  if (st != PKV_OK) return st;
  if (pl.workspace > 0 &&
      (!workspace || !aligned(workspace, 256) || workspace_bytes < pl.workspace))
    return PKV_ERR_WORKSPACE;
  CUtensorMap cmap;
  const bool tile_box =
      encode_cache_tile_map(&cmap, ckv_cache, dtype, latent_dim + rope_dim, 1, num_blocks);
  if (!tile_box && !encode_cache_map(&cmap, ckv_cache, dtype, latent_dim + rope_dim, 1, num_blocks))
    return PKV_ERR_CUDA;

  AttnParams p{};
  p.tile_box = tile_box ? 1 : 0;
  p.out = out;
  p.q = q;
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.err = error_word;
  p.num_blocks = num_blocks;
  p.batch = batch;
  p.num_queries = 1;
  p.num_heads = num_heads;
  p.num_kv_heads = 1;
  p.group = num_heads;
  p.rows = num_heads;
  p.rows_per_cta = kMlaHeadsPerCta;
  p.row_chunks = num_heads / kMlaHeadsPerCta;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_context_len = max_context_len;
  p.split_blocks = pl.split_blocks;
  p.num_splits = pl.num_splits;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.out_scale = 1.f;
  if (pl.num_splits > 1) {
    p.part_o = static_cast<float *>(workspace);
    p.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + pl.lse_off);
  }
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid(pl.num_splits, num_heads / kMlaHeadsPerCta, batch);
  if (mla_launch(dtype, rope_dim, options ? options->stages : 0, cmap, p, grid, cs) !=
      cudaSuccess)
    return PKV_ERR_CUDA;
  if (pl.num_splits > 1 && mla_merge_launch(dtype, p, cs) != cudaSuccess) return PKV_ERR_CUDA;
  return PKV_OK;
}

pkv_status pkv_mla_append(const void *ckv_new, void *ckv_cache, const int64_t *slot_mapping,
                          int64_t num_tokens, int width, int block_size, int64_t num_blocks,
                          pkv_dtype dtype, int32_t *error_word, pkv_stream_t stream) {
  if (num_tokens < 0 || width < 1 || block_size < 1 || num_blocks < 1 || !valid_dtype(dtype))
    return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!ckv_new || !ckv_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
  const int64_t row_bytes = static_cast<int64_t>(width) * elt_bytes(dtype);
  if (row_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (!aligned(ckv_new, 16) || !aligned(ckv_cache, 16) || !aligned(slot_mapping, 8) ||
      (error_word && !aligned(error_word, 4)))
    return PKV_ERR_ALIGNMENT;
  int device = 0, sms = 0;
  if (current_sm_count(&device, &sms) != cudaSuccess) return PKV_ERR_CUDA;
  return append_launch(ckv_new, nullptr, ckv_cache, nullptr, slot_mapping, num_tokens, 1,
                       static_cast<int>(row_bytes / 16), block_size, num_blocks, error_word, sms,
                       reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

pkv_status pkv_read_error_word(const int32_t *error_word, int32_t *host_code,
                               pkv_stream_t stream) {
  if (!error_word || !host_code) return PKV_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_code, error_word, sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return PKV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
  return PKV_OK;
}

}  // extern "C"

// ---- no-allocation variant --------------------------------------------
// Scratch for the split-K partials of pkv_paged_decode_attention_noalloc.
// In host code this name only stands in for the array; its device address
// is looked up per device below and passed to the kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {
std::atomic<void *> g_noalloc_ptr[pkv::kMaxDevices];
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device (looked up on
// the first call per device).
cudaError_t noalloc_scratch(void **ptr) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 0 || device >= pkv::kMaxDevices) return cudaErrorInvalidDevice;
  void *p = g_noalloc_ptr[device].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    p = g_noalloc_ptr[device].load(std::memory_order_acquire);
    if (!p) {
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return e;
      g_noalloc_ptr[device].store(p, std::memory_order_release);
    }
  }
  *ptr = p;
  return cudaSuccess;
}
}  // namespace

extern "C" pkv_status pkv_paged_decode_attention_noalloc(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_table, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int batch, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int64_t num_blocks, float scale, pkv_dtype dtype,
    const pkv_options *options, int32_t *error_word, pkv_stream_t stream) {
  if (batch == 0) return PKV_OK;
  // The size checked here and the size the launch below uses come from the
  // same planner (device_plan, on the current device, with these arguments
  // and options), so the launch never needs more than the bound checked.
  size_t need = 0;
  pkv_status st = pkv_attention_workspace_size(batch, 1, num_heads, num_kv_heads, head_dim,
                                               block_size, max_context_len, dtype, options, &need);
  if (st != PKV_OK) return st;
  if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return PKV_ERR_CUDA;
  return pkv_paged_decode_attention(out, q, k_cache, v_cache, block_table, max_blocks_per_seq,
                                    context_lens, max_context_len, batch, num_heads,
                                    num_kv_heads, head_dim, block_size, num_blocks, scale, dtype,
                                    scratch, PKV_NOALLOC_SCRATCH_BYTES, options, error_word,
                                    stream);
}
