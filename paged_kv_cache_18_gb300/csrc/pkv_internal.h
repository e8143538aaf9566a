// pkv_internal.h -- host-side declarations shared by the library's
// translation units (kernel families, their launchers and shared-memory
// needs).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/pkv.h"

namespace pkv {

struct AttnParams;
struct PrefillParams;

struct KernelInfo {
  const void *func = nullptr;
  int threads = 0;
  int warps = 0;
  int stages = 0;
  int warp_tiles = 1;
  int blocks_per_iter = 1;
  size_t smem = 0;
};

// Tensor-core kernel shape: n_tiles = query columns / 8, warp_tiles of them
// per warp (0 = one), blocks_per_iter KV blocks per loop iteration (0 =
// one), stages = per-lane ring depth (0 = default).
struct MmaShape {
  int n_tiles, warp_tiles, blocks_per_iter, stages;
};

// The cache type is q's 16-bit type, or FP8 E4M3 with bf16 / f16 q
// (head_dim 128 or 256).
int mma_max_tiles(int head_dim);
bool mma_kernel_info(pkv_dtype cache_dtype, pkv_dtype q_dtype, int head_dim, const MmaShape &m,
                     KernelInfo *info);
cudaError_t mma_launch(pkv_dtype cache_dtype, pkv_dtype q_dtype, int head_dim, const MmaShape &m,
                       const CUtensorMap &kmap, const CUtensorMap &vmap, const AttnParams &p,
                       dim3 grid, cudaStream_t stream);

// tcgen05 kernel (TMEM accumulators, 128-key chunks): bf16 / f16 caches, q of
// the same type, head_dim 128, up to 64 query rows per CTA.
constexpr int kTcMaxRows = 64;
// stages: V ring depth 1..3 (1..2 above 32 rows; 0 = default).
bool tc_kernel_info(pkv_dtype dtype, int head_dim, int rows_per_cta, int stages,
                    KernelInfo *info);
cudaError_t tc_launch(pkv_dtype dtype, int head_dim, int rows_per_cta, int stages,
                      const CUtensorMap &kmap, const CUtensorMap &vmap, const AttnParams &p,
                      dim3 grid, cudaStream_t stream);

// A one-thread wait on a barrier nothing arrives on, bounded by limit_ns.
cudaError_t bounded_wait_launch(int32_t *err, unsigned long long limit_ns,
                                unsigned long long *waited_ns, cudaStream_t stream);

// Chunked prefill on the tcgen05 tensor cores (attn_prefill.cu): head_dim 64
// or 128, bf16 / f16, group size dividing 128.  `stages` is the K/V ring
// depth (0: default).
bool prefill_supported(pkv_dtype dtype, int head_dim, int group, int stages);
int prefill_rows_per_cta();
cudaError_t prefill_launch(pkv_dtype dtype, int head_dim, int stages, const CUtensorMap &qmap,
                           const CUtensorMap &kmap, const CUtensorMap &vmap,
                           const PrefillParams &p, cudaStream_t stream);

// CUDA-core kernel: rows = query rows per CTA (1, 2, 4 or 8); the cache type
// may be FP8 E4M3 with q of another type, else both types are equal.
int simt_max_rows(int head_dim);
bool simt_kernel_info(pkv_dtype cache_dtype, pkv_dtype q_dtype, int head_dim, int rows,
                      KernelInfo *info);
cudaError_t simt_launch(pkv_dtype cache_dtype, pkv_dtype q_dtype, int head_dim, int rows,
                        const AttnParams &p, dim3 grid, cudaStream_t stream);

// MLA decode (attn_mla.cu): latent width 512, rotary part rope_dim 0 or 64,
// bf16 / f16, 16 query heads per CTA; `stages` 3..5 (0: default).  The
// partials and the merge are those of the other decode kernels.
constexpr int kMlaLatent = 512;
constexpr int kMlaHeadsPerCta = 16;
bool mla_kernel_info(pkv_dtype dtype, int rope_dim, int stages, KernelInfo *info);
cudaError_t mla_launch(pkv_dtype dtype, int rope_dim, int stages, const CUtensorMap &cmap,
                       const AttnParams &p, dim3 grid, cudaStream_t stream);
// Zero n 32-bit split-K arrival counters; the attention launch that follows
// is its programmatic dependent.
cudaError_t zero_counters_launch(unsigned int *words, int64_t n, cudaStream_t stream);
// Split-K log-sum-exp merge.
// The MLA step's split-K merge (512-wide rows, [row][split] partials).
cudaError_t mla_merge_launch(pkv_dtype dtype, const AttnParams &p, cudaStream_t stream);
cudaError_t merge_launch(pkv_dtype dtype, int head_dim, const AttnParams &p, int sm_count,
                         cudaStream_t stream);

// kv_append into an FP8 E4M3 cache: src_dtype rows quantised with the
// tensor scales (x / scale, round to nearest even, saturating).
cudaError_t append_fp8_launch(pkv_dtype src_dtype, const void *k_new, const void *v_new,
                              void *k_cache, void *v_cache, const int64_t *slots,
                              int64_t num_tokens, int num_kv_heads, int head_dim, int block_size,
                              int64_t num_blocks, float k_scale, float v_scale, int32_t *err,
                              int sm_count, cudaStream_t stream);

// Whole-block copies (copy-on-write) in both caches.
cudaError_t copy_blocks_launch(void *k_cache, void *v_cache, const int32_t *src,
                               const int32_t *dst, int num_pairs, int64_t block_bytes,
                               int64_t num_blocks, int32_t *err, int sm_count,
                               cudaStream_t stream);

// Copies of mapped host buffers into device memory, in one launch (the
// kernel after it is its programmatic dependent).  Sizes are multiples of 4
// bytes, addresses 4-byte aligned.
constexpr int kMaxGather = 6;
struct GatherItem {
  const void *src;
  void *dst;
  int64_t bytes;
};
struct GatherList {
  GatherItem item[kMaxGather];
  int count;
};
cudaError_t gather_launch(const GatherList &list, int sm_count, cudaStream_t stream);

// kv_append.
cudaError_t append_launch(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                          const int64_t *slots, int64_t num_tokens, int num_kv_heads,
                          int vec_per_row, int block_size, int64_t num_blocks, int32_t *err,
                          int sm_count, cudaStream_t stream);

}  // namespace pkv
