// kv_append.cu -- scatter the K/V rows of new tokens into their cache slots
// (the in-place write of a static KV cache, "Inference part 1", section "KV
// cache"; "Inference part 2", GPTlite_StaticCache; in paged form slot s is
// row s % block_size of physical block s / block_size, "KV cache, prefill va
// decode", section 05, "Block table").
//
// Pure data movement: one thread per 16-byte vector of a (token, kv head)
// row, for K and V (K only when no V cache is given: the single latent cache
// of MLA); the copy is bit-exact.  Negative slots are padding and skipped;
// slots past the cache are skipped and reported in the error word.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                     uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                     const int64_t *__restrict__ slots, int64_t num_tokens, int num_kv_heads,
                     int vec_per_row, int block_size, int64_t num_blocks, int32_t *err) {
  // An attention kernel launched next (a programmatic dependent) may be
  // scheduled now; it waits for this grid before it reads the cache.
  pdl_launch_dependents();
  const int64_t per_token = static_cast<int64_t>(num_kv_heads) * vec_per_row;
  const int64_t total = num_tokens * per_token;
  const int64_t capacity = num_blocks * block_size;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = idx / per_token;
    const int64_t rem = idx - t * per_token;
    const int h = static_cast<int>(rem / vec_per_row);
    const int v = static_cast<int>(rem - static_cast<int64_t>(h) * vec_per_row);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= capacity) {
      if (rem == 0) record_error(err, PKV_DEVERR_SLOT);
      continue;
    }
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * vec_per_row + v;
    const int64_t src = (t * num_kv_heads + h) * vec_per_row + v;
    k_cache[dst] = __ldg(k_new + src);
    if (v_cache != nullptr) v_cache[dst] = __ldg(v_new + src);
  }
}

}  // namespace

cudaError_t append_launch(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                          const int64_t *slots, int64_t num_tokens, int num_kv_heads,
                          int vec_per_row, int block_size, int64_t num_blocks, int32_t *err,
                          int sm_count, cudaStream_t stream) {
  const int64_t total = num_tokens * num_kv_heads * static_cast<int64_t>(vec_per_row);
  if (total == 0) return cudaSuccess;
  int64_t ctas = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  if (ctas > cap) ctas = cap;
  kv_append_kernel<<<static_cast<unsigned>(ctas), 256, 0, stream>>>(
      reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new),
      reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache), slots, num_tokens,
      num_kv_heads, vec_per_row, block_size, num_blocks, err);
  return cudaGetLastError();
}

}  // namespace pkv

// ---- FP8 E4M3 caches ------------------------------------------------------
// Quantised append ("Inference part 2", section "KV cache quantization": the
// cache is stored in FP8): each element becomes the e4m3 code nearest to
// x / scale (IEEE float32 division, round to nearest even, saturating at
// +-448).  One thread per 16 elements (one 16-byte store).
#include <cuda_fp8.h>

namespace pkv {
namespace {

template <typename TS> __device__ __forceinline__ float src_float(const TS *p, int64_t i);
template <> __device__ __forceinline__ float src_float<float>(const float *p, int64_t i) {
  return p[i];
}
template <> __device__ __forceinline__ float src_float<__nv_bfloat16>(const __nv_bfloat16 *p,
                                                                     int64_t i) {
  return __bfloat162float(p[i]);
}
template <> __device__ __forceinline__ float src_float<__half>(const __half *p, int64_t i) {
  return __half2float(p[i]);
}

template <typename TS>
__device__ __forceinline__ uint4 quantise16(const TS *src, int64_t base, float scale) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t word = 0;
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      const int64_t e = base + k * 4 + pr * 2;
      const float2 f = make_float2(__fdiv_rn(src_float<TS>(src, e), scale),
                                   __fdiv_rn(src_float<TS>(src, e + 1), scale));
      const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      word |= static_cast<uint32_t>(c) << (16 * pr);
    }
    w[k] = word;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename TS>
__global__ void __launch_bounds__(256)
    kv_append_fp8_kernel(const TS *__restrict__ k_new, const TS *__restrict__ v_new,
                         uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                         const int64_t *__restrict__ slots, int64_t num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int64_t num_blocks, float k_scale,
                         float v_scale, int32_t *err) {
  pdl_launch_dependents();  // as in kv_append_kernel
  const int vpr = head_dim / 16;  // 16-byte code vectors per row
  const int64_t per_token = static_cast<int64_t>(num_kv_heads) * vpr;
  const int64_t total = num_tokens * per_token;
  const int64_t capacity = num_blocks * block_size;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = idx / per_token;
    const int64_t rem = idx - t * per_token;
    const int h = static_cast<int>(rem / vpr);
    const int v = static_cast<int>(rem - static_cast<int64_t>(h) * vpr);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= capacity) {
      if (rem == 0) record_error(err, PKV_DEVERR_SLOT);
      continue;
    }
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    const int64_t src = ((t * num_kv_heads + h) * head_dim) + v * 16;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * vpr + v;
    k_cache[dst] = quantise16<TS>(k_new, src, k_scale);
    v_cache[dst] = quantise16<TS>(v_new, src, v_scale);
  }
}

template <typename TS>
cudaError_t append_fp8_t(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                         const int64_t *slots, int64_t num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int64_t num_blocks, float k_scale,
                         float v_scale, int32_t *err, int sm_count, cudaStream_t stream) {
  const int64_t total = num_tokens * num_kv_heads * static_cast<int64_t>(head_dim / 16);
  if (total == 0) return cudaSuccess;
  int64_t ctas = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  if (ctas > cap) ctas = cap;
  kv_append_fp8_kernel<TS><<<static_cast<unsigned>(ctas), 256, 0, stream>>>(
      static_cast<const TS *>(k_new), static_cast<const TS *>(v_new),
      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slots, num_tokens,
      num_kv_heads, head_dim, block_size, num_blocks, k_scale, v_scale, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t append_fp8_launch(pkv_dtype src_dtype, const void *k_new, const void *v_new,
                              void *k_cache, void *v_cache, const int64_t *slots,
                              int64_t num_tokens, int num_kv_heads, int head_dim, int block_size,
                              int64_t num_blocks, float k_scale, float v_scale, int32_t *err,
                              int sm_count, cudaStream_t stream) {
  switch (src_dtype) {
    case PKV_F32:
      return append_fp8_t<float>(k_new, v_new, k_cache, v_cache, slots, num_tokens, num_kv_heads,
                                 head_dim, block_size, num_blocks, k_scale, v_scale, err,
                                 sm_count, stream);
    case PKV_BF16:
      return append_fp8_t<__nv_bfloat16>(k_new, v_new, k_cache, v_cache, slots, num_tokens,
                                         num_kv_heads, head_dim, block_size, num_blocks, k_scale,
                                         v_scale, err, sm_count, stream);
    case PKV_F16:
      return append_fp8_t<__half>(k_new, v_new, k_cache, v_cache, slots, num_tokens, num_kv_heads,
                                  head_dim, block_size, num_blocks, k_scale, v_scale, err,
                                  sm_count, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv

// ---- copy_blocks: whole physical blocks, for copy-on-write ------------------
// ("KV cache, prefill và decode", section 05, "Chia sẻ block và
// copy-on-write": a shared block is copied to a fresh one before a sequence
// writes into it.)  One block of one cache is num_kv_heads x block_size x
// head_dim elements, contiguous; pair i copies block src[i] to dst[i] in both
// caches.  Out-of-range ids are skipped and recorded.
namespace pkv {
namespace {

__global__ void copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                   const int32_t *__restrict__ src,
                                   const int32_t *__restrict__ dst, int num_pairs,
                                   int64_t vec_per_block, int64_t num_blocks, int32_t *err) {
  const int64_t total = static_cast<int64_t>(num_pairs) * vec_per_block;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int pair = static_cast<int>(i / vec_per_block);
    const int64_t off = i - static_cast<int64_t>(pair) * vec_per_block;
    const int32_t s = __ldg(src + pair), d = __ldg(dst + pair);
    if (s < 0 || d < 0 || s >= num_blocks || d >= num_blocks) {
      if (off == 0) record_error(err, PKV_DEVERR_BLOCK_ID);
      continue;
    }
    k_cache[d * vec_per_block + off] = k_cache[s * vec_per_block + off];
    v_cache[d * vec_per_block + off] = v_cache[s * vec_per_block + off];
  }
}

}  // namespace

cudaError_t copy_blocks_launch(void *k_cache, void *v_cache, const int32_t *src,
                               const int32_t *dst, int num_pairs, int64_t block_bytes,
                               int64_t num_blocks, int32_t *err, int sm_count,
                               cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int64_t vpb = block_bytes / 16;
  const int64_t total = static_cast<int64_t>(num_pairs) * vpb;
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int grid = static_cast<int>(want < 8LL * sm_count ? want : 8LL * sm_count);
  copy_blocks_kernel<<<grid, threads, 0, stream>>>(static_cast<uint4 *>(k_cache),
                                                  static_cast<uint4 *>(v_cache), src, dst,
                                                  num_pairs, vpb, num_blocks, err);
  return cudaGetLastError();
}

}  // namespace pkv

// ---- host inputs gathered into device memory ---------------------------------
// One launch copies up to kMaxGather buffers from mapped page-locked host
// memory (reached over the chip-to-chip link) into device memory: every CTA
// walks all of them in 16-byte vectors (4-byte words for a buffer whose
// addresses or size are not multiples of 16), so the link sees many requests
// in flight at once.  The kernel that follows is its programmatic dependent.
namespace pkv {
namespace {

__global__ void __launch_bounds__(256) gather_kernel(const GatherList list) {
  pdl_launch_dependents();
  // All buffers' units (16-byte vectors of the wide ones, 4-byte words of the
  // others) form one index space, so every thread's loads are independent
  // and one round trip over the link serves the whole gather.
  int64_t first[kMaxGather + 1];
  bool wide[kMaxGather];
  first[0] = 0;
#pragma unroll
  for (int k = 0; k < kMaxGather; ++k) {
    const GatherItem &g = list.item[k];
    wide[k] = ((reinterpret_cast<uintptr_t>(g.src) | reinterpret_cast<uintptr_t>(g.dst) |
                static_cast<uintptr_t>(g.bytes)) & 15) == 0;
    first[k + 1] = first[k] + (k < list.count ? g.bytes / (wide[k] ? 16 : 4) : 0);
  }
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < first[list.count]; i += nthr) {
    int k = 0;
    while (i >= first[k + 1]) ++k;
    const int64_t j = i - first[k];
    const GatherItem &g = list.item[k];
    if (wide[k]) {
      static_cast<uint4 *>(g.dst)[j] = static_cast<const uint4 *>(g.src)[j];
    } else {
      static_cast<uint32_t *>(g.dst)[j] = static_cast<const uint32_t *>(g.src)[j];
    }
  }
}

}  // namespace

cudaError_t gather_launch(const GatherList &list, int sm_count, cudaStream_t stream) {
  if (list.count < 1 || list.count > kMaxGather) return list.count == 0 ? cudaSuccess
                                                                        : cudaErrorInvalidValue;
  int64_t units = 0;  // an upper bound: every buffer in 4-byte words
  for (int k = 0; k < list.count; ++k) units += list.item[k].bytes / 4;
  if (units == 0) return cudaSuccess;
  const int64_t want = (units + 255) / 256;
  const int grid = static_cast<int>(want < 4LL * sm_count ? want : 4LL * sm_count);
  gather_kernel<<<grid, 256, 0, stream>>>(list);
  return cudaGetLastError();
}

}  // namespace pkv

// ---- the bounded wait, exercised ---------------------------------------------
// Every wait of the library's kernels on an mbarrier gives up after a time
// limit, records PKV_DEVERR_TIMEOUT and lets the kernel return.  This kernel
// waits on a barrier that nothing ever arrives on, through the same wait
// loop with a caller-chosen limit, so the give-up path can be checked on a
// GPU without hanging or faulting it.
namespace pkv {
namespace {

__global__ void bounded_wait_kernel(int32_t *err, unsigned long long limit_ns,
                                    unsigned long long *waited_ns) {
  __shared__ uint64_t never;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&never), 1);
  fence_mbar_init();
  const unsigned long long t0 = global_ns();
  if (!mbar_wait_bounded_ns(smem_u32(&never), 0, limit_ns)) record_error(err, PKV_DEVERR_TIMEOUT);
  if (waited_ns) *waited_ns = global_ns() - t0;
}

}  // namespace

cudaError_t bounded_wait_launch(int32_t *err, unsigned long long limit_ns,
                                unsigned long long *waited_ns, cudaStream_t stream) {
  bounded_wait_kernel<<<1, 32, 0, stream>>>(err, limit_ns, waited_ns);
  return cudaGetLastError();
}

}  // namespace pkv
