// kv_append.cu -- scatter the K/V rows of new tokens into their cache slots
// (the in-place write of a static KV cache, "Inference part 1", section "KV
// cache"; "Inference part 2", GPTlite_StaticCache; in paged form slot s is
// row s % block_size of physical block s / block_size, "KV cache, prefill va
// decode", section 05, "Block table").
//
// Pure data movement: one thread per 16-byte vector of a (token, kv head)
// row, for K and V; the copy is bit-exact.  Negative slots are padding and
// skipped; slots past the cache are skipped and reported in the error word.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                     uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                     const int64_t *__restrict__ slots, int64_t num_tokens, int num_kv_heads,
                     int vec_per_row, int block_size, int64_t num_blocks, int32_t *err) {
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
    v_cache[dst] = __ldg(v_new + src);
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
