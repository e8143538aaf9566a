// attn_merge.cu -- the Flash-Decoding reduction: merge the per-split partial
// outputs of one query row by their log-sum-exps ("Inference part 1",
// section "FlashDecoding": a final reduction combines the chunks with the
// rescaling of the online softmax; "KV cache, prefill va decode", section 07:
// each chunk keeps its log-sum-exp and the chunks are combined by the online
// softmax's rescaling).
//
// For split s of row r the attention kernel wrote O_s (already divided by
// its own sum) and lse_s = m_s + log2(l_s) in log2 units of the scaled
// scores.  Then with M = max_s lse_s:
//   out = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M).
// A split with no visible row has lse_s = -inf and weight 0; a row with no
// visible row at all gets zeros.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

template <typename T, int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const AttnParams p) {
  constexpr int PER = D / 32;  // elements per lane (2, 4 or 8)
  const int64_t nrows = static_cast<int64_t>(p.batch) * p.num_queries * p.num_heads;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= nrows) return;
  const int b = static_cast<int>(row / (static_cast<int64_t>(p.num_queries) * p.num_heads));
  const SeqExtent ext = seq_extent(p, b, false);
  int ns = (ext.nblk + p.split_blocks - 1) / p.split_blocks;
  ns = ns < 1 ? 1 : (ns > p.num_splits ? p.num_splits : ns);

  const float *lse = p.part_lse + row * p.num_splits;
  float M = -INFINITY;
  for (int s = lane; s < ns; s += 32) M = fmaxf(M, lse[s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));

  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    const float *po = p.part_o + row * p.num_splits * D + lane * PER;
    for (int s = 0; s < ns; ++s) {
      const float w = ex2(lse[s] - M);
      wsum += w;
#pragma unroll
      for (int e = 0; e < PER; e += 2) {
        const float2 v = *reinterpret_cast<const float2 *>(po + static_cast<int64_t>(s) * D + e);
        acc[e] = fmaf(w, v.x, acc[e]);
        acc[e + 1] = fmaf(w, v.y, acc[e + 1]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  T *dst = reinterpret_cast<T *>(p.out) + row * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; ++e) dst[e] = from_float<T>(acc[e] * inv);
}

template <typename T>
cudaError_t merge_t(int D, const AttnParams &p, cudaStream_t stream) {
  const int64_t nrows = static_cast<int64_t>(p.batch) * p.num_queries * p.num_heads;
  const int rows_per_cta = 8;
  const dim3 grid(static_cast<unsigned>((nrows + rows_per_cta - 1) / rows_per_cta));
  switch (D) {
    case 64: attn_merge_kernel<T, 64><<<grid, 256, 0, stream>>>(p); break;
    case 128: attn_merge_kernel<T, 128><<<grid, 256, 0, stream>>>(p); break;
    case 256: attn_merge_kernel<T, 256><<<grid, 256, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t merge_launch(pkv_dtype dtype, int head_dim, const AttnParams &p, int /*sm_count*/,
                         cudaStream_t stream) {
  switch (dtype) {
    case PKV_F32: return merge_t<float>(head_dim, p, stream);
    case PKV_BF16: return merge_t<__nv_bfloat16>(head_dim, p, stream);
    case PKV_F16: return merge_t<__half>(head_dim, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
