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
//
// One CTA per output row.  Long contexts give rows of many splits, so the
// loads are spread: warp w takes splits w, w + 4, ..., four at a time, which
// keeps 16 partial vectors in flight per row; the warps meet in shared
// memory at the end.
// The kernel is a programmatic dependent of the attention kernel: it may be
// scheduled while that kernel still runs (which hides its launch), reads
// only the call's inputs before pdl_wait, and the partials after it.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kMergeWarps = 4;
constexpr int kMergeUnroll = 4;

template <typename T, int D>
__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_kernel(const AttnParams p) {
  constexpr int PER = D / 32;  // elements per lane: 2, 4 or 8
  const int64_t row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = static_cast<int>(row / (static_cast<int64_t>(p.num_queries) * p.num_heads));
  const SeqExtent ext = seq_extent(p, b, false);
  int ns = (ext.nblk + p.split_blocks - 1) / p.split_blocks;
  ns = ns < 1 ? 1 : (ns > p.num_splits ? p.num_splits : ns);

  __shared__ float red_max[kMergeWarps];
  __shared__ float red_sum[kMergeWarps];
  __shared__ float red_acc[kMergeWarps][D];

  pdl_wait();  // the attention kernel's partials are complete and visible
  const float *lse = p.part_lse + row * p.num_splits;
  float M = -INFINITY;
  for (int s = threadIdx.x; s < ns; s += kMergeWarps * 32) M = fmaxf(M, lse[s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  if (lane == 0) red_max[warp] = M;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, red_max[w]);

  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    const float *po = p.part_o + row * p.num_splits * D + lane * PER;
    for (int s0 = warp; s0 < ns; s0 += kMergeWarps * kMergeUnroll) {
      float w[kMergeUnroll];
      float v[kMergeUnroll][PER];
#pragma unroll
      for (int u = 0; u < kMergeUnroll; ++u) {
        const int s = s0 + u * kMergeWarps;
        const bool ok = s < ns;
        w[u] = ok ? ex2(lse[ok ? s : 0] - M) : 0.f;
#pragma unroll
        for (int e = 0; e < PER; e += 2) {
          const float2 x = ok ? *reinterpret_cast<const float2 *>(po + static_cast<int64_t>(s) * D + e)
                              : make_float2(0.f, 0.f);
          v[u][e] = x.x;
          v[u][e + 1] = x.y;
        }
      }
#pragma unroll
      for (int u = 0; u < kMergeUnroll; ++u) {
        wsum += w[u];
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = fmaf(w[u], v[u][e], acc[e]);
      }
    }
  }
  if (lane == 0) red_sum[warp] = wsum;
#pragma unroll
  for (int e = 0; e < PER; ++e) red_acc[warp][lane * PER + e] = acc[e];
  __syncthreads();
  float total = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) total += red_sum[w];
  const float inv = total > 0.f ? p.out_scale / total : 0.f;
  T *dst = reinterpret_cast<T *>(p.out) + row * D;
  for (int d = threadIdx.x; d < D; d += kMergeWarps * 32) {
    float x = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) x += red_acc[w][d];
    dst[d] = from_float<T>(x * inv);
  }
}

template <typename T>
cudaError_t merge_t(int D, const AttnParams &p, cudaStream_t stream) {
  const int64_t nrows = static_cast<int64_t>(p.batch) * p.num_queries * p.num_heads;
  if (nrows == 0) return cudaSuccess;
  if (nrows > 0x7fffffffLL) return cudaErrorInvalidValue;
  void (*kernel)(const AttnParams);
  switch (D) {
    case 64: kernel = attn_merge_kernel<T, 64>; break;
    case 128: kernel = attn_merge_kernel<T, 128>; break;
    case 256: kernel = attn_merge_kernel<T, 256>; break;
    default: return cudaErrorInvalidValue;
  }
  // launched as a programmatic dependent of the attention kernel before it
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nrows));
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
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
