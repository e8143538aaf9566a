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
// One CTA per output row, four warps.  Warp w merges splits w, w + 4, ...
// on its own, eight at a time (two for 512-wide rows): the log-sum-exps and
// partial vectors of a group are loaded together (one memory round trip per
// group; up to 32 splits are one group per warp), against the warp's own
// maximum M_w:
//   acc_w = sum_s 2^(lse_s - M_w) O_s,   l_w = sum_s 2^(lse_s - M_w).
// The warps then meet in shared memory: with M = max_w M_w,
//   out = sum_w 2^(M_w - M) acc_w / sum_w 2^(M_w - M) l_w.
// The kernel is a programmatic dependent of the attention kernel: it may be
// scheduled while that kernel still runs (which hides its launch) and reads
// nothing from global memory before pdl_wait.
#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kMergeWarps = 4;

// Splits a warp loads at once: eight (up to 32 splits in one round trip),
// two for the 512-wide latent rows of MLA (register budget).
template <int D> __host__ __device__ constexpr int merge_unroll() { return D <= 256 ? 8 : 2; }

// Where the partials of output row `row` are: split s at
// part_lse[first + s * stride] and part_o[(first + s * stride) * D ..], for
// s < ns.  LAYOUT 0: the host partition's partials, [row][split]; 1: the
// device partition's, [item][CTA column]; 2: the balanced partition's,
// [slot][CTA column] (sk_begin in pkv_device.cuh), where split s (CTA
// sk_c0 + s) holds nothing when that CTA's range is empty.  A device layout
// that cannot be the attention kernel's (never, unless that kernel did not
// publish it) is recorded (`report`) and merged as no split at all rather
// than read outside the workspace.
struct RowSplits {
  int ns, stride, sk_c0;
  int64_t first, sk_total;
};
template <int LAYOUT>
__device__ __forceinline__ RowSplits row_splits(const AttnParams &p, int64_t row, bool report) {
  RowSplits o{0, 1, 0, 0, 0};
  const int b = static_cast<int>(row / (static_cast<int64_t>(p.num_queries) * p.num_heads));
  if constexpr (LAYOUT == 0) {  // host partition: [row][split]
    const SeqExtent ext = seq_extent(p, b, false);
    int ns = (ext.nblk + p.split_blocks - 1) / p.split_blocks;
    o.ns = ns < 1 ? 1 : (ns > p.num_splits ? p.num_splits : ns);
    o.first = row * p.num_splits;
    o.stride = 1;
    return o;
  }
  const int units = p.num_kv_heads * p.row_chunks;
  const int h = static_cast<int>(row % p.num_heads);
  const int j = static_cast<int>((row / p.num_heads) % p.num_queries);
  const int kvh = h / p.group;
  const int r = j * p.group + (h - kvh * p.group);  // row within its KV head's rows
  const int chunk = r / p.rows_per_cta;
  const int u = kvh * p.row_chunks + chunk;
  const int col = r - chunk * p.rows_per_cta;
  o.stride = p.rows_per_cta;
  if constexpr (LAYOUT == 2) {  // balanced partition: [slot][CTA column]
    const int64_t s_b = p.split_info[2 * b], nb = p.split_info[2 * b + 1];
    const int64_t total = p.split_info[2 * p.batch];
    const int G = p.split_target;
    const int64_t vlen = nb > 0 ? nb + p.sk_weight : 0;  // places of each unit of b
    if (s_b < 0 || nb < 0 || total < 0 || s_b + vlen * units > total) {
      if (report) record_error(p.err, PKV_DEVERR_CONTEXT_LEN);
    } else if (nb > 0) {  // (a sequence without blocks gets zeros)
      // the unit's blocks (places s_u .. s_u + nb - 1) lie in CTAs c0 .. c1,
      // its splits in slots c0 + U .. c1 + U
      const int64_t s_u = s_b + static_cast<int64_t>(u) * vlen + p.sk_weight;
      const int c0 = sk_cta_of(total, G, s_u), c1 = sk_cta_of(total, G, s_u + nb - 1);
      const int64_t U = static_cast<int64_t>(b) * units + u;
      o.ns = c1 - c0 + 1;
      o.first = (c0 + U) * p.rows_per_cta + col;
      o.sk_c0 = c0;
      o.sk_total = total;
    }
  } else {  // device partition: [item][CTA column], the items of (b, unit) consecutive
    int ns = p.split_info[2 * b];
    int item0 = p.split_info[2 * b + 1];
    if (ns < 1 || item0 < 0 ||
        static_cast<int64_t>(item0) + static_cast<int64_t>(ns) * units > p.split_target) {
      if (report) record_error(p.err, PKV_DEVERR_CONTEXT_LEN);
      ns = 0;
      item0 = 0;
    }
    o.ns = ns;
    o.first = (static_cast<int64_t>(item0) + static_cast<int64_t>(u) * ns) * p.rows_per_cta + col;
  }
  return o;
}
// Split s of a row holds a partial (LAYOUT 2: its CTA's range is not empty).
template <int LAYOUT>
__device__ __forceinline__ bool split_present(const AttnParams &p, const RowSplits &rs, int s) {
  if constexpr (LAYOUT == 2)
    return sk_begin(rs.sk_total, p.split_target, rs.sk_c0 + s) <
           sk_begin(rs.sk_total, p.split_target, rs.sk_c0 + s + 1);
  return true;
}

// One CTA per row, four warps sharing its splits (many splits, few rows).
template <typename T, int D, int LAYOUT>
__global__ void __launch_bounds__(kMergeWarps * 32, (D <= 128 ? (LAYOUT ? 6 : 8) : 4))
    attn_merge_kernel(const AttnParams p) {
  constexpr int PER = D / 32;  // elements per lane: 2, 4, 8 or 16
  constexpr int kMergeUnroll = merge_unroll<D>();
  const int64_t row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The next kernel in the stream (the next call's, itself waiting before it
  // touches memory) may be scheduled from here on.  The attention kernel's
  // partials are complete and visible after the wait, and so is everything
  // enqueued before the attention kernel (which may itself have started
  // early, as a programmatic dependent): the context lengths are read only
  // after it.
  pdl_launch_dependents();
  pdl_wait();
  const RowSplits rs = row_splits<LAYOUT>(p, row, threadIdx.x == 0);
  const int ns = rs.ns, stride = rs.stride;
  const int64_t first = rs.first;

  __shared__ float red_max[kMergeWarps];
  __shared__ float red_sum[kMergeWarps];
  __shared__ float red_acc[kMergeWarps][D];

  const float *lse = p.part_lse + first;
  const float *po = p.part_o + first * D + lane * PER;
  float Mw = -INFINITY, wsum = 0.f;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int s0 = warp; s0 < ns; s0 += kMergeWarps * kMergeUnroll) {
    float ls[kMergeUnroll];
    float v[kMergeUnroll][PER];
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const int s = s0 + u * kMergeWarps;
      const bool ok = s < ns && split_present<LAYOUT>(p, rs, s);
      const int off = LAYOUT ? s * stride : s;  // < splits x rows per CTA: fits an int
      ls[u] = ok ? lse[off] : -INFINITY;
#pragma unroll
      for (int e = 0; e < PER; e += 2) {
        const float2 x = ok ? *reinterpret_cast<const float2 *>(po + off * D + e)
                            : make_float2(0.f, 0.f);
        v[u][e] = x.x;
        v[u][e + 1] = x.y;
      }
    }
    float mg = Mw;
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) mg = fmaxf(mg, ls[u]);
    if (mg == -INFINITY) continue;  // nothing visible in these splits yet
    const float r = ex2(Mw - mg);   // rescale what the warp holds (0 while it holds nothing)
    wsum *= r;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] *= r;
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const float w = ex2(ls[u] - mg);  // 0 for empty or absent splits
      wsum += w;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
    }
    Mw = mg;
  }
  if (lane == 0) {
    red_max[warp] = Mw;
    red_sum[warp] = wsum;
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) red_acc[warp][lane * PER + e] = acc[e];
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, red_max[w]);
  float f[kMergeWarps];
  float total = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) {
    f[w] = red_max[w] == -INFINITY ? 0.f : ex2(red_max[w] - M);
    total += f[w] * red_sum[w];
  }
  const float inv = total > 0.f ? p.out_scale / total : 0.f;
  T *dst = reinterpret_cast<T *>(p.out) + row * D;
  for (int d = threadIdx.x; d < D; d += kMergeWarps * 32) {
    float x = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) x = fmaf(f[w], red_acc[w][d], x);
    dst[d] = from_float<T>(x * inv);
  }
}

// One warp per row, kRowsPerCta rows a CTA (many rows, few splits: the
// speculative-verify and tree steps' thousands of rows): every row in one
// wave, no block-wide barrier.  The warp takes the row's log-sum-exps 32 at
// a time (lane s the split s), their maximum M and weights 2^(lse_s - M) by
// shuffles, then each lane accumulates its PER head dims over the splits,
// eight partial vectors in flight at once.
constexpr int kRowsPerCta = 8;
// Rows from which the warp-per-row kernel is used: with fewer, the rows are
// few CTAs' worth of warps, and a row's many splits (long contexts) go
// faster spread over the four warps of attn_merge_kernel.  The host plan's
// rows with more than 8 splits (the mma.sync verify step's 22) keep that
// kernel too: their step measured no faster with this one (76.6 against
// 75.2 us), while the device partitions' few splits a row gained (the
// tcgen05 verify step's merge from 13 to 5.5 us).
constexpr int64_t kMinRowsForRowKernel = 1024;
constexpr int kMaxSplitsForRowKernel = 8;
template <typename T, int D, int LAYOUT>
__global__ void __launch_bounds__(kRowsPerCta * 32)
    attn_merge_rows_kernel(const AttnParams p, int64_t nrows) {
  constexpr int PER = D / 32;  // 4 or 8: whole float4 loads
  static_assert(D == 128 || D == 256, "head_dim 128 or 256");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + warp;
  pdl_launch_dependents();  // as in attn_merge_kernel
  pdl_wait();
  if (row >= nrows) return;
  const RowSplits rs = row_splits<LAYOUT>(p, row, lane == 0);
  auto lse_of = [&](int s) -> float {
    return s < rs.ns && split_present<LAYOUT>(p, rs, s)
               ? __ldcg(p.part_lse + rs.first + static_cast<int64_t>(s) * rs.stride)
               : -INFINITY;
  };
  const float l0 = lse_of(lane);  // the first 32 splits (all of them, nearly always)
  float M = l0;
  for (int s0 = 32; s0 < rs.ns; s0 += 32) M = fmaxf(M, lse_of(s0 + lane));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < rs.ns; s0 += 32) {
      const float l = s0 == 0 ? l0 : lse_of(s0 + lane);
      const float w_mine = ex2(l - M);  // 0 for an empty or absent split
      wsum += w_mine;
      const int n = min(32, rs.ns - s0);
      for (int t0 = 0; t0 < n; t0 += 8) {
        float v[8][PER];
        float w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          w[u] = __shfl_sync(kFull, w_mine, (t0 + u) & 31);
          const bool ld = t0 + u < n && w[u] > 0.f;
          const float *src = p.part_o +
                             (rs.first + static_cast<int64_t>(s0 + t0 + u) * rs.stride) * D +
                             lane * PER;
#pragma unroll
          for (int e = 0; e < PER; e += 4) {
            const float4 x = ld ? __ldcg(reinterpret_cast<const float4 *>(src + e))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            v[u][e] = x.x;
            v[u][e + 1] = x.y;
            v[u][e + 2] = x.z;
            v[u][e + 3] = x.w;
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[e] = fmaf(t0 + u < n ? w[u] : 0.f, v[u][e], acc[e]);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(kFull, wsum, o);
  const float inv = wsum > 0.f ? p.out_scale / wsum : 0.f;
  T *dst = reinterpret_cast<T *>(p.out) + row * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; ++e) dst[e] = from_float<T>(acc[e] * inv);
}

template <typename T>
cudaError_t merge_t(int D, const AttnParams &p, cudaStream_t stream) {
  const int64_t nrows = static_cast<int64_t>(p.batch) * p.num_queries * p.num_heads;
  if (nrows == 0) return cudaSuccess;
  if (nrows > 0x7fffffffLL) return cudaErrorInvalidValue;
  void (*kernel)(const AttnParams);
  const int layout = p.split_target == 0 ? 0 : (p.stream_k ? 2 : 1);
  void (*const k64[3])(const AttnParams) = {attn_merge_kernel<T, 64, 0>,
                                            attn_merge_kernel<T, 64, 1>,
                                            attn_merge_kernel<T, 64, 2>};
  void (*const k128[3])(const AttnParams) = {attn_merge_kernel<T, 128, 0>,
                                             attn_merge_kernel<T, 128, 1>,
                                             attn_merge_kernel<T, 128, 2>};
  void (*const k256[3])(const AttnParams) = {attn_merge_kernel<T, 256, 0>,
                                             attn_merge_kernel<T, 256, 1>,
                                             attn_merge_kernel<T, 256, 2>};
  switch (D) {
    case 64: kernel = k64[layout]; break;
    case 128: kernel = k128[layout]; break;
    case 256: kernel = k256[layout]; break;
    case 512:  // MLA: host partition
      if (layout != 0) return cudaErrorInvalidValue;
      kernel = attn_merge_kernel<T, 512, 0>;
      break;
    default: return cudaErrorInvalidValue;
  }
  // launched as a programmatic dependent of the attention kernel before it
  if ((D == 128 || D == 256) && nrows >= kMinRowsForRowKernel &&
      (layout != 0 || p.num_splits <= kMaxSplitsForRowKernel)) {
    void (*const r128[3])(const AttnParams, int64_t) = {attn_merge_rows_kernel<T, 128, 0>,
                                                        attn_merge_rows_kernel<T, 128, 1>,
                                                        attn_merge_rows_kernel<T, 128, 2>};
    void (*const r256[3])(const AttnParams, int64_t) = {attn_merge_rows_kernel<T, 256, 0>,
                                                        attn_merge_rows_kernel<T, 256, 1>,
                                                        attn_merge_rows_kernel<T, 256, 2>};
    return launch_kernel(true, D == 128 ? r128[layout] : r256[layout],
                         dim3(static_cast<unsigned>((nrows + kRowsPerCta - 1) / kRowsPerCta)),
                         kRowsPerCta * 32, 0, stream, p, nrows);
  }
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

// Zero the split-K arrival counters of one call.  The attention kernel is
// launched right after it as its programmatic dependent, so that kernel's
// launch and main loop overlap this one; it waits for it (pdl_wait) only
// before its first arrival.
__global__ void __launch_bounds__(256) zero_words_kernel(unsigned int *words, int n) {
  pdl_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    words[i] = 0u;
}

}  // namespace

cudaError_t zero_counters_launch(unsigned int *words, int64_t n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  if (n > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int ctas = static_cast<int>(std::min<int64_t>((n + 255) / 256, 64));
  zero_words_kernel<<<ctas, 256, 0, stream>>>(words, static_cast<int>(n));
  return cudaGetLastError();
}

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
