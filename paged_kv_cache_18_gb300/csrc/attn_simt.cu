// attn_simt.cu -- CUDA-core attention for float32, bfloat16 and float16
// caches (q, cache and output of one type); the kernel is in attn_simt.cuh.
#include "attn_simt.cuh"

namespace pkv {
namespace simt {

template <typename T>
bool pick_d(int D, int r, KernelInfo *info, SimtLaunch *launch) {
  switch (D) {
    case 64: return simt_pick<T, T, 64>(r, info, launch);
    case 128: return simt_pick<T, T, 128>(r, info, launch);
    case 256: return simt_pick<T, T, 256>(r, info, launch);
    default: return false;
  }
}

bool pick_same(pkv_dtype dt, int D, int r, KernelInfo *info, SimtLaunch *launch) {
  switch (dt) {
    case PKV_F32: return pick_d<float>(D, r, info, launch);
    case PKV_BF16: return pick_d<__nv_bfloat16>(D, r, info, launch);
    case PKV_F16: return pick_d<__half>(D, r, info, launch);
    default: return false;
  }
}

// FP8 caches (attn_simt_fp8.cu).
bool pick_fp8(pkv_dtype q_dtype, int D, int r, KernelInfo *info, SimtLaunch *launch);

bool pick(pkv_dtype cache_dtype, pkv_dtype q_dtype, int D, int r, KernelInfo *info,
          SimtLaunch *launch) {
  if (cache_dtype == PKV_FP8_E4M3) return pick_fp8(q_dtype, D, r, info, launch);
  if (q_dtype != cache_dtype) return false;
  return pick_same(cache_dtype, D, r, info, launch);
}

}  // namespace simt

int simt_max_rows(int head_dim) { return head_dim <= 64 ? 8 : (head_dim <= 128 ? 4 : 2); }

bool simt_kernel_info(pkv_dtype cache_dtype, pkv_dtype q_dtype, int head_dim, int rows,
                      KernelInfo *info) {
  simt::SimtLaunch launch = nullptr;
  return simt::pick(cache_dtype, q_dtype, head_dim, rows, info, &launch);
}

cudaError_t simt_launch(pkv_dtype cache_dtype, pkv_dtype q_dtype, int head_dim, int rows,
                        const AttnParams &p, dim3 grid, cudaStream_t stream) {
  KernelInfo info;
  simt::SimtLaunch launch = nullptr;
  if (!simt::pick(cache_dtype, q_dtype, head_dim, rows, &info, &launch))
    return cudaErrorInvalidValue;
  return launch(p, grid, stream);
}

}  // namespace pkv
