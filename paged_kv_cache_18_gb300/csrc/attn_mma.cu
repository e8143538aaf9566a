// attn_mma.cu -- tensor-core attention over bf16 / fp16 caches (q, cache and
// output of one type); the kernel is in attn_mma.cuh.
#include "attn_mma.cuh"

namespace pkv {
namespace mma {

template <typename T>
bool pick_d(int D, int cg, int nt, int stages, KernelInfo *info, MmaLaunch *launch) {
  switch (D) {
    case 64: return mma_pick<T, T, 64>(cg, nt, stages, info, launch);
    case 128: return mma_pick<T, T, 128>(cg, nt, stages, info, launch);
    case 256: return mma_pick<T, T, 256>(cg, nt, stages, info, launch);
    default: return false;
  }
}

// FP8 caches (attn_mma_fp8.cu).
bool pick_fp8(pkv_dtype q_dtype, int D, int cg, int nt, int stages, KernelInfo *info,
              MmaLaunch *launch);

// n_tiles 8-column tiles, warp_tiles of them per warp (0: one).
bool pick(pkv_dtype cache_dtype, pkv_dtype q_dtype, int D, int n_tiles, int warp_tiles,
          int stages, KernelInfo *info, MmaLaunch *launch) {
  const int nt = warp_tiles > 0 ? warp_tiles : 1;
  if (nt > n_tiles && nt > 1) return false;
  const int cg = (n_tiles + nt - 1) / nt;
  if (cache_dtype == PKV_FP8_E4M3) return pick_fp8(q_dtype, D, cg, nt, stages, info, launch);
  if (q_dtype != cache_dtype) return false;
  if (cache_dtype == PKV_BF16) return pick_d<__nv_bfloat16>(D, cg, nt, stages, info, launch);
  if (cache_dtype == PKV_F16) return pick_d<__half>(D, cg, nt, stages, info, launch);
  return false;
}

}  // namespace mma

int mma_max_tiles(int head_dim) { return head_dim <= 64 ? 4 : (head_dim <= 128 ? 3 : 1); }

bool mma_kernel_info(pkv_dtype cache_dtype, pkv_dtype q_dtype, int head_dim, int n_tiles,
                     int warp_tiles, int stages, KernelInfo *info) {
  mma::MmaLaunch launch = nullptr;
  return mma::pick(cache_dtype, q_dtype, head_dim, n_tiles, warp_tiles, stages, info, &launch);
}

cudaError_t mma_launch(pkv_dtype cache_dtype, pkv_dtype q_dtype, int head_dim, int n_tiles,
                       int warp_tiles, int stages, const CUtensorMap &kmap,
                       const CUtensorMap &vmap, const AttnParams &p, dim3 grid,
                       cudaStream_t stream) {
  KernelInfo info;
  mma::MmaLaunch launch = nullptr;
  if (!mma::pick(cache_dtype, q_dtype, head_dim, n_tiles, warp_tiles, stages, &info, &launch))
    return cudaErrorInvalidValue;
  return launch(kmap, vmap, p, grid, stream);
}

}  // namespace pkv
