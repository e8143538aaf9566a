// attn_mma.cu -- tensor-core attention over bf16 caches (q, cache and output
// bf16), and the dispatch over every tensor-core instantiation; the kernel is
// in attn_mma.cuh.
#include "attn_mma.cuh"

namespace pkv {
namespace mma {

bool pick_bf16(int D, int cg, int nt, int kb, int stages, KernelInfo *info, MmaLaunch *launch) {
  switch (D) {
    case 64: return mma_pick<__nv_bfloat16, __nv_bfloat16, 64>(cg, nt, kb, stages, info, launch);
    case 128: return mma_pick<__nv_bfloat16, __nv_bfloat16, 128>(cg, nt, kb, stages, info, launch);
    case 256: return mma_pick<__nv_bfloat16, __nv_bfloat16, 256>(cg, nt, kb, stages, info, launch);
    default: return false;
  }
}

// fp16 caches (attn_mma_f16.cu) and FP8 caches (attn_mma_fp8.cu).
bool pick_f16(int D, int cg, int nt, int kb, int stages, KernelInfo *info, MmaLaunch *launch);
bool pick_fp8(pkv_dtype q_dtype, int D, int cg, int nt, int kb, int stages, KernelInfo *info,
              MmaLaunch *launch);

bool pick(pkv_dtype cache_dtype, pkv_dtype q_dtype, int D, const MmaShape &m, KernelInfo *info,
          MmaLaunch *launch) {
  const int nt = m.warp_tiles > 0 ? m.warp_tiles : 1;
  if (nt > m.n_tiles && nt > 1) return false;
  const int cg = (m.n_tiles + nt - 1) / nt;
  const int kb = m.blocks_per_iter > 0 ? m.blocks_per_iter : 1;
  if (cache_dtype == PKV_FP8_E4M3)
    return pick_fp8(q_dtype, D, cg, nt, kb, m.stages, info, launch);
  if (q_dtype != cache_dtype) return false;
  if (cache_dtype == PKV_BF16) return pick_bf16(D, cg, nt, kb, m.stages, info, launch);
  if (cache_dtype == PKV_F16) return pick_f16(D, cg, nt, kb, m.stages, info, launch);
  return false;
}

}  // namespace mma

int mma_max_tiles(int head_dim) { return head_dim <= 128 ? 5 : 1; }

bool mma_kernel_info(pkv_dtype cache_dtype, pkv_dtype q_dtype, int head_dim, const MmaShape &m,
                     KernelInfo *info) {
  mma::MmaLaunch launch = nullptr;
  return mma::pick(cache_dtype, q_dtype, head_dim, m, info, &launch);
}

cudaError_t mma_launch(pkv_dtype cache_dtype, pkv_dtype q_dtype, int head_dim, const MmaShape &m,
                       const CUtensorMap &kmap, const CUtensorMap &vmap, const AttnParams &p,
                       dim3 grid, cudaStream_t stream) {
  KernelInfo info;
  mma::MmaLaunch launch = nullptr;
  if (!mma::pick(cache_dtype, q_dtype, head_dim, m, &info, &launch)) return cudaErrorInvalidValue;
  return launch(kmap, vmap, p, grid, stream);
}

}  // namespace pkv
