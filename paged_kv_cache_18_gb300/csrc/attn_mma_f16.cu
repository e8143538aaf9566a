// attn_mma_f16.cu -- tensor-core attention over fp16 caches (q, cache and
// output fp16); the kernel is in attn_mma.cuh, the dispatch in attn_mma.cu.
#include "attn_mma.cuh"

namespace pkv {
namespace mma {

bool pick_f16(int D, int cg, int nt, int kb, int stages, KernelInfo *info, MmaLaunch *launch) {
  switch (D) {
    case 64: return mma_pick<__half, __half, 64>(cg, nt, kb, stages, info, launch);
    case 128: return mma_pick<__half, __half, 128>(cg, nt, kb, stages, info, launch);
    case 256: return mma_pick<__half, __half, 256>(cg, nt, kb, stages, info, launch);
    default: return false;
  }
}

}  // namespace mma
}  // namespace pkv
