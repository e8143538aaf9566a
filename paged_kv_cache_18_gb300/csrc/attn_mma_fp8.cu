// attn_mma_fp8.cu -- tensor-core attention over FP8 E4M3 caches with bf16 or
// fp16 queries ("Inference part 2", section "KV cache quantization": FP8
// halves the bytes read at each decode step).  Codes are widened exactly to
// f16 in registers and multiplied with f16 MMAs; the key scale is folded into
// the softmax scale, the value scale into the output.  head_dim 128 or 256.
#include "attn_mma.cuh"

namespace pkv {
namespace mma {

template <typename T>
bool pick_fp8_d(int D, int cg, int nt, int kb, int stages, KernelInfo *info, MmaLaunch *launch) {
  switch (D) {
    case 128: return mma_pick<T, E4M3, 128>(cg, nt, kb, stages, info, launch);
    case 256: return mma_pick<T, E4M3, 256>(cg, nt, kb, stages, info, launch);
    default: return false;
  }
}

bool pick_fp8(pkv_dtype q_dtype, int D, int cg, int nt, int kb, int stages, KernelInfo *info,
              MmaLaunch *launch) {
  if (q_dtype == PKV_BF16)
    return pick_fp8_d<__nv_bfloat16>(D, cg, nt, kb, stages, info, launch);
  if (q_dtype == PKV_F16) return pick_fp8_d<__half>(D, cg, nt, kb, stages, info, launch);
  return false;
}

}  // namespace mma
}  // namespace pkv
