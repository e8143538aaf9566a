// attn_simt_fp8.cu -- CUDA-core attention over FP8 E4M3 caches (one byte
// per element, one scale per cache tensor; "Inference part 2", section "KV
// cache quantization": FP8 halves the bytes read at each decode step).  The
// codes are widened to float32 in registers; the key scale is folded into the
// softmax scale and the value scale into the final output.  q and out are
// float32, bfloat16 or float16.  head_dim 128 or 256 (one row is a whole
// number of 128-byte lines).
#include "attn_simt.cuh"

namespace pkv {
namespace simt {

template <typename TQ>
bool pick_fp8_d(int D, int r, KernelInfo *info, SimtLaunch *launch) {
  switch (D) {
    case 128: return simt_pick<TQ, E4M3, 128>(r, info, launch);
    case 256: return simt_pick<TQ, E4M3, 256>(r, info, launch);
    default: return false;
  }
}

bool pick_fp8(pkv_dtype q_dtype, int D, int r, KernelInfo *info, SimtLaunch *launch) {
  switch (q_dtype) {
    case PKV_F32: return pick_fp8_d<float>(D, r, info, launch);
    case PKV_BF16: return pick_fp8_d<__nv_bfloat16>(D, r, info, launch);
    case PKV_F16: return pick_fp8_d<__half>(D, r, info, launch);
    default: return false;
  }
}

}  // namespace simt
}  // namespace pkv
