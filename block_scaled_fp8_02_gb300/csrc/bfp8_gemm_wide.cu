// bfp8_gemm_wide.cu -- wide-tile instantiations of the blocked FP8 GEMM (large
// M: 128 activation rows fill the MMA M slot, BN = 128 or 256 weight rows the
// N slot) and the per-instantiation launch constants.
#include "bfp8_gemm_kernel.cuh"
#include "bfp8_internal.h"

namespace bfp8 {

cudaError_t launch_gemm_wide(int bn, int mode, int mr, const CUtensorMap& tmP,
                             const CUtensorMap& tmQ, const GemmArgs& a, cudaStream_t stream) {
  if (mode != kModePlain) return launch_gemm_wide_ext(bn, mode, tmP, tmQ, a, stream);
  if (mr != 128) {
    if (bn != 256) return cudaErrorInvalidValue;
    return mr == 32 ? launch_instance<256, false, kModePlain, 32>(tmP, tmQ, a, stream)
         : mr == 64 ? launch_instance<256, false, kModePlain, 64>(tmP, tmQ, a, stream)
                    : cudaErrorInvalidValue;
  }
  switch (bn) {
    case 128: return launch_instance<128, false>(tmP, tmQ, a, stream);
    case 256: return launch_instance<256, false>(tmP, tmQ, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

#define BFP8_CFG_CASES(FIELD)                                                   \
  if (swap) {                                                                   \
    switch (bn) {                                                               \
      case 16: return GemmCfg<16, true>::FIELD;                                 \
      case 32: return GemmCfg<32, true>::FIELD;                                 \
      case 64: return GemmCfg<64, true>::FIELD;                                 \
      case 128: return GemmCfg<128, true>::FIELD;                               \
      case 256: return GemmCfg<256, true>::FIELD;                               \
      default: return 0;                                                        \
    }                                                                           \
  }                                                                             \
  switch (bn) {                                                                 \
    case 128: return GemmCfg<128, false>::FIELD;                                \
    case 256: return GemmCfg<256, false>::FIELD;                                \
    default: return 0;                                                          \
  }

int gemm_stages(bool swap, int bn, int mr) {
  if (!swap && bn == 256 && mr == 32) return GemmCfg<256, false, kModePlain, 32>::kStages;
  if (!swap && bn == 256 && mr == 64) return GemmCfg<256, false, kModePlain, 64>::kStages;
  BFP8_CFG_CASES(kStages)
}
int gemm_threads(bool swap, int bn) { BFP8_CFG_CASES(kThreads) }
size_t gemm_smem_bytes(bool swap, int bn) { BFP8_CFG_CASES(kSmemBytes) }

#undef BFP8_CFG_CASES

}  // namespace bfp8
