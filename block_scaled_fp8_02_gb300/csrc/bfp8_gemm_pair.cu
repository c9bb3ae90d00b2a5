// bfp8_gemm_pair.cu -- the paired wide-tile instantiation of the blocked FP8
// GEMM (large M): CTA pairs computing 256 x 256 output tiles with 2-SM MMAs
// (kModePair in bfp8_gemm_kernel.cuh).  Kept apart so that the translation
// units build in parallel.
#include "bfp8_gemm_kernel.cuh"
#include "bfp8_internal.h"

namespace bfp8 {

cudaError_t launch_gemm_pair(const CUtensorMap& tmP, const CUtensorMap& tmQ, const GemmArgs& a,
                             cudaStream_t stream) {
  // whole tiles only: each pair computes its tiles alone
  if (a.sched.cluster > 1 || a.sched.sk_units != 0) return cudaErrorInvalidValue;
  return launch_instance<256, false, kModePair>(tmP, tmQ, a, stream);
}

int gemm_pair_stages() { return GemmCfg<256, false, kModePair>::kStages; }

}  // namespace bfp8
