// bfp8_gemm_ext.cu -- wide-tile instantiations of the blocked FP8 GEMM's
// variants: the M-grouped (mixture-of-experts) GEMM and the GEMM with the
// fused epilogue (bias add and next-layer group quantisation).  Kept apart
// from the plain instantiations so that the translation units build in
// parallel.
#include "bfp8_gemm_kernel.cuh"
#include "bfp8_internal.h"

namespace bfp8 {

cudaError_t launch_gemm_wide_ext(int bn, int mode, const CUtensorMap& tmP, const CUtensorMap& tmQ,
                                 const GemmArgs& a, cudaStream_t stream) {
  if (mode == kModeGrouped) {
    switch (bn) {
      case 128: return launch_instance<128, false, kModeGrouped>(tmP, tmQ, a, stream);
      case 256: return launch_instance<256, false, kModeGrouped>(tmP, tmQ, a, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (mode == kModeFused) {
    switch (bn) {
      case 128: return launch_instance<128, false, kModeFused>(tmP, tmQ, a, stream);
      case 256: return launch_instance<256, false, kModeFused>(tmP, tmQ, a, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace bfp8
