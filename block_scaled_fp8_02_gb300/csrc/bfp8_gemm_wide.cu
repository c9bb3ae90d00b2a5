// bfp8_gemm_wide.cu -- wide-tile instantiations of the blocked FP8 GEMM (large
// M: 128 activation rows fill the MMA M slot, BN = 128 or 256 weight rows the
// N slot) and the per-instantiation launch constants.
#include <atomic>

#include "bfp8_gemm_kernel.cuh"
#include "bfp8_internal.h"

namespace bfp8 {

namespace {

template <int BN, bool SWAP>
cudaError_t launch_one(const CUtensorMap& tmP, const CUtensorMap& tmQ, const GemmArgs& a,
                       cudaStream_t stream) {
  using C = GemmCfg<BN, SWAP>;
  // The shared-memory opt-in is per device; set it once (a launch captured
  // into a CUDA graph then needs no attribute call).
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemm_kernel<BN, SWAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  // programmatic dependent launch: the prologue may overlap the preceding
  // kernel; the kernel waits for it (griddepcontrol.wait) before reading inputs
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.sched.grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<BN, SWAP>, tmP, tmQ, a);
}

}  // namespace

cudaError_t launch_gemm_wide(int bn, const CUtensorMap& tmP, const CUtensorMap& tmQ,
                             const GemmArgs& a, cudaStream_t stream) {
  switch (bn) {
    case 128: return launch_one<128, false>(tmP, tmQ, a, stream);
    case 256: return launch_one<256, false>(tmP, tmQ, a, stream);
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

int gemm_stages(bool swap, int bn) { BFP8_CFG_CASES(kStages) }
int gemm_threads(bool swap, int bn) { BFP8_CFG_CASES(kThreads) }
size_t gemm_smem_bytes(bool swap, int bn) { BFP8_CFG_CASES(kSmemBytes) }

#undef BFP8_CFG_CASES

}  // namespace bfp8
