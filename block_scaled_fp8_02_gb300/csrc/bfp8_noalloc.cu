// bfp8_noalloc.cu -- bfp8_gemm_noalloc: the blocked FP8 GEMM with its scratch
// space built into the library, for callers that cannot allocate device
// memory themselves (see include/bfp8.h for who they are and the limits).
//
// The scratch is one file-scope device array.  Host code cannot use the
// array's name as a device address (on the host it is only a stand-in), so
// the real address is looked up once per device with cudaGetSymbolAddress,
// with that device current, and cached.  The cached address belongs to the
// device's context of that moment: after cudaDeviceReset() on a device, this
// entry point must not be called on it again in the same process.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/bfp8.h"
#include "bfp8_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = BFP8_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bfp8_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" bfp8_status bfp8_gemm_noalloc(const void* A, const void* B, const float* As,
                                         int as_col_major, int64_t ld_as, const float* Bs,
                                         void* out, int64_t M, int64_t N, int64_t K,
                                         void* stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return bfp8::set_last_error(BFP8_ERR_UNSUPPORTED, "bfp8_gemm_noalloc: no usable CUDA device");
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_bfp8_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return bfp8::set_last_error(BFP8_ERR_CUDA,
                                    "bfp8_gemm_noalloc: cudaGetSymbolAddress of the built-in scratch failed");
      }
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  const bool unaligned = (reinterpret_cast<uintptr_t>(A) % 16) != 0 ||
                         (reinterpret_cast<uintptr_t>(B) % 16) != 0;
  size_t need = 0;
  bfp8_status st = bfp8_gemm_workspace_size(M, N, K, nullptr, unaligned ? 1 : 0, &need);
  if (st != BFP8_OK) return st;
  if (need > kNoAllocScratchBytes)
    return bfp8::set_last_error(BFP8_ERR_WORKSPACE,
                                "bfp8_gemm_noalloc: this problem needs more scratch than the "
                                "built-in BFP8_NOALLOC_SCRATCH_BYTES; use bfp8_gemm with a caller "
                                "workspace instead");
  if (need > 0) {
    // The array keeps the previous call's contents; the stream-K counters at
    // its start must read zero when the kernel starts.
    const size_t clear = need < bfp8::kCounterHeaderBytes ? need : bfp8::kCounterHeaderBytes;
    if (cudaMemsetAsync(scratch, 0, clear, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
      cudaGetLastError();
      return bfp8::set_last_error(BFP8_ERR_CUDA, "bfp8_gemm_noalloc: clearing the scratch failed");
    }
  }
  return bfp8_gemm(A, B, As, as_col_major, ld_as, Bs, out, M, N, K, scratch, kNoAllocScratchBytes,
                   stream);
}
