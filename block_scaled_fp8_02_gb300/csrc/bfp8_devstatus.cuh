// bfp8_devstatus.cuh -- the device-side failure word shared by the kernels
// that wait on barriers (bounded waits report here instead of hanging).
#pragma once

namespace bfp8 {

// Device-side failure codes (the first failure of a launch wins); the same
// values as BFP8_DEV_* in the public header.
enum : int {
  kDevOk = 0,
  kDevTimeoutProducer = 1,
  kDevTimeoutMma = 2,
  kDevTimeoutEpilogue = 3,
  kDevTimeoutTail = 4,
  kDevBadGroupedLayout = 5,   // grouped_layout not non-decreasing multiples of 128
};

__device__ __forceinline__ void report_failure(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

}  // namespace bfp8
