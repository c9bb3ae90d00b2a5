// bfp8_gemm_swap.cu -- swap-AB instantiations of the blocked FP8 GEMM (small
// M: 128 weight rows fill the MMA M slot, BN >= M activation rows the N slot)
// and the operand re-layout kernel for rows whose stride TMA cannot take.
#include "bfp8_gemm_kernel.cuh"
#include "bfp8_internal.h"

namespace bfp8 {

namespace {

__global__ void relayout_kernel(const uint8_t* __restrict__ src, int64_t rows, int64_t K,
                                uint8_t* __restrict__ dst, int64_t kp) {
  const int64_t chunks_per_row = kp / 16;
  const int64_t total = rows * chunks_per_row;
  for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < total;
       c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = c / chunks_per_row;
    const int64_t k0 = (c - r * chunks_per_row) * 16;
    uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t k = k0 + i;
      const uint32_t b = k < K ? src[r * K + k] : 0u;
      w[i / 4] |= b << (8 * (i % 4));
    }
    *reinterpret_cast<uint4*>(dst + r * kp + k0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Scales in the layout the GEMM kernel bulk-copies: As column-major
// [G][ld_out] (ld_out = M rounded up to 4; padding zero) and Bs contiguous
// with four zero floats after it.
__global__ void scale_relayout_kernel(const float* __restrict__ As, int32_t as_col_major,
                                      int64_t ld_as, int64_t M, int64_t G, float* __restrict__ As_out,
                                      int64_t ld_out, const float* __restrict__ Bs, int64_t nbs,
                                      float* __restrict__ Bs_out) {
  const int64_t n_as = As_out ? G * ld_out : 0;
  const int64_t total = n_as + (Bs_out ? nbs + 4 : 0);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (i < n_as) {
      const int64_t kb = i / ld_out, m = i - kb * ld_out;
      As_out[i] = m < M ? (as_col_major ? As[kb * ld_as + m] : As[m * ld_as + kb]) : 0.f;
    } else {
      const int64_t e = i - n_as;
      Bs_out[e] = e < nbs ? Bs[e] : 0.f;
    }
  }
}

}  // namespace

cudaError_t launch_scale_relayout(const float* As, int as_col_major, int64_t ld_as, int64_t M,
                                  int64_t G, float* As_out, int64_t ld_out, const float* Bs,
                                  int64_t nbs, float* Bs_out, int num_sms, cudaStream_t stream) {
  const int64_t total = (As_out ? G * ld_out : 0) + (Bs_out ? nbs + 4 : 0);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > static_cast<int64_t>(num_sms) * 4) blocks = static_cast<int64_t>(num_sms) * 4;
  scale_relayout_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      As, as_col_major, ld_as, M, G, As_out, ld_out, Bs, nbs, Bs_out);
  return cudaGetLastError();
}

cudaError_t launch_gemm_swap(int bn, const CUtensorMap& tmP, const CUtensorMap& tmQ,
                             const GemmArgs& a, cudaStream_t stream) {
  switch (bn) {
    case 16: return launch_instance<16, true>(tmP, tmQ, a, stream);
    case 32: return launch_instance<32, true>(tmP, tmQ, a, stream);
    case 64: return launch_instance<64, true>(tmP, tmQ, a, stream);
    case 128: return launch_instance<128, true>(tmP, tmQ, a, stream);
    case 256: return launch_instance<256, true>(tmP, tmQ, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_cluster_capacity(int cs, bool two_per_sm, int* clusters) {
  // the instantiations of each residency class share their answer
  return two_per_sm ? cluster_capacity_instance<16, true>(cs, clusters)
                    : cluster_capacity_instance<128, true>(cs, clusters);
}

cudaError_t launch_relayout(const uint8_t* src, int64_t rows, int64_t K, uint8_t* dst, int64_t kp,
                            int num_sms, cudaStream_t stream) {
  const int64_t total = rows * (kp / 16);
  int64_t blocks = (total + 255) / 256;
  if (blocks > static_cast<int64_t>(num_sms) * 8) blocks = static_cast<int64_t>(num_sms) * 8;
  if (blocks < 1) blocks = 1;
  relayout_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(src, rows, K, dst, kp);
  return cudaGetLastError();
}

}  // namespace bfp8
