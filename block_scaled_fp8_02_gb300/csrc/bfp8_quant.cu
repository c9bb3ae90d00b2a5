// bfp8_quant.cu -- per-token group quantisation to float8_e4m3fn (sm_103a).
//
// For every row m and every group g of 128 consecutive K elements
// (per_token_group_quant_fp8 with group 128, vLLM PR 49932 digest, "key
// source snippet"):
//   amax  = max |x[m, k]| over the group's real elements
//   scale = max(amax, 1e-10) / 448           (one IEEE fp32 division)
//   q     = e4m3_rn_satfinite(x / scale)     (x / scale as one IEEE fp32 division;
//                                             computed as x * (1/scale) except
//                                             near e4m3 rounding boundaries,
//                                             which gives the same codes)
// and the scale is stored row-major s[m * ld_s + g] or column-major
// s[g * ld_s + m] (the layout the GEMM kernels read; lmdeploy PR 4830 pads its
// stride to 16 bytes for TMA, transformers' _coerce_sf_for_kernel calls it
// MN-major).
//
// Memory-bound: each warp streams 512 input bytes per step with 16-byte loads
// (one 128-element group for fp32 input, two for bf16 input: a half-warp per
// group), reduces amax with warp shuffles inside the group's lanes and packs
// pairs of codes with cvt.rn.satfinite.e4m3x2.f32.  Four steps (2 KB) are in
// flight per warp to keep enough bytes outstanding.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bfp8_internal.h"
#include "bfp8_ptx.cuh"

namespace bfp8 {

namespace {

template <bool kF32>
struct QuantShape {
  static constexpr int kEPL = kF32 ? 4 : 8;     // elements per lane (16 bytes)
  static constexpr int kLPG = 128 / kEPL;       // lanes per group
  static constexpr int kGPW = 32 / kLPG;        // groups per warp step
};

// fl32(x / scale) as far as its e4m3 code is concerned.  y = x * rcp, with
// rcp = 1/scale rounded to nearest, differs from x / scale by at most 2 ulp
// and from its correctly rounded value by at most 2.5 ulp.  The e4m3 code of
// a value with |y| >= 2^-6 only changes at the midpoints between e4m3 values,
// fp32 numbers whose low 20 mantissa bits are exactly 0x80000; so unless y is
// within 3 ulp of such a midpoint (or in the e4m3 subnormal range, where the
// spacing is fixed) both round to the same code, and the IEEE division is
// only needed for those rare cases.
__device__ __forceinline__ float quotient_for_e4m3(float x, float scale, float rcp) {
  const float y = __fmul_rn(x, rcp);
  const uint32_t b = __float_as_uint(y) & 0x7FFFFFFFu;
  const bool tiny = b < 0x3C800000u;                            // |y| < 2^-6
  const bool near_mid = ((b - 0x80000u + 3u) & 0xFFFFFu) <= 6u;  // within 3 ulp of a midpoint
  return (tiny || near_mid) ? __fdiv_rn(x, scale) : y;
}

__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <bool kF32>
__device__ __forceinline__ float load_elem(const void* x, int64_t idx) {
  if constexpr (kF32) {
    return __ldg(static_cast<const float*>(x) + idx);
  } else {
    const unsigned short b = __ldg(static_cast<const unsigned short*>(x) + idx);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
}

template <bool kF32>
__device__ __forceinline__ void load_vec(const void* x, int64_t idx, float (&v)[QuantShape<kF32>::kEPL]) {
  if constexpr (kF32) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + idx));
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  } else {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(x) + idx));
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(words[i] << 16);
      v[2 * i + 1] = __uint_as_float(words[i] & 0xFFFF0000u);
    }
  }
}

constexpr int kUnroll = 4;
constexpr int kWarpsPerBlock = 8;

template <bool kF32>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, 4)
    group_quant_kernel(const void* __restrict__ x, int64_t M, int64_t K, int64_t ld_x,
                       uint8_t* __restrict__ q, int64_t ld_q, float* __restrict__ s,
                       int32_t col_major, int64_t ld_s, int32_t vec_x, int32_t vec_q) {
  using S = QuantShape<kF32>;
  constexpr int EPL = S::kEPL, LPG = S::kLPG, GPW = S::kGPW;
  // chunk indices fit in 32 bits (the host checks M * chunks_per_row < 2^31),
  // so the row / chunk split is a 32-bit division, not a 64-bit one
  const uint32_t G = static_cast<uint32_t>((K + 127) / 128);
  const uint32_t chunks_per_row = (G + GPW - 1) / GPW;
  const uint32_t total = static_cast<uint32_t>(M) * chunks_per_row;
  const int lane = threadIdx.x & 31;
  const int gi = lane / LPG;       // group within the warp step
  const int li = lane % LPG;       // lane within the group
  const uint32_t warp0 = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const uint32_t nwarps = gridDim.x * kWarpsPerBlock;
  // x may come from the kernel before this one; once it is visible, the next
  // kernel (the GEMM, which waits for this grid before reading q and s) may
  // start its prologue
  griddep_wait();
  griddep_launch_dependents();

  for (uint32_t base = warp0; base < total; base += nwarps * kUnroll) {
    float v[kUnroll][EPL];
    int64_t row[kUnroll], k[kUnroll], g[kUnroll];
    bool valid[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t c = base + u * nwarps;
      const uint32_t rr = c / chunks_per_row;
      row[u] = rr;
      g[u] = static_cast<int64_t>(c - rr * chunks_per_row) * GPW + gi;
      k[u] = g[u] * 128 + li * EPL;
      valid[u] = (c < total) && (g[u] < G);
      if (valid[u] && vec_x && k[u] + EPL <= K) {
        load_vec<kF32>(x, row[u] * ld_x + k[u], v[u]);
      } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e)
          v[u][e] = (valid[u] && k[u] + e < K) ? load_elem<kF32>(x, row[u] * ld_x + k[u] + e) : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(v[u][e]));
#pragma unroll
      for (int off = LPG / 2; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      if (!valid[u]) continue;
      const float scale = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
      const float rcp = __frcp_rn(scale);
      uint16_t pk[EPL / 2];
#pragma unroll
      for (int e = 0; e < EPL; e += 2)
        pk[e / 2] = cvt_e4m3x2(quotient_for_e4m3(v[u][e], scale, rcp),
                               quotient_for_e4m3(v[u][e + 1], scale, rcp));
      uint8_t* qrow = q + row[u] * ld_q;
      if (vec_q && k[u] + EPL <= K) {
        if constexpr (kF32) {
          *reinterpret_cast<uint32_t*>(qrow + k[u]) =
              static_cast<uint32_t>(pk[0]) | (static_cast<uint32_t>(pk[1]) << 16);
        } else {
          uint2 w;
          w.x = static_cast<uint32_t>(pk[0]) | (static_cast<uint32_t>(pk[1]) << 16);
          w.y = static_cast<uint32_t>(pk[2]) | (static_cast<uint32_t>(pk[3]) << 16);
          *reinterpret_cast<uint2*>(qrow + k[u]) = w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e)
          if (k[u] + e < K) qrow[k[u] + e] = static_cast<uint8_t>(pk[e / 2] >> (8 * (e & 1)));
      }
      if (li == 0) {
        if (col_major) s[g[u] * ld_s + row[u]] = scale;
        else s[row[u] * ld_s + g[u]] = scale;
      }
    }
  }
}

}  // namespace

cudaError_t launch_group_quant(const void* x, int in_f32, int64_t M, int64_t K, int64_t ld_x,
                               uint8_t* q, int64_t ld_q, float* s, int col_major, int64_t ld_s,
                               int num_sms, cudaStream_t stream) {
  const int64_t G = (K + 127) / 128;
  const int esize = in_f32 ? 4 : 2;
  const int epl = in_f32 ? 4 : 8;
  const int gpw = in_f32 ? 1 : 2;
  const int vec_x = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && ((ld_x * esize) % 16 == 0);
  const int vec_q = (reinterpret_cast<uintptr_t>(q) % epl == 0) && (ld_q % epl == 0);
  const int64_t total = M * ((G + gpw - 1) / gpw);
  if (total >= (int64_t{1} << 31) - static_cast<int64_t>(num_sms) * 8 * kWarpsPerBlock * kUnroll)
    return cudaErrorInvalidValue;
  int64_t blocks = (total + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kWarpsPerBlock * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int32_t cm = col_major;
  if (in_f32)
    return cudaLaunchKernelEx(&cfg, group_quant_kernel<true>, x, M, K, ld_x, q, ld_q, s, cm, ld_s,
                              vec_x, vec_q);
  return cudaLaunchKernelEx(&cfg, group_quant_kernel<false>, x, M, K, ld_x, q, ld_q, s, cm, ld_s,
                            vec_x, vec_q);
}

}  // namespace bfp8
