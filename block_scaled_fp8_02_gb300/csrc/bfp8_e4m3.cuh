// bfp8_e4m3.cuh -- the per-token-group quantisation arithmetic shared by the
// quantisation kernel and the fused GEMM epilogue (per_token_group_quant_fp8
// with group 128 of the vLLM PR 49932 digest, "key source snippet"):
//   scale = fl32(max(amax, 1e-10) / 448)      the IEEE fp32 quotient (div448)
//   code  = e4m3_rn_satfinite(fl32(x / scale)) one IEEE fp32 division per element
//
// The codes are found without dividing.  With r = rcp.approx(scale) (relative
// error <= 2^-23), r_lo = RN(r (1 - 2^-19)) and r_hi = RN(r (1 + 2^-19)), the
// products y_lo = RN(x r_lo) and y_hi = RN(x r_hi) differ from x / scale by a
// factor within (1 - 2^-19 +- 2^-21) and (1 + 2^-19 +- 2^-21), while
// fl32(x / scale) is within a factor 1 +- 2^-24 of it, so fl32(x / scale) lies
// strictly between y_lo and y_hi (for |x / scale| >= 2^-126; below that all
// three give e4m3 +-0).  Rounding to e4m3 (nearest-even, saturating) is
// monotone, so when y_lo and y_hi get the same code, that is the code of
// fl32(x / scale).  Only when an e4m3 rounding boundary falls in the 2^-18
// wide bracket must the IEEE division decide: about once in 30000 elements
// for data with full fp32 significands, but about once in 200 for bf16 data,
// whose quotients often fall exactly on a boundary (448 x / amax is then a
// ratio of small integers).  Callers therefore remember which pairs were
// undecided and divide only those, in a warp-uniform branch.
#pragma once

#include <cstdint>

namespace bfp8 {

// fl32(a / 448) for a >= 1e-10 without a division: q0 = RN(a * y) with
// y = RN(1 / 448), then one correction step with the exact residual
// a - q0 * 448 (one FMA), q = RN(q0 + r * y) (Markstein's corrected
// reciprocal product).  Checked exhaustively on the CPU against the IEEE
// quotient for every fp32 a from 1e-10 to the largest finite value (it differs
// only where the quotient is subnormal, below this range).
__device__ __forceinline__ float div448(float a) {
  constexpr float y = 0x1.24924ap-9f;           // RN(1 / 448)
  const float q0 = __fmul_rn(a, y);
  const float r = __fmaf_rn(-q0, 448.0f, a);
  return __fmaf_rn(r, y, q0);
}

__device__ __forceinline__ float group_scale(float amax) {
  return div448(fmaxf(amax, 1e-10f));
}

// Approximate reciprocal (PTX rcp.approx: at most 1 ulp from 1/s).
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// The two bracketing multipliers of a group.
struct E4m3Bracket {
  float lo, hi;
  __device__ __forceinline__ explicit E4m3Bracket(float scale) {
    const float r = rcp_approx(scale);
    lo = __fmul_rn(r, 1.0f - 0x1p-19f);
    hi = __fmul_rn(r, 1.0f + 0x1p-19f);
  }
};

// Codes of fl32(x0 / scale) and fl32(x1 / scale), low byte first, when the
// bracket decides them; `undecided` is set when it does not (branch-free, so
// that the conversions of many pairs can be interleaved).
__device__ __forceinline__ uint16_t e4m3_pair_bracketed(float x0, float x1, const E4m3Bracket& b,
                                                        bool& undecided) {
  const uint16_t lo = cvt_e4m3x2(__fmul_rn(x0, b.lo), __fmul_rn(x1, b.lo));
  const uint16_t hi = cvt_e4m3x2(__fmul_rn(x0, b.hi), __fmul_rn(x1, b.hi));
  undecided = lo != hi;
  return lo;
}

// UE8M0 scales (transformers DeepGEMM integration, _ceil_to_ue8m0): the fp32
// scale rounded up to the nearest power of two by adding 2^23 - 1 to its bit
// pattern and clearing the 23 mantissa bits (positive finite scales only).
__device__ __forceinline__ uint32_t ceil_ue8m0_bits(float s) {
  return (__float_as_uint(s) + 0x7FFFFFu) & 0xFF800000u;
}

// Group scale of the UE8M0 variant, and its exact reciprocal: for 2^e with
// biased exponent E (E = 85 .. 247 here: 2^-42 <= scale < 2^121), 1 / 2^e has
// biased exponent 254 - E, i.e. bits 0x7F000000 - bits.  x * (1 / scale) is
// then the correctly rounded x / scale (the same real number, rounded once),
// so the codes need neither a division nor a bracket.
struct Ue8m0Scale {
  float scale, inv;
  __device__ __forceinline__ explicit Ue8m0Scale(float amax) {
    const uint32_t b = ceil_ue8m0_bits(group_scale(amax));
    scale = __uint_as_float(b);
    inv = __uint_as_float(0x7F000000u - b);
  }
};

__device__ __forceinline__ uint16_t e4m3_pair_pow2(float x0, float x1, float inv) {
  return cvt_e4m3x2(__fmul_rn(x0, inv), __fmul_rn(x1, inv));
}

// The same codes by the IEEE division.
__device__ __forceinline__ uint16_t e4m3_pair_divided(float x0, float x1, float scale) {
  return cvt_e4m3x2(__fdiv_rn(x0, scale), __fdiv_rn(x1, scale));
}

}  // namespace bfp8
