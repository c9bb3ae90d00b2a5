// bfp8_internal.h -- declarations shared by the library's translation units
// (host side).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cstddef>
#include <cstdint>

#include "../../include/bfp8.h"
#include "bfp8_sched.h"

namespace bfp8 {

// Records `msg` as the calling thread's bfp8_last_error() and returns st.
bfp8_status set_last_error(bfp8_status st, const char* msg);

struct GemmArgs;

// Per-token group quantisation launcher (bfp8_quant.cu); ue8m0: scales
// rounded up to powers of two.
cudaError_t launch_group_quant(const void* x, int in_f32, int64_t M, int64_t K, int64_t ld_x,
                               uint8_t* q, int64_t ld_q, float* s, int col_major, int64_t ld_s,
                               int ue8m0, int num_sms, cudaStream_t stream);
// n fp32 scales rounded up to powers of two (bfp8_quant.cu).
cudaError_t launch_scale_ceil_ue8m0(const float* in, float* out, int64_t n, int num_sms,
                                    cudaStream_t stream);

// GEMM launchers (bfp8_gemm_swap.cu, bfp8_gemm_wide.cu).  `bn` selects the
// instantiation; returns cudaErrorInvalidValue for one that does not exist.
cudaError_t launch_gemm_swap(int bn, const CUtensorMap& tmP, const CUtensorMap& tmQ,
                             const GemmArgs& a, cudaStream_t stream);
// `mode` selects the plain, M-grouped or fused-epilogue variant (wide only;
// bfp8_gemm_kernel.cuh's kMode* values; the last two live in bfp8_gemm_ext.cu);
// `mr` the activation rows loaded per stage (128, or 32 / 64 for plain
// 256-wide tiles of decode-sized M).
cudaError_t launch_gemm_wide(int bn, int mode, int mr, const CUtensorMap& tmP,
                             const CUtensorMap& tmQ, const GemmArgs& a, cudaStream_t stream);
cudaError_t launch_gemm_wide_ext(int bn, int mode, const CUtensorMap& tmP, const CUtensorMap& tmQ,
                                 const GemmArgs& a, cudaStream_t stream);

// The GEMM for M <= kGemvMaxM activation rows on warp-level MMAs
// (bfp8_gemv.cu).  tmW: B [N, K] e4m3 viewed as [N][K/128][128] bytes, box
// 128 x 8 x 16 (eight k-blocks of 16 weight rows), 128-byte swizzle, zero
// fill; tmX: A [M, K] viewed the same way, box 128 x 8 x M.  K % 128 == 0.
constexpr int kGemvMaxM = 32;
struct GemvArgs {
  const float* As;       // activation scales, either layout (4-byte aligned)
  int64_t ld_as;
  int32_t as_col_major;
  const float* Bs;       // [ceil(N/128), G]
  __nv_bfloat16* out;    // [M, N] row-major
  int32_t M;
  int64_t N;
  int64_t G;             // K / 128
  int32_t prefetch_b;    // request the first weights before the grid dependency
  int* err;              // device failure word
  unsigned long long wait_limit;
  // 1: As is column-major with ld_as % 4 == 0, ld_as <= 8 * ceil(M / 8) and
  // 16-byte aligned: each stage's As slice (8 k-blocks x ld_as floats,
  // contiguous) is bulk-copied with the stage; 0: read by the scale warp
  int32_t as_bulk;
};
// max_ctas > 0 caps the grid (persistent CTAs; two or three per SM up to M = 24).
cudaError_t launch_gemv(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemvArgs& a,
                        int num_sms, int max_ctas, cudaStream_t stream);

// The paired wide-tile GEMM (bfp8_gemm_pair.cu): sched.grid counts CTA pairs,
// whole tiles of 256 x 256 only.
cudaError_t launch_gemm_pair(const CUtensorMap& tmP, const CUtensorMap& tmQ, const GemmArgs& a,
                             cudaStream_t stream);
int gemm_pair_stages();

// Clusters of `cs` GEMM CTAs the current device runs at once (bfp8_gemm_swap.cu),
// for the instantiations sized for two CTAs per SM (swap-AB tiles up to 64
// columns wide) or for the others (one CTA per SM).
cudaError_t gemm_cluster_capacity(int cs, bool two_per_sm, int* clusters);

// True for the GEMM instantiations sized for two CTAs per SM.
inline bool gemm_two_per_sm(bool swap, int bn) { return swap && bn <= 64; }

// Bytes at the start of every GEMM workspace that hold the stream-K tile
// counters (4096 of them); they must read zero when a GEMM starts, and every
// completed GEMM leaves them zero.
constexpr size_t kCounterHeaderBytes = 16384;

// Pipeline depth and dynamic shared memory of an instantiation (0 if none).
int gemm_stages(bool swap, int bn, int mr = 128);
int gemm_threads(bool swap, int bn);
size_t gemm_smem_bytes(bool swap, int bn);

// Copies rows x K bytes (row stride K) into rows x kp bytes (row stride kp,
// kp = K rounded up to 16) with zeros in columns K .. kp-1 (bfp8_gemm_swap.cu).
cudaError_t launch_relayout(const uint8_t* src, int64_t rows, int64_t K, uint8_t* dst, int64_t kp,
                            int num_sms, cudaStream_t stream);

// Copies the scales into the layout the GEMM kernel reads: As column-major
// [G][ld_out] with ld_out = M rounded up to 4 (when As_out != nullptr) and Bs
// with four zero floats appended (when Bs_out != nullptr).
cudaError_t launch_scale_relayout(const float* As, int as_col_major, int64_t ld_as, int64_t M,
                                  int64_t G, float* As_out, int64_t ld_out, const float* Bs,
                                  int64_t nbs, float* Bs_out, int num_sms, cudaStream_t stream);

}  // namespace bfp8
