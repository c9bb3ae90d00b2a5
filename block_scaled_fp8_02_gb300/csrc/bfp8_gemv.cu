// bfp8_gemv.cu -- the blocked FP8 GEMM for a handful of activation rows
// (M <= 8): a matrix-vector product bound by the weight stream.
//
// At M <= 8 the layer reads 16 MB of e4m3 weights (N = K = 4096) for at most
// 0.27 GFLOP.  The tcgen05 kernel spreads 32 weight tiles over the SMs by
// cluster split-K, with TMEM, a distributed reduction and one 128 x 16 MMA per
// 4 KB of weights; here the contraction is small enough for the warp-level
// tensor-core instruction mma.sync.m16n8k32 (e4m3 x e4m3 -> fp32), whose
// operands come straight from registers: no shared-memory staging, no TMEM, no
// clusters, no workspace.
//
// A CTA (8 warps) owns 16 weight rows (output columns n0 .. n0 + 15); warp w
// takes a contiguous 1/8 of the k-blocks.  Per k-block each lane loads 16
// bytes of weight rows g and g + 8 (g = lane / 4) and 16 bytes of activation
// row g at the same k offsets (64 bytes per group of 4 lanes, two 64-byte
// windows per 128-wide k-block) and feeds them to two MMAs per window.  The
// fragment slots are filled with the same absolute k positions on both
// operands, so each MMA sums 32 exact e4m3 products per output, in fp32; the
// four MMAs of a k-block start from zero, and the k-block's 16 x 8 partial is
// scaled by Bs[n/128, kb] * As[m, kb] into an fp32 accumulator (the blocked
// definition of the vLLM PR 49932 digest's matmul).  The 8 warps' partials
// are added in warp order in shared memory (deterministic) and rounded to bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bfp8_internal.h"
#include "bfp8_ptx.cuh"

namespace bfp8 {

namespace {

constexpr int kGemvWarps = 8;      // warps per CTA = k-slices of a 16-row tile
constexpr int kAhead = 2;          // k-blocks of loads in flight ahead of the one in use

// d += a (16 x 32 e4m3, row) * b (32 x 8 e4m3, col), fp32.  Fragments: lane
// (g = lane / 4, t = lane % 4) holds A rows g (a0, a2) and g + 8 (a1, a3) at
// k = 4t .. 4t + 3 (a0, a1) and 16 + 4t .. (a2, a3); B column g at the same k
// (b0, b1); D rows g (d0, d1) and g + 8 (d2, d3), columns 2t and 2t + 1.
__device__ __forceinline__ void mma_e4m3_16x8x32(float (&d)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One k-block's operands for this lane: weight rows g and g + 8 and
// activation row g, 16 bytes each, in each of the block's two windows, and
// the k-block's scales (Bs of the 16 rows; As of this lane's two columns),
// all requested kAhead k-blocks before they are used.
struct KbWords {
  uint4 w0[2], w1[2], x[2];
  float sb, sa0, sa1;
};

// Requires K % 16 == 0 and A, B 16-byte aligned (a 16-byte word of a row is
// wholly inside or wholly past K).  M <= 8.  Persistent: CTA b takes the
// 16-row tiles b, b + gridDim.x, ...; each warp walks the (tile, k-block)
// positions of its k-slice through all of them, with the loads of the next
// kAhead positions in flight (across tile boundaries too).
__global__ void __launch_bounds__(kGemvWarps * 32, 2)
    gemv_kernel(const uint8_t* __restrict__ A, int64_t lda, const float* __restrict__ As,
                int32_t as_col_major, int64_t ld_as, const uint8_t* __restrict__ B,
                const float* __restrict__ Bs, __nv_bfloat16* __restrict__ out, int32_t M, int64_t N,
                int64_t K, int32_t prefetch_b) {
  __shared__ float red[kGemvWarps][16][9];          // partial 16 x 8 tiles (padded)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t G = (K + 127) / 128;
  const int64_t tiles = (N + 15) / 16;
  const int64_t step = gridDim.x;
  const int64_t kb_begin = (G * warp) / kGemvWarps, kb_end = (G * (warp + 1)) / kGemvWarps;
  const bool x_row = g < M;
  const int c0 = 2 * t, c1 = 2 * t + 1;                 // this lane's output columns (m)
  // (tile, kb) -> the position `ahead` k-blocks later in this warp's walk
  auto advance = [&](int64_t& tile, int64_t& kb, int64_t ahead) {
    if (kb_end <= kb_begin) return;                     // no k-slice: nothing to walk
    kb += ahead;
    while (kb >= kb_end) {
      kb -= kb_end - kb_begin;
      tile += step;
    }
  };
  auto load_w = [&](int64_t tile, int64_t kb, KbWords& o) {
    const int64_t r0 = tile * 16 + g, r1 = r0 + 8;
    const bool live = tile < tiles;
    o.sb = live ? __ldg(Bs + (tile / 8) * G + kb) : 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t k = kb * 128 + h * 64 + t * 16;
      const bool in = live && k < K;
      o.w0[h] = (in && r0 < N) ? __ldg(reinterpret_cast<const uint4*>(B + r0 * K + k)) : make_uint4(0u, 0u, 0u, 0u);
      o.w1[h] = (in && r1 < N) ? __ldg(reinterpret_cast<const uint4*>(B + r1 * K + k)) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  auto load_x = [&](int64_t tile, int64_t kb, KbWords& o) {
    const bool live = tile < tiles;
    o.sa0 = (live && c0 < M) ? (as_col_major ? __ldg(As + kb * ld_as + c0) : __ldg(As + c0 * ld_as + kb)) : 0.f;
    o.sa1 = (live && c1 < M) ? (as_col_major ? __ldg(As + kb * ld_as + c1) : __ldg(As + c1 * ld_as + kb)) : 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t k = kb * 128 + h * 64 + t * 16;
      o.x[h] = (live && k < K && x_row) ? __ldg(reinterpret_cast<const uint4*>(A + g * lda + k))
                                        : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  const bool has_slice = kb_end > kb_begin;               // G < 8: some warps have none
  KbWords ring[kAhead + 1];
  // the weights are not written by the preceding kernel: with prefetch_b they
  // are requested before waiting for it; the activations only after
  if (prefetch_b && has_slice) {
    int64_t tt = blockIdx.x, kk = kb_begin;
#pragma unroll
    for (int s = 0; s <= kAhead; ++s) {
      load_w(tt, kk, ring[s]);
      advance(tt, kk, 1);
    }
  }
  griddep_launch_dependents();
  griddep_wait();
  if (has_slice) {
    int64_t tt = blockIdx.x, kk = kb_begin;
#pragma unroll
    for (int s = 0; s <= kAhead; ++s) {
      if (!prefetch_b) load_w(tt, kk, ring[s]);
      load_x(tt, kk, ring[s]);
      advance(tt, kk, 1);
    }
  }
  for (int64_t tile = blockIdx.x; tile < tiles; tile += step) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t kb = kb_begin; kb < kb_end; ++kb) {
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 w0 = ring[0].w0[h], w1 = ring[0].w1[h], x = ring[0].x[h];
        mma_e4m3_16x8x32(d, w0.x, w1.x, w0.y, w1.y, x.x, x.y);
        mma_e4m3_16x8x32(d, w0.z, w1.z, w0.w, w1.w, x.z, x.w);
      }
      const float s0 = __fmul_rn(ring[0].sb, ring[0].sa0), s1 = __fmul_rn(ring[0].sb, ring[0].sa1);
      acc[0] = fmaf(d[0], s0, acc[0]);
      acc[1] = fmaf(d[1], s1, acc[1]);
      acc[2] = fmaf(d[2], s0, acc[2]);
      acc[3] = fmaf(d[3], s1, acc[3]);
#pragma unroll
      for (int s = 0; s < kAhead; ++s) ring[s] = ring[s + 1];
      int64_t tt = tile, kk = kb;
      advance(tt, kk, kAhead + 1);
      load_w(tt, kk, ring[kAhead]);
      load_x(tt, kk, ring[kAhead]);
    }
    red[warp][g][c0] = acc[0];
    red[warp][g][c1] = acc[1];
    red[warp][g + 8][c0] = acc[2];
    red[warp][g + 8][c1] = acc[3];
    __syncthreads();
    if (threadIdx.x < 128) {
      const int row = threadIdx.x >> 3, col = threadIdx.x & 7;
      float v = red[0][row][col];
#pragma unroll
      for (int w = 1; w < kGemvWarps; ++w) v += red[w][row][col];
      const int64_t n = tile * 16 + row;
      if (col < M && n < N) out[static_cast<int64_t>(col) * N + n] = __float2bfloat16_rn(v);
    }
    __syncthreads();                                      // red is reused by the next tile
  }
}

}  // namespace

cudaError_t launch_gemv(const uint8_t* A, int64_t lda, const float* As, int as_col_major,
                        int64_t ld_as, const uint8_t* B, const float* Bs, __nv_bfloat16* out, int M,
                        int64_t N, int64_t K, int prefetch_b, int num_sms, cudaStream_t stream) {
  if (M < 1 || M > kGemvMaxM) return cudaErrorInvalidValue;
  // one wave: two CTAs per SM
  int64_t blocks = (N + 15) / 16;
  if (blocks > 2 * static_cast<int64_t>(num_sms)) blocks = 2 * static_cast<int64_t>(num_sms);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kGemvWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_kernel, A, lda, As, static_cast<int32_t>(as_col_major), ld_as,
                            B, Bs, out, static_cast<int32_t>(M), N, K, static_cast<int32_t>(prefetch_b));
}

}  // namespace bfp8
