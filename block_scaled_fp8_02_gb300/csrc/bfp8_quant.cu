// bfp8_quant.cu -- per-token group quantisation to float8_e4m3fn (sm_103a).
//
// For every row m and every group g of 128 consecutive K elements
// (per_token_group_quant_fp8 with group 128, vLLM PR 49932 digest, "key
// source snippet"):
//   amax  = max |x[m, k]| over the group's real elements
//   scale = max(amax, 1e-10) / 448           (one IEEE fp32 division)
//   q     = e4m3_rn_satfinite(x / scale)     (x / scale as one IEEE fp32 division;
//                                             its code is found from two
//                                             products that bracket it, with the
//                                             division only where they disagree)
// (the UE8M0 variant rounds each scale up to a power of two first, so the
// quotients are exact products), and the scale is stored row-major s[m * ld_s + g] or column-major
// s[g * ld_s + m] (the layout the GEMM kernels read; lmdeploy PR 4830 pads its
// stride to 16 bytes for TMA, transformers' _coerce_sf_for_kernel calls it
// MN-major).
//
// Memory-bound: each warp streams 512 input bytes per step with 16-byte loads
// (one 128-element group for fp32 input, two for bf16 input: a half-warp per
// group), reduces amax with warp shuffles inside the group's lanes and packs
// pairs of codes with cvt.rn.satfinite.e4m3x2.f32.  One wave of persistent
// blocks; each warp keeps the loads of its next kUnroll steps in flight while
// it quantises the current ones.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bfp8_e4m3.cuh"
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

template <bool kF32>
__device__ __forceinline__ void load_words(const void* x, int64_t idx, uint32_t (&w)[4]) {
  const uint4 t = kF32 ? __ldg(reinterpret_cast<const uint4*>(static_cast<const float*>(x) + idx))
                       : __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(x) + idx));
  w[0] = t.x; w[1] = t.y; w[2] = t.z; w[3] = t.w;
}

// Same for a lane whose elements run past K or whose row is not 16-byte
// aligned: element by element, zeros beyond `n`.
template <bool kF32>
__device__ __forceinline__ void load_words_tail(const void* x, int64_t idx, int64_t n, uint32_t (&w)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = 0u;
  if constexpr (kF32) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < n) w[e] = __float_as_uint(__ldg(static_cast<const float*>(x) + idx + e));
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (e < n) w[e / 2] |= static_cast<uint32_t>(__ldg(static_cast<const unsigned short*>(x) + idx + e))
                             << (16 * (e & 1));
  }
}

template <bool kF32>
__device__ __forceinline__ void unpack(const uint32_t (&w)[4], float (&v)[QuantShape<kF32>::kEPL]) {
  if constexpr (kF32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(w[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

constexpr int kUnroll = 2;              // warp steps per batch
constexpr int kWarpsPerBlock = 8;
constexpr int kBlocksPerSm = 4;

// Walks one warp's chunks, kUnroll at a time: chunk c = row * chunks_per_row
// + col; warp w takes chunks w, w + nwarps, ... (a chunk is one warp step:
// GPW groups of one row).  Positions advance without division (the host
// checks M * chunks_per_row < 2^31).
struct ChunkWalk {
  uint32_t rw[kUnroll], cl[kUnroll];
  uint32_t cpr, srow, scol;
  __device__ __forceinline__ void init(uint32_t warp0, uint32_t nwarps, uint32_t chunks_per_row) {
    cpr = chunks_per_row;
    const uint32_t stride = nwarps * kUnroll;
    srow = stride / cpr;
    scol = stride - srow * cpr;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t c = warp0 + u * nwarps;
      rw[u] = c / cpr;
      cl[u] = c - rw[u] * cpr;
    }
  }
  __device__ __forceinline__ void advance() {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      cl[u] += scol;
      rw[u] += srow;
      if (cl[u] >= cpr) {
        cl[u] -= cpr;
        ++rw[u];
      }
    }
  }
};

template <bool kF32>
__device__ __forceinline__ void load_batch(const void* x, const ChunkWalk& cw, uint32_t Mu, uint32_t G,
                                           int64_t K, int64_t ld_x, int32_t vec_x, int gi, int li,
                                           uint32_t (&w)[kUnroll][4]) {
  constexpr int EPL = QuantShape<kF32>::kEPL, GPW = QuantShape<kF32>::kGPW;
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const uint32_t gu = cw.cl[u] * GPW + gi;
    const int64_t ku = static_cast<int64_t>(gu) * 128 + li * EPL;
    const bool ok = cw.rw[u] < Mu && gu < G;
    const int64_t off = static_cast<int64_t>(cw.rw[u]) * ld_x + ku;
    if (ok && vec_x && ku + EPL <= K) {
      load_words<kF32>(x, off, w[u]);
    } else {
      load_words_tail<kF32>(x, off, ok ? K - ku : 0, w[u]);
    }
  }
}

// kUe8m0: every scale rounded up to a power of two (the UE8M0 variant).
template <bool kF32, bool kUe8m0>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, kBlocksPerSm)
    group_quant_kernel(const void* __restrict__ x, int64_t M, int64_t K, int64_t ld_x,
                       uint8_t* __restrict__ q, int64_t ld_q, float* __restrict__ s,
                       int32_t col_major, int64_t ld_s, int32_t vec_x, int32_t vec_q) {
  using S = QuantShape<kF32>;
  constexpr int EPL = S::kEPL, LPG = S::kLPG, GPW = S::kGPW;
  const uint32_t G = static_cast<uint32_t>((K + 127) / 128);
  const uint32_t Mu = static_cast<uint32_t>(M);
  const int lane = threadIdx.x & 31;
  const int gi = lane / LPG;       // group within the warp step
  const int li = lane % LPG;       // lane within the group
  const uint32_t warp0 = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const uint32_t nwarps = gridDim.x * kWarpsPerBlock;
  ChunkWalk cur, nxt;
  cur.init(warp0, nwarps, (G + GPW - 1) / GPW);
  // The next kernel (the GEMM, which waits for this grid to complete before
  // reading q and s) may be launched at once, so that its prologue and weight
  // prefetch overlap this kernel; x may come from the kernel before this one,
  // so nothing is read before the wait.
  griddep_launch_dependents();
  griddep_wait();

  // software pipeline: the next batch's loads are in flight while this one
  // is quantised and stored
  uint32_t w[kUnroll][4];
  load_batch<kF32>(x, cur, Mu, G, K, ld_x, vec_x, gi, li, w);
  while (cur.rw[0] < Mu) {
    nxt = cur;
    nxt.advance();
    uint32_t wn[kUnroll][4];
    if (nxt.rw[0] < Mu) load_batch<kF32>(x, nxt, Mu, G, K, ld_x, vec_x, gi, li, wn);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t gu = cur.cl[u] * GPW + gi;
      const int64_t ku = static_cast<int64_t>(gu) * 128 + li * EPL;
      const bool valid = cur.rw[u] < Mu && gu < G;
      float v[EPL];
      unpack<kF32>(w[u], v);
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
      for (int off = LPG / 2; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      float scale;
      uint16_t pk[EPL / 2];
      if constexpr (kUe8m0) {
        // power-of-two scale: exact quotients by one multiply each
        const Ue8m0Scale us(amax);
        scale = us.scale;
#pragma unroll
        for (int e = 0; e < EPL; e += 2) pk[e / 2] = e4m3_pair_pow2(v[e], v[e + 1], us.inv);
      } else {
        scale = group_scale(amax);
        // codes without dividing (bfp8_e4m3.cuh); the IEEE divisions run only
        // in warps where the bracket does not decide a code (warp-uniform branch)
        const E4m3Bracket br(scale);
        uint32_t undecided = 0;                 // one bit per pair
#pragma unroll
        for (int e = 0; e < EPL; e += 2) {
          bool u = false;
          pk[e / 2] = e4m3_pair_bracketed(v[e], v[e + 1], br, u);
          undecided |= static_cast<uint32_t>(u) << (e / 2);
        }
        if (__any_sync(0xffffffffu, undecided != 0)) {
#pragma unroll
          for (int e = 0; e < EPL; e += 2)
            if (undecided & (1u << (e / 2))) pk[e / 2] = e4m3_pair_divided(v[e], v[e + 1], scale);
        }
      }
      if (!valid) continue;
      uint8_t* qrow = q + static_cast<int64_t>(cur.rw[u]) * ld_q;
      if (vec_q && ku + EPL <= K) {
        if constexpr (kF32) {
          *reinterpret_cast<uint32_t*>(qrow + ku) =
              static_cast<uint32_t>(pk[0]) | (static_cast<uint32_t>(pk[1]) << 16);
        } else {
          uint2 wq;
          wq.x = static_cast<uint32_t>(pk[0]) | (static_cast<uint32_t>(pk[1]) << 16);
          wq.y = static_cast<uint32_t>(pk[2]) | (static_cast<uint32_t>(pk[3]) << 16);
          *reinterpret_cast<uint2*>(qrow + ku) = wq;
        }
      } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e)
          if (ku + e < K) qrow[ku + e] = static_cast<uint8_t>(pk[e / 2] >> (8 * (e & 1)));
      }
      if (li == 0) {
        if (col_major) s[static_cast<int64_t>(gu) * ld_s + cur.rw[u]] = scale;
        else s[static_cast<int64_t>(cur.rw[u]) * ld_s + gu] = scale;
      }
    }
    cur = nxt;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int i = 0; i < 4; ++i) w[u][i] = wn[u][i];
  }
}

// ---------------------------------------------------------------------------
// The common case on a lean path: bf16 rows of whole steps (K a multiple of
// 32 * EPL), 16-byte aligned rows of x and q.  A step is one warp's
// 32 * EPL elements of one row: 32 * EPL / 128 groups, 128 / EPL lanes each,
// EPL elements per lane (16-byte loads).  Each warp walks kStepU steps at a
// time (all their loads issued before any is used), with 32-bit offsets (the
// host checks that they fit) and products packed two per instruction.  Same
// arithmetic, bit for bit, as the general kernel above.  (kStepU: 64 bytes of
// loads in flight per lane either way.)
template <int EPL>
constexpr int kStepUFor = EPL == 16 ? 2 : 4;
template <bool kUe8m0, int EPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, kBlocksPerSm)
    group_quant_bf16_steps_kernel(const uint16_t* __restrict__ x, uint32_t M, uint32_t spr,
                                  uint32_t ld_x, uint8_t* __restrict__ q, uint32_t ld_q,
                                  float* __restrict__ s, int32_t col_major, uint32_t ld_s,
                                  uint32_t adv_row, uint32_t adv_col) {
  static_assert(EPL == 8 || EPL == 16, "8 or 16 elements per lane");
  constexpr int kStepU = kStepUFor<EPL>;
  constexpr int kLPG = 128 / EPL;                // lanes per group
  constexpr int kW = EPL / 8;                    // 16-byte words per lane
  constexpr uint32_t kStep = 32u * EPL;          // elements per step
  const int lane = threadIdx.x & 31;
  const uint32_t gi = static_cast<uint32_t>(lane) / kLPG;     // group within the step
  const uint32_t warp0 = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const uint32_t nwarps = gridDim.x * kWarpsPerBlock;
  // walker u visits steps warp0 + (u + kStepU * i) * nwarps; a step is
  // (row, column of kStep elements); each advance moves a walker
  // kStepU * nwarps steps = adv_row rows and adv_col columns (adv_col < spr)
  uint32_t rw[kStepU], cl[kStepU];
#pragma unroll
  for (int u = 0; u < kStepU; ++u) {
    const uint32_t st = warp0 + static_cast<uint32_t>(u) * nwarps;
    rw[u] = st / spr;
    cl[u] = st - rw[u] * spr;
  }
  griddep_launch_dependents();
  griddep_wait();
  while (rw[0] < M) {
    uint4 w[kStepU][kW];
#pragma unroll
    for (int u = 0; u < kStepU; ++u)
      if (rw[u] < M) {
        const uint4* src = reinterpret_cast<const uint4*>(x + rw[u] * ld_x + cl[u] * kStep) + lane * kW;
#pragma unroll
        for (int h = 0; h < kW; ++h) w[u][h] = __ldg(src + h);
      }
#pragma unroll
    for (int u = 0; u < kStepU; ++u) {
      if (rw[u] >= M) continue;
      float v[EPL];
#pragma unroll
      for (int h = 0; h < kW; ++h) {
        const uint32_t ww[4] = {w[u][h].x, w[u][h].y, w[u][h].z, w[u][h].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[8 * h + 2 * i] = __uint_as_float(ww[i] << 16);
          v[8 * h + 2 * i + 1] = __uint_as_float(ww[i] & 0xFFFF0000u);
        }
      }
      float amax = fabsf(v[0]);
#pragma unroll
      for (int e = 1; e < EPL; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
      for (int off = kLPG / 2; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      float scale;
      uint32_t pk[EPL / 2];
      if constexpr (kUe8m0) {
        const Ue8m0Scale us(amax);
        scale = us.scale;
        const uint64_t inv2 = pack_u32x2(__float_as_uint(us.inv), __float_as_uint(us.inv));
#pragma unroll
        for (int i = 0; i < EPL / 2; ++i) {
          float a0, a1;
          unpack_f32x2(mul_f32x2(pack_u32x2(__float_as_uint(v[2 * i]), __float_as_uint(v[2 * i + 1])), inv2),
                       a0, a1);
          pk[i] = cvt_e4m3x2(a0, a1);
        }
      } else {
        scale = group_scale(amax);
        const E4m3Bracket br(scale);
        const uint64_t lo2 = pack_u32x2(__float_as_uint(br.lo), __float_as_uint(br.lo));
        const uint64_t hi2 = pack_u32x2(__float_as_uint(br.hi), __float_as_uint(br.hi));
        uint32_t undecided = 0;
#pragma unroll
        for (int i = 0; i < EPL / 2; ++i) {
          const uint64_t x2 = pack_u32x2(__float_as_uint(v[2 * i]), __float_as_uint(v[2 * i + 1]));
          float a0, a1, b0, b1;
          unpack_f32x2(mul_f32x2(x2, lo2), a0, a1);
          unpack_f32x2(mul_f32x2(x2, hi2), b0, b1);
          const uint32_t lo = cvt_e4m3x2(a0, a1), hi = cvt_e4m3x2(b0, b1);
          pk[i] = lo;
          undecided |= static_cast<uint32_t>(lo != hi) << i;
        }
        // warp-uniform branch: IEEE divisions only for the undecided pairs
        if (__any_sync(0xffffffffu, undecided != 0)) {
#pragma unroll
          for (int i = 0; i < EPL / 2; ++i)
            if (undecided & (1u << i)) pk[i] = e4m3_pair_divided(v[2 * i], v[2 * i + 1], scale);
        }
      }
      uint8_t* dst = q + rw[u] * ld_q + cl[u] * kStep + static_cast<uint32_t>(lane) * EPL;
      if constexpr (EPL == 16) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0] | (pk[1] << 16), pk[2] | (pk[3] << 16),
                                                    pk[4] | (pk[5] << 16), pk[6] | (pk[7] << 16));
      } else {
        *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0] | (pk[1] << 16), pk[2] | (pk[3] << 16));
      }
      if ((static_cast<uint32_t>(lane) % kLPG) == 0) {
        const uint32_t g = cl[u] * (kStep / 128u) + gi;
        if (col_major) s[g * ld_s + rw[u]] = scale;
        else s[rw[u] * ld_s + g] = scale;
      }
    }
#pragma unroll
    for (int u = 0; u < kStepU; ++u) {
      cl[u] += adv_col;
      rw[u] += adv_row;
      if (cl[u] >= spr) {
        cl[u] -= spr;
        ++rw[u];
      }
    }
  }
}

// Rounds n fp32 scales up to powers of two (the UE8M0 variant's weight scales).
__global__ void scale_ceil_ue8m0_kernel(const float* __restrict__ in, float* __restrict__ out,
                                        int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = __uint_as_float(ceil_ue8m0_bits(in[i]));
}

}  // namespace

cudaError_t launch_scale_ceil_ue8m0(const float* in, float* out, int64_t n, int num_sms,
                                    cudaStream_t stream) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > static_cast<int64_t>(num_sms) * 4) blocks = static_cast<int64_t>(num_sms) * 4;
  if (blocks < 1) blocks = 1;
  scale_ceil_ue8m0_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(in, out, n);
  return cudaGetLastError();
}

namespace {

template <bool kF32, bool kUe8m0>
cudaError_t launch_quant_instance(const cudaLaunchConfig_t& cfg, const void* x, int64_t M,
                                  int64_t K, int64_t ld_x, uint8_t* q, int64_t ld_q, float* s,
                                  int32_t cm, int64_t ld_s, int32_t vec_x, int32_t vec_q) {
  return cudaLaunchKernelEx(&cfg, group_quant_kernel<kF32, kUe8m0>, x, M, K, ld_x, q, ld_q, s, cm,
                            ld_s, vec_x, vec_q);
}

}  // namespace

cudaError_t launch_group_quant(const void* x, int in_f32, int64_t M, int64_t K, int64_t ld_x,
                               uint8_t* q, int64_t ld_q, float* s, int col_major, int64_t ld_s,
                               int ue8m0, int num_sms, cudaStream_t stream) {
  // lean path: bf16, whole steps (512 elements: 16 per lane; else 256: 8 per
  // lane), 16-byte aligned rows of x and q (8-byte for 8 per lane), 32-bit
  // offsets
  const int lean_epl = (K % 512 == 0 && reinterpret_cast<uintptr_t>(q) % 16 == 0 && ld_q % 16 == 0) ? 16 : 8;
  const bool lean = !in_f32 && K % 256 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                    ld_x % 8 == 0 && reinterpret_cast<uintptr_t>(q) % 8 == 0 && ld_q % 8 == 0 &&
                    M * ld_x < (int64_t{1} << 31) && M * ld_q < (int64_t{1} << 31) &&
                    (col_major ? ((K / 128) * ld_s) : (M * ld_s)) < (int64_t{1} << 31);
  if (lean) {
    const uint32_t spr = static_cast<uint32_t>(K / (32 * lean_epl));
    const int64_t steps = M * spr;
    int64_t blocks = (steps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int64_t cap = static_cast<int64_t>(num_sms) * kBlocksPerSm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const uint32_t adv =
        static_cast<uint32_t>(blocks) * kWarpsPerBlock * (lean_epl == 16 ? kStepUFor<16> : kStepUFor<8>);
    if (steps + 2 * static_cast<int64_t>(adv) >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kWarpsPerBlock * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const auto* xb = static_cast<const uint16_t*>(x);
    const uint32_t Mu = static_cast<uint32_t>(M), ldx = static_cast<uint32_t>(ld_x),
                   ldq = static_cast<uint32_t>(ld_q), lds = static_cast<uint32_t>(ld_s);
    const int32_t cm = col_major;
    const uint32_t ar = adv / spr, ac = adv % spr;
    if (lean_epl == 16)
      return ue8m0 ? cudaLaunchKernelEx(&cfg, group_quant_bf16_steps_kernel<true, 16>, xb, Mu, spr, ldx,
                                        q, ldq, s, cm, lds, ar, ac)
                   : cudaLaunchKernelEx(&cfg, group_quant_bf16_steps_kernel<false, 16>, xb, Mu, spr, ldx,
                                        q, ldq, s, cm, lds, ar, ac);
    return ue8m0 ? cudaLaunchKernelEx(&cfg, group_quant_bf16_steps_kernel<true, 8>, xb, Mu, spr, ldx, q,
                                      ldq, s, cm, lds, ar, ac)
                 : cudaLaunchKernelEx(&cfg, group_quant_bf16_steps_kernel<false, 8>, xb, Mu, spr, ldx, q,
                                      ldq, s, cm, lds, ar, ac);
  }
  const int64_t G = (K + 127) / 128;
  const int esize = in_f32 ? 4 : 2;
  const int epl = in_f32 ? 4 : 8;
  const int gpw = in_f32 ? 1 : 2;
  const int vec_x = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && ((ld_x * esize) % 16 == 0);
  const int vec_q = (reinterpret_cast<uintptr_t>(q) % epl == 0) && (ld_q % epl == 0);
  const int64_t total = M * ((G + gpw - 1) / gpw);
  if (total >= (int64_t{1} << 31) - static_cast<int64_t>(num_sms) * 8 * kWarpsPerBlock * kUnroll)
    return cudaErrorInvalidValue;
  // one wave of persistent blocks (each warp then walks many chunks, which
  // keeps its software pipeline full)
  int64_t blocks = (total + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int64_t cap = static_cast<int64_t>(num_sms) * kBlocksPerSm;
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
    return ue8m0 ? launch_quant_instance<true, true>(cfg, x, M, K, ld_x, q, ld_q, s, cm, ld_s, vec_x, vec_q)
                 : launch_quant_instance<true, false>(cfg, x, M, K, ld_x, q, ld_q, s, cm, ld_s, vec_x, vec_q);
  return ue8m0 ? launch_quant_instance<false, true>(cfg, x, M, K, ld_x, q, ld_q, s, cm, ld_s, vec_x, vec_q)
               : launch_quant_instance<false, false>(cfg, x, M, K, ld_x, q, ld_q, s, cm, ld_s, vec_x, vec_q);
}

}  // namespace bfp8
