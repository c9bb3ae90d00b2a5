// bfp8_gemv.cu -- the blocked FP8 GEMM for a few activation rows (M <= 32):
// a matrix-vector-like product bound by the weight stream.
//
// At M <= 32 the layer reads 16.8 MB of e4m3 weights (N = K = 4096) for at
// most 1.1 GFLOP.  Here the contraction runs on the warp-level tensor-core
// instruction mma.sync.m16n8k32 (e4m3 x e4m3 -> fp32), with the weight rows
// in its 16-row slot (swap-AB: N in the MMA's M slot) and up to four 8-column
// groups of activation rows; no TMEM, no clusters, no workspace.
//
// The weights stream through TMA.  B [N, K] is viewed as a 3-D tensor of
// 128-byte k-block lines indexed (byte, row, k-block); one box is 16 weight
// rows x 8 k-blocks (16 KB, landing k-block-major as [k-block][row][128
// bytes] with the 128-byte swizzle, so that rows four apart in a k-block sit
// four swizzle phases apart), and the activations of the same 8 k-blocks
// come as one box of M rows: a stage.  A producer lane keeps a ring of
// 2 .. 4 stages in flight (up to 192 KB per SM), across tile boundaries, so
// each SM has a large share of the weights requested at once -- plain
// per-thread loads were limited by the requests a warp can keep
// outstanding.  With the weight prefetch, the first ring of weights and
// weight scales is requested before the preceding kernel completes.
// Each stage's scales land in a per-stage slot that completes on the stage's
// barrier, so the MMA warps never wait on a global load (reading the scales
// themselves, a few stages ahead, cost a third of the bandwidth on long
// weight streams): the As slice of the stage's 8 k-blocks (contiguous in the
// column-major layout) is bulk-copied with the activation box, and a third
// role, the scale warp, reads the Bs of the tile's 128-row block (and As in
// other layouts) with plain loads several stages ahead.
//
// A CTA (8 MMA warps, a TMA warp and a scale warp; two or three CTAs per SM
// for M <= 24, one above) takes 16-row weight tiles n0 = 16 * (blockIdx.x +
// i * gridDim.x).  In every stage warp w takes k-block w: lane (g = lane / 4,
// t = lane % 4) reads 16 bytes of weight rows p and p + 8 at k = 16t and
// k = 64 + 16t of the block, p = g / 2 + 4 (g % 2), and the same k of
// activation row p of each column group (the permutation spreads each
// quarter-warp's rows over all banks), and issues four MMAs per group whose
// fragment slots hold the same absolute k on both operands (the MMA's k
// order is a permutation of the block's, which a dot product does not see),
// as two chains of two that are added at the end.  The k-block's 16 x 8
// partial is scaled by Bs[n/128, kb] * As[m, kb] into fp32 accumulators (the
// blocked definition of the vLLM PR 49932 digest's matmul).  At the end of a
// tile the 8 warps' partials are added in warp order in shared memory
// (deterministic) and rounded to bf16.
//
// Every barrier wait is bounded: a wait that gives up records
// BFP8_DEV_TIMEOUT_* in the failure word and the kernel winds down.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bfp8_devstatus.cuh"
#include "bfp8_internal.h"
#include "bfp8_ptx.cuh"

namespace bfp8 {

namespace {

constexpr int kGvWarps = 8;                 // MMA warps = k-blocks per stage
constexpr int kGvThreads = (kGvWarps + 2) * 32;   // + TMA warp + scale warp
constexpr int kGvRows = 16;                 // weight rows per tile
constexpr int kGvBoxKb = 8;                 // k-blocks per TMA box = per stage

// NG: 8-column groups of activation rows (M <= 8 * NG); CTAS: CTAs per SM;
// STAGES: depth of the ring
template <int NG, int CTAS, int STAGES>
struct GvCfg {
  static constexpr int kCtas = CTAS;
  static constexpr int kWBytes = kGvRows * kGvBoxKb * 128;      // one weight box
  static constexpr int kXBytes = 8 * NG * kGvBoxKb * 128;       // room for one activation box
  static constexpr int kStageBytes = kWBytes + kXBytes;         // 8 k-blocks
  static constexpr int kStages = STAGES;
  // stages of scales the scale warp has in flight
  static constexpr int kScAhead = kCtas >= 3 ? 2 : 4;
  // scale slot of a stage: Bs of its 8 k-blocks, then As[k-block][column]
  static constexpr int kScFloats = kGvBoxKb + kGvBoxKb * 8 * NG;
  static constexpr int kRedPitch = 8 * NG + 1;                  // padded row of partials
  static constexpr int kOffSc = kStages * kStageBytes;
  static constexpr int kOffRed = kOffSc + kStages * kScFloats * 4;
  static constexpr int kOffBar = kOffRed + kGvWarps * kGvRows * kRedPitch * 4;
  static constexpr int kSmemBytes = kOffBar + 2 * kStages * 8 + 1024;   // + alignment slack
  static_assert(kXBytes % 1024 == 0 && kWBytes % 1024 == 0, "swizzled boxes start on 1 KB");
  static_assert(kScFloats % 4 == 0 && kOffBar % 8 == 0, "slot and barrier alignment");
  static_assert(kCtas * (kSmemBytes + 1024) <= 228 * 1024, "shared memory per SM");
};

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

// Byte offset, inside a box of `rows` rows landed as [8 k-blocks][rows][128
// bytes] with the 128-byte swizzle (16-byte chunk index XOR the 128-byte line
// index mod 8, the box starting on 1 KB), of chunk c of k-block j of row r.
__device__ __forceinline__ uint32_t box_off(int r, int j, int c, int rows) {
  const int line = j * rows + r;
  return static_cast<uint32_t>(line * 128 + ((c ^ (line & 7)) << 4));
}

template <int NG, int CTAS, int STAGES>
__global__ void __launch_bounds__(kGvThreads, CTAS)
    gemv_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ GemvArgs a) {
  using C = GvCfg<NG, CTAS, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  auto bar_full = [&](int s) { return sbase + static_cast<uint32_t>(C::kOffBar + 8 * s); };
  auto bar_empty = [&](int s) {
    return sbase + static_cast<uint32_t>(C::kOffBar + 8 * (C::kStages + s));
  };
  float* sc_slots = reinterpret_cast<float*>(smem + C::kOffSc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = a.G;
  const int64_t tiles = (a.N + kGvRows - 1) / kGvRows;
  const int64_t S = (G + kGvBoxKb - 1) / kGvBoxKb;            // stages per tile
  const int64_t my_tiles =
      tiles > blockIdx.x ? (tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int64_t total = my_tiles * S;                         // stages of this CTA
  // (tile, stage) cursor over this CTA's stages
  auto advance = [&](int64_t& tile, int64_t& st) {
    if (++st == S) {
      st = 0;
      tile += gridDim.x;
    }
  };

  if (threadIdx.x == kGvWarps * 32) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_full(s), 1 + 32);          // TMA bytes + the scale warp's lanes
      mbar_init(bar_empty(s), kGvWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == kGvWarps) {
    // ------------------------------------------------------------ TMA warp
    if (lane != 0) return;
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    // bytes of a stage: the weight and activation boxes, and (as_bulk) the
    // As slice of its k-blocks that exist
    auto as_bytes = [&](int64_t st) -> uint32_t {
      if (!a.as_bulk) return 0u;
      const int64_t kbs = G - st * kGvBoxKb < kGvBoxKb ? G - st * kGvBoxKb : kGvBoxKb;
      return static_cast<uint32_t>(kbs * a.ld_as * 4);
    };
    auto stage_bytes = [&](int64_t st) {
      return static_cast<uint32_t>(C::kWBytes + a.M * kGvBoxKb * 128) + as_bytes(st);
    };
    auto issue = [&](int64_t q, int64_t tile, int64_t st, bool w, bool x) {
      const int slot = static_cast<int>(q % C::kStages);
      const uint32_t stage = sbase + static_cast<uint32_t>(slot * C::kStageBytes);
      const int32_t kb = static_cast<int32_t>(st * kGvBoxKb);
      if (w) tma_load_3d(stage, &tmW, bar_full(slot), 0, static_cast<int32_t>(tile * kGvRows), kb);
      if (x) {
        tma_load_3d(stage + C::kWBytes, &tmX, bar_full(slot), 0, 0, kb);
        if (a.as_bulk)
          bulk_load(sbase + static_cast<uint32_t>(C::kOffSc + (slot * C::kScFloats + kGvBoxKb) * 4),
                    a.As + static_cast<int64_t>(kb) * a.ld_as, as_bytes(st), bar_full(slot));
      }
    };
    int64_t q = 0, tile = blockIdx.x, st = 0;
    if (a.prefetch_b) {
      // the weights are not written by the preceding kernel: the first ring's
      // worth is requested before waiting for it; the activations only after
      const int64_t pre = total < C::kStages ? total : C::kStages;
      for (; q < pre; ++q, advance(tile, st)) {
        mbar_arrive_expect_tx(bar_full(static_cast<int>(q)), stage_bytes(st));
        issue(q, tile, st, true, false);
      }
      griddep_wait();
      int64_t t2 = blockIdx.x, s2 = 0;
      for (int64_t p = 0; p < pre; ++p, advance(t2, s2)) issue(p, t2, s2, false, true);
    } else {
      griddep_wait();
    }
    for (; q < total; ++q, advance(tile, st)) {
      const int slot = static_cast<int>(q % C::kStages);
      const uint32_t ph = static_cast<uint32_t>((q / C::kStages) & 1);
      if (!mbar_wait_bounded(bar_empty(slot), ph ^ 1u, a.wait_limit)) {
        report_failure(a.err, kDevTimeoutProducer);
        break;
      }
      mbar_arrive_expect_tx(bar_full(slot), stage_bytes(st));
      issue(q, tile, st, true, true);
    }
    // no copy may still be landing in shared memory when the CTA exits
    for (int64_t p = q > C::kStages ? q - C::kStages : 0; p < q; ++p) {
      if (!mbar_wait_bounded(bar_full(static_cast<int>(p % C::kStages)),
                             static_cast<uint32_t>((p / C::kStages) & 1), a.wait_limit)) {
        report_failure(a.err, kDevTimeoutTail);
        break;
      }
    }
    return;
  }

  if (warp == kGvWarps + 1) {
    // ---------------------------------------------------------- scale warp
    // lane holds elements lane + 32 i of each stage's slot, kD stages ahead
    constexpr int kPer = (C::kScFloats + 31) / 32;
    constexpr int kD = C::kScAhead;
    // part 1: the Bs elements (slot 0 .. 7), part 2: the As elements
    auto load = [&](int64_t tile, int64_t st, float (&o)[kPer], int part) {
      const bool live = tile < tiles;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = lane + 32 * i;
        if (e < kGvBoxKb) {
          if (part != 1) continue;
          const int64_t kb = st * kGvBoxKb + e;
          o[i] = (live && kb < G) ? __ldg(a.Bs + (tile >> 3) * G + kb) : 0.f;
        } else {
          if (part != 2 || a.as_bulk) continue;
          float v = 0.f;
          if (live && e < C::kScFloats) {
            const int kbc = (e - kGvBoxKb) / (8 * NG), m = (e - kGvBoxKb) % (8 * NG);
            const int64_t kb = st * kGvBoxKb + kbc;
            if (kb < G && m < a.M)
              v = __ldg(a.as_col_major ? a.As + kb * a.ld_as + m : a.As + m * a.ld_as + kb);
          }
          o[i] = v;
        }
      }
    };
    float v[kD][kPer];
    int64_t lt = blockIdx.x, ls = 0;
    {
      // Bs is not written by the preceding kernel: with the weight prefetch
      // its first stages are requested before waiting for it; As only after
      if (a.prefetch_b) {
        int64_t t2 = blockIdx.x, s2 = 0;
#pragma unroll
        for (int d = 0; d < kD; ++d) {
          load(t2, s2, v[d], 1);
          advance(t2, s2);
        }
      }
      griddep_wait();
#pragma unroll
      for (int d = 0; d < kD; ++d) {
        if (!a.prefetch_b) load(lt, ls, v[d], 1);
        load(lt, ls, v[d], 2);
        advance(lt, ls);
      }
    }
    for (int64_t q = 0; q < total; ++q) {
      const int slot = static_cast<int>(q % C::kStages);
      const uint32_t ph = static_cast<uint32_t>((q / C::kStages) & 1);
      if (!mbar_wait_bounded(bar_empty(slot), ph ^ 1u, a.wait_limit)) {
        report_failure(a.err, kDevTimeoutProducer);
        break;
      }
      float* dst = sc_slots + slot * C::kScFloats;
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (lane + 32 * i < (a.as_bulk ? kGvBoxKb : C::kScFloats)) dst[lane + 32 * i] = v[0][i];
      mbar_arrive(bar_full(slot));             // each lane releases its own stores
#pragma unroll
      for (int d = 0; d + 1 < kD; ++d)
#pragma unroll
        for (int i = 0; i < kPer; ++i) v[d][i] = v[d + 1][i];
      load(lt, ls, v[kD - 1], 1);
      load(lt, ls, v[kD - 1], 2);
      advance(lt, ls);
    }
    return;
  }

  // ------------------------------------------------------------- MMA warps
  const int g = lane >> 2, t = lane & 3;
  // Fragment row (and column) g holds weight row (activation row) pg: a
  // 16-byte shared load is served a quarter-warp (lanes of g = 2q, 2q + 1) at
  // a time, and pg = q, q + 4 puts those two rows four swizzle phases apart,
  // on disjoint banks.  D column c therefore belongs to activation row
  // p(c): columns 2t, 2t + 1 to rows t, t + 4 of the column group.
  const int pg = (g >> 1) + 4 * (g & 1);
  // per-lane offsets inside a stage: weight rows pg and pg + 8, chunks t and
  // t + 4 (k = 16t .., 64 + 16t ..) of k-block `warp`
  const uint32_t w0a = box_off(pg, warp, t, kGvRows);
  const uint32_t w0b = box_off(pg, warp, t + 4, kGvRows);
  const uint32_t w1a = box_off(pg + 8, warp, t, kGvRows);
  const uint32_t w1b = box_off(pg + 8, warp, t + 4, kGvRows);
  uint32_t xa[NG], xb[NG];                   // activation row 8 grp + pg (rows past M: row M-1)
#pragma unroll
  for (int grp = 0; grp < NG; ++grp) {
    const int m = (8 * grp + pg < a.M) ? 8 * grp + pg : a.M - 1;
    xa[grp] = C::kWBytes + box_off(m, warp, t, a.M);
    xb[grp] = C::kWBytes + box_off(m, warp, t + 4, a.M);
  }
  // the output belongs to the preceding kernel's stream order
  griddep_wait();
  // As of a k-block in the scale slot: the bulk-copied slice keeps the
  // caller's column stride, the scale warp packs 8 * NG columns
  const int sa_ld = a.as_bulk ? static_cast<int>(a.ld_as) : 8 * NG;
  float* red = reinterpret_cast<float*>(smem + C::kOffRed);
  float acc[NG][4];
#pragma unroll
  for (int grp = 0; grp < NG; ++grp) acc[grp][0] = acc[grp][1] = acc[grp][2] = acc[grp][3] = 0.f;
  bool ok = true;
  int64_t tile = blockIdx.x, st = 0;
  for (int64_t q = 0; q < total; ++q, advance(tile, st)) {
    const int slot = static_cast<int>(q % C::kStages);
    if (ok && !mbar_wait_bounded(bar_full(slot), static_cast<uint32_t>((q / C::kStages) & 1),
                                 a.wait_limit)) {
      report_failure(a.err, kDevTimeoutEpilogue);
      ok = false;
    }
    if (ok && st * kGvBoxKb + warp < G) {
      const uint8_t* stage = smem + slot * C::kStageBytes;
      const float* sc = sc_slots + slot * C::kScFloats;
      const float sb = sc[warp];
      const uint4 u0a = *reinterpret_cast<const uint4*>(stage + w0a);
      const uint4 u0b = *reinterpret_cast<const uint4*>(stage + w0b);
      const uint4 u1a = *reinterpret_cast<const uint4*>(stage + w1a);
      const uint4 u1b = *reinterpret_cast<const uint4*>(stage + w1b);
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) {
        const uint4 va = *reinterpret_cast<const uint4*>(stage + xa[grp]);
        const uint4 vb = *reinterpret_cast<const uint4*>(stage + xb[grp]);
        // two independent chains of two MMAs (k = 16t .. and 64 + 16t ..)
        float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
        mma_e4m3_16x8x32(d, u0a.x, u1a.x, u0a.y, u1a.y, va.x, va.y);
        mma_e4m3_16x8x32(e, u0b.x, u1b.x, u0b.y, u1b.y, vb.x, vb.y);
        mma_e4m3_16x8x32(d, u0a.z, u1a.z, u0a.w, u1a.w, va.z, va.w);
        mma_e4m3_16x8x32(e, u0b.z, u1b.z, u0b.w, u1b.w, vb.z, vb.w);
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] += e[i];
        const float* sa = sc + kGvBoxKb + warp * sa_ld + 8 * grp + t;   // rows t, t + 4
        const float s0 = __fmul_rn(sb, sa[0]), s1 = __fmul_rn(sb, sa[4]);
        acc[grp][0] = fmaf(d[0], s0, acc[grp][0]);
        acc[grp][1] = fmaf(d[1], s1, acc[grp][1]);
        acc[grp][2] = fmaf(d[2], s0, acc[grp][2]);
        acc[grp][3] = fmaf(d[3], s1, acc[grp][3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty(slot));

    if (st == S - 1) {
      // tile done: the 8 warps' partials, added in warp order
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) {
        // weight rows pg, pg + 8; activation rows 8 grp + t, 8 grp + t + 4
        float* r0 = red + (warp * kGvRows + pg) * C::kRedPitch + 8 * grp + t;
        float* r1 = r0 + 8 * C::kRedPitch;
        r0[0] = acc[grp][0];
        r0[4] = acc[grp][1];
        r1[0] = acc[grp][2];
        r1[4] = acc[grp][3];
        acc[grp][0] = acc[grp][1] = acc[grp][2] = acc[grp][3] = 0.f;
      }
      named_bar_sync(1, kGvWarps * 32);
      for (int i = threadIdx.x; i < kGvRows * 8 * NG; i += kGvWarps * 32) {
        const int m = i / kGvRows, r = i % kGvRows;     // consecutive threads: consecutive n
        float v = red[r * C::kRedPitch + m];
#pragma unroll
        for (int w = 1; w < kGvWarps; ++w) v += red[(w * kGvRows + r) * C::kRedPitch + m];
        const int64_t n = tile * kGvRows + r;
        if (ok && m < a.M && n < a.N) a.out[static_cast<int64_t>(m) * a.N + n] = __float2bfloat16_rn(v);
      }
      named_bar_sync(1, kGvWarps * 32);              // red is rewritten by the next tile
    }
  }
}

template <int NG, int CTAS, int STAGES>
cudaError_t launch_ng(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemvArgs& a,
                      int num_sms, int max_ctas, cudaStream_t stream) {
  using C = GvCfg<NG, CTAS, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NG, CTAS, STAGES>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (a.N + kGvRows - 1) / kGvRows;
  int64_t slots = static_cast<int64_t>(C::kCtas) * num_sms;           // persistent
  if (max_ctas > 0 && max_ctas < slots) slots = max_ctas;
  const int64_t blocks = tiles < slots ? tiles : slots;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kGvThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<NG, CTAS, STAGES>, tmW, tmX, a);
}

}  // namespace

cudaError_t launch_gemv(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemvArgs& a,
                        int num_sms, int max_ctas, cudaStream_t stream) {
  if (a.M < 1 || a.M > kGemvMaxM || a.N < 1 || a.G < 1 || num_sms < 1) return cudaErrorInvalidValue;
  // M <= 8: two CTAs per SM while the tiles fit in one such wave, else three
  // with a 2-stage ring (more streams per SM, a shorter last wave): measured
  // N = K = 4096 6.2 against 6.8 us, N = 5120, K = 25600 42.7 against 32.0,
  // N = 51200, K = 5120 50.3 against 44.9 (two against three).  In one wave,
  // a 4-stage ring (a 4096-deep tile in flight at once) while each SM holds
  // one tile, a 3-stage ring once SMs hold two: N = K = 4096 4.96 against
  // 5.08 us, N = 4864 5.44 against 5.63, but N = 2048 4.40 against 4.20.
  const int64_t tiles = (a.N + kGvRows - 1) / kGvRows;
  const int64_t sms = num_sms;
  switch ((a.M + 7) / 8) {
    case 1:
      if (tiles > 2 * sms) return launch_ng<1, 3, 2>(tmW, tmX, a, num_sms, max_ctas, stream);
      if (tiles > sms) return launch_ng<1, 2, 3>(tmW, tmX, a, num_sms, max_ctas, stream);
      return launch_ng<1, 2, 4>(tmW, tmX, a, num_sms, max_ctas, stream);
    case 2: return launch_ng<2, 2, 3>(tmW, tmX, a, num_sms, max_ctas, stream);
    case 3: return launch_ng<3, 2, 2>(tmW, tmX, a, num_sms, max_ctas, stream);
    default: return launch_ng<4, 1, 4>(tmW, tmX, a, num_sms, max_ctas, stream);
  }
}

}  // namespace bfp8
