// bfp8_gemm_kernel.cuh -- blocked W8A8 FP8 GEMM for sm_103a (tcgen05 + TMA).
//
//   out[m, n] = bf16( sum_kb (A[m, kb] . B[n, kb]) * As[m, kb] * Bs[n / 128, kb] )
//
// with A [M, K] and B [N, K] float8_e4m3fn (K-major), As the per-token-group
// activation scales (1 x 128) and Bs the per-tile weight scales (128 x 128), as
// in native_w8a8_block_matmul / apply_block_scaled_mm of the vLLM PR 49932
// digest ("implementation breakdown", "key source snippet").
//
// The fp32 scales are arbitrary (not powers of two), so the tensor core's
// block-scaled MMA cannot apply them.  Each 128-wide K block is therefore its
// own MMA problem: the tensor core writes the block's fp32 sum into TMEM, and
// CUDA-core warps read it back, multiply by As * Bs and add it to an fp32
// accumulator held in registers (the "promotion" of the DeepGEMM design the
// lmdeploy PR 4830 page follows for large M).
//
// Roles (one CTA per SM, persistent):
//   warps 0 .. NE-1  promotion / epilogue warps; warp w reads TMEM lanes
//                    32*(w%4) .. +31 and column half w/4
//   warp  NE         TMA producer (one lane): A/B tiles into a STAGES-deep ring,
//                    and each unit's activation-scale slice
//   warp  NE+1       TMEM owner and MMA issuer (one lane)
//   (the 256-wide tile adds two idle warps so that the non-epilogue warps form
//   a whole warpgroup that can hand registers to the epilogue via setmaxnreg)
// TMEM holds two partial buffers of BN columns (four of 128 on 128-wide
// tiles), so the MMA of block kb+1 runs while block kb is promoted.
//
// SWAP = false: MMA M slot = 128 activation rows, N slot = BN weight rows
//               (large M).
// SWAP = true:  MMA M slot = 128 weight rows, N slot = BN >= M activation rows
//               ("swap AB": the transposed schedule the lmdeploy page uses for
//               small M, so the 128-row MMA is filled by weights).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstdint>

#include "bfp8_devstatus.cuh"
#include "bfp8_e4m3.cuh"
#include "bfp8_ptx.cuh"
#include "bfp8_sched.h"

namespace bfp8 {

struct GemmArgs {
  // Tensor map over out ([M, N] bf16, box 32 x 32, 64-byte swizzle) for the
  // wide tiles' TMA stores; set when tma_store (out 16-byte aligned, N % 8 == 0).
  CUtensorMap tmO;
  int32_t tma_store;
  const float* As;       // activation scales, column-major As[kb * ld_as + m],
  int64_t ld_as;         //   16-byte aligned, ld_as % 4 == 0
  int32_t NT;            // rows of Bs = ceil(N / 128); Bs row stride = G
  const float* Bs;       // 16-byte aligned; NT * G rounded up to 4 floats readable
  __nv_bfloat16* out;    // [M, N] row-major
  int64_t M, N;
  Sched sched;
  int* counters;         // one per stream-K tile, zero between launches
  float* partials;       // grid * 2 slots of 128 x BN fp32
  int32_t vec_store;     // out rows may be written 16 bytes at a time
  int* err;              // device failure word
  unsigned long long wait_limit;  // cycles before a wait gives up
  unsigned long long* trace;      // milestone timestamps (trace builds only)
  int32_t prefetch_b;    // stream B tiles before the preceding grid completes
  // M-grouped (MoE) mode, wide tiles only: B is [experts * N, K] and Bs
  // [experts * NT, G]; rows [psum[e-1], psum[e]) use expert e (psum =
  // cumulative per-expert row counts, each a multiple of 128); rows at or
  // past psum[experts-1] are not stored.  psum == nullptr: one plain GEMM.
  const int32_t* psum;
  int32_t experts;
  // Fused epilogue (wide tiles; each promotion thread holds one 128-column
  // group of one row): y = bf16(acc), then y = bf16(y + bias[n]) when bias is
  // set; y is stored to out when store_out, and quantised per 1 x 128 group
  // into q_out / s_out when q_out is set.
  const __nv_bfloat16* bias;
  int32_t bias_vec;      // bias may be read 16 bytes at a time
  int32_t store_out;
  uint8_t* q_out;        // [M, N] e4m3 codes, row-major
  float* s_out;          // scales: s_out[g * ld_s + m] (column-major) or s_out[m * ld_s + g]
  int32_t s_col_major;
  int64_t ld_s;
  int32_t q_vec;         // q_out rows may be written 16 bytes at a time
};

constexpr int kMaxExperts = 1024;   // psum entries cached in shared memory

// Kernel variants (compile-time, so that the plain GEMM carries none of the
// others' code): the plain GEMM, the M-grouped (MoE) GEMM and the GEMM with
// the fused epilogue (the last two on wide tiles only), and the paired plain
// GEMM (256-wide tiles only): a 1-D cluster of two CTAs, the pair computing
// 256 x 256 output tiles with 2-SM MMAs (tcgen05.mma.cta_group::2, M = 256).
// Each CTA loads its 128 activation rows and half of the 256 weight rows of a
// unit (32 KB against 48 KB unpaired, the per-SM operand ingest being what
// bounds the unpaired tile); the even CTA issues the MMAs for both, and each
// CTA promotes and stores its own 128 x 256 rows from its own TMEM.
enum : int { kModePlain = 0, kModeGrouped = 1, kModeFused = 2, kModePair = 3 };

// Expert of the 128-row tile starting at row m0: the first e with psum[e] >
// m0 (psum in shared memory); past the last expert, the last one (its
// results are not stored).
__device__ __forceinline__ uint32_t expert_of(const int32_t* spsum, int32_t experts, int64_t m0) {
  int32_t lo = 0, hi = experts;
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(spsum[mid]) > m0) hi = mid;
    else lo = mid + 1;
  }
  return static_cast<uint32_t>(lo < experts ? lo : experts - 1);
}

__host__ __device__ constexpr int tmem_cols_for(int n) {
  return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 512;
}

// MR (wide tiles only): activation rows the producer loads per stage.  The
// MMA always reads 128 rows of the A operand; with MR < 128 (decode-sized M,
// M <= MR) the rows past MR are whatever follows in shared memory, their
// results land in TMEM lanes >= MR and are never read: the promotion warps
// of those lane quadrants stay idle.
template <int BN, bool SWAP, int MODE = kModePlain, int MR = 128>
struct GemmCfg {
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M=128 is 16..256 step 16");
  static_assert(SWAP || BN % 128 == 0, "wide tiles cover whole 128-column weight-scale blocks");
  static_assert(MR == 128 || (!SWAP && MODE == kModePlain && (MR == 32 || MR == 64)),
                "partial activation tiles: plain wide tiles, 32 or 64 rows");
  static constexpr int kMR = MR;
  static constexpr bool kPair = !SWAP && MODE == kModePair;
  static_assert(!kPair || (BN == 256 && MR == 128), "paired tiles: 256 wide, 128 rows per CTA");
  // promotion warps: 4 per 128 TMEM columns (16 on the 256-wide tile, 64
  // columns each, ran slower: fewer registers per thread, shallower ring)
  static constexpr int kNE = BN > 128 ? 8 : 4;
  static constexpr int kNH = kNE / 4;            // column groups per lane quadrant
  static constexpr int kCPT = BN / kNH;          // accumulator columns per thread
  static constexpr int kCH = kCPT >= 32 ? 32 : 16;   // columns per tcgen05.ld
  // columns loaded per tcgen05.wait::ld: every wait costs a full TMEM load
  // latency, so batches are as large as the register budget allows
  // (64-column swap tiles: 32, so that two CTAs' registers fit on one SM)
  // (paired tiles: 32, their scale ring and rank bookkeeping leave fewer
  // registers to the promotion warps)
  static constexpr int kBatch = (!SWAP && MODE == kModePair) ? 32
                                : kNH == 2 ? 64 : (kCPT >= 64 ? (SWAP && BN == 64 ? 32 : 64) : kCPT);
  // 8 promotion warps: 12 warps in all so that warps 8..11 are one warpgroup
  // that gives registers to the promotion warpgroups (setmaxnreg).
  static constexpr int kWarps = kNE >= 8 ? kNE + 4 : kNE + 2;
  static constexpr int kThreads = kWarps * 32;
  static constexpr bool kRebalance = kNE >= 8;
  // 8 promotion warps at 232 registers, 4 others at 40: 256*232 + 128*40 <= 384*168
  static constexpr int kRegsEpi = 232;
  static constexpr int kRegsOther = 40;
  static constexpr int kPBytes = (SWAP ? 128 : MR) * 128;
  static constexpr int kQBytes = (kPair ? BN / 2 : BN) * 128;   // paired: half the weight rows
  static constexpr int kStageBytes = kPBytes + kQBytes;
  // Scales: the producer bulk-copies each unit's activation-scale slice
  // (column-major, contiguous) into a kSR-deep ring of slots (the library
  // hands the kernel scales in that layout).  Slot layout (floats):
  //   [0, kAsFloats)                       As of the tile's rows (wide) / columns (swap)
  //   [kAsFloats, kAsFloats + 4)           swap tiles: 16-byte chunk containing Bs
  // Wide tiles read their weight scales straight from global memory instead
  // (one load per lane covers 32 units; every bulk copy added to a unit's
  // stage lengthens the producer's per-unit issue time).
  // Swap tiles: the ring has its own full / empty barriers and runs ahead of
  // the operand ring (see kSR below).  Wide tiles: unit j's slot (j mod kSR) is copied with
  // unit j's operand tiles and completes on the same stage barrier; the MMA
  // issuer waits for that barrier before the MMAs whose completion the
  // promotion warps wait for, so no barrier of its own is needed.  The slot
  // is free again once unit j - kSR has been promoted: the producer writes it
  // after the MMAs of unit j - kStages have completed, which were issued after
  // the promotion of unit j - kStages - kTB, hence kSR >= kStages + kTB.
  // Swap tiles up to 64 columns wide are sized for two CTAs per SM, so that
  // the next launch's CTAs can be resident (and stream their weights) while
  // this launch finishes; the other instantiations hold one CTA per SM.
  static constexpr bool kTwoPerSm = SWAP && BN <= 64;
  // TMEM accumulator buffers: the MMA of a unit may start while the promotion
  // warps still read the kTB - 1 units before it.  Wide tiles: two 256-column
  // or four 128-column buffers (512 columns).  Swap tiles: as many as fit in
  // 256 columns (at most 16), so that the MMAs of a CTA's units run ahead of
  // their promotion instead of waiting for it unit by unit (512 columns for
  // the one-CTA-per-SM widths).
  static constexpr int kTB = !SWAP ? (BN == 128 ? 4 : 2)
                                   : (BN <= 64 ? (256 / BN > 16 ? 16 : 256 / BN) : 512 / BN);
  // Swap tiles' scale ring runs ahead of the operand ring: the producer is at
  // most kStages units ahead of the MMAs, which are at most kTB units ahead of
  // the promotion, so kStages + kTB slots never hold it back.
  // Paired tiles use the swap tiles' ring too: a unit's stage completes on
  // the even CTA's barrier, so each CTA tracks its own scale copies.
  static constexpr bool kRing = SWAP || kPair;
  static constexpr int kSRMax = kRing ? 10 + kTB : 12;
  static constexpr int kSRB = kRing ? kSRMax : 0;   // scale-ring barriers
  static constexpr int kAsFloats = SWAP ? BN : 128;
  static constexpr int kBsChunks = SWAP ? 1 : 0;
  static constexpr int kSlotFloats = kAsFloats + 4 * kBsChunks;
  static constexpr int kSmemLimit = 232448;      // 227 KB per CTA
  // two CTAs per SM: 2 x (dynamic shared memory + 1 KB reserved) <= 228 KB
  static constexpr int kSmemBudget = kTwoPerSm ? 115712 : kSmemLimit;
  // Wide tiles stage each promotion warp's bf16 output through shared memory,
  // 32 rows x 32 columns at a time.  Plain and fused tiles: a 2 KB tile in the
  // TMA store's 64-byte swizzle (conflict-free for lane-per-row 16-byte
  // writes), stored by one 2-D TMA store.  Grouped tiles, whose rows past the
  // last expert must not be written: rows padded to 80 bytes, read back and
  // stored by the warp with row masks (whole 32-byte sectors along a row).
  static constexpr bool kTmaStore = !SWAP && MODE != kModeGrouped;
  static constexpr int kOutPitch = 80;
  static constexpr int kOutTile = kTmaStore ? 2048 : 32 * kOutPitch;
  static constexpr int kOutBytes = SWAP ? 0 : kNE * kOutTile;
  static constexpr int kPsumBytes = MODE == kModeGrouped ? kMaxExperts * 4 : 0;
  // barriers: full, empty [kStages]; sfull, sempty [kSRB]; tfull, tempty [kTB]
  static constexpr int kBarBytes = ((2 * 10 + 2 * kSRB + 2 * kTB) * 8 + 16 + 127) / 128 * 128;
  static constexpr int kStagesFit =
      (kSmemBudget - 1024 /*align*/ - kBarBytes - kSRMax * kSlotFloats * 4 - kOutBytes -
       kPsumBytes) / kStageBytes;
  static constexpr int kStages = kStagesFit > 10 ? 10 : kStagesFit;
  static_assert(kStages >= 2, "ring too small");
  static constexpr int kSR = kRing ? kStages + kTB : 12;
  static_assert(kSR <= kSRMax, "scale ring");
  static constexpr int kScaleBytes = kSR * kSlotFloats * 4;
  static_assert(SWAP || kSR >= kStages + kTB, "wide scale slots reused too early");
  static constexpr int kOffBars = kStages * kStageBytes;
  static constexpr int kOffTmemPtr = kOffBars + (2 * kStages + 2 * kSRB + 2 * kTB) * 8;
  static_assert(kOffTmemPtr + 16 - kOffBars <= kBarBytes, "barrier area");
  static constexpr int kOffFlags = kOffTmemPtr + 8;
  static constexpr int kOffScale = (kOffFlags + 8 + 15) / 16 * 16;
  static constexpr int kOffOut = (kOffScale + kScaleBytes + 1023) / 1024 * 1024;
  static constexpr int kOffPsum = kOffOut + kOutBytes;
  static constexpr int kSmemBytes = kOffPsum + kPsumBytes + 1024;
  static_assert(kSmemBytes <= kSmemBudget, "shared memory budget");
  // one CTA per SM for the other instantiations (the planner's cluster
  // capacities for them assume it)
  static_assert(kTwoPerSm || 2 * kSmemBytes > kSmemLimit + 1024, "two CTAs would fit on one SM");
  static constexpr int kTmemCols = tmem_cols_for(kTB * BN);
  // Cluster split-K: a CTA's partial tile goes into its (then idle) operand
  // ring, laid out so that the reduction reads it contiguously along the
  // output's inner dimension (n): swap tiles as [column][row] with a 132-float
  // column pitch (TMEM rows are output columns), wide tiles as [row][column]
  // with a BN + 4 float row pitch (written 16 bytes at a time; the padding
  // spreads neighbouring rows over the banks).
  static constexpr int kPartPitch = SWAP ? 132 : BN + 4;
  static constexpr int kPartLines = SWAP ? BN : 128;
  static_assert(kPartLines * kPartPitch * 4 <= kStages * kStageBytes,
                "partial tile does not fit the ring");
  static constexpr uint32_t kIdesc = idesc_e4m3_f32(kPair ? 256 : 128, BN);
};

// Optional timeline trace (compiled in only with -DBFP8_TRACE): %globaltimer
// nanoseconds at role milestones, one row of kTraceEvents per CTA.
enum : int {
  kTrStart = 0,        // after set-up
  kTrProdFirst = 1,    // producer issued its first load
  kTrProdDone = 2,     // producer issued its last load
  kTrMmaFirst = 3,     // first stage of data seen by the MMA issuer
  kTrMmaDone = 4,      // last MMA issued
  kTrEpiFirst = 5,     // first TMEM partial seen by the promotion warps
  kTrEpiLoop = 6,      // last unit promoted
  kTrEpiEnd = 7,       // promotion warps done (after fixups and stores)
  // accumulated SM cycles (not timestamps)
  kTrEpiWaitCyc = 8,   // promotion warp 0 waiting for TMEM partials
  kTrEpiWorkCyc = 9,   // promotion warp 0 from partial ready to TMEM release
  kTrMmaWaitTmem = 10, // MMA issuer waiting for a free TMEM buffer
  kTrMmaWaitData = 11, // MMA issuer waiting for operand tiles
  kTrProdWait = 12,    // producer waiting for a free stage
  kTrEpiScaleCyc = 13, // promotion warp 0 staging / waiting for scales
  kTrEpiFixCyc = 14,   // promotion warp 0 in segment epilogues (fixup + stores)
  kTrClusterSync = 15, // cluster split-K: first cluster barrier passed
  kTrProdAtSync = 16,  // producer lane reaches the first cluster barrier
  kTrMmaAtSync = 17,   // MMA lane reaches it
  kTrEpiAtSync = 18,   // promotion warp 0 reaches it (partial parked)
  kTrEpiReduced = 19,  // promotion warp 0 done with its share of the reduction
  kTrMmaLoopCyc = 20,  // SM cycles of the MMA issuer's loop (with kTrMmaFirst /
                       // kTrMmaDone: the SM clock while it ran)
  kTrSmid = 21,        // the SM the CTA ran on
  kTraceEvents = 24
};
#if defined(BFP8_TRACE)
__device__ __forceinline__ void trace_event(unsigned long long* tr, uint32_t cta, int e) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  if (tr != nullptr && cta < 1024) tr[cta * kTraceEvents + e] = t;
}
__device__ __forceinline__ void trace_value(unsigned long long* tr, uint32_t cta, int e,
                                            unsigned long long v) {
  if (tr != nullptr && cta < 1024) tr[cta * kTraceEvents + e] = v;
}
#define BFP8_CLK(var) const long long var = clock64()
#define BFP8_ACC(acc, since) acc += static_cast<unsigned long long>(clock64() - (since))
#else
__device__ __forceinline__ void trace_event(unsigned long long*, uint32_t, int) {}
__device__ __forceinline__ void trace_value(unsigned long long*, uint32_t, int, unsigned long long) {}
#define BFP8_CLK(var)
#define BFP8_ACC(acc, since)
#endif

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* v) {
  if constexpr (N == 32) {
    tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(v));
  } else {
    tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(v));
  }
}

template <int N>
__device__ __forceinline__ void reg_fence(uint32_t* v) {
  static_assert(N % 16 == 0, "");
#pragma unroll
  for (int i = 0; i < N; i += 16) reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(v + i));
}

template <int BN, bool SWAP, int MODE, int MR>
__global__ void __launch_bounds__(GemmCfg<BN, SWAP, MODE, MR>::kThreads,
                                  GemmCfg<BN, SWAP, MODE, MR>::kTwoPerSm ? 2 : 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ,
                const __grid_constant__ GemmArgs a) {
#if defined(__CUDA_ARCH__)
  using C = GemmCfg<BN, SWAP, MODE, MR>;
  static_assert(MODE == kModePlain || !SWAP, "grouped and fused variants use wide tiles");
  constexpr bool kGrouped = MODE == kModeGrouped;
  constexpr bool kFused = MODE == kModeFused;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Sched& s = a.sched;
  constexpr bool kPair = C::kPair;
  // paired tiles: the pair is the scheduling unit; rank 0 issues the MMAs
  const uint32_t prank = kPair ? cluster_ctarank() : 0u;
  const uint32_t cta = kPair ? blockIdx.x >> 1 : blockIdx.x;
  // first output row of this CTA's share of the tile at p_tile
  auto row0 = [&](uint32_t p_tile) -> int64_t {
    return kPair ? static_cast<int64_t>(p_tile) * 256 + static_cast<int64_t>(prank) * 128
                 : static_cast<int64_t>(p_tile) * 128;
  };

  auto bar_full = [&](int i) { return sbase + C::kOffBars + 8u * i; };
  auto bar_empty = [&](int i) { return sbase + C::kOffBars + 8u * (C::kStages + i); };
  auto bar_sfull = [&](int i) { return sbase + C::kOffBars + 8u * (2 * C::kStages + i); };
  auto bar_sempty = [&](int i) { return sbase + C::kOffBars + 8u * (2 * C::kStages + C::kSRB + i); };
  auto bar_tfull = [&](int b) { return sbase + C::kOffBars + 8u * (2 * C::kStages + 2 * C::kSRB + b); };
  auto bar_tempty = [&](int b) {
    return sbase + C::kOffBars + 8u * (2 * C::kStages + 2 * C::kSRB + C::kTB + b);
  };
  auto stage_p = [&](int i) { return sbase + static_cast<uint32_t>(i * C::kStageBytes); };
  auto stage_q = [&](int i) { return sbase + static_cast<uint32_t>(i * C::kStageBytes + C::kPBytes); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemPtr);
  volatile int* s_last_flag = reinterpret_cast<volatile int*>(smem + C::kOffFlags);
  // set by any role of this CTA that gives up on a wait (copies may then still
  // be in flight into shared memory when the roles end)
  volatile int* s_fail = reinterpret_cast<volatile int*>(smem + C::kOffFlags + 4);
  auto fail = [&](int code) {
    report_failure(a.err, code);
    *s_fail = 1;
  };
  uint32_t prod_issued = 0, prod_sissued = 0;   // producer lane: copies requested

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), 1);
    }
    for (int i = 0; i < C::kSRB; ++i) {
      mbar_init(bar_sfull(i), 1);
      mbar_init(bar_sempty(i), C::kNE);    // one arrival per promotion warp
    }
    for (int b = 0; b < C::kTB; ++b) {
      mbar_init(bar_tfull(b), 1);
      // one arrival per promotion warp (paired: of both CTAs, on rank 0's)
      mbar_init(bar_tempty(b), kPair ? 2 * C::kNE : C::kNE);
    }
    *s_last_flag = 0;
    *s_fail = 0;
    fence_barrier_init();
  }
  if (warp == C::kNE && lane == 0) {
    tma_prefetch_desc(&tmP);
    tma_prefetch_desc(&tmQ);
  }
  // Barriers are initialised before anyone uses them; the producer then starts
  // streaming while the MMA warp allocates TMEM.  The TMEM address reaches the
  // MMA and promotion warps through named barrier 2 (producer not included).
  __syncthreads();
  // paired tiles: both CTAs' barriers are initialised before either CTA's
  // copies or arrivals reach the other's
  if (kPair) cluster_sync();
  if (threadIdx.x == 0) {
    trace_event(a.trace, blockIdx.x, kTrStart);
#if defined(BFP8_TRACE)
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    trace_value(a.trace, blockIdx.x, kTrSmid, smid);
#endif
  }
  // Everything above overlaps the tail of the preceding kernel in the stream
  // (programmatic dependent launch).  Global memory that kernel may have
  // written (A, As, the workspace; B and Bs unless prefetch_b) is touched only
  // after this wait; the producer waits inside its loop instead.  The next
  // kernel may be launched now: it reads what this one writes only after its
  // own wait, which returns when this grid has completed.
  if (threadIdx.x == 0) griddep_launch_dependents();
  if (warp != C::kNE) griddep_wait();
  const int32_t* spsum = reinterpret_cast<const int32_t*>(smem + C::kOffPsum);
  if (kGrouped) {
    // grouped mode: every role looks experts up from a shared-memory copy of
    // psum (written by an earlier kernel, so read after the wait).  A layout
    // that is not non-decreasing multiples of 128 (one tile would mix
    // experts) is reported in the failure word and the CTA does nothing else:
    // no copy has been issued and no TMEM allocated yet (grouped mode never
    // prefetches weights), and every CTA reaches the same verdict.
    griddep_wait();
    int32_t* dst = reinterpret_cast<int32_t*>(smem + C::kOffPsum);
    for (int i = threadIdx.x; i < a.experts; i += C::kThreads) dst[i] = __ldg(a.psum + i);
    __syncthreads();
    int bad = 0;
    for (int i = threadIdx.x; i < a.experts; i += C::kThreads) {
      const int32_t prev = i > 0 ? dst[i - 1] : 0;
      if ((dst[i] & 127) != 0 || dst[i] < prev) bad = 1;
    }
    if (__syncthreads_or(bad)) {
      if (threadIdx.x == 0) report_failure(a.err, kDevBadGroupedLayout);
      return;
    }
  }
  constexpr uint32_t kTmemSyncThreads = (C::kNE + 1) * 32;
  uint32_t tmem = 0;
  if (warp == C::kNE + 1) {
    if (kPair) {
      tmem_alloc_pair(smem_addr(tmem_slot), C::kTmemCols);   // both CTAs, same address
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    named_bar_sync(2, kTmemSyncThreads);
    tc_fence_after();
    tmem = *tmem_slot;
  } else if (warp < C::kNE) {
    named_bar_sync(2, kTmemSyncThreads);
    tc_fence_after();
    tmem = *tmem_slot;
  }

  if (warp >= C::kNE) {
    if constexpr (C::kRebalance) setmaxnreg_dec<C::kRegsOther>();
    if (warp == C::kNE && lane == 0) {
      // ----------------------------------------------------- TMA producer
      Cursor cur;
      cur.init(s, cta);
      int st = 0;
      uint32_t ph = 0;
      uint32_t issued = 0;
      unsigned long long t_wait = 0;
      (void)t_wait;
      int ss = 0;
      uint32_t sph = 0;
      const uint32_t sring = smem_addr(smem + C::kOffScale);
      // Scales of the unit at c (expert e): the As slice of its rows (wide) /
      // columns (swap) and the 16-byte chunk holding each weight scale, copied
      // into ring slot `slot`, completing on barrier `bar`.
      // first row of the unit's As slice; a paired tile's second half may lie
      // wholly past M (and past ld_as): it then copies row 0's slice instead,
      // whose values no stored row uses
      auto scale_m0 = [&](const Cursor& c) -> int64_t {
        const int64_t m0 = SWAP ? static_cast<int64_t>(c.q_tile) * BN : row0(c.p_tile);
        return m0 < a.ld_as ? m0 : 0;
      };
      auto scale_as_bytes = [&](const Cursor& c) -> uint32_t {
        int64_t n_as = a.ld_as - scale_m0(c);          // stay inside the As allocation
        if (n_as > C::kAsFloats) n_as = C::kAsFloats;
        return static_cast<uint32_t>(n_as) * 4u;
      };
      auto copy_scales = [&](const Cursor& c, uint32_t e, int slot_idx, uint32_t bar) {
        const int64_t kb = c.kb;
        const uint32_t slot = sring + 4u * (slot_idx * C::kSlotFloats);
        bulk_load(slot, a.As + kb * a.ld_as + scale_m0(c), scale_as_bytes(c), bar);
#pragma unroll
        for (int h = 0; h < C::kBsChunks; ++h) {
          int64_t nb = SWAP ? static_cast<int64_t>(c.p_tile)
                            : static_cast<int64_t>(c.q_tile) * (BN / 128) + h;
          if (nb >= a.NT) nb = a.NT - 1;               // block past N: any in-bounds value
          const int64_t ei = (static_cast<int64_t>(e) * a.NT + nb) * s.G + kb;
          bulk_load(slot + 4u * (C::kAsFloats + 4 * h), a.Bs + (ei & ~int64_t{3}), 16u, bar);
        }
      };
      // wide tiles: bytes of a unit's stage barrier (operand tiles + scales;
      // paired: both CTAs' operand tiles, on rank 0's barrier)
      auto stage_tx = [&](const Cursor& c) -> uint32_t {
        if (kPair) return 2u * C::kStageBytes;
        return C::kStageBytes + (SWAP ? 0u : scale_as_bytes(c) + 16u * C::kBsChunks);
      };
      // paired: this CTA's halves of the unit, counted on rank 0's barrier
      auto pair_load_p = [&](int stg, const Cursor& c, int32_t x) {
        tma_load_2d_pair(stage_p(stg), &tmP, mapa_shared(bar_full(stg), 0), x,
                         static_cast<int32_t>(row0(c.p_tile)));
      };
      auto pair_load_q = [&](int stg, const Cursor& c, int32_t x) {
        tma_load_2d_pair(stage_q(stg), &tmQ, mapa_shared(bar_full(stg), 0), x,
                         static_cast<int32_t>(c.q_tile * BN + prank * (BN / 2)));
      };
      // With prefetch_b, the weight tiles of the first stages are requested
      // before waiting for the preceding grid; their stages are then completed
      // with the activation tiles below.
      uint32_t pre = 0;
      if (a.prefetch_b) {
        Cursor pc = cur;
        for (; pre < static_cast<uint32_t>(C::kStages) && pc.valid(); ++pre, pc.next()) {
          if (prank == 0) mbar_arrive_expect_tx(bar_full(pre), stage_tx(pc));
          const int32_t x = static_cast<int32_t>(pc.kb * 128);
          if (kPair)
            pair_load_q(static_cast<int>(pre), pc, x);
          else if (SWAP)
            tma_load_2d(stage_p(pre), &tmP, bar_full(pre), x, static_cast<int32_t>(pc.p_tile * 128));
          else
            tma_load_2d(stage_q(pre), &tmQ, bar_full(pre), x, static_cast<int32_t>(pc.q_tile * BN));
        }
      }
      griddep_wait();
      uint32_t e_tile = 0xFFFFFFFFu, e_cur = 0;   // expert of the current p tile (grouped)
      for (; cur.valid(); cur.next()) {
        BFP8_CLK(c0);
        if (kGrouped && cur.p_tile != e_tile) {
          e_tile = cur.p_tile;
          e_cur = expert_of(spsum, a.experts, static_cast<int64_t>(cur.p_tile) * 128);
        }
        // B rows of this tile's expert (grouped mode) start at e_cur * N
        const int32_t q_row = static_cast<int32_t>(static_cast<int64_t>(e_cur) * a.N) +
                              static_cast<int32_t>(cur.q_tile * BN);
        if (C::kRing) {
          if (!mbar_wait_bounded(bar_sempty(ss), sph ^ 1u, a.wait_limit)) {
            fail(kDevTimeoutProducer);
            break;
          }
          mbar_arrive_expect_tx(bar_sfull(ss), scale_as_bytes(cur) + 16u * C::kBsChunks);
          copy_scales(cur, e_cur, ss, bar_sfull(ss));
          ++prod_sissued;
          if (++ss == C::kSR) { ss = 0; sph ^= 1u; }
        }
        if (!mbar_wait_bounded(bar_empty(st), ph ^ 1u, a.wait_limit)) {
          fail(kDevTimeoutProducer);
          break;
        }
        BFP8_ACC(t_wait, c0);
        const int32_t x = static_cast<int32_t>(cur.kb * 128);
        if (issued < pre) {
          // weight tile already requested: add the activation tile
          if (kPair)
            pair_load_p(st, cur, x);
          else if (SWAP)
            tma_load_2d(stage_q(st), &tmQ, bar_full(st), x, static_cast<int32_t>(cur.q_tile * BN));
          else
            tma_load_2d(stage_p(st), &tmP, bar_full(st), x, static_cast<int32_t>(cur.p_tile * 128));
        } else if (kPair) {
          if (prank == 0) mbar_arrive_expect_tx(bar_full(st), stage_tx(cur));
          pair_load_p(st, cur, x);
          pair_load_q(st, cur, x);
        } else {
          mbar_arrive_expect_tx(bar_full(st), stage_tx(cur));
          tma_load_2d(stage_p(st), &tmP, bar_full(st), x, static_cast<int32_t>(cur.p_tile * 128));
          tma_load_2d(stage_q(st), &tmQ, bar_full(st), x, SWAP ? static_cast<int32_t>(cur.q_tile * BN) : q_row);
        }
        // wide tiles: this unit's scales complete on the same stage barrier
        if (!C::kRing) copy_scales(cur, e_cur, static_cast<int>(issued % C::kSR), bar_full(st));
        if (issued == 0) trace_event(a.trace, blockIdx.x, kTrProdFirst);
        ++issued;
        if (++st == C::kStages) { st = 0; ph ^= 1u; }
      }
      trace_event(a.trace, blockIdx.x, kTrProdDone);
      trace_value(a.trace, blockIdx.x, kTrProdWait, t_wait);
      // When every role finishes normally, every copy has landed (the MMA
      // issuer waited for each operand stage, the swap-tile promotion warps
      // for each scale slot); otherwise the copies are drained at the end.
      prod_issued = issued;
    } else if (warp == C::kNE + 1 && lane == 0) {
      // -------------------------------------------------------- MMA issuer
      // (paired tiles: rank 0 issues for both CTAs; rank 1's lane idles)
      const uint32_t n = (kPair && prank != 0) ? 0u : num_units(s, cta);
      int st = 0;
      uint32_t ph = 0;
      uint32_t done = 0;
      unsigned long long t_tmem = 0, t_data = 0;
      (void)t_tmem; (void)t_data;
      BFP8_CLK(cl0);
      for (uint32_t j = 0; j < n; ++j) {
        const int b = static_cast<int>(j % C::kTB);
        const uint32_t tph = (j / C::kTB) & 1;
        BFP8_CLK(c0);
        const bool ok_t = mbar_wait_bounded(bar_tempty(b), tph ^ 1u, a.wait_limit);
        BFP8_ACC(t_tmem, c0);
        BFP8_CLK(c1);
        if (!ok_t || !mbar_wait_bounded(bar_full(st), ph, a.wait_limit)) {
          fail(kDevTimeoutMma);
          break;
        }
        BFP8_ACC(t_data, c1);
        tc_fence_after();
        if (j == 0) trace_event(a.trace, blockIdx.x, kTrMmaFirst);
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(b * BN);
        const uint64_t adesc = sdesc_k_sw128(stage_p(st));
        const uint64_t bdesc = sdesc_k_sw128(stage_q(st));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // advancing 32 fp8 elements along K = 32 bytes = 2 descriptor units
          if (kPair)
            mma_f8f6f4_pair(d_tmem, adesc + 2u * k, bdesc + 2u * k, C::kIdesc, k > 0 ? 1u : 0u);
          else
            mma_f8f6f4(d_tmem, adesc + 2u * k, bdesc + 2u * k, C::kIdesc, k > 0 ? 1u : 0u);
        }
        if (kPair) {
          // both CTAs' stages are free and both halves of the tile are in TMEM
          mma_commit_pair(bar_empty(st), static_cast<uint16_t>(3));
          mma_commit_pair(bar_tfull(b), static_cast<uint16_t>(3));
        } else {
          mma_commit(bar_empty(st));
          mma_commit(bar_tfull(b));
        }
        done = j + 1;
        if (++st == C::kStages) { st = 0; ph ^= 1u; }
      }
      trace_event(a.trace, blockIdx.x, kTrMmaDone);
      trace_value(a.trace, blockIdx.x, kTrMmaWaitTmem, t_tmem);
      trace_value(a.trace, blockIdx.x, kTrMmaWaitData, t_data);
#if defined(BFP8_TRACE)
      trace_value(a.trace, blockIdx.x, kTrMmaLoopCyc, static_cast<unsigned long long>(clock64() - cl0));
#endif
      // The last commit fires when every MMA issued above has completed.
      if (done > 0 && done < n) {
        const uint32_t j = done - 1;
        if (!mbar_wait_bounded(bar_tfull(static_cast<int>(j % C::kTB)), (j / C::kTB) & 1, a.wait_limit))
          fail(kDevTimeoutTail);
      }
    }
    __syncwarp();
    if (s.cluster > 1) {
      // every thread of the cluster takes part in both cluster barriers of
      // the split-K reduction (see the promotion warps)
      if (lane == 0 && warp == C::kNE) trace_event(a.trace, blockIdx.x, kTrProdAtSync);
      if (lane == 0 && warp == C::kNE + 1) trace_event(a.trace, blockIdx.x, kTrMmaAtSync);
      cluster_sync();
      cluster_sync_relaxed();
    }
  } else {
    // ---------------------------------------------- promotion and epilogue
    if constexpr (C::kRebalance) setmaxnreg_inc<C::kRegsEpi>();
    const int quad = warp & 3;
    const int half = warp >> 2;
    const int r = quad * 32 + lane;          // TMEM lane = row of the P tile
    const int col0 = half * C::kCPT;         // first TMEM column of this thread
    const int etid = threadIdx.x;            // 0 .. NE*32-1
    // partial activation tiles: warps whose lane quadrant holds no loaded row
    // skip the TMEM reads and FMAs (their rows are never stored)
    const bool idle = MR < 128 && quad * 32 >= MR;
    const float* sRing = reinterpret_cast<const float*>(smem + C::kOffScale);
    int ss = 0;
    uint32_t sph = 0;
    // fp32 accumulators, one per column of this thread's TMEM lane
    constexpr int kP = C::kCPT / 2;          // column pairs
    float acc[C::kCPT];
#pragma unroll
    for (int i = 0; i < C::kCPT; ++i) acc[i] = 0.f;

    Cursor cur;
    cur.init(s, cta);
    // rows that are stored: grouped mode stops at the end of the last expert
    const int64_t m_lim =
        (kGrouped && a.M > spsum[a.experts - 1]) ? spsum[a.experts - 1] : a.M;
    uint32_t e_tile = 0xFFFFFFFFu, e_cur = 0;      // expert of the current p tile (grouped)
    // Wide tiles: lane i holds the weight scale of this thread's column block
    // for k-block kb_win + i (loaded at each segment start and every 32
    // units; a shuffle hands each unit's value to the whole warp)
    float bs_win = 0.f;
    uint32_t kb_win = 0;

    unsigned long long t_ewait = 0, t_ework = 0, t_escale = 0, t_efix = 0;
    (void)t_ewait; (void)t_ework; (void)t_escale; (void)t_efix;
    for (; cur.valid(); cur.next()) {
      BFP8_CLK(e0);
      const uint32_t j = cur.j;
      float sr = 0.f;           // row scale (wide: As * Bs; swap: Bs)
      const float* sq = nullptr;              // column scales (swap)
      if (!SWAP) {
        if (kGrouped && cur.p_tile != e_tile) {
          e_tile = cur.p_tile;
          e_cur = expert_of(spsum, a.experts, static_cast<int64_t>(cur.p_tile) * 128);
        }
        if (cur.first() || cur.kb >= kb_win + 32) {
          kb_win = cur.kb;
          const uint32_t nb = cur.q_tile * (BN / 128) + static_cast<uint32_t>(col0 / 128);
          const uint32_t kbl = kb_win + static_cast<uint32_t>(lane);
          bs_win = (nb < static_cast<uint32_t>(a.NT) && kbl < s.G)
                       ? __ldg(a.Bs + (static_cast<int64_t>(e_cur) * a.NT + nb) * s.G + kbl)
                       : 0.f;   // columns past N are not stored
        }
        // paired tiles: this CTA's As slice comes through its own ring
        if (kPair && !mbar_wait_bounded(bar_sfull(ss), sph, a.wait_limit)) {
          fail(kDevTimeoutEpilogue);
          break;
        }
      } else {
        if (!mbar_wait_bounded(bar_sfull(ss), sph, a.wait_limit)) {
          fail(kDevTimeoutEpilogue);
          break;
        }
        const float* slot = sRing + ss * C::kSlotFloats;
        sr = slot[C::kAsFloats + ((cur.p_tile * s.G + cur.kb) & 3)];
        sq = slot + col0;
      }
      BFP8_ACC(t_escale, e0);
      BFP8_CLK(e1);
      const int b = static_cast<int>(j % C::kTB);
      if (!mbar_wait_bounded(bar_tfull(b), (j / C::kTB) & 1, a.wait_limit)) {
        fail(kDevTimeoutEpilogue);
        break;
      }
      tc_fence_after();
      BFP8_ACC(t_ewait, e1);
      BFP8_CLK(e2);
      if (j == 0 && etid == 0) trace_event(a.trace, blockIdx.x, kTrEpiFirst);
      if (j + 1 == cur.n && etid == 0) trace_event(a.trace, blockIdx.x, kTrEpiLoop);

      if (cur.first()) {
#pragma unroll
        for (int i = 0; i < C::kCPT; ++i) acc[i] = 0.f;
      }
      const uint32_t taddr = tmem + static_cast<uint32_t>(b * BN + col0) +
                             (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll
      for (int c0 = 0; c0 < (idle ? 0 : C::kCPT); c0 += C::kBatch) {
        uint32_t v[C::kBatch];
#pragma unroll
        for (int h = 0; h < C::kBatch; h += C::kCH) tmem_ld_cols<C::kCH>(taddr + c0 + h, v + h);
        if (!SWAP && c0 == 0) {
          // wide tiles: the scale slot landed before the MMAs were issued; it
          // is read while the first TMEM loads are in flight
          const float* slot = sRing + (kPair ? ss : static_cast<int>(j % C::kSR)) * C::kSlotFloats;
          const float bsv = __shfl_sync(0xffffffffu, bs_win, static_cast<int>(cur.kb - kb_win));
          sr = slot[r] * bsv;
        }
        tmem_wait_ld();
        reg_fence<C::kBatch>(v);
        // element (row r, column c) gets scale sr (wide) or sr * As[c] (swap);
        // two columns per packed fp32x2 FMA (one instruction, two IEEE FMAs)
        const uint64_t sr2 = pack_u32x2(__float_as_uint(sr), __float_as_uint(sr));
#pragma unroll
        for (int i = 0; i < C::kBatch; i += 2) {
          uint64_t sc2 = sr2;
          if (SWAP) {
            const float2 q2 = *reinterpret_cast<const float2*>(sq + c0 + i);
            sc2 = mul_f32x2(sr2, pack_u32x2(__float_as_uint(q2.x), __float_as_uint(q2.y)));
          }
          const uint64_t a2 =
              pack_u32x2(__float_as_uint(acc[c0 + i]), __float_as_uint(acc[c0 + i + 1]));
          unpack_f32x2(fma_f32x2(pack_u32x2(v[i], v[i + 1]), sc2, a2), acc[c0 + i],
                       acc[c0 + i + 1]);
        }
      }
      // every lane's TMEM reads are complete (wait::ld above); order them before
      // the release, then one lane per warp arrives
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // paired tiles: the buffer is free once both CTAs' warps have read it;
        // rank 0's MMA lane counts them on its barrier
        if (kPair) mbar_arrive_cluster(mapa_shared(bar_tempty(b), 0));
        else mbar_arrive(bar_tempty(b));
        if (C::kRing) mbar_arrive(bar_sempty(ss));
      }
      if (C::kRing) {
        if (++ss == C::kSR) { ss = 0; sph ^= 1u; }
      }
      BFP8_ACC(t_ework, e2);

      if (!cur.last()) continue;
      BFP8_CLK(e3);

      if (s.cluster > 1) {
        // cluster split-K: park this CTA's partial tile in its own shared
        // memory; the cluster adds the partials after the loop.  Every MMA
        // has completed (tfull of the last unit), so the operand ring is idle.
        float* part = reinterpret_cast<float*>(smem);
        if (SWAP) {
#pragma unroll
          for (int i = 0; i < C::kCPT; ++i) part[(col0 + i) * C::kPartPitch + r] = acc[i];
        } else {
          float4* row = reinterpret_cast<float4*>(part + r * C::kPartPitch + col0);
#pragma unroll
          for (int i = 0; i < C::kCPT / 4; ++i)
            row[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
        }
        BFP8_ACC(t_efix, e3);
        continue;
      }

      // ---- the segment is complete: emit it
      const int32_t ts = cur.sk_tile();
      uint32_t pf = cta, pl = cta;
      if (ts >= 0) {
        pf = sk_first_cta(s, ts);
        pl = sk_last_cta(s, ts);
      }
      if (pl > pf) {
        // stream-K fixup: publish this CTA's partial, the last arrival adds all.
        // Partial layout: column pairs interleaved, pair k of row r at
        // [(k * 128 + r) * 2, +2), so each lane moves 8 contiguous bytes.
        auto part = [&](uint32_t pp) {
          return reinterpret_cast<float2*>(
                     a.partials + static_cast<size_t>(pp * 2 + sk_slot(s, pp, ts)) * (128 * BN)) +
                 (col0 / 2) * 128 + r;
        };
        float2* mine = part(cta);
#pragma unroll
        for (int k = 0; k < kP; ++k) mine[k * 128] = make_float2(acc[2 * k], acc[2 * k + 1]);
        __threadfence();
        named_bar_sync(1, C::kNE * 32);
        if (etid == 0) {
          const int old = atomicAdd(a.counters + ts, 1);
          *s_last_flag = (old == static_cast<int>(pl - pf)) ? 1 : 0;
        }
        named_bar_sync(1, C::kNE * 32);
        const bool is_last = *s_last_flag != 0;
        if (!is_last) {
          BFP8_ACC(t_efix, e3);
          continue;
        }
        __threadfence();
        // Sum the contributors in ascending K order; each contributor's pairs
        // are loaded in chunks of kFixPairs so one L2 round trip serves many.
        constexpr int kFixPairs = C::kNH >= 2 ? 16 : (kP >= 32 ? 32 : kP);
        {
          const float2* p0 = part(pf);
#pragma unroll
          for (int k = 0; k < kP; ++k) {
            const float2 t = __ldcg(p0 + k * 128);
            acc[2 * k] = t.x;
            acc[2 * k + 1] = t.y;
          }
        }
#pragma unroll 1
        for (uint32_t pp = pf + 1; pp <= pl; ++pp) {
          const float2* pq = part(pp);
#pragma unroll
          for (int k0 = 0; k0 < kP; k0 += kFixPairs) {
            float2 t[kFixPairs];
#pragma unroll
            for (int k = 0; k < kFixPairs; ++k) t[k] = __ldcg(pq + (k0 + k) * 128);
#pragma unroll
            for (int k = 0; k < kFixPairs; ++k) {
              acc[2 * (k0 + k)] += t[k].x;
              acc[2 * (k0 + k) + 1] += t[k].y;
            }
          }
        }
        if (etid == 0) a.counters[ts] = 0;  // every contributor has arrived
      }

      if (kFused) {
        static_assert(SWAP || C::kCPT == 128, "fused epilogue: one 128-column group per thread");
        // ---- fused epilogue: bias, then the next layer's group quantisation
        const int64_t m = static_cast<int64_t>(cur.p_tile) * 128 + r;
        const int64_t nbase = static_cast<int64_t>(cur.q_tile) * BN + col0;
        const int64_t nv = a.N - nbase < 128 ? a.N - nbase : 128;   // columns in range
#pragma unroll
        for (int i = 0; i < C::kCPT; ++i) acc[i] = __bfloat162float(__float2bfloat16_rn(acc[i]));
        if (a.bias != nullptr && nv > 0) {
          if (a.bias_vec && nv == 128) {
#pragma unroll
            for (int g = 0; g < 16; ++g) {
              const uint4 w = __ldg(reinterpret_cast<const uint4*>(a.bias + nbase) + g);
              const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const float b0 = __uint_as_float(ww[h] << 16);
                const float b1 = __uint_as_float(ww[h] & 0xFFFF0000u);
                acc[8 * g + 2 * h] =
                    __bfloat162float(__float2bfloat16_rn(__fadd_rn(acc[8 * g + 2 * h], b0)));
                acc[8 * g + 2 * h + 1] =
                    __bfloat162float(__float2bfloat16_rn(__fadd_rn(acc[8 * g + 2 * h + 1], b1)));
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < C::kCPT; ++i)
              if (i < nv)
                acc[i] = __bfloat162float(
                    __float2bfloat16_rn(__fadd_rn(acc[i], __bfloat162float(a.bias[nbase + i]))));
          }
        }
        if (a.q_out != nullptr) {
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < C::kCPT; ++i)
            if (i < nv) amax = fmaxf(amax, fabsf(acc[i]));
          const float scale = group_scale(amax);
          const E4m3Bracket br(scale);
          uint32_t codes[C::kCPT / 4];
          uint64_t undecided = 0;             // one bit per pair of columns
#pragma unroll
          for (int i = 0; i < C::kCPT; i += 4) {
            bool u0 = false, u1 = false;
            const uint32_t lo = e4m3_pair_bracketed(acc[i], acc[i + 1], br, u0);
            const uint32_t hi = e4m3_pair_bracketed(acc[i + 2], acc[i + 3], br, u1);
            codes[i / 4] = lo | (hi << 16);
            undecided |= (static_cast<uint64_t>(u0) << (i / 2)) |
                         (static_cast<uint64_t>(u1) << (i / 2 + 1));
          }
          // warp-uniform branch: IEEE divisions only for the undecided pairs
          if (__any_sync(0xffffffffu, undecided != 0)) {
#pragma unroll
            for (int i = 0; i < C::kCPT; i += 2) {
              if (undecided & (uint64_t{1} << (i / 2))) {
                const uint32_t c = e4m3_pair_divided(acc[i], acc[i + 1], scale);
                const int sh = (i & 2) * 8;
                codes[i / 4] = (codes[i / 4] & ~(0xFFFFu << sh)) | (c << sh);
              }
            }
          }
          if (m < m_lim && nv > 0) {
            uint8_t* qrow = a.q_out + m * a.N + nbase;
            if (a.q_vec && nv == 128) {
#pragma unroll
              for (int g = 0; g < C::kCPT / 16; ++g)
                st_global_v4(qrow + 16 * g, codes[4 * g], codes[4 * g + 1], codes[4 * g + 2],
                             codes[4 * g + 3]);
            } else {
#pragma unroll
              for (int i = 0; i < C::kCPT; ++i)
                if (i < nv) qrow[i] = static_cast<uint8_t>(codes[i / 4] >> (8 * (i & 3)));
            }
            const int64_t g = nbase / 128;
            if (a.s_col_major) a.s_out[g * a.ld_s + m] = scale;
            else a.s_out[m * a.ld_s + g] = scale;
          }
        }
      }
      if (kFused && !a.store_out) {
        // fused epilogue without the bf16 output
      } else if (C::kTmaStore && a.tma_store && idle) {
        // no row of this warp is stored
      } else if (C::kTmaStore && a.tma_store) {
        // rows of 16-byte-aligned bf16: 32 columns at a time into this warp's
        // 2 KB tile (16-byte chunk c of row i at 64 i + 16 (c ^ ((i >> 1) & 3)),
        // the 64-byte swizzle), then one TMA store of the 32 x 32 box; rows
        // past M and columns past N are not written
        uint8_t* stg = smem + C::kOffOut + warp * C::kOutTile;
        const uint32_t stg_s = smem_addr(stg);
        const int32_t y = static_cast<int32_t>(row0(cur.p_tile) + quad * 32);
        const int32_t x0 = static_cast<int32_t>(cur.q_tile * BN + col0);
#pragma unroll
        for (int ch = 0; ch < C::kCPT; ch += 32) {
          if (lane == 0) bulk_wait_group_read<0>();   // the previous store has read the tile
          __syncwarp();
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const float* f = acc + ch + 8 * g;
            *reinterpret_cast<uint4*>(stg + lane * 64 + 16 * (g ^ ((lane >> 1) & 3))) =
                make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                           pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
          }
          fence_proxy_async_smem();                  // generic writes -> TMA reads
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&a.tmO, stg_s, x0 + ch, y);
            bulk_commit_group();
          }
        }
      } else if (!SWAP && a.vec_store) {
        // rows of 16-byte-aligned bf16 (N % 8 == 0): through this warp's
        // staging rows, 32 columns at a time; lanes 4i..4i+3 then store one
        // row's 64 contiguous bytes
        uint8_t* stg = smem + C::kOffOut + warp * C::kOutTile;
        const int64_t mrow0 = row0(cur.p_tile) + quad * 32;
        const int64_t nbase = static_cast<int64_t>(cur.q_tile) * BN + col0;
#pragma unroll
        for (int ch = 0; ch < C::kCPT; ch += 32) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const float* f = acc + ch + 8 * g;
            *reinterpret_cast<uint4*>(stg + lane * C::kOutPitch + 16 * g) =
                make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                           pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int pce = i * 32 + lane;
            const int row = pce >> 2, c16 = pce & 3;
            const uint4 w = *reinterpret_cast<const uint4*>(stg + row * C::kOutPitch + 16 * c16);
            const int64_t m = mrow0 + row;
            const int64_t n = nbase + ch + 8 * c16;
            if (m < m_lim && n < a.N) st_global_v4(a.out + m * a.N + n, w.x, w.y, w.z, w.w);
          }
          __syncwarp();
        }
      } else if (!SWAP) {
        const int64_t m = row0(cur.p_tile) + r;
        if (m < m_lim) {
          __nv_bfloat16* row = a.out + m * a.N;
          const int64_t nbase = static_cast<int64_t>(cur.q_tile) * BN + col0;
#pragma unroll
          for (int g = 0; g < C::kCPT / 8; ++g) {
            const int64_t n = nbase + g * 8;
            const float* f = acc + g * 8;
            if (a.vec_store && n + 8 <= a.N) {
              st_global_v4(row + n, pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                           pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (n + i < a.N) row[n + i] = __float2bfloat16_rn(f[i]);
            }
          }
        }
      } else {
        const int64_t n = static_cast<int64_t>(cur.p_tile) * 128 + r;
        if (n < a.N) {
          const int64_t mbase = static_cast<int64_t>(cur.q_tile) * BN + col0;
#pragma unroll
          for (int c = 0; c < C::kCPT; ++c) {
            const int64_t m = mbase + c;
            if (m < a.M) a.out[m * a.N + n] = __float2bfloat16_rn(acc[c]);
          }
        }
      }
      BFP8_ACC(t_efix, e3);
    }
    // this warp's TMA stores have completed (their staging tile is read and
    // the output written) before the CTA ends
    if (C::kTmaStore && lane == 0) bulk_wait_group<0>();
    if (s.cluster > 1) {
      // ---- cluster split-K reduction.  After the first cluster barrier every
      // CTA's partial is in its shared memory.  The output tile's valid part,
      // cut into runs of 4 elements along n, is divided evenly among the
      // cluster's CTAs; each adds the cs partials of its runs in rank order
      // (deterministic) through distributed shared memory and stores bf16.
      // The second barrier (relaxed: it orders nothing) keeps every CTA and
      // its shared memory alive until all reads of it are done.
      if (etid == 0) trace_event(a.trace, blockIdx.x, kTrEpiAtSync);
      cluster_sync();
      if (etid == 0) trace_event(a.trace, blockIdx.x, kTrClusterSync);
      BFP8_CLK(e4);
      const uint32_t cs = s.cluster;
      const uint32_t rank = cta % cs;            // 1-D clusters of consecutive CTAs
      const uint32_t tile = cta / cs;
      const uint32_t q_tile = tile / s.p_tiles;
      const uint32_t p_tile = tile - q_tile * s.p_tiles;
      const int64_t p0 = static_cast<int64_t>(p_tile) * 128;   // first row (TMEM lane)
      const int64_t q0 = static_cast<int64_t>(q_tile) * BN;    // first column
      const int64_t qlim = SWAP ? a.M : a.N;
      const int64_t plim = SWAP ? a.N : m_lim;
      const uint32_t qv = static_cast<uint32_t>(qlim - q0 < BN ? qlim - q0 : BN);
      const uint32_t pv = static_cast<uint32_t>(plim - p0 < 128 ? plim - p0 : 128);
      // swap: runs of 4 TMEM rows in each valid column; wide: runs of 4
      // columns in each valid row
      const uint32_t runs_per_line = SWAP ? (pv + 3) / 4 : (qv + 3) / 4;
      const uint32_t items = (SWAP ? qv : pv) * runs_per_line;
      const uint32_t beg = rank * items / cs;         // items <= 256 * 32: no overflow
      const uint32_t end = (rank + 1) * items / cs;
      const uint32_t part0 = smem_addr(smem);
      // kU runs per thread per round, all their loads issued before any is
      // used: distributed shared memory has a long round trip.
      constexpr int kU = 4;
      constexpr uint32_t kStride = C::kNE * 32;
      for (uint32_t i0 = beg + etid; i0 < end; i0 += kU * kStride) {
        uint32_t addr[kU];
        uint32_t cc[kU], rr[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const uint32_t i = i0 + u * kStride;
          // lanes walk along n: swap, down a column of TMEM rows; wide, across
          // the columns of one row
          const uint32_t line = i / runs_per_line;
          const uint32_t off4 = (i - line * runs_per_line) * 4;
          cc[u] = line;
          rr[u] = off4;
          addr[u] = part0 + 4u * (line * C::kPartPitch + off4);
        }
        // every rank's values are requested before any is added (one
        // distributed-shared-memory round trip), then summed in rank order
        float4 t[8][kU];
#pragma unroll
        for (uint32_t q = 0; q < 8; ++q)
#pragma unroll
          for (int u = 0; u < kU; ++u)
            if (q < cs && i0 + u * kStride < end) t[q][u] = ld_dsmem_v4(mapa_shared(addr[u], q));
        float4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) v[u] = t[0][u];
#pragma unroll
        for (uint32_t q = 1; q < 8; ++q) {
          if (q >= cs) break;
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            v[u].x += t[q][u].x;
            v[u].y += t[q][u].y;
            v[u].z += t[q][u].z;
            v[u].w += t[q][u].w;
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          if (i0 + u * kStride >= end) continue;
          const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          // output row m and first column n of the run
          const int64_t m = SWAP ? q0 + cc[u] : p0 + cc[u];
          const int64_t n = SWAP ? p0 + rr[u] : q0 + rr[u];
          __nv_bfloat16* row = a.out + m * a.N;
          if (a.vec_store && n + 4 <= a.N) {
            st_global_v2(row + n, pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (n + e < a.N) row[n + e] = __float2bfloat16_rn(f[e]);
          }
        }
      }
      BFP8_ACC(t_efix, e4);
      if (etid == 0) trace_event(a.trace, blockIdx.x, kTrEpiReduced);
      cluster_sync_relaxed();
    }
    if (etid == 0) {
      trace_event(a.trace, blockIdx.x, kTrEpiEnd);
      trace_value(a.trace, blockIdx.x, kTrEpiWaitCyc, t_ewait);
      trace_value(a.trace, blockIdx.x, kTrEpiWorkCyc, t_ework);
      trace_value(a.trace, blockIdx.x, kTrEpiScaleCyc, t_escale);
      trace_value(a.trace, blockIdx.x, kTrEpiFixCyc, t_efix);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kNE && lane == 0 && *s_fail) {
    // a role gave up: do not leave while copies into this CTA's shared memory
    // may still be in flight (paired tiles: rank 0's stage barriers count
    // both CTAs' operand copies, and rank 1 leaves only after the closing
    // cluster barrier, which rank 0 reaches after draining them)
    const uint32_t tail = (kPair && prank != 0) ? 0u
                          : (prod_issued < static_cast<uint32_t>(C::kStages) ? prod_issued : C::kStages);
    for (uint32_t t = 0; t < tail; ++t) {
      const uint32_t j = prod_issued - 1 - t;
      if (!mbar_wait_bounded(bar_full(j % C::kStages), (j / C::kStages) & 1u, a.wait_limit)) {
        report_failure(a.err, kDevTimeoutTail);
        break;
      }
    }
    const uint32_t stail = prod_sissued < static_cast<uint32_t>(C::kSR) ? prod_sissued : C::kSR;
    for (uint32_t t = 0; t < stail; ++t) {
      const uint32_t j = prod_sissued - 1 - t;
      if (!mbar_wait_bounded(bar_sfull(j % C::kSR), (j / C::kSR) & 1u, a.wait_limit)) {
        report_failure(a.err, kDevTimeoutTail);
        break;
      }
    }
  }
  if (kPair) {
    // rank 0's MMAs read rank 1's shared memory and both CTAs arrive on rank
    // 0's barriers: neither leaves (nor frees the pair's TMEM) before both
    // are done
    cluster_sync();
    if (warp == C::kNE + 1) tmem_dealloc_pair(tmem, C::kTmemCols);
  } else if (warp == C::kNE + 1) {
    tmem_dealloc(tmem, C::kTmemCols);
  }
#endif
}

// Host side.  The dynamic shared-memory opt-in is per device and set once (a
// launch captured into a CUDA graph then needs no attribute call).
template <int BN, bool SWAP, int MODE = kModePlain, int MR = 128>
cudaError_t configure_instance() {
  using C = GemmCfg<BN, SWAP, MODE, MR>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemm_kernel<BN, SWAP, MODE, MR>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  return cudaSuccess;
}

// How many clusters of `cs` CTAs of this instantiation the current device
// runs at once (the GPCs' sizes decide it, not just the SM count).
template <int BN, bool SWAP>
cudaError_t cluster_capacity_instance(int cs, int* clusters) {
  using C = GemmCfg<BN, SWAP>;
  cudaError_t e = configure_instance<BN, SWAP, kModePlain>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(cs);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, gemm_kernel<BN, SWAP, kModePlain, 128>, &cfg);
}

// Launches one instantiation with programmatic dependent launch (the
// prologue may overlap the preceding kernel in the stream; the kernel waits
// for it before reading its inputs) and, for cluster split-K, as 1-D
// clusters of sched.cluster consecutive CTAs.
template <int BN, bool SWAP, int MODE = kModePlain, int MR = 128>
cudaError_t launch_instance(const CUtensorMap& tmP, const CUtensorMap& tmQ, const GemmArgs& a,
                            cudaStream_t stream) {
  using C = GemmCfg<BN, SWAP, MODE, MR>;
  cudaError_t e = configure_instance<BN, SWAP, MODE, MR>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  // paired tiles: sched.grid counts pairs; each is a 1-D cluster of two CTAs
  cfg.gridDim = dim3(a.sched.grid * (C::kPair ? 2u : 1u));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (C::kPair || a.sched.cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = C::kPair ? 2u : a.sched.cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, gemm_kernel<BN, SWAP, MODE, MR>, tmP, tmQ, a);
}

}  // namespace bfp8
