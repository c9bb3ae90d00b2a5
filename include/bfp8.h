/*
 * bfp8.h -- libbfp8: DeepSeek-style blocked W8A8 FP8 linear layer on GB300
 * (sm_103a).  Plain C ABI: raw pointers, sizes and an opaque stream handle.
 *
 * The layer has two steps (vLLM PR 49932 digest, "implementation breakdown"
 * and "key source snippet"; lmdeploy PR 4830, "Kernel design"):
 *   1. per-token group quantisation of the activations to float8_e4m3fn in
 *      1 x 128 groups, with one fp32 scale per group (amax / 448);
 *   2. the block-scaled GEMM
 *        out[m, n] = sum over 128-wide K blocks kb of
 *                    (A[m, kb] . B[n, kb]) * As[m, kb] * Bs[n / 128, kb]
 *      with 128 x 128 weight-scale tiles and a bf16 output.
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device (or managed) addresses on the current
 *     device; the caller owns every buffer, including the GEMM workspace.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls only enqueue work: they neither allocate device memory
 *     nor synchronise.
 *   - Every argument is validated on the host before anything is launched; a
 *     rejected call returns a status other than BFP8_OK, launches nothing and
 *     leaves a reason in bfp8_last_error().  Nothing is thrown across the ABI.
 *   - Inputs must be finite.  NaN or infinite inputs give unspecified outputs
 *     (never a fault).
 *   - Only GB300-class devices (compute capability 10.3) are supported.
 */
#ifndef BFP8_H_
#define BFP8_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BFP8_VERSION 1

typedef enum {
  BFP8_OK = 0,
  BFP8_ERR_INVALID_ARG = 1,     /* null pointer, bad size, bad leading dimension */
  BFP8_ERR_ALIGNMENT = 2,       /* a pointer or stride breaks a stated alignment rule */
  BFP8_ERR_UNSUPPORTED = 3,     /* no device, or a device that is not sm_103 */
  BFP8_ERR_CUDA = 4,            /* a CUDA runtime / driver call failed */
  BFP8_ERR_WORKSPACE = 5,       /* workspace missing, too small or misaligned */
  BFP8_ERR_DEVICE_TIMEOUT = 6   /* a kernel-side wait gave up (see bfp8_device_status) */
} bfp8_status;

typedef enum { BFP8_IN_BF16 = 0, BFP8_IN_F32 = 1 } bfp8_in_dtype;

/* ------------------------------------------------------------------------ */
/* Step 1: per-token group quantisation                                      */
/* ------------------------------------------------------------------------ */

/*
 * bfp8_group_quant -- per_token_group_quant_fp8(x, group_size=128,
 * column_major_scales) as called in the vLLM PR 49932 digest's test.
 *
 *   x      [M, K] row-major activations, bf16 or fp32 (in_dtype), leading
 *          dimension ld_x elements (ld_x >= K).
 *   group  must be 128 (the only activation block shape the pages use).
 *   q      [M, K] float8_e4m3fn codes, leading dimension ld_q bytes (>= K).
 *   s      G = ceil(K / 128) fp32 scales per row:
 *            col_major = 0: s[m * ld_s + g], ld_s >= G
 *            col_major = 1: s[g * ld_s + m], ld_s >= M
 *          (bfp8_scale_ld(M) gives the 16-byte-aligned column-major stride the
 *          GEMM prefers).  Entries of a padded layout that hold no scale are
 *          not written.
 * For each group: amax = max |x| over the group's real elements (the last
 * group of a row has K - 128 * (G - 1) elements), scale = max(amax, 1e-10)
 * / 448 (IEEE fp32 division), q = round-to-nearest-even, saturating
 * e4m3(x / scale) with an IEEE fp32 division per element; a zero or an
 * underflow to zero keeps its sign.
 * Any M >= 0 and K >= 0 (empty inputs launch nothing).  No alignment is
 * required; 16-byte aligned rows take the vectorised path.
 */
bfp8_status bfp8_group_quant(const void* x, int in_dtype, int64_t M, int64_t K, int64_t ld_x,
                             int group, int col_major, void* q, int64_t ld_q, float* s,
                             int64_t ld_s, void* stream);

/* ------------------------------------------------------------------------ */
/* UE8M0 scale variant                                                       */
/* ------------------------------------------------------------------------ */

/*
 * The transformers DeepGEMM integration (`_ceil_to_ue8m0`, and
 * `_select_fp8_cast_kwargs` with use_ue8m0) rounds every fp32 scale UP to the
 * nearest power of two -- the UE8M0 format keeps only the biased exponent --
 * for the SM100 kernels.  That is a different function from the fp32-scale
 * layer above: activations are quantised with the rounded scale, and weight
 * scales are rounded the same way.  The blocked GEMM below computes it as it
 * stands (bfp8_gemm with such As and Bs); the scales stay fp32 values.
 */
typedef enum { BFP8_SCALE_FP32 = 0, BFP8_SCALE_UE8M0 = 1 } bfp8_scale_fmt;

/* bfp8_group_quant with a choice of scale format.  BFP8_SCALE_FP32: as
 * bfp8_group_quant.  BFP8_SCALE_UE8M0: each group's scale max(amax, 1e-10) /
 * 448 (IEEE fp32 division) is rounded up to a power of two (2^-42 for an
 * all-zero group), and q = e4m3(x / scale) with the quotient exact; |x / scale|
 * <= 448, so no code saturates.  Other arguments, layouts and errors as for
 * bfp8_group_quant; BFP8_ERR_INVALID_ARG for another scale_fmt. */
bfp8_status bfp8_group_quant_ex(const void* x, int in_dtype, int64_t M, int64_t K, int64_t ld_x,
                                int group, int col_major, int scale_fmt, void* q, int64_t ld_q,
                                float* s, int64_t ld_s, void* stream);

/* out[i] = in[i] rounded up to the nearest power of two, for n >= 0 positive
 * finite fp32 scales (e.g. a weight-scale tensor Bs for the UE8M0 variant);
 * other inputs give unspecified values.  in == out is allowed.  Device
 * pointers, 4-byte aligned; asynchronous on `stream`. */
bfp8_status bfp8_scale_ceil_ue8m0(const float* in, float* out, int64_t n, void* stream);

/* Column-major scale stride the GEMM prefers: M rounded up to a multiple of 4
 * (16 bytes of fp32, the TMA stride rule lmdeploy PR 4830 pads for). */
int64_t bfp8_scale_ld(int64_t M);

/* ------------------------------------------------------------------------ */
/* Step 2: block-scaled GEMM                                                 */
/* ------------------------------------------------------------------------ */

typedef enum {
  BFP8_SCHEDULE_AUTO = 0,
  BFP8_SCHEDULE_SWAP_AB = 1,  /* weights fill the 128-row MMA slot (small M) */
  BFP8_SCHEDULE_WIDE = 2,     /* activations fill it; 128 x 256 output tiles */
  BFP8_SCHEDULE_GEMV = 3      /* M <= 32 only: the decode kernel on warp-level
                                 MMAs (16-row weight tiles streamed by TMA, one
                                 k-block per MMA warp, no workspace use); needs
                                 K % 128 == 0 and 16-byte aligned A and B.  AUTO
                                 takes it for M <= 24 when its 16-row tiles fit
                                 one wave of 2 x SMs, and for M <= 16 when they
                                 spread evenly enough over the SMs or the
                                 weights take up to 64 MB */
} bfp8_schedule;

/* How the output tiles and their K dimension are shared out among CTAs when
 * the tiles do not fill whole waves of SMs (decode-sized M, few weight rows,
 * or a partly filled last wave). */
typedef enum {
  BFP8_KSPLIT_AUTO = 0,      /* the cheapest of the three below by a cost model
                                of this GPU */
  BFP8_KSPLIT_STREAM_K = 1,  /* persistent CTAs; tiles left after whole waves are
                                split into (tile, k-block) units, partial sums
                                meet in the workspace */
  BFP8_KSPLIT_CLUSTER = 2,   /* thread-block clusters of 2..8 CTAs share a tile,
                                each takes a slice of its k-blocks, and the
                                partial tiles are added in distributed shared
                                memory (no workspace traffic) */
  BFP8_KSPLIT_NONE = 3       /* whole tiles only, balanced over ceil(tiles /
                                waves) CTAs: nothing is split, some SMs may idle */
} bfp8_ksplit;

/* Wide tiles on CTA pairs: a 1-D cluster of two CTAs computes 256 x 256
 * output tiles with 2-SM MMAs (tcgen05.mma.cta_group::2), each CTA loading its
 * 128 activation rows and half of the 256 weight rows of every unit, so each
 * SM takes in a third less operand data per FLOP than with 128 x 256 tiles.
 * Whole tiles only (no k split), plain GEMM calls only (not grouped, not
 * fused), tiles of 256 weight rows. */
typedef enum {
  BFP8_PAIRS_AUTO = 0,    /* when the planner prefers them: never in this
                             version (they measured slower than 128 x 256
                             tiles on every shape tried) */
  BFP8_PAIRS_NEVER = 1,
  BFP8_PAIRS_ALWAYS = 2   /* whenever the call allows them; BFP8_ERR_UNSUPPORTED
                             when it does not (swap-AB or 128-wide tiles, at
                             most 64 rows, an explicit stream-K or cluster
                             split, grouped or fused calls) */
} bfp8_pairs;

/* Optional tuning / test controls; a NULL options pointer means all zero. */
typedef struct {
  int schedule;        /* bfp8_schedule */
  int max_ctas;        /* cap on CTAs; 0 = one per SM */
  int tile_n;          /* width of the second MMA operand's tile: wide 128 or
                          256 (0 = 256); swap-AB 16, 32, 64, 128 or 256 (0 =
                          the planner's choice for M) */
  int prefetch_weights;/* 1: the GEMM may start streaming B and Bs before the
                          kernel launched just before it on the stream has
                          finished (programmatic dependent launch).  Only valid
                          when that kernel does not write B or Bs, e.g. when it
                          is the bfp8_group_quant of this layer's activations. */
  int k_split;         /* bfp8_ksplit.  CLUSTER applies only when the output
                          has fewer tiles than max_ctas and K > 128; otherwise
                          stream-K runs. */
  int cluster_size;    /* CLUSTER: CTAs per tile, 2..8, clamped to ceil(K/128);
                          0 = the size the cost model prefers among those with
                          tiles * size <= max_ctas */
  int pairs;           /* bfp8_pairs: 256 x 256 tiles on CTA pairs (2-SM MMAs) */
  int reserved[1];
} bfp8_gemm_options;

/*
 * bfp8_gemm -- out = blocked_fp8_gemm(A, B, As, Bs), the computation of
 * native_w8a8_block_matmul / apply_block_scaled_mm in the vLLM PR 49932
 * digest, without its padding of M to a multiple of 4: ragged M, N and K
 * (including a partial last K block) are handled by the library.
 *
 *   A    [M, K] float8_e4m3fn, row-major, row stride K bytes.
 *   B    [N, K] float8_e4m3fn, row-major, row stride K bytes (the "NT" form:
 *        out = A @ B^T).
 *   As   activation scales, G = ceil(K / 128) per row:
 *          as_col_major = 1: As[kb * ld_as + m], ld_as >= M; the buffer holds
 *                            G * ld_as floats (rows are copied whole, as the
 *                            [G, bfp8_scale_ld(M)] buffers of bfp8_group_quant)
 *          as_col_major = 0: As[m * ld_as + kb], ld_as >= G
 *   Bs   [ceil(N / 128), G] fp32, row-major, one scale per 128 x 128 weight tile.
 *   out  [M, N] bfloat16, row-major; each element is the fp32 accumulation of
 *        the scaled block partial sums, rounded to nearest even.
 *   workspace / workspace_bytes
 *        caller-owned device scratch of at least the size bfp8_gemm_workspace_size
 *        reports for the same (M, N, K, options), 256-byte aligned.  It must be
 *        zero-filled once after allocation; every call that completes leaves it
 *        ready for the next (its counters return to zero), whatever the shapes
 *        of later calls.  Concurrent calls must not share a workspace.  After
 *        BFP8_ERR_DEVICE_TIMEOUT, zero it again.
 * Results are deterministic: the same inputs give bitwise the same output on
 * every call, whichever SM finishes first.
 * Requirements: M, N, K >= 1; As, Bs 4-byte aligned.  Fast path: A and B
 * 16-byte aligned with K % 16 == 0, As column-major with ld_as % 4 == 0 and
 * 16-byte aligned, Bs 16-byte aligned with ceil(N/128) * G % 4 == 0 (what
 * bfp8_group_quant and bfp8_scale_ld produce for column-major scales).  Other
 * inputs are first re-laid out into the workspace by the library, in the
 * same call, at the cost of one or two small extra kernels.
 */
bfp8_status bfp8_gemm(const void* A, const void* B, const float* As, int as_col_major,
                      int64_t ld_as, const float* Bs, void* out, int64_t M, int64_t N, int64_t K,
                      void* workspace, size_t workspace_bytes, void* stream);

/* bfp8_gemm with explicit schedule controls (opt may be NULL).  Every
 * schedule computes the same function; they differ only in speed. */
bfp8_status bfp8_gemm_ex(const void* A, const void* B, const float* As, int as_col_major,
                         int64_t ld_as, const float* Bs, void* out, int64_t M, int64_t N,
                         int64_t K, void* workspace, size_t workspace_bytes,
                         const bfp8_gemm_options* opt, void* stream);

/* Workspace bytes bfp8_gemm / bfp8_gemm_ex need for this problem on the
 * current device: a 16 KB counter header, the stream-K partial sums, room for
 * re-laid-out scales and, when K % 16 != 0 or `operands_unaligned` is nonzero
 * (A or B not 16-byte aligned), room for re-laid-out operands.  Writes
 * *bytes; returns BFP8_ERR_UNSUPPORTED without a suitable device. */
bfp8_status bfp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K,
                                     const bfp8_gemm_options* opt, int operands_unaligned,
                                     size_t* bytes);

/* Description of the schedule bfp8_gemm_ex runs.  num_sms = 0: for the
 * current device (its SM count and how many GEMM clusters of each size it
 * runs at once; needs the device).  num_sms > 0: host-only, for a device with
 * that many SMs whose cluster capacity is estimated (a little below
 * num_sms / size, since GPCs differ in size), so the cluster size may differ
 * from the one the current device would get. */
typedef struct {
  int swap_ab;          /* 1: weights in the MMA M slot */
  int tile_n;           /* MMA N (rows of the second operand per tile) */
  int stages;           /* shared-memory pipeline depth */
  int grid;             /* persistent CTAs */
  int64_t tiles;        /* output tiles */
  int64_t k_blocks;     /* G = ceil(K / 128) */
  int64_t dp_tiles;     /* tiles computed whole, round-robin */
  int64_t sk_units;     /* (tile, k-block) units split across CTAs */
  int relayout;         /* operands re-laid out into the workspace first */
  size_t workspace_bytes;
  int cluster;          /* CTAs per tile: > 1 for cluster split-K (grid =
                           tiles * cluster, dp_tiles = sk_units = 0), else 1.
                           Whole tiles only: dp_tiles = tiles, sk_units = 0,
                           grid possibly below the SM count. */
  int gemv;             /* 1: the warp-MMA decode kernel runs (BFP8_SCHEDULE_GEMV);
                           the tile fields above then describe the tensor-core
                           plan it replaces */
  int pair;             /* 1: 256 x 256 tiles on CTA pairs (grid counts CTAs,
                           tiles the 256 x 256 tiles) */
} bfp8_plan_info;

bfp8_status bfp8_gemm_plan(int64_t M, int64_t N, int64_t K, int num_sms,
                           const bfp8_gemm_options* opt, int operands_unaligned,
                           bfp8_plan_info* info);

/* The work split of a plan (num_sms as for bfp8_gemm_plan): for CTA `cta`,
 * the number of (tile, k-block) units it processes and, for unit j, its tile
 * and k-block.  Returns BFP8_ERR_INVALID_ARG for indices out of range. */
bfp8_status bfp8_plan_unit(int64_t M, int64_t N, int64_t K, int num_sms,
                           const bfp8_gemm_options* opt, int cta, int64_t j,
                           int64_t* num_units, int64_t* tile, int64_t* k_block);

/*
 * bfp8_gemm_grouped -- the same blocked FP8 GEMM for a mixture-of-experts
 * layer whose token rows are grouped by expert ("M-grouped contiguous"
 * layout: the transformers DeepGEMM integration, `_build_deepgemm_contiguous_
 * layout` and `deepgemm_fp8_fp4_experts_forward`, in its SM100 "psum" form).
 *
 *   A    [M, K] e4m3, row-major: rows sorted by expert, each expert's block
 *        padded to a multiple of 128 rows (padding rows hold anything; their
 *        outputs are computed and may be ignored).
 *   As   activation scales as for bfp8_gemm.
 *   B    [num_experts, N, K] e4m3, row-major (expert e's weights are rows
 *        e*N .. e*N+N-1 of a [num_experts*N, K] matrix).
 *   Bs   [num_experts, ceil(N/128), G] fp32, row-major.
 *   grouped_layout  device int32 [num_experts]: cumulative sums of the
 *        aligned per-expert row counts (grouped_layout[e] = end of expert e's
 *        block); non-decreasing multiples of 128.  Device memory, read by the
 *        kernel after the preceding kernel in the stream completes, so it may
 *        be produced on the device just before the call.
 *   out  [M, N] bf16: row m of expert e gets
 *          out[m, n] = sum_kb (A[m,kb] . B[e,n,kb]) * As[m,kb] * Bs[e, n/128, kb];
 *        rows m >= grouped_layout[num_experts-1] are not written (rows the
 *        caller's upper bound on M reserved but no expert uses).
 * Runs the wide schedule (128-row tiles, each inside one expert); options as
 * for bfp8_gemm_ex except `schedule` (ignored) and `prefetch_weights`
 * (ignored: the expert of a tile is known only after the wait).  Workspace
 * from bfp8_gemm_grouped_workspace_size.  Requirements as for bfp8_gemm plus
 * 1 <= num_experts <= 1024 and grouped_layout 4-byte aligned.  Its contents
 * live on the device and are checked there: when they are not non-decreasing
 * multiples of 128, the kernel writes nothing and records
 * BFP8_DEV_BAD_GROUPED_LAYOUT in the failure word (bfp8_device_status).
 */
bfp8_status bfp8_gemm_grouped(const void* A, const void* B, const float* As, int as_col_major,
                              int64_t ld_as, const float* Bs, const int32_t* grouped_layout,
                              int num_experts, void* out, int64_t M, int64_t N, int64_t K,
                              void* workspace, size_t workspace_bytes,
                              const bfp8_gemm_options* opt, void* stream);

/* Workspace bytes bfp8_gemm_grouped needs (current device). */
bfp8_status bfp8_gemm_grouped_workspace_size(int64_t M, int64_t N, int64_t K, int num_experts,
                                             const bfp8_gemm_options* opt,
                                             int operands_unaligned, size_t* bytes);

/*
 * bfp8_gemm_fused -- bfp8_gemm with the next steps of a linear layer folded
 * into the GEMM's epilogue (the transformers DeepGEMM integration's
 * `deepgemm_fp8_fp4_linear`: bias added to the bf16 product; and the next
 * layer's per_token_group_quant_fp8 of that bf16 result, vLLM PR 49932
 * digest, "key source snippet").  For every row m and column n:
 *   y[m, n] = bf16(bf16(sum_kb ...) + bias[n])     (bias == NULL: bf16(sum ...))
 * i.e. the bf16 GEMM result plus the bias as a bf16 tensor addition (one fp32
 * addition, rounded to bf16), then, when q != NULL, the 1 x 128 group
 * quantisation of y along n exactly as bfp8_group_quant computes it:
 *   s[m, g] = fl32(max(amax_g |y|, 1e-10) / 448),  q[m, n] = e4m3(fl32(y / s)).
 *   bias  bf16 [N] or NULL.
 *   out   bf16 [M, N] row-major, or NULL to skip the bf16 output.
 *   q     e4m3 [M, N] row-major (row stride N bytes), or NULL.
 *   s     fp32 scales of q: s_col_major = 1: s[g * ld_s + m], ld_s >= M;
 *         s_col_major = 0: s[m * ld_s + g], ld_s >= ceil(N / 128).  NULL iff q is.
 * Other arguments as for bfp8_gemm_ex; the fused epilogue runs on the wide
 * schedule with the stream-K split (options.schedule and options.k_split are
 * ignored when bias or q is given); workspace from
 * bfp8_gemm_fused_workspace_size.  Errors: BFP8_ERR_INVALID_ARG when out and
 * q are both NULL, q and s are not both given, or ld_s is too small;
 * BFP8_ERR_ALIGNMENT for s not 4-byte or bias not 2-byte aligned.
 */
bfp8_status bfp8_gemm_fused(const void* A, const void* B, const float* As, int as_col_major,
                            int64_t ld_as, const float* Bs, const void* bias, void* out, void* q,
                            float* s, int s_col_major, int64_t ld_s, int64_t M, int64_t N,
                            int64_t K, void* workspace, size_t workspace_bytes,
                            const bfp8_gemm_options* opt, void* stream);

/* Workspace bytes bfp8_gemm_fused needs (current device). */
bfp8_status bfp8_gemm_fused_workspace_size(int64_t M, int64_t N, int64_t K,
                                           const bfp8_gemm_options* opt, int operands_unaligned,
                                           size_t* bytes);

/*
 * bfp8_linear -- the whole W8A8 blocked linear layer from bf16 activations in
 * one call:
 *   out = bfp8_gemm(q, B, s, Bs)  with  (q, s) = bfp8_group_quant(x, group 128,
 *   column-major scales)
 * (per_token_group_quant_fp8 followed by w8a8_block_fp8_matmul, the two steps
 * of the vLLM PR 49932 digest's blocked FP8 linear), bitwise what those two
 * calls give with the same options.  Two kernels: the quantisation writes q
 * and s into the workspace, and the GEMM, launched behind it with
 * programmatic dependent launch, streams the weights while it runs.
 *   x    bf16 [M, K], row stride ld_x elements (ld_x >= K), 2-byte aligned.
 *   B, Bs, out, M, N, K, opt, stream as for bfp8_gemm_ex (opt.prefetch_weights
 *        is always on).
 *   workspace / workspace_bytes
 *        at least bfp8_linear_workspace_size bytes, 256-byte aligned, zero-filled
 *        once after allocation: its first part serves the GEMM as for
 *        bfp8_gemm (left ready for the next call), the rest holds q and s.
 * Errors: BFP8_ERR_INVALID_ARG / ALIGNMENT / WORKSPACE as for bfp8_gemm_ex.
 */
bfp8_status bfp8_linear(const void* x, int64_t ld_x, const void* B, const float* Bs, void* out,
                        int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                        const bfp8_gemm_options* opt, void* stream);

/* Workspace bytes bfp8_linear needs (current device); weights_unaligned: B
 * not 16-byte aligned. */
bfp8_status bfp8_linear_workspace_size(int64_t M, int64_t N, int64_t K, const bfp8_gemm_options* opt,
                                       int weights_unaligned, size_t* bytes);

/*
 * bfp8_gemm_noalloc -- bfp8_gemm for callers that cannot allocate device
 * memory.  (Not from the pages: they have no counterpart; this is a
 * convenience of this library.)
 *
 * Some callers have no way to provide the GEMM workspace: code running while a
 * stream is being captured into a CUDA graph in a mode that forbids
 * cudaMalloc, plug-ins living inside a host framework that owns every device
 * allocation through its own pool and exposes no hook to them, and
 * latency-critical loops that must not pay for an allocation or risk one
 * failing.  This entry point computes exactly what bfp8_gemm computes (same
 * arguments minus the workspace, same kernels, same results) but takes its
 * scratch from a fixed array built into the library: BFP8_NOALLOC_SCRATCH_BYTES
 * (16 MiB) of device memory that every GPU which loads the library holds until
 * the process exits.  It never calls cudaMalloc, cudaFree or any allocating
 * routine.
 *
 * Limits and rules:
 *   - Problems whose workspace (bfp8_gemm_workspace_size with default
 *     options) exceeds BFP8_NOALLOC_SCRATCH_BYTES are rejected with
 *     BFP8_ERR_WORKSPACE and a reason in bfp8_last_error(); nothing is
 *     launched.  Decode-sized problems fit (e.g. M <= 64 at N = K = 4096);
 *     large-M problems generally do not.
 *   - The first call on each device looks up the scratch's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.  The address is kept for the life of
 *     the process: after cudaDeviceReset() on a device, do not call this
 *     entry point on that device again.
 *   - Every call on a device shares the one scratch array, and it keeps the
 *     previous call's contents: each call first clears (cudaMemsetAsync on
 *     `stream`) the part that must start at zero.  Calls whose kernels can
 *     overlap on the GPU (different streams without ordering between them)
 *     race on the scratch and give wrong results; serialise them.
 */
#define BFP8_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
bfp8_status bfp8_gemm_noalloc(const void* A, const void* B, const float* As, int as_col_major,
                              int64_t ld_as, const float* Bs, void* out, int64_t M, int64_t N,
                              int64_t K, void* stream);

/* ------------------------------------------------------------------------ */
/* Status and diagnostics                                                    */
/* ------------------------------------------------------------------------ */

/* Reason for the last failure on the calling thread ("" if none). */
const char* bfp8_last_error(void);

/* Static name of a status code. */
const char* bfp8_status_string(int status);

/* Synchronises the current device and reads the library's device-side failure
 * word for it; clears it when `clear` is nonzero.  The word holds the first
 * failure a kernel reported since the last clear: */
#define BFP8_DEV_OK 0                       /* none */
#define BFP8_DEV_TIMEOUT_PRODUCER 1         /* a bounded wait gave up: operand loader */
#define BFP8_DEV_TIMEOUT_MMA 2              /*   MMA issuer */
#define BFP8_DEV_TIMEOUT_EPILOGUE 3         /*   promotion / epilogue warps */
#define BFP8_DEV_TIMEOUT_TAIL 4             /*   draining copies before exit */
#define BFP8_DEV_BAD_GROUPED_LAYOUT 5       /* bfp8_gemm_grouped: invalid grouped_layout */
/* After a timeout code, a workspace the call used may hold non-zero counters:
 * zero it before reusing it. */
bfp8_status bfp8_device_status(int* code, int clear);

/* Self-test of the bounded wait every kernel uses: launches one warp that
 * waits on a shared-memory barrier nothing ever arrives on, giving up after
 * `limit_cycles` SM cycles.  Synchronises the stream and returns
 * BFP8_ERR_DEVICE_TIMEOUT when the wait gave up as designed (and *elapsed
 * holds the cycles it waited), BFP8_OK if the barrier completed. */
bfp8_status bfp8_selftest_bounded_wait(uint64_t limit_cycles, uint64_t* elapsed, void* stream);

int bfp8_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BFP8_H_ */
