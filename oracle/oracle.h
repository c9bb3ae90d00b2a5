/*
 * oracle.h -- plain, slow CPU oracle for the blocked W8A8 FP8 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this code; only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library (libbfp8): every definition below is written out again from
 * the pages and from the OCP FP8 format definition.
 *
 * What it computes (sources are the four pages on DeepSeek-style blocked FP8):
 *   - float8_e4m3fn decode / encode: the vLLM PR 49932 digest
 *     "torch._scaled_mm FP8 block-scale kernel backend" (section "key source
 *     snippet", test_w8a8_block_fp8_torch_scaled_mm_matmul) takes fp8 max/min from
 *     torch.finfo(float8_e4m3fn) = +-448; the bit layout is OCP E4M3 "fn"
 *     (bias 7, no infinities, S.1111.111 is the only NaN).
 *   - per-token group quantisation: same snippet, per_token_group_quant_fp8
 *     with a group of 128 and row- or column-major activation scales.
 *   - blocked GEMM: same snippet, native_w8a8_block_matmul with
 *     block_size [128, 128]: out[m,n] = sum_kb (A[m,kb].B[n,kb]) As[m,kb]
 *     Bs[n/128,kb], rounded to bf16.
 *
 * Every function returns 0 on success and a negative value on a bad argument.
 */
#ifndef BFP8_ORACLE_H
#define BFP8_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Value of one float8_e4m3fn code as a double (NaN for 0x7F / 0xFF). */
double oracle_e4m3_decode(uint8_t code);

/* Copy the 256-entry decode table into out[256]. */
void oracle_e4m3_table(double* out);

/* Round-to-nearest-even, saturating encode of one fp32 value to e4m3fn.
 * NaN -> 0x7F; |x| > 448 (including +-inf) -> +-448; the sign of a zero or
 * of an underflow to zero is kept (0x80 for negatives). */
uint8_t oracle_e4m3_encode(float x);

/* Encode n values (used by the exhaustive checks). */
void oracle_e4m3_encode_array(const float* x, uint8_t* out, int64_t n);

/* Round a double to bfloat16 (round to nearest, ties to even), directly from
 * the double with no intermediate fp32 rounding.  Returns the bf16 bits. */
uint16_t oracle_bf16_from_double(double v);
void oracle_bf16_from_double_array(const double* v, uint16_t* out, int64_t n);

/* Per-token group quantisation, group = 128 along K.
 *   x        : [M, K] row-major, leading dimension ld_x elements;
 *              in_is_f32 = 1 -> float, 0 -> bfloat16 bits (uint16).
 *   q        : [M, K] e4m3 codes, leading dimension ld_q bytes.
 *   s        : G = ceil(K/128) scales per row; col_major = 0 -> s[m*ld_s + g]
 *              (ld_s >= G), col_major = 1 -> s[g*ld_s + m] (ld_s >= M).
 *              Entries of the padded layout that hold no scale are set to 0.
 * amax = max |x| over the group's real elements, scale = max(amax, 1e-10)/448
 * in fp32 (one IEEE division), q = encode(x / scale) with one IEEE fp32
 * division per element. */
int oracle_group_quant(const void* x, int in_is_f32, int64_t M, int64_t K, int64_t ld_x,
                       int col_major, int64_t ld_s, uint8_t* q, int64_t ld_q, float* s);

/* UE8M0 variant (transformers integrations/deepgemm.py, _ceil_to_ue8m0 and
 * the use_ue8m0 cast of _select_fp8_cast_kwargs): oracle_ceil_pow2 rounds a
 * positive finite fp32 scale up to the nearest power of two;
 * oracle_group_quant_ue8m0 is oracle_group_quant with every group's scale
 * max(amax, 1e-10) / 448 so rounded before the codes are computed (the codes
 * are then encode(x / scale), each division exact). */
float oracle_ceil_pow2(float s);
int oracle_group_quant_ue8m0(const void* x, int in_is_f32, int64_t M, int64_t K, int64_t ld_x,
                             int col_major, int64_t ld_s, uint8_t* q, int64_t ld_q, float* s);

/* Blocked GEMM over selected output rows.
 *   A  : [M, K] e4m3 codes (row stride K), B : [N, K] e4m3 codes (row stride K)
 *   As : activation scales, layout as in oracle_group_quant (as_col_major, ld_as)
 *   Bs : [ceil(N/128), ceil(K/128)] fp32, row-major, one per 128x128 weight tile
 *   rows: n_rows row indices (NULL -> all M rows in order)
 * For each selected row r and every n:
 *   acc = sum over kb ascending of ((double)D_kb * As[m,kb]) * Bs[n/128,kb]
 *   with D_kb = sum over the block's real k of dec(A[m,k]) * dec(B[n,k])
 *   (exact in fp64), then out = bf16(acc).
 * out_bf16  (may be NULL) : [n_rows, N] bf16 bits
 * out_f64   (may be NULL) : [n_rows, N] the fp64 sum before rounding
 * abs_f64   (may be NULL) : [n_rows, N] sum over kb of |D_kb * As * Bs|
 * Work is spread over nthreads POSIX threads (<= 0: one per online core);
 * the result does not depend on the thread count. */
int oracle_blocked_gemm(const uint8_t* A, const uint8_t* B, const float* As, int as_col_major,
                        int64_t ld_as, const float* Bs, int64_t M, int64_t N, int64_t K,
                        const int64_t* rows, int64_t n_rows, uint16_t* out_bf16, double* out_f64,
                        double* abs_f64, int nthreads);

/* Number of threads oracle_blocked_gemm uses for nthreads <= 0. */
int oracle_default_threads(void);

#ifdef __cplusplus
}
#endif
#endif
