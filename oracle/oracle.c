/*
 * oracle.c -- plain CPU oracle for the blocked W8A8 FP8 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Built with -ffp-contract=off and
 * without fast-math so that every float / double operation below is one IEEE
 * operation, identical on x86-64 and aarch64.
 *
 * Sources:
 *   [P2] vLLM PR 49932 digest, "torch._scaled_mm FP8 block-scale kernel
 *        backend" -- section "key source snippet", test_w8a8_block_fp8_torch_scaled_mm_matmul: fp8 limits
 *        from torch.finfo(float8_e4m3fn) (+-448), per_token_group_quant_fp8
 *        with group 128 and row/column-major scales, native_w8a8_block_matmul
 *        with block_size [128, 128], weight scales [ceil(N/128), ceil(K/128)],
 *        bf16 output.
 *   [P4] transformers integrations/deepgemm.py, _coerce_sf_for_kernel: the
 *        column-major (MN-major) scale layout with a padded leading dimension;
 *        _ceil_to_ue8m0 and _select_fp8_cast_kwargs (use_ue8m0): scales rounded
 *        up to powers of two (UE8M0, the scale format of the SM100 kernels).
 *   OCP 8-bit floating point specification, E4M3: sign, 4 exponent bits
 *        (bias 7), 3 mantissa bits, no infinities, S.1111.111 = NaN.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------------------------------------------------------------- e4m3 --- */

/* OCP E4M3: s = bit 7, e = bits 6..3, m = bits 2..0.
 *   e = 15 and m = 7      -> NaN (the format has no infinities)
 *   e = 0                 -> (-1)^s * m * 2^-9          (subnormal: m/8 * 2^-6)
 *   otherwise             -> (-1)^s * (1 + m/8) * 2^(e-7)                    */
double oracle_e4m3_decode(uint8_t code) {
    int s = code >> 7;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

void oracle_e4m3_table(double* out) {
    for (int c = 0; c < 256; ++c) out[c] = oracle_e4m3_decode((uint8_t)c);
}

/* Magnitudes of the 127 non-negative finite codes 0x00..0x7E, ascending
 * (the encoding is monotone in the code for a fixed sign). */
static double g_mag[127];
static pthread_once_t g_mag_once = PTHREAD_ONCE_INIT;
static void build_mag(void) {
    for (int c = 0; c < 127; ++c) g_mag[c] = oracle_e4m3_decode((uint8_t)c);
}

/* Round to nearest, ties to the even code (even mantissa), saturating at 448.
 * The two neighbours of |x| are found by binary search in the ascending
 * magnitude table; the distances are exact in double because |x| has a
 * 24-bit significand and the table entries have 4. */
uint8_t oracle_e4m3_encode(float x) {
    pthread_once(&g_mag_once, build_mag);
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a > 448.0) return (uint8_t)(sign | 0x7E); /* satfinite, includes inf */
    int lo = 0, hi = 126;                          /* g_mag[lo] <= a */
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (g_mag[mid] <= a) lo = mid; else hi = mid - 1;
    }
    int c = lo;
    if (g_mag[lo] != a && lo < 126) {
        double dl = a - g_mag[lo];
        double dh = g_mag[lo + 1] - a;
        if (dh < dl || (dh == dl && ((lo + 1) & 1) == 0)) c = lo + 1;
    }
    return (uint8_t)(sign | c);
}

void oracle_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

/* ---------------------------------------------------------------- bf16 --- */

/* bfloat16: 8-bit significand (1 implicit + 7 stored), 8 exponent bits.
 * Normal numbers from 2^-126, subnormals step 2^-133.  The double is scaled
 * by a power of two so that one unit of the result's last place is 1, rounded
 * to an integer with rint() (ties to even under the default rounding mode),
 * and scaled back; both scalings are exact. */
uint16_t oracle_bf16_from_double(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e);            /* a = f * 2^e, f in [0.5, 1) */
    int q = e - 8;                 /* quantum exponent of a normal bf16 */
    if (q < -133) q = -133;        /* subnormal range */
    double r = ldexp(rint(ldexp(a, -q)), q);
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float f = (float)r;            /* exact: <= 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

void oracle_bf16_from_double_array(const double* v, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_from_double(v[i]);
}

/* ------------------------------------------------------ group quantise --- */

static float load_x(const void* x, int in_is_f32, int64_t idx) {
    if (in_is_f32) return ((const float*)x)[idx];
    uint32_t bits = (uint32_t)((const uint16_t*)x)[idx] << 16; /* exact widening */
    float f;
    memcpy(&f, &bits, 4);
    return f;
}

/* [P4] _ceil_to_ue8m0: a positive fp32 scale rounded up to the nearest power
 * of two.  Written from that definition: with s = f * 2^e and f in [0.5, 1),
 * s is itself a power of two exactly when f = 0.5; otherwise the smallest
 * power of two above s is 2^e. */
float oracle_ceil_pow2(float s) {
    if (!(s > 0.0f) || isinf(s)) return s;   /* defined for positive finite scales */
    int e;
    const double f = frexp((double)s, &e);
    if (f == 0.5) return s;
    return (float)ldexp(1.0, e);             /* 2^128 and above: +inf */
}

static int group_quant_impl(const void* x, int in_is_f32, int64_t M, int64_t K, int64_t ld_x,
                            int col_major, int64_t ld_s, uint8_t* q, int64_t ld_q, float* s,
                            int ue8m0);

int oracle_group_quant(const void* x, int in_is_f32, int64_t M, int64_t K, int64_t ld_x,
                       int col_major, int64_t ld_s, uint8_t* q, int64_t ld_q, float* s) {
    return group_quant_impl(x, in_is_f32, M, K, ld_x, col_major, ld_s, q, ld_q, s, 0);
}

int oracle_group_quant_ue8m0(const void* x, int in_is_f32, int64_t M, int64_t K, int64_t ld_x,
                             int col_major, int64_t ld_s, uint8_t* q, int64_t ld_q, float* s) {
    return group_quant_impl(x, in_is_f32, M, K, ld_x, col_major, ld_s, q, ld_q, s, 1);
}

static int group_quant_impl(const void* x, int in_is_f32, int64_t M, int64_t K, int64_t ld_x,
                            int col_major, int64_t ld_s, uint8_t* q, int64_t ld_q, float* s,
                            int ue8m0) {
    if (!x || !q || !s || M < 0 || K < 0 || ld_x < K || ld_q < K) return -1;
    const int64_t G = (K + 127) / 128;
    if (col_major ? ld_s < M : ld_s < G) return -1;
    /* padded layout entries hold no scale: zero them */
    if (col_major) {
        for (int64_t g = 0; g < G; ++g)
            for (int64_t m = M; m < ld_s; ++m) s[g * ld_s + m] = 0.0f;
    } else {
        for (int64_t m = 0; m < M; ++m)
            for (int64_t g = G; g < ld_s; ++g) s[m * ld_s + g] = 0.0f;
    }
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < G; ++g) {
            const int64_t k0 = g * 128;
            const int64_t k1 = (k0 + 128 < K) ? k0 + 128 : K;
            float amax = 0.0f;
            for (int64_t k = k0; k < k1; ++k) {
                float v = fabsf(load_x(x, in_is_f32, m * ld_x + k));
                if (v > amax) amax = v;
            }
            const float floor_amax = 1e-10f;
            float scale = (amax > floor_amax ? amax : floor_amax) / 448.0f;
            if (ue8m0) scale = oracle_ceil_pow2(scale);
            for (int64_t k = k0; k < k1; ++k) {
                const float v = load_x(x, in_is_f32, m * ld_x + k);
                const float y = v / scale;
                q[m * ld_q + k] = oracle_e4m3_encode(y);
            }
            if (col_major) s[g * ld_s + m] = scale;
            else s[m * ld_s + g] = scale;
        }
    }
    return 0;
}

/* -------------------------------------------------------- blocked GEMM --- */

typedef struct {
    const uint8_t* A; const uint8_t* B; const float* As; const float* Bs;
    int as_col_major; int64_t ld_as; int64_t M, N, K;
    const int64_t* rows; int64_t n_rows;
    uint16_t* out_bf16; double* out_f64; double* abs_f64;
    int tid, nthreads; int status;
} gemm_job;

static void* gemm_worker(void* arg) {
    gemm_job* j = (gemm_job*)arg;
    double tab[256];
    oracle_e4m3_table(tab);
    const int64_t K = j->K, N = j->N;
    const int64_t G = (K + 127) / 128;
    const int64_t G_n = (N + 127) / 128;
    (void)G_n;
    double* arow = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    if (!arow) { j->status = -2; return NULL; }
    for (int64_t i = j->tid; i < j->n_rows; i += j->nthreads) {
        const int64_t m = j->rows ? j->rows[i] : i;
        for (int64_t k = 0; k < K; ++k) arow[k] = tab[j->A[m * K + k]];
        for (int64_t n = 0; n < N; ++n) {
            const uint8_t* brow = j->B + n * K;
            double acc = 0.0, abs_acc = 0.0;
            for (int64_t kb = 0; kb < G; ++kb) {
                const int64_t k0 = kb * 128;
                const int64_t k1 = (k0 + 128 < K) ? k0 + 128 : K;
                /* exact in fp64: each product of two e4m3 values has at most 8
                 * significant bits and lies in [2^-18, 2^17.6]; 128 of them sum
                 * to < 2^25, so every partial sum fits in 43 bits < 53. */
                double d = 0.0;
                for (int64_t k = k0; k < k1; ++k) d += arow[k] * tab[brow[k]];
                const double as = j->as_col_major ? (double)j->As[kb * j->ld_as + m]
                                                  : (double)j->As[m * j->ld_as + kb];
                const double bs = (double)j->Bs[(n / 128) * G + kb];
                const double term = (d * as) * bs;
                acc += term;
                abs_acc += fabs(term);
            }
            if (j->out_f64) j->out_f64[i * N + n] = acc;
            if (j->abs_f64) j->abs_f64[i * N + n] = abs_acc;
            if (j->out_bf16) j->out_bf16[i * N + n] = oracle_bf16_from_double(acc);
        }
    }
    free(arow);
    return NULL;
}

int oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    if (n < 1) n = 1;
    if (n > 256) n = 256;
    return (int)n;
}

int oracle_blocked_gemm(const uint8_t* A, const uint8_t* B, const float* As, int as_col_major,
                        int64_t ld_as, const float* Bs, int64_t M, int64_t N, int64_t K,
                        const int64_t* rows, int64_t n_rows, uint16_t* out_bf16, double* out_f64,
                        double* abs_f64, int nthreads) {
    if (!A || !B || !As || !Bs || M < 0 || N < 0 || K < 0) return -1;
    const int64_t G = (K + 127) / 128;
    if (as_col_major ? ld_as < M : ld_as < G) return -1;
    if (!rows) n_rows = M;
    for (int64_t i = 0; rows && i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= M) return -1;
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > n_rows) nthreads = n_rows > 0 ? (int)n_rows : 1;
    gemm_job* jobs = (gemm_job*)calloc((size_t)nthreads, sizeof(gemm_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -2; }
    for (int t = 0; t < nthreads; ++t) {
        gemm_job jb = {A, B, As, Bs, as_col_major, ld_as, M, N, K, rows, n_rows,
                       out_bf16, out_f64, abs_f64, t, nthreads, 0};
        jobs[t] = jb;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, gemm_worker, &jobs[t]) != 0) break;
        started = t;
    }
    /* threads that failed to start have their rows done by the caller */
    if (started < nthreads - 1) {
        for (int t = started + 1; t < nthreads; ++t) gemm_worker(&jobs[t]);
    }
    gemm_worker(&jobs[0]);
    int status = 0;
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads; ++t) if (jobs[t].status) status = jobs[t].status;
    free(jobs);
    free(th);
    return status;
}
