/*
 * CPU oracle for dense GEMM  C <- alpha * A * B + beta * C   (TEST INFRASTRUCTURE)
 *
 * This file is test infrastructure.  Only the tests, the smoke check and the
 * bench's CPU-baseline leg call it; the library's GPU path never does.  It
 * shares no code with the CUDA path: its own format decoders, its own
 * rounding, its own loop.
 *
 * What it computes (the plain definition, no blocking or reordering):
 *   a_ik, b_kj : the exact values of the stored fp16/bf16 bit patterns
 *                ("rounded-input" reference: the two-reference testing protocol
 *                of "GEMM From Naive CUDA to Tensor Cores", leetllm.com)
 *   s_ij       = sum over k = 0..K-1, ascending, of a_ik * b_kj, in binary64
 *                (the scalar dot product C_ij = sum_k A_ik B_kj of the same page,
 *                "Compute one output before launching a warp")
 *   r_ij       = alpha * s_ij + beta * c_ij   in binary64; the beta term is
 *                dropped when beta == 0 so C is not read (the same page's
 *                preamble: the alpha = 1, beta = 0 case does not read the old
 *                output buffer)
 *   r_ij      += bias_j (per-column bias) or bias_i (per-row bias), in binary64,
 *                when a bias is given; then r_ij = 0 if r_ij < 0 when ReLU is
 *                asked for (NaN stays NaN).  This is the epilogue folded into the
 *                GEMM of "A dense FP16 matrix-multiply kernel for NVIDIA Ada", its
 *                bias + ReLU paragraph after the L2-rasterization table: the
 *                intermediate is kept in wide precision and rounded once; the
 *                per-row form is the one the "mma.sync and ldmatrix" page names
 *                (an epilogue applying a per-row bias).
 *   out_ij     = round-to-nearest-even(r_ij) in the output format
 *   S_ij       = sum_k |a_ik| |b_kj|, the scale of the error bound.
 *
 * Formats: IEEE binary16 (1/5/10), bfloat16 (1/8/7), binary32 (1/8/23), decoded
 * from their definitions (the binary16 facts -- 5 exponent bits, 10 mantissa
 * bits, spacing 1 above 1024 -- are the ones the leetllm page states in "What FP32
 * accumulation preserves").
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { OR_F16 = 0, OR_BF16 = 1, OR_F32 = 2, OR_E4M3 = 3, OR_E5M2 = 4 };
enum { OR_BIAS_NONE = 0, OR_BIAS_COL = 1, OR_BIAS_ROW = 2 };
enum { OR_ACT_NONE = 0, OR_ACT_RELU = 1 };

/* ---------------------------------------------------------------- decoding */

static double decode_f16(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);      /* (1 + m/2^10) 2^(e-15) */
    return s ? -v : v;
}

static double decode_bf16(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 7) & 0xFF, m = h & 0x7F;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);                /* m/2^7 * 2^-126 */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + m), e - 134);      /* (1 + m/2^7) 2^(e-127) */
    return s ? -v : v;
}

/* The two 8-bit formats of the OCP FP8 definition (the FP8 variant the Ada GEMM
 * page lists as written but untested):
 *   E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; no infinities, the
 *         pattern S.1111.111 is NaN, the largest finite value is 448.
 *   E5M2: 1 sign, 5 exponent bits (bias 15), 2 mantissa bits; IEEE-style
 *         infinities (exponent 31, mantissa 0) and NaNs. */
static double decode_e4m3(uint8_t b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 0xF, m = b & 0x7;
    double v;
    if (e == 0)
        v = ldexp((double)m, -9);                  /* m/8 * 2^(1-7) */
    else if (e == 15 && m == 7)
        v = NAN;
    else
        v = ldexp((double)(8 + m), e - 10);         /* (1 + m/8) 2^(e-7) */
    return s ? -v : v;
}

static double decode_e5m2(uint8_t b) {
    int s = (b >> 7) & 1, e = (b >> 2) & 0x1F, m = b & 0x3;
    double v;
    if (e == 0)
        v = ldexp((double)m, -16);                 /* m/4 * 2^(1-15) */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(4 + m), e - 17);         /* (1 + m/4) 2^(e-15) */
    return s ? -v : v;
}

static double decode_f32(uint32_t w) {
    int s = (w >> 31) & 1, e = (w >> 23) & 0xFF;
    uint32_t m = w & 0x7FFFFF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -149);
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(0x800000u + m), e - 150);
    return s ? -v : v;
}

static double decode(const void* base, int fmt, int64_t idx) {
    if (fmt == OR_F32) return decode_f32(((const uint32_t*)base)[idx]);
    if (fmt == OR_BF16) return decode_bf16(((const uint16_t*)base)[idx]);
    if (fmt == OR_E4M3) return decode_e4m3(((const uint8_t*)base)[idx]);
    if (fmt == OR_E5M2) return decode_e5m2(((const uint8_t*)base)[idx]);
    return decode_f16(((const uint16_t*)base)[idx]);
}

/* ----------------------------------------------- rounding (nearest, ties even) */

/* Round x to a binary format with p significand bits (hidden bit included) and
 * normal exponents emin..emax, round-to-nearest-even, overflow to infinity. */
static double round_fmt(double x, int p, int emin, int emax) {
    if (isnan(x) || isinf(x) || x == 0.0) return x;
    double ax = fabs(x);
    int e;
    frexp(ax, &e);                 /* ax in [2^(e-1), 2^e) */
    int E = e - 1;
    if (E > emax) return copysign(INFINITY, x);
    if (E < emin) E = emin;        /* subnormal range: fixed quantum */
    double q = ldexp(1.0, E - (p - 1));
    double t = ax / q;             /* exact: scaling by a power of two */
    double fl = floor(t);
    double d = t - fl;             /* exact */
    double r;
    if (d > 0.5)
        r = fl + 1.0;
    else if (d < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double y = r * q;
    double maxf = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (y > maxf) return copysign(INFINITY, x);
    return copysign(y, x);
}

static uint32_t encode_f32(double x) {
    if (isnan(x)) return 0x7FC00000u;
    double y = round_fmt(x, 24, -126, 127);
    float f = (float)y;            /* exact: y is representable */
    uint32_t w;
    memcpy(&w, &f, 4);
    return w;
}

static uint16_t encode_bf16(double x) {
    if (isnan(x)) return 0x7FC0u;
    double y = round_fmt(x, 8, -126, 127);
    float f = (float)y;            /* exact: every bfloat16 value is a binary32 value */
    uint32_t w;
    memcpy(&w, &f, 4);
    return (uint16_t)(w >> 16);    /* exact: the low 16 bits are zero */
}

static uint16_t encode_f16(double x) {
    if (isnan(x)) return 0x7E00u;
    double y = round_fmt(x, 11, -14, 15);
    uint16_t s = signbit(y) ? 0x8000u : 0;
    double ay = fabs(y);
    if (isinf(ay)) return s | 0x7C00u;
    if (ay == 0.0) return s;
    int e;
    frexp(ay, &e);
    int E = e - 1;
    if (E < -14) return s | (uint16_t)ldexp(ay, 24);              /* subnormal */
    return s | (uint16_t)((E + 15) << 10) | (uint16_t)(ldexp(ay, 10 - E) - 1024.0);
}

/* ------------------------------------------------------------------ the GEMM */

typedef struct {
    int64_t M, N, K;
    double alpha, beta;
    const void* A; int64_t lda; int a_col;
    const float* Bk;                /* B decoded to exact values, [K][N] */
    int in_fmt;
    const void* C_in; int64_t ldc;
    int out_fmt;
    const float* bias; int bias_kind; int act;
    const int64_t* rows; int64_t nrows;
    void* out_bits; double* out_exact; double* out_scale;
    int64_t r0, r1;                 /* this worker's slice of rows[] */
} job_t;

static void* run_rows(void* arg) {
    job_t* J = (job_t*)arg;
    const int64_t N = J->N, K = J->K;
    double* acc = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double* scl = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    for (int64_t t = J->r0; t < J->r1; ++t) {
        const int64_t i = J->rows ? J->rows[t] : t;
        for (int64_t j = 0; j < N; ++j) { acc[j] = 0.0; scl[j] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            /* A is [M, K] row-major (a_ik at i*lda + k) or [K, M] column-major
             * storage (a_ik at k*lda + i). */
            const double a = decode(J->A, J->in_fmt, J->a_col ? k * J->lda + i : i * J->lda + k);
            const double aa = fabs(a);
            const float* brow = J->Bk + k * N;
            for (int64_t j = 0; j < N; ++j) {
                const double b = (double)brow[j];
                acc[j] += a * b;
                scl[j] += aa * fabs(b);
            }
        }
        for (int64_t j = 0; j < N; ++j) {
            double r = J->alpha * acc[j];
            if (J->beta != 0.0)
                r += J->beta * decode(J->C_in, J->out_fmt, i * J->ldc + j);
            if (J->bias_kind == OR_BIAS_COL) r += (double)J->bias[j];
            else if (J->bias_kind == OR_BIAS_ROW) r += (double)J->bias[i];
            if (J->act == OR_ACT_RELU && r < 0.0) r = 0.0;
            const int64_t o = t * N + j;
            if (J->out_exact) J->out_exact[o] = r;
            if (J->out_scale) J->out_scale[o] = scl[j];
            if (J->out_bits) {
                if (J->out_fmt == OR_F32) ((uint32_t*)J->out_bits)[o] = encode_f32(r);
                else if (J->out_fmt == OR_BF16) ((uint16_t*)J->out_bits)[o] = encode_bf16(r);
                else ((uint16_t*)J->out_bits)[o] = encode_f16(r);
            }
        }
    }
    free(acc);
    free(scl);
    return NULL;
}

/* Computes the rows listed in rows[0..nrows) (all M rows, in order, when rows is
 * NULL; nrows must then equal M).  Outputs are packed [nrows, N].
 * B is [K, N] row-major (b_kj at k*ldb + j) or [N, K] column-major storage
 * (b_kj at j*ldb + k).  C_in is [M, N] row-major in out_fmt with leading
 * dimension ldc; it is read only when beta != 0.  bias: N floats (bias_kind 1,
 * per column) or M floats (bias_kind 2, per row), unused for bias_kind 0; act 1
 * applies ReLU.  Returns 0, or -1 on bad input. */
int oracle_gemm_epilogue(int64_t M, int64_t N, int64_t K, double alpha,
                         const void* A, int64_t lda, int a_col,
                         const void* B, int64_t ldb, int b_col, int in_fmt,
                         double beta, const void* C_in, int64_t ldc, int out_fmt,
                         const float* bias, int bias_kind, int act,
                         const int64_t* rows, int64_t nrows,
                         void* out_bits, double* out_exact, double* out_scale, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (!rows && nrows != M) return -1;
    if (beta != 0.0 && !C_in) return -1;
    if (bias_kind < OR_BIAS_NONE || bias_kind > OR_BIAS_ROW || act < OR_ACT_NONE || act > OR_ACT_RELU)
        return -1;
    if (bias_kind != OR_BIAS_NONE && !bias) return -1;
    for (int64_t t = 0; rows && t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= M) return -1;
    float* Bk = (float*)malloc(sizeof(float) * (size_t)(K * N > 0 ? K * N : 1));
    if (!Bk) return -1;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N; ++j)
            Bk[k * N + j] = (float)decode(B, in_fmt, b_col ? j * ldb + k : k * ldb + j);
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = nrows > 0 ? (int)nrows : 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    job_t* jobs = (job_t*)malloc(sizeof(job_t) * (size_t)nthreads);
    for (int w = 0; w < nthreads; ++w) {
        job_t J = {M, N, K, alpha, beta, A, lda, a_col, Bk, in_fmt, C_in, ldc, out_fmt,
                   bias, bias_kind, act, rows, nrows, out_bits, out_exact, out_scale,
                   nrows * w / nthreads, nrows * (w + 1) / nthreads};
        jobs[w] = J;
        pthread_create(&th[w], NULL, run_rows, &jobs[w]);
    }
    for (int w = 0; w < nthreads; ++w) pthread_join(th[w], NULL);
    free(th);
    free(jobs);
    free(Bk);
    return 0;
}

/* The plain GEMM: no bias, no activation. */
int oracle_gemm(int64_t M, int64_t N, int64_t K, double alpha,
                const void* A, int64_t lda, int a_col,
                const void* B, int64_t ldb, int b_col, int in_fmt,
                double beta, const void* C_in, int64_t ldc, int out_fmt,
                const int64_t* rows, int64_t nrows,
                void* out_bits, double* out_exact, double* out_scale, int nthreads) {
    return oracle_gemm_epilogue(M, N, K, alpha, A, lda, a_col, B, ldb, b_col, in_fmt, beta, C_in,
                                ldc, out_fmt, NULL, OR_BIAS_NONE, OR_ACT_NONE, rows, nrows,
                                out_bits, out_exact, out_scale, nthreads);
}

/* Element-wise helpers exposed for the oracle's own pins. */
void oracle_decode(const void* bits, int fmt, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = decode(bits, fmt, i);
}

void oracle_encode(const double* x, int fmt, int64_t n, void* bits) {
    for (int64_t i = 0; i < n; ++i) {
        if (fmt == OR_F32) ((uint32_t*)bits)[i] = encode_f32(x[i]);
        else if (fmt == OR_BF16) ((uint16_t*)bits)[i] = encode_bf16(x[i]);
        else ((uint16_t*)bits)[i] = encode_f16(x[i]);
    }
}
