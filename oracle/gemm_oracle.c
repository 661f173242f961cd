/*
 * CPU oracle for the bf16 GEMM  C_out = alpha * A * B + beta * C_in.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA library is checked against.  It shares no code,
 * header, table or constant with the CUDA library, and only the tests, the
 * package's smoke check and the benchmark's CPU-baseline leg may load it.
 *
 * What it computes (the definition, written out):
 *
 *   S[i,j]     = sum_{k=0}^{K-1} A[i,k] * B[k,j]            (k ascending, fp64)
 *   D[i,j]     = alpha * S[i,j] + beta * C_in[i,j]          (fp64; the beta
 *                term is skipped entirely when beta == 0, so C_in is not read)
 *   C_out[i,j] = round_out(D[i,j])                          (one rounding)
 *
 * Sources:
 *  - The product C[m,n] = A[m,k] x B[k,n] and the layouts -- A row-major,
 *    B and C column-major, bf16 -- are from the H100 work log
 *    "在 H100 上超越 cuBLAS：一份工作日志", sections "Simon 博客的快速回顾"
 *    (recap of the blocked GEMM structure) and "实验设置" (experimental
 *    setup).
 *  - The alpha/beta form C = alpha*A*B + beta*C is from the "DeepGEMM"
 *    article (demingchina.com), section 1.1; its extracted formula lost the
 *    "=" and "+" signs, and we read it as the standard BLAS update.
 *  - fp32 accumulation of low-precision products is the precision contract of
 *    the same article, section 3.1; the oracle accumulates in fp64, which is
 *    at least as accurate, so the GPU's fp32 sum is compared against the
 *    exact-up-to-fp64 value.
 *
 * Indexing: A[i,k] = A[i*lda + k], B[k,j] = B[j*ldb + k], C[i,j] = C[j*ldc + i].
 * bf16 values are the upper 16 bits of an IEEE binary32 and decode exactly to
 * double.  Every product of two bf16 values is exact in double.
 *
 * round_out: fp32 output rounds the double to nearest-even binary32; bf16
 * output rounds the double directly (once) to nearest-even bf16.
 *
 * Fused epilogue (the "DeepGEMM" article, section 6.1: after a fully
 * connected layer a bias is added and then ReLU or GELU applied, fused into
 * the end of the GEMM kernel).  The article fixes the order -- bias first,
 * then the activation, then the output -- but not where alpha and beta enter,
 * which axis the bias runs along, nor which GELU.  Readings taken:
 *
 *   E[i,j]     = act( D[i,j] + bias[j] )                    (fp64)
 *   C_out[i,j] = round_out(E[i,j])
 *
 * bias[j] is one value per output column j (per output feature of the layer
 * whose weights are B), fp32 or bf16, decoded exactly to double.  act is one
 * of
 *   none       act(x) = x
 *   relu       act(x) = max(x, 0); NaN stays NaN and -0 becomes +0
 *   gelu       act(x) = x * Phi(x), Phi the standard normal distribution
 *              function, Phi(x) = erfc(-x / sqrt(2)) / 2 (the definition of
 *              Hendrycks and Gimpel, "Gaussian Error Linear Units", 2016);
 *              written with erfc rather than 1 + erf so that negative x does
 *              not cancel
 *   gelu_tanh  the same paper's approximation
 *              x/2 * (1 + tanh( sqrt(2/pi) * (x + 0.044715 x^3) )),
 *              evaluated through the identity (1 + tanh z)/2 = 1/(1 + e^-2z)
 *              so that negative x does not cancel
 * Both sides of every identity above are equal in exact arithmetic; the
 * formulas produce NaN for x = -inf (0 * inf), and so does the oracle.
 *
 * FP8 inputs (the "DeepGEMM" article, section 6.3, names an FP8 input path as
 * the next step; it gives no format or scaling rules).  Readings taken: A and
 * B hold 8-bit floats in one of the two formats of the OCP 8-bit floating
 * point specification (Micikevicius et al., "FP8 Formats for Deep Learning",
 * 2022): E4M3 (bias 7, no infinities, S.1111.111 is NaN, largest 448) or E5M2
 * (bias 15, IEEE-style infinities and NaNs, largest 57344); both operands in
 * the same format, or A in one and B in the other (the two formats have
 * different range and precision; a product of one code of each is still
 * exact in double); same layouts and definition as above, with per-tensor
 * scale factors folded into alpha.  Every FP8 value decodes exactly to double
 * and every product of two is exact in double.
 *
 * Other operand layouts (the work log fixes A row-major and B column-major in
 * "实验设置"; the other three combinations are the same product with an
 * operand stored transposed): A column-major puts A[i,k] at A[k*lda + i]
 * (lda >= M), B row-major puts B[k,j] at B[k*ldb + j] (ldb >= N).  C stays
 * column-major.
 *
 * Quantising epilogue (the same article, section 6.2: y = round(x * scale +
 * zero_point) with one scale per row -- per token -- fused after the GEMM).
 * Readings taken: x is the epilogue's value E[i,j] above (with beta = 0: the
 * int8 output is not read); scale[i] is an fp32 value per row i of C; the
 * zero point is one integer; "round" is to nearest with ties to even; the
 * result saturates to the int8 range [-128, 127]; NaN gives 0, +-inf
 * saturate.  The code is an integer decided by floating point, so the oracle
 * takes that decision in the kernel's precision: E rounded once to fp32, then
 * q = rne(fmaf(E32, scale[i], zero_point)) with one fp32 rounding of the
 * fused multiply-add (C99 fmaf), then saturation.
 *
 * Planted mistakes: when compiled with -DORACLE_MUTANT=n (n > 0) one
 * deliberate error is switched on.  The test suite builds these variants to
 * prove that its pins catch every such error; the normal build has n = 0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ---- number formats --------------------------------------------------- */

/* bf16 -> double: bf16 is the upper half of a binary32, so widening the bit
 * pattern gives the exact float, and float -> double is exact. */
static double bf16_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_bf16_to_double(uint16_t h) { return bf16_to_double(h); }

/* double -> bf16, round to nearest, ties to even, in one step.
 * bf16 has 8 exponent bits (like binary32) and 7 stored fraction bits, so the
 * spacing of representable values in the binade [2^e, 2^(e+1)) is 2^(e-7),
 * and below the smallest normal 2^-126 the spacing stays 2^-133.  Dividing by
 * that spacing is an exact power-of-two scaling; nearbyint() in the default
 * rounding mode rounds to the nearest integer with ties to even. */
uint16_t oracle_round_bf16(double x) {
    if (isnan(x)) return (uint16_t)(signbit(x) ? 0xFFC0u : 0x7FC0u);
    if (isinf(x)) return (uint16_t)(signbit(x) ? 0xFF80u : 0x7F80u);
    if (x == 0.0) return (uint16_t)(signbit(x) ? 0x8000u : 0x0000u);
    int e;
    (void)frexp(fabs(x), &e);       /* |x| = m * 2^e, m in [0.5, 1)      */
    int lead = e - 1;               /* 2^lead <= |x| < 2^(lead+1)        */
    if (lead < -126) lead = -126;   /* subnormal range: fixed spacing    */
    double q = ldexp(1.0, lead - 7);
#if ORACLE_MUTANT == 7
    double r = trunc(x / q) * q;    /* planted: truncation instead of RNE */
#else
    double r = nearbyint(x / q) * q;
#endif
    if (fabs(r) >= ldexp(1.0, 128)) /* beyond the largest finite bf16    */
        return (uint16_t)(signbit(x) ? 0xFF80u : 0x7F80u);
    float f = (float)r;             /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* double -> binary32, round to nearest even (C's conversion in the default
 * rounding mode). */
float oracle_round_f32(double x) { return (float)x; }

void oracle_round_bf16_array(const double* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(x[i]);
}

void oracle_round_f32_array(const double* x, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_f32(x[i]);
}

/* ---- one output element ------------------------------------------------ */

typedef struct {
    int64_t M, N, K;
    const void* A; int64_t lda;
    const void* B; int64_t ldb;
    int in_kind;        /* 0 bf16; FP8: 1 both E4M3, 2 both E5M2, 3 A E4M3 and B E5M2, 4 A E5M2 and B E4M3 */
    int a_col, b_row;   /* 1: A column-major (A[k*lda + i]); 1: B row-major (B[k*ldb + j]) */
    const void* Cin; int64_t ldc; int cin_bf16; /* C_in dtype: 0 fp32, 1 bf16 */
    double alpha, beta;
    int absolute;       /* 1: sum |A[i,k]*B[k,j]| instead (error model, no alpha/beta) */
    const void* bias; int bias_kind;  /* 0 none, 1 fp32, 2 bf16 bits; one value per column j */
    int act;            /* 0 none, 1 relu, 2 gelu, 3 gelu_tanh */
} problem_t;

/* ---- activations (see the header) ------------------------------------- */

static double activation(double x, int act) {
    switch (act) {
    case 1:
        return (x > 0.0 || isnan(x)) ? x : 0.0;
    case 2:
#if ORACLE_MUTANT == 13
        return 0.5 * x * erfc(-x);                      /* planted: 1/sqrt(2) dropped */
#else
        return 0.5 * x * erfc(-x / sqrt(2.0));
#endif
    case 3: {
        const double c = sqrt(2.0 / acos(-1.0));        /* sqrt(2/pi) */
#if ORACLE_MUTANT == 14
        const double z = c * x;                         /* planted: cubic term dropped */
#else
        const double z = c * (x + 0.044715 * x * x * x);
#endif
        return x / (1.0 + exp(-2.0 * z));
    }
    default:
        return x;
    }
}

void oracle_activation_array(const double* x, double* out, int64_t n, int act) {
    for (int64_t i = 0; i < n; ++i) out[i] = activation(x[i], act);
}

static double bias_at(const problem_t* p, int64_t i, int64_t j) {
#if ORACLE_MUTANT == 11
    const int64_t idx = i;                              /* planted: bias along rows */
#else
    const int64_t idx = j;
    (void)i;
#endif
    if (p->bias_kind == 1) return (double)((const float*)p->bias)[idx];
    if (p->bias_kind == 2) return bf16_to_double(((const uint16_t*)p->bias)[idx]);
    return 0.0;
}

/* ---- FP8 formats ------------------------------------------------------ */

/* E4M3: sign, 4 exponent bits (bias 7), 3 fraction bits.  Exponent field 0
 * holds subnormals m/8 * 2^-6; the pattern S.1111.111 is NaN and there are no
 * infinities. */
static double e4m3_to_double(uint8_t v) {
    const int s = v >> 7, e = (v >> 3) & 0xF, m = v & 0x7;
    double x;
    if (e == 0xF && m == 0x7) return NAN;
#if ORACLE_MUTANT == 16
    if (e == 0) x = ldexp((double)m, -10);             /* planted: subnormal scale off by two */
#else
    if (e == 0) x = ldexp((double)m, -9);              /* (m/8) * 2^(1-7) */
#endif
    else x = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -x : x;
}

/* E5M2: sign, 5 exponent bits (bias 15), 2 fraction bits; exponent field 31
 * holds infinity (fraction 0) and NaN; field 0 holds subnormals m/4 * 2^-14. */
static double e5m2_to_double(uint8_t v) {
    const int s = v >> 7, e = (v >> 2) & 0x1F, m = v & 0x3;
    double x;
    if (e == 0x1F) x = m ? NAN : INFINITY;
    else if (e == 0) x = ldexp((double)m, -16);         /* (m/4) * 2^(1-15) */
#if ORACLE_MUTANT == 17
    else x = ldexp(1.0 + m / 4.0, e - 7);               /* planted: E4M3's bias used */
#else
    else x = ldexp(1.0 + m / 4.0, e - 15);
#endif
    return s ? -x : x;
}

double oracle_fp8_to_double(uint8_t v, int format) {
    return format == 0 ? e4m3_to_double(v) : e5m2_to_double(v);
}

/* The FP8 format of A (0 E4M3, 1 E5M2) and of B under an input kind. */
static int a_fp8_format(int kind) { return (kind == 2 || kind == 4) ? 1 : 0; }
static int b_fp8_format(int kind) {
#if ORACLE_MUTANT == 22
    return (kind == 2 || kind == 4) ? 1 : 0;            /* planted: B decoded in A's format */
#else
    return (kind == 2 || kind == 3) ? 1 : 0;
#endif
}

static double a_at(const problem_t* p, int64_t idx) {
    if (p->in_kind != 0) return oracle_fp8_to_double(((const uint8_t*)p->A)[idx], a_fp8_format(p->in_kind));
    return bf16_to_double(((const uint16_t*)p->A)[idx]);
}

static double b_at(const problem_t* p, int64_t idx) {
    if (p->in_kind != 0) return oracle_fp8_to_double(((const uint8_t*)p->B)[idx], b_fp8_format(p->in_kind));
    return bf16_to_double(((const uint16_t*)p->B)[idx]);
}

static double c_in_at(const problem_t* p, int64_t i, int64_t j) {
#if ORACLE_MUTANT == 8
    int64_t idx = i * p->N + j;     /* planted: C_in read row-major */
#else
    int64_t idx = j * p->ldc + i;
#endif
    if (p->cin_bf16) return bf16_to_double(((const uint16_t*)p->Cin)[idx]);
    return (double)((const float*)p->Cin)[idx];
}

static double element(const problem_t* p, int64_t i, int64_t j) {
#if ORACLE_MUTANT == 10
    float s = 0.0f;                 /* planted: fp32 accumulation */
#else
    double s = 0.0;
#endif
#if ORACLE_MUTANT == 5
    const int64_t kend = p->K > 0 ? p->K - 1 : 0;   /* planted: drops the last term */
#else
    const int64_t kend = p->K;
#endif
    for (int64_t k = 0; k < kend; ++k) {
#if ORACLE_MUTANT == 1
        double a = a_at(p, k * p->M + i);                /* planted: A as column-major */
#elif ORACLE_MUTANT == 21
        double a = a_at(p, p->a_col ? i * p->lda + k : i * p->lda + k);  /* planted: column-major A ignored */
#else
        double a = a_at(p, p->a_col ? k * p->lda + i : i * p->lda + k);
#endif
#if ORACLE_MUTANT == 2
        double b = b_at(p, k * p->N + j);                /* planted: B as row-major */
#else
        double b = b_at(p, p->b_row ? k * p->ldb + j : j * p->ldb + k);
#endif
        s += p->absolute ? fabs(a * b) : a * b;
    }
    if (p->absolute) return (double)s;
#if ORACLE_MUTANT == 4
    double d = p->beta * (double)s;                     /* planted: alpha and beta swapped */
    if (p->beta != 0.0) d += p->alpha * c_in_at(p, i, j);
#elif ORACLE_MUTANT == 3
    double d = p->alpha * (double)s;                    /* planted: beta term dropped */
#elif ORACLE_MUTANT == 6
    double d = p->alpha * (double)s;                    /* planted: wrong sign */
    if (p->beta != 0.0) d -= p->beta * c_in_at(p, i, j);
#elif ORACLE_MUTANT == 9
    double d = p->alpha * (double)s;                    /* planted: reads C even when beta == 0 */
    if (p->Cin != NULL) d += p->beta * c_in_at(p, i, j);
#elif ORACLE_MUTANT == 15
    double d = (double)s;                               /* planted: bias added before alpha */
    if (p->bias_kind != 0) d += bias_at(p, i, j);
    d *= p->alpha;
    if (p->beta != 0.0) d += p->beta * c_in_at(p, i, j);
    return activation(d, p->act);
#else
    double d = p->alpha * (double)s;
    if (p->beta != 0.0) d += p->beta * c_in_at(p, i, j);
#endif
    if (p->bias_kind == 0 && p->act == 0) return d;
#if ORACLE_MUTANT == 12
    return activation(d, p->act) + bias_at(p, i, j);    /* planted: activation before bias */
#else
    return activation(d + bias_at(p, i, j), p->act);
#endif
}

/* ---- full matrix, threaded over columns ------------------------------- */

int oracle_gemm_epi_f64(int64_t M, int64_t N, int64_t K,
                        const void* A, int64_t lda, const void* B, int64_t ldb, int in_kind,
                        const void* Cin, int64_t ldc, int cin_bf16,
                        float alpha, float beta, const void* bias, int bias_kind, int act,
                        double* D, int nthreads);
int oracle_gemm_epi_sampled_f64(int64_t M, int64_t N, int64_t K,
                                const void* A, int64_t lda, const void* B, int64_t ldb, int in_kind,
                                const void* Cin, int64_t ldc, int cin_bf16,
                                float alpha, float beta, const void* bias, int bias_kind, int act,
                                int64_t count, const int64_t* rows, const int64_t* cols,
                                double* out);

typedef struct {
    const problem_t* p;
    int64_t j0, j1;
    double* D; /* column-major, leading dimension M */
} job_t;

static void* run_columns(void* arg) {
    job_t* job = (job_t*)arg;
    const problem_t* p = job->p;
    for (int64_t j = job->j0; j < job->j1; ++j)
        for (int64_t i = 0; i < p->M; ++i)
            job->D[j * p->M + i] = element(p, i, j);
    return NULL;
}

static int pick_threads(int nthreads, int64_t units) {
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > units) nthreads = (int)(units > 0 ? units : 1);
    return nthreads;
}

int oracle_threads(int nthreads) { return pick_threads(nthreads, 1 << 30); }

/* D (column-major M x N, leading dimension M) = alpha*A*B + beta*C_in in fp64.
 * Returns 0 on success, -1 on a bad argument. */
static int run_full(const problem_t* pp, double* D, int nthreads);

int oracle_gemm_f64(int64_t M, int64_t N, int64_t K,
                    const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                    const void* Cin, int64_t ldc, int cin_bf16,
                    float alpha, float beta, double* D, int nthreads) {
    return oracle_gemm_epi_f64(M, N, K, A, lda, B, ldb, 0, Cin, ldc, cin_bf16, alpha, beta, NULL, 0, 0, D,
                               nthreads);
}

/* E = act(alpha*A*B + beta*C_in + bias) in fp64 (the fused epilogue, see the
 * header); bias_kind 0 and act 0 give D itself. */
int oracle_gemm_epi_f64(int64_t M, int64_t N, int64_t K,
                        const void* A, int64_t lda, const void* B, int64_t ldb, int in_kind,
                        const void* Cin, int64_t ldc, int cin_bf16,
                        float alpha, float beta, const void* bias, int bias_kind, int act,
                        double* D, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || ldc < M) return -1;
    if (beta != 0.0f && Cin == NULL) return -1;
    if (bias_kind < 0 || bias_kind > 2 || (bias_kind != 0 && bias == NULL) || act < 0 || act > 3) return -1;
    if (in_kind < 0 || in_kind > 4) return -1;
    problem_t p = {M, N, K, A, lda, B, ldb, in_kind, 0, 0, Cin, ldc, cin_bf16, (double)alpha, (double)beta, 0,
                   bias, bias_kind, act};
    return run_full(&p, D, nthreads);
}

static int run_full(const problem_t* pp, double* D, int nthreads) {
    const problem_t p = *pp;
    const int64_t N = p.N;
    if (p.M == 0 || N == 0) return 0;
    int nt = pick_threads(nthreads, N);
    pthread_t tid[256];
    int spawned[256];
    job_t jobs[256];
    int64_t per = (N + nt - 1) / nt;
    for (int t = 0; t < nt; ++t) {
        jobs[t].p = &p;
        jobs[t].j0 = t * per < N ? t * per : N;
        jobs[t].j1 = (t + 1) * per < N ? (t + 1) * per : N;
        jobs[t].D = D;
        spawned[t] = 0;
        if (t < nt - 1 && pthread_create(&tid[t], NULL, run_columns, &jobs[t]) == 0)
            spawned[t] = 1;
        else
            run_columns(&jobs[t]);  /* the last slice, or a failed spawn, runs here */
    }
    for (int t = 0; t < nt; ++t)
        if (spawned[t]) pthread_join(tid[t], NULL);
    return 0;
}

/* The same definition at selected (row, col) positions only. */
int oracle_gemm_sampled_f64(int64_t M, int64_t N, int64_t K,
                            const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                            const void* Cin, int64_t ldc, int cin_bf16,
                            float alpha, float beta,
                            int64_t count, const int64_t* rows, const int64_t* cols,
                            double* out) {
    return oracle_gemm_epi_sampled_f64(M, N, K, A, lda, B, ldb, 0, Cin, ldc, cin_bf16, alpha, beta, NULL, 0, 0,
                                       count, rows, cols, out);
}

int oracle_gemm_epi_sampled_f64(int64_t M, int64_t N, int64_t K,
                                const void* A, int64_t lda, const void* B, int64_t ldb, int in_kind,
                                const void* Cin, int64_t ldc, int cin_bf16,
                                float alpha, float beta, const void* bias, int bias_kind, int act,
                                int64_t count, const int64_t* rows, const int64_t* cols,
                                double* out) {
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || ldc < M) return -1;
    if (beta != 0.0f && Cin == NULL) return -1;
    if (bias_kind < 0 || bias_kind > 2 || (bias_kind != 0 && bias == NULL) || act < 0 || act > 3) return -1;
    if (in_kind < 0 || in_kind > 4) return -1;
    problem_t p = {M, N, K, A, lda, B, ldb, in_kind, 0, 0, Cin, ldc, cin_bf16, (double)alpha, (double)beta, 0,
                   bias, bias_kind, act};
    for (int64_t s = 0; s < count; ++s) {
        if (rows[s] < 0 || rows[s] >= M || cols[s] < 0 || cols[s] >= N) return -1;
        out[s] = element(&p, rows[s], cols[s]);
    }
    return 0;
}

/* Error model for the fp32-accumulation bound: G[i,j] = sum_k |A[i,k]*B[k,j]|
 * in fp64, at selected positions.  A recursive fp32 sum of these K products,
 * in any order, differs from the exact sum by at most about
 * K * 2^-24 * G[i,j] (the classical bound for floating-point summation). */
int oracle_absdot_kind_sampled_f64(int64_t M, int64_t N, int64_t K,
                                   const void* A, int64_t lda, const void* B, int64_t ldb, int in_kind,
                                   int64_t count, const int64_t* rows, const int64_t* cols,
                                   double* out) {
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || in_kind < 0 || in_kind > 4) return -1;
    problem_t p = {M, N, K, A, lda, B, ldb, in_kind, 0, 0, NULL, M, 0, 1.0, 0.0, 1, NULL, 0, 0};
    for (int64_t s = 0; s < count; ++s) {
        if (rows[s] < 0 || rows[s] >= M || cols[s] < 0 || cols[s] >= N) return -1;
        out[s] = element(&p, rows[s], cols[s]);
    }
    return 0;
}

int oracle_absdot_sampled_f64(int64_t M, int64_t N, int64_t K,
                              const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                              int64_t count, const int64_t* rows, const int64_t* cols,
                              double* out) {
    return oracle_absdot_kind_sampled_f64(M, N, K, A, lda, B, ldb, 0, count, rows, cols, out);
}

/* ---- quantising epilogue (see the header) ----------------------------- */

static int8_t quant_i8(double e, float scale, int32_t zero_point) {
    const float e32 = (float)e;
#if ORACLE_MUTANT == 20
    const float v = fmaf(e32, scale, 0.0f);               /* planted: zero point added after rounding */
#else
    const float v = fmaf(e32, scale, (float)zero_point);
#endif
    if (isnan(v)) return 0;
#if ORACLE_MUTANT == 18
    double r = trunc((double)v);                          /* planted: truncation instead of rounding */
#else
    double r = nearbyint((double)v);                      /* ties to even in the default rounding mode */
#endif
#if ORACLE_MUTANT == 20
    r += (double)zero_point;
#endif
#if ORACLE_MUTANT == 19
    return (int8_t)(uint8_t)(int64_t)fmod(r, 256.0);      /* planted: wraps instead of saturating */
#else
    if (r > 127.0) r = 127.0;
    if (r < -128.0) r = -128.0;
    return (int8_t)r;
#endif
}

/* Q (column-major M x N int8, leading dimension M) from E (same layout,
 * fp64): q[i,j] = quant(E[i,j], row_scale[i], zero_point). */
void oracle_quantize_i8(const double* E, int64_t M, int64_t N, const float* row_scale, int32_t zero_point,
                        int8_t* Q) {
    for (int64_t j = 0; j < N; ++j)
        for (int64_t i = 0; i < M; ++i) Q[j * M + i] = quant_i8(E[j * M + i], row_scale[i], zero_point);
}

/* The same at sampled positions: values[s] is E at (rows[s], any column). */
void oracle_quantize_i8_sampled(const double* values, int64_t count, const int64_t* rows, const float* row_scale,
                                int32_t zero_point, int8_t* out) {
    for (int64_t s = 0; s < count; ++s) out[s] = quant_i8(values[s], row_scale[rows[s]], zero_point);
}

/* D = alpha*A*B + beta*C_in in fp64 for bf16 operands in any of the four
 * layouts: a_col = 1 for column-major A (lda >= M), b_row = 1 for row-major
 * B (ldb >= N).  D as in oracle_gemm_f64. */
int oracle_gemm_layout_f64(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, int a_col,
                           const uint16_t* B, int64_t ldb, int b_row, const void* Cin, int64_t ldc, int cin_bf16,
                           float alpha, float beta, double* D, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || ldc < M) return -1;
    if (lda < (a_col ? M : K) || ldb < (b_row ? N : K)) return -1;
    if (beta != 0.0f && Cin == NULL) return -1;
    problem_t p = {M, N, K, A, lda, B, ldb, 0, a_col != 0, b_row != 0, Cin, ldc, cin_bf16, (double)alpha,
                   (double)beta, 0, NULL, 0, 0};
    return run_full(&p, D, nthreads);
}

int oracle_gemm_layout_sampled_f64(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, int a_col,
                                   const uint16_t* B, int64_t ldb, int b_row, const void* Cin, int64_t ldc,
                                   int cin_bf16, float alpha, float beta, int64_t count, const int64_t* rows,
                                   const int64_t* cols, double* out, int absolute) {
    if (M < 0 || N < 0 || K < 0 || ldc < M) return -1;
    if (lda < (a_col ? M : K) || ldb < (b_row ? N : K)) return -1;
    if (!absolute && beta != 0.0f && Cin == NULL) return -1;
    problem_t p = {M, N, K, A, lda, B, ldb, 0, a_col != 0, b_row != 0, absolute ? NULL : Cin, ldc, cin_bf16,
                   absolute ? 1.0 : (double)alpha, absolute ? 0.0 : (double)beta, absolute != 0, NULL, 0, 0};
    for (int64_t s = 0; s < count; ++s) {
        if (rows[s] < 0 || rows[s] >= M || cols[s] < 0 || cols[s] >= N) return -1;
        out[s] = element(&p, rows[s], cols[s]);
    }
    return 0;
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }
