/*
 * oracle_gemm.c -- the fp64 CPU oracle for C = A*B.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check in __graft_entry__ and the CPU-baseline leg of bench.py may load
 * this library.  It shares no code, header, table or constant with the CUDA
 * path under hierarchical_gemm_gb300/.
 *
 * What it follows.  The tile-level GEMM skeleton of "TileScale 与 TileLang比较"
 * (yaopepe.com, section 核心抽象与编程模型对比, the TileLang single-device
 * GEMM) clears an accumulator C_r, adds the product of every BK-slice of A and
 * B into it, and copies C_r to C.  Up to the order of the additions that is
 * the plain definition
 *
 *     C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j],
 *
 * with A (M x K) and B (K x N) row-major, which the TileScale README (section
 * "Example of GEMM") also uses.  This file writes that definition out with no
 * tiling, fusion or reordering: for every (i, j) the K products are added in
 * the order k = 0, 1, ..., K-1 in double precision.  Inputs are 16-bit or
 * 8-bit floats; the product of two of them has at most 22 significant bits, so
 * every product is exact in double and only the additions round (relative
 * error of the sum <= K * 2^-53, far below any tolerance used against it).
 *
 * It also returns sabs[i][j] = sum_k |A[i][k] * B[k][j]|, the scale that the
 * acceptance rule |C - ref| <= 1e-3 * sabs + 1e-5 is measured against.
 *
 * Number formats are decoded from their IEEE-style definitions:
 *   binary16 : 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits
 *   bfloat16 : 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits
 *   FP8 E4M3 : 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; no
 *              infinities, S.1111.111 is NaN, largest finite 448 (OCP 8-bit
 *              floating point specification)
 *   FP8 E5M2 : 1 sign bit, 5 exponent bits (bias 15), 2 fraction bits, with
 *              IEEE infinities and NaNs (same specification)
 * and the output rounding (fp32 accumulator to a 16-bit output) is
 * round-to-nearest, ties-to-even, written out from the same definitions.
 *
 * Compiled with -ffp-contract=off so that no multiply-add is fused.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1
#define ORACLE_F32 2
#define ORACLE_E4M3 3
#define ORACLE_E5M2 4

/* Field widths of the two 16-bit formats. */
static int frac_bits(int dtype) { return dtype == ORACLE_F16 ? 10 : 7; }
static int exp_bits(int dtype) { return dtype == ORACLE_F16 ? 5 : 8; }
static int exp_bias(int dtype) { return dtype == ORACLE_F16 ? 15 : 127; }

/* Exact value of a 16-bit float given by its bit pattern. */
double oracle_decode(uint16_t bits, int dtype) {
    const int fb = frac_bits(dtype), eb = exp_bits(dtype), bias = exp_bias(dtype);
    const int sign = (bits >> 15) & 1;
    const int e = (bits >> fb) & ((1 << eb) - 1);
    const int f = bits & ((1 << fb) - 1);
    double v;
    if (e == (1 << eb) - 1) {
        v = f ? NAN : INFINITY;
    } else if (e == 0) {
        /* subnormal: f * 2^(1 - bias - fb) */
        v = ldexp((double)f, 1 - bias - fb);
    } else {
        /* normal: (2^fb + f) * 2^(e - bias - fb) */
        v = ldexp((double)((1 << fb) + f), e - bias - fb);
    }
    return sign ? -v : v;
}

/* Exact value of an 8-bit float given by its bit pattern. */
double oracle_decode8(uint8_t bits, int dtype) {
    const int sign = (bits >> 7) & 1;
    double v;
    if (dtype == ORACLE_E4M3) {
        const int e = (bits >> 3) & 15, f = bits & 7;
        if (e == 15 && f == 7)
            v = NAN;
        else if (e == 0)
            v = ldexp((double)f, 1 - 7 - 3);       /* subnormal: f * 2^-9 */
        else
            v = ldexp((double)(8 + f), e - 7 - 3); /* (1 + f/8) * 2^(e - 7) */
    } else {
        const int e = (bits >> 2) & 31, f = bits & 3;
        if (e == 31)
            v = f ? NAN : INFINITY;
        else if (e == 0)
            v = ldexp((double)f, 1 - 15 - 2);       /* subnormal: f * 2^-16 */
        else
            v = ldexp((double)(4 + f), e - 15 - 2); /* (1 + f/4) * 2^(e - 15) */
    }
    return sign ? -v : v;
}

void oracle_decode8_n(const uint8_t* bits, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_decode8(bits[i], dtype);
}

/* Round a double to the nearest 16-bit float, ties to even; returns the bits.
 * Values at or beyond the rounding boundary above the largest finite number
 * become +-infinity; NaN stays NaN. */
uint16_t oracle_round16(double x, int dtype) {
    const int fb = frac_bits(dtype), eb = exp_bits(dtype), bias = exp_bias(dtype);
    const int emax = (1 << eb) - 2 - bias; /* largest unbiased exponent */
    const int emin = 1 - bias;             /* smallest normal exponent */
    const uint16_t inf_bits = (uint16_t)(((1 << eb) - 1) << fb);
    uint16_t sign = 0;
    if (isnan(x)) return (uint16_t)(inf_bits | (1 << (fb - 1)));
    if (signbit(x)) { sign = 0x8000; x = -x; }
    if (isinf(x)) return (uint16_t)(sign | inf_bits);
    if (x == 0.0) return sign;

    int e2;
    (void)frexp(x, &e2);       /* x = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;            /* x in [2^E, 2^(E+1)) */
    if (E < emin) E = emin;    /* subnormal range shares the quantum of emin */
    /* quantum of the target format in this binade is 2^(E - fb) */
    double n = ldexp(x, fb - E); /* exact: scaling by a power of two */
    double fl = floor(n);
    double r = n - fl;           /* exact: n < 2^(fb+1) so fl and r are exact */
    double q = fl;
    if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) != 0.0)) q = fl + 1.0;
    /* q in [0, 2^(fb+1)]; a carry to 2^(fb+1) moves to the next binade */
    if (q == ldexp(1.0, fb + 1)) { q = ldexp(1.0, fb); E += 1; }
    if (q < ldexp(1.0, fb)) {
        /* subnormal (only possible when E == emin): exponent field 0 */
        return (uint16_t)(sign | (uint16_t)q);
    }
    if (E > emax) return (uint16_t)(sign | inf_bits);
    uint16_t efield = (uint16_t)(E + bias);
    uint16_t ffield = (uint16_t)(q - ldexp(1.0, fb));
    return (uint16_t)(sign | (efield << fb) | ffield);
}

/* Round a double to binary32 (the C conversion is round-to-nearest-even in
 * the default rounding mode); returns the value. */
float oracle_round32(double x) { return (float)x; }

/* Vector forms used from Python. */
void oracle_decode_n(const uint16_t* bits, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_decode(bits[i], dtype);
}
void oracle_round16_n(const double* x, int64_t n, int dtype, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round16(x[i], dtype);
}
void oracle_round32_n(const double* x, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round32(x[i]);
}

/* ---------------------------------------------------------------- GEMM -- */

typedef struct {
    int64_t M, N, K;
    const void* A;    /* 16-bit (elem 2) or 8-bit (elem 1) values, M x K row-major */
    int elem;
    const double* Bd; /* B decoded to double, K x N row-major */
    int dtype_in;
    double* ref;
    double* sabs;
    int64_t row_begin, row_end;
} gemm_job_t;

static double decode_a(const gemm_job_t* j, int64_t idx) {
    return j->elem == 1 ? oracle_decode8(((const uint8_t*)j->A)[idx], j->dtype_in)
                        : oracle_decode(((const uint16_t*)j->A)[idx], j->dtype_in);
}

/* Rows [row_begin, row_end) of ref and sabs.  For each row i the products
 * A[i][k] * B[k][j] are added into ref[i][j] for k = 0..K-1 in order, so each
 * output element is the definition's sum taken left to right. */
static void* gemm_rows(void* p) {
    gemm_job_t* j = (gemm_job_t*)p;
    const int64_t N = j->N, K = j->K;
    for (int64_t i = j->row_begin; i < j->row_end; ++i) {
        double* r = j->ref + i * N;
        double* s = j->sabs + i * N;
        for (int64_t c = 0; c < N; ++c) { r[c] = 0.0; s[c] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            const double a = decode_a(j, i * K + k);
            const double* b = j->Bd + k * N;
            for (int64_t c = 0; c < N; ++c) {
                const double p_ = a * b[c]; /* exact */
                r[c] += p_;
                s[c] += fabs(p_);
            }
        }
    }
    return NULL;
}

int oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int gemm_any(int64_t M, int64_t N, int64_t K, const void* A, const void* B, int elem,
                    int dtype_in, double* ref, double* sabs, int nthreads) {
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > M) nthreads = (int)(M > 0 ? M : 1);
    double* Bd = (double*)malloc((size_t)(K * N > 0 ? K * N : 1) * sizeof(double));
    if (!Bd) return -1;
    if (elem == 1)
        oracle_decode8_n((const uint8_t*)B, K * N, dtype_in, Bd);
    else
        oracle_decode_n((const uint16_t*)B, K * N, dtype_in, Bd);
    gemm_job_t* jobs = (gemm_job_t*)calloc((size_t)nthreads, sizeof(gemm_job_t));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(Bd); free(jobs); free(th); return -1; }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (gemm_job_t){M, N, K, A, elem, Bd, dtype_in, ref, sabs,
                               M * t / nthreads, M * (t + 1) / nthreads};
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, gemm_rows, &jobs[t]) != 0) break;
        started = t;
    }
    gemm_rows(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    /* rows of any thread that failed to start are done here */
    for (int t = started + 1; t < nthreads; ++t) gemm_rows(&jobs[t]);
    free(Bd);
    free(jobs);
    free(th);
    return nthreads;
}

/* ref, sabs: M x N row-major outputs of A (M x K) times B (K x N), both of
 * 16-bit floats.  nthreads <= 0 means one per online core.  Returns the
 * number of threads used, or -1 on allocation failure. */
int oracle_gemm(int64_t M, int64_t N, int64_t K, const uint16_t* A,
                const uint16_t* B, int dtype_in, double* ref, double* sabs,
                int nthreads) {
    return gemm_any(M, N, K, A, B, 2, dtype_in, ref, sabs, nthreads);
}

/* The same for 8-bit float inputs (FP8 E4M3 or E5M2). */
int oracle_gemm8(int64_t M, int64_t N, int64_t K, const uint8_t* A,
                 const uint8_t* B, int dtype_in, double* ref, double* sabs,
                 int nthreads) {
    return gemm_any(M, N, K, A, B, 1, dtype_in, ref, sabs, nthreads);
}

/* The same definition evaluated only at `count` output positions
 * (rows[s], cols[s]); used where the full product would take too long. */
void oracle_gemm_sampled(int64_t M, int64_t N, int64_t K, const uint16_t* A,
                         const uint16_t* B, int dtype_in, int64_t count,
                         const int64_t* rows, const int64_t* cols, double* ref,
                         double* sabs) {
    (void)M;
    for (int64_t s = 0; s < count; ++s) {
        const int64_t i = rows[s], c = cols[s];
        double r = 0.0, a_ = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double p_ = oracle_decode(A[i * K + k], dtype_in) *
                              oracle_decode(B[k * N + c], dtype_in);
            r += p_;
            a_ += fabs(p_);
        }
        ref[s] = r;
        sabs[s] = a_;
    }
}

void oracle_gemm8_sampled(int64_t M, int64_t N, int64_t K, const uint8_t* A,
                          const uint8_t* B, int dtype_in, int64_t count,
                          const int64_t* rows, const int64_t* cols, double* ref,
                          double* sabs) {
    (void)M;
    for (int64_t s = 0; s < count; ++s) {
        const int64_t i = rows[s], c = cols[s];
        double r = 0.0, a_ = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double p_ = oracle_decode8(A[i * K + k], dtype_in) *
                              oracle_decode8(B[k * N + c], dtype_in);
            r += p_;
            a_ += fabs(p_);
        }
        ref[s] = r;
        sabs[s] = a_;
    }
}
