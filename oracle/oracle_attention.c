/*
 * oracle_attention.c -- the fp64 CPU oracle for the attention block.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE (same rules as oracle_gemm.c: only
 * the tests, the smoke check and bench.py's CPU legs load it; it shares
 * nothing with the CUDA path).
 *
 * What it follows.  The FlashMLA example of the TileScale README (section
 * "Example of FlashMLA") runs, per block of query rows, a loop over key /
 * value blocks: scores acc_s = Q K^T, a running row maximum (scores_max),
 * the rescale factor of the previous partial results (scores_scale), the
 * exponentials of the scaled scores, their row sums (logsum), and an output
 * accumulator acc_o = acc_o * scores_scale + P V, divided by logsum at the
 * end.  Up to the order of operations and the running-maximum bookkeeping
 * (which cancels exactly in exact arithmetic), that computes
 *
 *     O[i] = sum_t w_it V[t],   w_it = exp(scale * s_it) / sum_u exp(scale * s_iu),
 *     s_it = sum_d Q[i][d] K[t][d],
 *
 * over the keys t that row i may see (all of them, or t <= i + Sk - Sq with
 * the causal mask).  This file writes that definition out in double
 * precision: the scores in order d = 0..D-1, the largest scaled score m_i,
 * the weights exp(scale * s_it - m_i) (the same ratio), their sum, and the
 * weighted sum of V in order t = 0, 1, ...  It also returns, per output
 * element, bound = sum_t w_it |V[t][e]|, the scale of the acceptance rule.
 * A row with no visible key is defined to be all zero.
 *
 * Tensors are [B][H][S][D] row-major 16-bit floats (decoded exactly by
 * oracle_decode in oracle_gemm.c).  Compiled with -ffp-contract=off.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

double oracle_decode(uint16_t bits, int dtype);
int oracle_default_threads(void);

typedef struct {
    int64_t B, H, Sq, Sk, D, Dv;
    const uint16_t *Q, *K, *V;
    int dtype, causal;
    double scale;
    double *O, *bound;
    int64_t bh_begin, bh_end; /* the (batch, head) pairs of this thread */
    int failed;
} attn_job_t;

/* Every output row of the (batch, head) pairs [bh_begin, bh_end).  A head's
 * keys and values are decoded once (exactly) into double; the arithmetic is
 * the definition above, row by row. */
static void* attn_heads(void* p) {
    attn_job_t* j = (attn_job_t*)p;
    const int64_t Sq = j->Sq, Sk = j->Sk, D = j->D, Dv = j->Dv;
    double* w = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
    double* kd = (double*)malloc(sizeof(double) * (size_t)(Sk * D > 0 ? Sk * D : 1));
    double* vd = (double*)malloc(sizeof(double) * (size_t)(Sk * Dv > 0 ? Sk * Dv : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)(D > 0 ? D : 1));
    if (!w || !kd || !vd || !qd) {
        j->failed = 1;
        free(w); free(kd); free(vd); free(qd);
        return NULL;
    }
    for (int64_t bh = j->bh_begin; bh < j->bh_end; ++bh) {
        const uint16_t* q = j->Q + bh * Sq * D;
        const uint16_t* k = j->K + bh * Sk * D;
        const uint16_t* v = j->V + bh * Sk * Dv;
        for (int64_t x = 0; x < Sk * D; ++x) kd[x] = oracle_decode(k[x], j->dtype);
        for (int64_t x = 0; x < Sk * Dv; ++x) vd[x] = oracle_decode(v[x], j->dtype);
        for (int64_t i = 0; i < Sq; ++i) {
            const int64_t last = j->causal ? i + Sk - Sq : Sk - 1;  /* last visible key */
            const int64_t n = last < 0 ? 0 : (last >= Sk ? Sk : last + 1);
            double* o = j->O + (bh * Sq + i) * Dv;
            double* bd = j->bound + (bh * Sq + i) * Dv;
            if (n == 0) {
                for (int64_t e = 0; e < Dv; ++e) o[e] = bd[e] = 0.0;
                continue;
            }
            for (int64_t d = 0; d < D; ++d) qd[d] = oracle_decode(q[i * D + d], j->dtype);
            double m = -INFINITY;
            for (int64_t t = 0; t < n; ++t) {
                double s = 0.0;
                for (int64_t d = 0; d < D; ++d) s += qd[d] * kd[t * D + d];
                w[t] = j->scale * s;
                if (w[t] > m) m = w[t];
            }
            double l = 0.0;
            for (int64_t t = 0; t < n; ++t) {
                w[t] = exp(w[t] - m);
                l += w[t];
            }
            for (int64_t e = 0; e < Dv; ++e) {
                double acc = 0.0, mag = 0.0;
                for (int64_t t = 0; t < n; ++t) {
                    const double xv = vd[t * Dv + e];
                    acc += w[t] * xv;
                    mag += w[t] * fabs(xv);
                }
                o[e] = acc / l;
                bd[e] = mag / l;
            }
        }
    }
    free(w); free(kd); free(vd); free(qd);
    return NULL;
}

/* Returns 0, or -1 when it cannot allocate its scratch.  The (batch, head)
 * pairs are shared out over one thread per online core; each output
 * element is computed by one thread in the order above, so the result does
 * not depend on the thread count. */
int oracle_attention(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t D, int64_t Dv,
                     const uint16_t* Q, const uint16_t* K, const uint16_t* V, int dtype,
                     double scale, int causal, double* O, double* bound) {
    const int64_t nbh = B * H;
    int nthreads = oracle_default_threads();
    if (nthreads > nbh) nthreads = (int)(nbh > 0 ? nbh : 1);
    attn_job_t* jobs = (attn_job_t*)calloc((size_t)nthreads, sizeof(attn_job_t));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -1; }
    for (int t = 0; t < nthreads; ++t)
        jobs[t] = (attn_job_t){B, H, Sq, Sk, D, Dv, Q, K, V, dtype, causal, scale, O, bound,
                               nbh * t / nthreads, nbh * (t + 1) / nthreads, 0};
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, attn_heads, &jobs[t]) != 0) break;
        started = t;
    }
    attn_heads(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    for (int t = started + 1; t < nthreads; ++t) attn_heads(&jobs[t]);
    int failed = 0;
    for (int t = 0; t < nthreads; ++t) failed |= jobs[t].failed;
    free(jobs);
    free(th);
    return failed ? -1 : 0;
}
