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
#include <stdint.h>
#include <stdlib.h>

double oracle_decode(uint16_t bits, int dtype);

/* Returns 0, or -1 when it cannot allocate its scratch. */
int oracle_attention(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t D, int64_t Dv,
                     const uint16_t* Q, const uint16_t* K, const uint16_t* V, int dtype,
                     double scale, int causal, double* O, double* bound) {
    double* w = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
    if (!w) return -1;
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const uint16_t* q = Q + bh * Sq * D;
        const uint16_t* k = K + bh * Sk * D;
        const uint16_t* v = V + bh * Sk * Dv;
        for (int64_t i = 0; i < Sq; ++i) {
            const int64_t last = causal ? i + Sk - Sq : Sk - 1;  /* last visible key */
            const int64_t n = last < 0 ? 0 : (last >= Sk ? Sk : last + 1);
            double* o = O + (bh * Sq + i) * Dv;
            double* bd = bound + (bh * Sq + i) * Dv;
            if (n == 0) {
                for (int64_t e = 0; e < Dv; ++e) o[e] = bd[e] = 0.0;
                continue;
            }
            double m = -INFINITY;
            for (int64_t t = 0; t < n; ++t) {
                double s = 0.0;
                for (int64_t d = 0; d < D; ++d)
                    s += oracle_decode(q[i * D + d], dtype) * oracle_decode(k[t * D + d], dtype);
                w[t] = scale * s;
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
                    const double x = oracle_decode(v[t * Dv + e], dtype);
                    acc += w[t] * x;
                    mag += w[t] * fabs(x);
                }
                o[e] = acc / l;
                bd[e] = mag / l;
            }
        }
    }
    free(w);
    return 0;
}
