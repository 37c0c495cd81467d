/*
 * router_oracle.c -- plain CPU oracle of the quantile-balancing router-bias
 * update (aux-loss-free load balancing).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes, for routing logits x [T, E] of a statistics window and a
 * per-expert bias [E] [P1 §4.2, P2 §3.2, P3 §4.3, P4 §3.2]:
 *   1. score s_te = x_te + bias_e, added in binary32 (the bias only steers the
 *      selection); each token picks the k experts of largest score, ties
 *      going to the lower expert index;
 *   2. load_e += the number of tokens that picked expert e (int64 counts,
 *      accumulated over calls, so a window may span several batches);
 *   3. quantiles of the E loads by linear interpolation between order
 *      statistics (x sorted ascending, p = q (E - 1), i = floor(p),
 *      Q = x_i + (p - i)(x_{i+1} - x_i)), in binary64;
 *   4. the update, in one of the two forms the pages print:
 *      sign:         bias_e -= eta where load_e > Q(q_hi),
 *                    bias_e += eta where load_e < Q(q_lo)
 *                    (q_lo = q_hi = q is the single-threshold form);
 *      proportional: bias_e += eta (Q(q_hi) - load_e) / Q(q_hi), skipped when
 *                    Q(q_hi) = 0; computed in binary64, rounded once to binary32.
 *
 * Citation keys (page title, section):
 *   P1 = "Deep Dive: The Next Generation of Ultra-Long Context Sparse MoE LLMs"
 *   P2 = "Core Technologies Behind Ultra-Long-Context Sparse MoE Large Models"
 *   P3 = "How Trillion-Scale Sparse MoE Models Achieve Million-Token Long
 *         Context Capabilities"
 *   P4 = "Evaluating Next-Gen Sparse MoE and Long-Context LLMs"
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { RO_BF16 = 0, RO_F32 = 1 };
enum { RO_SIGN = 0, RO_PROPORTIONAL = 1 };

static float logit_at(const void *x, int dtype, int64_t i)
{
    if (dtype == RO_F32) return ((const float *)x)[i];
    uint32_t u = (uint32_t)((const uint16_t *)x)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Top-k of every token by repeated selection of the best remaining expert. */
int gdr_oracle_router_topk(const void *logits, int dtype, const float *bias, int64_t T, int E,
                           int k, int32_t *idx, float *sel_logit, int64_t *load)
{
    if (T < 0 || E < 1 || k < 1 || k > E || (dtype != RO_BF16 && dtype != RO_F32)) return 1;
    float *s = (float *)malloc(sizeof(float) * (size_t)E);
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    for (int64_t t = 0; t < T; t++) {
        for (int e = 0; e < E; e++) {
            s[e] = logit_at(logits, dtype, t * E + e) + bias[e];
            taken[e] = 0;
        }
        for (int r = 0; r < k; r++) {
            int best = -1;
            for (int e = 0; e < E; e++) {
                if (taken[e]) continue;
                if (best < 0 || s[e] > s[best]) best = e;   /* strict: ties keep the lower index */
            }
            taken[best] = 1;
            idx[t * k + r] = best;
            if (sel_logit) sel_logit[t * k + r] = logit_at(logits, dtype, t * E + best);
            if (load) load[best] += 1;
        }
    }
    free(s);
    free(taken);
    return 0;
}

static int cmp_i64(const void *a, const void *b)
{
    const int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return (x > y) - (x < y);
}

static double quantile_sorted(const int64_t *xs, int E, double q)
{
    const double p = q * (double)(E - 1);
    int i = (int)floor(p);
    if (i > E - 1) i = E - 1;
    const int j = i + 1 < E ? i + 1 : i;
    return (double)xs[i] + (p - (double)i) * ((double)xs[j] - (double)xs[i]);
}

int gdr_oracle_router_update(const int64_t *load, int E, float *bias, int mode, double q_lo,
                             double q_hi, float eta, double *thresholds)
{
    if (E < 1 || !(q_lo >= 0.0 && q_lo <= 1.0) || !(q_hi >= 0.0 && q_hi <= 1.0)) return 1;
    if (mode != RO_SIGN && mode != RO_PROPORTIONAL) return 1;
    int64_t *xs = (int64_t *)malloc(sizeof(int64_t) * (size_t)E);
    memcpy(xs, load, sizeof(int64_t) * (size_t)E);
    qsort(xs, (size_t)E, sizeof(int64_t), cmp_i64);
    const double Qlo = quantile_sorted(xs, E, q_lo), Qhi = quantile_sorted(xs, E, q_hi);
    free(xs);
    if (thresholds) {
        thresholds[0] = Qlo;
        thresholds[1] = Qhi;
    }
    for (int e = 0; e < E; e++) {
        const double l = (double)load[e];
        if (mode == RO_SIGN) {
            if (l > Qhi) bias[e] = bias[e] - eta;
            else if (l < Qlo) bias[e] = bias[e] + eta;
        } else if (Qhi != 0.0) {
            bias[e] = (float)((double)bias[e] + (double)eta * (Qhi - l) / Qhi);
        }
    }
    return 0;
}
