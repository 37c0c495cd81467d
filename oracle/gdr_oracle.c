/*
 * gdr_oracle.c -- fp64 CPU oracle for the gated delta-rule forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes (the plain definition, token by token, no chunking):
 *
 *   g_t   = -b * sigmoid(a_t)            bounded log-decay          [P1 §3.3, P2 §2.2,
 *                                                                     P3 §3.2, P4 §2.3]
 *   g_t   = -softplus(a_t)               unbounded variant the pages replace
 *                                                                    [P1 §3.3, P3 §3.2]
 *   alpha = exp(g_t)
 *   H_t   = alpha * H_{t-1} + beta_t * k_t (v_t - alpha * H_{t-1}^T k_t)^T
 *   o_t   = H_t^T q_t
 *
 * H is the dk x dv state (H = S^T for the dv x dk state S of the delta rule
 * written as S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 * o_t = S_t q_t).  The pages describe the layer only as a fixed-size matrix
 * state updated token by token by a delta-rule write with a data-dependent
 * decay [P4 §2.2 "Incremental Linear Attention", P3 §2.2]; the closed form
 * above is the plainest reading of that description.  With erase = 0 the
 * correction term is dropped (H_t = alpha H_{t-1} + beta k v^T): that is
 * the plain gated linear-attention recurrence, used only by the pins.
 *
 * Citation keys (page title, section):
 *   P1 = "Deep Dive: The Next Generation of Ultra-Long Context Sparse MoE LLMs"
 *   P2 = "Core Technologies Behind Ultra-Long-Context Sparse MoE Large Models"
 *   P3 = "How Trillion-Scale Sparse MoE Models Achieve Million-Token Long
 *         Context Capabilities"
 *   P4 = "Evaluating Next-Gen Sparse MoE and Long-Context LLMs"
 *
 * Layouts (row-major, contiguous):
 *   dense  : q,k [B,T,H,dk]  v [B,T,H,dv]  a,beta [B,T,H]
 *   varlen : the same with B = 1 and T = total tokens; cu_seqlens[N+1]
 *            splits the token axis into N sequences (cu[0]=0, cu[N]=T).
 *   h0, hT : [N,H,dk,dv] fp64 (N = B for dense input)
 *   out    : [B,T,H,dv] fp64
 * Inputs are read in their stored precision (bf16 bit patterns, fp32 or
 * fp64) and widened exactly to fp64 before any arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_BF16 = 0, OR_F32 = 1, OR_F64 = 2 };
enum { OR_GATE_BOUNDED = 0, OR_GATE_SOFTPLUS = 1 };

/* Widen element i of a buffer stored as dtype to double (exact). */
static double widen(const void *p, int dtype, int64_t i)
{
    if (dtype == OR_F64) return ((const double *)p)[i];
    if (dtype == OR_F32) return (double)((const float *)p)[i];
    /* bf16: the upper 16 bits of an IEEE binary32 */
    uint32_t bits = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Logistic function, evaluated without overflow for either sign. */
static double sigmoid(double x)
{
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}

/* log(1 + exp(x)) without overflow. */
static double softplus(double x)
{
    if (x > 0.0) return x + log1p(exp(-x));
    return log1p(exp(x));
}

/* The log-decay g_t of one token [P1 §3.3, P2 §2.2, P3 §3.2, P4 §2.3]. */
double gdr_oracle_gate(double a, double b, int gate)
{
    if (gate == OR_GATE_SOFTPLUS) return -softplus(a);
    return -b * sigmoid(a);
}

/*
 * Run the recurrence for every (sequence, head) and a block of dv columns.
 * Columns of H evolve independently given (k, beta, g): column j only ever
 * sees k, q, beta, g and v[:, j].  That is what the OpenMP split uses.
 */
int gdr_oracle_fwd(const void *q, const void *k, const void *v, const void *a,
                   const void *beta, int in_dtype, const double *h0, double *out,
                   double *hT, const int64_t *cu_seqlens, int B, int64_t T, int H,
                   int dk, int dv, double b, int gate, int erase, int nthreads)
{
    if (B < 1 || T < 0 || H < 1 || dk < 1 || dv < 1) return 1;
    if (in_dtype < OR_BF16 || in_dtype > OR_F64) return 1;
    int N = B;
    if (cu_seqlens) {
        if (cu_seqlens[0] != 0) return 2;
        for (int n = 0; n < N; n++)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return 2;
        if (cu_seqlens[N] != T) return 2;
    }
    const int CB = 16; /* dv columns per task */
    const int ncb = (dv + CB - 1) / CB;
    const int64_t ntask = (int64_t)N * H * ncb;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel
    {
        double *Hs = (double *)malloc(sizeof(double) * (size_t)dk * CB);
        double *kt = (double *)malloc(sizeof(double) * (size_t)dk);
        double *qt = (double *)malloc(sizeof(double) * (size_t)dk);
#pragma omp for schedule(dynamic, 1)
        for (int64_t task = 0; task < ntask; task++) {
            const int cb = (int)(task % ncb);
            const int h = (int)((task / ncb) % H);
            const int n = (int)(task / ((int64_t)ncb * H));
            const int j0 = cb * CB;
            const int nc = (dv - j0) < CB ? (dv - j0) : CB;
            /* token range of this sequence, as rows of the [*, H, *] tensors */
            int64_t t_begin, t_end;
            if (cu_seqlens) {
                t_begin = cu_seqlens[n];
                t_end = cu_seqlens[n + 1];
            } else {
                t_begin = (int64_t)n * T;
                t_end = t_begin + T;
            }
            /* H <- h0 (or 0) */
            for (int i = 0; i < dk; i++)
                for (int c = 0; c < nc; c++)
                    Hs[i * CB + c] = h0 ? h0[(((int64_t)n * H + h) * dk + i) * dv + j0 + c] : 0.0;

            for (int64_t t = t_begin; t < t_end; t++) {
                const int64_t row = t * H + h; /* (token, head) row */
                const double g = gdr_oracle_gate(widen(a, in_dtype, row), b, gate);
                const double alpha = exp(g);
                const double bt = widen(beta, in_dtype, row);
                for (int i = 0; i < dk; i++) {
                    kt[i] = widen(k, in_dtype, row * dk + i);
                    qt[i] = widen(q, in_dtype, row * dk + i);
                }
                for (int c = 0; c < nc; c++) {
                    const double vj = widen(v, in_dtype, row * dv + j0 + c);
                    /* p = alpha * H^T k  (decayed prediction for column j) */
                    double p = 0.0;
                    if (erase) {
                        for (int i = 0; i < dk; i++) p += Hs[i * CB + c] * kt[i];
                        p *= alpha;
                    }
                    const double delta = bt * (vj - p);
                    double o = 0.0;
                    for (int i = 0; i < dk; i++) {
                        const double hij = alpha * Hs[i * CB + c] + kt[i] * delta;
                        Hs[i * CB + c] = hij;
                        o += hij * qt[i];
                    }
                    out[row * dv + j0 + c] = o;
                }
            }
            if (hT)
                for (int i = 0; i < dk; i++)
                    for (int c = 0; c < nc; c++)
                        hT[(((int64_t)n * H + h) * dk + i) * dv + j0 + c] = Hs[i * CB + c];
        }
        free(Hs);
        free(kt);
        free(qt);
    }
    return 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int gdr_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
