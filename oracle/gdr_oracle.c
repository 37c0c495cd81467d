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

/*
 * Per-channel (vector) decay: a carries one gate input per key channel, a is
 * [rows, dk], and token t decays row i of H by its own factor
 * alpha_{t,i} = exp(g(a_{t,i})) [P1 §2.1-2.2 and P4 §3 give the decay as the
 * data-dependent factor whose log is bounded; a decay per key channel is the
 * plainest reading of a vector-valued log-decay g_t]:
 *
 *   Hb  = diag(alpha_t) H_{t-1}
 *   H_t = Hb + beta_t k_t (v_t - Hb^T k_t)^T = (I - beta_t k_t k_t^T) Hb + beta_t k_t v_t^T
 *   o_t = H_t^T q_t
 *
 * With every channel given the same a this is gdr_oracle_fwd exactly.
 */
int gdr_oracle_fwd_vec(const void *q, const void *k, const void *v, const void *a,
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
    const int CB = 16;
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
        double *al = (double *)malloc(sizeof(double) * (size_t)dk);
#pragma omp for schedule(dynamic, 1)
        for (int64_t task = 0; task < ntask; task++) {
            const int cb = (int)(task % ncb);
            const int h = (int)((task / ncb) % H);
            const int n = (int)(task / ((int64_t)ncb * H));
            const int j0 = cb * CB;
            const int nc = (dv - j0) < CB ? (dv - j0) : CB;
            const int64_t t_begin = cu_seqlens ? cu_seqlens[n] : (int64_t)n * T;
            const int64_t t_end = cu_seqlens ? cu_seqlens[n + 1] : t_begin + T;
            for (int i = 0; i < dk; i++)
                for (int c = 0; c < nc; c++)
                    Hs[i * CB + c] = h0 ? h0[((int64_t)(n * H + h) * dk + i) * dv + j0 + c] : 0.0;
            for (int64_t t = t_begin; t < t_end; t++) {
                const int64_t row = t * H + h;
                const double bt = widen(beta, in_dtype, row);
                for (int i = 0; i < dk; i++) {
                    al[i] = exp(gdr_oracle_gate(widen(a, in_dtype, row * dk + i), b, gate));
                    kt[i] = widen(k, in_dtype, row * dk + i);
                    qt[i] = widen(q, in_dtype, row * dk + i);
                }
                for (int c = 0; c < nc; c++) {
                    /* decay each row by its channel's factor, then predict v */
                    double p = 0.0;
                    for (int i = 0; i < dk; i++) {
                        Hs[i * CB + c] *= al[i];
                        p += kt[i] * Hs[i * CB + c];
                    }
                    const double delta = bt * (widen(v, in_dtype, row * dv + j0 + c) - (erase ? p : 0.0));
                    double o = 0.0;
                    for (int i = 0; i < dk; i++) {
                        Hs[i * CB + c] += kt[i] * delta;
                        o += Hs[i * CB + c] * qt[i];
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
        free(al);
    }
    return 0;
}

/* d g / d a of the log-decay, for the backward pass. */
static double gate_grad(double a, double b, int gate)
{
    const double s = sigmoid(a);
    if (gate == OR_GATE_SOFTPLUS) return -s;
    return -b * s * (1.0 - s);
}

/*
 * Gradients of L = <dout, out> + <dhT, hT> with respect to q, k, v, a, beta
 * and h0, for the recurrence of gdr_oracle_fwd (erase on).  Per token, with
 * Hb = alpha H_{t-1}, p = Hb^T k, delta = beta (v - p), H_t = Hb + k delta^T,
 * o = H_t^T q, the adjoints run backwards over the tokens:
 *     dH     += q do^T            dq     = H_t do
 *     dk     += dH delta          ddelta = dH^T k
 *     dv      = beta ddelta       dbeta  = ddelta . (v - p)
 *     dp      = -beta ddelta      dHb    = dH + k dp^T        dk += Hb dp
 *     dalpha  = <H_{t-1}, dHb>    da     = dalpha alpha g'(a)  dH <- alpha dHb
 * and dh0 is the final dH.  The states are recomputed forward from
 * checkpoints kept every CK tokens.  dout and dhT may be NULL (zero); dhT and
 * dh0 are [N,H,dk,dv]; the token gradients have the input layouts.
 */
int gdr_oracle_bwd(const void *q, const void *k, const void *v, const void *a,
                   const void *beta, int in_dtype, const double *h0, const double *dout,
                   const double *dhT, double *dq, double *dk_out, double *dv_out, double *da,
                   double *dbeta, double *dh0, const int64_t *cu_seqlens, int B, int64_t T,
                   int H, int dk, int dv, double b, int gate, int nthreads)
{
    if (B < 1 || T < 0 || H < 1 || dk < 1 || dv < 1) return 1;
    if (in_dtype < OR_BF16 || in_dtype > OR_F64) return 1;
    const int N = B;
    if (cu_seqlens) {
        if (cu_seqlens[0] != 0) return 2;
        for (int n = 0; n < N; n++)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return 2;
        if (cu_seqlens[N] != T) return 2;
    }
    enum { CK = 64 };
    const int64_t S = (int64_t)dk * dv;
    const int64_t nunit = (int64_t)N * H;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int rc = 0;
#pragma omp parallel
    {
        double *blk = (double *)malloc(sizeof(double) * (size_t)(CK + 1) * S); /* states of a block */
        double *dH = (double *)malloc(sizeof(double) * (size_t)S);
        double *kt = (double *)malloc(sizeof(double) * (size_t)dk);
        double *qt = (double *)malloc(sizeof(double) * (size_t)dk);
        double *p = (double *)malloc(sizeof(double) * (size_t)dv);
        double *dl = (double *)malloc(sizeof(double) * (size_t)dv);
        double *ddl = (double *)malloc(sizeof(double) * (size_t)dv);
        double *dp = (double *)malloc(sizeof(double) * (size_t)dv);
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < nunit; u++) {
            const int h = (int)(u % H);
            const int n = (int)(u / H);
            int64_t t_begin, t_end;
            if (cu_seqlens) {
                t_begin = cu_seqlens[n];
                t_end = cu_seqlens[n + 1];
            } else {
                t_begin = (int64_t)n * T;
                t_end = t_begin + T;
            }
            const int64_t len = t_end - t_begin;
            const int64_t nck = (len + CK - 1) / CK + 1;
            double *ck = (double *)malloc(sizeof(double) * (size_t)(nck > 0 ? nck : 1) * S);
            if (!ck) {
                rc = 3;
                continue;
            }
            /* one forward step: from state Hp to Hn at token row, also p and delta */
#define STEP(Hp, Hn, row, alpha, bt)                                                   \
    do {                                                                               \
        for (int i = 0; i < dk; i++) kt[i] = widen(k, in_dtype, (row) * dk + i);       \
        for (int j = 0; j < dv; j++) {                                                 \
            double acc = 0.0;                                                          \
            for (int i = 0; i < dk; i++) acc += (Hp)[i * dv + j] * kt[i];              \
            p[j] = (alpha) * acc;                                                      \
            dl[j] = (bt) * (widen(v, in_dtype, (row) * dv + j) - p[j]);                \
        }                                                                              \
        for (int i = 0; i < dk; i++)                                                   \
            for (int j = 0; j < dv; j++)                                               \
                (Hn)[i * dv + j] = (alpha) * (Hp)[i * dv + j] + kt[i] * dl[j];         \
    } while (0)
            /* forward: checkpoints at tokens 0, CK, 2 CK, ... of the sequence */
            double *Hc = blk, *Hn = blk + S;
            for (int64_t e = 0; e < S; e++) Hc[e] = h0 ? h0[u * S + e] : 0.0;
            memcpy(ck, Hc, sizeof(double) * (size_t)S);
            for (int64_t t = 0; t < len; t++) {
                const int64_t row = (t_begin + t) * H + h;
                const double alpha = exp(gdr_oracle_gate(widen(a, in_dtype, row), b, gate));
                const double bt = widen(beta, in_dtype, row);
                STEP(Hc, Hn, row, alpha, bt);
                double *tmp = Hc;
                Hc = Hn;
                Hn = tmp;
                if ((t + 1) % CK == 0) memcpy(ck + ((t + 1) / CK) * S, Hc, sizeof(double) * (size_t)S);
            }
            /* backward */
            for (int64_t e = 0; e < S; e++) dH[e] = dhT ? dhT[u * S + e] : 0.0;
            for (int64_t c0 = ((len - 1) / CK) * CK; len > 0 && c0 >= 0; c0 -= CK) {
                const int64_t c1 = (c0 + CK < len) ? c0 + CK : len;
                /* states H_{c0} .. H_{c1} of this block */
                memcpy(blk, ck + (c0 / CK) * S, sizeof(double) * (size_t)S);
                for (int64_t t = c0; t < c1; t++) {
                    const int64_t row = (t_begin + t) * H + h;
                    const double alpha = exp(gdr_oracle_gate(widen(a, in_dtype, row), b, gate));
                    const double bt = widen(beta, in_dtype, row);
                    STEP(blk + (t - c0) * S, blk + (t - c0 + 1) * S, row, alpha, bt);
                }
                for (int64_t t = c1 - 1; t >= c0; t--) {
                    const int64_t row = (t_begin + t) * H + h;
                    const double av = widen(a, in_dtype, row);
                    const double alpha = exp(gdr_oracle_gate(av, b, gate));
                    const double bt = widen(beta, in_dtype, row);
                    const double *Hp = blk + (t - c0) * S;     /* H_{t-1} */
                    const double *Ht = blk + (t - c0 + 1) * S; /* H_t */
                    for (int i = 0; i < dk; i++) {
                        kt[i] = widen(k, in_dtype, row * dk + i);
                        qt[i] = widen(q, in_dtype, row * dk + i);
                    }
                    /* p and delta of this token */
                    for (int j = 0; j < dv; j++) {
                        double acc = 0.0;
                        for (int i = 0; i < dk; i++) acc += Hp[i * dv + j] * kt[i];
                        p[j] = alpha * acc;
                        dl[j] = bt * (widen(v, in_dtype, row * dv + j) - p[j]);
                    }
                    /* o = H_t^T q */
                    for (int i = 0; i < dk; i++) {
                        double acc = 0.0;
                        for (int j = 0; j < dv; j++) {
                            const double g_o = dout ? dout[row * dv + j] : 0.0;
                            dH[i * dv + j] += qt[i] * g_o;
                            acc += Ht[i * dv + j] * g_o;
                        }
                        dq[row * dk + i] = acc;
                    }
                    /* H_t = Hb + k delta^T */
                    double dbt = 0.0;
                    for (int j = 0; j < dv; j++) {
                        double acc = 0.0;
                        for (int i = 0; i < dk; i++) acc += dH[i * dv + j] * kt[i];
                        ddl[j] = acc;
                        dv_out[row * dv + j] = bt * acc;
                        dbt += acc * (widen(v, in_dtype, row * dv + j) - p[j]);
                        dp[j] = -bt * acc;
                    }
                    dbeta[row] = dbt;
                    double dalpha = 0.0;
                    for (int i = 0; i < dk; i++) {
                        double g_k = 0.0;
                        for (int j = 0; j < dv; j++) {
                            g_k += dH[i * dv + j] * dl[j];                   /* from k delta^T */
                            g_k += alpha * Hp[i * dv + j] * dp[j];           /* from p = Hb^T k */
                            const double dhb = dH[i * dv + j] + kt[i] * dp[j];
                            dalpha += Hp[i * dv + j] * dhb;
                            dH[i * dv + j] = alpha * dhb;
                        }
                        dk_out[row * dk + i] = g_k;
                    }
                    da[row] = dalpha * alpha * gate_grad(av, b, gate);
                }
            }
#undef STEP
            for (int64_t e = 0; e < S; e++)
                if (dh0) dh0[u * S + e] = dH[e];
            free(ck);
        }
        free(blk);
        free(dH);
        free(kt);
        free(qt);
        free(p);
        free(dl);
        free(ddl);
        free(dp);
    }
    return rc;
}

/*
 * Gradients for the per-channel decay form of gdr_oracle_fwd_vec: row i of the
 * state decays by al_i = exp(g(a_{t,i})).  With Hb = diag(al) H_{t-1}, the
 * token's adjoint step is that of gdr_oracle_bwd with alpha replaced row by row:
 *     dk_i += sum_j al_i H_{t-1}[i][j] dp_j       (from p = Hb^T k)
 *     dal_i = sum_j H_{t-1}[i][j] dHb[i][j]       dH[i][j] <- al_i dHb[i][j]
 *     da_{t,i} = dal_i al_i g'(a_{t,i})           (da is [rows, dk])
 */
int gdr_oracle_bwd_vec(const void *q, const void *k, const void *v, const void *a,
                       const void *beta, int in_dtype, const double *h0, const double *dout,
                       const double *dhT, double *dq, double *dk_out, double *dv_out, double *da,
                       double *dbeta, double *dh0, const int64_t *cu_seqlens, int B, int64_t T,
                       int H, int dk, int dv, double b, int gate, int nthreads)
{
    if (B < 1 || T < 0 || H < 1 || dk < 1 || dv < 1) return 1;
    if (in_dtype < OR_BF16 || in_dtype > OR_F64) return 1;
    const int N = B;
    if (cu_seqlens) {
        if (cu_seqlens[0] != 0) return 2;
        for (int n = 0; n < N; n++)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return 2;
        if (cu_seqlens[N] != T) return 2;
    }
    const int64_t S = (int64_t)dk * dv;
    const int64_t nunit = (int64_t)N * H;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int rc = 0;
#pragma omp parallel
    {
        double *dH = (double *)malloc(sizeof(double) * (size_t)S);
        double *al = (double *)malloc(sizeof(double) * (size_t)dk);
        double *kt = (double *)malloc(sizeof(double) * (size_t)dk);
        double *qt = (double *)malloc(sizeof(double) * (size_t)dk);
        double *pr = (double *)malloc(sizeof(double) * (size_t)dv);
        double *de = (double *)malloc(sizeof(double) * (size_t)dv);
        double *gp = (double *)malloc(sizeof(double) * (size_t)dv);
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < nunit; u++) {
            const int h = (int)(u % H);
            const int n = (int)(u / H);
            const int64_t t_begin = cu_seqlens ? cu_seqlens[n] : (int64_t)n * T;
            const int64_t len = (cu_seqlens ? cu_seqlens[n + 1] : t_begin + T) - t_begin;
            /* every state H_0 .. H_len of this (sequence, head): small cases only */
            double *Hs = (double *)malloc(sizeof(double) * (size_t)(len + 1) * S);
            if (!Hs) {
                rc = 3;
                continue;
            }
            for (int64_t e = 0; e < S; e++) Hs[e] = h0 ? h0[u * S + e] : 0.0;
            for (int64_t t = 0; t < len; t++) {
                const int64_t row = (t_begin + t) * H + h;
                const double bt = widen(beta, in_dtype, row);
                const double *Hp = Hs + t * S;
                double *Hn = Hs + (t + 1) * S;
                for (int i = 0; i < dk; i++) {
                    al[i] = exp(gdr_oracle_gate(widen(a, in_dtype, (row * dk) + i), b, gate));
                    kt[i] = widen(k, in_dtype, row * dk + i);
                }
                for (int j = 0; j < dv; j++) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; i++) acc += al[i] * Hp[i * dv + j] * kt[i];
                    de[j] = bt * (widen(v, in_dtype, row * dv + j) - acc);
                }
                for (int i = 0; i < dk; i++)
                    for (int j = 0; j < dv; j++) Hn[i * dv + j] = al[i] * Hp[i * dv + j] + kt[i] * de[j];
            }
            for (int64_t e = 0; e < S; e++) dH[e] = dhT ? dhT[u * S + e] : 0.0;
            for (int64_t t = len - 1; t >= 0; t--) {
                const int64_t row = (t_begin + t) * H + h;
                const double bt = widen(beta, in_dtype, row);
                const double *Hp = Hs + t * S, *Ht = Hs + (t + 1) * S;
                for (int i = 0; i < dk; i++) {
                    al[i] = exp(gdr_oracle_gate(widen(a, in_dtype, (row * dk) + i), b, gate));
                    kt[i] = widen(k, in_dtype, row * dk + i);
                    qt[i] = widen(q, in_dtype, row * dk + i);
                }
                for (int j = 0; j < dv; j++) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; i++) acc += al[i] * Hp[i * dv + j] * kt[i];
                    pr[j] = acc;
                    de[j] = bt * (widen(v, in_dtype, row * dv + j) - acc);
                }
                /* o = H_t^T q: dq, and dH gains q do^T */
                for (int i = 0; i < dk; i++) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; j++) {
                        const double go = dout ? dout[row * dv + j] : 0.0;
                        acc += Ht[i * dv + j] * go;
                        dH[i * dv + j] += go * qt[i];
                    }
                    dq[row * dk + i] = acc;
                }
                /* H_t = Hb + k delta^T, delta = beta (v - Hb^T k) */
                double db = 0.0;
                for (int j = 0; j < dv; j++) {
                    double gd = 0.0;
                    for (int i = 0; i < dk; i++) gd += kt[i] * dH[i * dv + j];
                    dv_out[row * dv + j] = bt * gd;
                    db += gd * (widen(v, in_dtype, row * dv + j) - pr[j]);
                    gp[j] = -bt * gd;
                }
                dbeta[row] = db;
                for (int i = 0; i < dk; i++) {
                    double gk = 0.0, dal = 0.0;
                    for (int j = 0; j < dv; j++) {
                        const double hb_bar = dH[i * dv + j] + kt[i] * gp[j];
                        gk += dH[i * dv + j] * de[j] + al[i] * Hp[i * dv + j] * gp[j];
                        dal += Hp[i * dv + j] * hb_bar;
                        dH[i * dv + j] = al[i] * hb_bar;
                    }
                    dk_out[row * dk + i] = gk;
                    da[row * dk + i] = dal * al[i] * gate_grad(widen(a, in_dtype, (row * dk) + i), b, gate);
                }
            }
            if (dh0)
                for (int64_t e = 0; e < S; e++) dh0[u * S + e] = dH[e];
            free(Hs);
        }
        free(dH);
        free(al);
        free(kt);
        free(qt);
        free(pr);
        free(de);
        free(gp);
    }
    return rc;
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
