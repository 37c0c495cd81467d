// gdr_vec.cu -- the chunked forward pass with one decay factor per key
// channel (per-channel or "vector" decay), in the factored exp(+-G) form.
//
// Per token the state's row i decays by alpha_{t,i} = exp(g(a_{t,i})) before
// the delta-rule write [P1 §2.1-2.2, P4 §3]:
//     H_t = (I - beta k k^T) diag(alpha_t) H_{t-1} + beta k v^T,   o_t = H_t^T q_t.
// Inside a tile of C tokens with per-channel cumulative log-decay G_{i,d}
// (G_i = sum_{r<=i} g_r, resetting at every tile) and entering state H:
//     Kt = K (.) exp(G),  Kh = K (.) exp(-G),  Qt = Q (.) exp(G)
//     A_ij = beta_i Kt_i . Kh_j  (j < i),  T = (I + A)^{-1}
//     W = T diag(beta) Kt,  U = T diag(beta) V,  D = U - W H
//     O = Qt H + (Qt Kh^T (.) [j <= i]) D
//     H <- diag(exp(G_C)) H + (Kh (.) exp(G_C))^T D
// Every pairwise decay exp(G_i - G_j) is the product of two factors taken
// separately, so the in-tile products are plain matrix products of Kt, Kh and
// Qt.  That is what the bounded gate buys [P1 §2.2, P3 §3.2]: with
// g in (-b, 0) the factor exp(-G) stays below exp(C b), finite in fp32 for
// C b < 88; an unbounded gate can overflow it, so this path takes the bounded
// gate only.
//
// Two kernels: wy_vec_kernel (one block per (tile, head), all tiles at once)
// builds W, U, Qt, Kh exp(G_C), the masked Qt Kh^T and exp(G_C); then
// state_vec_kernel (one block per (sequence, head, 32 state columns)) runs the
// state pass over the tiles of its sequence and writes the outputs.
#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr int kVC = 16;      // tile length of this path
constexpr int kVCols = 32;   // state columns per state-pass block

struct VecScratch {
    float *W, *U, *Qt, *Ke;  // [tokens][H][dk] (U: [tokens][H][dv])
    float *P;                // [tiles][H][C][C]
    float *eGC;              // [tiles][H][dk]
};

template <typename T, int DK>
__global__ void __launch_bounds__(128)
wy_vec_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
              const T *__restrict__ a, const T *__restrict__ beta, VecScratch S, Plan p, int H,
              int dv, float b) {
    __shared__ float Kt[kVC][DK + 1], Kh[kVC][DK + 1], Qt[kVC][DK + 1];
    __shared__ float Am[kVC][kVC + 1], Tm[kVC][kVC + 1];
    __shared__ float bs[kVC];
    const int64_t c = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int n = find_owner(p.chunk_base, p.N, c);
    if (n < 0) return;
    const int64_t t0 = p.seq_start[n] + (c - p.chunk_base[n]) * kVC;
    const int len = (int)min((int64_t)kVC, p.seq_start[n + 1] - t0);
    // per-channel cumulative log-decay: thread d owns key channel d
    float eGC = 1.f;
    if (tid < DK) {
        float G = 0.f;
#pragma unroll
        for (int i = 0; i < kVC; ++i) {
            float kt = 0.f, kh = 0.f, qt = 0.f;
            if (i < len) {
                const int64_t r = (t0 + i) * H + h;
                G += gate_logdecay(to_f32(a[r * DK + tid]), b, GDR_GATE_BOUNDED);
                const float e = expf(G), en = expf(-G);
                const float kd = to_f32(k[r * DK + tid]);
                kt = kd * e;
                kh = kd * en;
                qt = to_f32(q[r * DK + tid]) * e;
                eGC = e;
            }
            Kt[i][tid] = kt;
            Kh[i][tid] = kh;
            Qt[i][tid] = qt;
        }
    }
    if (tid < kVC) bs[tid] = tid < len ? to_f32(beta[(t0 + tid) * H + h]) : 0.f;
    __syncthreads();
    // A_ij = beta_i Kt_i . Kh_j (j < i) and P_ij = Qt_i . Kh_j (j <= i)
    float *P = S.P + (c * H + h) * (int64_t)(kVC * kVC);
    for (int e = tid; e < kVC * kVC; e += 128) {
        const int i = e / kVC, j = e % kVC;
        float da = 0.f, dp = 0.f;
        if (j <= i) {
#pragma unroll 8
            for (int d = 0; d < DK; ++d) {
                da = fmaf(Kt[i][d], Kh[j][d], da);
                dp = fmaf(Qt[i][d], Kh[j][d], dp);
            }
        }
        Am[i][j] = j < i ? bs[i] * da : 0.f;
        P[e] = dp;
    }
    __syncthreads();
    // T = (I + A)^{-1}: forward substitution, one column per thread
    if (tid < kVC) {
        const int col = tid;
        for (int i = 0; i < kVC; ++i) {
            float acc = (i == col) ? 1.f : 0.f;
            for (int j = col; j < i; ++j) acc = fmaf(-Am[i][j], Tm[j][col], acc);
            Tm[i][col] = (i < col) ? 0.f : acc;
        }
    }
    __syncthreads();
    // W = T diag(beta) Kt, and the per-token factors the state pass reads
    if (tid < DK) {
        for (int i = 0; i < len; ++i) {
            float acc = 0.f;
            for (int j = 0; j <= i; ++j) acc = fmaf(Tm[i][j] * bs[j], Kt[j][tid], acc);
            const int64_t r = ((t0 + i) * H + h) * DK + tid;
            S.W[r] = acc;
            S.Qt[r] = Qt[i][tid];
            S.Ke[r] = Kh[i][tid] * eGC;
        }
        S.eGC[(c * H + h) * DK + tid] = eGC;
    }
    // U = T diag(beta) V
    for (int d = tid; d < dv; d += 128) {
        float vc[kVC];
#pragma unroll
        for (int j = 0; j < kVC; ++j) vc[j] = j < len ? to_f32(v[((t0 + j) * H + h) * dv + d]) : 0.f;
#pragma unroll
        for (int i = 0; i < kVC; ++i) {
            if (i >= len) break;
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j <= i; ++j) acc = fmaf(Tm[i][j] * bs[j], vc[j], acc);
            S.U[((t0 + i) * H + h) * dv + d] = acc;
        }
    }
}

// State pass over the tiles of one sequence; 256 threads: tx = column of the
// 32-column slice, ty = row group.
template <typename T>
__global__ void __launch_bounds__(256)
state_vec_kernel(VecScratch S, const float *__restrict__ h0, T *__restrict__ out,
                 float *__restrict__ hT, Plan p, int H, int dk, int dv) {
    extern __shared__ float sm[];
    const int nslices = dv / kVCols;
    const int slice = blockIdx.x % nslices;
    const int h = (blockIdx.x / nslices) % H;
    const int n = blockIdx.x / (nslices * H);
    const int j0 = slice * kVCols;
    const int tid = threadIdx.x, tx = tid % 32, ty = tid / 32;
    float *Hs = sm;                     // [dk][32]
    float *Ws = Hs + dk * kVCols;       // [C][dk]
    float *Ks = Ws + kVC * dk;          // [C][dk]  Kh exp(G_C)
    float *Qs = Ks + kVC * dk;          // [C][dk]  Qt
    float *Ds = Qs + kVC * dk;          // [C][32]  U, then D
    float *Ps = Ds + kVC * kVCols;      // [C][C]
    float *eg = Ps + kVC * kVC;         // [dk]
    const size_t hbase = ((size_t)n * H + h) * dk * dv;
    for (int e = tid; e < dk * kVCols; e += 256) {
        const int d = e / kVCols, j = e % kVCols;
        Hs[e] = h0 ? h0[hbase + (size_t)d * dv + j0 + j] : 0.f;
    }
    const int64_t s = p.seq_start[n], e_end = p.seq_start[n + 1];
    int64_t c = p.chunk_base[n];
    for (int64_t t0 = s; t0 < e_end; t0 += kVC, ++c) {
        const int len = (int)min((int64_t)kVC, e_end - t0);
        __syncthreads();   // the previous tile is done with the staging arrays
        for (int e = tid; e < len * dk; e += 256) {
            const int i = e / dk, d = e % dk;
            const int64_t r = ((t0 + i) * H + h) * dk + d;
            Ws[e] = S.W[r];
            Ks[e] = S.Ke[r];
            Qs[e] = S.Qt[r];
        }
        for (int e = tid; e < len * kVCols; e += 256) {
            const int i = e / kVCols, j = e % kVCols;
            Ds[e] = S.U[((t0 + i) * H + h) * dv + j0 + j];
        }
        const float *P = S.P + (c * H + h) * (int64_t)(kVC * kVC);
        for (int e = tid; e < kVC * kVC; e += 256) Ps[e] = P[e];
        for (int d = tid; d < dk; d += 256) eg[d] = S.eGC[(c * H + h) * dk + d];
        __syncthreads();
        // D = U - W H
        float dreg[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = ty + 8 * r;
            float acc = 0.f;
            if (i < len) {
                acc = Ds[i * kVCols + tx];
                for (int d = 0; d < dk; ++d) acc = fmaf(-Ws[i * dk + d], Hs[d * kVCols + tx], acc);
            }
            dreg[r] = acc;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = ty + 8 * r;
            if (i < len) Ds[i * kVCols + tx] = dreg[r];
        }
        __syncthreads();
        // O = Qt H + P D
        for (int i = ty; i < len; i += 8) {
            float acc = 0.f;
            for (int d = 0; d < dk; ++d) acc = fmaf(Qs[i * dk + d], Hs[d * kVCols + tx], acc);
            for (int j = 0; j <= i; ++j) acc = fmaf(Ps[i * kVC + j], Ds[j * kVCols + tx], acc);
            out[((t0 + i) * H + h) * dv + j0 + tx] = from_f32<T>(acc);
        }
        __syncthreads();
        // H <- diag(exp(G_C)) H + (Kh exp(G_C))^T D
        for (int d = ty; d < dk; d += 8) {
            float acc = eg[d] * Hs[d * kVCols + tx];
            for (int i = 0; i < len; ++i) acc = fmaf(Ks[i * dk + d], Ds[i * kVCols + tx], acc);
            Hs[d * kVCols + tx] = acc;
        }
    }
    __syncthreads();
    if (hT)
        for (int e = tid; e < dk * kVCols; e += 256) {
            const int d = e / kVCols, j = e % kVCols;
            hT[hbase + (size_t)d * dv + j0 + j] = Hs[e];
        }
}

template <typename T>
cudaError_t launch_vec_t(const void *q, const void *k, const void *v, const void *a,
                         const void *beta, const float *h0, void *out, float *hT,
                         const VecScratch &S, Plan plan, int H, int dk, int dv, int64_t max_tiles,
                         float b, cudaStream_t stream) {
    if (max_tiles > 0) {
        ProfScope prof(stream, "wy_vec_kernel");
        const dim3 grid((unsigned)max_tiles, (unsigned)H);
        if (dk == 128)
            wy_vec_kernel<T, 128><<<grid, 128, 0, stream>>>((const T *)q, (const T *)k, (const T *)v,
                                                            (const T *)a, (const T *)beta, S, plan,
                                                            H, dv, b);
        else
            wy_vec_kernel<T, 64><<<grid, 128, 0, stream>>>((const T *)q, (const T *)k, (const T *)v,
                                                           (const T *)a, (const T *)beta, S, plan, H,
                                                           dv, b);
        count_launch();
        const cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    const size_t smem = sizeof(float) * ((size_t)dk * kVCols + 3 * (size_t)kVC * dk +
                                         (size_t)kVC * kVCols + kVC * kVC + dk);
    auto kern = state_vec_kernel<T>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    ProfScope prof(stream, "state_vec_kernel");
    kern<<<(unsigned)((size_t)plan.N * H * (dv / kVCols)), 256, smem, stream>>>(S, h0, (T *)out, hT,
                                                                              plan, H, dk, dv);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

size_t vec_scratch_bytes(int64_t tiles, int64_t T_total, int H, int dk, int dv) {
    return sizeof(float) * ((size_t)T_total * H * (3 * (size_t)dk + dv) +
                            (size_t)tiles * H * (kVC * kVC + dk)) + 6 * 256;
}

cudaError_t launch_vec_forward(const void *q, const void *k, const void *v, const void *a,
                               const void *beta, const float *h0, void *out, float *hT,
                               gdr_dtype_t dtype, Plan plan, int H, int dk, int dv,
                               int64_t T_total, int64_t max_tiles, float b, void *scratch,
                               cudaStream_t stream) {
    if (plan.C != kVC) return cudaErrorInvalidValue;
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    char *p = (char *)scratch;
    VecScratch S;
    const size_t tok_k = sizeof(float) * (size_t)T_total * H * dk;
    S.W = (float *)p;
    p += al(tok_k);
    S.Qt = (float *)p;
    p += al(tok_k);
    S.Ke = (float *)p;
    p += al(tok_k);
    S.U = (float *)p;
    p += al(sizeof(float) * (size_t)T_total * H * dv);
    S.P = (float *)p;
    p += al(sizeof(float) * (size_t)max_tiles * H * kVC * kVC);
    S.eGC = (float *)p;
    if (dtype == GDR_BF16)
        return launch_vec_t<__nv_bfloat16>(q, k, v, a, beta, h0, out, hT, S, plan, H, dk, dv,
                                           max_tiles, b, stream);
    return launch_vec_t<float>(q, k, v, a, beta, h0, out, hT, S, plan, H, dk, dv, max_tiles, b,
                               stream);
}

}  // namespace gdr
