// gdr_simt.cu -- planning, the gate stage and the fp32 CUDA-core path.
//
// This path computes every stage of the chunked forward pass in fp32 on the
// CUDA cores.  It serves the fp32 dtype, dk/dv = 64, any tile length, and is
// the reference GPU path the tensor-core path is checked against.
//
// Per tile of C tokens with in-tile cumulative log-decay G (G_i = sum_{r<=i} g_r)
// and entering state H (dk x dv) [P1 §3.2, P2 §2.1, P3 §3.1]:
//   A_ij = beta_i exp(G_i - G_j) k_i.k_j (j < i),   T = (I + A)^{-1}
//   W = T diag(beta exp(G)) K,   U = T diag(beta) V,   D = U - W H
//   O = diag(exp(G)) Q H + (Q K^T (.) [j <= i] (.) exp(G_i - G_j)) D
//   H <- exp(G_C) H + (K (.) exp(G_C - G))^T D
// Every decay factor is exp of a non-positive number (G is non-increasing
// inside a tile), so nothing overflows for any gate, bounded or not.
#include <algorithm>

#include "gdr_internal.cuh"

namespace gdr {

GDR_DEBUG_TU()

// ---------------------------------------------------------------------------
// plan: sequence starts, tile bases and segment bases (exclusive prefix sums)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
plan_kernel(const int32_t *__restrict__ cu, int N, int64_t T_per, int64_t T_total, int C,
            int seg_chunks, int64_t *__restrict__ seq_start, int64_t *__restrict__ chunk_base,
            int64_t *__restrict__ seg_base, int *__restrict__ status) {
    __shared__ int64_t s_ch[1024];
    __shared__ int64_t s_sg[1024];
    __shared__ int bad;
    const int tid = threadIdx.x;
    if (tid == 0) bad = 0;
    __syncthreads();
    const int per = (N + 1023) / 1024;
    const int n0 = min(N, tid * per), n1 = min(N, n0 + per);
    int64_t lc = 0, ls = 0;
    for (int n = n0; n < n1; ++n) {
        int64_t s, e;
        if (cu) {
            s = cu[n];
            e = cu[n + 1];
            if (e < s) bad = 1;
        } else {
            s = (int64_t)n * T_per;
            e = s + T_per;
        }
        const int64_t len = e > s ? e - s : 0;
        const int64_t nc = (len + C - 1) / C;
        lc += nc;
        ls += nc > seg_chunks ? (nc + seg_chunks - 1) / seg_chunks : 1;  // >= 1 segment per sequence
    }
    if (cu && tid == 0 && (cu[0] != 0 || (int64_t)cu[N] != T_total)) bad = 1;
    s_ch[tid] = lc;
    s_sg[tid] = ls;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        const int64_t x = tid >= off ? s_ch[tid - off] : 0;
        const int64_t y = tid >= off ? s_sg[tid - off] : 0;
        __syncthreads();
        s_ch[tid] += x;
        s_sg[tid] += y;
        __syncthreads();
    }
    if (bad) {  // an empty plan: every sequence has zero tokens
        for (int n = n0; n < n1; ++n) seq_start[n] = chunk_base[n] = seg_base[n] = 0;
        if (tid == 0) {
            seq_start[N] = chunk_base[N] = seg_base[N] = 0;
            set_status(status, GDR_ERR_BAD_SEQLENS);
        }
        return;
    }
    int64_t cb = s_ch[tid] - lc, sb = s_sg[tid] - ls;
    for (int n = n0; n < n1; ++n) {
        const int64_t s = cu ? (int64_t)cu[n] : (int64_t)n * T_per;
        const int64_t e = cu ? (int64_t)cu[n + 1] : s + T_per;
        const int64_t nc = (e - s + C - 1) / C;
        seq_start[n] = s;
        chunk_base[n] = cb;
        seg_base[n] = sb;
        cb += nc;
        sb += nc > seg_chunks ? (nc + seg_chunks - 1) / seg_chunks : 1;
    }
    if (tid == 1023) {
        seq_start[N] = cu ? T_total : (int64_t)N * T_per;
        chunk_base[N] = s_ch[1023];
        seg_base[N] = s_sg[1023];
    }
}

cudaError_t launch_plan(const int32_t *cu_seqlens, int N, int64_t T_per, int64_t T_total, int C,
                        int seg_chunks, int64_t *seq_start, int64_t *chunk_base,
                        int64_t *seg_base, int *status, cudaStream_t stream) {
    ProfScope prof(stream, "plan_kernel");
    plan_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, N, T_per, T_total, C, seg_chunks, seq_start,
                                        chunk_base, seg_base, status);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// stage 1: gate + in-tile cumulative sum [P1 §3.3, P2 §2.2, P3 §3.2, P4 §2.3]
// G and the transposed beta are head-major so a tile's values are contiguous
// for the later stages.  One block per 128 / C consecutive tiles (at most 128
// tokens, contiguous along the token axis) and 32 heads: a and beta are read
// row by row (coalesced), transposed through shared memory, summed per
// (tile, head), and written head row by head row (coalesced).
// ---------------------------------------------------------------------------
constexpr int kGateTok = 128, kGateMaxTiles = kGateTok / 16, kGateHeads = 32;

template <typename T>
__global__ void __launch_bounds__(256)
gate_cumsum_kernel(const T *__restrict__ a, const T *__restrict__ beta, float *__restrict__ G,
                   float *__restrict__ Bt, Plan p, int H, int64_t T_total, int64_t max_chunks,
                   float b, int gate) {
    __shared__ float gsm[2 * kGateHeads * (kGateTok + 1)];   // [head][token] gates, then beta
    __shared__ int64_t tstart[kGateMaxTiles];
    __shared__ int tlen[kGateMaxTiles];
    const int tid = threadIdx.x;
    const int nt = kGateTok / p.C;                           // tiles per block
    const int64_t c0 = (int64_t)blockIdx.x * nt;
    const int h0 = blockIdx.y * kGateHeads;
    const int nh = min(kGateHeads, H - h0);
    if (tid < kGateMaxTiles) {
        const int64_t c = c0 + tid;
        const int n = (tid < nt && c < max_chunks) ? find_owner(p.chunk_base, p.N, c) : -1;
        int64_t t0 = 0;
        int len = 0;
        if (n >= 0) {
            t0 = p.seq_start[n] + (c - p.chunk_base[n]) * p.C;
            len = (int)min((int64_t)p.C, p.seq_start[n + 1] - t0);
        }
        tstart[tid] = t0;
        tlen[tid] = len;
    }
    __syncthreads();
    if (tlen[0] == 0) return;   // tiles are enumerated densely: nothing from here on
    // the tiles present are consecutive and cover [Tb, Te) without gaps
    const int64_t Tb = tstart[0];
    int64_t Te = Tb;
    for (int j = 0; j < nt; ++j)
        if (tlen[j] > 0) Te = tstart[j] + tlen[j];
    const int ntok = (int)(Te - Tb);
    const int ld = ntok + 1;
    float *sg = gsm;
    float *sb = gsm + kGateHeads * ld;
    const int warp = tid >> 5, lane = tid & 31;
    constexpr int kRows = kGateTok / 8;   // token rows per warp (8 warps)
    const int64_t base = Tb * H + h0;
    if (nh == H && ntok * H % 8 == 0 && ((uintptr_t)(a + base) | (uintptr_t)(beta + base)) % (8 * sizeof(T)) == 0 &&
        GDR_INBOUNDS(Te <= T_total)) {
        // every head of the block's tokens: one contiguous [ntok][H] region, read 8
        // elements (16 or 32 bytes) per thread and load
        for (int e0 = 8 * tid; e0 < ntok * H; e0 += 8 * 256) {
            T av[8], bv[8];
            *(uint4 *)av = *(const uint4 *)(a + base + e0);
            if (sizeof(T) == 4) *((uint4 *)av + 1) = *((const uint4 *)(a + base + e0) + 1);
            if (Bt) {
                *(uint4 *)bv = *(const uint4 *)(beta + base + e0);
                if (sizeof(T) == 4) *((uint4 *)bv + 1) = *((const uint4 *)(beta + base + e0) + 1);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = (e0 + u) / H, hh = (e0 + u) - t * H;
                sg[hh * ld + t] = gate_logdecay(to_f32(av[u]), b, gate);
                sb[hh * ld + t] = Bt ? to_f32(bv[u]) : 0.f;
            }
        }
    } else if (lane < nh) {   // warp per token row, lane per head; all loads in flight at once
        float av[kRows], bv[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int t = warp + 8 * r;
            const int64_t src = (Tb + min(t, ntok - 1)) * H + h0 + lane;
            av[r] = bv[r] = 0.f;
            if (GDR_INBOUNDS(Tb + min(t, ntok - 1) < T_total && h0 + lane < H)) {
                av[r] = to_f32(a[src]);
                bv[r] = Bt ? to_f32(beta[src]) : 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int t = warp + 8 * r;
            if (t < ntok) {
                sg[lane * ld + t] = gate_logdecay(av[r], b, gate);
                sb[lane * ld + t] = bv[r];
            }
        }
    }
    __syncthreads();
    {
        const int j = tid / kGateHeads, hh = tid % kGateHeads;
        if (j < nt && hh < nh && tlen[j] > 0) {
            float *row = sg + hh * ld + (int)(tstart[j] - Tb);
            float acc = 0.f;
            for (int i = 0; i < tlen[j]; ++i) {
                acc += row[i];
                row[i] = acc;
            }
        }
    }
    __syncthreads();
    for (int hh = warp; hh < nh; hh += 8) {   // warp per head row, lane per token
        const int64_t dst = (int64_t)(h0 + hh) * T_total + Tb;
        for (int t = lane; t < ntok; t += 32) {
            if (!GDR_INBOUNDS(Tb + t < T_total)) continue;
            G[dst + t] = sg[hh * ld + t];
            if (Bt) Bt[dst + t] = sb[hh * ld + t];
        }
    }
}

cudaError_t launch_gate_cumsum(const void *a, const void *beta, gdr_dtype_t dtype, float *G,
                               float *Bt, Plan plan, int H, int64_t T_total,
                               int64_t max_chunks, float b, gdr_gate_t gate,
                               cudaStream_t stream) {
    if (max_chunks == 0 || H == 0) return cudaSuccess;
    if (plan.C < 16 || plan.C > kGateTok || kGateTok % plan.C != 0) return cudaErrorInvalidValue;
    const int nt = kGateTok / plan.C;
    const dim3 grid((unsigned)((max_chunks + nt - 1) / nt), (unsigned)((H + kGateHeads - 1) / kGateHeads));
    const size_t smem = 0;
    ProfScope prof(stream, "gate_cumsum_kernel");
    if (dtype == GDR_BF16)
        gate_cumsum_kernel<__nv_bfloat16><<<grid, 256, smem, stream>>>(
            (const __nv_bfloat16 *)a, (const __nv_bfloat16 *)beta, G, Bt, plan, H, T_total,
            max_chunks, b, (int)gate);
    else
        gate_cumsum_kernel<float><<<grid, 256, smem, stream>>>(
            (const float *)a, (const float *)beta, G, Bt, plan, H, T_total, max_chunks, b,
            (int)gate);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// stage 2 (CUDA cores): the WY / UT representation of every tile
// one block of 128 threads per (tile, head)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(128)
wy_simt_kernel(const T *__restrict__ k, const T *__restrict__ v, const T *__restrict__ beta,
               const float *__restrict__ G, float *__restrict__ W, float *__restrict__ U, Plan p,
               int H, int dk, int dv, int64_t T_total, int64_t max_chunks) {
    extern __shared__ float sm[];
    const int64_t c = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int C = p.C;
    const int n = find_owner(p.chunk_base, p.N, c);
    if (n < 0) return;
    const int64_t t0 = p.seq_start[n] + (c - p.chunk_base[n]) * C;
    const int len = (int)min((int64_t)C, p.seq_start[n + 1] - t0);
    if (!GDR_INBOUNDS(h < H && t0 >= 0 && t0 + len <= T_total)) return;
    float *Ks = sm;                  // [C][dk]
    float *Vs = Ks + C * dk;         // [C][dv]
    float *A = Vs + C * dv;          // [C][C+1]
    float *Tm = A + C * (C + 1);     // [C][C+1]
    float *bs = Tm + C * (C + 1);    // beta           [C]
    float *be = bs + C;              // beta * exp(G)  [C]
    float *Gs = be + C;              // G              [C]
    for (int e = tid; e < len * dk; e += blockDim.x) {
        const int i = e / dk, d = e % dk;
        Ks[e] = to_f32(k[((t0 + i) * H + h) * dk + d]);
    }
    for (int e = tid; e < len * dv; e += blockDim.x) {
        const int i = e / dv, d = e % dv;
        Vs[e] = to_f32(v[((t0 + i) * H + h) * dv + d]);
    }
    if (tid < len) {
        const float gi = G[(int64_t)h * T_total + t0 + tid];
        const float bi = to_f32(beta[(t0 + tid) * H + h]);
        Gs[tid] = gi;
        bs[tid] = bi;
        be[tid] = bi * expf(gi);
    }
    __syncthreads();
    // A (strictly lower): decay-scaled Gram matrix of the keys
    for (int e = tid; e < len * len; e += blockDim.x) {
        const int i = e / len, j = e % len;
        float val = 0.f;
        if (j < i) {
            float dot = 0.f;
            for (int d = 0; d < dk; ++d) dot = fmaf(Ks[i * dk + d], Ks[j * dk + d], dot);
            val = bs[i] * expf(Gs[i] - Gs[j]) * dot;
        }
        A[i * (C + 1) + j] = val;
    }
    __syncthreads();
    // T = (I + A)^{-1}: forward substitution, one column per thread
    if (tid < len) {
        const int col = tid;
        for (int i = 0; i < len; ++i) {
            float acc = (i == col) ? 1.f : 0.f;
            for (int j = col; j < i; ++j) acc = fmaf(-A[i * (C + 1) + j], Tm[j * (C + 1) + col], acc);
            Tm[i * (C + 1) + col] = (i < col) ? 0.f : acc;
        }
    }
    __syncthreads();
    // W = T diag(beta exp(G)) K,  U = T diag(beta) V
    for (int e = tid; e < len * dk; e += blockDim.x) {
        const int i = e / dk, d = e % dk;
        float acc = 0.f;
        for (int j = 0; j <= i; ++j) acc = fmaf(Tm[i * (C + 1) + j] * be[j], Ks[j * dk + d], acc);
        W[((t0 + i) * H + h) * dk + d] = acc;
    }
    for (int e = tid; e < len * dv; e += blockDim.x) {
        const int i = e / dv, d = e % dv;
        float acc = 0.f;
        for (int j = 0; j <= i; ++j) acc = fmaf(Tm[i * (C + 1) + j] * bs[j], Vs[j * dv + d], acc);
        U[((t0 + i) * H + h) * dv + d] = acc;
    }
}

cudaError_t launch_wy_simt(const void *k, const void *v, const void *beta, const float *G,
                           float *W, float *U, gdr_dtype_t dtype, Plan plan, int H, int dk,
                           int dv, int64_t T_total, int64_t max_chunks, cudaStream_t stream) {
    if (max_chunks == 0) return cudaSuccess;
    const int C = plan.C;
    const size_t smem = sizeof(float) * ((size_t)C * dk + (size_t)C * dv + 2 * (size_t)C * (C + 1) + 3 * C);
    const dim3 grid((unsigned)max_chunks, (unsigned)H);
    cudaError_t err;
    ProfScope prof(stream, "wy_simt_kernel");
    if (dtype == GDR_BF16) {
        auto kern = wy_simt_kernel<__nv_bfloat16>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        kern<<<grid, 128, smem, stream>>>((const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v,
                                          (const __nv_bfloat16 *)beta, G, W, U, plan, H, dk, dv,
                                          T_total, max_chunks);
    } else {
        auto kern = wy_simt_kernel<float>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        kern<<<grid, 128, smem, stream>>>((const float *)k, (const float *)v,
                                          (const float *)beta, G, W, U, plan, H, dk, dv, T_total,
                                          max_chunks);
    }
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// stages 3+4 (CUDA cores): state pass over the tiles of one sequence and the
// outputs; one block of 256 threads per (sequence, head, 32 state columns).
// The columns of H evolve independently given (k, beta, g), so the column
// split needs no exchange.
// ---------------------------------------------------------------------------
constexpr int kSimtCols = 32;

template <typename T>
__global__ void __launch_bounds__(256)
state_out_simt_kernel(const T *__restrict__ q, const T *__restrict__ k,
                      const float *__restrict__ W, const float *__restrict__ U,
                      const float *__restrict__ G, const float *__restrict__ h0,
                      T *__restrict__ out, float *__restrict__ hT, Plan p, int H, int dk, int dv,
                      int64_t T_total) {
    extern __shared__ float sm[];
    const int nslices = dv / kSimtCols;
    const int slice = blockIdx.x % nslices;
    const int h = (blockIdx.x / nslices) % H;
    const int n = blockIdx.x / (nslices * H);
    const int j0 = slice * kSimtCols;
    const int C = p.C;
    const int tid = threadIdx.x, tx = tid % 32, ty = tid / 32;
    float *Hs = sm;                      // [dk][32]
    float *Ws = Hs + dk * kSimtCols;     // [C][dk]
    float *Ks = Ws + C * dk;             // [C][dk]
    float *Qs = Ks + C * dk;             // [C][dk]
    float *Ds = Qs + C * dk;             // [C][32]   U, then D
    float *P = Ds + C * kSimtCols;       // [C][C+1]
    float *Gs = P + C * (C + 1);         // [C]
    float *eG = Gs + C;                  // exp(G_i)
    float *eR = eG + C;                  // exp(G_C - G_i)

    if (!GDR_INBOUNDS(n < p.N)) return;
    const size_t hbase = ((size_t)n * H + h) * dk * dv;
    for (int e = tid; e < dk * kSimtCols; e += 256) {
        const int d = e / kSimtCols, j = e % kSimtCols;
        Hs[e] = h0 ? h0[hbase + (size_t)d * dv + j0 + j] : 0.f;
    }
    const int64_t s = p.seq_start[n], e_end = p.seq_start[n + 1];
    if (!GDR_INBOUNDS(s >= 0 && e_end <= T_total)) return;
    for (int64_t t0 = s; t0 < e_end; t0 += C) {
        const int len = (int)min((int64_t)C, e_end - t0);
        __syncthreads();  // previous tile done with Ws/Ks/Qs/Ds/P
        for (int e = tid; e < len * dk; e += 256) {
            const int i = e / dk, d = e % dk;
            const int64_t r = ((t0 + i) * H + h) * dk + d;
            Ws[e] = W[r];
            Ks[e] = to_f32(k[r]);
            Qs[e] = to_f32(q[r]);
        }
        for (int e = tid; e < len * kSimtCols; e += 256) {
            const int i = e / kSimtCols, j = e % kSimtCols;
            Ds[e] = U[((t0 + i) * H + h) * dv + j0 + j];
        }
        if (tid < len) Gs[tid] = G[(int64_t)h * T_total + t0 + tid];
        __syncthreads();
        const float GC = Gs[len - 1];
        if (tid < len) {
            eG[tid] = expf(Gs[tid]);
            eR[tid] = expf(GC - Gs[tid]);
        }
        // D = U - W H  (rows ty, ty+8, ...; column tx)
        float dreg[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int i = ty + 8 * r;
            float acc = 0.f;
            if (i < len) {
                acc = Ds[i * kSimtCols + tx];
                for (int d = 0; d < dk; ++d) acc = fmaf(-Ws[i * dk + d], Hs[d * kSimtCols + tx], acc);
            }
            dreg[r] = acc;
        }
        // P = (Q K^T) (.) [j <= i] (.) exp(G_i - G_j)
        for (int e = tid; e < len * len; e += 256) {
            const int i = e / len, j = e % len;
            float val = 0.f;
            if (j <= i) {
                float dot = 0.f;
                for (int d = 0; d < dk; ++d) dot = fmaf(Qs[i * dk + d], Ks[j * dk + d], dot);
                val = dot * expf(Gs[i] - Gs[j]);
            }
            P[i * (C + 1) + j] = val;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int i = ty + 8 * r;
            if (i < len) Ds[i * kSimtCols + tx] = dreg[r];
        }
        __syncthreads();
        // O = diag(exp(G)) Q H + P D
        for (int i = ty; i < len; i += 8) {
            float acc = 0.f;
            for (int d = 0; d < dk; ++d) acc = fmaf(Qs[i * dk + d], Hs[d * kSimtCols + tx], acc);
            acc *= eG[i];
            for (int j = 0; j <= i; ++j) acc = fmaf(P[i * (C + 1) + j], Ds[j * kSimtCols + tx], acc);
            out[((t0 + i) * H + h) * dv + j0 + tx] = from_f32<T>(acc);
        }
        __syncthreads();
        // H <- exp(G_C) H + (K (.) exp(G_C - G))^T D
        const float eGC = expf(GC);
        for (int d = ty; d < dk; d += 8) {
            float acc = eGC * Hs[d * kSimtCols + tx];
            for (int i = 0; i < len; ++i) acc = fmaf(Ks[i * dk + d] * eR[i], Ds[i * kSimtCols + tx], acc);
            Hs[d * kSimtCols + tx] = acc;
        }
    }
    __syncthreads();
    if (hT)
        for (int e = tid; e < dk * kSimtCols; e += 256) {
            const int d = e / kSimtCols, j = e % kSimtCols;
            hT[hbase + (size_t)d * dv + j0 + j] = Hs[e];
        }
}

cudaError_t launch_state_out_simt(const void *q, const void *k, const float *W, const float *U,
                                  const float *G, const float *h0, void *out, float *hT,
                                  gdr_dtype_t dtype, Plan plan, int H, int dk, int dv,
                                  int64_t T_total, cudaStream_t stream) {
    const int C = plan.C;
    const size_t smem = sizeof(float) * ((size_t)dk * kSimtCols + 3 * (size_t)C * dk +
                                         (size_t)C * kSimtCols + (size_t)C * (C + 1) + 3 * C);
    const unsigned grid = (unsigned)((size_t)plan.N * H * (dv / kSimtCols));
    cudaError_t err;
    ProfScope prof(stream, "state_out_simt_kernel");
    if (dtype == GDR_BF16) {
        auto kern = state_out_simt_kernel<__nv_bfloat16>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        kern<<<grid, 256, smem, stream>>>((const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, W, U,
                                          G, h0, (__nv_bfloat16 *)out, hT, plan, H, dk, dv,
                                          T_total);
    } else {
        auto kern = state_out_simt_kernel<float>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        kern<<<grid, 256, smem, stream>>>((const float *)q, (const float *)k, W, U, G, h0,
                                          (float *)out, hT, plan, H, dk, dv, T_total);
    }
    count_launch();
    return cudaGetLastError();
}

}  // namespace gdr
