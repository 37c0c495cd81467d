// gdr_backward.cu -- the backward pass: gradients of <dout, out> + <dhT, hT>
// with respect to q, k, v, a, beta and h0.
//
// Per token, the forward is [P4 §2.2, P1 §3.3]
//     Hb = alpha H_{t-1},  p = Hb^T k,  delta = beta (v - p),  H_t = Hb + k delta^T,
//     o = H_t^T q,         alpha = exp(g(a)),
// and the adjoints run backwards over the tokens, dH being dL/dH_t:
//     dH += q do^T,        dq = H_t do,
//     ddelta = dH^T k,     dv = beta ddelta,   dbeta = ddelta . (v - p),
//     dp = -beta ddelta,   dk = dH delta + Hb dp,
//     dHb = dH + k dp^T,   dalpha = <H_{t-1}, dHb>,  dH <- alpha dHb,
// with da = dalpha alpha g'(a) and dh0 the final dH.
//
// Columns of the state are independent in the forward, so one block owns one
// (sequence, head, 32-column slice), like the decoding kernel: it keeps its
// slice of the state in registers, runs the forward once storing the slice at
// every tile start (checkpoints), then walks the tiles backwards.  In a tile it
// first recomputes every token's delta and p (one reduction over dk each) and
// keeps them in shared memory with the tile's k, q, v and do; then for each
// token, last to first, it rebuilds H_{t-1} from the checkpoint with those
// deltas (FMAs only) and applies the adjoint step.  The sums over the value
// columns (dq, dk, dbeta, dalpha) are written per slice and added by a second
// kernel in a fixed order: the result does not depend on scheduling.
#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr int kBwCols = 32;       // state columns per block
constexpr int kBwThreads = 256;   // lane & 7 -> 4 columns; warp, lane >> 3 -> row group
constexpr int kBwMaxC = 16;       // tokens between checkpoints (the plan's tile)

struct BwArgs {
    const void *q, *k, *v, *a, *beta;
    const void *dout;  // [tokens, H, dv] (input dtype) or null
    const float *h0, *dhT;
    void *dv;         // [tokens, H, dv] (input dtype)
    float *dh0;       // [N, H, dk, dv] or null
    float *ck;        // checkpoints [tiles][H][dk][dv]
    float *pdq, *pdk; // [slices][tokens][H][dk] partial sums over this slice's columns
    float *pdb, *pda; // [slices][tokens][H]
    Plan plan;
    int H, dv_, C;
    int64_t T_total;
    float b;
    int gate;
};

__device__ __forceinline__ float gate_dgda(float a, float b, int gate) {
    const float s = 1.f / (1.f + expf(-a));
    return gate == GDR_GATE_SOFTPLUS ? -s : -b * s * (1.f - s);
}

template <typename T, int DK>
__global__ void __launch_bounds__(kBwThreads)
bwd_slice_kernel(const BwArgs A) {
    constexpr int kRows = DK / 32;
    __shared__ float red[8][kBwCols];
    __shared__ float vec[kBwCols];
    __shared__ float sc[8];
    __shared__ float ks[kBwMaxC][DK], qs[kBwMaxC][DK];
    __shared__ float dls[kBwMaxC][kBwCols], vps[kBwMaxC][kBwCols], dos[kBwMaxC][kBwCols];
    __shared__ float als[kBwMaxC], bts[kBwMaxC];
    const T *q = (const T *)A.q, *k = (const T *)A.k, *v = (const T *)A.v;
    const T *a = (const T *)A.a, *beta = (const T *)A.beta;
    const int H = A.H, dv = A.dv_, C = A.C;
    const int nslices = dv / kBwCols;
    const int slice = blockIdx.x % nslices;
    const int h = (blockIdx.x / nslices) % H;
    const int n = blockIdx.x / (nslices * H);
    if (n >= A.plan.N) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c4 = (lane & 7) * 4, rg = warp * 4 + (lane >> 3);
    const int col0 = slice * kBwCols;
    const int64_t tok0 = A.plan.seq_start[n], len = A.plan.seq_start[n + 1] - tok0;
    const int64_t tile0 = A.plan.chunk_base[n];
    const int64_t ntiles = (len + C - 1) / C;
    const int64_t S = (int64_t)DK * dv;
    auto ckp = [&](int64_t tile) { return A.ck + (tile * H + h) * S + col0 + c4; };

    // sum over the row groups of a per-thread 4-column partial -> vec[0..31]
    auto reduce_cols = [&](float (&part)[4]) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            part[u] += __shfl_xor_sync(0xffffffffu, part[u], 8);
            part[u] += __shfl_xor_sync(0xffffffffu, part[u], 16);
        }
        if (lane < 8)
#pragma unroll
            for (int u = 0; u < 4; ++u) red[warp][c4 + u] = part[u];
        __syncthreads();
        if (tid < kBwCols) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) acc += red[w][tid];
            vec[tid] = acc;
        }
        __syncthreads();
    };
    // sum of a per-thread scalar over the block -> returned to every thread
    auto reduce_scalar = [&](float x) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) sc[warp] = x;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) tot += sc[w];
        __syncthreads();
        return tot;
    };
    // per-row sum over this thread's 4 columns and the 8 lanes sharing its rows
    auto rowsum = [&](float x) {
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        return x;
    };

    // ---- forward: checkpoints at every tile start
    float s[kRows][4];
#pragma unroll
    for (int j = 0; j < kRows; ++j)
#pragma unroll
        for (int u = 0; u < 4; ++u)
            s[j][u] = A.h0 ? A.h0[((int64_t)n * H + h) * S + (int64_t)(rg + 32 * j) * dv + col0 + c4 + u] : 0.f;
    for (int64_t tt = 0; tt < len; ++tt) {
        if (tt % C == 0) {
            float *cp = ckp(tile0 + tt / C);
#pragma unroll
            for (int j = 0; j < kRows; ++j)
                *(float4 *)&cp[(int64_t)(rg + 32 * j) * dv] = make_float4(s[j][0], s[j][1], s[j][2], s[j][3]);
        }
        const int64_t row = (tok0 + tt) * H + h;
        for (int d = tid; d < DK; d += kBwThreads) ks[0][d] = to_f32(k[row * DK + d]);
        const float alpha = expf(gate_logdecay(to_f32(a[row]), A.b, A.gate));
        const float bt = to_f32(beta[row]);
        __syncthreads();
        float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            const float kd = ks[0][rg + 32 * j];
#pragma unroll
            for (int u = 0; u < 4; ++u) part[u] = fmaf(s[j][u], kd, part[u]);
        }
        reduce_cols(part);
        float dl[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            dl[u] = bt * (to_f32(v[row * dv + col0 + c4 + u]) - alpha * vec[c4 + u]);
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            const float kd = ks[0][rg + 32 * j];
#pragma unroll
            for (int u = 0; u < 4; ++u) s[j][u] = fmaf(alpha, s[j][u], kd * dl[u]);
        }
        __syncthreads();   // ks is reloaded next token
    }

    // ---- backward over the tiles
    float dh[kRows][4];
#pragma unroll
    for (int j = 0; j < kRows; ++j)
#pragma unroll
        for (int u = 0; u < 4; ++u)
            dh[j][u] = A.dhT ? A.dhT[((int64_t)n * H + h) * S + (int64_t)(rg + 32 * j) * dv + col0 + c4 + u] : 0.f;
    for (int64_t tile = ntiles - 1; tile >= 0; --tile) {
        const int64_t t0 = tile * C;
        const int tl = (int)min((int64_t)C, len - t0);
        const float *cp = ckp(tile0 + tile);
        // the tile's inputs, and delta and v - p of each token (recomputed)
        for (int e = tid; e < tl * DK; e += kBwThreads) {
            const int i = e / DK, d = e - i * DK;
            const int64_t row = (tok0 + t0 + i) * H + h;
            ks[i][d] = to_f32(k[row * DK + d]);
            qs[i][d] = to_f32(q[row * DK + d]);
        }
        for (int e = tid; e < tl * kBwCols; e += kBwThreads) {
            const int i = e / kBwCols, c = e - i * kBwCols;
            const int64_t row = (tok0 + t0 + i) * H + h;
            vps[i][c] = to_f32(v[row * dv + col0 + c]);
            dos[i][c] = A.dout ? to_f32(((const T *)A.dout)[row * dv + col0 + c]) : 0.f;
        }
        if (tid < tl) {
            const int64_t row = (tok0 + t0 + tid) * H + h;
            als[tid] = expf(gate_logdecay(to_f32(a[row]), A.b, A.gate));
            bts[tid] = to_f32(beta[row]);
        }
        __syncthreads();
        {
            float hs[kRows][4];
#pragma unroll
            for (int j = 0; j < kRows; ++j) {
                const float4 x = *(const float4 *)&cp[(int64_t)(rg + 32 * j) * dv];
                hs[j][0] = x.x;
                hs[j][1] = x.y;
                hs[j][2] = x.z;
                hs[j][3] = x.w;
            }
            for (int i = 0; i < tl; ++i) {
                float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < kRows; ++j) {
                    const float kd = ks[i][rg + 32 * j];
#pragma unroll
                    for (int u = 0; u < 4; ++u) part[u] = fmaf(hs[j][u], kd, part[u]);
                }
                reduce_cols(part);
                const float al = als[i], bt = bts[i];
                float dl[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) dl[u] = bt * (vps[i][c4 + u] - al * vec[c4 + u]);
                __syncthreads();   // every thread has read vec
                if (lane < 8)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (warp == 0) {
                            dls[i][c4 + u] = dl[u];
                            vps[i][c4 + u] = vps[i][c4 + u] - al * vec[c4 + u];   // v - p
                        }
                    }
#pragma unroll
                for (int j = 0; j < kRows; ++j) {
                    const float kd = ks[i][rg + 32 * j];
#pragma unroll
                    for (int u = 0; u < 4; ++u) hs[j][u] = fmaf(al, hs[j][u], kd * dl[u]);
                }
                __syncthreads();
            }
        }
        for (int i = tl - 1; i >= 0; --i) {
            const int64_t row = (tok0 + t0 + i) * H + h;
            // H_{i-1} rebuilt from the checkpoint, then H_i
            float hp[kRows][4];
#pragma unroll
            for (int j = 0; j < kRows; ++j) {
                const float4 x = *(const float4 *)&cp[(int64_t)(rg + 32 * j) * dv];
                hp[j][0] = x.x;
                hp[j][1] = x.y;
                hp[j][2] = x.z;
                hp[j][3] = x.w;
            }
            for (int r = 0; r < i; ++r) {
                const float al = als[r];
#pragma unroll
                for (int j = 0; j < kRows; ++j) {
                    const float kd = ks[r][rg + 32 * j];
#pragma unroll
                    for (int u = 0; u < 4; ++u) hp[j][u] = fmaf(al, hp[j][u], kd * dls[r][c4 + u]);
                }
            }
            const float al = als[i], bt = bts[i];
            float dd[4], dl[4], dof[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                dl[u] = dls[i][c4 + u];
                dof[u] = dos[i][c4 + u];
            }
            // dH += q do^T;  dq = H_i do (partial over the slice);  ddelta = dH^T k
            float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < kRows; ++j) {
                const int d = rg + 32 * j;
                const float qd = qs[i][d], kd = ks[i][d];
                float dqp = 0.f;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    dh[j][u] = fmaf(qd, dof[u], dh[j][u]);
                    dqp = fmaf(fmaf(al, hp[j][u], kd * dl[u]), dof[u], dqp);
                    part[u] = fmaf(dh[j][u], kd, part[u]);
                }
                dqp = rowsum(dqp);
                if ((lane & 7) == 0) A.pdq[(((int64_t)slice * A.T_total + tok0 + t0 + i) * H + h) * DK + d] = dqp;
            }
            reduce_cols(part);
#pragma unroll
            for (int u = 0; u < 4; ++u) dd[u] = vec[c4 + u];
            if (tid < kBwCols)
                ((T *)A.dv)[row * dv + col0 + tid] = from_f32<T>(bt * vec[tid]);
            float dbp = 0.f;
            if (tid < kBwCols) dbp = vec[tid] * vps[i][tid];
            const float db = reduce_scalar(dbp);
            // dk = dH delta + Hb dp (partial);  dHb = dH + k dp^T;  dalpha = <H_{i-1}, dHb>
            float dap = 0.f;
#pragma unroll
            for (int j = 0; j < kRows; ++j) {
                const int d = rg + 32 * j;
                const float kd = ks[i][d];
                float dkp = 0.f;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float dp = -bt * dd[u];
                    dkp = fmaf(dh[j][u], dl[u], dkp);
                    dkp = fmaf(al * hp[j][u], dp, dkp);
                    const float dhb = fmaf(kd, dp, dh[j][u]);
                    dap = fmaf(hp[j][u], dhb, dap);
                    dh[j][u] = al * dhb;
                }
                dkp = rowsum(dkp);
                if ((lane & 7) == 0) A.pdk[(((int64_t)slice * A.T_total + tok0 + t0 + i) * H + h) * DK + d] = dkp;
            }
            const float da_ = reduce_scalar(dap);
            if (tid == 0) {
                A.pdb[((int64_t)slice * A.T_total + tok0 + t0 + i) * H + h] = db;
                A.pda[((int64_t)slice * A.T_total + tok0 + t0 + i) * H + h] = da_;
            }
        }
        __syncthreads();   // the tile's shared arrays are reloaded for the previous tile
    }
    if (A.dh0)
#pragma unroll
        for (int j = 0; j < kRows; ++j)
            *(float4 *)&A.dh0[((int64_t)n * H + h) * S + (int64_t)(rg + 32 * j) * dv + col0 + c4] =
                make_float4(dh[j][0], dh[j][1], dh[j][2], dh[j][3]);
}

// Sum the per-slice partials and apply the gate derivative; one thread per
// (token, head, key index) for dq and dk, plus dbeta and da at key index 0.
template <typename T>
__global__ void __launch_bounds__(256)
bwd_finish_kernel(const BwArgs A, T *dq, T *dk, T *da, T *dbeta, int dk_dim) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t rows = A.T_total * A.H;
    if (e >= rows * dk_dim) return;
    const int64_t row = e / dk_dim;
    const int nslices = A.dv_ / kBwCols;
    float sq = 0.f, sk = 0.f;
    for (int s = 0; s < nslices; ++s) {
        sq += A.pdq[(int64_t)s * rows * dk_dim + e];
        sk += A.pdk[(int64_t)s * rows * dk_dim + e];
    }
    dq[e] = from_f32<T>(sq);
    dk[e] = from_f32<T>(sk);
    if (e % dk_dim == 0) {
        float sb = 0.f, sa = 0.f;
        for (int s = 0; s < nslices; ++s) {
            sb += A.pdb[(int64_t)s * rows + row];
            sa += A.pda[(int64_t)s * rows + row];
        }
        const float av = to_f32(((const T *)A.a)[row]);
        const float alpha = expf(gate_logdecay(av, A.b, A.gate));
        dbeta[row] = from_f32<T>(sb);
        da[row] = from_f32<T>(sa * alpha * gate_dgda(av, A.b, A.gate));
    }
}

template <typename T>
cudaError_t launch_bwd_t(const BwArgs &A, int N, int dk, void *dq, void *dkk, void *da,
                         void *dbeta, cudaStream_t stream) {
    const int64_t blocks = (int64_t)N * A.H * (A.dv_ / kBwCols);
    if (blocks > 0) {
        ProfScope prof(stream, "bwd_slice_kernel");
        if (dk == 128)
            bwd_slice_kernel<T, 128><<<(unsigned)blocks, kBwThreads, 0, stream>>>(A);
        else
            bwd_slice_kernel<T, 64><<<(unsigned)blocks, kBwThreads, 0, stream>>>(A);
        count_launch();
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    const int64_t n = A.T_total * A.H * dk;
    if (n > 0) {
        ProfScope prof(stream, "bwd_finish_kernel");
        bwd_finish_kernel<T><<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(
            A, (T *)dq, (T *)dkk, (T *)da, (T *)dbeta, dk);
        count_launch();
    }
    return cudaGetLastError();
}

}  // namespace

size_t bwd_scratch_bytes(int64_t tiles, int64_t T_total, int H, int dk, int dv) {
    const int64_t nsl = dv / kBwCols;
    return sizeof(float) * ((size_t)tiles * H * dk * dv + 2 * (size_t)nsl * T_total * H * dk +
                            2 * (size_t)nsl * T_total * H) + 4 * 256;
}

cudaError_t launch_bwd(const void *q, const void *k, const void *v, const void *a, const void *beta,
                       const float *h0, const void *dout, const float *dhT, void *dq, void *dk_,
                       void *dv, void *da, void *dbeta, float *dh0, gdr_dtype_t dtype, Plan plan,
                       int H, int dk, int dv_dim, int64_t T_total, int64_t tiles, float b,
                       gdr_gate_t gate, void *scratch, cudaStream_t stream) {
    if (plan.C != kBwMaxC) return cudaErrorInvalidValue;
    const int64_t nsl = dv_dim / kBwCols;
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    char *p = (char *)scratch;
    BwArgs A;
    A.q = q;
    A.k = k;
    A.v = v;
    A.a = a;
    A.beta = beta;
    A.h0 = h0;
    A.dout = dout;
    A.dhT = dhT;
    A.dv = dv;
    A.dh0 = dh0;
    A.ck = (float *)p;
    p += al(sizeof(float) * (size_t)tiles * H * dk * dv_dim);
    A.pdq = (float *)p;
    p += al(sizeof(float) * (size_t)nsl * T_total * H * dk);
    A.pdk = (float *)p;
    p += al(sizeof(float) * (size_t)nsl * T_total * H * dk);
    A.pdb = (float *)p;
    p += al(sizeof(float) * (size_t)nsl * T_total * H);
    A.pda = (float *)p;
    A.plan = plan;
    A.H = H;
    A.dv_ = dv_dim;
    A.C = plan.C;
    A.T_total = T_total;
    A.b = b;
    A.gate = (int)gate;
    if (dtype == GDR_BF16) return launch_bwd_t<__nv_bfloat16>(A, plan.N, dk, dq, dk_, da, dbeta, stream);
    return launch_bwd_t<float>(A, plan.N, dk, dq, dk_, da, dbeta, stream);
}

}  // namespace gdr
