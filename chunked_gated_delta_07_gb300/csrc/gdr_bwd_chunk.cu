// gdr_bwd_chunk.cu -- the backward pass in the chunked (WY) form, bf16 inputs,
// dk = dv = 128, 16-token tiles, bounded gate: every dense product on the tensor
// cores (mma.sync m16n8k8, tf32 operands, fp32 accumulation).
//
// Per tile with entering state H0, factored decays Kt = K (.) e^G, Kh = K (.) e^-G,
// Qt = Q (.) e^G (G the in-tile cumulative log-decay, per key channel), the
// forward is [P1 §3.2, P2 §2.1, P3 §3.1]
//   A = beta (.) strict_lower(Kt Kh^T),  S = lower(Qt Kh^T),  T = (I + A)^{-1}
//   W = T diag(beta) Kt,  U = T diag(beta) V,  D = U - W H0
//   O = Qt H0 + S D,      H1 = diag(e^{G_C}) H0 + Ke^T D,  Ke = Kh (.) e^{G_C}
// and, for L = <dO, O> + <dH_T, H_T>, with dH1 the gradient at the tile's end:
//   dD  = S^T dO + Ke dH1                       dH0 = diag(e^{G_C}) dH1 + Qt^T dO - W^T dD
//   dS  = lower(dO D^T)     dKe = D dH1^T       dW  = -dD H0^T        dQt = dO H0^T + dS Kh
//   dYu = T^T dD,  dYw = T^T dW  (back substitution)
//   dA  = -strict_lower(dYu U^T + dYw W^T)      dV  = diag(beta) dYu
//   dKt = diag(beta) dYw + (beta (.) dA) Kh     dKh = (beta (.) dA)^T Kt + dS^T Qt + dKe (.) e^{G_C}
//   dbeta_i = dYu_i . V_i + dYw_i . Kt_i + sum_j dA_ij (Kt Kh^T)_ij
//   dG = dQt (.) Qt + dKt (.) Kt - dKh (.) Kh, plus at the tile's last token
//        sum_i dKe (.) Ke + e^{G_C} (.) rowsum(dH1 (.) H0);  dg = reverse cumsum of dG
//   dq = dQt (.) e^G,  dk = dKt (.) e^G + dKh (.) e^-G,  da = dg g'(a)
// Three kernels:
//   bwd_fwd_chain_kernel  per (sequence, head): the state chain; stores H0 and D of
//                         every tile
//   bwd_adj_chain_kernel  per (sequence, head), tiles in reverse: the dH chain; stores
//                         dH1 of every tile and writes dh0
//   bwd_tile_kernel       per (tile, head), all tiles at once: every input gradient
// The scalar-gate form is the per-channel form with every channel's gate equal.
#include "gdr_internal.cuh"
#include "gdr_mma.cuh"

namespace gdr {
namespace {

constexpr int kT = 16;
constexpr int kD = 128;
constexpr int kLd = 132;
constexpr int kPd = 20;
constexpr int kThreads = 256;
constexpr int kTile2 = kT * kLd;   // floats of one [16][kLd] buffer

struct BcArgs {
    const __nv_bfloat16 *q, *k, *v, *a, *beta, *dout;
    const float *h0, *dhT;
    __nv_bfloat16 *dq, *dk, *dv, *da, *dbeta;
    float *dh0;
    float *Hst, *dHst, *Dst;   // [tiles][H][128][128], [tiles][H][128][128], [tiles][H][16][128]
    Plan p;
    int H;
    float b;
};

template <bool VEC>
__device__ __forceinline__ float gate_in(const __nv_bfloat16 *a, int64_t row, int d) {
    return __bfloat162float(VEC ? a[row * kD + d] : a[row]);
}

// Stage one tile: per key channel (threads 0..127) the cumulative log-decay and the
// factored rows; the other 128 threads load one 128-wide input (V or dO) and beta.
template <bool VEC>
__device__ __forceinline__ void stage_tile(const BcArgs &A, int64_t t0, int len, int h, float *Kt,
                                           float *Kh, float *Qt, float *Gb, float *eg,
                                           const __nv_bfloat16 *other, float *Ob, float *bs) {
    const int tid = threadIdx.x;
    if (tid < kD) {
        const int d = tid;
        float G = 0.f, eGC = 1.f;
#pragma unroll 4
        for (int i = 0; i < kT; ++i) {
            float kt = 0.f, kh = 0.f, qt = 0.f, gg = 0.f;
            if (i < len) {
                const int64_t row = (t0 + i) * A.H + h;
                G += gate_logdecay(gate_in<VEC>(A.a, row, d), A.b, GDR_GATE_BOUNDED);
                const float e = expf(G), en = expf(-G), kd = __bfloat162float(A.k[row * kD + d]);
                kt = kd * e;
                kh = kd * en;
                if (Qt) qt = __bfloat162float(A.q[row * kD + d]) * e;
                eGC = e;
                gg = G;
            }
            Kt[i * kLd + d] = kt;
            Kh[i * kLd + d] = kh;
            if (Qt) Qt[i * kLd + d] = qt;
            if (Gb) Gb[i * kLd + d] = gg;
        }
        eg[d] = eGC;
    } else {
        const int c = tid - kD;
#pragma unroll 4
        for (int i = 0; i < kT; ++i)
            Ob[i * kLd + c] = (i < len && other) ? __bfloat162float(other[((t0 + i) * A.H + h) * kD + c]) : 0.f;
        if (c < kT) bs[c] = c < len ? __bfloat162float(A.beta[(t0 + c) * A.H + h]) : 0.f;
    }
}

// 16 x 16 product X Y^T over K = 128 (one 8-column half of the output per warp):
// out[i][j] for j in j0..j0+7.
__device__ __forceinline__ void gram_half(float (&acc)[4], const float *X, const float *Y, int j0,
                                          int g, int t) {
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll 4
    for (int k0 = 0; k0 < kD; k0 += 8) {
        uint32_t af[4], b0, b1;
        load_a(af, X, kLd, 0, k0, g, t);
        load_bt(b0, b1, Y, kLd, k0, j0, g, t);
        mma8(acc, af, b0, b1);
    }
}

// Forward substitution x = (I + A)^{-1} diag(beta) y on one column of a [16][kLd]
// buffer, in place (A strictly lower, row stride kPd).
__device__ __forceinline__ void fwd_subst(float *X, int col, const float *Am, const float *bs) {
    float x[kT];
#pragma unroll
    for (int i = 0; i < kT; ++i) {
        float acc = bs[i] * X[i * kLd + col];
#pragma unroll
        for (int j = 0; j < i; ++j) acc = fmaf(-Am[i * kPd + j], x[j], acc);
        x[i] = acc;
    }
#pragma unroll
    for (int i = 0; i < kT; ++i) X[i * kLd + col] = x[i];
}

// Back substitution y = (I + A)^{-T} x on one column, from src into dst.
__device__ __forceinline__ void back_subst(const float *src, float *dst, int col, const float *Am) {
    float y[kT];
#pragma unroll
    for (int i = kT - 1; i >= 0; --i) {
        float acc = src[i * kLd + col];
#pragma unroll
        for (int j = i + 1; j < kT; ++j) acc = fmaf(-Am[j * kPd + i], y[j], acc);
        y[i] = acc;
    }
#pragma unroll
    for (int i = 0; i < kT; ++i) dst[i * kLd + col] = y[i];
}

// A = beta (.) strict_lower(Kt Kh^T) into Am (warps 0-1 call this)
__device__ __forceinline__ void build_A(const float *Kt, const float *Kh, const float *bs, float *Am,
                                        float *KK, int half, int g, int t) {
    float acc[4];
    const int j0 = 8 * half;
    gram_half(acc, Kt, Kh, j0, g, t);
    const int i0 = g, i1 = g + 8, ja = j0 + 2 * t, jb = ja + 1;
    Am[i0 * kPd + ja] = ja < i0 ? bs[i0] * acc[0] : 0.f;
    Am[i0 * kPd + jb] = jb < i0 ? bs[i0] * acc[1] : 0.f;
    Am[i1 * kPd + ja] = ja < i1 ? bs[i1] * acc[2] : 0.f;
    Am[i1 * kPd + jb] = jb < i1 ? bs[i1] * acc[3] : 0.f;
    if (KK) {
        KK[i0 * kPd + ja] = acc[0];
        KK[i0 * kPd + jb] = acc[1];
        KK[i1 * kPd + ja] = acc[2];
        KK[i1 * kPd + jb] = acc[3];
    }
}

// lower (j <= i) part of X Y^T into M
__device__ __forceinline__ void build_lower(const float *X, const float *Y, float *M, int half, int g,
                                            int t) {
    float acc[4];
    const int j0 = 8 * half;
    gram_half(acc, X, Y, j0, g, t);
    const int i0 = g, i1 = g + 8, ja = j0 + 2 * t, jb = ja + 1;
    M[i0 * kPd + ja] = ja <= i0 ? acc[0] : 0.f;
    M[i0 * kPd + jb] = jb <= i0 ? acc[1] : 0.f;
    M[i1 * kPd + ja] = ja <= i1 ? acc[2] : 0.f;
    M[i1 * kPd + jb] = jb <= i1 ? acc[3] : 0.f;
}

__device__ __forceinline__ void copy_state_out(const float *Hs, float *dst) {
    for (int e = threadIdx.x * 4; e < kD * kD; e += kThreads * 4) {
        const int r = e >> 7, c = e & (kD - 1);
        *(float4 *)&dst[e] = *(const float4 *)&Hs[r * kLd + c];
    }
}

__device__ __forceinline__ void copy_state_in(float *Hs, const float *src) {
    for (int e = threadIdx.x * 4; e < kD * kD; e += kThreads * 4) {
        const int r = e >> 7, c = e & (kD - 1);
        *(float4 *)&Hs[r * kLd + c] = src ? *(const float4 *)&src[e] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// ---------------------------------------------------------------------------
// forward state chain: stores H0 and D of every tile
// ---------------------------------------------------------------------------
constexpr int kF_H = 0, kF_Kt = kF_H + kD * kLd, kF_Kh = kF_Kt + kTile2, kF_U = kF_Kh + kTile2,
              kF_A = kF_U + kTile2, kF_eg = kF_A + kT * kPd, kF_b = kF_eg + kD,
              kF_total = kF_b + kT;

template <bool VEC>
__global__ void __launch_bounds__(kThreads)
bwd_fwd_chain_kernel(const BcArgs A) {
    extern __shared__ float sm[];
    float *Hs = sm + kF_H, *Kt = sm + kF_Kt, *Kh = sm + kF_Kh, *Ub = sm + kF_U, *Am = sm + kF_A;
    float *eg = sm + kF_eg, *bs = sm + kF_b;
    const int h = blockIdx.x % A.H, n = blockIdx.x / A.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
    const int c0 = 16 * warp;
    const size_t sbase = ((size_t)n * A.H + h) * kD * kD;
    copy_state_in(Hs, A.h0 ? A.h0 + sbase : nullptr);
    const int64_t s = A.p.seq_start[n], e_end = A.p.seq_start[n + 1], tile0 = A.p.chunk_base[n];
    int64_t c = tile0;
    for (int64_t t0 = s; t0 < e_end; t0 += kT, ++c) {
        const int len = (int)min((int64_t)kT, e_end - t0);
        __syncthreads();
        copy_state_out(Hs, A.Hst + ((size_t)c * A.H + h) * kD * kD);
        stage_tile<VEC>(A, t0, len, h, Kt, Kh, nullptr, nullptr, eg, A.v, Ub, bs);
        __syncthreads();
        if (warp < 2) build_A(Kt, Kh, bs, Am, nullptr, warp, g, t);
        __syncthreads();
        fwd_subst(tid < kD ? Kt : Ub, tid & (kD - 1), Am, bs);   // Kt -> W, V -> U
        if (tid < kD)
            for (int i = 0; i < kT; ++i) Kh[i * kLd + tid] *= eg[tid];   // Ke
        __syncthreads();
        // D = U - W H0 on this warp's columns; stored for the tile-gradient kernel
        float dacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int n0 = c0 + 8 * nt;
            dacc[nt][0] = Ub[g * kLd + n0 + 2 * t];
            dacc[nt][1] = Ub[g * kLd + n0 + 2 * t + 1];
            dacc[nt][2] = Ub[(g + 8) * kLd + n0 + 2 * t];
            dacc[nt][3] = Ub[(g + 8) * kLd + n0 + 2 * t + 1];
        }
#pragma unroll 2
        for (int k0 = 0; k0 < kD; k0 += 8) {
            uint32_t aw[4];
            load_a(aw, Kt, kLd, 0, k0, g, t);
            aw[0] ^= 0x80000000u;   // -W: flip the sign bits
            aw[1] ^= 0x80000000u;
            aw[2] ^= 0x80000000u;
            aw[3] ^= 0x80000000u;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t b0, b1;
                load_b(b0, b1, Hs, kLd, k0, c0 + 8 * nt, g, t);
                mma8(dacc[nt], aw, b0, b1);
            }
        }
        float *Dg = A.Dst + ((size_t)c * A.H + h) * kT * kD;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int col = c0 + 8 * nt + 2 * t;
            Ub[g * kLd + col] = dacc[nt][0];
            Ub[g * kLd + col + 1] = dacc[nt][1];
            Ub[(g + 8) * kLd + col] = dacc[nt][2];
            Ub[(g + 8) * kLd + col + 1] = dacc[nt][3];
            *(float2 *)&Dg[g * kD + col] = make_float2(dacc[nt][0], dacc[nt][1]);
            *(float2 *)&Dg[(g + 8) * kD + col] = make_float2(dacc[nt][2], dacc[nt][3]);
        }
        __syncwarp();
        // H1 = diag(e^{G_C}) H0 + Ke^T D on this warp's columns
        uint32_t bd[2][2][2];
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) load_b(bd[ks][nt][0], bd[ks][nt][1], Ub, kLd, 8 * ks, c0 + 8 * nt, g, t);
#pragma unroll 2
        for (int mt = 0; mt < kD / 16; ++mt) {
            const int r0 = 16 * mt;
            const float e0 = eg[r0 + g], e1 = eg[r0 + g + 8];
            uint32_t ak[2][4];
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) load_at(ak[ks], Kh, kLd, r0, 8 * ks, g, t);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int col = c0 + 8 * nt + 2 * t;
                float *p0 = &Hs[(r0 + g) * kLd + col], *p1 = &Hs[(r0 + g + 8) * kLd + col];
                float acc[4] = {e0 * p0[0], e0 * p0[1], e1 * p1[0], e1 * p1[1]};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) mma8(acc, ak[ks], bd[ks][nt][0], bd[ks][nt][1]);
                p0[0] = acc[0];
                p0[1] = acc[1];
                p1[0] = acc[2];
                p1[1] = acc[3];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// adjoint state chain, tiles in reverse: stores dH1 of every tile, writes dh0
// ---------------------------------------------------------------------------
constexpr int kA_H = 0, kA_Kt = kA_H + kD * kLd, kA_Kh = kA_Kt + kTile2, kA_Qt = kA_Kh + kTile2,
              kA_O = kA_Qt + kTile2, kA_E = kA_O + kTile2, kA_A = kA_E + kTile2,
              kA_S = kA_A + kT * kPd, kA_eg = kA_S + kT * kPd, kA_b = kA_eg + kD,
              kA_total = kA_b + kT;

template <bool VEC>
__global__ void __launch_bounds__(kThreads)
bwd_adj_chain_kernel(const BcArgs A) {
    extern __shared__ float sm[];
    float *dH = sm + kA_H, *Kt = sm + kA_Kt, *Kh = sm + kA_Kh, *Qt = sm + kA_Qt, *Ob = sm + kA_O;
    float *Eb = sm + kA_E, *Am = sm + kA_A, *Sm = sm + kA_S, *eg = sm + kA_eg, *bs = sm + kA_b;
    const int h = blockIdx.x % A.H, n = blockIdx.x / A.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
    const int c0 = 16 * warp;
    const size_t sbase = ((size_t)n * A.H + h) * kD * kD;
    copy_state_in(dH, A.dhT ? A.dhT + sbase : nullptr);
    const int64_t s = A.p.seq_start[n], e_end = A.p.seq_start[n + 1], tile0 = A.p.chunk_base[n];
    const int64_t ntiles = A.p.chunk_base[n + 1] - tile0;
    for (int64_t tt = ntiles - 1; tt >= 0; --tt) {
        const int64_t t0 = s + tt * kT, c = tile0 + tt;
        const int len = (int)min((int64_t)kT, e_end - t0);
        __syncthreads();
        copy_state_out(dH, A.dHst + ((size_t)c * A.H + h) * kD * kD);
        stage_tile<VEC>(A, t0, len, h, Kt, Kh, Qt, nullptr, eg, A.dout, Ob, bs);
        __syncthreads();
        if (warp < 2) build_A(Kt, Kh, bs, Am, nullptr, warp, g, t);
        else if (warp < 4) build_lower(Qt, Kh, Sm, warp - 2, g, t);
        __syncthreads();
        if (tid < kD) {
            fwd_subst(Kt, tid, Am, bs);   // Kt -> W
            for (int i = 0; i < kT; ++i) Kh[i * kLd + tid] *= eg[tid];   // Ke
        }
        __syncthreads();
        // dD = S^T dO + Ke dH1 on this warp's columns
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 2
        for (int k0 = 0; k0 < kD; k0 += 8) {
            uint32_t ak[4];
            load_a(ak, Kh, kLd, 0, k0, g, t);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t b0, b1;
                load_b(b0, b1, dH, kLd, k0, c0 + 8 * nt, g, t);
                mma8(acc[nt], ak, b0, b1);
            }
        }
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            uint32_t as[4];
            load_at(as, Sm, kPd, 0, 8 * ks, g, t);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t b0, b1;
                load_b(b0, b1, Ob, kLd, 8 * ks, c0 + 8 * nt, g, t);
                mma8(acc[nt], as, b0, b1);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int col = c0 + 8 * nt + 2 * t;
            Eb[g * kLd + col] = acc[nt][0];
            Eb[g * kLd + col + 1] = acc[nt][1];
            Eb[(g + 8) * kLd + col] = acc[nt][2];
            Eb[(g + 8) * kLd + col + 1] = acc[nt][3];
        }
        __syncwarp();
        // dH0 = diag(e^{G_C}) dH1 + Qt^T dO - W^T dD on this warp's columns
        uint32_t bo[2][2][2], be[2][2][2];
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                load_b(bo[ks][nt][0], bo[ks][nt][1], Ob, kLd, 8 * ks, c0 + 8 * nt, g, t);
                load_b(be[ks][nt][0], be[ks][nt][1], Eb, kLd, 8 * ks, c0 + 8 * nt, g, t);
            }
#pragma unroll 2
        for (int mt = 0; mt < kD / 16; ++mt) {
            const int r0 = 16 * mt;
            const float e0 = eg[r0 + g], e1 = eg[r0 + g + 8];
            uint32_t aq[2][4], aw[2][4];
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                load_at(aq[ks], Qt, kLd, r0, 8 * ks, g, t);
                load_at(aw[ks], Kt, kLd, r0, 8 * ks, g, t);
#pragma unroll
                for (int u = 0; u < 4; ++u) aw[ks][u] ^= 0x80000000u;   // -W^T
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int col = c0 + 8 * nt + 2 * t;
                float *p0 = &dH[(r0 + g) * kLd + col], *p1 = &dH[(r0 + g + 8) * kLd + col];
                float d4[4] = {e0 * p0[0], e0 * p0[1], e1 * p1[0], e1 * p1[1]};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    mma8(d4, aq[ks], bo[ks][nt][0], bo[ks][nt][1]);
                    mma8(d4, aw[ks], be[ks][nt][0], be[ks][nt][1]);
                }
                p0[0] = d4[0];
                p0[1] = d4[1];
                p1[0] = d4[2];
                p1[1] = d4[3];
            }
        }
    }
    __syncthreads();
    if (A.dh0) copy_state_out(dH, A.dh0 + sbase);
}

// ---------------------------------------------------------------------------
// per-tile gradients
// ---------------------------------------------------------------------------
constexpr int kG_S = 0;                            // dH1, then H0   [128][kLd]
constexpr int kG_Kt = kG_S + kD * kLd;             // Kt
constexpr int kG_Kh = kG_Kt + kTile2;              // Kh
constexpr int kG_Qt = kG_Kh + kTile2;              // Qt
constexpr int kG_G = kG_Qt + kTile2;               // G
constexpr int kG_V = kG_G + kTile2;                // V
constexpr int kG_O = kG_V + kTile2;                // dO
constexpr int kG_W = kG_O + kTile2;                // W
constexpr int kG_U = kG_W + kTile2;                // U
constexpr int kG_D = kG_U + kTile2;                // D
constexpr int kG_E = kG_D + kTile2;                // dD
constexpr int kG_F1 = kG_E + kTile2;               // dW, then dYu
constexpr int kG_F2 = kG_F1 + kTile2;              // dYw
constexpr int kG_X = kG_F2 + kTile2;               // dG (per token, channel)
constexpr int kG_A = kG_X + kTile2;                // A        [16][kPd]
constexpr int kG_KK = kG_A + kT * kPd;             // Kt Kh^T
constexpr int kG_Sm = kG_KK + kT * kPd;            // S
constexpr int kG_dS = kG_Sm + kT * kPd;            // dS
constexpr int kG_dA = kG_dS + kT * kPd;            // dA
constexpr int kG_bdA = kG_dA + kT * kPd;           // beta_i dA_ij
constexpr int kG_eg = kG_bdA + kT * kPd;           // e^{G_C} [128]
constexpr int kG_rG = kG_eg + kD;                  // extra dG_C [128]
constexpr int kG_b = kG_rG + kD;                   // beta [16]
constexpr int kG_total = kG_b + kT;

template <bool VEC>
__global__ void __launch_bounds__(kThreads)
bwd_tile_kernel(const BcArgs A) {
    extern __shared__ float sm[];
    float *Sb = sm + kG_S, *Kt = sm + kG_Kt, *Kh = sm + kG_Kh, *Qt = sm + kG_Qt, *Gb = sm + kG_G;
    float *Vb = sm + kG_V, *Ob = sm + kG_O, *Wb = sm + kG_W, *Ub = sm + kG_U, *Db = sm + kG_D;
    float *Eb = sm + kG_E, *F1 = sm + kG_F1, *F2 = sm + kG_F2, *Xb = sm + kG_X;
    float *Am = sm + kG_A, *KK = sm + kG_KK, *Sm = sm + kG_Sm, *dS = sm + kG_dS, *dA = sm + kG_dA;
    float *bdA = sm + kG_bdA, *eg = sm + kG_eg, *rG = sm + kG_rG, *bs = sm + kG_b;
    const int64_t c = blockIdx.x;
    const int h = blockIdx.y;
    const int n = find_owner(A.p.chunk_base, A.p.N, c);
    if (n < 0) return;
    const int64_t t0 = A.p.seq_start[n] + (c - A.p.chunk_base[n]) * kT;
    const int len = (int)min((int64_t)kT, A.p.seq_start[n + 1] - t0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
    const int c0 = 16 * warp;
    const size_t st = ((size_t)c * A.H + h) * kD * kD;
    // ---- stage: factored rows, G, V, dO, beta, D; dH1 into the state buffer
    stage_tile<VEC>(A, t0, len, h, Kt, Kh, Qt, Gb, eg, A.v, Vb, bs);
    for (int e = tid; e < kT * kD; e += kThreads) {
        const int i = e >> 7, col = e & (kD - 1);
        const int64_t row = (t0 + i) * A.H + h;
        Ob[i * kLd + col] = (i < len && A.dout) ? __bfloat162float(A.dout[row * kD + col]) : 0.f;
        Db[i * kLd + col] = A.Dst[((size_t)c * A.H + h) * kT * kD + e];
        Ub[i * kLd + col] = i < len ? __bfloat162float(A.v[row * kD + col]) : 0.f;   // U built in place
    }
    copy_state_in(Sb, A.dHst + st);
    __syncthreads();
    // ---- 16 x 16 products
    if (warp < 2) build_A(Kt, Kh, bs, Am, KK, warp, g, t);
    else if (warp < 4) build_lower(Qt, Kh, Sm, warp - 2, g, t);
    else if (warp < 6) build_lower(Ob, Db, dS, warp - 4, g, t);   // dS = lower(dO D^T)
    if (tid < kD)
        for (int i = 0; i < kT; ++i) Wb[i * kLd + tid] = Kt[i * kLd + tid];
    __syncthreads();
    // ---- W and U
    fwd_subst(tid < kD ? Wb : Ub, tid & (kD - 1), Am, bs);
    __syncthreads();
    // ---- dD = S^T dO + Ke dH1 (this warp's dv columns); dKe = D dH1^T (this warp's dk columns)
    float dke[2][4];
    {
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int u = 0; u < 4; ++u) dke[nt][u] = 0.f;
#pragma unroll 2
        for (int k0 = 0; k0 < kD; k0 += 8) {
            uint32_t ak[4], ad[4];
            // Ke = Kh (.) e^{G_C}: scale the A fragment by the channel factors
            ak[0] = tf32(Kh[g * kLd + k0 + t] * eg[k0 + t]);
            ak[1] = tf32(Kh[(g + 8) * kLd + k0 + t] * eg[k0 + t]);
            ak[2] = tf32(Kh[g * kLd + k0 + t + 4] * eg[k0 + t + 4]);
            ak[3] = tf32(Kh[(g + 8) * kLd + k0 + t + 4] * eg[k0 + t + 4]);
            load_a(ad, Db, kLd, 0, k0, g, t);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t b0, b1;
                load_b(b0, b1, Sb, kLd, k0, c0 + 8 * nt, g, t);    // dH1[k][c]
                mma8(acc[nt], ak, b0, b1);
                load_bt(b0, b1, Sb, kLd, k0, c0 + 8 * nt, g, t);   // dH1^T[k][d] = dH1[d][k]
                mma8(dke[nt], ad, b0, b1);
            }
        }
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            uint32_t as[4];
            load_at(as, Sm, kPd, 0, 8 * ks, g, t);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t b0, b1;
                load_b(b0, b1, Ob, kLd, 8 * ks, c0 + 8 * nt, g, t);
                mma8(acc[nt], as, b0, b1);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int col = c0 + 8 * nt + 2 * t;
            Eb[g * kLd + col] = acc[nt][0];
            Eb[g * kLd + col + 1] = acc[nt][1];
            Eb[(g + 8) * kLd + col] = acc[nt][2];
            Eb[(g + 8) * kLd + col + 1] = acc[nt][3];
        }
    }
    __syncthreads();
    // ---- H0 into the state buffer, and e^{G_C} rowsum(dH1 (.) H0) (dH1 reread from HBM)
    {
        const float *H0g = A.Hst + st, *dH1g = A.dHst + st;
        for (int r = warp; r < kD; r += 8) {
            const float4 x = *(const float4 *)&H0g[r * kD + 4 * lane];
            const float4 y = *(const float4 *)&dH1g[r * kD + 4 * lane];
            *(float4 *)&Sb[r * kLd + 4 * lane] = x;
            float p = x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
            if (lane == 0) rG[r] = eg[r] * p;
        }
    }
    __syncthreads();
    // ---- dQt_a = dO H0^T and dW = -dD H0^T (this warp's dk columns)
    float dq[2][4];
    {
        float dw[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int u = 0; u < 4; ++u) dq[nt][u] = dw[nt][u] = 0.f;
#pragma unroll 2
        for (int k0 = 0; k0 < kD; k0 += 8) {
            uint32_t ao[4], ae[4];
            load_a(ao, Ob, kLd, 0, k0, g, t);
            load_a(ae, Eb, kLd, 0, k0, g, t);
#pragma unroll
            for (int u = 0; u < 4; ++u) ae[u] ^= 0x80000000u;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t b0, b1;
                load_bt(b0, b1, Sb, kLd, k0, c0 + 8 * nt, g, t);   // H0^T[k][d] = H0[d][k]
                mma8(dq[nt], ao, b0, b1);
                mma8(dw[nt], ae, b0, b1);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int col = c0 + 8 * nt + 2 * t;
            F1[g * kLd + col] = dw[nt][0];
            F1[g * kLd + col + 1] = dw[nt][1];
            F1[(g + 8) * kLd + col] = dw[nt][2];
            F1[(g + 8) * kLd + col + 1] = dw[nt][3];
        }
    }
    __syncthreads();
    // ---- dYw = T^T dW (threads 0..127, dk columns); dYu = T^T dD (threads 128..255)
    if (tid < kD) back_subst(F1, F2, tid, Am);
    __syncthreads();
    if (tid >= kD) back_subst(Eb, F1, tid - kD, Am);   // F1 <- dYu (dW no longer needed)
    __syncthreads();
    // ---- dA = -strict_lower(dYu U^T + dYw W^T) (warps 0-1); dV = diag(beta) dYu
    if (warp < 2) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int j0 = 8 * warp;
#pragma unroll 4
        for (int k0 = 0; k0 < kD; k0 += 8) {
            uint32_t af[4], b0, b1;
            load_a(af, F1, kLd, 0, k0, g, t);
            load_bt(b0, b1, Ub, kLd, k0, j0, g, t);
            mma8(acc, af, b0, b1);
            load_a(af, F2, kLd, 0, k0, g, t);
            load_bt(b0, b1, Wb, kLd, k0, j0, g, t);
            mma8(acc, af, b0, b1);
        }
        const int i0 = g, i1 = g + 8, ja = j0 + 2 * t, jb = ja + 1;
        const float v00 = ja < i0 ? -acc[0] : 0.f, v01 = jb < i0 ? -acc[1] : 0.f;
        const float v10 = ja < i1 ? -acc[2] : 0.f, v11 = jb < i1 ? -acc[3] : 0.f;
        dA[i0 * kPd + ja] = v00;
        dA[i0 * kPd + jb] = v01;
        dA[i1 * kPd + ja] = v10;
        dA[i1 * kPd + jb] = v11;
        bdA[i0 * kPd + ja] = bs[i0] * v00;
        bdA[i0 * kPd + jb] = bs[i0] * v01;
        bdA[i1 * kPd + ja] = bs[i1] * v10;
        bdA[i1 * kPd + jb] = bs[i1] * v11;
    }
    for (int e = tid; e < kT * kD; e += kThreads) {
        const int i = e >> 7, col = e & (kD - 1);
        if (i < len) A.dv[((t0 + i) * A.H + h) * kD + col] = __float2bfloat16_rn(bs[i] * F1[i * kLd + col]);
    }
    __syncthreads();
    // ---- dKt, dKh, dQt on this warp's dk columns; dG into Xb
    {
        float dkt[2][4], dkh[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int u = 0; u < 4; ++u) dkt[nt][u] = dkh[nt][u] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            uint32_t a_bdA[4], a_bdAt[4], a_dS[4], a_dSt[4];
            load_a(a_bdA, bdA, kPd, 0, 8 * ks, g, t);
            load_at(a_bdAt, bdA, kPd, 0, 8 * ks, g, t);
            load_a(a_dS, dS, kPd, 0, 8 * ks, g, t);
            load_at(a_dSt, dS, kPd, 0, 8 * ks, g, t);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t bh0, bh1, bt0, bt1, bq0, bq1;
                load_b(bh0, bh1, Kh, kLd, 8 * ks, c0 + 8 * nt, g, t);
                load_b(bt0, bt1, Kt, kLd, 8 * ks, c0 + 8 * nt, g, t);
                load_b(bq0, bq1, Qt, kLd, 8 * ks, c0 + 8 * nt, g, t);
                mma8(dkt[nt], a_bdA, bh0, bh1);    // (beta dA) Kh
                mma8(dkh[nt], a_bdAt, bt0, bt1);   // (beta dA)^T Kt
                mma8(dkh[nt], a_dSt, bq0, bq1);    // dS^T Qt
                mma8(dq[nt], a_dS, bh0, bh1);      // dS Kh
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = g + 8 * (u >> 1), d = c0 + 8 * nt + 2 * t + (u & 1);
                const float kt = Kt[i * kLd + d], kh = Kh[i * kLd + d], qt = Qt[i * kLd + d];
                const float dKt = dkt[nt][u] + bs[i] * F2[i * kLd + d];
                const float dKh = dkh[nt][u] + dke[nt][u] * eg[d];
                float dG = dq[nt][u] * qt + dKt * kt - dKh * kh;
                Xb[i * kLd + d] = dG;
                const float G = Gb[i * kLd + d];
                if (i < len) {
                    const int64_t r = ((t0 + i) * A.H + h) * kD + d;
                    A.dq[r] = __float2bfloat16_rn(dq[nt][u] * expf(G));
                    A.dk[r] = __float2bfloat16_rn(dKt * expf(G) + dKh * expf(-G));
                }
                // sum_i dKe (.) Ke, folded into the last token's dG below
                dke[nt][u] *= kh * eg[d];
            }
        // column sums over the 16 rows of dKe (.) Ke: rows g and g+8 of the 8 lane groups
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float x = dke[nt][u] + dke[nt][u + 2];
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                if (g == 0) rG[c0 + 8 * nt + 2 * t + u] += x;
            }
    }
    __syncthreads();
    // ---- dbeta (threads 0..15, one token each)
    if (tid < kT && tid < len) {
        const int i = tid;
        float acc = 0.f;
        for (int col = 0; col < kD; ++col)
            acc = fmaf(F1[i * kLd + col], Vb[i * kLd + col], fmaf(F2[i * kLd + col], Kt[i * kLd + col], acc));
        for (int j = 0; j < i; ++j) acc = fmaf(dA[i * kPd + j], KK[i * kPd + j], acc);
        A.dbeta[(t0 + i) * A.H + h] = __float2bfloat16_rn(acc);
    }
    // ---- da: the last token also carries dG_C; reverse cumsum over the tile
    if (VEC) {
        if (tid < kD) {
            const int d = tid;
            float acc = 0.f;
            for (int i = len - 1; i >= 0; --i) {
                acc += Xb[i * kLd + d] + (i == len - 1 ? rG[d] : 0.f);
                const int64_t r = ((t0 + i) * A.H + h) * kD + d;
                const float av = __bfloat162float(A.a[r]);
                const float sg = 1.f / (1.f + expf(-av));
                A.da[r] = __float2bfloat16_rn(acc * (-A.b * sg * (1.f - sg)));
            }
        }
    } else {
        // per-token sums over the channels, then the reverse cumsum (warp 0)
        __shared__ float rowsum[kT];
        if (warp < 4) {
            for (int i = warp; i < kT; i += 4) {
                float x = 0.f;
                for (int d = lane; d < kD; d += 32) x += Xb[i * kLd + d] + (i == len - 1 ? rG[d] : 0.f);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                if (lane == 0) rowsum[i] = x;
            }
        }
        __syncthreads();
        if (tid == 0) {
            float acc = 0.f;
            for (int i = len - 1; i >= 0; --i) {
                acc += rowsum[i];
                const int64_t r = (t0 + i) * A.H + h;
                const float av = __bfloat162float(A.a[r]);
                const float sg = 1.f / (1.f + expf(-av));
                A.da[r] = __float2bfloat16_rn(acc * (-A.b * sg * (1.f - sg)));
            }
        }
    }
}

template <bool VEC>
cudaError_t launch_chunk_bwd_t(const BcArgs &A, int64_t max_tiles) {
    cudaError_t err;
    const int N = A.p.N, H = A.H;
    auto kf = bwd_fwd_chain_kernel<VEC>;
    auto ka = bwd_adj_chain_kernel<VEC>;
    auto kt = bwd_tile_kernel<VEC>;
    const size_t sf = sizeof(float) * kF_total, sa = sizeof(float) * kA_total, sg = sizeof(float) * kG_total;
    if ((err = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sf)) != cudaSuccess) return err;
    if ((err = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sa)) != cudaSuccess) return err;
    if ((err = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sg)) != cudaSuccess) return err;
    return cudaSuccess;
}

}  // namespace

size_t chunk_bwd_scratch_bytes(int64_t tiles, int H) {
    return sizeof(float) * (size_t)tiles * H * (2 * (size_t)kD * kD + (size_t)kT * kD) + 3 * 256;
}

cudaError_t launch_chunk_bwd(const void *q, const void *k, const void *v, const void *a,
                             const void *beta, const float *h0, const void *dout, const float *dhT,
                             void *dq, void *dk, void *dv, void *da, void *dbeta, float *dh0,
                             Plan plan, int H, int64_t max_tiles, float b, bool per_channel,
                             void *scratch, cudaStream_t stream) {
    if (plan.C != kT) return cudaErrorInvalidValue;
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    BcArgs A;
    A.q = (const __nv_bfloat16 *)q;
    A.k = (const __nv_bfloat16 *)k;
    A.v = (const __nv_bfloat16 *)v;
    A.a = (const __nv_bfloat16 *)a;
    A.beta = (const __nv_bfloat16 *)beta;
    A.dout = (const __nv_bfloat16 *)dout;
    A.h0 = h0;
    A.dhT = dhT;
    A.dq = (__nv_bfloat16 *)dq;
    A.dk = (__nv_bfloat16 *)dk;
    A.dv = (__nv_bfloat16 *)dv;
    A.da = (__nv_bfloat16 *)da;
    A.dbeta = (__nv_bfloat16 *)dbeta;
    A.dh0 = dh0;
    char *p = (char *)scratch;
    const size_t st = sizeof(float) * (size_t)max_tiles * H * kD * kD;
    A.Hst = (float *)p;
    p += al(st);
    A.dHst = (float *)p;
    p += al(st);
    A.Dst = (float *)p;
    A.p = plan;
    A.H = H;
    A.b = b;
    cudaError_t err = per_channel ? launch_chunk_bwd_t<true>(A, max_tiles) : launch_chunk_bwd_t<false>(A, max_tiles);
    if (err != cudaSuccess) return err;
    const int64_t chains = (int64_t)plan.N * H;
    if (chains > 0x7fffffff) return cudaErrorInvalidValue;
    {
        ProfScope prof(stream, "bwd_fwd_chain_kernel");
        if (per_channel)
            bwd_fwd_chain_kernel<true><<<(unsigned)chains, kThreads, sizeof(float) * kF_total, stream>>>(A);
        else
            bwd_fwd_chain_kernel<false><<<(unsigned)chains, kThreads, sizeof(float) * kF_total, stream>>>(A);
        count_launch();
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    {
        ProfScope prof(stream, "bwd_adj_chain_kernel");
        if (per_channel)
            bwd_adj_chain_kernel<true><<<(unsigned)chains, kThreads, sizeof(float) * kA_total, stream>>>(A);
        else
            bwd_adj_chain_kernel<false><<<(unsigned)chains, kThreads, sizeof(float) * kA_total, stream>>>(A);
        count_launch();
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if (max_tiles > 0) {
        ProfScope prof(stream, "bwd_tile_kernel");
        const dim3 grid((unsigned)max_tiles, (unsigned)H);
        if (per_channel)
            bwd_tile_kernel<true><<<grid, kThreads, sizeof(float) * kG_total, stream>>>(A);
        else
            bwd_tile_kernel<false><<<grid, kThreads, sizeof(float) * kG_total, stream>>>(A);
        count_launch();
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace gdr
