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
//   bwd_fwd_chain_kernel  per (segment, head): the state chain (state in registers);
//                         stores H0 and D of every tile (tc_fwd_chain_kernel in
//                         gdr_tc_fwd_chain.cu is the same chain on tcgen05)
//   bwd_adj_chain_kernel  per (segment, head), tiles in reverse: the dH chain (state in
//                         shared memory); stores X = diag(e^{G_C}) dH1 of every tile, and dh0
//                         (tc_adj_kernel in gdr_tc_adj.cu is the same chain on tcgen05)
//   bwd_tile_kernel       per (tile, head), all tiles at once: every input gradient
// The scalar-gate form is the per-channel form with every channel's gate equal.
//
// The two chains run in segments of S tiles (the plan's seg_chunks: 64 to 256,
// longer when enough (segment, head) blocks remain), one block per (segment, head), each
// started at a warm-up tile whose neglected transition is provably below 2^-64:
// the forward chain from a zero state some tiles before its segment, the adjoint
// chain from a zero gradient some tiles after it.  Both transitions have norm at
// most prod_t max(1, |1 - beta_t |k_t|^2|) max_d alpha_{t,d} (the adjoint one is
// the transpose), summed in log form per tile by bwd_bound_kernel.  A (sequence,
// head) pair without such a warm-up within 4 S tiles of every segment
// boundary runs as one block, as without segments (bwd_decide_kernel).
// The stored states are bf16 (they only feed the per-tile products).
#include <cstdlib>

#include "gdr_bwd_chunk.cuh"
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
constexpr int kSegMin = 64, kSegMax = 256;   // segment lengths in tiles
constexpr int kWarmFactor = 4;   // longest warm-up, in segments
constexpr int kLdh = 136;               // row stride (elements) of the bf16 state in shared memory
// row stride of the per-tile kernel's fp32 [16][.] buffers: 8 mod 32 words, so that its
// k-permuted fragment loads (8 bytes per lane) meet no bank conflict
constexpr int kLt = 136;
constexpr int kTileT = kT * kLt;

using bwdc::BcArgs;
using bwdc::kHorizonLog;
using bwdc::segment_of;
using bwdc::warm_walk;



// Staging of one tile over all 256 threads: lanes 2d and 2d + 1 of a warp take key
// channel d (and column d of the 128-wide input `other`, V or dO), tokens 0-7 and 8-15;
// the second half gets the first half's cumulative log-decay from its neighbour lane.
// stage_fetch issues every global load of the tile into registers; stage_compute
// writes the factored rows, G (if Gb), e^{G_C} per channel and beta.
struct StageRegs {
    __nv_bfloat16 ra[8], rk[8], rq[8], ro[8];
    float bt;
};

template <bool VEC>
__device__ __forceinline__ void stage_fetch(const BcArgs &A, int64_t t0, int len, int h, bool with_q,
                                            const __nv_bfloat16 *other, StageRegs &R) {
    const int tid = threadIdx.x;
    const int d = tid >> 1, i0 = 8 * (tid & 1);
#pragma unroll
    for (int u = 0; u < 8; ++u)
        if (i0 + u < len) {
            const int64_t row = (t0 + i0 + u) * A.H + h;
            R.ra[u] = VEC ? A.a[row * kD + d] : A.a[row];
            R.rk[u] = A.k[row * kD + d];
            if (with_q) R.rq[u] = A.q[row * kD + d];
            if (other) R.ro[u] = other[row * kD + d];
        }
    R.bt = tid < len ? __bfloat162float(A.beta[(t0 + tid) * A.H + h]) : 0.f;
}

template <int LD = kLd>
__device__ __forceinline__ void stage_compute(const BcArgs &A, int len, const StageRegs &R, float *Kt,
                                              float *Kh, float *Qt, float *Gb, float *eg, bool has_other,
                                              float *Ob, float *bs) {
    const int tid = threadIdx.x;
    const int d = tid >> 1, half = tid & 1, i0 = 8 * half;
    float gl[8], G = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        gl[u] = i0 + u < len ? gate_logdecay(__bfloat162float(R.ra[u]), A.b, GDR_GATE_BOUNDED) : 0.f;
        G += gl[u];
    }
    const float Gfirst = __shfl_xor_sync(0xffffffffu, G, 1);
    G = half ? Gfirst : 0.f;
    float eGC = 1.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int i = i0 + u;
        float kt = 0.f, kh = 0.f, qt = 0.f, gg = 0.f, ov = 0.f;
        if (i < len) {
            G += gl[u];
            const float e = expf(G), en = expf(-G), kd = __bfloat162float(R.rk[u]);
            kt = kd * e;
            kh = kd * en;
            if (Qt) qt = __bfloat162float(R.rq[u]) * e;
            if (has_other) ov = __bfloat162float(R.ro[u]);
            eGC = e;
            gg = G;
        }
        Kt[i * LD + d] = kt;
        Kh[i * LD + d] = kh;
        if (Qt) Qt[i * LD + d] = qt;
        if (Gb) Gb[i * LD + d] = gg;
        Ob[i * LD + d] = ov;
    }
    const float eo = __shfl_xor_sync(0xffffffffu, eGC, 1);
    if (half == 0) eg[d] = len > 8 ? eo : eGC;
    if (tid < kT) bs[tid] = R.bt;
}

// The same staging with the raw values packed two bf16 per register (for a kernel
// whose state takes most of its registers).
struct StageRegsPacked {
    uint32_t pa[4], pk[4], pq[4], po[4];   // two bf16 per register: tokens i0 + 2m, i0 + 2m + 1
    float bt;
};

__device__ __forceinline__ float bf_half(uint32_t x, int u) {
    return __uint_as_float(u ? (x & 0xffff0000u) : (x << 16));
}

template <bool VEC>
__device__ __forceinline__ void stage_fetch_packed(const BcArgs &A, int64_t t0, int len, int h, bool with_q,
                                            const __nv_bfloat16 *other, StageRegsPacked &R) {
    const int tid = threadIdx.x;
    const int d = tid >> 1, i0 = 8 * (tid & 1);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        uint32_t xa = 0, xk = 0, xq = 0, xo = 0;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = i0 + 2 * m + u;
            if (i < len) {
                const int64_t row = (t0 + i) * A.H + h;
                xa |= (uint32_t)__bfloat16_as_ushort(VEC ? A.a[row * kD + d] : A.a[row]) << (16 * u);
                xk |= (uint32_t)__bfloat16_as_ushort(A.k[row * kD + d]) << (16 * u);
                if (with_q) xq |= (uint32_t)__bfloat16_as_ushort(A.q[row * kD + d]) << (16 * u);
                if (other) xo |= (uint32_t)__bfloat16_as_ushort(other[row * kD + d]) << (16 * u);
            }
        }
        R.pa[m] = xa;
        R.pk[m] = xk;
        R.pq[m] = xq;
        R.po[m] = xo;
    }
    R.bt = tid < len ? __bfloat162float(A.beta[(t0 + tid) * A.H + h]) : 0.f;
}

__device__ __forceinline__ void stage_compute_packed(const BcArgs &A, int len, const StageRegsPacked &R, float *Kt,
                                              float *Kh, float *Qt, float *Gb, float *eg, bool has_other,
                                              float *Ob, float *bs) {
    const int tid = threadIdx.x;
    const int d = tid >> 1, half = tid & 1, i0 = 8 * half;
    float gl[8], G = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        gl[u] = i0 + u < len ? gate_logdecay(bf_half(R.pa[u >> 1], u & 1), A.b, GDR_GATE_BOUNDED) : 0.f;
        G += gl[u];
    }
    const float Gfirst = __shfl_xor_sync(0xffffffffu, G, 1);
    G = half ? Gfirst : 0.f;
    float eGC = 1.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int i = i0 + u;
        float kt = 0.f, kh = 0.f, qt = 0.f, gg = 0.f, ov = 0.f;
        if (i < len) {
            G += gl[u];
            const float e = expf(G), en = expf(-G), kd = bf_half(R.pk[u >> 1], u & 1);
            kt = kd * e;
            kh = kd * en;
            if (Qt) qt = bf_half(R.pq[u >> 1], u & 1) * e;
            if (has_other) ov = bf_half(R.po[u >> 1], u & 1);
            eGC = e;
            gg = G;
        }
        Kt[i * kLd + d] = kt;
        Kh[i * kLd + d] = kh;
        if (Qt) Qt[i * kLd + d] = qt;
        if (Gb) Gb[i * kLd + d] = gg;
        Ob[i * kLd + d] = ov;
    }
    const float eo = __shfl_xor_sync(0xffffffffu, eGC, 1);
    if (half == 0) eg[d] = len > 8 ? eo : eGC;
    if (tid < kT) bs[tid] = R.bt;
}

template <bool VEC>
__device__ __forceinline__ void stage_tile(const BcArgs &A, int64_t t0, int len, int h, float *Kt,
                                           float *Kh, float *Qt, float *Gb, float *eg,
                                           const __nv_bfloat16 *other, float *Ob, float *bs) {
    StageRegs R;
    stage_fetch<VEC>(A, t0, len, h, Qt != nullptr, other, R);
    stage_compute(A, len, R, Kt, Kh, Qt, Gb, eg, other != nullptr, Ob, bs);
}

// 16 x 16 product X Y^T over K = 128 (one 8-column half of the output per warp):
// out[i][j] for j in j0..j0+7.
template <int LD = kLd>
__device__ __forceinline__ void gram_half(float (&acc)[4], const float *X, const float *Y, int j0,
                                          int g, int t) {
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll 4
    for (int k0 = 0; k0 < kD; k0 += 8) {
        uint32_t af[4], b0, b1;
        if constexpr (LD % 32 == 8) {
            load_a_kp(af, X, LD, 0, k0, g, t);
            load_bt_kp(b0, b1, Y, LD, k0, j0, g, t);
        } else {
            load_a(af, X, LD, 0, k0, g, t);
            load_bt(b0, b1, Y, LD, k0, j0, g, t);
        }
        mma8(acc, af, b0, b1);
    }
}

// Forward substitution x = (I + A)^{-1} diag(beta) y on one column of a [16][kLd]
// buffer, in place (A strictly lower, row stride kPd).
template <int LD = kLd>
__device__ __forceinline__ void fwd_subst(float *X, int col, const float *Am, const float *bs) {
    float x[kT];
#pragma unroll
    for (int i = 0; i < kT; ++i) {
        float acc = bs[i] * X[i * LD + col];
#pragma unroll
        for (int j = 0; j < i; ++j) acc = fmaf(-Am[i * kPd + j], x[j], acc);
        x[i] = acc;
    }
#pragma unroll
    for (int i = 0; i < kT; ++i) X[i * LD + col] = x[i];
}

// Back substitution y = (I + A)^{-T} x on one column, from src into dst.
template <int LD = kLd>
__device__ __forceinline__ void back_subst(const float *src, float *dst, int col, const float *Am) {
    float y[kT];
#pragma unroll
    for (int i = kT - 1; i >= 0; --i) {
        float acc = src[i * LD + col];
#pragma unroll
        for (int j = i + 1; j < kT; ++j) acc = fmaf(-Am[j * kPd + i], y[j], acc);
        y[i] = acc;
    }
#pragma unroll
    for (int i = 0; i < kT; ++i) dst[i * LD + col] = y[i];
}

// A = beta (.) strict_lower(Kt Kh^T) into Am (warps 0-1 call this)
template <int LD = kLd>
__device__ __forceinline__ void build_A(const float *Kt, const float *Kh, const float *bs, float *Am,
                                        float *KK, int half, int g, int t) {
    float acc[4];
    const int j0 = 8 * half;
    gram_half<LD>(acc, Kt, Kh, j0, g, t);
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
template <int LD = kLd>
__device__ __forceinline__ void build_lower(const float *X, const float *Y, float *M, int half, int g,
                                            int t) {
    float acc[4];
    const int j0 = 8 * half;
    gram_half<LD>(acc, X, Y, j0, g, t);
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

// bf16 copy of the fp32 state by threads [first, kThreads), row r scaled by rs[r]
__device__ __forceinline__ void copy_state_out_h(const float *Hs, __nv_bfloat16 *dst, const float *rs,
                                                 int first = 0) {
    if ((int)threadIdx.x < first) return;
    const int n = kThreads - first;
    for (int e = ((int)threadIdx.x - first) * 4; e < kD * kD; e += n * 4) {
        const int r = e >> 7, c = e & (kD - 1);
        float4 x = *(const float4 *)&Hs[r * kLd + c];
        const float sr = rs[r];
        x.x *= sr;
        x.y *= sr;
        x.z *= sr;
        x.w *= sr;
        __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
        uint2 u;
        u.x = *(uint32_t *)&lo;
        u.y = *(uint32_t *)&hi;
        *(uint2 *)&dst[e] = u;
    }
}

__device__ __forceinline__ void copy_state_in(float *Hs, const float *src) {
    for (int e = threadIdx.x * 4; e < kD * kD; e += kThreads * 4) {
        const int r = e >> 7, c = e & (kD - 1);
        *(float4 *)&Hs[r * kLd + c] = src ? *(const float4 *)&src[e] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Per (tile, head): sum over its tokens of max_d g_{t,d} + ln max(1, |1 - beta |k|^2|).
// One warp per (tile, head): lane l reads key channels 4l..4l+3 of every token (8-byte
// loads), and the 16 per-token partial sums (and gate minima) are reduced across the
// warp by halving exchanges (16 + 8 + 4 + 2 + 1 values), after which lane pair
// (2i, 2i + 1) holds token i's totals.
constexpr int kBoundWarps = 8;   // (tile, head) pairs per block

// v[0..15] summed (MIN: minimised) over the warp; token (lane >> 1)'s result in v[0]
template <bool MIN>
__device__ __forceinline__ void fold16(float (&v)[kT], int lane) {
#pragma unroll
    for (int w = kT / 2; w >= 1; w >>= 1) {
        const bool hi = (lane & (2 * w)) != 0;   // keeps the upper w of the 2w values
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float keep = hi ? v[j + w] : v[j], send = hi ? v[j] : v[j + w];
            const float r = __shfl_xor_sync(0xffffffffu, send, 2 * w);
            v[j] = MIN ? fminf(keep, r) : keep + r;
        }
    }
    const float r = __shfl_xor_sync(0xffffffffu, v[0], 1);
    v[0] = MIN ? fminf(v[0], r) : v[0] + r;
}

// four consecutive bf16 values: one 8-byte load when the tensors are 8-byte aligned
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, bool wide, float (&x)[4]) {
    if (wide) {
        const uint2 r = *(const uint2 *)p;
        const float2 lo = __bfloat1622float2(*(const __nv_bfloat162 *)&r.x);
        const float2 hi = __bfloat1622float2(*(const __nv_bfloat162 *)&r.y);
        x[0] = lo.x;
        x[1] = lo.y;
        x[2] = hi.x;
        x[3] = hi.y;
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = __bfloat162float(p[u]);
    }
}

template <bool VEC>
__global__ void __launch_bounds__(32 * kBoundWarps)
bwd_bound_kernel(const BcArgs A, float *lam, int64_t max_tiles, bool wide) {
    const int lane = threadIdx.x & 31;
    const int64_t c = (int64_t)blockIdx.x * kBoundWarps + (threadIdx.x >> 5);
    const int h = blockIdx.y;
    if (c >= max_tiles) return;
    const int n = find_owner(A.p.chunk_base, A.p.N, c);
    if (n < 0) return;
    const int64_t t0 = A.p.seq_start[n] + (c - A.p.chunk_base[n]) * kT;
    const int len = (int)min((int64_t)kT, A.p.seq_start[n + 1] - t0);
    float kk[kT], m[kT];
#pragma unroll
    for (int i = 0; i < kT; ++i) {
        kk[i] = 0.f;
        m[i] = 3.0e38f;
        if (i < len) {
            const int64_t row = (t0 + i) * A.H + h;
            float kv[4], av[4];
            load4(&A.k[row * kD + 4 * lane], wide, kv);
            kk[i] = kv[0] * kv[0] + kv[1] * kv[1] + kv[2] * kv[2] + kv[3] * kv[3];
            if (VEC) {
                load4(&A.a[row * kD + 4 * lane], wide, av);
                m[i] = fminf(fminf(av[0], av[1]), fminf(av[2], av[3]));
            }
        }
    }
    fold16<false>(kk, lane);
    if (VEC) fold16<true>(m, lane);
    const int i = lane >> 1;
    float x = 0.f;
    if ((lane & 1) == 0 && i < len) {
        const int64_t row = (t0 + i) * A.H + h;
        const float mi = VEC ? m[0] : __bfloat162float(A.a[row]);
        const float bt = __bfloat162float(A.beta[row]);
        x = gate_logdecay(mi, A.b, GDR_GATE_BOUNDED) + logf(fmaxf(1.f, fabsf(1.f - bt * kk[0])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) lam[c * A.H + h] = x;
}

// Per (sequence, head): 1 if every interior segment boundary has a bound <= e^-46
// within 4 S tiles on both sides (or the sequence's end within reach).
__global__ void __launch_bounds__(32)
bwd_decide_kernel(const float *__restrict__ lam, int *__restrict__ ok, Plan p, int H) {
    const int h = blockIdx.x % H, n = blockIdx.x / H;
    const int lane = threadIdx.x;
    const int64_t base = p.chunk_base[n], nt = p.chunk_base[n + 1] - base;
    int good = 1;
    const int seg = p.seg_chunks, max_warm = kWarmFactor * seg;
    for (int64_t B = seg; B < nt && good; B += seg) {
        float before = 0.f, after = 0.f;
        for (int i = lane; i < max_warm; i += 32) {
            if (B - 1 - i >= 0) before += lam[(base + B - 1 - i) * H + h];
            if (B + i < nt) after += lam[(base + B + i) * H + h];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            before += __shfl_xor_sync(0xffffffffu, before, o);
            after += __shfl_xor_sync(0xffffffffu, after, o);
        }
        good = (B <= max_warm || before <= kHorizonLog) && (B + max_warm >= nt || after <= kHorizonLog);
    }
    if (lane == 0) ok[(int64_t)n * H + h] = good;
}

// ---------------------------------------------------------------------------
// forward state chain: stores H0 and D of every tile
// ---------------------------------------------------------------------------
// The state is held in registers as transposed accumulator fragments (as in the
// per-channel forward): warp w owns value channels 16w..16w+15; hs[nd][u] = H[d][c]
// with c = c0 + g + 8 (u >> 1), d = 8 nd + 2t + (u & 1).  An 8-wide block of a
// thread's fragments is an A operand if the reduction order inside the block is
// (2t, 2t + 1) <-> slots (t, t + 4), and the shared-memory B operand is read in that
// order too.  Each tile's entering state goes out in bf16 through Hb, its D through
// Db, both written by the warps idle during the Gram products one step later.
constexpr int kF_Kt = 0, kF_Kh = kF_Kt + kTile2, kF_U = kF_Kh + kTile2, kF_D = kF_U + kTile2,
              kF_A = kF_D + kTile2, kF_eg = kF_A + kT * kPd, kF_b = kF_eg + kD,
              kF_Hb = kF_b + kT,                                   // bf16 [128][kLdh]
              kF_total = kF_Hb + kD * kLdh / 2;

template <bool VEC>
__global__ void __launch_bounds__(kThreads, 2)
bwd_fwd_chain_kernel(const BcArgs A) {
    extern __shared__ float sm[];
    float *Kt = sm + kF_Kt, *Kh = sm + kF_Kh, *Ub = sm + kF_U, *Db = sm + kF_D, *Am = sm + kF_A;
    float *eg = sm + kF_eg, *bs = sm + kF_b;
    __nv_bfloat16 *Hb = (__nv_bfloat16 *)(sm + kF_Hb);
    __shared__ int64_t first;
    const int h = blockIdx.x % A.H;
    int n;
    int64_t s0, s1;
    if (!segment_of(A, blockIdx.x / A.H, h, n, s0, s1)) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
    const int c0 = 16 * warp;
    const int64_t s = A.p.seq_start[n], e_end = A.p.seq_start[n + 1], tile0 = A.p.chunk_base[n];
    const int64_t ntiles = A.p.chunk_base[n + 1] - tile0;
    if (warp == 0) {
        const int64_t w = warm_walk(A.lam, tile0, ntiles, A.H, h, s0, -1);
        if (lane == 0) first = w;
    }
    __syncthreads();
    const int64_t w0 = first;
    const size_t sbase = ((size_t)n * A.H + h) * kD * kD;
    const bool from_h0 = w0 == 0 && A.h0;
    float hs[kD / 8][4];
#pragma unroll
    for (int nd = 0; nd < kD / 8; ++nd)
#pragma unroll
        for (int u = 0; u < 4; ++u)
            hs[nd][u] = from_h0 ? A.h0[sbase + (size_t)(8 * nd + 2 * t + (u & 1)) * kD + c0 + g + 8 * (u >> 1)] : 0.f;
    int64_t d_tile = -1;   // tile whose D waits in Db
    // bf16 state in Hb and D in Db go out as whole rows (threads [64, 256))
    auto copy_out = [&](int64_t c_state, int64_t c_d) {
        if (tid < 64) return;
        const int q = tid - 64;
        if (c_state >= 0) {
            __nv_bfloat16 *dst = A.Hst + ((size_t)c_state * A.H + h) * kD * kD;
            for (int e = q; e < kD * kD / 8; e += kThreads - 64) {
                const int r = e >> 4, c8 = e & 15;
                *(uint4 *)&dst[r * kD + 8 * c8] = *(const uint4 *)&Hb[r * kLdh + 8 * c8];
            }
        }
        if (c_d >= 0) {
            float *dst = A.Dst + ((size_t)c_d * A.H + h) * kT * kD;
            for (int e = q; e < kT * kD / 4; e += kThreads - 64) {
                const int i = e >> 5, c4 = e & 31;
                *(float4 *)&dst[i * kD + 4 * c4] = *(const float4 *)&Db[i * kLd + 4 * c4];
            }
        }
    };
    for (int64_t tt = w0; tt < s1; ++tt) {
        const int64_t t0 = s + tt * kT, c = tile0 + tt;
        const int len = (int)min((int64_t)kT, e_end - t0);
        const bool keep = tt >= s0;   // warm-up tiles only advance the state
        __syncthreads();
        {
            StageRegsPacked R;
            stage_fetch_packed<VEC>(A, t0, len, h, false, A.v, R);
            stage_compute_packed(A, len, R, Kt, Kh, nullptr, nullptr, eg, true, Ub, bs);
        }
        if (keep)
#pragma unroll
            for (int nd = 0; nd < kD / 8; ++nd)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    Hb[(8 * nd + 2 * t + (u & 1)) * kLdh + c0 + g + 8 * (u >> 1)] = __float2bfloat16_rn(hs[nd][u]);
        __syncthreads();
        if (warp < 2) build_A(Kt, Kh, bs, Am, nullptr, warp, g, t);
        else copy_out(keep ? c : -1, d_tile);
        __syncthreads();
        fwd_subst(tid < kD ? Kt : Ub, tid & (kD - 1), Am, bs);   // Kt -> W, V -> U
        if (tid < kD)
            for (int i = 0; i < kT; ++i) Kh[i * kLd + tid] *= eg[tid];   // Ke
        __syncthreads();
        // D^T = U^T - H^T W^T (this warp's value channels)
        float dt[2][4];   // (c, i = 8 it + 2t + (u & 1))
#pragma unroll
        for (int it = 0; it < 2; ++it)
#pragma unroll
            for (int u = 0; u < 4; ++u) dt[it][u] = Ub[(8 * it + 2 * t + (u & 1)) * kLd + c0 + g + 8 * (u >> 1)];
#pragma unroll
        for (int nd = 0; nd < kD / 8; ++nd) {
            const uint32_t ah[4] = {tf32(hs[nd][0]), tf32(hs[nd][2]), tf32(hs[nd][1]), tf32(hs[nd][3])};
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const float2 w2 = *(const float2 *)&Kt[(8 * it + g) * kLd + 8 * nd + 2 * t];
                mma8(dt[it], ah, tf32(-w2.x), tf32(-w2.y));
            }
        }
        if (keep) {
#pragma unroll
            for (int it = 0; it < 2; ++it)
#pragma unroll
                for (int u = 0; u < 4; ++u) Db[(8 * it + 2 * t + (u & 1)) * kLd + c0 + g + 8 * (u >> 1)] = dt[it][u];
            d_tile = c;
        } else {
            d_tile = -1;
        }
        // H1^T = H0^T diag(e^{G_C}) + D^T Ke
        uint32_t ad[2][4];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            ad[kk][0] = tf32(dt[kk][0]);
            ad[kk][1] = tf32(dt[kk][2]);
            ad[kk][2] = tf32(dt[kk][1]);
            ad[kk][3] = tf32(dt[kk][3]);
        }
#pragma unroll
        for (int nd = 0; nd < kD / 8; ++nd) {
            const float e0 = eg[8 * nd + 2 * t], e1 = eg[8 * nd + 2 * t + 1];
            hs[nd][0] *= e0;
            hs[nd][1] *= e1;
            hs[nd][2] *= e0;
            hs[nd][3] *= e1;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const uint32_t b0 = tf32(Kh[(8 * kk + 2 * t) * kLd + 8 * nd + g]);
                const uint32_t b1 = tf32(Kh[(8 * kk + 2 * t + 1) * kLd + 8 * nd + g]);
                mma8(hs[nd], ad[kk], b0, b1);
            }
        }
    }
    __syncthreads();
    copy_out(-1, d_tile);   // the last tile's D
}

// ---------------------------------------------------------------------------
// adjoint state chain, tiles in reverse: stores X = diag(e^{G_C}) dH1 of every tile, writes dh0
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
    __shared__ int64_t last;
    const int h = blockIdx.x % A.H;
    int n;
    int64_t s0, s1;
    if (!segment_of(A, blockIdx.x / A.H, h, n, s0, s1)) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
    const int c0 = 16 * warp;
    const int64_t s = A.p.seq_start[n], e_end = A.p.seq_start[n + 1], tile0 = A.p.chunk_base[n];
    const int64_t ntiles = A.p.chunk_base[n + 1] - tile0;
    if (warp == 0) {
        const int64_t e = warm_walk(A.lam, tile0, ntiles, A.H, h, s1, +1);
        if (lane == 0) last = e;
    }
    __syncthreads();
    const int64_t e0 = last;
    const size_t sbase = ((size_t)n * A.H + h) * kD * kD;
    copy_state_in(dH, (e0 == ntiles && A.dhT) ? A.dhT + sbase : nullptr);
    for (int64_t tt = e0 - 1; tt >= s0; --tt) {
        const int64_t t0 = s + tt * kT, c = tile0 + tt;
        const int len = (int)min((int64_t)kT, e_end - t0);
        __syncthreads();
        stage_tile<VEC>(A, t0, len, h, Kt, Kh, Qt, nullptr, eg, A.dout, Ob, bs);
        __syncthreads();
        if (warp < 2) build_A(Kt, Kh, bs, Am, nullptr, warp, g, t);
        else if (warp < 4) build_lower(Qt, Kh, Sm, warp - 2, g, t);
        else if (tt < s1) copy_state_out_h(dH, A.dHst + ((size_t)c * A.H + h) * kD * kD, eg, 128);   // X
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
        if (tt < s1) {   // dD of the segment's tiles for the tile kernel (this warp's columns)
            const int i = lane >> 1, cc = c0 + 8 * (lane & 1);
            float *dst = A.dDst + ((size_t)c * A.H + h) * kT * kD + (size_t)i * kD + cc;
            *(float4 *)dst = *(const float4 *)&Eb[i * kLd + cc];
            *(float4 *)(dst + 4) = *(const float4 *)&Eb[i * kLd + cc + 4];
        }
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
    if (A.dh0 && s0 == 0) copy_state_out(dH, A.dh0 + sbase);
}

// ---------------------------------------------------------------------------
// per-tile gradients.  Buffers are reused by lifetime:
//   Ob: dO, then dG        Db: D, then dW, then dYw     Eb: dD, then dYu
//   Ub: V, then U          Wb: W                        Sh: dH1, then H0 (bf16)
// ---------------------------------------------------------------------------
template <bool VEC> struct TileLayout {
    static constexpr int kt = 0, kh = kt + kTileT, qt = kh + kTileT, ob = qt + kTileT,
                         db = ob + kTileT, ub = db + kTileT, wb = ub + kTileT, eb = wb + kTileT,
                         am = eb + kTileT, kk = am + kT * kPd,
                         ds = kk + kT * kPd, da = ds + kT * kPd, bda = da + kT * kPd,
                         eg = bda + kT * kPd, rg = eg + kD, bs = rg + kD, rs = bs + kT,
                         gb = rs + 4 * kT + kT, egt = gb + 2 * kT, dgp = egt + 2 * kT,
                         sh = dgp + 8 * kT, total_f = sh;
    static constexpr size_t bytes = sizeof(float) * total_f + sizeof(__nv_bfloat16) * kD * kLdh;
};

template <bool VEC>
__global__ void __launch_bounds__(kThreads)
bwd_tile_kernel(const BcArgs A) {
    using L = TileLayout<VEC>;
    extern __shared__ float sm[];
    float *Kt = sm + L::kt, *Kh = sm + L::kh, *Qt = sm + L::qt, *Ob = sm + L::ob, *Db = sm + L::db;
    float *Ub = sm + L::ub, *Wb = sm + L::wb, *Eb = sm + L::eb;
    float *Am = sm + L::am, *KK = sm + L::kk, *dS = sm + L::ds, *dA = sm + L::da;
    float *bdA = sm + L::bda, *eg = sm + L::eg, *rG = sm + L::rg, *bs = sm + L::bs, *rowsum = sm + L::rs;
    float *Gb = sm + L::gb;
    float *eGt = sm + L::egt;   // scalar gate: e^{G_i}, then e^{-G_i}, per token
    float *dGp = sm + L::dgp;   // scalar gate: per (warp, token) partial sums of dG
    __nv_bfloat16 *Sh = (__nv_bfloat16 *)(sm + L::sh);
    const int64_t c = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
    const int c0 = 16 * warp;
    const size_t st = ((size_t)c * A.H + h) * kD * kD;
    // this tile's H0 goes to L2 now (one 128-byte line per thread): the row sums below
    // and its copy into shared memory then wait on L2 rather than HBM
    asm volatile("prefetch.global.L2 [%0];" ::"l"(A.Hst + st + threadIdx.x * 64));
    // a bf16 state into Sh and, asynchronously, without registers
    auto stage_state = [&](const __nv_bfloat16 *src) {
#pragma unroll
        for (int e = tid * 8; e < kD * kD; e += kThreads * 8) {
            const int r = e >> 7, col = e & (kD - 1);
            cp_async16(&Sh[r * kLdh + col], &src[e]);
        }
    };
    // ---- stage: X, D and dD by asynchronous copies, then the factored rows, G, dO, V
    stage_state(A.dHst + st);
    {
        const float *Dg = A.Dst + ((size_t)c * A.H + h) * kT * kD;
        const float *dDg = A.dDst + ((size_t)c * A.H + h) * kT * kD;
#pragma unroll
        for (int e = tid * 4; e < kT * kD; e += kThreads * 4) {
            const int i = e >> 7, col = e & (kD - 1);
            cp_async16(&Db[i * kLt + col], &Dg[e]);
            cp_async16(&Eb[i * kLt + col], &dDg[e]);
        }
    }
    cp_async_commit();
    // the tile's sequence and tokens (its copies above need only the tile index); a block
    // past the last tile leaves once its own copies have landed
    const int n = find_owner(A.p.chunk_base, A.p.N, c);
    if (n < 0) {
        cp_async_wait_all();
        return;
    }
    const int64_t t0 = A.p.seq_start[n] + (c - A.p.chunk_base[n]) * kT;
    const int len = (int)min((int64_t)kT, A.p.seq_start[n + 1] - t0);
    // per-channel gate: the raw inputs of this thread's (channel, 8 tokens) stay packed in
    // registers, and G is formed again from them once V's buffer is free (see below),
    // so that no [16][128] G buffer holds shared memory through the tile
    uint32_t ra_keep[kT / 4] = {};
    // V, kept in registers for the dV / dbeta pass (same element per thread there), and
    // the scalar gate's inputs: loaded with the tile's other inputs, before any is used
    __nv_bfloat16 rv[kT / 2];   // per-channel gate: V by (channel, token pair)
    uint4 rv8 = make_uint4(0, 0, 0, 0);   // scalar gate: V by (token, 8 channels)
    if constexpr (VEC) {
        StageRegs R;
        stage_fetch<VEC>(A, t0, len, h, true, A.dout, R);
#pragma unroll
        for (int m = 0; m < kT / 2; ++m) {
            const int i = (tid >> 7) + 2 * m, col = tid & (kD - 1);
            rv[m] = i < len ? A.v[((t0 + i) * A.H + h) * kD + col] : __float2bfloat16_rn(0.f);
        }
        stage_compute<kLt>(A, len, R, Kt, Kh, Qt, nullptr, eg, A.dout != nullptr, Ob, bs);
#pragma unroll
        for (int m = 0; m < kT / 4; ++m)
            ra_keep[m] = (uint32_t)__bfloat16_as_ushort(R.ra[2 * m]) |
                         ((uint32_t)__bfloat16_as_ushort(R.ra[2 * m + 1]) << 16);
#pragma unroll
        for (int m = 0; m < kT / 2; ++m) {
            const int i = (tid >> 7) + 2 * m, col = tid & (kD - 1);
            Ub[i * kLt + col] = __bfloat162float(rv[m]);
        }
    } else {
        // thread (token si, channels 8 sch .. 8 sch + 7): one 16-byte load per tensor; the
        // gate of the tile's 16 tokens is formed in every warp (lanes 0..15), G by an
        // inclusive prefix sum over the lanes
        const int si = tid >> 4, sch = tid & 15;
        uint4 rq = make_uint4(0, 0, 0, 0), rk = rq, rdo = rq;
        float a_l = 0.f, b_l = 0.f;
        if (si < len) {
            const int64_t off = ((t0 + si) * A.H + h) * kD + 8 * sch;
            rq = *(const uint4 *)(A.q + off);
            rk = *(const uint4 *)(A.k + off);
            if (A.dout) rdo = *(const uint4 *)(A.dout + off);   // NULL: zero
            rv8 = *(const uint4 *)(A.v + off);
        }
        if (lane < len) {
            const int64_t row = (t0 + lane) * A.H + h;
            a_l = __bfloat162float(A.a[row]);
            b_l = __bfloat162float(A.beta[row]);
        }
        float G_l = lane < len ? gate_logdecay(a_l, A.b, GDR_GATE_BOUNDED) : 0.f;
#pragma unroll
        for (int o = 1; o < kT; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, G_l, o);
            if (lane >= o) G_l += y;
        }
        const float Gi = __shfl_sync(0xffffffffu, G_l, si & (kT - 1));
        const float GC = __shfl_sync(0xffffffffu, G_l, kT - 1);   // lanes past the end add 0
        const float bi = __shfl_sync(0xffffffffu, b_l, si & (kT - 1));
        const float e = expf(Gi), en = expf(-Gi);
        const uint32_t wq[4] = {rq.x, rq.y, rq.z, rq.w}, wk[4] = {rk.x, rk.y, rk.z, rk.w};
        const uint32_t wo[4] = {rdo.x, rdo.y, rdo.z, rdo.w}, wv[4] = {rv8.x, rv8.y, rv8.z, rv8.w};
        float kt[8], kh[8], qt[8], ob[8], ub[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float kd = bf_half(wk[u >> 1], u & 1);
            kt[u] = kd * e;
            kh[u] = kd * en;
            qt[u] = bf_half(wq[u >> 1], u & 1) * e;
            ob[u] = bf_half(wo[u >> 1], u & 1);
            ub[u] = bf_half(wv[u >> 1], u & 1);
        }
        const int so = si * kLt + 8 * sch;
        *(float4 *)&Kt[so] = make_float4(kt[0], kt[1], kt[2], kt[3]);
        *(float4 *)&Kt[so + 4] = make_float4(kt[4], kt[5], kt[6], kt[7]);
        *(float4 *)&Kh[so] = make_float4(kh[0], kh[1], kh[2], kh[3]);
        *(float4 *)&Kh[so + 4] = make_float4(kh[4], kh[5], kh[6], kh[7]);
        *(float4 *)&Qt[so] = make_float4(qt[0], qt[1], qt[2], qt[3]);
        *(float4 *)&Qt[so + 4] = make_float4(qt[4], qt[5], qt[6], qt[7]);
        *(float4 *)&Ob[so] = make_float4(ob[0], ob[1], ob[2], ob[3]);
        *(float4 *)&Ob[so + 4] = make_float4(ob[4], ob[5], ob[6], ob[7]);
        *(float4 *)&Ub[so] = make_float4(ub[0], ub[1], ub[2], ub[3]);
        *(float4 *)&Ub[so + 4] = make_float4(ub[4], ub[5], ub[6], ub[7]);
        if (si == 0) {
            const float eGC = expf(GC);
            *(float4 *)&eg[8 * sch] = make_float4(eGC, eGC, eGC, eGC);
            *(float4 *)&eg[8 * sch + 4] = make_float4(eGC, eGC, eGC, eGC);
        }
        if (sch == 0) bs[si] = si < len ? bi : 0.f;
        if (warp == kThreads / 32 - 1 && lane < kT) {
            // g and g'(a) per token for the outputs and da (the cumsum follows the barrier)
            float gi = 0.f, dgi = 0.f;
            if (lane < len) {
                const float sg = 1.f / (1.f + expf(-a_l));
                gi = -A.b * sg;
                dgi = -A.b * sg * (1.f - sg);
            }
            Gb[lane] = gi;
            Gb[kT + lane] = dgi;
        }
    }
    cp_async_wait_all();
    __syncthreads();
    // ---- dKe (.) e^{G_C} = D X^T (this warp's dk columns), then the 16 x 16 products
    // (dD = S^T dO + Kh X comes from the adjoint chain, which forms it for its own step)
    // this warp's H0 rows for the row sums below, loaded first so that the product's
    // time covers their latency
    const __nv_bfloat16 *H0g = A.Hst + st;
    uint2 xh[kD / 8];
#pragma unroll
    for (int m = 0; m < kD / 8; ++m) xh[m] = *(const uint2 *)&H0g[(warp + 8 * m) * kD + 4 * lane];
    float dke[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u) dke[nt][u] = 0.f;
#pragma unroll 2
    for (int k0 = 0; k0 < kD; k0 += 8) {
        uint32_t ad[4];
        load_a_kp(ad, Db, kLt, 0, k0, g, t);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            uint32_t b0, b1;
            load_bt_h_kp(b0, b1, Sh, kLdh, k0, c0 + 8 * nt, g, t);   // X^T[k][d] = X[d][k]
            mma8(dke[nt], ad, b0, b1);
        }
    }
    // e^{G_C} rowsum(dH1 (.) H0) = rowsum(X (.) H0): X from shared memory, H0 rows from
    // the stored copy
    {
        // this lane's part of the 16 rows (warp + 8 m), then one halving reduction over the
        // warp for all of them: lane pair (2m, 2m + 1) ends with row warp + 8 m
        float pr[kT];
#pragma unroll
        for (int m = 0; m < kD / 8; ++m) {
            const int r = warp + 8 * m;
            const uint2 yh = *(const uint2 *)&Sh[r * kLdh + 4 * lane];
            const __nv_bfloat162 *x2 = (const __nv_bfloat162 *)&xh[m], *y2 = (const __nv_bfloat162 *)&yh;
            const float2 xa = __bfloat1622float2(x2[0]), xb = __bfloat1622float2(x2[1]);
            const float2 ya = __bfloat1622float2(y2[0]), yb = __bfloat1622float2(y2[1]);
            pr[m] = xa.x * ya.x + xa.y * ya.y + xb.x * yb.x + xb.y * yb.y;
        }
        fold16<false>(pr, lane);
        if ((lane & 1) == 0) rG[warp + 8 * (lane >> 1)] = pr[0];
    }
    if (warp < 2) build_A<kLt>(Kt, Kh, bs, Am, KK, warp, g, t);
    else if (warp < 4) build_lower<kLt>(Ob, Db, dS, warp - 2, g, t);   // dS = lower(dO D^T)
    else if (!VEC && warp == 7) {
        // in-tile inclusive cumsum of g (lanes 0..15), in place
        float x = lane < kT ? Gb[lane] : 0.f;
#pragma unroll
        for (int o = 1; o < kT; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane < kT) {
            Gb[lane] = x;
            eGt[lane] = expf(x);
            eGt[kT + lane] = expf(-x);
        }
    }
    if (tid < kD)
        for (int i = 0; i < kT; ++i) Wb[i * kLt + tid] = Kt[i * kLt + tid];
    __syncthreads();
    // ---- H0 into the state buffer (asynchronous: dH1 is no longer needed)
    stage_state(A.Hst + st);
    cp_async_commit();
    // ---- W and U
    fwd_subst<kLt>(tid < kD ? Wb : Ub, tid & (kD - 1), Am, bs);
    cp_async_wait_all();   // H0 landed (own copies); the barrier publishes them
    __syncthreads();
    // ---- dQt_a = dO H0^T and dW = -dD H0^T (this warp's dk columns); dW into Db
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
            load_a_kp(ao, Ob, kLt, 0, k0, g, t);
            load_a_kp(ae, Eb, kLt, 0, k0, g, t);
#pragma unroll
            for (int u = 0; u < 4; ++u) ae[u] ^= 0x80000000u;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t b0, b1;
                load_bt_h_kp(b0, b1, Sh, kLdh, k0, c0 + 8 * nt, g, t);   // H0^T[k][d] = H0[d][k]
                mma8(dq[nt], ao, b0, b1);
                mma8(dw[nt], ae, b0, b1);
            }
        }
        // D's last readers (dS and dKe) finished two barriers ago: dW can take its place
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int col = c0 + 8 * nt + 2 * t;
            *(float2 *)&Db[g * kLt + col] = make_float2(dw[nt][0], dw[nt][1]);
            *(float2 *)&Db[(g + 8) * kLt + col] = make_float2(dw[nt][2], dw[nt][3]);
        }
    }
    __syncthreads();
    // ---- dYw = T^T dW in place (dk columns, threads 0..127); dYu = T^T dD in place
    back_subst<kLt>(tid < kD ? Db : Eb, tid < kD ? Db : Eb, tid & (kD - 1), Am);
    __syncthreads();
    // ---- dA = -strict_lower(dYu U^T + dYw W^T) (warps 0-1); dV = diag(beta) dYu
    if (warp < 2) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};   // two chains
        const int j0 = 8 * warp;
#pragma unroll 4
        for (int k0 = 0; k0 < kD; k0 += 8) {
            uint32_t af[4], b0, b1;
            load_a_kp(af, Eb, kLt, 0, k0, g, t);
            load_bt_kp(b0, b1, Ub, kLt, k0, j0, g, t);
            mma8(acc, af, b0, b1);
            load_a_kp(af, Db, kLt, 0, k0, g, t);
            load_bt_kp(b0, b1, Wb, kLt, k0, j0, g, t);
            mma8(acc2, af, b0, b1);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] += acc2[u];
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
    // dV = diag(beta) dYu, and the per-token sums dYu . V + dYw . Kt for dbeta: the
    // scalar gate's staging thread (token i, 8 channels), a 16-byte store of dV each
    if constexpr (!VEC) {
        const int i = tid >> 4, ch = tid & 15;
        float x = 0.f;
        if (i < len) {
            const int so = i * kLt + 8 * ch;
            const float4 y0 = *(const float4 *)&Eb[so], y1 = *(const float4 *)&Eb[so + 4];
            const float4 d0 = *(const float4 *)&Db[so], d1 = *(const float4 *)&Db[so + 4];
            const float4 k0 = *(const float4 *)&Kt[so], k1 = *(const float4 *)&Kt[so + 4];
            const float yu[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
            const float dw[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
            const float kt[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
            const uint32_t wv[4] = {rv8.x, rv8.y, rv8.z, rv8.w};
            const float bi = bs[i];
            uint32_t pv[4];
#pragma unroll
            for (int u = 0; u < 8; ++u) x = fmaf(yu[u], bf_half(wv[u >> 1], u & 1), fmaf(dw[u], kt[u], x));
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                __nv_bfloat162 v2 = __floats2bfloat162_rn(bi * yu[2 * m], bi * yu[2 * m + 1]);
                pv[m] = *reinterpret_cast<uint32_t *>(&v2);
            }
            *(uint4 *)(A.dv + ((t0 + i) * A.H + h) * kD + 8 * ch) = make_uint4(pv[0], pv[1], pv[2], pv[3]);
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);   // the 16 lanes of token i
        if (ch == 0) {
            rowsum[i * 4] = x;
            rowsum[i * 4 + 1] = rowsum[i * 4 + 2] = rowsum[i * 4 + 3] = 0.f;
        }
    } else {
        const int col = tid & (kD - 1), half = tid >> 7;
        float x[kT / 2];
#pragma unroll
        for (int m = 0; m < kT / 2; ++m) {
            const int i = half + 2 * m;
            x[m] = 0.f;
            if (i < len) {
                const int64_t r = ((t0 + i) * A.H + h) * kD + col;
                const float yu = Eb[i * kLt + col];
                A.dv[r] = __float2bfloat16_rn(bs[i] * yu);
                x[m] = fmaf(yu, __bfloat162float(rv[m]), Db[i * kLt + col] * Kt[i * kLt + col]);
            }
        }
        // the 8 row sums by one halving exchange: row half + 2 ((lane >> 1) & 7) in x[0]
        // of the lanes with bits 0 and 4 clear
#pragma unroll
        for (int w = kT / 4; w >= 1; w >>= 1) {
            const bool hi = (lane & (2 * w)) != 0;
#pragma unroll
            for (int j = 0; j < w; ++j) {
                const float keep = hi ? x[j + w] : x[j], send = hi ? x[j] : x[j + w];
                x[j] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * w);
            }
        }
        x[0] += __shfl_xor_sync(0xffffffffu, x[0], 1);
        x[0] += __shfl_xor_sync(0xffffffffu, x[0], 16);
        if ((lane & 17) == 0) rowsum[(half + 2 * ((lane >> 1) & 7)) * 4 + (warp & 3)] = x[0];   // 4 warps per half
    }
    __syncthreads();
    // ---- per-channel gate: G again, into V's buffer (its last reader was dA, above), in
    // the staging's order (lane pair (2d, 2d + 1): channel d, tokens 0-7 and 8-15)
    float *Gv = VEC ? Ub : Gb;
    if (VEC) {
        const int d = tid >> 1, half = tid & 1, i0 = 8 * half;
        float gl[8], G = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            gl[u] = i0 + u < len ? gate_logdecay(bf_half(ra_keep[u >> 1], u & 1), A.b, GDR_GATE_BOUNDED) : 0.f;
            G += gl[u];
        }
        const float Gfirst = __shfl_xor_sync(0xffffffffu, G, 1);
        G = half ? Gfirst : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u;
            float gg = 0.f;
            if (i < len) {
                G += gl[u];
                gg = G;
            }
            Ub[i * kLt + d] = gg;
        }
    }
    // ---- dKt, dKh, dQt on this warp's dk columns; dG into Ob
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
                load_b(bh0, bh1, Kh, kLt, 8 * ks, c0 + 8 * nt, g, t);
                load_b(bt0, bt1, Kt, kLt, 8 * ks, c0 + 8 * nt, g, t);
                load_b(bq0, bq1, Qt, kLt, 8 * ks, c0 + 8 * nt, g, t);
                mma8(dkt[nt], a_bdA, bh0, bh1);    // (beta dA) Kh
                mma8(dkh[nt], a_bdAt, bt0, bt1);   // (beta dA)^T Kt
                mma8(dkh[nt], a_dSt, bq0, bq1);    // dS^T Qt
                mma8(dq[nt], a_dS, bh0, bh1);      // dS Kh
            }
        }
        if (VEC) __syncthreads();   // G (written above by other threads) is complete
        float pg[2] = {0.f, 0.f};   // scalar gate: this thread's part of dG's row sums (rows g, g + 8)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {   // the pair (u, u + 1) = columns (d, d + 1) of row i
                const int i = g + 8 * hr, d = c0 + 8 * nt + 2 * t;
                const float2 kt2 = *(const float2 *)&Kt[i * kLt + d], kh2 = *(const float2 *)&Kh[i * kLt + d];
                const float2 qt2 = *(const float2 *)&Qt[i * kLt + d], dw2 = *(const float2 *)&Db[i * kLt + d];
                float oq[2], ok[2];
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int u = 2 * hr + w, dd = d + w;
                    const float kt = w ? kt2.y : kt2.x, kh = w ? kh2.y : kh2.x, qt = w ? qt2.y : qt2.x;
                    const float dKt = dkt[nt][u] + bs[i] * (w ? dw2.y : dw2.x);
                    const float dKh = dkh[nt][u] + dke[nt][u];   // dke = D X^T = dKe (.) e^{G_C}
                    const float dG = dq[nt][u] * qt + dKt * kt - dKh * kh;
                    if constexpr (VEC) Ob[i * kLt + dd] = dG;
                    else pg[hr] += dG;
                    // e^G and e^-G: per (token, channel), or per token from the table (scalar gate)
                    const float ep = VEC ? expf(Gv[i * kLt + dd]) : eGt[i];
                    const float em = VEC ? expf(-Gv[i * kLt + dd]) : eGt[kT + i];
                    oq[w] = dq[nt][u] * ep;
                    ok[w] = dKt * ep + dKh * em;
                    dke[nt][u] *= kh;   // dKe (.) Ke, summed over the tile below
                }
                if (i < len) {
                    const int64_t r = ((t0 + i) * A.H + h) * kD + d;
                    if constexpr (VEC) {   // (dq and dk of any alignment)
                        A.dq[r] = __float2bfloat16_rn(oq[0]);
                        A.dq[r + 1] = __float2bfloat16_rn(oq[1]);
                        A.dk[r] = __float2bfloat16_rn(ok[0]);
                        A.dk[r + 1] = __float2bfloat16_rn(ok[1]);
                    } else {   // (the scalar gate's chunked form takes 16-byte aligned outputs)
                        *(__nv_bfloat162 *)&A.dq[r] = __floats2bfloat162_rn(oq[0], oq[1]);
                        *(__nv_bfloat162 *)&A.dk[r] = __floats2bfloat162_rn(ok[0], ok[1]);
                    }
                }
            }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float x = dke[nt][u] + dke[nt][u + 2];
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                if (g == 0) rG[c0 + 8 * nt + 2 * t + u] += x;
            }
        if constexpr (!VEC) {   // dG's row sums over this warp's 16 columns
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                float x = pg[hr];
                x += __shfl_xor_sync(0xffffffffu, x, 1);
                x += __shfl_xor_sync(0xffffffffu, x, 2);
                if (t == 0) dGp[warp * kT + g + 8 * hr] = x;
            }
        }
    }
    __syncthreads();
    // ---- dbeta (threads 0..15, one token each)
    if (tid < kT && tid < len) {
        const int i = tid;
        float acc = rowsum[i * 4] + rowsum[i * 4 + 1] + rowsum[i * 4 + 2] + rowsum[i * 4 + 3];
        // sum_j dA_ij (Kt Kh^T)_ij over the whole row: dA is 0 on and above the diagonal
#pragma unroll
        for (int j4 = 0; j4 < kT; j4 += 4) {
            const float4 a4 = *(const float4 *)&dA[i * kPd + j4], k4 = *(const float4 *)&KK[i * kPd + j4];
            acc = fmaf(a4.x, k4.x, fmaf(a4.y, k4.y, fmaf(a4.z, k4.z, fmaf(a4.w, k4.w, acc))));
        }
        A.dbeta[(t0 + i) * A.H + h] = __float2bfloat16_rn(acc);
    }
    // ---- da: the last token also carries dG_C; reverse cumsum over the tile
    if (VEC) {
        if (tid < kD) {
            const int d = tid;
            float acc = 0.f;
            for (int i = len - 1; i >= 0; --i) {
                acc += Ob[i * kLt + d] + (i == len - 1 ? rG[d] : 0.f);
                // g'(a) = -b s (1 - s) with s = -g / b, i.e. g (1 + g / b); g from the cumsum
                const float gi = Gv[i * kLt + d] - (i > 0 ? Gv[(i - 1) * kLt + d] : 0.f);
                const int64_t r = ((t0 + i) * A.H + h) * kD + d;
                A.da[r] = __float2bfloat16_rn(acc * gi * (1.f + gi / A.b));
            }
        }
    } else {
        if (warp == 0) {
            // per token: dG's row sum (the warps' partial sums), the last token also
            // carries dG_C summed over the channels; then the reverse cumsum over the
            // tile's tokens (lanes 0..15), times g'(a)
            float rgs = rG[lane] + rG[lane + 32] + rG[lane + 64] + rG[lane + 96];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) rgs += __shfl_xor_sync(0xffffffffu, rgs, o);
            float x = 0.f;
            if (lane < len) {
#pragma unroll
                for (int w = 0; w < kThreads / 32; ++w) x += dGp[w * kT + lane];
                if (lane == len - 1) x += rgs;
            }
#pragma unroll
            for (int o = 1; o < kT; o <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, x, o);
                if (lane + o < kT) x += y;
            }
            if (lane < len) A.da[(t0 + lane) * A.H + h] = __float2bfloat16_rn(x * Gb[kT + lane]);
        }
    }
}

// GDR_BWD_ADJ_MMA=1 / GDR_BWD_FWD_MMA=1 run the adjoint / forward state chain on the
// mma.sync kernel (for comparisons).
bool env_on(const char *name) {
    const char *e = std::getenv(name);
    return e && e[0] == '1';
}

template <bool VEC>
cudaError_t run_chunk_bwd(const BcArgs &A, int64_t T_total, int64_t max_tiles, int64_t max_segs, float *lam,
                          int *ok, int *status, cudaStream_t stream, const AuxStream &aux) {
    cudaError_t err;
    const int H = A.H;
    auto kf = bwd_fwd_chain_kernel<VEC>;
    auto ka = bwd_adj_chain_kernel<VEC>;
    auto kt = bwd_tile_kernel<VEC>;
    const size_t sf = sizeof(float) * kF_total, sa = sizeof(float) * kA_total, sg = TileLayout<VEC>::bytes;
    if ((err = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sf)) != cudaSuccess) return err;
    if ((err = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sa)) != cudaSuccess) return err;
    if ((err = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sg)) != cudaSuccess) return err;
    const int64_t segs = max_segs * H;
    if (segs > 0x7fffffff) return cudaErrorInvalidValue;
    if (max_tiles > 0) {
        ProfScope prof(stream, "bwd_bound_kernel");
        const int64_t nb = (max_tiles + kBoundWarps - 1) / kBoundWarps;
        const bool wide = (uintptr_t)A.k % 8 == 0 && (!VEC || (uintptr_t)A.a % 8 == 0);
        bwd_bound_kernel<VEC><<<dim3((unsigned)nb, (unsigned)H), 32 * kBoundWarps, 0, stream>>>(A, lam, max_tiles,
                                                                                               wide);
        count_launch();
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    {
        ProfScope prof(stream, "bwd_decide_kernel");
        bwd_decide_kernel<<<(unsigned)((int64_t)A.p.N * H), 32, 0, stream>>>(lam, ok, A.p, H);
        count_launch();
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    // The two chains are independent (the adjoint recurrence needs no forward state):
    // with an auxiliary stream the adjoint chain runs beside the forward chain, and the
    // tile kernel waits for both.
    const bool fork = aux.stream != nullptr;
    if (fork) {
        if ((err = cudaEventRecord(aux.fork, stream)) != cudaSuccess) return err;
        if ((err = cudaStreamWaitEvent(aux.stream, aux.fork, 0)) != cudaSuccess) return err;
    }
    {
        // the adjoint chain on tcgen05 unless a tensor map cannot be made (or the
        // mma.sync chain is asked for)
        cudaStream_t sa_stream = fork ? aux.stream : stream;
        err = env_on("GDR_BWD_ADJ_MMA") ? cudaErrorNotSupported
                                 : launch_tc_adj(A, VEC, T_total, max_tiles, max_segs, status, sa_stream);
        if (err == cudaErrorNotSupported) {
            ProfScope prof(sa_stream, "bwd_adj_chain_kernel");
            ka<<<(unsigned)segs, kThreads, sa, sa_stream>>>(A);
            count_launch();
            err = cudaGetLastError();
        }
        if (err != cudaSuccess) return err;
    }
    if (fork && (err = cudaEventRecord(aux.join, aux.stream)) != cudaSuccess) return err;
    {
        err = env_on("GDR_BWD_FWD_MMA") ? cudaErrorNotSupported
                                        : launch_tc_fwd_chain(A, VEC, T_total, max_tiles, max_segs, status, stream);
        if (err == cudaErrorNotSupported) {
            ProfScope prof(stream, "bwd_fwd_chain_kernel");
            kf<<<(unsigned)segs, kThreads, sf, stream>>>(A);
            count_launch();
            err = cudaGetLastError();
        }
        if (err != cudaSuccess) return err;
    }
    if (fork && (err = cudaStreamWaitEvent(stream, aux.join, 0)) != cudaSuccess) return err;
    if (max_tiles > 0) {
        ProfScope prof(stream, "bwd_tile_kernel");
        kt<<<dim3((unsigned)max_tiles, (unsigned)H), kThreads, sg, stream>>>(A);
        count_launch();
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace

// Segment length: the longest of 64, 128, 256 tiles that still leaves about eight
// (segment, head) blocks per resident block (two per SM).
int chunk_bwd_segment_tiles(int64_t tiles, int H, int sms) {
    int seg = kSegMin;
    while (seg < kSegMax && tiles * H / (2 * seg) >= (int64_t)16 * sms) seg *= 2;
    return seg;
}

size_t chunk_bwd_scratch_bytes(int64_t tiles, int N, int H) {
    return sizeof(__nv_bfloat16) * (size_t)tiles * H * 2 * kD * kD +
           sizeof(float) * (size_t)tiles * H * (2 * kT * kD + 1) + sizeof(int) * (size_t)N * H + 6 * 256;
}

cudaError_t launch_chunk_bwd(const void *q, const void *k, const void *v, const void *a,
                             const void *beta, const float *h0, const void *dout, const float *dhT,
                             void *dq, void *dk, void *dv, void *da, void *dbeta, float *dh0,
                             Plan plan, int H, int64_t T_total, int64_t max_tiles, int64_t max_segs,
                             float b, bool per_channel, void *scratch, int *status, cudaStream_t stream,
                             const AuxStream &aux) {
    if (plan.C != kT || plan.seg_chunks < kSegMin || plan.seg_chunks > kSegMax) return cudaErrorInvalidValue;
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
    const size_t sth = sizeof(__nv_bfloat16) * (size_t)max_tiles * H * kD * kD;
    A.Hst = (__nv_bfloat16 *)p;
    p += al(sth);
    A.dHst = (__nv_bfloat16 *)p;
    p += al(sth);
    A.Dst = (float *)p;
    p += al(sizeof(float) * (size_t)max_tiles * H * kT * kD);
    A.dDst = (float *)p;
    p += al(sizeof(float) * (size_t)max_tiles * H * kT * kD);
    float *lam = (float *)p;
    p += al(sizeof(float) * (size_t)max_tiles * H);
    int *ok = (int *)p;
    A.lam = lam;
    A.seg_ok = ok;
    A.p = plan;
    A.H = H;
    A.b = b;
    return per_channel ? run_chunk_bwd<true>(A, T_total, max_tiles, max_segs, lam, ok, status, stream, aux)
                       : run_chunk_bwd<false>(A, T_total, max_tiles, max_segs, lam, ok, status, stream, aux);
}

}  // namespace gdr
