// gdr_tc.cu -- the tensor-core (tcgen05) path of the chunked gated delta rule.
//
// Shape: bf16 inputs, dk = dv = 128, tile C = 16.  One CTA runs one stream:
// the tiles of one (sequence, head) segment in order.  The state never
// leaves the tensor memory: it is the fp32 accumulator of the state-update
// MMA and the (tf32) A operand of the W.H / Q.H products.
//
// Per tile, with in-tile cumulative log-decay G and entering state H
// (transposed in TMEM: lane = value index e, column = key index d)
// [P1 §3.2-3.3, P2 §2.1-2.2, P3 §3.1-3.3]:
//   prep warps (CUDA cores + mma.sync):  Skk = K K^T, Sqk = Q K^T,
//       A = strict_lower(beta_i e^{G_i-G_j} Skk),  T = (I + A)^{-1},
//       Bu = T diag(beta),  Bw = T diag(beta e^G),  W = Bw K,  Qt = diag(e^G) Q,
//       P = Sqk (.) [j<=i] (.) e^{G_i-G_j}
//   tensor cores (one issuing thread):
//       D_U  = V^T Bu^T                  (U^T, kind::f16)
//       D_X  = H^T [-W ; Qt]^T           (kind::tf32, A = the state in TMEM)
//       D    = U + Gamma * D_X[:, :C]    (the delta-rule writes, per lane)
//       H^   += Dt^T K                   (kind::f16, A = Dt in TMEM, the state update)
//       D_X[:, C:] += (D/Gamma)^T P^T    (in-tile output term)
// Decays are never applied to the whole state per tile: the state is kept
// as H = Gamma * H^ with a running scalar Gamma (product of tile decays),
// and the tile's writes enter H^ scaled by 1/Gamma.  Gamma is folded back
// into H^ only when it would fall below 2^-100, so the factor is always a
// bounded reciprocal of accumulated decay -- the quantity the pages bound
// with the scaled-sigmoid gate -- and fp32 range is never left.
//
// A long sequence is split into segments processed in parallel:
//   pass A (per non-last segment): the segment's transition H_out = M H_in + B
//           as two streams of the same kernel: B from a zero state (or from
//           h0 for the first segment) and M from the identity with v = 0;
//   combine: H_in(s+1) = M_s H_in(s) + B_s, serial over segments (fp32);
//   pass C (every segment): the outputs from the true entering state.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "gdr_sm100.cuh"
#include "gdr_tc.cuh"

namespace gdr {
namespace {

using namespace sm100;

constexpr int kD = 128;          // dk = dv
constexpr int kC = 16;           // tile length on this path
constexpr int kNS = 3;           // pipeline stages, one per prep warp
constexpr int kThreads = 32 * (4 + kNS);   // 4 state warps + kNS prep warps
constexpr uint64_t kWaitNs = 2000000000ull;  // bounded waits: 2 s

// TMEM columns
constexpr uint32_t kColH = 0;                    // state H^ (128 fp32 columns)
constexpr uint32_t kColX = 128;                  // D_X, 2 buffers x 2C
constexpr uint32_t kColU = kColX + 2 * 2 * kC;   // D_U, C columns
constexpr uint32_t kColA = kColU + kC;           // bf16 A operands: Dt (C/2) and D/Gamma (C/2)
constexpr uint32_t kTmemCols = 256;
static_assert(kColA + kC <= kTmemCols, "TMEM budget");

// Shared memory, per stage
constexpr uint32_t kBox = kC * 128;              // one 64-column box of a [C][128] bf16 tile
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + 2 * kBox;
constexpr uint32_t kOffQ = kOffV + 2 * kBox;
constexpr uint32_t kOffWQ = kOffQ + 2 * kBox;    // tf32 [2C rows][128], 4 swizzled 32-wide column blocks
constexpr uint32_t kWQBlock = 2 * kC * 128;
constexpr uint32_t kOffBU = kOffWQ + 4 * kWQBlock;
constexpr uint32_t kOffP = kOffBU + kC * kC * 2;
constexpr uint32_t kOffHdr = kOffP + kC * kC * 2;
constexpr uint32_t kStage = 30720;
static_assert(kOffHdr + 256 <= kStage, "stage layout");
// per-prep-warp scratch after the stages
constexpr uint32_t kScrSkk = 0;                  // fp32 [C][C+1]
constexpr uint32_t kScrSqk = kScrSkk + kC * (kC + 1) * 4;
constexpr uint32_t kScrBW = 2304;                // bf16 [C][C] row-major (32 B rows)
constexpr uint32_t kScr = 2816;
static_assert(kScrSqk + kC * (kC + 1) * 4 <= kScrBW, "scratch layout");
constexpr uint32_t kOffScr = kNS * kStage;
constexpr uint32_t kOffBar = kOffScr + kNS * kScr;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // + alignment slack

// core-matrix (no swizzle) K-major layout of a C x C bf16 operand [n][k]
__device__ __forceinline__ uint32_t cc_off(int n, int k) {
    return core_off((uint32_t)n, (uint32_t)k * 2u, (kC / 8) * 128u, 128u);
}

struct Hdr {
    float G[kC];
    float beta[kC];
    int len;
};

enum Mode : int { kModeOut = 0, kModeB = 1, kModeM = 2 };

struct TcArgs {
    const float *G;
    const float *Bt;
    const float *h0;
    void *out;
    float *hT;
    float *Hin;   // [segs][H][D][D] entering states (pass C, s >= 1)
    float *Bs;    // [segs][H][D][D] transition offsets
    float *Ms;    // [segs][H][D][D] transition matrices
    Plan plan;
    int H;
    int64_t T_total;
    int mode;
    int *status;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9},"
        " {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Segment geometry of CTA (gseg, h): sequence n, first tile, tile count, last?
struct SegInfo {
    int n;
    int s;            // segment index within the sequence
    int nseg;         // segments of the sequence
    int64_t tok0;     // first token row of the sequence
    int64_t len;      // tokens of the sequence
    int64_t c0, c1;   // tile range [c0, c1) of this segment
};
__device__ __forceinline__ bool seg_info(const Plan &p, int64_t gseg, SegInfo &si) {
    const int n = find_owner(p.seg_base, p.N, gseg);
    if (n < 0) return false;
    si.n = n;
    si.s = (int)(gseg - p.seg_base[n]);
    si.nseg = (int)(p.seg_base[n + 1] - p.seg_base[n]);
    si.tok0 = p.seq_start[n];
    si.len = p.seq_start[n + 1] - si.tok0;
    const int64_t nch = (si.len + kC - 1) / kC;
    si.c0 = min((int64_t)si.s * p.seg_chunks, nch);
    si.c1 = min(si.c0 + (int64_t)p.seg_chunks, nch);
    if (si.s == si.nseg - 1) si.c1 = nch;
    return true;
}

// ---------------------------------------------------------------------------
// the chunk kernel (all three modes)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 2)
tc_chunk_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const TcArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bar_full = (uint64_t *)(smem + kOffBar);
    uint64_t *bar_prep = bar_full + kNS;
    uint64_t *bar_free = bar_prep + kNS;
    uint64_t *bar_x = bar_free + kNS;    // [2]
    uint64_t *bar_h = bar_x + 2;         // [1]
    uint64_t *bar_fin = bar_h + 1;       // [1]
    uint32_t *tmem_slot = (uint32_t *)(bar_fin + 1);
    volatile int *abort_prep = (volatile int *)(tmem_slot + 1);   // set by prep warps
    volatile int *abort_state = abort_prep + 1;                   // set by state warps only

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mode = args.mode;
    const int h = blockIdx.y;
    SegInfo si;
    if (!seg_info(args.plan, blockIdx.x, si)) return;
    const bool last_seg = si.s == si.nseg - 1;
    if (mode != kModeOut) {  // transition passes: only non-last segments
        if (last_seg) return;
        if (mode == kModeM && si.s == 0) return;
    }
    const int H = args.H;
    const int64_t gsh = (int64_t)blockIdx.x * H + h;   // (global segment, head) slot
    const float *h_in = nullptr;
    float *h_out = nullptr;
    if (mode == kModeOut) {
        h_in = si.s == 0 ? (args.h0 ? args.h0 + ((int64_t)si.n * H + h) * kD * kD : nullptr)
                         : args.Hin + gsh * kD * kD;
        h_out = (last_seg && args.hT) ? args.hT + ((int64_t)si.n * H + h) * kD * kD : nullptr;
    } else if (mode == kModeB) {
        h_in = (si.s == 0 && args.h0) ? args.h0 + ((int64_t)si.n * H + h) * kD * kD : nullptr;
        h_out = args.Bs + gsh * kD * kD;
    } else {
        h_out = args.Ms + gsh * kD * kD;
    }
    const bool use_v = mode != kModeM, use_q = mode == kModeOut;
    const int nch = (int)(si.c1 - si.c0);
    constexpr unsigned kFull = 0xffffffffu;

    if (tid == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_prep[i], 1);
            mbar_init(&bar_free[i], 1);
        }
        mbar_init(&bar_x[0], 1);
        mbar_init(&bar_x[1], 1);
        mbar_init(&bar_h[0], 1);
        mbar_init(&bar_fin[0], 1);
        *abort_prep = 0;
        *abort_state = 0;
        fence_mbar_init();
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 32) {
        prefetch_tensormap(&tmQ);
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;

    if (warp >= 4) {
        // ============================ prep warps ============================
        const int pw = warp - 4;
        uint8_t *scr = smem + kOffScr + pw * kScr;
        float *Skk = (float *)(scr + kScrSkk);
        float *Sqk = (float *)(scr + kScrSqk);
        uint8_t *BW = scr + kScrBW;
        const uint32_t tx_bytes = 2 * kBox * (1 + (use_v ? 1 : 0) + (use_q ? 1 : 0));
        int pend_st = -1;          // stage whose TMA is issued but not yet seen complete
        uint32_t pend_ph = 0;
        // prep warp pw owns stage pw and tiles pw, pw + kNS, ...: every wait on a
        // stage barrier is for the phase right after the one this warp consumed
        for (int c = pw; c < nch; c += kNS) {
            if (__any_sync(kFull, *abort_prep != 0 || *abort_state != 0)) break;
            const int st = pw;
            const uint32_t ph = (uint32_t)(c / kNS) & 1u;
            uint8_t *stg = smem + st * kStage;
            Hdr *hdr = (Hdr *)(stg + kOffHdr);
            const int64_t tc = si.c0 + c;                  // tile index within the sequence
            const int64_t t0 = si.tok0 + tc * kC;         // first token row
            const int len = (int)min((int64_t)kC, si.len - tc * kC);
            // gates of the tile (issued before the waits)
            float g_i = 0.f, b_i = 0.f;
            if (lane < kC) {
                const int i = min(lane, len - 1);
                g_i = args.G[(int64_t)h * args.T_total + t0 + i];
                b_i = lane < len ? args.Bt[(int64_t)h * args.T_total + t0 + lane] : 0.f;
            }
            if (c >= kNS && !__all_sync(kFull, mbar_wait(&bar_free[st], ph ^ 1u, kWaitNs))) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_prep = 1;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar_full[st], tx_bytes);
                tma_load_3d(stg + kOffK, &tmK, 0, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffK + kBox, &tmK, 64, h, (int)t0, &bar_full[st]);
                if (use_v) {
                    tma_load_3d(stg + kOffV, &tmV, 0, h, (int)t0, &bar_full[st]);
                    tma_load_3d(stg + kOffV + kBox, &tmV, 64, h, (int)t0, &bar_full[st]);
                }
                if (use_q) {
                    tma_load_3d(stg + kOffQ, &tmQ, 0, h, (int)t0, &bar_full[st]);
                    tma_load_3d(stg + kOffQ + kBox, &tmQ, 64, h, (int)t0, &bar_full[st]);
                }
            }
            pend_st = st;
            pend_ph = ph;
            if (lane < kC) {
                hdr->G[lane] = g_i;
                hdr->beta[lane] = b_i;
            }
            if (lane == 0) hdr->len = len;
            if (!__all_sync(kFull, mbar_wait(&bar_full[st], ph, kWaitNs))) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_prep = 1;
                break;
            }
            pend_st = -1;
            // rows past the end of the sequence hold another sequence's tokens: zero them
            if (len < kC) {
                const int nt = 1 + (use_v ? 1 : 0) + (use_q ? 1 : 0);
                const int nrow = kC - len;
                for (int e = lane; e < nt * 2 * nrow * 8; e += 32) {
                    const int chunk16 = e & 7, rem = e >> 3;
                    const int row = len + rem % nrow, box = (rem / nrow) & 1;
                    const int tsel = rem / (nrow * 2);
                    const uint32_t toff =
                        tsel == 0 ? kOffK : ((tsel == 1 && use_v) ? kOffV : kOffQ);
                    *(uint4 *)(stg + toff + box * kBox + sw128_off(row, chunk16 * 16)) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            __syncwarp();
            // ---- Gram matrices Skk = K K^T, Sqk = Q K^T (mma.sync, bf16 -> fp32)
            float skk[2][4] = {}, sqk[2][4] = {};
            {
                const int r = lane & 15, half = lane >> 4;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * kBox + sw128_off(r, 32 * (ks & 3) + 16 * half);
                    uint32_t kf[4];
                    ldsm_x4(smem_u32(stg + kOffK + off), kf);
                    mma16816(skk[0], kf, kf[0], kf[2]);
                    mma16816(skk[1], kf, kf[1], kf[3]);
                    if (use_q) {
                        uint32_t qf[4];
                        ldsm_x4(smem_u32(stg + kOffQ + off), qf);
                        mma16816(sqk[0], qf, kf[0], kf[2]);
                        mma16816(sqk[1], qf, kf[1], kf[3]);
                    }
                }
            }
            {
                const int r0 = lane >> 2;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int col = 8 * nt + 2 * (lane & 3);
                    Skk[r0 * (kC + 1) + col] = skk[nt][0];
                    Skk[r0 * (kC + 1) + col + 1] = skk[nt][1];
                    Skk[(r0 + 8) * (kC + 1) + col] = skk[nt][2];
                    Skk[(r0 + 8) * (kC + 1) + col + 1] = skk[nt][3];
                    Sqk[r0 * (kC + 1) + col] = sqk[nt][0];
                    Sqk[r0 * (kC + 1) + col + 1] = sqk[nt][1];
                    Sqk[(r0 + 8) * (kC + 1) + col] = sqk[nt][2];
                    Sqk[(r0 + 8) * (kC + 1) + col + 1] = sqk[nt][3];
                }
            }
            __syncwarp();
            // ---- A (in place over Skk) and P (bf16, core-matrix layout in the stage)
            for (int e = lane; e < kC * kC; e += 32) {
                const int i = e / kC, j = e % kC;
                const float dg = __expf(fminf(hdr->G[i] - hdr->G[j], 0.f));
                const float a_ij = j < i ? hdr->beta[i] * dg * Skk[i * (kC + 1) + j] : 0.f;
                Skk[i * (kC + 1) + j] = a_ij;
                if (use_q) {
                    const float p_ij = j <= i ? Sqk[i * (kC + 1) + j] * dg : 0.f;
                    *(__nv_bfloat16 *)(stg + kOffP + cc_off(i, j)) = __float2bfloat16_rn(p_ij);
                }
            }
            __syncwarp();
            // ---- T = (I + A)^{-1}, one column per lane (forward substitution)
            {
                const int j = lane & (kC - 1);
                float tcol[kC];
#pragma unroll
                for (int i = 0; i < kC; ++i) {
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < i; ++m) acc = fmaf(Skk[i * (kC + 1) + m], tcol[m], acc);
                    tcol[i] = (i < j) ? 0.f : ((i == j) ? 1.f : -acc);
                }
                if (lane < kC) {
                    const float bj = hdr->beta[j];
                    const float bej = bj * __expf(hdr->G[j]);
#pragma unroll
                    for (int i = 0; i < kC; ++i) {
                        if (use_v)
                            *(__nv_bfloat16 *)(stg + kOffBU + cc_off(i, j)) =
                                __float2bfloat16_rn(tcol[i] * bj);
                        *(__nv_bfloat16 *)(BW + i * 32 + j * 2) = __float2bfloat16_rn(tcol[i] * bej);
                    }
                }
            }
            __syncwarp();
            // ---- W = Bw K (mma.sync) -> rows [0, C) of WQ as -W in tf32
            {
                uint32_t af[4];
                ldsm_x4(smem_u32(BW + (lane & 15) * 32 + (lane >> 4) * 16), af);
                const int jrow = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    const int d0 = 16 * np + 8 * (lane >> 4);
                    uint32_t bf[4];
                    ldsm_x4_t(smem_u32(stg + kOffK + (d0 >> 6) * kBox + sw128_off(jrow, (d0 & 63) * 2)), bf);
                    float w0[4] = {}, w1[4] = {};
                    mma16816(w0, af, bf[0], bf[1]);
                    mma16816(w1, af, bf[2], bf[3]);
                    const int i0 = lane >> 2;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const float *w = t == 0 ? w0 : w1;
                        const int d = 16 * np + 8 * t + 2 * (lane & 3);
                        uint8_t *base = stg + kOffWQ + (d >> 5) * kWQBlock;
                        *(float2 *)(base + sw128_off(i0, (d & 31) * 4)) = make_float2(-w[0], -w[1]);
                        *(float2 *)(base + sw128_off(i0 + 8, (d & 31) * 4)) = make_float2(-w[2], -w[3]);
                    }
                }
            }
            // ---- rows [C, 2C) of WQ: diag(e^G) Q in tf32
            if (use_q) {
                const int i = lane >> 1, hb = lane & 1;
                const float eg = __expf(hdr->G[i]);
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint4 raw = *(const uint4 *)(stg + kOffQ + hb * kBox + sw128_off(i, 16 * c8));
                    const __nv_bfloat162 *bp = (const __nv_bfloat162 *)&raw;
                    float f[8];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 x = __bfloat1622float2(bp[u]);
                        f[2 * u] = x.x * eg;
                        f[2 * u + 1] = x.y * eg;
                    }
                    const int d = 64 * hb + 8 * c8;
                    uint8_t *base = stg + kOffWQ + (d >> 5) * kWQBlock;
                    *(float4 *)(base + sw128_off(kC + i, (d & 31) * 4)) = make_float4(f[0], f[1], f[2], f[3]);
                    *(float4 *)(base + sw128_off(kC + i, (d & 31) * 4 + 16)) = make_float4(f[4], f[5], f[6], f[7]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_prep[st]);
        }
        // never leave with a tile copy still in flight
        if (pend_st >= 0) {
            mbar_wait(&bar_full[pend_st], pend_ph, kWaitNs);
            __syncwarp();
        }
    } else {
        // ============================ state warps ============================
        const int e = tid;                       // value index = TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        // H^ <- h_in (or 0, or the identity for the transition matrix)
        for (int d0 = 0; d0 < kD; d0 += 16) {
            uint32_t r[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float x = 0.f;
                if (h_in) x = h_in[(int64_t)(d0 + j) * kD + e];
                else if (mode == kModeM) x = (d0 + j == e) ? 1.f : 0.f;
                r[j] = __float_as_uint(x);
            }
            __syncwarp();
            tmem_st16(tm + lane_base + kColH + d0, r);
        }
        tmem_st_wait();
        tc_fence_before();
        named_barrier(1, 128);
        float Gamma = 1.f;                // H = Gamma * H^
        float gamma_prev = 1.f;           // Gamma of the previous tile's output
        int64_t t0_prev = 0;
        int len_prev = 0;
        const uint32_t id_u = instr_desc(128, kC, 1, true, false);
        const uint32_t id_x = instr_desc(128, use_q ? 2 * kC : kC, 2, false, false);
        const uint32_t id_h = instr_desc(128, kD, 1, false, true);
        const uint32_t id_o = instr_desc(128, kC, 1, false, false);
        int done = 0;                     // tiles whose state update was issued
        for (int c = 0; c < nch; ++c) {
            const int st = c % kNS;
            const uint32_t ph = (uint32_t)(c / kNS) & 1u;
            const int buf = c & 1;
            uint8_t *stg = smem + st * kStage;
            const uint32_t sb = smem_u32(stg);
            if (tid == 0) {
                tc_fence_after();
                bool okw = c == 0 || mbar_wait(&bar_h[0], (uint32_t)(c - 1) & 1u, kWaitNs);
                okw = okw && mbar_wait(&bar_prep[st], ph, kWaitNs);
                if (okw) {
                    tc_fence_after();
                    if (use_v)
                        mma_f16_ss(tm + kColU, smem_desc(sb + kOffV, kBox, 1024, kSw128),
                                   smem_desc(sb + kOffBU, 128, (kC / 8) * 128, kSwNone), id_u, 0);
#pragma unroll
                    for (int s8 = 0; s8 < kD / 8; ++s8)
                        mma_tf32_ts(tm + kColX + buf * 2 * kC, tm + kColH + 8 * s8,
                                    smem_desc(sb + kOffWQ + (s8 >> 2) * kWQBlock + 32 * (s8 & 3), 16, 1024, kSw128),
                                    id_x, s8 > 0);
                    mma_commit(&bar_x[buf]);
                } else {
                    set_status(args.status, GDR_ERR_TIMEOUT);
                    *abort_state = 1;
                }
            }
            __syncwarp();
            // everyone: the tile's header and the MMA results (a missing result times out)
            const bool okw = mbar_wait(&bar_prep[st], ph, kWaitNs) &&
                             mbar_wait(&bar_x[buf], (uint32_t)(c >> 1) & 1u, kWaitNs);
            if (!okw) {
                set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_state = 1;
            }
            __syncwarp();
            named_barrier(1, 128);        // one view of abort_state for the whole group
            if (*abort_state) break;
            tc_fence_after();
            const Hdr *hdr = (const Hdr *)(stg + kOffHdr);
            const int len_c = hdr->len;   // read before the stage can be recycled
            uint32_t xr[kC], ur[kC], orr[kC];
            tmem_ld16(tm + lane_base + kColX + buf * 2 * kC, xr);
            if (use_v) tmem_ld16(tm + lane_base + kColU, ur);
            if (use_q && c > 0) tmem_ld16(tm + lane_base + kColX + (buf ^ 1) * 2 * kC + kC, orr);
            tmem_ld_wait();
            const float GC = hdr->G[kC - 1];
            const float gam = __expf(GC);
            float Gp = Gamma * gam;
            const bool renorm = !(Gp >= 1e-30f);   // ~2^-100; also catches gam == 0
            float s2;
            if (renorm) {
                // fold Gamma * gam into H^ (the MMAs reading H^ for this tile are done)
                const float f = Gamma * gam;
                for (int d0 = 0; d0 < kD; d0 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tm + lane_base + kColH + d0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
                    tmem_st16(tm + lane_base + kColH + d0, r);
                }
                tmem_st_wait();
                s2 = 1.f;
                Gp = 1.f;
            } else {
                s2 = 1.f / Gp;
            }
            uint32_t a2[kC / 2], a3[kC / 2];
            const float inv_g = 1.f / Gamma;
#pragma unroll
            for (int i = 0; i < kC; i += 2) {
                float dl0 = Gamma * __uint_as_float(xr[i]);
                float dl1 = Gamma * __uint_as_float(xr[i + 1]);
                if (use_v) {
                    dl0 += __uint_as_float(ur[i]);
                    dl1 += __uint_as_float(ur[i + 1]);
                }
                const float r0 = __expf(fminf(GC - hdr->G[i], 0.f)) * s2;
                const float r1 = __expf(fminf(GC - hdr->G[i + 1], 0.f)) * s2;
                a2[i / 2] = pack_bf16(dl0 * r0, dl1 * r1);
                a3[i / 2] = pack_bf16(dl0 * inv_g, dl1 * inv_g);
            }
            tmem_st8(tm + lane_base + kColA, a2);
            if (use_q) tmem_st8(tm + lane_base + kColA + kC / 2, a3);
            tmem_st_wait();
            tc_fence_before();
            named_barrier(1, 128);
            if (tid == 0) {
                tc_fence_after();
                mma_f16_ts(tm + kColH, tm + kColA, smem_desc(sb + kOffK, kBox, 1024, kSw128), id_h, 1);
                if (use_q)
                    mma_f16_ts(tm + kColX + buf * 2 * kC + kC, tm + kColA + kC / 2,
                               smem_desc(sb + kOffP, 128, (kC / 8) * 128, kSwNone), id_o, 1);
                mma_commit(&bar_free[st]);
                mma_commit(&bar_h[0]);
            }
            __syncwarp();
            // output of the previous tile (its MMAs completed before this tile's D_X)
            if (use_q && c > 0) {
                __nv_bfloat16 *out = (__nv_bfloat16 *)args.out;
                for (int i = 0; i < len_prev; ++i)
                    out[((t0_prev + i) * H + h) * kD + e] =
                        __float2bfloat16_rn(__uint_as_float(orr[i]) * gamma_prev);
            }
            gamma_prev = Gamma;
            t0_prev = si.tok0 + (si.c0 + c) * kC;
            len_prev = len_c;
            Gamma = renorm ? 1.f : Gp;
            done = c + 1;
        }
        // drain: the last tile's output, then the final state
        if (done > 0 && done == nch) {
            if (!mbar_wait(&bar_h[0], (uint32_t)(nch - 1) & 1u, kWaitNs)) {
                set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_state = 1;
            }
        }
        __syncwarp();
        named_barrier(1, 128);
        const bool ok = *abort_state == 0 && done == nch;
        tc_fence_after();
        if (ok && use_q && nch > 0) {
            uint32_t orr[kC];
            tmem_ld16(tm + lane_base + kColX + ((nch - 1) & 1) * 2 * kC + kC, orr);
            tmem_ld_wait();
            __nv_bfloat16 *out = (__nv_bfloat16 *)args.out;
            for (int i = 0; i < len_prev; ++i)
                out[((t0_prev + i) * H + h) * kD + e] =
                    __float2bfloat16_rn(__uint_as_float(orr[i]) * gamma_prev);
        }
        if (ok && h_out) {
            for (int d0 = 0; d0 < kD; d0 += 16) {
                uint32_t r[16];
                tmem_ld16(tm + lane_base + kColH + d0, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) h_out[(int64_t)(d0 + j) * kD + e] = __uint_as_float(r[j]) * Gamma;
            }
        }
    }
    // teardown: no tensor-core operation may still be running when the TMEM is released
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after();
        mma_commit(&bar_fin[0]);
        mbar_wait(&bar_fin[0], 0, kWaitNs);
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// combine: H_in(s+1) = M_s H_in(s) + B_s, serial over the segments of one
// (sequence, head); one block per 32 state columns, fp32 FMA.
// ---------------------------------------------------------------------------
constexpr int kCombCols = 32;

__global__ void __launch_bounds__(256)
tc_combine_kernel(float *Hin, const float *Bs, const float *Ms, Plan p, int H) {
    extern __shared__ float cs[];
    float *Msh = cs;                  // [128][129]
    float *Hs = Msh + kD * (kD + 1);  // [128][32]
    const int slice = blockIdx.x % (kD / kCombCols);
    const int h = (blockIdx.x / (kD / kCombCols)) % H;
    const int n = blockIdx.x / ((kD / kCombCols) * H);
    if (n >= p.N) return;
    const int64_t g0 = p.seg_base[n];
    const int nseg = (int)(p.seg_base[n + 1] - g0);
    const int j0 = slice * kCombCols, tid = threadIdx.x;
    for (int s = 1; s < nseg; ++s) {
        const int64_t prev = (g0 + s - 1) * H + h, cur = (g0 + s) * H + h;
        const float *B = Bs + prev * kD * kD;
        float *Hc = Hin + cur * kD * kD;
        if (s == 1) {
            for (int e = tid; e < kD * kCombCols; e += 256) {
                const int d = e / kCombCols, j = e % kCombCols;
                const float x = B[d * kD + j0 + j];
                Hc[d * kD + j0 + j] = x;
                Hs[e] = x;
            }
            __syncthreads();
            continue;
        }
        const float *M = Ms + prev * kD * kD;
        for (int e = tid; e < kD * kD; e += 256) Msh[(e / kD) * (kD + 1) + e % kD] = M[e];
        __syncthreads();
        // out[d][j] = sum_m M[d][m] Hs[m][j] + B[d][j];  thread: rows d = tid/8 + 32r, cols j = 4(tid%8)..+3
        float acc[4][4];
        const int dr = tid >> 3, jc = (tid & 7) * 4;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[r][q] = B[(dr + 32 * r) * kD + j0 + jc + q];
        for (int m = 0; m < kD; ++m) {
            const float4 hv = *(const float4 *)&Hs[m * kCombCols + jc];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float mv = Msh[(dr + 32 * r) * (kD + 1) + m];
                acc[r][0] = fmaf(mv, hv.x, acc[r][0]);
                acc[r][1] = fmaf(mv, hv.y, acc[r][1]);
                acc[r][2] = fmaf(mv, hv.z, acc[r][2]);
                acc[r][3] = fmaf(mv, hv.w, acc[r][3]);
            }
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int d = dr + 32 * r, j = jc + q;
                Hc[d * kD + j0 + j] = acc[r][q];
                Hs[d * kCombCols + j] = acc[r][q];
            }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    });
    return fn;
}

// [rows][H][128] bf16 viewed as (d, h, row), box (64, 1, C), 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *base, int H, int64_t rows) {
    auto fn = encode_fn();
    if (!fn || ((uintptr_t)base & 15)) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)std::max<int64_t>(rows, 1)};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)kD * 2 * H};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kC};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
    }
    return n;
}

int64_t max_segments(int N, int64_t T_total, int seg_chunks) {
    const int64_t tiles = (T_total + kC - 1) / kC + N;
    return tiles / seg_chunks + 2 * (int64_t)N + 1;
}

}  // namespace

bool tc_supported(gdr_dtype_t dtype, int dk, int dv, int chunk) {
    return dtype == GDR_BF16 && dk == kD && dv == kD && chunk == kC;
}

int tc_segment_chunks(int N, int H, int64_t T_total, int C) {
    if (const char *env = std::getenv("GDR_TC_SEG_CHUNKS")) {
        const int v = std::atoi(env);
        if (v > 0) return v;
    }
    // about two resident streams per SM in the output pass
    const int64_t target = 2 * (int64_t)sm_count();
    const int64_t tiles = (T_total + C - 1) / C + N;
    int64_t sc = (tiles * H + target - 1) / target;
    return (int)std::max<int64_t>(32, std::min<int64_t>(sc, 1 << 30));
}

size_t tc_workspace_bytes(int N, int H, int64_t T_total, int C) {
    const int sc = tc_segment_chunks(N, H, T_total, C);
    const size_t per = (size_t)max_segments(N, T_total, sc) * H * kD * kD * sizeof(float);
    return 3 * ((per + 255) / 256 * 256);
}

cudaError_t launch_tc_forward(const void *q, const void *k, const void *v, const float *G,
                              const float *Bt, const float *h0, void *out, float *hT, Plan plan,
                              int H, int64_t T_total, int64_t max_chunks, void *scratch,
                              int *status, cudaStream_t stream) {
    (void)max_chunks;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, H, T_total) || !make_map(&mk, k, H, T_total) || !make_map(&mv, v, H, T_total))
        return cudaErrorInvalidValue;
    const int64_t nseg = max_segments(plan.N, T_total, plan.seg_chunks);
    const size_t per = ((size_t)nseg * H * kD * kD * sizeof(float) + 255) / 256 * 256;
    TcArgs a{};
    a.G = G;
    a.Bt = Bt;
    a.h0 = h0;
    a.out = out;
    a.hT = hT;
    a.Hin = (float *)scratch;
    a.Bs = (float *)((char *)scratch + per);
    a.Ms = (float *)((char *)scratch + 2 * per);
    a.plan = plan;
    a.H = H;
    a.T_total = T_total;
    a.status = status;
    cudaError_t err = cudaFuncSetAttribute(tc_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    const size_t comb_smem = sizeof(float) * (kD * (kD + 1) + kD * kCombCols);
    err = cudaFuncSetAttribute(tc_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)comb_smem);
    if (err != cudaSuccess) return err;
    const dim3 grid((unsigned)nseg, (unsigned)H);
    {   // pass A: transitions of every non-last segment (B and M streams)
        ProfScope prof(stream, "tc_transition_B");
        a.mode = kModeB;
        tc_chunk_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, a);
        count_launch();
    }
    {
        ProfScope prof(stream, "tc_transition_M");
        a.mode = kModeM;
        tc_chunk_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, a);
        count_launch();
    }
    {
        ProfScope prof(stream, "tc_combine_kernel");
        tc_combine_kernel<<<(unsigned)(plan.N * H * (kD / kCombCols)), 256, comb_smem, stream>>>(
            a.Hin, a.Bs, a.Ms, plan, H);
        count_launch();
    }
    {
        ProfScope prof(stream, "tc_output_kernel");
        a.mode = kModeOut;
        tc_chunk_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, a);
        count_launch();
    }
    return cudaGetLastError();
}

}  // namespace gdr
