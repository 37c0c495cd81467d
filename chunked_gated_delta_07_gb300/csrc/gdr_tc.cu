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
//           where M_s is negligible, H_in(s+1) = B_s is read in place;
//   pass C (every segment): the outputs from the true entering state.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <mutex>

#include "gdr_sm100.cuh"
#include "gdr_tc.cuh"

namespace gdr {

GDR_DEBUG_TU()

namespace {

using namespace sm100;

constexpr int kD = 128;          // dk = dv
constexpr int kC = 16;           // tile length on this path
constexpr int kNS = 4;           // pipeline stages, one per prep warp
constexpr int kThreads = 32 * (4 + kNS + 1);   // 4 state warps, kNS prep warps, 1 MMA issuer
// Every wait is bounded.  The pipeline waits use the launch's limit (TcArgs::wait_ns,
// 2 s unless GDR_TC_WAIT_NS is set, which the tests use to make waits run out); the
// drains before exit -- a tile copy still in flight, the CTA's last MMAs -- always
// allow kDrainNs, since the CTA may not leave while either is pending.
constexpr uint64_t kWaitNs = 2000000000ull;   // default pipeline limit: 2 s
constexpr uint64_t kDrainNs = 2000000000ull;  // drain limit: 2 s
// The state is kept as H = Gamma * H^.  Gamma runs down by each tile's decay and
// is folded into H^ (Gamma reset to 1) before it would drop below kGammaMin, so
// H^ stays within |H| / kGammaMin and the scaled writes within |Delta| /
// kGammaMin: both far inside fp32 / bf16 range.  (Resetting to a large Gamma
// instead, to fold less often, measured slower.)
constexpr float kGammaMin = 1e-30f;

// TMEM columns
constexpr uint32_t kColH = 0;                    // state H^ (128 fp32 columns)
constexpr uint32_t kColB = 128;                  // 2 buffers of [U (C) | -W H (C) | out (C)]
constexpr uint32_t kColBuf = 3 * kC;
constexpr uint32_t kColA = kColB + 2 * kColBuf;  // bf16 A operands: Dt (C/2) and D/Gamma (C/2)
constexpr uint32_t kTmemCols = 256;
static_assert(kColA + kC <= kTmemCols, "TMEM budget");

// Shared memory, per stage (26 KB, so that 4 stages fit at 2 CTAs per SM).
// [-W ; Qt] in tf32 is 4 column blocks of 2C rows x 128 B (rows 0..C-1: -W,
// rows C..2C-1: Qt).  The -W rows are written last, so until then they hold
// the raw Q tile (blocks 0, 1: one 64-column box each) and the prep warp's
// scratch (blocks 2, 3).
constexpr uint32_t kBox = kC * 128;              // one 64-column box of a [C][128] bf16 tile
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + 2 * kBox;
constexpr uint32_t kOffWQ = kOffV + 2 * kBox;
constexpr uint32_t kWQBlock = 2 * kC * 128;
constexpr uint32_t kOffQ0 = kOffWQ;                  // raw Q, columns 0..63
constexpr uint32_t kOffQ1 = kOffWQ + kWQBlock;       // raw Q, columns 64..127
constexpr uint32_t kOffSkk = kOffWQ + 2 * kWQBlock;  // fp32 [C][C] K K^T, then A
constexpr uint32_t kOffSqk = kOffSkk + kC * kC * 4;  // fp32 [C][C] Q K^T
constexpr uint32_t kOffBW = kOffWQ + 3 * kWQBlock;   // bf16 [C][C] row-major (32 B rows)
constexpr uint32_t kOffBU = kOffWQ + 4 * kWQBlock;
constexpr uint32_t kOffP = kOffBU + kC * kC * 2;
constexpr uint32_t kOffHdr = kOffP + kC * kC * 2;
constexpr uint32_t kStage = 26624;
static_assert(kOffSqk + kC * kC * 4 <= kOffWQ + 2 * kWQBlock + kC * 128, "scratch in -W rows");
static_assert(kOffBW + kC * kC * 2 <= kOffWQ + 3 * kWQBlock + kC * 128, "scratch in -W rows");
static_assert(kOffHdr + 256 <= kStage && kStage % 1024 == 0, "stage layout");
__host__ __device__ constexpr uint32_t q_box(int b) { return b == 0 ? kOffQ0 : kOffQ1; }
constexpr uint32_t kOffBar = kNS * kStage;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // + alignment slack

// core-matrix (no swizzle) K-major layout of a C x C bf16 operand [n][k]
__device__ __forceinline__ uint32_t cc_off(int n, int k) {
    return core_off((uint32_t)n, (uint32_t)k * 2u, (kC / 8) * 128u, 128u);
}

struct Hdr {
    float G[kC];       // in-tile cumulative log-decay (padded past the end with the last value)
    float beta[kC];    // write strengths (0 past the end)
    float eR[kC];      // exp(G_C - G_i)
    float gam;         // exp(G_C), the tile's decay
    int len;
};

enum Mode : int { kModeOut = 0, kModeB = 1, kModeM = 2 };

struct TcArgs {
    const float *G;
    const __nv_bfloat16 *beta;   // [rows][H] write strengths
    const float *h0;
    void *out;
    float *hT;
    float *Hin;   // [segs][H][D][D] entering states (pass C, s >= 1)
    float *Bs;    // [segs][H][D][D] transition offsets
    float *Ms;    // [segs][H][D][D] transition matrices
    const int *first;   // [segs][H] first tile of the B stream (truncated transition)
    const int *mneed;   // [segs][H] 1 if the transition matrix is not negligible
    Plan plan;
    int H;
    int64_t T_total;
    int mode;
    int *status;
    uint64_t wait_ns;   // limit of every pipeline wait
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Per-tile clock stamps of CTA (0, 0) for performance work; compiled only with
// -DGDR_TC_TRACE (then gdr_tc_trace_buffer points at a [3 modes][64 tiles][16] buffer).
#ifdef GDR_TC_TRACE
}  // namespace
__device__ long long *gdr_tc_trace_buffer = nullptr;
__device__ int gdr_tc_trace_first = 0;
namespace {
#define TC_TRACE(c, slot)                                                                    \
    do {                                                                                     \
        long long *tb_ = gdr_tc_trace_buffer;                                                \
        const int r_ = (c) - gdr_tc_trace_first;                                             \
        if (tb_ && blockIdx.x == 0 && blockIdx.y == 0 && r_ >= 0 && r_ < 64)                 \
            tb_[(args.mode * 64 + r_) * 16 + (slot)] = clock64();                           \
    } while (0)
#else
#define TC_TRACE(c, slot) \
    do {                  \
    } while (0)
#endif

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
    uint64_t *bar_a = bar_fin + 1;       // [1] A operands of the tile written (4 state warps)
    uint64_t *bar_init = bar_a + 1;      // [1] state initialised (4 state warps)
    uint32_t *tmem_slot = (uint32_t *)(bar_init + 1);
    volatile int *abort_prep = (volatile int *)(tmem_slot + 1);   // set by prep warps
    volatile int *abort_state = abort_prep + 1;                   // set by state warps only

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mode = args.mode;
    const int h = blockIdx.y;
    SegInfo si;
    if (!seg_info(args.plan, blockIdx.x, si)) return;
    const bool last_seg = si.s == si.nseg - 1;
    const int H = args.H;
    const int64_t gsh = (int64_t)blockIdx.x * H + h;   // (global segment, head) slot
    if (mode != kModeOut) {  // transition passes: only non-last segments
        if (last_seg) return;
        if (mode == kModeM && (si.s == 0 || args.mneed[gsh] == 0)) return;
    }
    // the B stream may start late: earlier tiles' contributions to the segment's
    // end state are attenuated below the truncation bound
    const bool truncated = mode == kModeB && args.first[gsh] > si.c0;
    if (truncated) si.c0 = args.first[gsh];
    const float *h_in = nullptr;
    float *h_out = nullptr;
    if (mode == kModeOut) {
        if (si.s == 0) {
            h_in = args.h0 ? args.h0 + ((int64_t)si.n * H + h) * kD * kD : nullptr;
        } else {
            // the previous segment's transition: with no (or a negligible) matrix the
            // entering state is its offset B, which the combine does not copy
            const int64_t prev = gsh - H;
            h_in = (si.s == 1 || args.mneed[prev] == 0) ? args.Bs + prev * kD * kD
                                                         : args.Hin + gsh * kD * kD;
        }
        h_out = (last_seg && args.hT) ? args.hT + ((int64_t)si.n * H + h) * kD * kD : nullptr;
    } else if (mode == kModeB) {
        h_in = (si.s == 0 && args.h0 && !truncated) ? args.h0 + ((int64_t)si.n * H + h) * kD * kD
                                                      : nullptr;
        h_out = args.Bs + gsh * kD * kD;
    } else {
        h_out = args.Ms + gsh * kD * kD;
    }
    const bool use_v = mode != kModeM, use_q = mode == kModeOut;
    const int nch = (int)(si.c1 - si.c0);
    constexpr unsigned kFull = 0xffffffffu;
    // (checking build) the segment's tokens and its sequence lie inside the tensors; a
    // failed check leaves the CTA's work undone (block-uniform, before any barrier)
    if (!GDR_INBOUNDS(si.n < args.plan.N && h < H && si.tok0 >= 0 && si.tok0 + si.len <= args.T_total &&
                      si.c0 >= 0 && si.c1 * kC <= si.len + kC - 1))
        return;

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
        mbar_init(&bar_a[0], 4);
        mbar_init(&bar_init[0], 4);
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

    if (warp >= 4 && warp < 4 + kNS) {
        // ============================ prep warps ============================
        const int pw = warp - 4;
        float *Skk = (float *)(smem + pw * kStage + kOffSkk);
        float *Sqk = (float *)(smem + pw * kStage + kOffSqk);
        uint8_t *BW = smem + pw * kStage + kOffBW;
        const uint32_t tx_bytes = 2 * kBox * (1 + (use_v ? 1 : 0) + (use_q ? 1 : 0));
        int pend_st = -1;          // stage whose TMA is issued but not yet seen complete
        uint32_t pend_ph = 0;
        // prep warp pw owns stage pw and tiles pw, pw + kNS, ...: every wait on a
        // stage barrier is for the phase right after the one this warp consumed
        for (int c = pw; c < nch; c += kNS) {
            if (__any_sync(kFull, *abort_prep != 0 || *abort_state != 0)) break;
            if (lane == 0) TC_TRACE(c, 0);
            const int st = pw;
            const uint32_t ph = (uint32_t)(c / kNS) & 1u;
            uint8_t *stg = smem + st * kStage;
            Hdr *hdr = (Hdr *)(stg + kOffHdr);
            const int64_t tc = si.c0 + c;                  // tile index within the sequence
            const int64_t t0 = si.tok0 + tc * kC;         // first token row
            const int len = (int)min((int64_t)kC, si.len - tc * kC);
            // gates of the tile (issued before the waits)
            float g_i = 0.f, b_i = 0.f;
            if (lane < kC && GDR_INBOUNDS(t0 >= 0 && t0 + len <= args.T_total && len >= 1)) {
                const int i = min(lane, len - 1);
                g_i = args.G[(int64_t)h * args.T_total + t0 + i];
                b_i = lane < len ? __bfloat162float(args.beta[(t0 + lane) * H + h]) : 0.f;
            }
            if (c >= kNS && !__all_sync(kFull, mbar_wait(&bar_free[st], ph ^ 1u, args.wait_ns))) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_prep = 1;
                break;
            }
            if (lane == 0) {
                TC_TRACE(c, 1);
                mbar_arrive_expect_tx(&bar_full[st], tx_bytes);
                tma_load_3d(stg + kOffK, &tmK, 0, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffK + kBox, &tmK, 64, h, (int)t0, &bar_full[st]);
                if (use_v) {
                    tma_load_3d(stg + kOffV, &tmV, 0, h, (int)t0, &bar_full[st]);
                    tma_load_3d(stg + kOffV + kBox, &tmV, 64, h, (int)t0, &bar_full[st]);
                }
                if (use_q) {
                    tma_load_3d(stg + kOffQ0, &tmQ, 0, h, (int)t0, &bar_full[st]);
                    tma_load_3d(stg + kOffQ1, &tmQ, 64, h, (int)t0, &bar_full[st]);
                }
            }
            pend_st = st;
            pend_ph = ph;
            {
                const float g_last = __shfl_sync(kFull, g_i, kC - 1);
                if (lane < kC) {
                    hdr->G[lane] = g_i;
                    hdr->beta[lane] = b_i;
                    hdr->eR[lane] = __expf(fminf(g_last - g_i, 0.f));
                }
                if (lane == 0) {
                    hdr->len = len;
                    hdr->gam = __expf(g_last);
                }
            }
            if (!__all_sync(kFull, mbar_wait(&bar_full[st], ph, args.wait_ns))) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_prep = 1;
                break;
            }
            pend_st = -1;
            if (lane == 0) TC_TRACE(c, 2);
            // rows past the end of the sequence hold another sequence's tokens: zero them
            if (len < kC) {
                const int nt = 1 + (use_v ? 1 : 0) + (use_q ? 1 : 0);
                const int nrow = kC - len;
                for (int e = lane; e < nt * 2 * nrow * 8; e += 32) {
                    const int chunk16 = e & 7, rem = e >> 3;
                    const int row = len + rem % nrow, box = (rem / nrow) & 1;
                    const int tsel = rem / (nrow * 2);
                    const uint32_t toff = tsel == 0 ? kOffK + box * kBox
                                          : ((tsel == 1 && use_v) ? kOffV + box * kBox : q_box(box));
                    *(uint4 *)(stg + toff + sw128_off(row, chunk16 * 16)) = make_uint4(0, 0, 0, 0);
                }
            }
            __syncwarp();
            // ---- Gram matrices Skk = K K^T, Sqk = Q K^T (mma.sync, bf16 -> fp32)
            float skk[2][4] = {}, sqk[2][4] = {};
            {
                const int r = lane & 15, half = lane >> 4;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = sw128_off(r, 32 * (ks & 3) + 16 * half);
                    uint32_t kf[4];
                    ldsm_x4(smem_u32(stg + kOffK + (ks >> 2) * kBox + off), kf);
                    mma16816(skk[0], kf, kf[0], kf[2]);
                    mma16816(skk[1], kf, kf[1], kf[3]);
                    if (use_q) {
                        uint32_t qf[4];
                        ldsm_x4(smem_u32(stg + q_box(ks >> 2) + off), qf);
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
                    *(float2 *)&Skk[r0 * kC + col] = make_float2(skk[nt][0], skk[nt][1]);
                    *(float2 *)&Skk[(r0 + 8) * kC + col] = make_float2(skk[nt][2], skk[nt][3]);
                    *(float2 *)&Sqk[r0 * kC + col] = make_float2(sqk[nt][0], sqk[nt][1]);
                    *(float2 *)&Sqk[(r0 + 8) * kC + col] = make_float2(sqk[nt][2], sqk[nt][3]);
                }
            }
            __syncwarp();
            if (lane == 0) TC_TRACE(c, 3);
            // ---- A (in place over Skk) and P (bf16, core-matrix layout in the stage):
            // lane -> row i = lane / 2, columns 8 (lane & 1) .. + 7
            {
                const int i = lane >> 1, j0 = 8 * (lane & 1);
                const float Gi = hdr->G[i], bi = hdr->beta[i];
                const float4 k0 = *(const float4 *)&Skk[i * kC + j0];
                const float4 k1 = *(const float4 *)&Skk[i * kC + j0 + 4];
                const float sk[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
                float a[8], pv[8];
                float sq[8];
                if (use_q) {
                    const float4 q0 = *(const float4 *)&Sqk[i * kC + j0];
                    const float4 q1 = *(const float4 *)&Sqk[i * kC + j0 + 4];
                    sq[0] = q0.x; sq[1] = q0.y; sq[2] = q0.z; sq[3] = q0.w;
                    sq[4] = q1.x; sq[5] = q1.y; sq[6] = q1.z; sq[7] = q1.w;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = j0 + u;
                    const float dg = __expf(fminf(Gi - hdr->G[j], 0.f));
                    a[u] = j < i ? bi * dg * sk[u] : 0.f;
                    pv[u] = (use_q && j <= i) ? sq[u] * dg : 0.f;
                }
                __syncwarp();   // every lane has read its Skk row segment before it is overwritten
                *(float4 *)&Skk[i * kC + j0] = make_float4(a[0], a[1], a[2], a[3]);
                *(float4 *)&Skk[i * kC + j0 + 4] = make_float4(a[4], a[5], a[6], a[7]);
                if (use_q)
                    *(uint4 *)(stg + kOffP + cc_off(i, j0)) =
                        make_uint4(pack_bf16(pv[0], pv[1]), pack_bf16(pv[2], pv[3]),
                                   pack_bf16(pv[4], pv[5]), pack_bf16(pv[6], pv[7]));
            }
            __syncwarp();
            // ---- T = (I + A)^{-1}, one column per lane (forward substitution over
            // broadcast row loads); lanes 16..31 repeat lanes 0..15
            {
                const int j = lane & (kC - 1);
                float tcol[kC];
#pragma unroll
                for (int i = 0; i < kC; ++i) {
                    float row[kC];
#pragma unroll
                    for (int q4 = 0; q4 < kC / 4; ++q4) {
                        const float4 v4 = *(const float4 *)&Skk[i * kC + 4 * q4];
                        row[4 * q4] = v4.x;
                        row[4 * q4 + 1] = v4.y;
                        row[4 * q4 + 2] = v4.z;
                        row[4 * q4 + 3] = v4.w;
                    }
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < i; ++m) acc = fmaf(row[m], tcol[m], acc);
                    tcol[i] = (i < j) ? 0.f : ((i == j) ? 1.f : -acc);
                }
                const float bj = hdr->beta[j];
                if (lane < kC) {          // Bu = T diag(beta)
                    if (use_v)
#pragma unroll
                        for (int i = 0; i < kC; ++i)
                            *(__nv_bfloat16 *)(stg + kOffBU + cc_off(i, j)) = __float2bfloat16_rn(tcol[i] * bj);
                } else {                  // -Bw = -T diag(beta e^G), row-major for ldmatrix
                    const float bej = -bj * __expf(hdr->G[j]);
#pragma unroll
                    for (int i = 0; i < kC; ++i)
                        *(__nv_bfloat16 *)(BW + i * 32 + j * 2) = __float2bfloat16_rn(tcol[i] * bej);
                }
            }
            __syncwarp();
            if (lane == 0) TC_TRACE(c, 4);
            // ---- rows [C, 2C) of WQ: diag(e^G) Q in tf32 (reads the raw Q tile, which
            // the -W rows below overwrite)
            if (use_q) {
                const int i = lane >> 1, hb = lane & 1;
                const float eg = __expf(hdr->G[i]);
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint4 raw = *(const uint4 *)(stg + q_box(hb) + sw128_off(i, 16 * c8));
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
            __syncwarp();
            if (lane == 0) TC_TRACE(c, 5);
            // ---- -W = (-Bw) K (mma.sync) -> rows [0, C) of WQ in tf32
            {
                uint32_t af[4];
                ldsm_x4(smem_u32(BW + (lane & 15) * 32 + (lane >> 4) * 16), af);
                __syncwarp();   // Bw is read before the -W rows (which hold it) are written
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
                        *(float2 *)(base + sw128_off(i0, (d & 31) * 4)) = make_float2(w[0], w[1]);
                        *(float2 *)(base + sw128_off(i0 + 8, (d & 31) * 4)) = make_float2(w[2], w[3]);
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) TC_TRACE(c, 6);
            if (lane == 0) mbar_arrive(&bar_prep[st]);
        }
        // never leave with a tile copy still in flight
        if (pend_st >= 0) {
            if (!__all_sync(kFull, mbar_wait(&bar_full[pend_st], pend_ph, kDrainNs)) && lane == 0)
                set_status(args.status, GDR_ERR_TIMEOUT);
            __syncwarp();
        }
    } else if (warp == 4 + kNS) {
        // ============================ MMA issuer ============================
        // One thread issues every tcgen05 MMA of the CTA, in tile order, so the
        // tensor pipe executes them in that order: a tile's front MMAs may read
        // the state the previous tile's update MMA writes without waiting for it.
        // The warp runs the loop converged (operand descriptors are warp-uniform)
        // and elects the issuing lane at each group of MMAs.
        {
            const uint32_t id_u = instr_desc(128, kC, 1, true, false);
            const uint32_t id_x = instr_desc(128, use_q ? 2 * kC : kC, 2, false, false);
            const uint32_t id_h = instr_desc(128, kD, 1, false, true);
            const uint32_t id_o = instr_desc(128, kC, 1, false, false);
            // operand descriptors of stage 0; stage st adds st * kStage to the
            // start-address field (shared addresses are below 256 KiB: no carry)
            const uint32_t s0 = smem_u32(smem);
            const uint64_t dV = smem_desc(s0 + kOffV, kBox, 1024, kSw128);
            const uint64_t dK = smem_desc(s0 + kOffK, kBox, 1024, kSw128);
            const uint64_t dBU = smem_desc(s0 + kOffBU, 128, (kC / 8) * 128, kSwNone);
            const uint64_t dP = smem_desc(s0 + kOffP, 128, (kC / 8) * 128, kSwNone);
            const uint64_t dWQ = smem_desc(s0 + kOffWQ, 16, 1024, kSw128);
            bool ok = nch == 0 || __all_sync(kFull, mbar_wait(&bar_init[0], 0, args.wait_ns));
            for (int c = 0; c < nch && ok; ++c) {
                if (__any_sync(kFull, *abort_state != 0 || *abort_prep != 0)) {
                    ok = false;
                    break;
                }
                const int st = c % kNS, buf = c & 1;
                const uint64_t so = (uint64_t)((st * kStage) >> 4);   // stage offset in descriptor units
                const uint32_t cb = kColB + buf * kColBuf;
                if (!__all_sync(kFull, mbar_wait(&bar_prep[st], (uint32_t)(c / kNS) & 1u, args.wait_ns))) {
                    ok = false;
                    break;
                }
                if (lane == 0) TC_TRACE(c, 14);
                tc_fence_after();
                // front: U^T and [-W ; Qt] H^ into buffer c & 1
                if (elect_one()) {
                    if (use_v)
                        mma_f16_ss(tm + cb, dV + so, dBU + so, id_u, 0);
                    // K-step s8 of [-W ; Qt] starts (s8 / 4) column blocks and 32 (s8 % 4)
                    // bytes in: added to the start-address field (shared addresses are
                    // below 256 KiB, so the 14-bit field never carries)
                    const uint64_t dwq = dWQ + so;
#pragma unroll
                    for (int s8 = 0; s8 < kD / 8; ++s8)
                        mma_tf32_ts(tm + cb + kC, tm + kColH + 8 * s8,
                                    dwq + (uint64_t)(((s8 >> 2) * kWQBlock + 32 * (s8 & 3)) >> 4), id_x, s8 > 0);
                    mma_commit(&bar_x[buf]);
                }
                __syncwarp();
                if (lane == 0) TC_TRACE(c, 15);
                // back: the state update and the in-tile output term, once the
                // state warps have written this tile's A operands
                if (!__all_sync(kFull, mbar_wait(&bar_a[0], (uint32_t)c & 1u, args.wait_ns))) {
                    ok = false;
                    break;
                }
                if (lane == 0) TC_TRACE(c, 11);
                tc_fence_after();
                if (elect_one()) {
                    mma_f16_ts(tm + kColH, tm + kColA, dK + so, id_h, 1);
                    if (use_q)
                        mma_f16_ts(tm + cb + 2 * kC, tm + kColA + kC / 2,
                                   dP + so, id_o, 1);
                    mma_commit(&bar_free[st]);
                }
                __syncwarp();
                if (lane == 0) TC_TRACE(c, 12);
            }
            // the state warps' drain waits on the last tile's MMAs; on a failure, no
            // tensor-core operation may still run when the TMEM is released
            if (elect_one()) {
                if (ok) mma_commit(&bar_h[0]);
                mma_commit(&bar_fin[0]);
            }
            __syncwarp();
            if (!ok) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_state = 1;
            }
            __all_sync(kFull, mbar_wait(&bar_fin[0], 0, kDrainNs));
        }
        __syncwarp();
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
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_init[0]);
        // One tile's output for this warp's 32 value columns: per token row, the
        // warp writes 64 contiguous bytes.
        const int64_t orow = (int64_t)H * kD;   // elements between token rows
        auto store_out = [&](const uint32_t (&o)[kC], int len, int64_t t0, float scale) {
            if (!GDR_INBOUNDS(t0 >= 0 && t0 + len <= args.T_total)) return;
            __nv_bfloat16 *out = (__nv_bfloat16 *)args.out + (t0 * H + h) * kD + e;
            if (len == kC) {
#pragma unroll
                for (int i = 0; i < kC; ++i) out[i * orow] = __float2bfloat16_rn(__uint_as_float(o[i]) * scale);
            } else {
#pragma unroll
                for (int i = 0; i < kC; ++i)
                    if (i < len) out[i * orow] = __float2bfloat16_rn(__uint_as_float(o[i]) * scale);
            }
        };
        float Gamma = 1.f;                // H = Gamma * H^
        float gamma_prev = 1.f;           // Gamma of the previous tile's output
        int64_t t0_prev = 0;
        int len_prev = 0;
        int done = 0;
        for (int c = 0; c < nch; ++c) {
            if (__any_sync(kFull, *abort_state != 0 || *abort_prep != 0)) break;
            const int st = c % kNS;
            const uint32_t ph = (uint32_t)(c / kNS) & 1u;
            const int buf = c & 1;
            uint8_t *stg = smem + st * kStage;
            const uint32_t cb = kColB + buf * kColBuf;
            if (lane == 0) TC_TRACE(c, 8);
            // the tile's header and its front MMAs (a missing result times out)
            const bool okw = mbar_wait(&bar_prep[st], ph, args.wait_ns) &&
                             mbar_wait(&bar_x[buf], (uint32_t)(c >> 1) & 1u, args.wait_ns);
            if (!__all_sync(kFull, okw)) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_state = 1;
                break;
            }
            tc_fence_after();
            if (lane == 0) TC_TRACE(c, 9);
            const Hdr *hdr = (const Hdr *)(stg + kOffHdr);
            const int len_c = hdr->len;
            const float gam = hdr->gam;
            float Gp = Gamma * gam;                  // Gamma after this tile, if not reset
            const bool renorm = !(Gp >= kGammaMin);  // also catches gam == 0
            if (renorm) {
                // fold Gp into H^ and reset Gamma to 1; no MMA reads or writes H^ now
                // (this tile's front is done, its update not issued)
                for (int d0 = 0; d0 < kD; d0 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tm + lane_base + kColH + d0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        r[j] = __float_as_uint(__uint_as_float(r[j]) * Gp);
                    tmem_st16(tm + lane_base + kColH + d0, r);
                }
                Gp = 1.f;
            }
            const float s2 = __frcp_rn(Gp);               // the tile's writes enter H^ scaled by 1 / Gamma
            // [U | -W H^] of this tile, and the previous tile's output (complete with
            // this tile's bar_x; read before the arrive, since the next front MMA
            // overwrites its buffer)
            uint32_t ux[2 * kC], orr[kC];
            tmem_ld32(tm + lane_base + cb, ux);
            if (use_q && c > 0) tmem_ld16(tm + lane_base + kColB + (buf ^ 1) * kColBuf + 2 * kC, orr);
            tmem_ld_wait();
            uint32_t a2[kC / 2], a3[kC / 2];
            const float inv_g = __frcp_rn(Gamma);
#pragma unroll
            for (int i = 0; i < kC; i += 4) {
                const float4 e4 = *(const float4 *)&hdr->eR[i];
                float dl[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    dl[u] = Gamma * __uint_as_float(ux[kC + i + u]);
                    if (use_v) dl[u] += __uint_as_float(ux[i + u]);
                }
                a2[i / 2] = pack_bf16(dl[0] * (e4.x * s2), dl[1] * (e4.y * s2));
                a2[i / 2 + 1] = pack_bf16(dl[2] * (e4.z * s2), dl[3] * (e4.w * s2));
                a3[i / 2] = pack_bf16(dl[0] * inv_g, dl[1] * inv_g);
                a3[i / 2 + 1] = pack_bf16(dl[2] * inv_g, dl[3] * inv_g);
            }
            tmem_st8(tm + lane_base + kColA, a2);
            if (use_q) tmem_st8(tm + lane_base + kColA + kC / 2, a3);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_a[0]);
            if (lane == 0) TC_TRACE(c, 10);
            if (use_q && c > 0) store_out(orr, len_prev, t0_prev, gamma_prev);
            if (lane == 0) TC_TRACE(c, 13);
            gamma_prev = Gamma;
            t0_prev = si.tok0 + (si.c0 + c) * kC;
            len_prev = len_c;
            Gamma = Gp;
            done = c + 1;
        }
        // drain: the last tile's output, then the final state
        bool ok = done == nch;
        if (ok && nch > 0) ok = __all_sync(kFull, mbar_wait(&bar_h[0], 0, args.wait_ns));
        ok = __all_sync(kFull, ok && *abort_state == 0);
        tc_fence_after();
        if (ok && use_q && nch > 0) {
            uint32_t orr[kC];
            tmem_ld16(tm + lane_base + kColB + ((nch - 1) & 1) * kColBuf + 2 * kC, orr);
            tmem_ld_wait();
            store_out(orr, len_prev, t0_prev, gamma_prev);
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
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// transition truncation: for each non-last segment, the first tile r such that
// the bound on the state transition from the start of tile r to the segment's
// end is at most exp(-kTruncLog) = 2^-64.  One token multiplies the state by
// Phi_t = alpha_t (I - beta_t k_t k_t^T), whose norm is
// alpha_t max(1, |1 - beta_t |k_t|^2|) (the erase factor's eigenvalues are 1
// and 1 - beta |k|^2), so the log of the bound over a tile is its summed
// log-decay plus the tokens' log max(1, |1 - beta |k|^2|).  Everything that
// enters the recurrence before tile r then reaches the segment's end
// attenuated by at least 2^-64 relative to the state at tile r, so the
// segment's offset B is computed from a zero state at r and its transition
// matrix M is taken as zero.  When no such r exists the full transition is
// computed.  [P3 §3.1-3.2: the state passed from chunk to chunk]
//
// One warp per (segment, head), walking back from the segment's end.  The decay
// alone gives a weaker bound (erase factors are >= 1), so a first walk over G
// (32 tiles per step) finds whether the horizon can fall inside the segment at
// all, and where; only then are keys read, from the segment's end back to that
// horizon or a little past it (two tiles per step, a lane per token).  A walk that
// does not cross within a few times the first horizon's distance gives up and the
// full transition is used, which is always exact.
// ---------------------------------------------------------------------------
constexpr float kTruncLog = 44.3614195558365f;   // 64 ln 2

// Inclusive scan of x over the lanes of a warp.
__device__ __forceinline__ float warp_scan(float x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// log of the decay of one tile (its summed log-decay, the last in-tile cumsum)
__device__ __forceinline__ float tile_log_decay(const float *G, const SegInfo &si, int64_t c, int h,
                                                int64_t T_total) {
    const int len = (int)min((int64_t)kC, si.len - c * kC);
    const int64_t row0 = si.tok0 + c * kC;
    if (!GDR_INBOUNDS(len >= 1 && row0 >= 0 && row0 + len <= T_total)) return 0.f;
    return G[(int64_t)h * T_total + row0 + len - 1];
}

__global__ void __launch_bounds__(128)
tc_horizon_kernel(const float *G, const __nv_bfloat16 *beta, const __nv_bfloat16 *k, Plan p, int H,
                  int64_t T_total, int64_t nslots, int *first, int *mneed, int truncate) {
    const int64_t slot = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    constexpr unsigned kFull = 0xffffffffu;
    if (slot >= nslots) return;   // warp-uniform
    const int64_t gseg = slot / H;
    const int h = (int)(slot % H);
    SegInfo si;
    if (!seg_info(p, gseg, si)) return;
    int r = (int)si.c0;
    int need = 1;
    if (truncate) {
        // pass 0, the decay alone, 32 tiles per step (lane j: the j-th tile back): is
        // there a horizon inside the segment at all, and where (r0)?
        int64_t r0 = -1;
        {
            float acc = 0.f;
            for (int64_t cs = si.c1 - 1; cs >= si.c0 && r0 < 0; cs -= 32) {
                const int64_t c = cs - lane;
                const bool valid = c >= si.c0;
                const float run = acc + warp_scan(valid ? tile_log_decay(G, si, c, h, T_total) : 0.f, lane);
                const unsigned hit = __ballot_sync(kFull, valid && run <= -kTruncLog);
                if (hit) r0 = cs - (__ffs(hit) - 1);
                acc = __shfl_sync(kFull, run, 31);
            }
        }
        // pass 1, with the erase factors (its horizon lies at or before r0), two tiles
        // per step, lane = token (tile cs - lane / 16, token lane % 16); a walk that has
        // not crossed a few segment-end distances past r0 gives up (full transition)
        if (r0 >= 0) {
            const int64_t limit = max(si.c0, r0 - 4 * (si.c1 - r0) - 64);
            float acc = 0.f;
            for (int64_t cs = si.c1 - 1; cs >= limit; cs -= 2) {
                const int64_t c = cs - (lane >> 4);
                const int i = lane & 15;
                float part = 0.f;
                if (c >= limit) {
                    const int len = (int)min((int64_t)kC, si.len - c * kC);
                    const int64_t row = si.tok0 + c * kC + i;
                    if (i < len && GDR_INBOUNDS(row < T_total)) {
                        const uint4 *kp = (const uint4 *)(k + (row * H + h) * kD);
                        float kk = 0.f;
#pragma unroll
                        for (int u = 0; u < kD / 8; ++u) {
                            const uint4 w = kp[u];
                            const __nv_bfloat162 *p2 = (const __nv_bfloat162 *)&w;
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                const float2 f = __bfloat1622float2(p2[m]);
                                kk = fmaf(f.x, f.x, fmaf(f.y, f.y, kk));
                            }
                        }
                        const float e = fabsf(1.f - __bfloat162float(beta[row * H + h]) * kk);
                        if (e > 1.f) part = logf(e);
                    }
                    if (i == 0) part += tile_log_decay(G, si, c, h, T_total);
                }
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);   // per half
                const float t_hi = __shfl_sync(kFull, part, 0), t_lo = __shfl_sync(kFull, part, 16);
                acc += t_hi;
                if (acc <= -kTruncLog) {
                    r = (int)cs;
                    need = 0;
                    break;
                }
                acc += t_lo;
                if (cs - 1 >= limit && acc <= -kTruncLog) {
                    r = (int)(cs - 1);
                    need = 0;
                    break;
                }
            }
        }
    }
    if (lane == 0) {
        first[slot] = r;
        mneed[slot] = need;
    }
}

// ---------------------------------------------------------------------------
// combine: H_in(s+1) = M_s H_in(s) + B_s, serial over the segments of one
// (sequence, head); one block per 32 state columns, fp32 FMA.
// ---------------------------------------------------------------------------
constexpr int kCombCols = 32;

__global__ void __launch_bounds__(256)
tc_combine_kernel(float *Hin, const float *Bs, const float *Ms, const int *mneed, Plan p, int H) {
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
    // Hs holds H_in(s - 1) for this block's columns, or (lazily) it is B of the
    // segment before, still in global memory: a run of negligible transitions
    // costs nothing until a transition that needs H_in arrives
    const float *pending = nullptr;
    for (int s = 1; s < nseg; ++s) {
        const int64_t prev = (g0 + s - 1) * H + h, cur = (g0 + s) * H + h;
        if (!GDR_INBOUNDS(cur < p.seg_base[p.N] * H)) return;   // (block-uniform)
        const float *B = Bs + prev * kD * kD;
        float *Hc = Hin + cur * kD * kD;
        if (s == 1 || mneed[prev] == 0) {
            // M of the previous segment is negligible (or s = 1): H_in(s) = B(s-1),
            // which the output pass reads in place
            pending = B;
            continue;
        }
        if (pending) {
            for (int e = tid; e < kD * kCombCols; e += 256) {
                const int d = e / kCombCols, j = e % kCombCols;
                Hs[e] = pending[d * kD + j0 + j];
            }
            pending = nullptr;
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

// Streaming multiprocessors of the current device, looked up once per device (a
// benign race: concurrent first calls store the same value).
int sm_count() {
    constexpr int kMaxDev = 64;
    static std::atomic<int> cache[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    if (dev >= 0 && dev < kMaxDev) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    if (dev >= 0 && dev < kMaxDev) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

int64_t max_segments(int N, int64_t T_total, int seg_chunks) {
    const int64_t tiles = (T_total + kC - 1) / kC + N;
    return tiles / seg_chunks + 2 * (int64_t)N + 1;
}

}  // namespace

bool tc_make_map(CUtensorMap *map, const void *base, int H, int64_t rows) {
    return make_map(map, base, H, rows);
}

bool tc_supported(gdr_dtype_t dtype, int dk, int dv, int chunk) {
    static_assert(kC == kTcTile, "tile length");
    return dtype == GDR_BF16 && dk == kD && dv == kD && (chunk == 16 || chunk == 32 || chunk == 64);
}

// Tiles per segment.  The output pass runs one CTA per (segment, head), two per SM,
// and takes as long as its slowest wave.
//   Dense input (N sequences of equal length): the segments per sequence s that
//   minimise waves(s) x tiles per segment, with waves(s) = ceil(N H s / slots), plus a
//   small charge per extra segment (its transition pass and start-up).
//   Packed input (lengths unknown on the host): segments of a quarter of an even share
//   of the tiles, so that the block scheduler balances the many unequal CTAs.
int tc_segment_chunks(int N, int H, int64_t T_total, int C, bool varlen) {
    if (const char *env = std::getenv("GDR_TC_SEG_CHUNKS")) {
        const int v = std::atoi(env);
        if (v > 0) return v;
    }
    constexpr int64_t kMinTiles = 32;
    const int64_t slots = 2 * (int64_t)sm_count();
    if (varlen) {
        const int64_t tiles = (T_total + C - 1) / C + N;
        const int64_t sc = (tiles * H + 4 * slots - 1) / (4 * slots);
        return (int)std::max<int64_t>(kMinTiles, std::min<int64_t>(sc, 1 << 30));
    }
    const int64_t L = (T_total / std::max(N, 1) + C - 1) / C;   // tiles per sequence
    if (L <= kMinTiles) return (int)kMinTiles;
    int64_t best_s = 1;
    double best = 1e300;
    const int64_t s_max = std::min<int64_t>(L / kMinTiles, 4096);
    for (int64_t s = 1; s <= s_max; ++s) {
        const int64_t ctas = (int64_t)N * H * s;
        const int64_t waves = (ctas + slots - 1) / slots;
        const int64_t per = (L + s - 1) / s;
        const double cost = (double)waves * (double)per + 4.0 * (double)waves * (double)(s > 1);
        if (cost < best) {
            best = cost;
            best_s = s;
        }
    }
    return (int)((L + best_s - 1) / best_s);
}

size_t tc_workspace_bytes(int N, int H, int64_t T_total, int C, bool varlen) {
    const int sc = tc_segment_chunks(N, H, T_total, C, varlen);
    const int64_t nseg = max_segments(N, T_total, sc);
    const size_t per = (size_t)nseg * H * kD * kD * sizeof(float);
    const size_t flags = (size_t)nseg * H * sizeof(int);
    return 3 * ((per + 255) / 256 * 256) + 2 * ((flags + 255) / 256 * 256);
}

cudaError_t launch_tc_forward(const void *q, const void *k, const void *v, const float *G,
                              const void *beta, const float *h0, void *out, float *hT, Plan plan,
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
    a.beta = (const __nv_bfloat16 *)beta;
    a.h0 = h0;
    a.out = out;
    a.hT = hT;
    a.Hin = (float *)scratch;
    a.Bs = (float *)((char *)scratch + per);
    a.Ms = (float *)((char *)scratch + 2 * per);
    const size_t flags_b = ((size_t)nseg * H * sizeof(int) + 255) / 256 * 256;
    int *first = (int *)((char *)scratch + 3 * per);
    int *mneed = (int *)((char *)scratch + 3 * per + flags_b);
    a.first = first;
    a.mneed = mneed;
    a.plan = plan;
    a.H = H;
    a.T_total = T_total;
    a.status = status;
    const char *exact = std::getenv("GDR_TC_EXACT");
    const int truncate = (exact && std::atoi(exact) != 0) ? 0 : 1;
    a.wait_ns = kWaitNs;
    if (const char *w = std::getenv("GDR_TC_WAIT_NS")) {   // test hook: shorter pipeline waits
        const long long v = std::atoll(w);                  // (0: look once, never wait)
        if (v >= 0 && (uint64_t)v < kWaitNs) a.wait_ns = (uint64_t)v;
    }
    {
        ProfScope prof(stream, "tc_horizon_kernel");
        const int64_t nslots = nseg * H;   // one warp each
        tc_horizon_kernel<<<(unsigned)((nslots + 3) / 4), 128, 0, stream>>>(
            G, (const __nv_bfloat16 *)beta, (const __nv_bfloat16 *)k, plan, H, T_total, nslots, first, mneed,
            truncate);
        count_launch();
    }
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
            a.Hin, a.Bs, a.Ms, mneed, plan, H);
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

#ifdef GDR_TC_TRACE
extern "C" __attribute__((visibility("default"))) int gdr_tc_trace_set(long long *buf, int first) {
    if (cudaMemcpyToSymbol(gdr::gdr_tc_trace_buffer, &buf, sizeof(buf)) != cudaSuccess) return 1;
    return cudaMemcpyToSymbol(gdr::gdr_tc_trace_first, &first, sizeof(first)) == cudaSuccess ? 0 : 1;
}
#endif
