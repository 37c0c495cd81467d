// gdr_tc_adj.cu -- the adjoint state chain of the chunked backward on the
// 5th-generation tensor cores (tcgen05): bf16 inputs, dk = dv = 128, tiles of 16,
// bounded gate, one decay per token or one per key channel.
//
// The chain runs the tiles of one (segment, head) in reverse.  With dH1 the gradient
// of the loss with respect to a tile's end state, the tile's in-tile cumulative
// log-decay G (per key channel), gamma = e^{G_C}, the factored decays Kt = K (.) e^G,
// Kh = K (.) e^-G, Qt = Q (.) e^G and
//   A = beta (.) strict_lower(Kt Kh^T),  S = lower(Qt Kh^T),
//   Bu = (I + A)^{-1} diag(beta),        W = Bu Kt,
// the gradient with respect to the tile's entering state is [P1 §3.2, P2 §2.1, P3 §3.1]
//   X   = diag(gamma) dH1                     (the decay of every key channel)
//   dD  = S^T dO + Ke dH1 = S^T dO + Kh X     (Ke = Kh (.) gamma)
//   dH0 = X + Qt^T dO - W^T dD.
// The gradient lives in the tensor memory, transposed (lane = value index e, column =
// key index d), as the fp32 accumulator of the products that update it:
//   state warps   X^T = dH1^T diag(gamma)       a pass over the tensor memory; X also
//                                              goes out in bf16 for the tile kernel
//   tensor cores  dD^T  = dO^T S + X^T Kh^T     kind::f16, then kind::tf32 with the
//                                              state as the A operand (16 K-steps)
//   state warps   dD^T -> bf16                 the A operand of the next product; dD
//                                              also goes out (fp32) for the tile kernel
//   tensor cores  dH0^T = X^T + dO^T Qt + dD^T (-W)   kind::f16, into the state
// Every product that reads the state waits (on an mbarrier) for the pass that wrote
// it, and the pass waits for the products that wrote it before.
//
// Roles (288 threads, two CTAs per SM): warps 0-3 own the state's lane quarters; prep
// warp 4 + s owns pipeline stage s and tiles s, s + 4, ... (the TMA loads of K, Q, dO
// and the per-channel gate inputs, the factored tiles, the Gram products and W on
// mma.sync, the substitution); warp 8 issues every tcgen05 MMA from one elected lane.
//
// Segments and warm-ups are those of the mma.sync chain (bwd_adj_chain_kernel): a
// segment's chain starts from a zero gradient at the first tile past its end whose
// transition bound to the segment end is below 2^-64 (or from dhT at the sequence's
// end) and stores X only for its own tiles.
#include <cudaTypedefs.h>

#include <cstdlib>

#include "gdr_bwd_chunk.cuh"
#include "gdr_sm100.cuh"
#include "gdr_tc.cuh"
#include "gdr_tc_prep.cuh"

namespace gdr {

GDR_DEBUG_TU()

namespace {

using namespace sm100;
using namespace tcp;
using bwdc::BcArgs;

constexpr int kD = 128;          // dk = dv
constexpr int kC = 16;           // tile length
constexpr int kNS = 4;           // pipeline stages, one per prep warp
constexpr int kThreads = 32 * (4 + kNS + 1);   // 4 state warps, kNS prep warps, 1 MMA issuer
constexpr uint64_t kWaitNs = 2000000000ull;    // default pipeline wait limit: 2 s
constexpr uint64_t kDrainNs = 2000000000ull;   // drains before exit: 2 s

// TMEM columns
constexpr uint32_t kColH = 0;            // the gradient dH^T (128 fp32 columns)
constexpr uint32_t kColD = 128;          // dD^T (C fp32 columns)
constexpr uint32_t kColA = kColD + kC;   // dD^T in bf16 (C/2 columns)
constexpr uint32_t kTmemCols = 256;
static_assert(kColA + kC / 2 <= kTmemCols, "TMEM budget");

// Shared memory per stage (27 KB: four stages at two CTAs per SM).  [C][128] bf16
// tiles are two 64-column boxes of C rows x 128 B, 128-byte swizzled, as the TMA
// writes them.
constexpr uint32_t kBox = kC * 128;
constexpr uint32_t kOffDO = 0;                   // dO: A operand (MN-major) of dO^T S and dO^T Qt
constexpr uint32_t kOffK = kOffDO + 2 * kBox;    // raw K -> Kt (bf16) -> -W (bf16, B operand)
constexpr uint32_t kOffQ = kOffK + 2 * kBox;     // raw Q -> Qt (bf16, B operand)
constexpr uint32_t kOffG = kOffQ + 2 * kBox;     // raw gate inputs (per channel) -> Kh (bf16)
constexpr uint32_t kOffKH = kOffG + 2 * kBox;    // Kh in tf32: 4 column blocks of C rows x 128 B
constexpr uint32_t kKhBlock = kC * 128;
constexpr uint32_t kOffAm = kOffKH + 4 * kKhBlock;   // A (fp32 [C][C])
constexpr uint32_t kOffBu = kOffAm + kC * kC * 4;    // Bu (bf16 [C][C], 32-byte rows)
constexpr uint32_t kOffST = kOffBu + kC * kC * 2;    // S^T: K-major B operand, core-matrix layout
constexpr uint32_t kOffHdr = kOffST + kC * kC * 2;
constexpr uint32_t kStage = 27648;
constexpr uint32_t kOffBar = kNS * kStage;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;   // + alignment slack

struct Hdr {
    float gam[kD];     // e^{G_C} per key channel
    float beta[kC];    // write strengths (0 past the end)
    int len;           // tokens of the tile
    int emit;          // 1: X goes out (a tile of the segment), 0: a warm-up tile
};
static_assert(kOffHdr + sizeof(Hdr) <= kStage && kStage % 1024 == 0, "stage layout");

struct TaArgs {
    BcArgs A;
    int64_t T_total;
    int64_t max_tiles;   // tiles of the stored-gradient buffer
    int *status;
    uint64_t wait_ns;    // limit of every pipeline wait
};

// byte offset of element (row, col) of a [C][128] bf16 tile
__device__ __forceinline__ uint32_t tile_off(int row, int col) {
    return (uint32_t)(col >> 6) * kBox + sw128_off((uint32_t)row, (uint32_t)(col & 63) * 2u);
}
// S^T[n][k] in the K-major core-matrix layout (8-row groups at 256 B, 16-byte column
// groups at 128 B)
__device__ __forceinline__ uint32_t st_off(int n, int k) {
    return core_off((uint32_t)n, (uint32_t)k * 2u, (kC / 8) * 128u, 128u);
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads, 2)
tc_adj_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmA,
              const TaArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bar_full = (uint64_t *)(smem + kOffBar);
    uint64_t *bar_prep = bar_full + kNS;
    uint64_t *bar_free = bar_prep + kNS;   // the stage's products complete (also: the state updated)
    uint64_t *bar_s = bar_free + kNS;      // [1] state scaled by gamma (4 state warps)
    uint64_t *bar_x = bar_s + 1;           // [1] dD^T complete
    uint64_t *bar_a = bar_x + 1;           // [1] dD^T in bf16 written (4 state warps)
    uint64_t *bar_fin = bar_a + 1;         // [1] every MMA of the CTA complete
    uint32_t *tmem_slot = (uint32_t *)(bar_fin + 1);
    volatile int *abort_prep = (volatile int *)(tmem_slot + 1);   // set by prep warps
    volatile int *abort_state = abort_prep + 1;                   // set by state warps and the issuer
    __shared__ int64_t s_last;

    const BcArgs &A = args.A;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    const int H = A.H;
    const Plan &p = A.p;
    int n;
    int64_t s0, s1;
    if (!bwdc::segment_of(A, blockIdx.x, h, n, s0, s1)) return;
    const int64_t sstart = p.seq_start[n], send = p.seq_start[n + 1], tile0 = p.chunk_base[n];
    const int64_t ntiles = p.chunk_base[n + 1] - tile0;
    if (warp == 0) {
        const int64_t e = bwdc::warm_walk(A.lam, tile0, ntiles, H, h, s1, +1);
        if (lane == 0) s_last = e;
    }
    __syncthreads();
    const int64_t e0 = s_last;   // the chain runs tiles e0 - 1, ..., s0
    const int nch = (int)max((int64_t)0, e0 - s0);
    const size_t sbase = ((size_t)n * H + h) * kD * kD;
    const float *h_in = (e0 == ntiles && A.dhT) ? A.dhT + sbase : nullptr;
    float *h_out = (s0 == 0 && A.dh0) ? A.dh0 + sbase : nullptr;
    constexpr unsigned kFull = 0xffffffffu;
    // (checking build) the segment's tokens and tiles lie inside the tensors; a failed
    // check leaves the CTA's work undone (block-uniform, before any barrier)
    if (!GDR_INBOUNDS(n < p.N && h < H && sstart >= 0 && send <= args.T_total && s0 >= 0 && e0 <= ntiles &&
                      tile0 + ntiles <= args.max_tiles && e0 - s0 < (int64_t)1 << 30))
        return;

    if (tid == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_prep[i], 1);
            mbar_init(&bar_free[i], 1);
        }
        mbar_init(&bar_s[0], 4);
        mbar_init(&bar_x[0], 1);
        mbar_init(&bar_a[0], 4);
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
        prefetch_tensormap(&tmO);
        if (VEC) prefetch_tensormap(&tmA);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;

    if (warp >= 4 && warp < 4 + kNS) {
        // ============================ prep warps ============================
        const int pw = warp - 4;
        const int g = lane >> 2, t = lane & 3;
        // ldmatrix row addresses: lanes 0-7 / 8-15 / 16-23 / 24-31 give the rows of the
        // 8x8 blocks (rows 0-7, cols 0-7) / (8-15, 0-7) / (0-7, 8-15) / (8-15, 8-15)
        const int lr = (lane & 7) + 8 * ((lane >> 3) & 1), lc = lane >> 4;
        int pend_st = -1;          // stage whose TMA is issued but not yet seen complete
        uint32_t pend_ph = 0;
        for (int c = pw; c < nch; c += kNS) {
            if (__any_sync(kFull, *abort_prep != 0 || *abort_state != 0)) break;
            const int st = pw;
            const uint32_t ph = (uint32_t)(c / kNS) & 1u;
            uint8_t *stg = smem + st * kStage;
            Hdr *hdr = (Hdr *)(stg + kOffHdr);
            const int64_t tt = e0 - 1 - c;                // tile index within the sequence
            const int64_t t0 = sstart + tt * kC;          // first token row
            const int len = (int)min((int64_t)kC, send - t0);
            float b_i = 0.f, g_i = 0.f;
            if (lane < len && GDR_INBOUNDS(t0 >= 0 && t0 + len <= args.T_total)) {
                b_i = __bfloat162float(A.beta[(t0 + lane) * H + h]);
                if (!VEC) g_i = -A.b * fast_sigmoid(__bfloat162float(A.a[(t0 + lane) * H + h]));
            }
            if (c >= kNS && !__all_sync(kFull, mbar_wait(&bar_free[st], ph ^ 1u, args.wait_ns))) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_prep = 1;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar_full[st], 2 * kBox * (VEC ? 4 : 3));
                tma_load_3d(stg + kOffDO, &tmO, 0, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffDO + kBox, &tmO, 64, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffK, &tmK, 0, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffK + kBox, &tmK, 64, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffQ, &tmQ, 0, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffQ + kBox, &tmQ, 64, h, (int)t0, &bar_full[st]);
                if (VEC) {
                    tma_load_3d(stg + kOffG, &tmA, 0, h, (int)t0, &bar_full[st]);
                    tma_load_3d(stg + kOffG + kBox, &tmA, 64, h, (int)t0, &bar_full[st]);
                }
            }
            pend_st = st;
            pend_ph = ph;
            if (lane < kC) hdr->beta[lane] = b_i;
            if (lane == 0) {
                hdr->len = len;
                hdr->emit = tt < s1 ? 1 : 0;
            }
            // scalar gate: G_i by a prefix sum over lanes 0..15 (0 past the end)
            float Es = 1.f, Ens = 1.f;
            if (!VEC) {
                float Gs = g_i;
#pragma unroll
                for (int o = 1; o < kC; o <<= 1) {
                    const float y = __shfl_up_sync(kFull, Gs, o);
                    if (lane >= o) Gs += y;
                }
                Es = __expf(Gs);
                Ens = __expf(-Gs);
            }
            if (!__all_sync(kFull, mbar_wait(&bar_full[st], ph, args.wait_ns))) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_prep = 1;
                break;
            }
            pend_st = -1;
            // rows past the end of the sequence hold another sequence's tokens: zero
            // those of dO, K and Q (their gates are taken as 0 below)
            if (len < kC) {
                const int nrow = kC - len;
                for (int e = lane; e < 3 * 2 * nrow * 8; e += 32) {
                    const int chunk16 = e & 7, rem = e >> 3;
                    const int row = len + rem % nrow, box = (rem / nrow) & 1;
                    const int tsel = rem / (nrow * 2);
                    const uint32_t toff = (tsel == 0 ? kOffDO : (tsel == 1 ? kOffK : kOffQ)) + box * kBox;
                    *(uint4 *)(stg + toff + sw128_off(row, chunk16 * 16)) = make_uint4(0, 0, 0, 0);
                }
            }
            __syncwarp();
            // ---- the factored tiles: lane l runs key channels 4l..4l+3 down the tile's
            // tokens.  Kt (bf16) over the raw K, Qt (bf16) over the raw Q, Kh (bf16) over
            // the raw gate inputs, Kh (tf32) into its own area; e^{G_C} to the header
            {
                const int d = 4 * lane;
                const float nb = -A.b;
                float G0 = 0.f, G1 = 0.f, G2 = 0.f, G3 = 0.f;
                const uint32_t kh_off = kOffKH + (uint32_t)(d >> 5) * kKhBlock;
#pragma unroll 4
                for (int i = 0; i < kC; ++i) {
                    const uint32_t off = tile_off(i, d);
                    float E[4], En[4];
                    if (VEC) {
                        if (i < len) {
                            const uint2 raw = *(const uint2 *)(stg + kOffG + off);
                            const float2 x0 = unpack_bf16(raw.x), x1 = unpack_bf16(raw.y);
                            G0 = fmaf(nb, fast_sigmoid(x0.x), G0);
                            G1 = fmaf(nb, fast_sigmoid(x0.y), G1);
                            G2 = fmaf(nb, fast_sigmoid(x1.x), G2);
                            G3 = fmaf(nb, fast_sigmoid(x1.y), G3);
                        }
                        E[0] = __expf(G0);
                        E[1] = __expf(G1);
                        E[2] = __expf(G2);
                        E[3] = __expf(G3);
#pragma unroll
                        for (int u = 0; u < 4; ++u) En[u] = __fdividef(1.f, E[u]);
                    } else {
                        const float ei = __shfl_sync(kFull, Es, i), eni = __shfl_sync(kFull, Ens, i);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            E[u] = ei;
                            En[u] = eni;
                        }
                    }
                    const uint2 kr = *(const uint2 *)(stg + kOffK + off);
                    const uint2 qr = *(const uint2 *)(stg + kOffQ + off);
                    const float2 k01 = unpack_bf16(kr.x), k23 = unpack_bf16(kr.y);
                    const float2 q01 = unpack_bf16(qr.x), q23 = unpack_bf16(qr.y);
                    const float kv[4] = {k01.x, k01.y, k23.x, k23.y};
                    const float qv[4] = {q01.x, q01.y, q23.x, q23.y};
                    float kt[4], kh[4], qt[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        kt[u] = kv[u] * E[u];
                        kh[u] = kv[u] * En[u];
                        qt[u] = qv[u] * E[u];
                    }
                    *(uint2 *)(stg + kOffK + off) = make_uint2(pack_bf16(kt[0], kt[1]), pack_bf16(kt[2], kt[3]));
                    *(uint2 *)(stg + kOffQ + off) = make_uint2(pack_bf16(qt[0], qt[1]), pack_bf16(qt[2], qt[3]));
                    *(uint2 *)(stg + kOffG + off) = make_uint2(pack_bf16(kh[0], kh[1]), pack_bf16(kh[2], kh[3]));
                    *(float4 *)(stg + kh_off + sw128_off((uint32_t)i, (uint32_t)(d & 31) * 4u)) =
                        make_float4(kh[0], kh[1], kh[2], kh[3]);
                }
                if (VEC) {
                    *(float4 *)&hdr->gam[d] = make_float4(__expf(G0), __expf(G1), __expf(G2), __expf(G3));
                } else {
                    const float ec = __shfl_sync(kFull, Es, kC - 1);
                    *(float4 *)&hdr->gam[d] = make_float4(ec, ec, ec, ec);
                }
            }
            __syncwarp();
            // ---- Skk = Kt Kh^T and Sqk = Qt Kh^T over 16-key slabs (bf16 in, fp32 out)
            float skk[2][4] = {}, sqk[2][4] = {};
#pragma unroll 2
            for (int sl = 0; sl < kD / 16; ++sl) {
                const uint32_t off = (uint32_t)(sl >> 2) * kBox +
                                     sw128_off((uint32_t)lr, (uint32_t)(sl & 3) * 32u + 16u * (uint32_t)lc);
                uint32_t ktf[4], khf[4], qtf[4];
                ldsm_x4(smem_u32(stg + kOffK + off), ktf);
                ldsm_x4(smem_u32(stg + kOffG + off), khf);
                ldsm_x4(smem_u32(stg + kOffQ + off), qtf);
                mma16816(skk[0], ktf, khf[0], khf[2]);
                mma16816(skk[1], ktf, khf[1], khf[3]);
                mma16816(sqk[0], qtf, khf[0], khf[2]);
                mma16816(sqk[1], qtf, khf[1], khf[3]);
            }
            // ---- A = beta (.) strict_lower(Skk) (fp32) and S^T = lower(Sqk)^T (bf16, the
            // B operand of dO^T S); skk[nt][r] is (row g + 8 (r >> 1), column 8 nt + 2t + (r & 1))
            {
                float *Am = (float *)(stg + kOffAm);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int i = g + 8 * hr, j0 = 8 * nt + 2 * t;
                        const float bi = hdr->beta[i];
                        const float a0 = j0 < i ? bi * skk[nt][2 * hr] : 0.f;
                        const float a1 = j0 + 1 < i ? bi * skk[nt][2 * hr + 1] : 0.f;
                        *(float2 *)&Am[i * kC + j0] = make_float2(a0, a1);
                        const float p0 = j0 <= i ? sqk[nt][2 * hr] : 0.f;
                        const float p1 = j0 + 1 <= i ? sqk[nt][2 * hr + 1] : 0.f;
                        *(__nv_bfloat16 *)(stg + kOffST + st_off(j0, i)) = __float2bfloat16_rn(p0);
                        *(__nv_bfloat16 *)(stg + kOffST + st_off(j0 + 1, i)) = __float2bfloat16_rn(p1);
                    }
            }
            __syncwarp();
            // ---- T = (I + A)^{-1}, one column per lane (lanes 16..31 repeat 0..15);
            // Bu = T diag(beta) in bf16, row-major
            {
                const int jc = lane & (kC - 1);
                const float *Am = (const float *)(stg + kOffAm);
                float tcol[kC];
#pragma unroll
                for (int i = 0; i < kC; ++i) {
                    float row[kC];
#pragma unroll
                    for (int q4 = 0; q4 < kC / 4; ++q4) {
                        const float4 v4 = *(const float4 *)&Am[i * kC + 4 * q4];
                        row[4 * q4] = v4.x;
                        row[4 * q4 + 1] = v4.y;
                        row[4 * q4 + 2] = v4.z;
                        row[4 * q4 + 3] = v4.w;
                    }
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < i; ++m) acc = fmaf(row[m], tcol[m], acc);
                    tcol[i] = (i < jc) ? 0.f : ((i == jc) ? 1.f : -acc);
                }
                const float bj = hdr->beta[jc];
                if (lane < kC) {
#pragma unroll
                    for (int i = 0; i < kC; ++i)
                        *(__nv_bfloat16 *)(stg + kOffBu + i * 32 + jc * 2) = __float2bfloat16_rn(tcol[i] * bj);
                }
            }
            __syncwarp();
            // ---- -W = -Bu Kt, 16 key columns at a time, in bf16 over Kt (the slab's Kt is
            // read by ldmatrix before its -W is written)
            {
                uint32_t bua[4];
                ldsm_x4(smem_u32(stg + kOffBu + lr * 32 + 16 * lc), bua);
#pragma unroll 2
                for (int sl = 0; sl < kD / 16; ++sl) {
                    const uint32_t off = (uint32_t)(sl >> 2) * kBox +
                                         sw128_off((uint32_t)lr, (uint32_t)(sl & 3) * 32u + 16u * (uint32_t)lc);
                    uint32_t kf[4];
                    ldsm_x4_trans(smem_u32(stg + kOffK + off), kf);
                    float w[2][4] = {};
                    mma16816(w[0], bua, kf[0], kf[1]);
                    mma16816(w[1], bua, kf[2], kf[3]);
                    __syncwarp();
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr)
                            *(uint32_t *)(stg + kOffK + tile_off(g + 8 * hr, 16 * sl + 8 * nt + 2 * t)) =
                                pack_bf16(-w[nt][2 * hr], -w[nt][2 * hr + 1]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
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
        {
            const uint32_t id_s = instr_desc(128, kC, 1, true, false);    // dO^T S
            const uint32_t id_k = instr_desc(128, kC, 2, false, false);   // X^T Kh^T (tf32)
            const uint32_t id_q = instr_desc(128, kD, 1, true, true);     // dO^T Qt
            const uint32_t id_w = instr_desc(128, kD, 1, false, true);    // dD^T (-W)
            const uint32_t s0a = smem_u32(smem);
            const uint64_t dDO = smem_desc(s0a + kOffDO, kBox, 1024, kSw128);
            const uint64_t dQT = smem_desc(s0a + kOffQ, kBox, 1024, kSw128);
            const uint64_t dWN = smem_desc(s0a + kOffK, kBox, 1024, kSw128);
            const uint64_t dST = smem_desc(s0a + kOffST, 128, (kC / 8) * 128, kSwNone);
            const uint64_t dKH = smem_desc(s0a + kOffKH, 16, 1024, kSw128);
            bool ok = true;
            for (int c = 0; c < nch; ++c) {
                if (__any_sync(kFull, *abort_state != 0 || *abort_prep != 0)) {
                    ok = false;
                    break;
                }
                const int st = c % kNS;
                const uint64_t so = (uint64_t)((st * kStage) >> 4);   // stage offset in descriptor units
                const bool okw = mbar_wait(&bar_prep[st], (uint32_t)(c / kNS) & 1u, args.wait_ns) &&
                                 mbar_wait(&bar_s[0], (uint32_t)c & 1u, args.wait_ns);
                if (!__all_sync(kFull, okw)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    mma_f16_ss(tm + kColD, dDO + so, dST + so, id_s, 0);
#pragma unroll
                    for (int s8 = 0; s8 < kD / 8; ++s8)
                        mma_tf32_ts(tm + kColD, tm + kColH + 8 * s8,
                                    dKH + so + (uint64_t)(((s8 >> 2) * kKhBlock + 32 * (s8 & 3)) >> 4), id_k, 1);
                    mma_commit(&bar_x[0]);
                }
                __syncwarp();
                if (!__all_sync(kFull, mbar_wait(&bar_a[0], (uint32_t)c & 1u, args.wait_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    mma_f16_ss(tm + kColH, dDO + so, dQT + so, id_q, 1);
                    mma_f16_ts(tm + kColH, tm + kColA, dWN + so, id_w, 1);
                    mma_commit(&bar_free[st]);
                }
                __syncwarp();
            }
            // no tensor-core operation may still run when the TMEM is released
            if (elect_one()) mma_commit(&bar_fin[0]);
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
        for (int d0 = 0; d0 < kD; d0 += 16) {
            uint32_t r[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) r[jj] = __float_as_uint(h_in ? h_in[(int64_t)(d0 + jj) * kD + e] : 0.f);
            __syncwarp();
            tmem_st16(tm + lane_base + kColH + d0, r);
        }
        tmem_st_wait();
        int done = 0;
        for (int c = 0; c < nch; ++c) {
            if (__any_sync(kFull, *abort_state != 0 || *abort_prep != 0)) break;
            const int st = c % kNS;
            const uint32_t ph = (uint32_t)(c / kNS) & 1u;
            uint8_t *stg = smem + st * kStage;
            const bool okw = mbar_wait(&bar_prep[st], ph, args.wait_ns) &&
                             (c == 0 || mbar_wait(&bar_free[(c - 1) % kNS], (uint32_t)((c - 1) / kNS) & 1u,
                                                  args.wait_ns));
            if (!__all_sync(kFull, okw)) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_state = 1;
                break;
            }
            tc_fence_after();
            const Hdr *hdr = (const Hdr *)(stg + kOffHdr);
            // X^T = dH1^T diag(gamma), 16 columns at a time, the next chunk's load in
            // flight while this one is scaled
            {
                uint32_t ra[16], rb[16];
                tmem_ld16(tm + lane_base + kColH, ra);
#pragma unroll
                for (int q = 0; q < kD / 16; ++q) {
                    uint32_t(&cur)[16] = (q & 1) ? rb : ra;
                    uint32_t(&nxt)[16] = (q & 1) ? ra : rb;
                    tmem_ld_wait();
                    if (q + 1 < kD / 16) tmem_ld16(tm + lane_base + kColH + 16 * (q + 1), nxt);
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const uint4 g4 = *(const uint4 *)&hdr->gam[16 * q + 4 * j4];
                        const uint64_t y0 = mul_f32x2(((uint64_t)cur[4 * j4 + 1] << 32) | cur[4 * j4],
                                                      ((uint64_t)g4.y << 32) | g4.x);
                        const uint64_t y1 = mul_f32x2(((uint64_t)cur[4 * j4 + 3] << 32) | cur[4 * j4 + 2],
                                                      ((uint64_t)g4.w << 32) | g4.z);
                        cur[4 * j4] = (uint32_t)y0;
                        cur[4 * j4 + 1] = (uint32_t)(y0 >> 32);
                        cur[4 * j4 + 2] = (uint32_t)y1;
                        cur[4 * j4 + 3] = (uint32_t)(y1 >> 32);
                    }
                    tmem_st16(tm + lane_base + kColH + 16 * q, cur);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_s[0]);
            // X in bf16 for the tile kernel, [dk][dv], while the front products run (they
            // only read the state)
            if (hdr->emit) {
                const int64_t tt = e0 - 1 - c;
                unsigned short *xs = (unsigned short *)A.dHst + ((size_t)(tile0 + tt) * H + h) * kD * kD + e;
                uint32_t ra[16], rb[16];
                tmem_ld16(tm + lane_base + kColH, ra);
#pragma unroll
                for (int q = 0; q < kD / 16; ++q) {
                    uint32_t(&cur)[16] = (q & 1) ? rb : ra;
                    uint32_t(&nxt)[16] = (q & 1) ? ra : rb;
                    tmem_ld_wait();
                    if (q + 1 < kD / 16) tmem_ld16(tm + lane_base + kColH + 16 * (q + 1), nxt);
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 2) {
                        const uint32_t pr = pack_bf16(__uint_as_float(cur[jj]), __uint_as_float(cur[jj + 1]));
                        xs[(size_t)(16 * q + jj) * kD] = (unsigned short)(pr & 0xffffu);
                        xs[(size_t)(16 * q + jj + 1) * kD] = (unsigned short)(pr >> 16);
                    }
                }
            }
            if (!__all_sync(kFull, mbar_wait(&bar_x[0], (uint32_t)c & 1u, args.wait_ns))) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_state = 1;
                break;
            }
            tc_fence_after();
            // dD^T to bf16: the A operand of dD^T (-W); dD of the segment's tiles also goes
            // out, [C][dv] fp32, for the tile kernel
            {
                uint32_t dr[kC], a2[kC / 2];
                tmem_ld16(tm + lane_base + kColD, dr);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < kC / 2; ++i)
                    a2[i] = pack_bf16(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1]));
                tmem_st8(tm + lane_base + kColA, a2);
                if (hdr->emit) {
                    float *dst = A.dDst + ((size_t)(tile0 + e0 - 1 - c) * H + h) * kC * kD + e;
#pragma unroll
                    for (int i = 0; i < kC; ++i) dst[i * kD] = __uint_as_float(dr[i]);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_a[0]);
            done = c + 1;
        }
        // the gradient at the segment's first tile
        bool ok = done == nch;
        if (ok && nch > 0)
            ok = __all_sync(kFull, mbar_wait(&bar_free[(nch - 1) % kNS], (uint32_t)((nch - 1) / kNS) & 1u,
                                             args.wait_ns));
        ok = __all_sync(kFull, ok && *abort_state == 0);
        tc_fence_after();
        if (ok && h_out) {
            for (int d0 = 0; d0 < kD; d0 += 16) {
                uint32_t r[16];
                tmem_ld16(tm + lane_base + kColH + d0, r);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) h_out[(int64_t)(d0 + jj) * kD + e] = __uint_as_float(r[jj]);
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

template <bool VEC>
cudaError_t launch_impl(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mo,
                        const CUtensorMap &ma, const TaArgs &args, int64_t max_segs, cudaStream_t stream) {
    auto kern = tc_adj_kernel<VEC>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    ProfScope prof(stream, "tc_adj_kernel");
    kern<<<dim3((unsigned)max_segs, (unsigned)args.A.H), kThreads, kSmemBytes, stream>>>(mq, mk, mo, ma, args);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_adj(const bwdc::BcArgs &A, bool per_channel, int64_t T_total, int64_t max_tiles,
                          int64_t max_segs, int *status, cudaStream_t stream) {
    CUtensorMap mq, mk, mo, ma;
    if (!A.dout)   // dout = NULL (zero): the mma.sync chain reads it as zero
        return cudaErrorNotSupported;
    if (!tc_make_map(&mq, A.q, A.H, T_total) || !tc_make_map(&mk, A.k, A.H, T_total) ||
        !tc_make_map(&mo, A.dout, A.H, T_total))
        return cudaErrorNotSupported;
    if (per_channel) {
        if (!tc_make_map(&ma, A.a, A.H, T_total)) return cudaErrorNotSupported;
    } else {
        ma = mk;   // not read
    }
    if (max_segs <= 0) return cudaSuccess;
    if (max_segs > 0x7fffffff || A.H > 65535) return cudaErrorInvalidValue;
    TaArgs args{};
    args.A = A;
    args.T_total = T_total;
    args.max_tiles = max_tiles;
    args.status = status;
    args.wait_ns = kWaitNs;
    if (const char *w = std::getenv("GDR_TC_WAIT_NS")) {   // test hook: shorter pipeline waits
        const long long x = std::atoll(w);
        if (x >= 0 && (uint64_t)x < kWaitNs) args.wait_ns = (uint64_t)x;
    }
    return per_channel ? launch_impl<true>(mq, mk, mo, ma, args, max_segs, stream)
                       : launch_impl<false>(mq, mk, mo, ma, args, max_segs, stream);
}

}  // namespace gdr
