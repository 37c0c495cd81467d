// gdr_tc_fwd_chain.cu -- the forward state chain of the chunked backward on the
// 5th-generation tensor cores (tcgen05): bf16 inputs, dk = dv = 128, tiles of 16,
// bounded gate, one decay per token or one per key channel.
//
// The chain runs the tiles of one (segment, head) in order and stores, for the tile
// kernel, each tile's entering state H0 (bf16, [dk][dv]) and its D (fp32, [C][dv]).
// Per tile, with the in-tile cumulative log-decay G (per key channel), gamma = e^{G_C},
// Kt = K (.) e^G, Kh = K (.) e^-G, K'' = Kh (.) gamma and [P1 §3.2, P2 §2.1, P3 §3.1]
//   A = beta (.) strict_lower(Kt Kh^T),  Bu = (I + A)^{-1} diag(beta),  W = Bu Kt,
//   D  = Bu V - W H0 = U - W H0,
//   H1 = diag(gamma) H0 + K''^T D.
// The state lives in the tensor memory, transposed (lane = value index e, column = key
// index d), as the fp32 accumulator of the update:
//   tensor cores  D^T  = V^T Bu^T + H0^T (-W)^T   kind::f16, then kind::tf32 with the
//                                                 state as the A operand (16 K-steps)
//   state warps   D^T -> bf16 (A operand of the update) and to global memory;
//                 H^T <- H0^T diag(gamma)         a pass over the tensor memory
//   tensor cores  H1^T = H^T + D^T K''            kind::f16, the update
// H0 goes out while the front products run (they only read the state), after the
// previous tile's update is complete.  As in the forward kernels, one thread issues
// every MMA, so the update of one tile and the front products of the next (which
// read the state as their A operand, with the V^T Bu^T product issued between them)
// run in issue order.
//
// Roles as in the adjoint chain (gdr_tc_adj.cu): four state warps, four prep warps
// (one pipeline stage each: TMA loads of K, V and the per-channel gate inputs, the
// factored tiles, the Gram product and W on mma.sync, the substitution), one issuer.
// Segments and warm-ups are those of the mma.sync chain (bwd_fwd_chain_kernel): a
// segment's chain starts from a zero state at the latest tile before its start whose
// transition bound to the segment start is below 2^-64 (or from h0 at the sequence's
// start) and stores only for its own tiles.
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
constexpr uint32_t kColH = 0;            // the state H^T (128 fp32 columns)
constexpr uint32_t kColD = 128;          // D^T (C fp32 columns)
constexpr uint32_t kColA = kColD + kC;   // D^T in bf16 (C/2 columns)
constexpr uint32_t kTmemCols = 256;
static_assert(kColA + kC / 2 <= kTmemCols, "TMEM budget");

// Shared memory per stage (27 KB: four stages at two CTAs per SM).  [C][128] bf16
// tiles are two 64-column boxes of C rows x 128 B, 128-byte swizzled.
constexpr uint32_t kBox = kC * 128;
constexpr uint32_t kOffV = 0;                    // V: A operand (MN-major) of V^T Bu^T
constexpr uint32_t kOffK = kOffV + 2 * kBox;     // raw K -> Kt (bf16, Gram and W operand)
constexpr uint32_t kOffG = kOffK + 2 * kBox;     // raw gate inputs (per channel) -> Kh (bf16)
constexpr uint32_t kOffKP = kOffG + 2 * kBox;    // K'' (bf16, B operand of the update)
constexpr uint32_t kOffWT = kOffKP + 2 * kBox;   // -W in tf32 (4 column blocks of C rows x 128 B);
                                                 // Kh in fp32 before (per-channel gate)
constexpr uint32_t kWBlock = kC * 128;
constexpr uint32_t kOffAm = kOffWT + 4 * kWBlock;    // A (fp32 [C][C])
constexpr uint32_t kOffBu = kOffAm + kC * kC * 4;    // Bu (bf16 [C][C], 32-byte rows): W's operand
constexpr uint32_t kOffBc = kOffBu + kC * kC * 2;    // Bu: K-major B operand of V^T Bu^T (core matrices)
constexpr uint32_t kOffHdr = kOffBc + kC * kC * 2;
constexpr uint32_t kStage = 27648;
constexpr uint32_t kOffBar = kNS * kStage;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;   // + alignment slack

struct Hdr {
    float gam[kD];     // e^{G_C} per key channel
    float beta[kC];    // write strengths (0 past the end)
    int len;           // tokens of the tile
    int emit;          // 1: H0 and D go out (a tile of the segment), 0: a warm-up tile
};
static_assert(kOffHdr + sizeof(Hdr) <= kStage && kStage % 1024 == 0, "stage layout");

struct TfArgs {
    BcArgs A;
    int64_t T_total;
    int64_t max_tiles;   // tiles of the stored-state buffers
    int *status;
    uint64_t wait_ns;    // limit of every pipeline wait
};

// byte offset of element (row, col) of a [C][128] bf16 tile
__device__ __forceinline__ uint32_t tile_off(int row, int col) {
    return (uint32_t)(col >> 6) * kBox + sw128_off((uint32_t)row, (uint32_t)(col & 63) * 2u);
}
// byte offset of element (row, d) of the [C][128] fp32 (tf32) -W area
__device__ __forceinline__ uint32_t wt_off(int row, int d) {
    return kOffWT + (uint32_t)(d >> 5) * kWBlock + sw128_off((uint32_t)row, (uint32_t)(d & 31) * 4u);
}
// Bu[n][k] in the K-major core-matrix layout (8-row groups at 256 B, 16-byte column
// groups at 128 B)
__device__ __forceinline__ uint32_t cc_off(int n, int k) {
    return core_off((uint32_t)n, (uint32_t)k * 2u, (kC / 8) * 128u, 128u);
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads, 2)
tc_fwd_chain_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmA, const TfArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bar_full = (uint64_t *)(smem + kOffBar);
    uint64_t *bar_prep = bar_full + kNS;
    uint64_t *bar_free = bar_prep + kNS;   // the stage's products complete (the state updated)
    uint64_t *bar_init = bar_free + kNS;   // [1] state initialised (4 state warps)
    uint64_t *bar_x = bar_init + 1;        // [1] D^T complete
    uint64_t *bar_a = bar_x + 1;           // [1] state scaled and D^T in bf16 written (4 state warps)
    uint64_t *bar_fin = bar_a + 1;         // [1] every MMA of the CTA complete
    uint32_t *tmem_slot = (uint32_t *)(bar_fin + 1);
    volatile int *abort_prep = (volatile int *)(tmem_slot + 1);   // set by prep warps
    volatile int *abort_state = abort_prep + 1;                   // set by state warps and the issuer
    __shared__ int64_t s_first;

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
        const int64_t w = bwdc::warm_walk(A.lam, tile0, ntiles, H, h, s0, -1);
        if (lane == 0) s_first = w;
    }
    __syncthreads();
    const int64_t w0 = s_first;   // the chain runs tiles w0, ..., s1 - 1
    const int nch = (int)max((int64_t)0, s1 - w0);
    const size_t sbase = ((size_t)n * H + h) * kD * kD;
    const float *h_in = (w0 == 0 && A.h0) ? A.h0 + sbase : nullptr;
    constexpr unsigned kFull = 0xffffffffu;
    // (checking build) the segment's tokens and tiles lie inside the tensors; a failed
    // check leaves the CTA's work undone (block-uniform, before any barrier)
    if (!GDR_INBOUNDS(n < p.N && h < H && sstart >= 0 && send <= args.T_total && w0 >= 0 && s1 <= ntiles &&
                      tile0 + ntiles <= args.max_tiles && s1 - w0 < (int64_t)1 << 30))
        return;

    if (tid == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_prep[i], 1);
            mbar_init(&bar_free[i], 1);
        }
        mbar_init(&bar_init[0], 4);
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
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
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
            const int64_t tt = w0 + c;                    // tile index within the sequence
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
                mbar_arrive_expect_tx(&bar_full[st], 2 * kBox * (VEC ? 3 : 2));
                tma_load_3d(stg + kOffV, &tmV, 0, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffV + kBox, &tmV, 64, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffK, &tmK, 0, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffK + kBox, &tmK, 64, h, (int)t0, &bar_full[st]);
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
                hdr->emit = tt >= s0 ? 1 : 0;
            }
            // scalar gate: G_i by a prefix sum over lanes 0..15 (0 past the end)
            float Es = 1.f, Ens = 1.f, Eps = 1.f;
            if (!VEC) {
                float Gs = g_i;
#pragma unroll
                for (int o = 1; o < kC; o <<= 1) {
                    const float y = __shfl_up_sync(kFull, Gs, o);
                    if (lane >= o) Gs += y;
                }
                const float Gc = __shfl_sync(kFull, Gs, kC - 1);
                Es = __expf(Gs);
                Ens = __expf(-Gs);
                Eps = __expf(Gc - Gs);   // e^{G_C - G_i}: K'' = K e^{G_C - G}
            }
            if (!__all_sync(kFull, mbar_wait(&bar_full[st], ph, args.wait_ns))) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_prep = 1;
                break;
            }
            pend_st = -1;
            // rows past the end of the sequence hold another sequence's tokens: zero
            // those of V and K (their gates are taken as 0 below)
            if (len < kC) {
                const int nrow = kC - len;
                for (int e = lane; e < 2 * 2 * nrow * 8; e += 32) {
                    const int chunk16 = e & 7, rem = e >> 3;
                    const int row = len + rem % nrow, box = (rem / nrow) & 1;
                    const int tsel = rem / (nrow * 2);
                    const uint32_t toff = (tsel == 0 ? kOffV : kOffK) + box * kBox;
                    *(uint4 *)(stg + toff + sw128_off(row, chunk16 * 16)) = make_uint4(0, 0, 0, 0);
                }
            }
            __syncwarp();
            // ---- the factored tiles: lane l runs key channels 4l..4l+3 down the tile's
            // tokens.  Kt (bf16) over the raw K, Kh (bf16) over the raw gate inputs; K''
            // directly (scalar gate) or Kh in fp32 to the -W area, scaled by e^{G_C} once
            // the last token is in (per-channel gate); e^{G_C} to the header
            {
                const int d = 4 * lane;
                const float nb = -A.b;
                float G0 = 0.f, G1 = 0.f, G2 = 0.f, G3 = 0.f;
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
                    const float2 k01 = unpack_bf16(kr.x), k23 = unpack_bf16(kr.y);
                    const float kv[4] = {k01.x, k01.y, k23.x, k23.y};
                    float kt[4], kh[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        kt[u] = kv[u] * E[u];
                        kh[u] = kv[u] * En[u];
                    }
                    *(uint2 *)(stg + kOffK + off) = make_uint2(pack_bf16(kt[0], kt[1]), pack_bf16(kt[2], kt[3]));
                    *(uint2 *)(stg + kOffG + off) = make_uint2(pack_bf16(kh[0], kh[1]), pack_bf16(kh[2], kh[3]));
                    if (VEC) {
                        *(float4 *)(stg + wt_off(i, d)) = make_float4(kh[0], kh[1], kh[2], kh[3]);
                    } else {
                        const float ep = __shfl_sync(kFull, Eps, i);
                        *(uint2 *)(stg + kOffKP + off) =
                            make_uint2(pack_bf16(kv[0] * ep, kv[1] * ep), pack_bf16(kv[2] * ep, kv[3] * ep));
                    }
                }
                if (VEC) {
                    const float4 gc = make_float4(__expf(G0), __expf(G1), __expf(G2), __expf(G3));
                    *(float4 *)&hdr->gam[d] = gc;
                    // K'' = Kh (.) e^{G_C}
#pragma unroll 4
                    for (int i = 0; i < kC; ++i) {
                        const float4 kh = *(const float4 *)(stg + wt_off(i, d));
                        *(uint2 *)(stg + kOffKP + tile_off(i, d)) =
                            make_uint2(pack_bf16(kh.x * gc.x, kh.y * gc.y), pack_bf16(kh.z * gc.z, kh.w * gc.w));
                    }
                } else {
                    const float ec = __shfl_sync(kFull, Es, kC - 1);
                    *(float4 *)&hdr->gam[d] = make_float4(ec, ec, ec, ec);
                }
            }
            __syncwarp();
            // ---- Skk = Kt Kh^T over 16-key slabs (bf16 in, fp32 out)
            float skk[2][4] = {};
#pragma unroll 2
            for (int sl = 0; sl < kD / 16; ++sl) {
                const uint32_t off = (uint32_t)(sl >> 2) * kBox +
                                     sw128_off((uint32_t)lr, (uint32_t)(sl & 3) * 32u + 16u * (uint32_t)lc);
                uint32_t ktf[4], khf[4];
                ldsm_x4(smem_u32(stg + kOffK + off), ktf);
                ldsm_x4(smem_u32(stg + kOffG + off), khf);
                mma16816(skk[0], ktf, khf[0], khf[2]);
                mma16816(skk[1], ktf, khf[1], khf[3]);
            }
            // ---- A = beta (.) strict_lower(Skk) (fp32); skk[nt][r] is (row g + 8 (r >> 1),
            // column 8 nt + 2t + (r & 1))
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
                    }
            }
            __syncwarp();
            // ---- T = (I + A)^{-1}, one column per lane (lanes 16..31 repeat 0..15);
            // Bu = T diag(beta) in bf16, row-major (lanes 0..15) and as the K-major
            // operand of V^T Bu^T (lanes 16..31)
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
                } else {
#pragma unroll
                    for (int i = 0; i < kC; ++i)
                        *(__nv_bfloat16 *)(stg + kOffBc + cc_off(i, jc)) = __float2bfloat16_rn(tcol[i] * bj);
                }
            }
            __syncwarp();
            // ---- -W = -Bu Kt, 16 key columns at a time, in fp32 (tf32 operand) into the
            // -W area (the per-channel Kh there was read by the K'' pass above)
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
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr)
                            *(float2 *)(stg + wt_off(g + 8 * hr, 16 * sl + 8 * nt + 2 * t)) =
                                make_float2(-w[nt][2 * hr], -w[nt][2 * hr + 1]);
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
            const uint32_t id_u = instr_desc(128, kC, 1, true, false);    // V^T Bu^T
            const uint32_t id_w = instr_desc(128, kC, 2, false, false);   // H0^T (-W)^T (tf32)
            const uint32_t id_h = instr_desc(128, kD, 1, false, true);    // D^T K''
            const uint32_t s0a = smem_u32(smem);
            const uint64_t dV = smem_desc(s0a + kOffV, kBox, 1024, kSw128);
            const uint64_t dBc = smem_desc(s0a + kOffBc, 128, (kC / 8) * 128, kSwNone);
            const uint64_t dWT = smem_desc(s0a + kOffWT, 16, 1024, kSw128);
            const uint64_t dKP = smem_desc(s0a + kOffKP, kBox, 1024, kSw128);
            bool ok = nch == 0 || __all_sync(kFull, mbar_wait(&bar_init[0], 0, args.wait_ns));
            for (int c = 0; c < nch && ok; ++c) {
                if (__any_sync(kFull, *abort_state != 0 || *abort_prep != 0)) {
                    ok = false;
                    break;
                }
                const int st = c % kNS;
                const uint64_t so = (uint64_t)((st * kStage) >> 4);   // stage offset in descriptor units
                if (!__all_sync(kFull, mbar_wait(&bar_prep[st], (uint32_t)(c / kNS) & 1u, args.wait_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    mma_f16_ss(tm + kColD, dV + so, dBc + so, id_u, 0);
#pragma unroll
                    for (int s8 = 0; s8 < kD / 8; ++s8)
                        mma_tf32_ts(tm + kColD, tm + kColH + 8 * s8,
                                    dWT + so + (uint64_t)(((s8 >> 2) * kWBlock + 32 * (s8 & 3)) >> 4), id_w, 1);
                    mma_commit(&bar_x[0]);
                }
                __syncwarp();
                if (!__all_sync(kFull, mbar_wait(&bar_a[0], (uint32_t)c & 1u, args.wait_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    mma_f16_ts(tm + kColH, tm + kColA, dKP + so, id_h, 1);
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
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_init[0]);
        for (int c = 0; c < nch; ++c) {
            if (__any_sync(kFull, *abort_state != 0 || *abort_prep != 0)) break;
            const int st = c % kNS;
            const uint32_t ph = (uint32_t)(c / kNS) & 1u;
            uint8_t *stg = smem + st * kStage;
            if (!__all_sync(kFull, mbar_wait(&bar_prep[st], ph, args.wait_ns))) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_state = 1;
                break;
            }
            const Hdr *hdr = (const Hdr *)(stg + kOffHdr);
            const bool emit = hdr->emit != 0;
            const size_t cg = (size_t)(tile0 + w0 + c) * H + h;   // global (tile, head)
            // H0 in bf16, [dk][dv], once the previous update is complete, while the front
            // products run (they only read the state)
            if (emit) {
                if (c > 0 && !__all_sync(kFull, mbar_wait(&bar_free[(c - 1) % kNS], (uint32_t)((c - 1) / kNS) & 1u,
                                                          args.wait_ns))) {
                    if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                    *abort_state = 1;
                    break;
                }
                tc_fence_after();
                unsigned short *hs = (unsigned short *)A.Hst + cg * kD * kD + e;
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
                        hs[(size_t)(16 * q + jj) * kD] = (unsigned short)(pr & 0xffffu);
                        hs[(size_t)(16 * q + jj + 1) * kD] = (unsigned short)(pr >> 16);
                    }
                }
            }
            if (!__all_sync(kFull, mbar_wait(&bar_x[0], (uint32_t)c & 1u, args.wait_ns))) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_state = 1;
                break;
            }
            tc_fence_after();
            // D^T: to bf16 (the update's A operand) and, for a tile of the segment, to
            // global memory ([C][dv] fp32, one token row per register)
            {
                uint32_t dr[kC], a2[kC / 2];
                tmem_ld16(tm + lane_base + kColD, dr);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < kC / 2; ++i)
                    a2[i] = pack_bf16(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1]));
                tmem_st8(tm + lane_base + kColA, a2);
                if (emit) {
                    float *dst = A.Dst + cg * kC * kD + e;
#pragma unroll
                    for (int i = 0; i < kC; ++i) dst[i * kD] = __uint_as_float(dr[i]);
                }
            }
            // H^T <- H0^T diag(gamma), 16 columns at a time, the next chunk's load in
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
            if (lane == 0) mbar_arrive(&bar_a[0]);
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
cudaError_t launch_impl(const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &ma,
                        const TfArgs &args, int64_t max_segs, cudaStream_t stream) {
    auto kern = tc_fwd_chain_kernel<VEC>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    ProfScope prof(stream, "tc_fwd_chain_kernel");
    kern<<<dim3((unsigned)max_segs, (unsigned)args.A.H), kThreads, kSmemBytes, stream>>>(mk, mv, ma, args);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_fwd_chain(const bwdc::BcArgs &A, bool per_channel, int64_t T_total, int64_t max_tiles,
                                int64_t max_segs, int *status, cudaStream_t stream) {
    CUtensorMap mk, mv, ma;
    if (!tc_make_map(&mk, A.k, A.H, T_total) || !tc_make_map(&mv, A.v, A.H, T_total))
        return cudaErrorNotSupported;
    if (per_channel) {
        if (!tc_make_map(&ma, A.a, A.H, T_total)) return cudaErrorNotSupported;
    } else {
        ma = mk;   // not read
    }
    if (max_segs <= 0) return cudaSuccess;
    if (max_segs > 0x7fffffff || A.H > 65535) return cudaErrorInvalidValue;
    TfArgs args{};
    args.A = A;
    args.T_total = T_total;
    args.max_tiles = max_tiles;
    args.status = status;
    args.wait_ns = kWaitNs;
    if (const char *w = std::getenv("GDR_TC_WAIT_NS")) {   // test hook: shorter pipeline waits
        const long long x = std::atoll(w);
        if (x >= 0 && (uint64_t)x < kWaitNs) args.wait_ns = (uint64_t)x;
    }
    return per_channel ? launch_impl<true>(mk, mv, ma, args, max_segs, stream)
                       : launch_impl<false>(mk, mv, ma, args, max_segs, stream);
}

}  // namespace gdr
