// gdr_tc_vec.cu -- the per-channel decay forward on the 5th-generation tensor
// cores (tcgen05): bf16 inputs, dk = dv = 128, tile C = 16, bounded gate.
//
// One CTA runs the tiles of one (segment, head) in order, with the same roles as
// the scalar-gate tile kernel: four prep warps (one pipeline stage each), one MMA
// issuer and four state warps.  The state never leaves the tensor memory: it is
// the fp32 accumulator of the state-update MMA and the tf32 A operand of the
// products with the keys and queries.
//
// Per tile, with per-channel cumulative log-decay G (resetting each tile),
// gamma = exp(G_C) (the tile's decay of each key channel), the factored decays
// Kt = K (.) e^G, Kh = K (.) e^-G, Qt = Q (.) e^G and the entering state H
// (transposed in TMEM: lane = value index e, column = key index d)
// [P1 §2.1-2.2, P3 §3.2]:
//   prep warps (CUDA cores + mma.sync):
//       G by a running sum over the tile's tokens, per channel;
//       Skk = Kt Kh^T, Sqk = Qt Kh^T;  A = beta (.) strict_lower(Skk),
//       P = lower(Sqk);  Bu = (I + A)^{-1} diag(beta);  K'' = Kh (.) gamma
//   tensor cores (one issuing thread):
//       D^T  = V^T Bu^T                 (U^T, kind::f16)
//       [Y | O^T] = H^T [-Kt ; Qt]^T    (kind::tf32, A = the state in TMEM)
//       D^T += Y Bu^T                   (kind::tf32, A = Y in TMEM):
//                                        D = Bu (V - Kt H) = U - W H, W = Bu Kt
//       H^T += D^T K''                  (kind::f16, A = D^T in bf16, the update)
//       O^T += D^T P^T                  (in-tile output term)
//   state warps, between the front products and the update:
//       H^T <- H^T diag(gamma)          (the decay of every key channel: a pass
//                                        over the state in TMEM, read, scaled and
//                                        written back by the lane that owns it)
//       D^T -> bf16 A operand of the update and the output term.
// So H_next = diag(gamma) H + K''^T D = diag(gamma) H + (Kh gamma)^T D, the
// chunked per-channel form; the state kept in TMEM is always the true state.
//
// Long sequences are cut into segments of S tiles, one CTA per (segment, head),
// each starting from a zero state at a warm-up tile before its segment (found by
// the per-channel path's warm-up kernel: the latest tile whose bound on the
// transition to the segment start is below 2^-64) and storing outputs only for
// its own tiles.  A (sequence, head) pair with a segment start that has no such
// warm-up runs as one CTA over the whole sequence.
#include <cudaTypedefs.h>

#include <cstdlib>

#include "gdr_sm100.cuh"
#include "gdr_tc.cuh"
#include "gdr_tc_prep.cuh"

namespace gdr {

GDR_DEBUG_TU()

namespace {

using namespace sm100;
using namespace tcp;

constexpr int kD = 128;          // dk = dv
constexpr int kC = 16;           // tile length
constexpr int kNS = 4;           // pipeline stages, one per prep warp
constexpr int kThreads = 32 * (4 + kNS + 1);   // 4 state warps, kNS prep warps, 1 MMA issuer
static_assert(kNS == 4, "the prep warps form warpgroup 1 (register hand-over below)");
constexpr uint64_t kWaitNs = 2000000000ull;    // default pipeline wait limit: 2 s
constexpr uint64_t kDrainNs = 2000000000ull;   // drains before exit: 2 s

// TMEM columns
constexpr uint32_t kColH = 0;                    // state H^T (128 fp32 columns)
constexpr uint32_t kColB = 128;                  // 2 buffers of [D (C) | Y (C) | out (C)]
constexpr uint32_t kColBuf = 3 * kC;
constexpr uint32_t kColA = kColB + 2 * kColBuf;  // D^T in bf16 (C/2 columns)
constexpr uint32_t kTmemCols = 256;
static_assert(kColA + kC / 2 <= kTmemCols, "TMEM budget");

// Shared memory per stage (27 KB, so that 4 stages fit at 2 CTAs per SM).
// [-Kt ; Qt] in tf32 is 4 column blocks of 2C rows x 128 B (rows 0..C-1: -Kt,
// rows C..2C-1: Qt).  Until the prep warp writes them, the -Kt rows hold the raw
// gate inputs (blocks 0, 1) and the raw Q tile (blocks 2, 3), one 64-column box
// each, and the Qt rows hold exp(G) in fp32.
constexpr uint32_t kBox = kC * 128;              // one 64-column box of a [C][128] bf16 tile
constexpr uint32_t kOffK = 0;                    // raw K, then K'' (bf16, the update's operand)
constexpr uint32_t kOffV = kOffK + 2 * kBox;
constexpr uint32_t kOffWQ = kOffV + 2 * kBox;
constexpr uint32_t kWQBlock = 2 * kC * 128;
constexpr uint32_t kOffA0 = kOffWQ;                  // raw gate inputs, columns 0..63
constexpr uint32_t kOffA1 = kOffWQ + kWQBlock;       // raw gate inputs, columns 64..127
constexpr uint32_t kOffQ0 = kOffWQ + 2 * kWQBlock;   // raw Q, columns 0..63
constexpr uint32_t kOffQ1 = kOffWQ + 3 * kWQBlock;   // raw Q, columns 64..127
constexpr uint32_t kOffBT = kOffWQ + 4 * kWQBlock;   // A (fp32 [C][C]), then Bu in tf32
constexpr uint32_t kOffBU = kOffBT + kC * kC * 4;    // Bu in bf16
constexpr uint32_t kOffP = kOffBU + kC * kC * 2;     // P in bf16
constexpr uint32_t kOffHdr = kOffP + kC * kC * 2;
constexpr uint32_t kStage = 27648;
__host__ __device__ constexpr uint32_t q_box(int b) { return b == 0 ? kOffQ0 : kOffQ1; }
__host__ __device__ constexpr uint32_t a_box(int b) { return b == 0 ? kOffA0 : kOffA1; }
constexpr uint32_t kOffBar = kNS * kStage;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;   // + alignment slack

struct Hdr {
    float gam[kD];     // exp(G_C) per key channel: the tile's decay of the state
    float beta[kC];    // write strengths (0 past the end)
    int len;           // tokens of the tile
    int emit;          // 1: the tile's outputs are stored (0: a warm-up tile)
};
static_assert(kOffHdr + sizeof(Hdr) <= kStage && kStage % 1024 == 0, "stage layout");

// core-matrix (no swizzle) K-major layout of a C x C bf16 operand [n][k]
__device__ __forceinline__ uint32_t cc_off(int n, int k) {
    return core_off((uint32_t)n, (uint32_t)k * 2u, (kC / 8) * 128u, 128u);
}
// the same for a C x C tf32 operand: 16-byte core rows hold 4 elements
constexpr uint32_t kTfRowGroup = (kC / 4) * 128u;   // bytes between 8-row groups
__device__ __forceinline__ uint32_t cc_off_tf32(int n, int k) {
    return core_off((uint32_t)n, (uint32_t)k * 4u, kTfRowGroup, 128u);
}
// byte offset of element (row, d) of a fp32 row block of [-Kt ; Qt] (row in [0, 2C))
__device__ __forceinline__ uint32_t wq_off(int row, int d) {
    return kOffWQ + (uint32_t)(d >> 5) * kWQBlock + sw128_off((uint32_t)row, (uint32_t)(d & 31) * 4u);
}
struct TvArgs {
    const __nv_bfloat16 *beta;
    const float *h0;
    __nv_bfloat16 *out;
    float *hT;
    const int *warm;     // [segments][H] warm-up tiles before each segment start (-1: none)
    Plan plan;
    int H;
    int64_t T_total;
    float b;
    int *status;
    uint64_t wait_ns;    // limit of every pipeline wait
};

__global__ void __launch_bounds__(kThreads, 2)
tc_vec_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmA,
              const TvArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bar_full = (uint64_t *)(smem + kOffBar);
    uint64_t *bar_prep = bar_full + kNS;
    uint64_t *bar_free = bar_prep + kNS;
    uint64_t *bar_x = bar_free + kNS;    // [2]
    uint64_t *bar_h = bar_x + 2;         // [1]
    uint64_t *bar_fin = bar_h + 1;       // [1]
    uint64_t *bar_a = bar_fin + 1;       // [1] state rescaled and D^T written (4 state warps)
    uint64_t *bar_init = bar_a + 1;      // [1] state initialised (4 state warps)
    uint64_t *bar_y = bar_init + 1;      // [1] the front products complete (Y written)
    uint32_t *tmem_slot = (uint32_t *)(bar_y + 1);
    volatile int *abort_prep = (volatile int *)(tmem_slot + 1);   // set by prep warps
    volatile int *abort_state = abort_prep + 1;                   // set by state warps only
    __shared__ int s_warm, s_seg_all;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    const int H = args.H;
    const Plan &p = args.plan;
    const int64_t sg = blockIdx.x;   // global segment
    const int n = find_owner(p.seg_base, p.N, sg);
    if (n < 0) return;
    const int64_t ntiles = p.chunk_base[n + 1] - p.chunk_base[n];
    const int64_t j = sg - p.seg_base[n];
    // the pair runs in segments only if every segment start found its warm-up
    if (warp == 0) {
        const int64_t first = p.seg_base[n], nseg = p.seg_base[n + 1] - first;
        bool ok = true;
        for (int64_t i = lane; i < nseg; i += 32) ok = ok && args.warm[(first + i) * H + h] >= 0;
        ok = __all_sync(0xffffffffu, ok);
        if (lane == 0) {
            s_seg_all = ok;
            s_warm = ok ? args.warm[sg * H + h] : 0;
        }
    }
    __syncthreads();
    const bool segmented = s_seg_all != 0;
    if (!segmented && j > 0) return;   // one CTA runs the whole sequence
    const int64_t s0 = segmented ? j * p.seg_chunks : 0;
    const int64_t s1 = segmented ? min(ntiles, s0 + (int64_t)p.seg_chunks) : ntiles;
    const int64_t w0 = s0 - s_warm;   // first tile run
    const int nch = (int)max((int64_t)0, s1 - w0);
    const int64_t sstart = p.seq_start[n], send = p.seq_start[n + 1];
    const size_t hbase = ((size_t)n * H + h) * kD * kD;
    const float *h_in = (w0 == 0 && args.h0) ? args.h0 + hbase : nullptr;
    float *h_out = (args.hT && s1 == ntiles) ? args.hT + hbase : nullptr;
    constexpr unsigned kFull = 0xffffffffu;
    // (checking build) the segment's tokens lie inside the tensors; a failed check
    // leaves the CTA's work undone (block-uniform, before any barrier)
    if (!GDR_INBOUNDS(n < p.N && h < H && sstart >= 0 && send <= args.T_total && w0 >= 0 &&
                      s1 * kC <= send - sstart + kC - 1 && s1 - w0 < (int64_t)1 << 30))
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
        mbar_init(&bar_y[0], 1);
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
        prefetch_tensormap(&tmA);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;

    if (warp >= 4 && warp < 4 + kNS) {
        // ============================ prep warps ============================
        // The state warps (warpgroup 0) hand 8 registers per thread over to the prep
        // warps (warpgroup 1): 4 x 32 x (88 + 104) = 2 x 4 x 32 x 96, the two warpgroups'
        // launch allocation, so the increase never waits on more than the decrease frees.
        asm volatile("setmaxnreg.inc.sync.aligned.u32 104;");
        const int pw = warp - 4;
        const int g = lane >> 2, t = lane & 3;
        int pend_st = -1;          // stage whose TMA is issued but not yet seen complete
        uint32_t pend_ph = 0;
        // prep warp pw owns stage pw and tiles pw, pw + kNS, ...
        for (int c = pw; c < nch; c += kNS) {
            if (__any_sync(kFull, *abort_prep != 0 || *abort_state != 0)) break;
            const int st = pw;
            const uint32_t ph = (uint32_t)(c / kNS) & 1u;
            uint8_t *stg = smem + st * kStage;
            Hdr *hdr = (Hdr *)(stg + kOffHdr);
            const int64_t tt = w0 + c;                     // tile index within the sequence
            const int64_t t0 = sstart + tt * kC;          // first token row
            const int len = (int)min((int64_t)kC, send - t0);
            const bool use_q = tt >= s0;
            float b_i = 0.f;
            if (lane < len && GDR_INBOUNDS(t0 >= 0 && t0 + len <= args.T_total))
                b_i = __bfloat162float(args.beta[(t0 + lane) * H + h]);
            if (c >= kNS && !__all_sync(kFull, mbar_wait(&bar_free[st], ph ^ 1u, args.wait_ns))) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_prep = 1;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar_full[st], 2 * kBox * (use_q ? 4 : 3));
                tma_load_3d(stg + kOffK, &tmK, 0, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffK + kBox, &tmK, 64, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffV, &tmV, 0, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffV + kBox, &tmV, 64, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffA0, &tmA, 0, h, (int)t0, &bar_full[st]);
                tma_load_3d(stg + kOffA1, &tmA, 64, h, (int)t0, &bar_full[st]);
                if (use_q) {
                    tma_load_3d(stg + kOffQ0, &tmQ, 0, h, (int)t0, &bar_full[st]);
                    tma_load_3d(stg + kOffQ1, &tmQ, 64, h, (int)t0, &bar_full[st]);
                }
            }
            pend_st = st;
            pend_ph = ph;
            if (lane < kC) hdr->beta[lane] = b_i;
            if (lane == 0) {
                hdr->len = len;
                hdr->emit = use_q ? 1 : 0;
            }
            if (!__all_sync(kFull, mbar_wait(&bar_full[st], ph, args.wait_ns))) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_prep = 1;
                break;
            }
            pend_st = -1;
            // rows past the end of the sequence hold another sequence's tokens: zero
            // those of K, V and Q (their gates are taken as 0 below)
            if (len < kC) {
                const int nt = use_q ? 3 : 2;
                const int nrow = kC - len;
                for (int e = lane; e < nt * 2 * nrow * 8; e += 32) {
                    const int chunk16 = e & 7, rem = e >> 3;
                    const int row = len + rem % nrow, box = (rem / nrow) & 1;
                    const int tsel = rem / (nrow * 2);
                    const uint32_t toff = tsel == 0 ? kOffK + box * kBox
                                          : (tsel == 1 ? kOffV + box * kBox : q_box(box));
                    *(uint4 *)(stg + toff + sw128_off(row, chunk16 * 16)) = make_uint4(0, 0, 0, 0);
                }
            }
            // ---- G: lane l runs channels 4l..4l+3 down the tile's tokens (gates past the
            // end are 0); exp(G) goes to the Qt rows (fp32), exp(G_C) to the header
            {
                const int d = 4 * lane;
                const float nb = -args.b;
                const uint8_t *abase = stg + a_box(d >> 6);
                const uint32_t dcol = (uint32_t)(d & 63) * 2u;
                float G[4] = {0.f, 0.f, 0.f, 0.f};
                // four tokens per group; the next group's raw rows are read before this
                // group's exp(G) rows are stored (rows C..2C-1, never the raw rows 0..C-1,
                // which the compiler cannot see), so their latency overlaps the gates
                uint2 raw[4], nxt[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) raw[u] = *(const uint2 *)(abase + sw128_off((uint32_t)u, dcol));
                float e[4];
#pragma unroll 1
                for (int grp = 0; grp < kC / 4; ++grp) {
                    if (grp + 1 < kC / 4) {
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            nxt[u] = *(const uint2 *)(abase + sw128_off((uint32_t)(4 * grp + 4 + u), dcol));
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 x0 = unpack_bf16(raw[u].x), x1 = unpack_bf16(raw[u].y);
                        const float xs[4] = {x0.x, x0.y, x1.x, x1.y};
                        const bool live = 4 * grp + u < len;   // gates past the end are 0
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            G[v] = live ? fmaf(nb, fast_sigmoid(xs[v]), G[v]) : G[v];
                            e[v] = __expf(G[v]);
                        }
                        *(float4 *)(stg + wq_off(kC + 4 * grp + u, d)) = make_float4(e[0], e[1], e[2], e[3]);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) raw[u] = nxt[u];
                }
                // exp(G_C): G stops at the tile's last token, so the last row's values
                *(float4 *)&hdr->gam[d] = make_float4(e[0], e[1], e[2], e[3]);
            }
            __syncwarp();
            // ---- per 16-column slab s: lane (g, t) = (lane / 4, lane % 4) forms rows g and
            // g + 8, columns 2t, 2t + 1, 2t + 8, 2t + 9 of Kt, Kh, Qt and K'' = Kh (.) gamma
            // from the raw tiles and exp(G), which is the m16n8k16 fragment layout: its own
            // bf16 pairs are the A fragments of Kt and Qt and the B fragments of Kh^T, so the
            // Gram products Skk = Kt Kh^T and Sqk = Qt Kh^T need no scratch.  It writes K''
            // over the raw K, -Kt (tf32) over the raw gate inputs / raw Q and Qt (tf32) over
            // exp(G).  Slab s writes -Kt over raw data that slabs <= s have read: raw gate
            // inputs (slabs 0-3), raw Q columns 0..63 (slabs 4, 5) and 64..127 (slabs 6, 7).
            float skk[2][4] = {}, sqk[2][4] = {};
            {
#pragma unroll 1
                for (int sl = 0; sl < kD / 16; ++sl) {
                    // element (hr, w, u): row g + 8 hr, column 16 sl + 2t + 8 w + u
                    uint32_t kw[2][2], qw[2][2];
                    float2 ev[2][2];
                    float2 gm[2];
#pragma unroll
                    for (int w = 0; w < 2; ++w) {
                        const int c = 16 * sl + 2 * t + 8 * w;
                        gm[w] = *(const float2 *)&hdr->gam[c];
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const int r = g + 8 * hr;
                            const uint32_t kq_off = sw128_off((uint32_t)r, (uint32_t)(c & 63) * 2u);
                            kw[hr][w] = *(const uint32_t *)(stg + kOffK + (c >> 6) * kBox + kq_off);
                            qw[hr][w] = use_q ? *(const uint32_t *)(stg + q_box(c >> 6) + kq_off) : 0u;
                            ev[hr][w] = *(const float2 *)(stg + wq_off(kC + r, c));
                        }
                    }
                    // -Kt overwrites raw Q that other lanes read: slabs 4 and 5 that of slabs
                    // 0-3, slab 6 that of slabs 4 and 5, slab 7 that of slabs 6 and 7 (its
                    // own); slabs 0-3 overwrite only gate inputs (read before the slabs) and
                    // each lane's own elements
                    if (sl == 4 || sl >= 6) __syncwarp();
                    uint32_t ktf[4], khf[4], qtf[4];   // fragment order: (g, w 0), (g+8, w 0), (g, w 1), (g+8, w 1)
#pragma unroll
                    for (int w = 0; w < 2; ++w) {
                        const int c = 16 * sl + 2 * t + 8 * w;
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const int r = g + 8 * hr;
                            const float2 kv = unpack_bf16(kw[hr][w]), qv = unpack_bf16(qw[hr][w]);
                            const float2 E = ev[hr][w];
                            const float n0 = __fdividef(1.f, E.x), n1 = __fdividef(1.f, E.y);
                            const float kt0 = kv.x * E.x, kt1 = kv.y * E.y;
                            const float kh0 = kv.x * n0, kh1 = kv.y * n1;
                            const float qt0 = qv.x * E.x, qt1 = qv.y * E.y;
                            const uint32_t kq_off = sw128_off((uint32_t)r, (uint32_t)(c & 63) * 2u);
                            *(uint32_t *)(stg + kOffK + (c >> 6) * kBox + kq_off) =
                                pack_bf16(kh0 * gm[w].x, kh1 * gm[w].y);
                            *(float2 *)(stg + wq_off(r, c)) = make_float2(-kt0, -kt1);
                            if (use_q) *(float2 *)(stg + wq_off(kC + r, c)) = make_float2(qt0, qt1);
                            ktf[2 * w + hr] = pack_bf16(kt0, kt1);
                            khf[2 * w + hr] = pack_bf16(kh0, kh1);
                            qtf[2 * w + hr] = pack_bf16(qt0, qt1);
                        }
                    }
                    mma16816(skk[0], ktf, khf[0], khf[2]);
                    mma16816(skk[1], ktf, khf[1], khf[3]);
                    if (use_q) {
                        mma16816(sqk[0], qtf, khf[0], khf[2]);
                        mma16816(sqk[1], qtf, khf[1], khf[3]);
                    }
                }
            }
            __syncwarp();   // every lane's slab stores are done before A and P are formed
            // ---- A = beta (.) strict_lower(Skk) (fp32, for the substitution) and
            // P = lower(Sqk) (bf16, the output term's operand), from the accumulators:
            // skk[nt][r] is (row g + 8 (r >> 1), column 8 nt + 2t + (r & 1))
            {
                float *Am = (float *)(stg + kOffBT);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int i = g + 8 * hr, j0 = 8 * nt + 2 * t;
                        const float bi = hdr->beta[i];
                        const float a0 = j0 < i ? bi * skk[nt][2 * hr] : 0.f;
                        const float a1 = j0 + 1 < i ? bi * skk[nt][2 * hr + 1] : 0.f;
                        *(float2 *)&Am[i * kC + j0] = make_float2(a0, a1);
                        if (use_q) {
                            const float p0 = j0 <= i ? sqk[nt][2 * hr] : 0.f;
                            const float p1 = j0 + 1 <= i ? sqk[nt][2 * hr + 1] : 0.f;
                            *(uint32_t *)(stg + kOffP + cc_off(i, j0)) = pack_bf16(p0, p1);
                        }
                    }
            }
            __syncwarp();
            // ---- T = (I + A)^{-1}, one column per lane (forward substitution over
            // broadcast row loads); lanes 16..31 repeat lanes 0..15.  Bu = T diag(beta)
            // in bf16 (lanes 0..15) and in tf32 over A (lanes 16..31, after every
            // lane has read A)
            {
                const int jc = lane & (kC - 1);
                const float *Am = (const float *)(stg + kOffBT);
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
                __syncwarp();   // A is read by every lane before Bu in tf32 overwrites it
                if (lane < kC) {
#pragma unroll
                    for (int i = 0; i < kC; ++i)
                        *(__nv_bfloat16 *)(stg + kOffBU + cc_off(i, jc)) = __float2bfloat16_rn(tcol[i] * bj);
                } else {
#pragma unroll
                    for (int i = 0; i < kC; ++i)
                        *(float *)(stg + kOffBT + cc_off_tf32(i, jc)) = tcol[i] * bj;
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
        // One thread issues every tcgen05 MMA of the CTA, in tile order, so the
        // tensor pipe executes them in that order; the product D^T += Y Bu^T waits on
        // an mbarrier for the products that write Y (see below).
        {
            const uint32_t id_u = instr_desc(128, kC, 1, true, false);
            const uint32_t id_x2 = instr_desc(128, 2 * kC, 2, false, false);
            const uint32_t id_x1 = instr_desc(128, kC, 2, false, false);
            const uint32_t id_y = instr_desc(128, kC, 2, false, false);
            const uint32_t id_h = instr_desc(128, kD, 1, false, true);
            const uint32_t id_o = instr_desc(128, kC, 1, false, false);
            const uint32_t s0a = smem_u32(smem);
            const uint64_t dV = smem_desc(s0a + kOffV, kBox, 1024, kSw128);
            const uint64_t dK = smem_desc(s0a + kOffK, kBox, 1024, kSw128);
            const uint64_t dBU = smem_desc(s0a + kOffBU, 128, (kC / 8) * 128, kSwNone);
            const uint64_t dBT = smem_desc(s0a + kOffBT, 128, kTfRowGroup, kSwNone);
            const uint64_t dP = smem_desc(s0a + kOffP, 128, (kC / 8) * 128, kSwNone);
            const uint64_t dWQ = smem_desc(s0a + kOffWQ, 16, 1024, kSw128);
            bool ok = nch == 0 || __all_sync(kFull, mbar_wait(&bar_init[0], 0, args.wait_ns));
            for (int c = 0; c < nch && ok; ++c) {
                if (__any_sync(kFull, *abort_state != 0 || *abort_prep != 0)) {
                    ok = false;
                    break;
                }
                const int st = c % kNS, buf = c & 1;
                const bool use_q = w0 + c >= s0;
                const uint64_t so = (uint64_t)((st * kStage) >> 4);   // stage offset in descriptor units
                const uint32_t cb = kColB + buf * kColBuf;
                if (!__all_sync(kFull, mbar_wait(&bar_prep[st], (uint32_t)(c / kNS) & 1u, args.wait_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    mma_f16_ss(tm + cb, dV + so, dBU + so, id_u, 0);
                    const uint64_t dwq = dWQ + so;
                    const uint32_t id_x = use_q ? id_x2 : id_x1;
#pragma unroll
                    for (int s8 = 0; s8 < kD / 8; ++s8)
                        mma_tf32_ts(tm + cb + kC, tm + kColH + 8 * s8,
                                    dwq + (uint64_t)(((s8 >> 2) * kWQBlock + 32 * (s8 & 3)) >> 4), id_x, s8 > 0);
                    mma_commit(&bar_y[0]);
                }
                __syncwarp();
                // Y is read as an operand only after the products that write it are
                // complete: the tensor pipe does not order a TMEM write and a later MMA's
                // read of it as the A operand (measured: without this wait the read
                // takes partly stale values)
                if (!__all_sync(kFull, mbar_wait(&bar_y[0], (uint32_t)c & 1u, args.wait_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    mma_tf32_ts(tm + cb, tm + cb + kC, dBT + so, id_y, 1);
                    mma_tf32_ts(tm + cb, tm + cb + kC + 8, dBT + so + (uint64_t)(256 >> 4), id_y, 1);
                    mma_commit(&bar_x[buf]);
                }
                __syncwarp();
                if (!__all_sync(kFull, mbar_wait(&bar_a[0], (uint32_t)c & 1u, args.wait_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    mma_f16_ts(tm + kColH, tm + kColA, dK + so, id_h, 1);
                    if (use_q) mma_f16_ts(tm + cb + 2 * kC, tm + kColA, dP + so, id_o, 1);
                    mma_commit(&bar_free[st]);
                }
                __syncwarp();
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
        asm volatile("setmaxnreg.dec.sync.aligned.u32 88;");
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
        const int64_t orow = (int64_t)H * kD;   // elements between token rows
        // one tile's output (bf16 pairs of consecutive tokens) for value index e
        auto store_out = [&](const uint32_t (&o)[kC / 2], int len, int64_t t0) {
            if (!GDR_INBOUNDS(t0 >= 0 && t0 + len <= args.T_total)) return;
            unsigned short *out = (unsigned short *)args.out + (t0 * H + h) * kD + e;
#pragma unroll
            for (int i = 0; i < kC; ++i) {
                if (i < len) *out = (unsigned short)(i & 1 ? o[i / 2] >> 16 : o[i / 2] & 0xffffu);
                out += orow;
            }
        };
        int64_t t0_prev = 0;
        int len_prev = 0, emit_prev = 0;
        int done = 0;
        for (int c = 0; c < nch; ++c) {
            if (__any_sync(kFull, *abort_state != 0 || *abort_prep != 0)) break;
            const int st = c % kNS;
            const uint32_t ph = (uint32_t)(c / kNS) & 1u;
            const int buf = c & 1;
            uint8_t *stg = smem + st * kStage;
            const uint32_t cb = kColB + buf * kColBuf;
            const bool okw = mbar_wait(&bar_prep[st], ph, args.wait_ns) &&
                             mbar_wait(&bar_x[buf], (uint32_t)(c >> 1) & 1u, args.wait_ns);
            if (!__all_sync(kFull, okw)) {
                if (lane == 0) set_status(args.status, GDR_ERR_TIMEOUT);
                *abort_state = 1;
                break;
            }
            tc_fence_after();
            const Hdr *hdr = (const Hdr *)(stg + kOffHdr);
            // the header is read before the arrive below: the update that follows it frees
            // the stage, and the prep warp then writes the header of the stage's next tile
            const int len_c = hdr->len, emit_c = hdr->emit;
            // D^T of this tile (to bf16, the A operand of the update and the output
            // term) and the previous tile's output (complete with this tile's bar_x; read
            // before the arrive, since the next front overwrites its buffer)
            uint32_t ob[kC / 2];   // the previous output, bf16 pairs
            {
                uint32_t dr[kC], orr[kC];
                tmem_ld16(tm + lane_base + cb, dr);
                if (emit_prev) tmem_ld16(tm + lane_base + kColB + (buf ^ 1) * kColBuf + 2 * kC, orr);
                tmem_ld_wait();
                uint32_t a2[kC / 2];
#pragma unroll
                for (int i = 0; i < kC / 2; ++i) {
                    a2[i] = pack_bf16(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1]));
                    ob[i] = pack_bf16(__uint_as_float(orr[2 * i]), __uint_as_float(orr[2 * i + 1]));
                }
                tmem_st8(tm + lane_base + kColA, a2);
            }
            // H^T <- H^T diag(gamma), 16 columns at a time, the next chunk's load in
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
            if (emit_prev) store_out(ob, len_prev, t0_prev);
            t0_prev = sstart + (w0 + c) * kC;
            len_prev = len_c;
            emit_prev = emit_c;
            done = c + 1;
        }
        // drain: the last tile's output, then the final state
        bool ok = done == nch;
        if (ok && nch > 0) ok = __all_sync(kFull, mbar_wait(&bar_h[0], 0, args.wait_ns));
        ok = __all_sync(kFull, ok && *abort_state == 0);
        tc_fence_after();
        if (ok && emit_prev && nch > 0) {
            uint32_t orr[kC], ob[kC / 2];
            tmem_ld16(tm + lane_base + kColB + ((nch - 1) & 1) * kColBuf + 2 * kC, orr);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < kC / 2; ++i)
                ob[i] = pack_bf16(__uint_as_float(orr[2 * i]), __uint_as_float(orr[2 * i + 1]));
            store_out(ob, len_prev, t0_prev);
        }
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

}  // namespace

cudaError_t launch_tc_vec(const void *q, const void *k, const void *v, const void *a,
                          const void *beta, const float *h0, void *out, float *hT, Plan plan,
                          int H, int64_t T_total, float b, int64_t max_segs, const int *warm,
                          int *status, cudaStream_t stream) {
    CUtensorMap mq, mk, mv, ma;
    if (!tc_make_map(&mq, q, H, T_total) || !tc_make_map(&mk, k, H, T_total) ||
        !tc_make_map(&mv, v, H, T_total) || !tc_make_map(&ma, a, H, T_total))
        return cudaErrorInvalidValue;
    if (max_segs <= 0) return cudaSuccess;
    if (max_segs > 0x7fffffff || H > 65535) return cudaErrorInvalidValue;
    TvArgs args{};
    args.beta = (const __nv_bfloat16 *)beta;
    args.h0 = h0;
    args.out = (__nv_bfloat16 *)out;
    args.hT = hT;
    args.warm = warm;
    args.plan = plan;
    args.H = H;
    args.T_total = T_total;
    args.b = b;
    args.status = status;
    args.wait_ns = kWaitNs;
    if (const char *w = std::getenv("GDR_TC_WAIT_NS")) {   // test hook: shorter pipeline waits
        const long long x = std::atoll(w);
        if (x >= 0 && (uint64_t)x < kWaitNs) args.wait_ns = (uint64_t)x;
    }
    cudaError_t err = cudaFuncSetAttribute(tc_vec_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    ProfScope prof(stream, "tc_vec_kernel");
    tc_vec_kernel<<<dim3((unsigned)max_segs, (unsigned)H), kThreads, kSmemBytes, stream>>>(mq, mk, mv, ma,
                                                                                           args);
    count_launch();
    return cudaGetLastError();
}

}  // namespace gdr
