// gdr_vec_mma.cu -- per-channel decay forward, bf16 inputs, dk = dv = 128:
// one fused kernel per (segment, head) that keeps the 128 x 128 fp32 state in
// registers and runs every dense product of a 16-token tile on the tensor cores
// (mma.sync m16n8k8, tf32 operands, fp32 accumulation).
//
// The state is held transposed, H^T (value channel x key channel), as accumulator
// fragments: warp w owns value channels 16w..16w+15, every thread 64 values.  A
// thread's accumulator holds key channels 2t and 2t + 1 of each 8-wide block, which
// is exactly what an A-operand fragment needs if the reduction index inside the
// block is read in the order (2t, 2t + 1) <-> slots (t, t + 4); the B operand is
// loaded from shared memory in the same order, so the sum is unchanged and the
// state never leaves the registers.
//
// Per tile, with per-channel cumulative log-decay G (resetting each tile) and
// the factored decays Kt = K (.) exp(G), Kh = K (.) exp(-G), Qt = Q (.) exp(G)
// [P1 §2.1-2.2, P3 §3.2]:
//   A = beta (.) strict_lower(Kt Kh^T),  P = lower(Qt Kh^T)          (tensor cores)
//   W = (I + A)^{-1} diag(beta) Kt,  U = (I + A)^{-1} diag(beta) V    (forward
//        substitution, one column per thread: no explicit inverse)
//   D = U - W H,  O = Qt H + P D                                       (tensor cores)
//   H <- diag(exp(G_C)) H + (Kh exp(G_C))^T D                          (tensor cores)
// In the transposed form D^T = U^T - H^T W^T, O^T = H^T Qt^T + D^T P^T and
// H^T <- H^T diag(exp(G_C)) + D^T (Kh exp(G_C)) are per-warp; a tile takes four
// block barriers (staging, the Gram products, the substitutions, reuse).
// The next tile's q, k, v and a rows are copied into shared memory (16-byte cp.async,
// bf16 as stored) while the current tile runs its products, so the staging reads
// shared memory instead of waiting on global loads; two blocks share an SM.  The
// outputs of a tile wait in shared memory and go out as whole rows after the next
// barrier.
//
// Long sequences are cut into segments of S tiles (the plan's seg_chunks, 64 to 512,
// larger when there are enough (segment, head) blocks to fill the GPU), one block per
// (segment, head).  A block starts from a zero state at a warm-up tile w before
// its segment and runs the state update alone up to the segment start.  The
// state entering tile w reaches the segment start multiplied by a product of
// (I - beta k k^T) diag(alpha_t); each factor has norm at most
// max(1, |1 - beta |k|^2|) max_d alpha_{t,d}, so the neglected term is at most
// the product of those times that state.  w is the latest tile that makes this
// bound <= e^-46 < 2^-64 (far below fp32 resolution), or the sequence start,
// where the block starts from h0 exactly.  vec_warm_kernel finds w for every
// (segment, head) before the main kernel runs: it walks back from the segment
// start eight tiles at a time, bounding each tile from its a, k and beta, so it
// reads only the tiles its warm-up spans.  A (sequence, head) pair with a segment
// start that has no such w within 4 S tiles runs as one block over the whole
// sequence, exactly as without segments.
#include "gdr_internal.cuh"
#include "gdr_mma.cuh"

namespace gdr {
namespace {

constexpr int kT = 16;       // tile
constexpr int kD = 128;      // dk = dv
constexpr int kLd = 132;     // row stride (floats) of 128-wide shared matrices
constexpr int kPd = 20;      // row stride of 16 x 16 shared matrices
constexpr int kThreads = 256;
constexpr int kSegMin = 64, kSegMax = 512;   // segment lengths in tiles
constexpr int kWarmFactor = 4;   // longest warm-up, in segments, before a pair runs unsegmented
constexpr float kHorizonLog = -46.0f;    // below ln(2^-64) = -44.4, with room for fp32 sums

// shared layout, in floats
constexpr int kOffKt = 0;                     // Kt, then -W   [16][kLd]
constexpr int kOffKh = kOffKt + kT * kLd;     // Kh, then Kh exp(G_C)
constexpr int kOffQt = kOffKh + kT * kLd;     // Qt
constexpr int kOffU = kOffQt + kT * kLd;      // V, then U
constexpr int kOffA = kOffU + kT * kLd;       // A [16][kPd]
constexpr int kOffP = kOffA + kT * kPd;       // P [16][kPd]
constexpr int kOffEg = kOffP + kT * kPd;      // exp(G_C) [128]
constexpr int kOffB = kOffEg + kD;            // beta [16]
constexpr int kOffO = kOffB + kT;             // the tile's outputs, bf16 [16][128]
constexpr int kOffRaw = kOffO + kT * kD / 2;  // next tile's q, k, v, a as stored: bf16 [4][16][128]
constexpr int kSmemFloats = kOffRaw + 4 * kT * kD / 2;
static_assert(kOffO % 4 == 0 && kOffRaw % 4 == 0, "16-byte aligned bf16 tiles");
static_assert(kOffA % 4 == 0 && kPd % 4 == 0, "A rows read in 16-byte pieces");
// Rows 8-15 of a raw tile keep their 16-byte pieces in the order c ^ 2, so that the
// two staging lanes of a channel (tokens i and i + 8) read different banks.
__device__ __forceinline__ int raw_slot(int i, int c16) { return i * kD + 8 * (c16 ^ ((i >> 3) << 1)); }
constexpr size_t kSmemBytes = sizeof(float) * kSmemFloats;

// The log of a bound on the norm of a tile's transition, sum over its tokens of
//   max_d g_{t,d} + ln max(1, |1 - beta_t |k_t|^2|),
// with max_d g = -b sigmoid(min_d a) (the gate is decreasing in a).  One warp per
// tile: lane l loads channels 4l..4l+3 of every token.  The 16 per-token reductions
// over the lanes run as one butterfly that halves the tokens a lane keeps at each
// step: afterwards lanes 2j and 2j + 1 hold the complete minimum and squared norm
// of token j (in a lane-bit order), and each token's term is evaluated once.
// Returns the sum in every lane.

// One butterfly step over n tokens: lanes whose bit `o` is clear keep the first
// n/2, the others the last n/2, each combining its kept half with its partner's.
template <int N, bool MIN>
__device__ __forceinline__ void bound_step(float (&x)[kT], int o, bool upper) {
#pragma unroll
    for (int j = 0; j < N / 2; ++j) {
        const float keep = upper ? x[j + N / 2] : x[j];
        const float give = upper ? x[j] : x[j + N / 2];
        const float got = __shfl_xor_sync(0xffffffffu, give, o);
        x[j] = MIN ? fminf(keep, got) : keep + got;
    }
}

__device__ __forceinline__ float tile_bound_log(const __nv_bfloat16 *__restrict__ a,
                                                const __nv_bfloat16 *__restrict__ k,
                                                const __nv_bfloat16 *__restrict__ beta, int64_t t0,
                                                int len, int H, int h, float b, int lane) {
    uint2 ra[kT], rk[kT];
#pragma unroll
    for (int i = 0; i < kT; ++i) {
        ra[i] = make_uint2(0u, 0u);
        rk[i] = make_uint2(0u, 0u);
        if (i < len) {
            const int64_t r = ((t0 + i) * H + h) * kD + 4 * lane;
            ra[i] = *(const uint2 *)&a[r];
            rk[i] = *(const uint2 *)&k[r];
        }
    }
    // the token this lane ends up holding: bits 4, 3, 2, 1 of the lane, high to low
    const int tk = 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
    const float bt = tk < len ? __bfloat162float(beta[(t0 + tk) * H + h]) : 0.f;
    float m[kT], kk[kT];
#pragma unroll
    for (int i = 0; i < kT; ++i) {
        const float2 a0 = __bfloat1622float2(*(const __nv_bfloat162 *)&ra[i].x);
        const float2 a1 = __bfloat1622float2(*(const __nv_bfloat162 *)&ra[i].y);
        const float2 k0 = __bfloat1622float2(*(const __nv_bfloat162 *)&rk[i].x);
        const float2 k1 = __bfloat1622float2(*(const __nv_bfloat162 *)&rk[i].y);
        m[i] = fminf(fminf(a0.x, a0.y), fminf(a1.x, a1.y));
        kk[i] = k0.x * k0.x + k0.y * k0.y + k1.x * k1.x + k1.y * k1.y;
    }
    bound_step<16, true>(m, 16, (lane >> 4) & 1);
    bound_step<16, false>(kk, 16, (lane >> 4) & 1);
    bound_step<8, true>(m, 8, (lane >> 3) & 1);
    bound_step<8, false>(kk, 8, (lane >> 3) & 1);
    bound_step<4, true>(m, 4, (lane >> 2) & 1);
    bound_step<4, false>(kk, 4, (lane >> 2) & 1);
    bound_step<2, true>(m, 2, (lane >> 1) & 1);
    bound_step<2, false>(kk, 2, (lane >> 1) & 1);
    const float mt = fminf(m[0], __shfl_xor_sync(0xffffffffu, m[0], 1));
    const float kt = kk[0] + __shfl_xor_sync(0xffffffffu, kk[0], 1);
    // token tk's term, counted once (by the even lane of the pair)
    float x = 0.f;
    if (tk < len && (lane & 1) == 0)
        x = gate_logdecay(mt, b, GDR_GATE_BOUNDED) + logf(fmaxf(1.f, fabsf(1.f - bt * kt)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Per (segment, head): the warm-up length s0 - w, where w is the latest tile
// <= s0 (the segment start) whose bound to s0 is <= e^-46, or the sequence start
// when none is; -1 when s0 > 4 S and no w >= s0 - 4 S exists.  Segment 0 writes 0.
// Warp i bounds tile top - 1 - i; warp 0 scans the eight sums from the top down.
// The walk ends after at most 4 S / 8 steps.
constexpr int kWarmWarps = 8;
constexpr int64_t kWalking = -2;

__global__ void __launch_bounds__(32 * kWarmWarps)
vec_warm_kernel(const __nv_bfloat16 *__restrict__ a, const __nv_bfloat16 *__restrict__ k,
                const __nv_bfloat16 *__restrict__ beta, int *__restrict__ warm, Plan p, int H,
                float b) {
    __shared__ float lam_s[kWarmWarps];
    __shared__ long long res;
    const int h = blockIdx.x % H;
    const int64_t sg = blockIdx.x / H;
    const int n = find_owner(p.seg_base, p.N, sg);
    if (n < 0) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t s0 = (sg - p.seg_base[n]) * p.seg_chunks;
    if (s0 == 0) {
        if (threadIdx.x == 0) warm[sg * H + h] = 0;
        return;
    }
    const int64_t sstart = p.seq_start[n], send = p.seq_start[n + 1];
    const int64_t max_warm = (int64_t)kWarmFactor * p.seg_chunks;
    const int64_t floor_w = s0 > max_warm ? s0 - max_warm : 0;   // lowest tile the walk visits
    if (threadIdx.x == 0) res = kWalking;
    float acc = 0.f;   // warp 0: the bound's log over [top, s0)
    for (int64_t top = s0;; top -= kWarmWarps) {
        const int64_t c = top - 1 - warp;
        float lw = 0.f;
        if (c >= floor_w) {
            const int64_t t0 = sstart + c * kT;
            lw = tile_bound_log(a, k, beta, t0, (int)min((int64_t)kT, send - t0), H, h, b, lane);
        }
        if (lane == 0) lam_s[warp] = lw;
        __syncthreads();
        if (warp == 0) {
            const bool valid = lane < kWarmWarps && top - 1 - lane >= floor_w;
            float x = valid ? lam_s[lane] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, valid && acc + x <= kHorizonLog);
            if (lane == 0) {
                if (hit)
                    res = s0 - (top - 1 - (__ffs(hit) - 1));
                else if (top - kWarmWarps <= floor_w)
                    res = floor_w == 0 ? s0 : -1;   // from h0 at the sequence start, or none
            }
            acc += __shfl_sync(0xffffffffu, x, 31);
        }
        __syncthreads();
        const long long r = res;   // written again only after the next first barrier
        if (r != kWalking) {
            if (threadIdx.x == 0) warm[sg * H + h] = (int)r;
            return;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2)
vec_mma_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
               const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ a,
               const __nv_bfloat16 *__restrict__ beta, const float *__restrict__ h0,
               __nv_bfloat16 *__restrict__ out, float *__restrict__ hT, Plan p, int H, float b,
               const int *__restrict__ warm) {
    extern __shared__ float sm[];
    float *Kt = sm + kOffKt, *Kh = sm + kOffKh, *Qt = sm + kOffQt;
    float *Ub = sm + kOffU, *Am = sm + kOffA, *Pm = sm + kOffP, *eg = sm + kOffEg, *bs = sm + kOffB;
    __nv_bfloat16 *Os = (__nv_bfloat16 *)(sm + kOffO);
    __shared__ int warm_start, seg_all;
    const int h = blockIdx.x % H;
    const int64_t sg = blockIdx.x / H;   // global segment
    const int n = find_owner(p.seg_base, p.N, sg);
    if (n < 0) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int c0 = 16 * warp;   // this warp's 16 value channels
    const int64_t tile0 = p.chunk_base[n], ntiles = p.chunk_base[n + 1] - tile0;
    const int64_t j = sg - p.seg_base[n];
    // the pair runs in segments only if every segment start found its warm-up
    if (warp == 0) {
        const int64_t first = p.seg_base[n], nseg = p.seg_base[n + 1] - first;
        bool ok = true;
        for (int64_t i = lane; i < nseg; i += 32) ok = ok && warm[(first + i) * H + h] >= 0;
        ok = __all_sync(0xffffffffu, ok);
        if (lane == 0) {
            seg_all = ok;
            warm_start = ok ? warm[sg * H + h] : 0;
        }
    }
    __syncthreads();
    const bool segmented = seg_all != 0;
    if (!segmented && j > 0) return;   // one block runs the whole sequence
    const int64_t s0 = segmented ? j * p.seg_chunks : 0;
    const int64_t s1 = segmented ? min(ntiles, s0 + (int64_t)p.seg_chunks) : ntiles;
    const int64_t w0 = s0 - warm_start;   // first tile run
    const size_t hbase = ((size_t)n * H + h) * kD * kD;
    const bool from_h0 = w0 == 0 && h0;
    // H^T fragments: hs[nd][u] = H[d][c], c = c0 + g + 8 (u >> 1), d = 8 nd + 2t + (u & 1)
    float hs[kD / 8][4];
#pragma unroll
    for (int nd = 0; nd < kD / 8; ++nd)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + g + 8 * (u >> 1), d = 8 * nd + 2 * t + (u & 1);
            hs[nd][u] = from_h0 ? h0[hbase + (size_t)d * kD + c] : 0.f;
        }
    const int64_t sstart = p.seq_start[n], e_end = p.seq_start[n + 1];
    // Staging is split over all 256 threads: lanes 2d and 2d + 1 of a warp take key
    // (and value) channel d, tokens 0-7 and 8-15; the second half gets the first
    // half's cumulative log-decay from its neighbour lane.
    const int sd = tid >> 1, shalf = tid & 1, si0 = 8 * shalf;
    __nv_bfloat16 *Raw = (__nv_bfloat16 *)(sm + kOffRaw);
    unsigned short rb = 0;   // beta of token tid of the fetched tile, as stored (converted at staging)
    // Copies of a tile's rows into Raw: thread tid takes row tid / 16, 16-byte piece
    // tid % 16, of q, k, v and a; rows past the sequence end are not copied (staging
    // masks them).  Waited for by cp_async_wait_all before the next barrier.
    auto prefetch = [&](int64_t tt) {
        const int64_t t0 = sstart + tt * kT;
        const int len = (int)min((int64_t)kT, e_end - t0);
        const int i = tid >> 4, c16 = tid & 15;
        if (i < len) {
            const int64_t r = ((t0 + i) * H + h) * kD + 8 * c16;
            const int dst = raw_slot(i, c16);
            cp_async16(&Raw[0 * kT * kD + dst], &q[r]);
            cp_async16(&Raw[1 * kT * kD + dst], &k[r]);
            cp_async16(&Raw[2 * kT * kD + dst], &v[r]);
            cp_async16(&Raw[3 * kT * kD + dst], &a[r]);
        }
        cp_async_commit();
        if (tid < len) rb = __bfloat16_as_ushort(beta[(t0 + tid) * H + h]);
    };
    // channel sd of token si0 + u of raw tile X (0 q, 1 k, 2 v, 3 a)
    const int rs0 = raw_slot(si0, sd >> 3) + (sd & 7);
    auto raw = [&](int X, int u) { return __bfloat162float(Raw[X * kT * kD + rs0 + u * kD]); };
    // outputs of a tile wait in Os until the next barrier, then go out as 256-byte rows
    int64_t o_t0 = 0;
    int o_len = 0;
    auto flush_out = [&]() {
        for (int e = tid; e < o_len * (kD / 8); e += kThreads) {
            const int i = e / (kD / 8), c8 = e % (kD / 8);
            *(uint4 *)&out[((o_t0 + i) * H + h) * kD + 8 * c8] = *(const uint4 *)&Os[i * kD + 8 * c8];
        }
        o_len = 0;
    };
    if (w0 < s1) prefetch(w0);
    for (int64_t tt = w0; tt < s1; ++tt) {
        const int64_t t0 = sstart + tt * kT;
        const int len = (int)min((int64_t)kT, e_end - t0);
        const bool emit = tt >= s0;   // warm-up tiles only advance the state
        cp_async_wait_all();   // this thread's copies of the tile have landed
        __syncthreads();       // all copies visible; the previous tile is done with every buffer
        flush_out();           // the previous tile's outputs, whole rows
        // ---- stage the tile: factored decays per key channel, V and beta
        {
            float gl[8], G = 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                gl[u] = si0 + u < len ? gate_logdecay(raw(3, u), b, GDR_GATE_BOUNDED) : 0.f;
                G += gl[u];
            }
            const float Gfirst = __shfl_xor_sync(0xffffffffu, G, 1);   // the other half's total
            G = shalf ? Gfirst : 0.f;                                    // offset of this half
            float eGC = 1.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = si0 + u;
                float kt = 0.f, kh = 0.f, qt = 0.f, vv = 0.f;
                if (i < len) {
                    G += gl[u];
                    const float e = expf(G), en = expf(-G), kd = raw(1, u);
                    kt = kd * e;
                    kh = kd * en;
                    qt = raw(0, u) * e;
                    vv = raw(2, u);
                    eGC = e;
                }
                Kt[i * kLd + sd] = kt;
                Kh[i * kLd + sd] = kh;
                Qt[i * kLd + sd] = qt;
                Ub[i * kLd + sd] = vv;
            }
        // e^{G_C} of channel d: from the half that holds the tile's last token
            const float other = __shfl_xor_sync(0xffffffffu, eGC, 1);
            if (shalf == 0) eg[sd] = len > 8 ? other : eGC;
            if (tid < kT) bs[tid] = tid < len ? __bfloat162float(__ushort_as_bfloat16(rb)) : 0.f;
        }
        __syncthreads();
        if (tt + 1 < s1) prefetch(tt + 1);   // Raw and rb are free until the next staging
        // ---- A = beta (.) strict_lower(Kt Kh^T) and P = lower(Qt Kh^T): warps 0-3
        if (warp < 4) {
            const float *Aop = (warp < 2) ? Kt : Qt;
            const int j0 = 8 * (warp & 1);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int k0 = 0; k0 < kD; k0 += 8) {
                uint32_t af[4];
                load_a(af, Aop, kLd, 0, k0, g, t);
                mma8(acc, af, tf32(Kh[(j0 + g) * kLd + k0 + t]), tf32(Kh[(j0 + g) * kLd + k0 + t + 4]));
            }
            const int i0 = g, i1 = g + 8, ja = j0 + 2 * t, jb = ja + 1;
            if (warp < 2) {
                Am[i0 * kPd + ja] = ja < i0 ? bs[i0] * acc[0] : 0.f;
                Am[i0 * kPd + jb] = jb < i0 ? bs[i0] * acc[1] : 0.f;
                Am[i1 * kPd + ja] = ja < i1 ? bs[i1] * acc[2] : 0.f;
                Am[i1 * kPd + jb] = jb < i1 ? bs[i1] * acc[3] : 0.f;
            } else {
                Pm[i0 * kPd + ja] = ja <= i0 ? acc[0] : 0.f;
                Pm[i0 * kPd + jb] = jb <= i0 ? acc[1] : 0.f;
                Pm[i1 * kPd + ja] = ja <= i1 ? acc[2] : 0.f;
                Pm[i1 * kPd + jb] = jb <= i1 ? acc[3] : 0.f;
            }
        }
        __syncthreads();
        // ---- W and U by forward substitution, one column per thread
        {
            const int col = tid & (kD - 1);
            float *X = tid < kD ? Kt : Ub;   // Kt -> -W, V -> U
            float x[kT];
#pragma unroll
            for (int i = 0; i < kT; ++i) {
                float acc = bs[i] * X[i * kLd + col];
                // row i of A in 16-byte pieces (entries j >= i are zero and unused)
#pragma unroll
                for (int j4 = 0; j4 < i; j4 += 4) {
                    const float4 a4 = *(const float4 *)&Am[i * kPd + j4];
                    const float ar[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (j4 + u < i) acc = fmaf(-ar[u], x[j4 + u], acc);
                }
                x[i] = acc;
            }
            if (tid < kD) {
                const float egc = eg[col];
#pragma unroll
                for (int i = 0; i < kT; ++i) {
                    X[i * kLd + col] = -x[i];
                    Kh[i * kLd + col] *= egc;   // Kh exp(G_C) = K exp(G_C - G)
                }
            } else {
#pragma unroll
                for (int i = 0; i < kT; ++i) X[i * kLd + col] = x[i];
            }
        }
        __syncthreads();
        // ---- D^T = U^T - H^T W^T and O^T = H^T Qt^T (value channels c0..c0+15)
        float dt[2][4], ot[2][4];   // [token tile][fragment]: (c, i = 8 it + 2t + (u & 1))
#pragma unroll
        for (int it = 0; it < 2; ++it)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                dt[it][u] = Ub[(8 * it + 2 * t + (u & 1)) * kLd + c0 + g + 8 * (u >> 1)];
                ot[it][u] = 0.f;
            }
#pragma unroll
        for (int nd = 0; nd < kD / 8; ++nd) {
            const uint32_t ah[4] = {tf32(hs[nd][0]), tf32(hs[nd][2]), tf32(hs[nd][1]), tf32(hs[nd][3])};
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const float2 w2 = *(const float2 *)&Kt[(8 * it + g) * kLd + 8 * nd + 2 * t];   // -W
                const float2 q2 = *(const float2 *)&Qt[(8 * it + g) * kLd + 8 * nd + 2 * t];
                mma8(dt[it], ah, tf32(w2.x), tf32(w2.y));
                mma8(ot[it], ah, tf32(q2.x), tf32(q2.y));
            }
        }
        // D^T as A operands over the tokens (reduction order 2t, 2t + 1 as above)
        uint32_t ad[2][4];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            ad[kk][0] = tf32(dt[kk][0]);
            ad[kk][1] = tf32(dt[kk][2]);
            ad[kk][2] = tf32(dt[kk][1]);
            ad[kk][3] = tf32(dt[kk][3]);
        }
        // ---- O^T += D^T P^T, then the outputs
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const float2 p2 = *(const float2 *)&Pm[(8 * it + g) * kPd + 8 * kk + 2 * t];
                mma8(ot[it], ad[kk], tf32(p2.x), tf32(p2.y));
            }
        if (emit) {
#pragma unroll
            for (int it = 0; it < 2; ++it)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = 8 * it + 2 * t + (u & 1), c = c0 + g + 8 * (u >> 1);
                    Os[i * kD + c] = __float2bfloat16_rn(ot[it][u]);
                }
            o_t0 = t0;
            o_len = len;
        }
        // ---- H^T <- H^T diag(exp(G_C)) + D^T (Kh exp(G_C))
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
    flush_out();
    if (hT && s1 == ntiles)
#pragma unroll
        for (int nd = 0; nd < kD / 8; ++nd)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + g + 8 * (u >> 1), d = 8 * nd + 2 * t + (u & 1);
                hT[hbase + (size_t)d * kD + c] = hs[nd][u];
            }
}

}  // namespace

size_t vec_mma_scratch_bytes(int64_t max_segs, int H) {
    return sizeof(int) * (size_t)max_segs * H + 256;
}

// Segment length: the longest of 64, 128, 256, 512 tiles that still gives about three
// quarters of a wave of (segment, head) blocks (two resident per SM).  Longer segments
// spend less on warm-up tiles (about 20 per segment at the benchmark's decay) and on
// each block's start; measured on the tensor-core kernel, 512-tile segments beat 256
// by 3 % on 1M packed tokens and by 17 % (against 64) on 32 heads x 64K tokens.
int vec_mma_segment_tiles(int64_t tiles, int H, int sms) {
    const int64_t want = (int64_t)3 * 2 * sms / 4;
    int seg = kSegMax;
    while (seg > kSegMin && tiles * H / seg < want) seg /= 2;
    return seg;
}

cudaError_t launch_vec_warm(const void *a, const void *k, const void *beta, int *warm, Plan plan,
                            int H, float b, int64_t max_segs, cudaStream_t stream) {
    if (plan.C != kT || plan.seg_chunks < kSegMin || plan.seg_chunks > kSegMax) return cudaErrorInvalidValue;
    const int64_t blocks = max_segs * H;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    if (blocks == 0) return cudaSuccess;
    ProfScope prof(stream, "vec_warm_kernel");
    vec_warm_kernel<<<(unsigned)blocks, 32 * kWarmWarps, 0, stream>>>(
        (const __nv_bfloat16 *)a, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)beta, warm,
        plan, H, b);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_vec_mma(const void *q, const void *k, const void *v, const void *a,
                           const void *beta, const float *h0, void *out, float *hT, Plan plan,
                           int H, float b, int64_t max_segs, void *scratch, cudaStream_t stream) {
    if (plan.C != kT || plan.seg_chunks < kSegMin || plan.seg_chunks > kSegMax) return cudaErrorInvalidValue;
    const int64_t blocks = max_segs * H;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    if (blocks == 0) return cudaSuccess;
    int *warm = (int *)scratch;
    cudaError_t err = launch_vec_warm(a, k, beta, warm, plan, H, b, max_segs, stream);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(vec_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    ProfScope prof(stream, "vec_mma_kernel");
    vec_mma_kernel<<<(unsigned)blocks, kThreads, kSmemBytes, stream>>>(
        (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v,
        (const __nv_bfloat16 *)a, (const __nv_bfloat16 *)beta, h0, (__nv_bfloat16 *)out, hT, plan,
        H, b, warm);
    count_launch();
    return cudaGetLastError();
}

}  // namespace gdr
