// gdr_router.cu -- the quantile-balancing router-bias update (aux-loss-free
// load balancing) [P1 §4.2, P2 §3.2, P3 §4.3, P4 §3.2]:
//   1. every token picks the k experts of largest score logit + bias
//      (binary32 add; equal scores go to the lower expert index);
//   2. load_e counts the tokens that picked expert e (int64, accumulated);
//   3. quantiles of the loads by linear interpolation between order statistics;
//   4. sign step (bias -= eta above Q(q_hi), += eta below Q(q_lo)) or
//      proportional step (bias += eta (Q - load) / Q), binary64 then rounded.
//
// router_topk_kernel is the hot part: it reads the [T, E] logits once.  One
// warp per token; lane l owns experts 4c..4c+3 for c = l, l + 32, ...  The scores
// stay in registers as floats and each lane keeps their maximum.  The k-th largest
// of the 32 lane maxima, found with k warp-wide max reductions, bounds the k-th
// largest score from below; the reductions run on order-preserving 32-bit keys whose
// low 5 bits are replaced by the lane index (which makes them distinct, and only
// lowers the bound).  Only scores >= that bound can be selected: each lane marks
// them in a bit mask, the warp gathers them (usually a dozen; the logit is read back
// from a per-warp copy of the row in shared memory) and ranks them exactly by
// (score, -index).  When more than kCap scores pass, or fewer than k (NaN scores
// never pass), the warp falls back to k rounds of a warp-wide arg-max over (score,
// -index).  Loads are counted in a shared-memory histogram per block and added to
// the int64 counts once per block.
#include <algorithm>

#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr int kRtThreads = 256;
constexpr int kRtWarps = kRtThreads / 32;
constexpr int kCap = 64;     // gathered candidates per warp

// Order-preserving map of a binary32 score onto uint32 (-0 taken as +0).
__device__ __forceinline__ uint32_t score_key(float s) {
    const uint32_t u = __float_as_uint(s + 0.0f);
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);   // negative: ~u, else u | sign
}

// The score of a key (the inverse of score_key).
__device__ __forceinline__ float key_score(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

// max(a, b, c) in one instruction (the three-input form of max.f32).  Only the lane
// maxima use it; they feed a lower bound, so its choice between -0 and +0, or its
// handling of NaN, cannot change a selection (a NaN bound sends the token to the
// arg-max rounds).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// (key, -index) packed so that a larger value is the better expert.
__device__ __forceinline__ uint64_t pack(uint32_t key, int e) {
    return ((uint64_t)key << 32) | (uint64_t)(0xffffffffu - (uint32_t)e);
}

// Asynchronous copy of one lane's four logits (8 or 16 bytes) into shared memory;
// complete for the issuing thread after cp.async.wait_group.
__device__ __forceinline__ void copy_async(void *smem, const void *gmem, int bytes) {
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    if (bytes == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(sa), "l"(gmem) : "memory");
}

template <typename T> struct Vec4;
template <> struct Vec4<__nv_bfloat16> {
    using type = uint2;   // four bf16 in 8 bytes
    __device__ static void unpack(const type &x, float (&f)[4]) {
        f[0] = __uint_as_float(x.x << 16);
        f[1] = __uint_as_float(x.x & 0xffff0000u);
        f[2] = __uint_as_float(x.y << 16);
        f[3] = __uint_as_float(x.y & 0xffff0000u);
    }
    __device__ static float at(const __nv_bfloat16 *row, int e) { return __bfloat162float(row[e]); }
};
template <> struct Vec4<float> {
    using type = float4;
    __device__ static void unpack(const type &x, float (&f)[4]) {
        f[0] = x.x;
        f[1] = x.y;
        f[2] = x.z;
        f[3] = x.w;
    }
    __device__ static float at(const float *row, int e) { return row[e]; }
};

// Bit mask of a lane's NCH * 4 scores.
template <int NCH> struct LaneMask { using type = uint32_t; };
template <> struct LaneMask<16> { using type = uint64_t; };
__device__ __forceinline__ int lowest_bit(uint32_t m) { return __ffs(m) - 1; }
__device__ __forceinline__ int lowest_bit(uint64_t m) { return __ffsll((long long)m) - 1; }
__device__ __forceinline__ int bit_count(uint32_t m) { return __popc(m); }
__device__ __forceinline__ int bit_count(uint64_t m) { return __popcll(m); }

// ECT > 0 fixes the expert count and KCT > 0 the pick count at compile time (the
// bounds checks fold away, the threshold rounds unroll).
template <typename T, int NCH, int ECT, int KCT>
__global__ void __launch_bounds__(kRtThreads, NCH > 8 ? 1 : (NCH > 7 ? 2 : 3))
router_topk_kernel(const T *__restrict__ logits, const float *__restrict__ bias,
                   int32_t *__restrict__ idx, float *__restrict__ sel,
                   unsigned long long *__restrict__ load, int64_t Tn, int E_arg, int k_arg) {
    static_assert(NCH * 4 <= 8 * (int)sizeof(typename LaneMask<NCH>::type), "mask too narrow");
    using M = typename LaneMask<NCH>::type;
    using V = typename Vec4<T>::type;
    const int E = ECT > 0 ? ECT : E_arg;
    const int k = KCT > 0 ? KCT : k_arg;
    // [E] counts, [E] bias, then two rows of logits per warp ([kRtWarps][2][E]): the
    // current token's, and the next one's, in flight
    extern __shared__ unsigned int hist[];
    float *bsm = (float *)(hist + E);
    __shared__ __align__(16) uint64_t cand[kRtWarps][kCap];
    __shared__ float cand_x[kRtWarps][kCap];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    T *rows = (T *)(bsm + E) + (size_t)warp * 2 * E;
    for (int e = threadIdx.x; e < E; e += kRtThreads) {
        hist[e] = 0;
        bsm[e] = bias[e];
    }
    __syncthreads();
    const int64_t nwarps = (int64_t)gridDim.x * kRtWarps;
    // each lane copies its own chunks of a row (and reads only those), so the row
    // buffers need no barrier between the lanes
    int64_t t = (int64_t)blockIdx.x * kRtWarps + warp;
    auto fetch = [&](int64_t tt, T *dst) {
        if (tt < Tn) {
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
                const int c = lane + 32 * j;
                if (4 * c < E) copy_async(dst + 4 * c, logits + tt * E + 4 * c, (int)sizeof(V));
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    fetch(t, rows);
    for (int buf = 0; t < Tn; t += nwarps, buf ^= 1) {
        const T *row = rows + buf * E;
        fetch(t + nwarps, rows + (buf ^ 1) * E);
        asm volatile("cp.async.wait_group 1;" ::: "memory");   // this row's copies landed
        // the scores and the lane maximum
        float sc[NCH][4];
        float lmax = -INFINITY;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
            const int c = lane + 32 * j;
            if (4 * c < E) {
                float x[4];
                Vec4<T>::unpack(*(const V *)&row[4 * c], x);
                const float4 bz = *(const float4 *)&bsm[4 * c];
                sc[j][0] = x[0] + bz.x;
                sc[j][1] = x[1] + bz.y;
                sc[j][2] = x[2] + bz.z;
                sc[j][3] = x[3] + bz.w;
                lmax = max3(lmax, max3(sc[j][0], sc[j][1], sc[j][2]), sc[j][3]);
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u) sc[j][u] = -INFINITY;
            }
        }
        // tau: the k-th largest lane maximum, as a key with the lane index in its low 5
        // bits (lanes without experts offer 0); with fewer than k lanes the last rounds
        // find 0, and tau takes every score
        uint32_t tau_key;
        {
            const uint32_t lk = 4 * lane < E ? (score_key(lmax) & ~31u) | (uint32_t)lane : 0u;
            bool alive = true;
            uint32_t m = 0;
#pragma unroll
            for (int r = 0; r < k; ++r) {
                m = __reduce_max_sync(0xffffffffu, alive ? lk : 0u);
                alive = alive && (int)(m & 31u) != lane;
            }
            tau_key = m & ~31u;
        }
        const float tau = key_score(max(tau_key, 0x007fffffu));   // at least -inf
        // the scores >= tau: a bit per score, then their positions in the warp's list
        M mask = 0;
#pragma unroll
        for (int j = 0; j < NCH; ++j)
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (4 * (lane + 32 * j) + u < E && sc[j][u] >= tau) mask |= (M)1 << (4 * j + u);
        const int cnt = bit_count(mask);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (total >= k && total <= kCap) {
            int pos = incl - cnt;
            while (mask) {
                const int b = lowest_bit(mask);
                mask &= mask - 1;
                const int e = 4 * (lane + 32 * (b >> 2)) + (b & 3);
                const float x = Vec4<T>::at(row, e);
                cand[warp][pos] = pack(score_key(x + bsm[e]), e);
                cand_x[warp][pos] = x;
                ++pos;
            }
            if (lane == 0 && (total & 1)) cand[warp][total] = 0;   // pads the list to pairs
            __syncwarp();
            for (int ci = lane; ci < total; ci += 32) {
                const uint64_t me = cand[warp][ci];
                int rank = 0;
                for (int cj = 0; cj < total; cj += 2) {   // two candidates per load
                    const ulonglong2 q = *(const ulonglong2 *)&cand[warp][cj];
                    rank += (q.x > me ? 1 : 0) + (q.y > me ? 1 : 0);
                }
                if (rank < k) {
                    const int e = (int)(0xffffffffu - (uint32_t)me);
                    idx[t * k + rank] = e;
                    if (sel) sel[t * k + rank] = cand_x[warp][ci];
                    atomicAdd(&hist[e], 1u);
                }
            }
            __syncwarp();
        } else {
            // many ties at the threshold (or NaN scores): k rounds of a warp-wide arg-max;
            // a NaN score ranks as -inf, and every pick is a valid expert index
            M taken = 0;
            for (int r = 0; r < k; ++r) {
                uint64_t best = 0;
                int bb = -1;
#pragma unroll
                for (int j = 0; j < NCH; ++j)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int b = 4 * j + u, e = 4 * (lane + 32 * j) + u;
                        const float s = sc[j][u] != sc[j][u] ? -INFINITY : sc[j][u];
                        const uint64_t p = (e < E && !((taken >> b) & 1)) ? pack(score_key(s), e) : 0ull;
                        if (p > best) {
                            best = p;
                            bb = b;
                        }
                    }
                uint64_t w = best;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const uint64_t y = __shfl_xor_sync(0xffffffffu, w, o);
                    w = y > w ? y : w;
                }
                if (best == w && bb >= 0) {   // the lane that owns the winner records and removes it
                    const int e = (int)(0xffffffffu - (uint32_t)w);
                    taken |= (M)1 << bb;
                    idx[t * k + r] = e;
                    if (sel) sel[t * k + r] = Vec4<T>::at(row, e);
                    atomicAdd(&hist[e], 1u);
                }
                __syncwarp();
            }
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");   // (the last, empty group)
    __syncthreads();
    if (load)
        for (int e = threadIdx.x; e < E; e += kRtThreads)
            if (hist[e]) atomicAdd(&load[e], (unsigned long long)hist[e]);
}

// One block: rank sort of the loads, the two quantiles, then the bias step.
__global__ void __launch_bounds__(1024)
router_update_kernel(const long long *__restrict__ load, float *__restrict__ bias,
                     double *__restrict__ thr, int E, int mode, double q_lo, double q_hi,
                     float eta) {
    extern __shared__ long long sm_load[];   // [E] loads, then [E] sorted
    long long *srt = sm_load + E;
    __shared__ double Q[2];
    for (int e = threadIdx.x; e < E; e += blockDim.x) sm_load[e] = load[e];
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
        const long long li = sm_load[i];
        int r = 0;
        for (int j = 0; j < E; ++j) {
            const long long lj = sm_load[j];
            r += (lj < li || (lj == li && j < i)) ? 1 : 0;
        }
        srt[r] = li;
    }
    __syncthreads();
    if (threadIdx.x < 2) {
        const double q = threadIdx.x == 0 ? q_lo : q_hi;
        const double p = __dmul_rn(q, (double)(E - 1));
        int i = (int)floor(p);
        if (i > E - 1) i = E - 1;
        const int j = i + 1 < E ? i + 1 : i;
        const double xi = (double)srt[i], xj = (double)srt[j];
        Q[threadIdx.x] = __dadd_rn(xi, __dmul_rn(__dsub_rn(p, (double)i), __dsub_rn(xj, xi)));
        if (thr) thr[threadIdx.x] = Q[threadIdx.x];
    }
    __syncthreads();
    const double Qlo = Q[0], Qhi = Q[1];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const double l = (double)sm_load[e];
        const float b0 = bias[e];
        float b1 = b0;
        if (mode == GDR_QB_SIGN) {
            if (l > Qhi) b1 = __fsub_rn(b0, eta);
            else if (l < Qlo) b1 = __fadd_rn(b0, eta);
        } else if (Qhi != 0.0) {
            b1 = __double2float_rn(
                __dadd_rn((double)b0, __ddiv_rn(__dmul_rn((double)eta, __dsub_rn(Qhi, l)), Qhi)));
        }
        bias[e] = b1;
    }
}

template <typename T, int NCH, int ECT = 0, int KCT = 0>
cudaError_t launch_topk_t(const void *logits, const float *bias, int32_t *idx, float *sel,
                          int64_t *load, int64_t Tn, int E, int k, cudaStream_t stream) {
    auto kern = router_topk_kernel<T, NCH, ECT, KCT>;
    const size_t smem = (sizeof(unsigned int) + sizeof(float) + sizeof(T) * 2 * kRtWarps) * (size_t)E;
    int dev = 0, sms = 0;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err == cudaSuccess) err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    // one wave of resident blocks (each warp then walks its tokens with the next row
    // in flight), so that every SM holds as many warps as registers allow
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRtThreads, smem);
    if (err != cudaSuccess) return err;
    const int64_t want = (Tn + kRtWarps - 1) / kRtWarps;
    const int64_t grid = std::min<int64_t>(want, (int64_t)sms * std::max(per_sm, 1));
    ProfScope prof(stream, "router_topk_kernel");
    kern<<<(unsigned)grid, kRtThreads, smem, stream>>>((const T *)logits, bias, idx, sel,
                                                       (unsigned long long *)load, Tn, E, k);
    count_launch();
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_topk_dt(const void *logits, const float *bias, int32_t *idx, float *sel,
                           int64_t *load, int64_t Tn, int E, int k, cudaStream_t stream) {
    if (E <= 128) return launch_topk_t<T, 1>(logits, bias, idx, sel, load, Tn, E, k, stream);
    if (E <= 256) return launch_topk_t<T, 2>(logits, bias, idx, sel, load, Tn, E, k, stream);
    if (E <= 512) return launch_topk_t<T, 4>(logits, bias, idx, sel, load, Tn, E, k, stream);
    if (E == 896 && k == 8) return launch_topk_t<T, 7, 896, 8>(logits, bias, idx, sel, load, Tn, E, k, stream);
    if (E == 896) return launch_topk_t<T, 7, 896>(logits, bias, idx, sel, load, Tn, E, k, stream);
    if (E <= 896) return launch_topk_t<T, 7>(logits, bias, idx, sel, load, Tn, E, k, stream);
    if (E <= 1024) return launch_topk_t<T, 8>(logits, bias, idx, sel, load, Tn, E, k, stream);
    return launch_topk_t<T, 16>(logits, bias, idx, sel, load, Tn, E, k, stream);
}

}  // namespace

cudaError_t launch_router_topk(const void *logits, const float *bias, int32_t *idx, float *sel,
                               int64_t *load, int64_t T, int E, int k, gdr_dtype_t dtype,
                               cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (dtype == GDR_BF16)
        return launch_topk_dt<__nv_bfloat16>(logits, bias, idx, sel, load, T, E, k, stream);
    return launch_topk_dt<float>(logits, bias, idx, sel, load, T, E, k, stream);
}

cudaError_t launch_router_update(const int64_t *load, float *bias, double *thr, int E, int mode,
                                 double q_lo, double q_hi, float eta, cudaStream_t stream) {
    const size_t smem = 2 * sizeof(long long) * (size_t)E;
    cudaError_t err = cudaFuncSetAttribute(router_update_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    ProfScope prof(stream, "router_update_kernel");
    router_update_kernel<<<1, 1024, smem, stream>>>((const long long *)load, bias, thr, E, mode,
                                                    q_lo, q_hi, eta);
    count_launch();
    return cudaGetLastError();
}

}  // namespace gdr
