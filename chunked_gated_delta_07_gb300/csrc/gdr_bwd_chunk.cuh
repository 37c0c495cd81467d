// gdr_bwd_chunk.cuh -- what the chunked backward's kernels share: the argument
// block and the walk that finds each segment's warm-up tiles.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdr_internal.cuh"

namespace gdr {
namespace bwdc {

constexpr float kHorizonLog = -46.0f;   // below ln(2^-64) = -44.4, with room for fp32 sums

// Stored per tile and head: Hst the entering state H0 ([dk][dv], bf16), dHst the
// end-of-tile gradient scaled by the tile's decay, X = diag(e^{G_C}) dH1 ([dk][dv],
// bf16; every use of dH1 in the tile gradients is through X), Dst the tile's D.
struct BcArgs {
    const __nv_bfloat16 *q, *k, *v, *a, *beta, *dout;
    const float *h0, *dhT;
    __nv_bfloat16 *dq, *dk, *dv, *da, *dbeta;
    float *dh0;
    __nv_bfloat16 *Hst, *dHst;   // [tiles][H][128][128]: H0, and X = diag(e^{G_C}) dH1
    float *Dst;                  // [tiles][H][16][128]: D of the forward chain
    float *dDst;                 // [tiles][H][16][128]: dD of the adjoint chain
    const float *lam;            // [tiles][H]: log bound of each tile's transition
    const int *seg_ok;           // [N][H]: 1 if the pair runs in segments
    Plan p;
    int H;
    float b;
};

// Warp-wide walk over the per-tile log bounds from tile `from` of a sequence with
// `nt` tiles: backwards (dir < 0) to the latest start w <= from whose tiles
// [w, from) sum to <= e^-46, or 0; forwards (dir > 0) to the earliest end
// e >= from whose tiles [from, e) do, or nt.
__device__ __forceinline__ int64_t warm_walk(const float *lam, int64_t tile0, int64_t nt, int H, int h,
                                             int64_t from, int dir) {
    const int lane = threadIdx.x & 31;
    int64_t w = from;
    float acc = 0.f;
    bool done = dir < 0 ? from == 0 : from >= nt;
    while (!done) {
        const int64_t i = dir < 0 ? w - 1 - lane : w + lane;
        const bool in = i >= 0 && i < nt;
        float x = in ? lam[(tile0 + i) * H + h] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, in && acc + x <= kHorizonLog);
        if (hit) {
            const int l = __ffs(hit) - 1;
            w = dir < 0 ? w - 1 - l : w + 1 + l;
            done = true;
        } else {
            acc += __shfl_sync(0xffffffffu, x, 31);
            w = dir < 0 ? max(w - 32, (int64_t)0) : min(w + 32, nt);
            done = dir < 0 ? w == 0 : w == nt;
        }
    }
    return w;
}

// Segment of block `sg` (global segment index): sequence n and tiles [s0, s1);
// false when the block has nothing to do.
__device__ __forceinline__ bool segment_of(const BcArgs &A, int64_t sg, int h, int &n, int64_t &s0,
                                           int64_t &s1) {
    n = find_owner(A.p.seg_base, A.p.N, sg);
    if (n < 0) return false;
    const int64_t nt = A.p.chunk_base[n + 1] - A.p.chunk_base[n];
    const int64_t j = sg - A.p.seg_base[n];
    if (A.seg_ok[(int64_t)n * A.H + h]) {
        s0 = j * A.p.seg_chunks;
        s1 = min(nt, s0 + (int64_t)A.p.seg_chunks);
    } else {
        if (j > 0) return false;
        s0 = 0;
        s1 = nt;
    }
    return true;
}

}  // namespace bwdc

// The adjoint chain on tcgen05 (gdr_tc_adj.cu), a drop-in for bwd_adj_chain_kernel:
// cudaErrorNotSupported (and nothing launched) when a tensor map cannot be made
// (a base not 16-byte aligned).
cudaError_t launch_tc_adj(const bwdc::BcArgs &A, bool per_channel, int64_t T_total, int64_t max_tiles,
                          int64_t max_segs, int *status, cudaStream_t stream);

// The forward state chain on tcgen05 (gdr_tc_fwd_chain.cu), a drop-in for
// bwd_fwd_chain_kernel, with the same fallback rule.
cudaError_t launch_tc_fwd_chain(const bwdc::BcArgs &A, bool per_channel, int64_t T_total, int64_t max_tiles,
                                int64_t max_segs, int *status, cudaStream_t stream);

}  // namespace gdr
