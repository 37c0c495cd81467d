// gdr_sm100.cuh -- thin inline-PTX wrappers for the sm_100-family features the
// tensor-core path uses: mbarriers (with bounded waits), TMA tile loads,
// tcgen05 (TMEM allocation, MMA, commit, TMEM loads/stores) and the shared-
// memory matrix / instruction descriptors, plus the byte-offset functions
// of the shared-memory operand layouts the kernels write by hand.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gdr {
namespace sm100 {

// ---------------------------------------------------------------- addresses
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// Non-blocking: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for the phase with the given parity to complete.  Gives up after
// `limit_ns` of wall time and returns false (the caller records a timeout
// and unwinds); never spins forever.  (try_wait may itself suspend the thread
// for a while before it reports an incomplete phase.)  A limit of 0 only looks
// once, without suspending: a test hook that makes any wait not already
// satisfied run out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (limit_ns == 0) return mbar_test_wait(bar, parity);
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------- fences
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- TMA
// 3-D tiled load into shared memory, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}
// Bring a 3-D tile of a tensor into L2 ahead of its load (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"((uint64_t)map),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// ---------------------------------------------------------------- tcgen05
// TMEM allocation (one full warp executes these).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_f16_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t accum) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0;"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                           uint32_t accum) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0;"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
__device__ __forceinline__ void mma_tf32_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accum) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0;"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p; }" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
__device__ __forceinline__ void mma_tf32_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accum) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0;"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p; }" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
// D[tmem] = A[tmem] * B[smem] + 2^-S * D[tmem] (kind::tf32; S in [0, 15] is an
// immediate of the instruction: the accumulator is scaled by an exact power of two
// as it is read).
template <int S>
__device__ __forceinline__ void mma_tf32_ts_scale(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc) {
    static_assert(S >= 0 && S <= 15, "scale-input-d range");
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, 1, 0;"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p, %4; }" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "n"(S)
        : "memory");
}
// The same with a run-time S in [0, 15] (one branch per value).
__device__ __forceinline__ void mma_tf32_ts_scaled(uint32_t d, uint32_t a, uint64_t b,
                                                   uint32_t idesc, int s) {
    switch (s) {
        case 0: mma_tf32_ts_scale<0>(d, a, b, idesc); break;
        case 1: mma_tf32_ts_scale<1>(d, a, b, idesc); break;
        case 2: mma_tf32_ts_scale<2>(d, a, b, idesc); break;
        case 3: mma_tf32_ts_scale<3>(d, a, b, idesc); break;
        case 4: mma_tf32_ts_scale<4>(d, a, b, idesc); break;
        case 5: mma_tf32_ts_scale<5>(d, a, b, idesc); break;
        case 6: mma_tf32_ts_scale<6>(d, a, b, idesc); break;
        case 7: mma_tf32_ts_scale<7>(d, a, b, idesc); break;
        case 8: mma_tf32_ts_scale<8>(d, a, b, idesc); break;
        case 9: mma_tf32_ts_scale<9>(d, a, b, idesc); break;
        case 10: mma_tf32_ts_scale<10>(d, a, b, idesc); break;
        case 11: mma_tf32_ts_scale<11>(d, a, b, idesc); break;
        case 12: mma_tf32_ts_scale<12>(d, a, b, idesc); break;
        case 13: mma_tf32_ts_scale<13>(d, a, b, idesc); break;
        case 14: mma_tf32_ts_scale<14>(d, a, b, idesc); break;
        default: mma_tf32_ts_scale<15>(d, a, b, idesc); break;
    }
}
// True in exactly one lane of a converged warp (the warp stays converged around it).
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile("{ .reg .pred p; elect.sync _|p, 0xffffffff; selp.u32 %0, 1, 0, p; }" : "=r"(pred));
    return pred != 0;
}
// Arrive (once) on `bar` when every tcgen05 operation this thread issued so far is complete.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// TMEM -> registers, 32 lanes x 32 bits, N consecutive columns (lane = thread of the warp).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// TMEM address of lane `lane`, column `col` relative to an allocation base.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
    return base + (lane << 16) + col;
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (sm_100 format): start address, leading-
// and stride-dimension byte offsets (all >> 4), version 1, layout type.
enum Swizzle : uint32_t { kSwNone = 0, kSw128 = 2, kSw64 = 4, kSw32 = 6 };

__host__ __device__ constexpr uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                                 uint32_t swizzle) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) |
           ((uint64_t)(swizzle & 7) << 61);
}

// Instruction descriptor of a dense MMA with fp32 accumulation.
//   ab_format: 0 = f16, 1 = bf16, 2 = tf32; a_mn / b_mn: operand is MN-major.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t M, uint32_t N, uint32_t ab_format,
                                                  bool a_mn, bool b_mn) {
    return (1u << 4)                  // D format: f32
           | (ab_format << 7)         // A format
           | (ab_format << 10)        // B format
           | ((a_mn ? 1u : 0u) << 15) // A major
           | ((b_mn ? 1u : 0u) << 16) // B major
           | ((N >> 3) << 17)         // N / 8
           | ((M >> 4) << 24);        // M / 16
}

// ---------------------------------------------------------------- operand layouts
// Byte offset of (row, byte-in-row) inside a 128-byte-swizzled region whose
// rows are 128 bytes (8-row atoms of 1 KiB, 16-byte chunks permuted by the
// row index).  The region must start on a 1 KiB boundary.
__host__ __device__ constexpr uint32_t sw128_off(uint32_t row, uint32_t byte) {
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((((byte >> 4) ^ (row & 7u)) & 7u) << 4) +
           (byte & 15u);
}
// Byte offset in a non-swizzled core-matrix layout: core matrices of 8
// rows x 16 bytes (128 B each); `row` runs within a core matrix at 16 B,
// row groups at `row_group_stride`, 16-byte column groups at `col_group_stride`.
__host__ __device__ constexpr uint32_t core_off(uint32_t row, uint32_t byte,
                                                uint32_t row_group_stride,
                                                uint32_t col_group_stride) {
    return (row >> 3) * row_group_stride + (byte >> 4) * col_group_stride + (row & 7u) * 16u +
           (byte & 15u);
}

}  // namespace sm100
}  // namespace gdr
