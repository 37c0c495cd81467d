// gdr_mma.cuh -- warp-level tensor-core helpers (mma.sync m16n8k8, tf32 inputs,
// fp32 accumulators) shared by the fused per-tile kernels.
//
// Fragment layout of m16n8k8 with g = lane / 4 and t = lane % 4:
//   A (16 x 8, row major): a0 = A[g][t], a1 = A[g+8][t], a2 = A[g][t+4], a3 = A[g+8][t+4]
//   B (8 x 8):             b0 = B[t][g], b1 = B[t+4][g]
//   C (16 x 8):            c0 = C[g][2t], c1 = C[g][2t+1], c2 = C[g+8][2t], c3 = C[g+8][2t+1]
#pragma once

#include <cstdint>

#include <cuda_bf16.h>

namespace gdr {

// The tensor cores read the top 19 bits of an fp32 operand (sign, exponent and 10
// mantissa bits); the low bits are ignored, which truncates rather than rounds.
__device__ __forceinline__ uint32_t tf32(float x) { return __float_as_uint(x); }

// d += a * b
__device__ __forceinline__ void mma8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A fragment: rows r0..r0+15, columns k0..k0+7 of a row-major matrix M (stride ld)
__device__ __forceinline__ void load_a(uint32_t (&a)[4], const float *M, int ld, int r0, int k0,
                                       int g, int t) {
    a[0] = tf32(M[(r0 + g) * ld + k0 + t]);
    a[1] = tf32(M[(r0 + g + 8) * ld + k0 + t]);
    a[2] = tf32(M[(r0 + g) * ld + k0 + t + 4]);
    a[3] = tf32(M[(r0 + g + 8) * ld + k0 + t + 4]);
}

// A fragment of the transpose: A = M^T, i.e. A[r][k] = M[k][r]
__device__ __forceinline__ void load_at(uint32_t (&a)[4], const float *M, int ld, int r0, int k0,
                                        int g, int t) {
    a[0] = tf32(M[(k0 + t) * ld + r0 + g]);
    a[1] = tf32(M[(k0 + t) * ld + r0 + g + 8]);
    a[2] = tf32(M[(k0 + t + 4) * ld + r0 + g]);
    a[3] = tf32(M[(k0 + t + 4) * ld + r0 + g + 8]);
}

// B fragment: B[k][n] = M[k][n] (row-major K x N), k0..k0+7, n0..n0+7
__device__ __forceinline__ void load_b(uint32_t &b0, uint32_t &b1, const float *M, int ld, int k0,
                                       int n0, int g, int t) {
    b0 = tf32(M[(k0 + t) * ld + n0 + g]);
    b1 = tf32(M[(k0 + t + 4) * ld + n0 + g]);
}

// B fragment of the transpose: B[k][n] = M[n][k]
__device__ __forceinline__ void load_bt(uint32_t &b0, uint32_t &b1, const float *M, int ld, int k0,
                                        int n0, int g, int t) {
    b0 = tf32(M[(n0 + g) * ld + k0 + t]);
    b1 = tf32(M[(n0 + g) * ld + k0 + t + 4]);
}

}  // namespace gdr

namespace gdr {

// B fragments from a bf16 row-major matrix (values widened exactly, then tf32)
__device__ __forceinline__ void load_b_h(uint32_t &b0, uint32_t &b1, const __nv_bfloat16 *M, int ld,
                                         int k0, int n0, int g, int t) {
    b0 = tf32(__bfloat162float(M[(k0 + t) * ld + n0 + g]));
    b1 = tf32(__bfloat162float(M[(k0 + t + 4) * ld + n0 + g]));
}

__device__ __forceinline__ void load_bt_h(uint32_t &b0, uint32_t &b1, const __nv_bfloat16 *M, int ld,
                                          int k0, int n0, int g, int t) {
    b0 = tf32(__bfloat162float(M[(n0 + g) * ld + k0 + t]));
    b1 = tf32(__bfloat162float(M[(n0 + g) * ld + k0 + t + 4]));
}

// Fragments of a product whose k index runs along the rows of both operands, with k
// permuted the same way on both sides (slot t <-> column k0 + 2t, slot t + 4 <-> column
// k0 + 2t + 1), which leaves the product unchanged: each pair of slots is one 8-byte
// (fp32) or 4-byte (bf16) load.  A row stride of 8 mod 32 words keeps the fp32 loads
// free of bank conflicts (a half warp reads 4 rows x 8 words).
__device__ __forceinline__ void load_a_kp(uint32_t (&a)[4], const float *M, int ld, int r0, int k0,
                                          int g, int t) {
    const float2 x = *(const float2 *)&M[(r0 + g) * ld + k0 + 2 * t];
    const float2 y = *(const float2 *)&M[(r0 + g + 8) * ld + k0 + 2 * t];
    a[0] = tf32(x.x);
    a[2] = tf32(x.y);
    a[1] = tf32(y.x);
    a[3] = tf32(y.y);
}

// B[k][n] = M[n][k], k permuted as in load_a_kp
__device__ __forceinline__ void load_bt_kp(uint32_t &b0, uint32_t &b1, const float *M, int ld, int k0,
                                           int n0, int g, int t) {
    const float2 x = *(const float2 *)&M[(n0 + g) * ld + k0 + 2 * t];
    b0 = tf32(x.x);
    b1 = tf32(x.y);
}

// B[k][n] = M[n][k] from a bf16 row-major matrix, k permuted as in load_a_kp (the two
// values widened exactly: a bf16 is the top half of its fp32)
__device__ __forceinline__ void load_bt_h_kp(uint32_t &b0, uint32_t &b1, const __nv_bfloat16 *M, int ld,
                                             int k0, int n0, int g, int t) {
    const uint32_t x = *(const uint32_t *)&M[(n0 + g) * ld + k0 + 2 * t];
    b0 = x << 16;
    b1 = x & 0xffff0000u;
}

}  // namespace gdr

namespace gdr {

// 16-byte asynchronous copy global -> shared (completion: cp_async_wait_all)
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

}  // namespace gdr
