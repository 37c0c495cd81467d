// gdr_recurrent.cu -- the token-by-token (recurrent) form of the gated delta
// rule, for decoding: T tokens per sequence (T = 1 is one decode step), the
// fp32 state read from and written back to HBM once per call.
//
// Per token, with alpha = exp(g(a)) and the dk x dv state H [P4 §2.2, P1 §3.3]:
//     p     = alpha H^T k                (the decayed prediction of v)
//     H    <- alpha H + beta k (v - p)^T
//     o     = H^T q
// The dv columns of H are independent, so one block owns one (sequence, head,
// 32-column slice): 256 threads hold the slice in registers (dk / 32 rows x 4
// columns each) for all T tokens; each token needs two reductions over dk
// (p and o), done with warp shuffles and a shared-memory pass over the 8 warps.
// The kernel is bound by HBM traffic of the state (2 x dk x dv x 4 B per
// sequence and head) when T is small.
#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr int kRecCols = 32;       // state columns per block
constexpr int kRecThreads = 256;   // 8 warps: lane & 7 -> 4 columns, the rest -> rows

template <typename T, int DK>
__global__ void __launch_bounds__(kRecThreads)
recurrent_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                 const T *__restrict__ a, const T *__restrict__ beta, float *__restrict__ state,
                 T *__restrict__ out, int N, int64_t Tn, int H, int dv, float b, int gate) {
    constexpr int kRows = DK / 32;   // rows per thread
    __shared__ float red[8][kRecCols];
    __shared__ float vec[2][kRecCols];   // p, then o, for the slice
    __shared__ float kq[2][DK];          // k and q of the current token
    const int nslices = dv / kRecCols;
    const int slice = blockIdx.x % nslices;
    const int64_t nh = blockIdx.x / nslices;   // (sequence, head)
    const int h = (int)(nh % H);
    const int64_t n = nh / H;
    if (n >= N) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c4 = (lane & 7) * 4;            // first of this thread's 4 columns
    const int rg = warp * 4 + (lane >> 3);    // row group 0..31: rows rg + 32 j
    float *S = state + nh * (int64_t)DK * dv + slice * kRecCols + c4;
    float s[kRows][4];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
        const float4 x = *(const float4 *)&S[(int64_t)(rg + 32 * j) * dv];
        s[j][0] = x.x;
        s[j][1] = x.y;
        s[j][2] = x.z;
        s[j][3] = x.w;
    }
    // sum over the 32 row groups of a per-thread 4-column partial; the slice's
    // 32 totals land in dst[0..31]
    auto reduce = [&](float (&part)[4], float *dst) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            part[u] += __shfl_xor_sync(0xffffffffu, part[u], 8);
            part[u] += __shfl_xor_sync(0xffffffffu, part[u], 16);
        }
        if (lane < 8)
#pragma unroll
            for (int u = 0; u < 4; ++u) red[warp][c4 + u] = part[u];
        __syncthreads();
        if (tid < kRecCols) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) acc += red[w][tid];
            dst[tid] = acc;
        }
        __syncthreads();
    };
    for (int64_t t = 0; t < Tn; ++t) {
        const int64_t row = (n * Tn + t) * H + h;   // token row of [N, T, H, .]
        for (int d = tid; d < DK; d += kRecThreads) {
            kq[0][d] = to_f32(k[row * DK + d]);
            kq[1][d] = to_f32(q[row * DK + d]);
        }
        const float alpha = expf(gate_logdecay(to_f32(a[row]), b, gate));
        const float bt = to_f32(beta[row]);
        __syncthreads();
        // p = alpha H^T k
        float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            const float kd = kq[0][rg + 32 * j];
#pragma unroll
            for (int u = 0; u < 4; ++u) part[u] = fmaf(s[j][u], kd, part[u]);
        }
        reduce(part, vec[0]);
        // H <- alpha H + beta k (v - alpha H^T k)^T, and the partials of o = H^T q
        float dl[4], op[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < 4; ++u)
            dl[u] = bt * (to_f32(v[row * dv + slice * kRecCols + c4 + u]) - alpha * vec[0][c4 + u]);
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            const float kd = kq[0][rg + 32 * j], qd = kq[1][rg + 32 * j];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                s[j][u] = fmaf(alpha, s[j][u], kd * dl[u]);
                op[u] = fmaf(s[j][u], qd, op[u]);
            }
        }
        reduce(op, vec[1]);
        if (tid < kRecCols) out[row * dv + slice * kRecCols + tid] = from_f32<T>(vec[1][tid]);
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j)
        *(float4 *)&S[(int64_t)(rg + 32 * j) * dv] = make_float4(s[j][0], s[j][1], s[j][2], s[j][3]);
}

template <typename T>
cudaError_t launch_t(const void *q, const void *k, const void *v, const void *a, const void *beta,
                     float *state, void *out, int N, int64_t Tn, int H, int dk, int dv, float b,
                     int gate, cudaStream_t stream) {
    const int64_t blocks = (int64_t)N * H * (dv / kRecCols);
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    ProfScope prof(stream, "recurrent_kernel");
    if (dk == 128)
        recurrent_kernel<T, 128><<<(unsigned)blocks, kRecThreads, 0, stream>>>(
            (const T *)q, (const T *)k, (const T *)v, (const T *)a, (const T *)beta, state, (T *)out,
            N, Tn, H, dv, b, gate);
    else
        recurrent_kernel<T, 64><<<(unsigned)blocks, kRecThreads, 0, stream>>>(
            (const T *)q, (const T *)k, (const T *)v, (const T *)a, (const T *)beta, state, (T *)out,
            N, Tn, H, dv, b, gate);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent(const void *q, const void *k, const void *v, const void *a,
                             const void *beta, float *state, void *out, gdr_dtype_t dtype, int N,
                             int64_t T, int H, int dk, int dv, float b, gdr_gate_t gate,
                             cudaStream_t stream) {
    if (N == 0 || T == 0) return cudaSuccess;
    if (dtype == GDR_BF16)
        return launch_t<__nv_bfloat16>(q, k, v, a, beta, state, out, N, T, H, dk, dv, b, (int)gate,
                                       stream);
    return launch_t<float>(q, k, v, a, beta, state, out, N, T, H, dk, dv, b, (int)gate, stream);
}

}  // namespace gdr
