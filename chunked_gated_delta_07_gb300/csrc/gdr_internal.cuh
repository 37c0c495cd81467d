// gdr_internal.cuh -- shared declarations of the library's translation units.
//
// Citation keys used across csrc/ (page title, section):
//   P1 = "Deep Dive: The Next Generation of Ultra-Long Context Sparse MoE LLMs"
//   P2 = "Core Technologies Behind Ultra-Long-Context Sparse MoE Large Models"
//   P3 = "How Trillion-Scale Sparse MoE Models Achieve Million-Token Long
//         Context Capabilities"
//   P4 = "Evaluating Next-Gen Sparse MoE and Long-Context LLMs"
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdr.h"

namespace gdr {

// Description of the packed token axis, built on the device by plan_kernel
// from cu_seqlens (or synthesised for dense input).  All arrays have N+1
// entries; entry N is the total.
struct Plan {
    int N;                        // sequences
    int C;                        // tile length
    int seg_chunks;               // tiles per segment (tensor-core path)
    const int64_t *seq_start;     // token offset of sequence n (seq_start[N] = total)
    const int64_t *chunk_base;    // first global tile of sequence n
    const int64_t *seg_base;      // first global segment of sequence n
};

// Device status word codes (a subset of gdr_status_t).
constexpr int kStatusOk = 0;

// Checking build (-DGDR_DEBUG).  Each translation unit with kernels that check their
// indexes declares GDR_DEBUG_TU() once at namespace scope: a failed GDR_INBOUNDS(cond)
// sets that unit's device flag and the caller skips the access; gdr_get_status reads
// and clears every unit's flag and reports GDR_ERR_BOUNDS.  In regular builds both
// macros compile to nothing.
#ifdef GDR_DEBUG
using DebugFlagReader = int (*)();
bool register_debug_flag(DebugFlagReader fn);
#define GDR_DEBUG_TU()                                                                  \
    namespace {                                                                         \
    __device__ int g_debug_flag = 0;                                                    \
    int read_debug_flag() {                                                             \
        int v = 0, z = 0;                                                               \
        if (cudaMemcpyFromSymbol(&v, g_debug_flag, sizeof(int)) != cudaSuccess) return 0; \
        if (v) cudaMemcpyToSymbol(g_debug_flag, &z, sizeof(int));                       \
        return v;                                                                       \
    }                                                                                   \
    [[maybe_unused]] const bool g_debug_registered = register_debug_flag(&read_debug_flag); \
    }
#define GDR_INBOUNDS(cond) ((cond) ? true : (atomicExch(&g_debug_flag, 1), false))
#else
#define GDR_DEBUG_TU()
#define GDR_INBOUNDS(cond) true
#endif

// First error wins; later ones are dropped.
__device__ __forceinline__ void set_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Index of the sequence that owns global item `idx`, given exclusive bases
// base[0..N] (base[0] = 0, non-decreasing).  Returns -1 when idx >= base[N].
__device__ __forceinline__ int find_owner(const int64_t *base, int N, int64_t idx) {
    if (idx < 0 || idx >= base[N]) return -1;
    int lo = 0, hi = N - 1;  // largest n with base[n] <= idx
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (base[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Log-decay of one token: bounded scaled sigmoid or unbounded negative
// softplus [P1 §3.3, P2 §2.2, P3 §3.2, P4 §2.3].  Both forms are evaluated
// without overflow for any finite a.
__device__ __forceinline__ float gate_logdecay(float a, float b, int gate) {
    if (gate == GDR_GATE_SOFTPLUS) {
        // softplus(a) = max(a, 0) + log1p(exp(-|a|))
        return -(fmaxf(a, 0.f) + log1pf(expf(-fabsf(a))));
    }
    // sigmoid(a) = 1 / (1 + exp(-a)); exp(-a) may be inf for a << 0, giving 0
    return -b / (1.f + expf(-a));
}

// The argument checks of gdr_chunk_fwd_ex (sizes, dtypes, gate, path, null and
// overlapping buffers), for entry points that take the same arguments.
gdr_status_t validate_forward(const void *q, const void *k, const void *v, const void *a,
                              const void *beta, const float *h0, const void *out, const float *hT,
                              const int32_t *cu, int B, int64_t T, int H, int dk, int dv,
                              int chunk, float b, gdr_dtype_t dtype, gdr_gate_t gate,
                              gdr_path_t path);

// ---- launchers (host side; each returns the launch error) -------------------

// Builds the plan arrays (seq_start, chunk_base, seg_base; N+1 each) and
// validates cu_seqlens (NULL => N sequences of T_per tokens each).
cudaError_t launch_plan(const int32_t *cu_seqlens, int N, int64_t T_per, int64_t T_total, int C,
                        int seg_chunks, int64_t *seq_start, int64_t *chunk_base,
                        int64_t *seg_base, int *status, cudaStream_t stream);

// Stage 1: G[h, row] (in-tile inclusive cumsum of the log-decay), and
// optionally beta transposed to head-major fp32 Bt[h, row].
cudaError_t launch_gate_cumsum(const void *a, const void *beta, gdr_dtype_t dtype, float *G,
                               float *Bt, Plan plan, int H, int64_t T_total,
                               int64_t max_chunks, float b, gdr_gate_t gate,
                               cudaStream_t stream);

// Stage 2 on CUDA cores: W, U of every tile (fp32, layouts of k and v).
cudaError_t launch_wy_simt(const void *k, const void *v, const void *beta, const float *G,
                           float *W, float *U, gdr_dtype_t dtype, Plan plan, int H, int dk,
                           int dv, int64_t T_total, int64_t max_chunks, cudaStream_t stream);

// Stages 3+4 on CUDA cores: the tile-to-tile state pass and the outputs.
// The backward pass (gdr_backward.cu).  The plan must be built with 16-token
// tiles (the checkpoint interval); scratch holds bwd_scratch_bytes(...) bytes.
constexpr int kBwTile = 16;
constexpr int kVecTile = 16;        // tile of the per-channel decay path
constexpr float kVecMaxB = 5.0f;    // largest gate bound it takes: exp(16 b) < FLT_MAX
size_t bwd_scratch_bytes(int64_t tiles, int64_t T_total, int H, int dk, int dv);
cudaError_t launch_bwd(const void *q, const void *k, const void *v, const void *a, const void *beta,
                       const float *h0, const void *dout, const float *dhT, void *dq, void *dk_,
                       void *dv, void *da, void *dbeta, float *dh0, gdr_dtype_t dtype, Plan plan,
                       int H, int dk, int dv_dim, int64_t T_total, int64_t tiles, float b,
                       gdr_gate_t gate, void *scratch, cudaStream_t stream);

// The recurrent form over T tokens per sequence, the fp32 state updated in place.
cudaError_t launch_recurrent(const void *q, const void *k, const void *v, const void *a,
                             const void *beta, float *state, void *out, gdr_dtype_t dtype, int N,
                             int64_t T, int H, int dk, int dv, float b, gdr_gate_t gate,
                             cudaStream_t stream);
cudaError_t launch_state_out_simt(const void *q, const void *k, const float *W, const float *U,
                                  const float *G, const float *h0, void *out, float *hT,
                                  gdr_dtype_t dtype, Plan plan, int H, int dk, int dv,
                                  int64_t T_total, cudaStream_t stream);

// Count of kernels launched by the library (incremented by every launcher).
// per-channel decay path (gdr_vec.cu); tiles of 16 tokens, bounded gate
size_t vec_scratch_bytes(int64_t tiles, int64_t T_total, int H, int dk, int dv);
cudaError_t launch_vec_forward(const void *q, const void *k, const void *v, const void *a,
                               const void *beta, const float *h0, void *out, float *hT,
                               gdr_dtype_t dtype, Plan plan, int H, int dk, int dv,
                               int64_t T_total, int64_t max_tiles, float b, void *scratch,
                               cudaStream_t stream);

// per-channel decay, bf16 and dk = dv = 128: fused tensor-core kernel (gdr_vec_mma.cu)
size_t vec_mma_scratch_bytes(int64_t max_segs, int H);
int vec_mma_segment_tiles(int64_t tiles, int H, int sms);
cudaError_t launch_vec_mma(const void *q, const void *k, const void *v, const void *a,
                           const void *beta, const float *h0, void *out, float *hT, Plan plan,
                           int H, float b, int64_t max_segs, void *scratch, cudaStream_t stream);
// The warm-up of every (segment, head) of the plan (int [max_segs][H] in `warm`):
// tiles to run from a zero state before the segment start, 0 at a sequence start,
// -1 when no warm-up within 4 segments bounds the dropped state below 2^-64.
cudaError_t launch_vec_warm(const void *a, const void *k, const void *beta, int *warm, Plan plan,
                            int H, float b, int64_t max_segs, cudaStream_t stream);

// An internal stream and the two events that fork work onto it from the caller's
// stream and join it back (stream = nullptr: run everything on the caller's stream).
struct AuxStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

// backward in the chunked form, bf16 d = 128, bounded gate (gdr_bwd_chunk.cu)
int chunk_bwd_segment_tiles(int64_t tiles, int H, int sms);
size_t chunk_bwd_scratch_bytes(int64_t tiles, int N, int H);
cudaError_t launch_chunk_bwd(const void *q, const void *k, const void *v, const void *a,
                             const void *beta, const float *h0, const void *dout, const float *dhT,
                             void *dq, void *dk, void *dv, void *da, void *dbeta, float *dh0,
                             Plan plan, int H, int64_t T_total, int64_t max_tiles, int64_t max_segs,
                             float b, bool per_channel, void *scratch, int *status, cudaStream_t stream,
                             const AuxStream &aux);

// quantile-balancing router-bias update (gdr_router.cu)
constexpr int kRouterMaxE = 2048;
constexpr int kRouterMaxK = 32;
cudaError_t launch_router_topk(const void *logits, const float *bias, int32_t *idx, float *sel,
                               int64_t *load, int64_t T, int E, int k, gdr_dtype_t dtype,
                               cudaStream_t stream);
cudaError_t launch_router_update(const int64_t *load, float *bias, double *thr, int E, int mode,
                                 double q_lo, double q_hi, float eta, cudaStream_t stream);

void count_launch(uint64_t n = 1);

// Brackets one kernel launch with CUDA events while profiling is enabled
// (gdr_profile_enable); a no-op otherwise.
class ProfScope {
  public:
    ProfScope(cudaStream_t stream, const char *name);
    ~ProfScope();
    ProfScope(const ProfScope &) = delete;
    ProfScope &operator=(const ProfScope &) = delete;

  private:
    cudaStream_t stream_;
    long slot_;
};

}  // namespace gdr
