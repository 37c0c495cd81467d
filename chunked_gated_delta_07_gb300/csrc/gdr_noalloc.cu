// gdr_noalloc.cu -- gdr_chunk_fwd_noalloc: the fp32 CUDA-core forward pass
// for dense input, with all of its scratch in one statically allocated device
// array instead of memory obtained from cudaMalloc.
//
// Why it exists.  Some callers are not allowed to allocate device memory at
// the moment they run the pass: code that executes while a CUDA graph is
// being captured (cudaMalloc is not capturable), engines that reserve all
// device memory for their own pool at start-up and forbid later
// allocations, and latency-critical loops where an allocation (and the
// device synchronisation that freeing a grown buffer implies) is not
// acceptable.  Those callers still pass their own inputs and outputs; this
// entry point only removes the library's own scratch allocation.
//
// The scratch array below is part of the module: every GPU that loads the
// library holds it until the process exits.  Its host-side name is only a
// stand-in for the symbol, so the device address is looked up once per
// device with cudaGetSymbolAddress (on the first call made on that device,
// which should therefore come before any stream capture) and that address
// is what the kernels receive.
#include <mutex>

#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per device).
cudaError_t noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

inline size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace gdr

using namespace gdr;

extern "C" gdr_status_t gdr_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                              const void *a, const void *beta, const float *h0,
                                              void *out, float *hT, int B, int64_t T, int H,
                                              int dk, int dv, int chunk, float b,
                                              gdr_dtype_t dtype, gdr_gate_t gate,
                                              gdr_stream_t stream) {
    // the same checks as gdr_chunk_fwd_ex (dense input, CUDA-core path)
    const gdr_status_t chk = validate_forward(q, k, v, a, beta, h0, out, hT, nullptr, B, T, H, dk,
                                              dv, chunk, b, dtype, gate, GDR_PATH_SIMT);
    if (chk != GDR_OK) return chk;
    const int64_t T_total = (int64_t)B * T;   // <= 2^40 after the checks

    // scratch layout: plan arrays, G [H, B*T], W [B*T, H, dk], U [B*T, H, dv].
    // The (token, head) rows are bounded first, by division, so that no byte
    // count below can wrap whatever H is.
    const int64_t row_bytes = 4 * (int64_t)(1 + dk + dv);
    const int64_t max_rows = (int64_t)kNoAllocScratchBytes / row_bytes;
    if (T_total > max_rows / H) return GDR_ERR_NO_WORKSPACE;
    if ((int64_t)B > (int64_t)kNoAllocScratchBytes / (3 * (int64_t)sizeof(int64_t)))
        return GDR_ERR_NO_WORKSPACE;
    const size_t plan_b = round256(3 * sizeof(int64_t) * (size_t)(B + 1));
    const size_t g_b = round256(sizeof(float) * (size_t)H * T_total);
    const size_t w_b = round256(sizeof(float) * (size_t)T_total * H * dk);
    const size_t u_b = round256(sizeof(float) * (size_t)T_total * H * dv);
    if (plan_b + g_b + w_b + u_b > kNoAllocScratchBytes) return GDR_ERR_NO_WORKSPACE;

    void *base = nullptr;
    if (noalloc_scratch(&base) != cudaSuccess) return GDR_ERR_CUDA;
    char *ws = (char *)base;
    int64_t *seq_start = (int64_t *)ws;
    int64_t *chunk_base = seq_start + (B + 1);
    int64_t *seg_base = chunk_base + (B + 1);
    float *G = (float *)(ws + plan_b);
    float *W = (float *)(ws + plan_b + g_b);
    float *U = (float *)(ws + plan_b + g_b + w_b);
    const int64_t max_chunks = (int64_t)B * ((T + chunk - 1) / chunk);
    Plan plan{B, chunk, 1 << 30, seq_start, chunk_base, seg_base};
    cudaStream_t st = (cudaStream_t)stream;
    // Every scratch element a kernel reads is written earlier in the same call,
    // so nothing left by a previous call needs clearing.
    if (launch_plan(nullptr, B, T, T_total, chunk, 1 << 30, seq_start, chunk_base, seg_base,
                    nullptr, st) != cudaSuccess)
        return GDR_ERR_CUDA;
    if (launch_gate_cumsum(a, nullptr, dtype, G, nullptr, plan, H, T_total, max_chunks, b, gate,
                           st) != cudaSuccess)
        return GDR_ERR_CUDA;
    if (launch_wy_simt(k, v, beta, G, W, U, dtype, plan, H, dk, dv, T_total, max_chunks, st) !=
        cudaSuccess)
        return GDR_ERR_CUDA;
    if (launch_state_out_simt(q, k, W, U, G, h0, out, hT, dtype, plan, H, dk, dv, T_total, st) !=
        cudaSuccess)
        return GDR_ERR_CUDA;
    return GDR_OK;
}
