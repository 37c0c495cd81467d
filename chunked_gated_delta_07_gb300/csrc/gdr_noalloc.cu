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
    if (dtype != GDR_BF16 && dtype != GDR_F32) return GDR_ERR_INVALID_ARG;
    if (gate != GDR_GATE_BOUNDED && gate != GDR_GATE_SOFTPLUS) return GDR_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || chunk < 1) return GDR_ERR_INVALID_ARG;
    if (gate == GDR_GATE_BOUNDED && !(b > 0.f && b < 3.4e38f)) return GDR_ERR_INVALID_ARG;
    if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return GDR_ERR_UNSUPPORTED;
    if (chunk != 16 && chunk != 32 && chunk != 64) return GDR_ERR_UNSUPPORTED;
    if (T > ((int64_t)1 << 40) || (int64_t)B * T > ((int64_t)1 << 40)) return GDR_ERR_NO_WORKSPACE;
    const int64_t T_total = (int64_t)B * T;
    if (T_total > 0 && (!q || !k || !v || !a || !beta || !out)) return GDR_ERR_INVALID_ARG;

    // scratch layout: plan arrays, G [H, B*T], W [B*T, H, dk], U [B*T, H, dv]
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
