// gdr_tc.cu -- the tcgen05 path (not yet enabled: every query reports unsupported).
#include "gdr_tc.cuh"

namespace gdr {

bool tc_supported(gdr_dtype_t, int, int, int) { return false; }
int tc_segment_chunks(int, int, int64_t, int) { return 1 << 30; }
size_t tc_workspace_bytes(int, int, int64_t, int) { return 0; }
cudaError_t launch_tc_forward(const void *, const void *, const void *, const float *,
                              const float *, const float *, void *, float *, Plan, int, int64_t,
                              int64_t, void *, int *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace gdr
