// gdr_tc.cuh -- the tcgen05 (5th-generation tensor core) path: host-side entry points.
#pragma once

#include <cuda.h>

#include "gdr_internal.cuh"

namespace gdr {

// Tile length of the tensor-core path.  A call with chunk 32 or 64 runs it on 16-token
// tiles: the chunked form's result does not depend on the tile length (it is exact, and
// the pairwise in-tile decays need no bound at any length), so the chunk a caller names
// is a statement of blocking that this path is free to refine.
constexpr int kTcTile = 16;

// True when the tensor-core path implements this shape and dtype.
bool tc_supported(gdr_dtype_t dtype, int dk, int dv, int chunk);

// Tiles per segment for the segment-parallel state pass.
int tc_segment_chunks(int N, int H, int64_t T_total, int C, bool varlen);

// Scratch bytes of the tensor-core path beyond the plan and G.
size_t tc_workspace_bytes(int N, int H, int64_t T_total, int C, bool varlen);

// Stages 2-4 on the tensor cores (stage 1 and the plan already enqueued; beta is read
// as given, [rows][H] bf16).
cudaError_t launch_tc_forward(const void *q, const void *k, const void *v, const float *G,
                              const void *beta, const float *h0, void *out, float *hT, Plan plan,
                              int H, int64_t T_total, int64_t max_chunks, void *scratch,
                              int *status, cudaStream_t stream);

// Tensor map of a [rows][H][128] bf16 tensor for 64-column x C-row tile loads
// (128-byte swizzle); false when the driver entry point is missing or the base is
// not 16-byte aligned.
bool tc_make_map(CUtensorMap *map, const void *base, int H, int64_t rows);

// The per-channel decay forward on the tensor cores (gdr_tc_vec.cu): bf16, d = 128,
// tiles of 16, bounded gate.  `warm` holds the warm-up of every (segment, head),
// written by launch_vec_warm on the same plan.
cudaError_t launch_tc_vec(const void *q, const void *k, const void *v, const void *a,
                          const void *beta, const float *h0, void *out, float *hT, Plan plan,
                          int H, int64_t T_total, float b, int64_t max_segs, const int *warm,
                          int *status, cudaStream_t stream);

}  // namespace gdr
