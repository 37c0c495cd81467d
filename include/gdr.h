/*
 * gdr.h -- C ABI of the chunked gated delta-rule forward pass on GB300 (sm_103a).
 *
 * The operation.  For every (sequence, head) unit, with per-token inputs
 * q_t, k_t in R^dk, v_t in R^dv, a gate logit a_t and a write strength
 * beta_t, the library computes
 *
 *     g_t   = -b * sigmoid(a_t)        (bounded gate, GDR_GATE_BOUNDED)
 *           = -softplus(a_t)           (unbounded gate, GDR_GATE_SOFTPLUS)
 *     H_t   = exp(g_t) H_{t-1} + beta_t k_t (v_t - exp(g_t) H_{t-1}^T k_t)^T
 *     o_t   = H_t^T q_t
 *
 * with H the dk x dv fp32 state (H = S^T for the dv x dk delta-rule state
 * S_t = alpha_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = S_t q_t,
 * alpha_t = exp(g_t)),
 * starting from h0 and ending in hT.  The bounded gate is the scaled-sigmoid
 * log-decay the pages introduce in place of the unbounded negative softplus
 * ("Deep Dive: The Next Generation of Ultra-Long Context Sparse MoE LLMs",
 * §3.3; "Core Technologies Behind Ultra-Long-Context Sparse MoE Large
 * Models", §2.2; "How Trillion-Scale Sparse MoE Models Achieve Million-Token
 * Long Context Capabilities", §3.2; "Evaluating Next-Gen Sparse MoE and
 * Long-Context LLMs", §2.3); the pages fix b = 5 there, b is a parameter
 * here.  The state update is the delta-rule write with data-dependent decay
 * of the incremental linear-attention layer ("Evaluating Next-Gen Sparse MoE
 * and Long-Context LLMs", §2.2).  It is computed chunk-parallel: the
 * sequence is cut into tiles of `chunk` tokens, each tile is a set of dense
 * products, and the state is passed from tile to tile ("Deep Dive ...",
 * §3.2; "Core Technologies ...", §2.1).  The result does not depend on
 * `chunk` beyond rounding.
 *
 * Layouts (row-major, contiguous, element type = dtype unless stated):
 *   dense  (cu_seqlens == NULL): q,k [B,T,H,dk]  v,out [B,T,H,dv]  a,beta [B,T,H]
 *   varlen (cu_seqlens != NULL): the same tensors with a leading 1 instead of B
 *          and T = total tokens; cu_seqlens holds N+1 int32 offsets (device
 *          memory), cu[0] = 0, non-decreasing, cu[N] = T; B is then N.
 *          Tiles restart at every sequence start; a partial last tile is masked.
 *   h0, hT : [N,H,dk,dv] fp32 (N = B for dense input).  h0 == NULL means zero.
 *          hT may be NULL (not written) and may alias h0 (in-place carry).
 *   beta is a probability (used as given, not passed through a sigmoid).
 *   q and k are used as given: no scaling, no normalisation.
 *
 * Segments of the tensor-core path.  A long sequence is cut into segments
 * whose state transitions are computed in parallel and chained.  A transition
 * skips what enters its segment so early that it reaches the segment's end
 * attenuated below 2^-64 of the state: the bound multiplies, per token, the
 * decay exp(g_t) by the erase factor's norm max(1, |1 - beta_t |k_t|^2|), so
 * it holds for any keys and write strengths (with unit keys and beta in
 * [0, 1] the erase factors are 1 and the decay alone sets it).  Where no such
 * point lies inside a segment the full transition is used.  The environment
 * variable GDR_TC_EXACT=1 turns the skipping off.
 *
 * Ownership and concurrency.  All tensor pointers of gdr_chunk_fwd* and of
 * the stage calls are DEVICE pointers owned by the caller; the library
 * retains none of them.  Calls are asynchronous on `stream` (NULL = the
 * legacy default stream).  Scratch memory comes from `workspace` if given,
 * else from a cache the library keeps per device (grown with cudaMalloc,
 * freed by gdr_release).  Calls that share the internal cache must not
 * overlap on the GPU: issue them on one stream, or pass each stream its own
 * workspace.
 *
 * Errors.  Arguments are checked before anything is launched: unsupported
 * sizes return GDR_ERR_UNSUPPORTED, malformed ones GDR_ERR_INVALID_ARG.  A
 * failed CUDA call returns GDR_ERR_CUDA.  Conditions only the device can see
 * (cu_seqlens that are not a valid offset list, a bounded wait that gave
 * up) set a per-device status word; gdr_get_status() reads and clears it.
 */
#ifndef GDR_H_
#define GDR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GDR_API __attribute__((visibility("default")))
#else
#define GDR_API
#endif

struct CUstream_st;
typedef struct CUstream_st *gdr_stream_t; /* the same type as cudaStream_t */

typedef enum {
    GDR_OK = 0,
    GDR_ERR_INVALID_ARG = 1,  /* null required pointer, negative size, ...     */
    GDR_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. dk = 96)       */
    GDR_ERR_CUDA = 3,         /* a CUDA runtime call failed                      */
    GDR_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out              */
    GDR_ERR_NO_WORKSPACE = 5, /* caller workspace smaller than required          */
    GDR_ERR_BAD_SEQLENS = 6,  /* cu_seqlens is not 0 = c0 <= c1 <= ... <= cN = T */
    GDR_ERR_BOUNDS = 7        /* checking build (GDR_DEBUG) only: a device-side index
                                 check failed and its access was skipped           */
} gdr_status_t;

typedef enum { GDR_BF16 = 0, GDR_F32 = 1 } gdr_dtype_t;

typedef enum {
    GDR_GATE_BOUNDED = 0, /* g = -b * sigmoid(a), g in [-b, 0]   */
    GDR_GATE_SOFTPLUS = 1 /* g = -softplus(a),    g in (-inf, 0) */
} gdr_gate_t;

typedef enum {
    GDR_PATH_AUTO = 0, /* tensor-core path where supported and q, k, v are 16-byte
                          aligned (TMA tiles), else SIMT                            */
    GDR_PATH_SIMT = 1, /* fp32 CUDA-core path (any supported shape and dtype)     */
    GDR_PATH_TC = 2    /* tcgen05 path; GDR_ERR_UNSUPPORTED where it does not apply
                          (shape, dtype, or q, k, v not 16-byte aligned)            */
} gdr_path_t;

/*
 * The forward pass with the defaults: dtype bf16, bounded gate with bound b,
 * automatic path, internal workspace.
 *   q,k,v,a,beta : inputs, layouts above (bf16)
 *   h0           : initial state or NULL (zero)
 *   out          : output, bf16, layout above; must not alias an input
 *   hT           : final state or NULL
 *   cu_seqlens   : NULL (dense) or N+1 int32 device offsets (varlen)
 *   B, T, H      : batch (or N), tokens per sequence (or total), heads
 *   dk, dv       : key / value width, each 64 or 128
 *   chunk        : tile length, 16, 32 or 64.  The CUDA-core path tiles by
 *                  chunk; the tensor-core path (bf16, dk = dv = 128) tiles by
 *                  16 tokens for every chunk, since the result does not depend
 *                  on the tile length beyond rounding (its in-tile decays are
 *                  pairwise, bounded for any tile length and gate)
 *   b            : gate bound, > 0 and finite
 * Supported sizes: B, H >= 1, T >= 0 (T = 0 copies h0 to hT, or zeroes hT).
 */
GDR_API gdr_status_t gdr_chunk_fwd(const void *q, const void *k, const void *v, const void *a,
                           const void *beta, const float *h0, void *out, float *hT,
                           const int32_t *cu_seqlens, int B, int64_t T, int H, int dk,
                           int dv, int chunk, float b, gdr_stream_t stream);

/*
 * The forward pass with every option.
 *   dtype       : element type of q, k, v, a, beta and out
 *   gate        : gate form; b is ignored for GDR_GATE_SOFTPLUS
 *   path        : kernel family (see gdr_path_t)
 *   workspace   : device scratch of workspace_bytes >= gdr_chunk_fwd_workspace_size(...),
 *                 or NULL for the internal per-device cache
 */
GDR_API gdr_status_t gdr_chunk_fwd_ex(const void *q, const void *k, const void *v, const void *a,
                              const void *beta, const float *h0, void *out, float *hT,
                              const int32_t *cu_seqlens, int B, int64_t T, int H, int dk,
                              int dv, int chunk, float b, gdr_dtype_t dtype, gdr_gate_t gate,
                              gdr_path_t path, void *workspace, size_t workspace_bytes,
                              gdr_stream_t stream);

/* Scratch bytes gdr_chunk_fwd_ex needs for these sizes (0 on invalid sizes).
 * B is N (the sequence count) for varlen input.  For GDR_PATH_AUTO it covers
 * both paths, since the pointers' alignment decides between them. */
GDR_API size_t gdr_chunk_fwd_workspace_size(int B, int64_t T, int H, int dk, int dv, int chunk,
                                    gdr_dtype_t dtype, gdr_path_t path);

/*
 * The forward pass on HOST buffers: inputs are copied to the device, the
 * pass runs, out (and hT) are copied back, and the call returns after the
 * copies have finished (it synchronises `stream`).  Same arguments and
 * layouts as gdr_chunk_fwd_ex except that every tensor pointer, including
 * cu_seqlens, is host memory (pinned memory gives full copy bandwidth).
 * Device buffers come from the internal per-device cache.
 * From 2^21 (token, head) units up, the call is pipelined: the tokens are cut
 * into up to 8 pieces (dense input: tile-aligned token ranges of every
 * sequence, the state carried from piece to piece; packed input: groups of
 * whole sequences, when cu_seqlens is well formed) and a piece's copies in
 * and out overlap the neighbouring pieces' passes, on two internal copy
 * streams.  The result then differs from gdr_chunk_fwd_ex's only by the
 * rounding of the different segment split.
 */
GDR_API gdr_status_t gdr_chunk_fwd_host(const void *q, const void *k, const void *v, const void *a,
                                const void *beta, const float *h0, void *out, float *hT,
                                const int32_t *cu_seqlens, int B, int64_t T, int H, int dk,
                                int dv, int chunk, float b, gdr_dtype_t dtype, gdr_gate_t gate,
                                gdr_path_t path, gdr_stream_t stream);

/*
 * The forward pass without any device allocation by the library.  The pages
 * have no counterpart to this call; it exists for callers that must not
 * allocate device memory when they run the pass (during CUDA graph capture,
 * inside engines that pre-reserve all device memory, in allocation-free
 * latency loops).  It runs the fp32 CUDA-core path on DENSE input only (no
 * cu_seqlens) and keeps its scratch in one statically allocated 32 MiB device
 * array that every GPU loading the library holds until exit.
 *   Arguments, layouts and ownership are those of gdr_chunk_fwd_ex.
 *   Limit: sizes whose scratch (4 * B*T*H * (1 + dk + dv) bytes plus
 *   24 * (B+1) bytes, each part rounded up to 256) exceeds 32 MiB return
 *   GDR_ERR_NO_WORKSPACE before anything is launched -- about 32K
 *   (token, head) pairs at dk = dv = 128.
 *   The first call on a device looks up the array's device address once
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   Every call reuses the same array, so calls that overlap on the GPU (on
 *   different streams, or from several threads) race and must be
 *   serialised by the caller.  Nothing in the array needs clearing between
 *   calls: each call writes every scratch element before reading it.
 */
GDR_API gdr_status_t gdr_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                           const void *a, const void *beta, const float *h0,
                                           void *out, float *hT, int B, int64_t T, int H, int dk,
                                           int dv, int chunk, float b, gdr_dtype_t dtype,
                                           gdr_gate_t gate, gdr_stream_t stream);

/*
 * Stage 1 alone: the gate and its in-tile cumulative sum.
 *   G[h, r] = sum over tokens r' of r's tile with r' <= r of g(a[r', h]),
 * written head-major as G [H, B*T] fp32 (token rows packed as in a).
 * Tiles restart at every sequence start ("Deep Dive ...", §3.2-3.3).
 */
GDR_API gdr_status_t gdr_gate_cumsum(const void *a, float *G, const int32_t *cu_seqlens, int B,
                             int64_t T, int H, int chunk, float b, gdr_dtype_t dtype,
                             gdr_gate_t gate, gdr_stream_t stream);

/*
 * Stage 2 alone: the per-tile WY / UT representation.  With G from
 * gdr_gate_cumsum (layout above), per tile of length C
 *   A_ij = beta_i exp(G_i - G_j) (k_i . k_j) for j < i,  T = (I + A)^{-1},
 *   W = T diag(beta exp(G)) K  [C x dk],  U = T diag(beta) V  [C x dv],
 * written fp32 in the layouts of k and v: W [B,T,H,dk], U [B,T,H,dv].
 */
GDR_API gdr_status_t gdr_wy_repr(const void *k, const void *v, const void *beta, const float *G,
                         float *W, float *U, const int32_t *cu_seqlens, int B, int64_t T,
                         int H, int dk, int dv, int chunk, gdr_dtype_t dtype,
                         gdr_stream_t stream);

/*
 * The recurrent (token-by-token) form, for decoding: advances each sequence's
 * state over T tokens and writes their outputs; T = 1 is one decode step of
 * an inference engine that keeps a constant-size state per sequence instead
 * of a cache that grows with the context ("Evaluating Next-Gen Sparse MoE and
 * Long-Context LLMs", §2.2: the state is updated token by token; §4, §5:
 * chunked prefill and constant-state layers on the inference side).  A prompt
 * is prefilled with gdr_chunk_fwd_ex (its hT is the state), then decoded here.
 *
 *   q, k   [N, T, H, dk]   v, out [N, T, H, dv]   a, beta [N, T, H]   (dtype)
 *   state  [N, H, dk, dv]  fp32, read as the entering state and overwritten
 *          with the state after the last token (same layout as h0 / hT)
 * Per token: alpha = exp(g(a)), H <- alpha H + beta k (v - alpha H^T k)^T,
 * o = H^T q (the same recurrence as gdr_chunk_fwd_ex, computed without tiles).
 * Device pointers owned by the caller; nothing is retained or allocated.
 * dk, dv in {64, 128}; N, H >= 1; T >= 0 (T = 0 leaves state untouched).
 * out must not alias any input or state; state must be 16-byte aligned (it
 * is read and written as float4).  Returns GDR_ERR_INVALID_ARG or
 * GDR_ERR_UNSUPPORTED before any launch, GDR_ERR_CUDA on a launch failure;
 * the call is asynchronous on `stream`.
 */
GDR_API gdr_status_t gdr_recurrent_fwd(const void *q, const void *k, const void *v, const void *a,
                               const void *beta, float *state, void *out, int N, int64_t T,
                               int H, int dk, int dv, float b, gdr_dtype_t dtype,
                               gdr_gate_t gate, gdr_stream_t stream);

/*
 * Per-channel (vector) decay: the forward pass of gdr_chunk_fwd_ex with one
 * gate input per key channel.  Token t decays row i of the dk x dv state by
 * exp(g(a[t, h, i])) before the delta-rule write:
 *     H_t = (I - beta k k^T) diag(exp(g(a_t))) H_{t-1} + beta k v^T,  o_t = H_t^T q_t,
 * g(a) = -b sigmoid(a) (the bounded gate).  Inside each 16-token tile the
 * pairwise decays exp(G_i - G_j) are split into the factors exp(G_i) and
 * exp(-G_j), which turns every in-tile product into a plain matrix product;
 * the bound keeps exp(-G) finite ("Deep Dive: The Next Generation of
 * Ultra-Long Context Sparse MoE LLMs", §2.1-2.2; "How Trillion-Scale Sparse
 * MoE Models Achieve Million-Token Long Context Capabilities", §3.2).
 *   a    [B, T, H, dk] in dtype (varlen: [1, T, H, dk]); every other argument as
 *        for gdr_chunk_fwd_ex.
 * chunk must be 16 and 0 < b <= 5 (exp(16 b) must stay below FLT_MAX):
 * GDR_ERR_UNSUPPORTED otherwise; b <= 0 is GDR_ERR_INVALID_ARG.  Only the
 * bounded gate is taken (an unbounded one can overflow exp(-G)).  bf16 with
 * dk = dv = 128 runs a fused tensor-core kernel when q, k, v, a and `out` are
 * 16-byte aligned; other shapes, fp32 and unaligned pointers run the CUDA-core
 * kernels (same results within the stated tolerances).  Scratch
 * comes from the internal per-device cache; asynchronous on `stream`.
 */
GDR_API gdr_status_t gdr_chunk_fwd_vec(const void *q, const void *k, const void *v, const void *a,
                               const void *beta, const float *h0, void *out, float *hT,
                               const int32_t *cu_seqlens, int B, int64_t T, int H, int dk, int dv,
                               int chunk, float b, gdr_dtype_t dtype, gdr_stream_t stream);

/*
 * Backward of the per-channel decay form (gdr_chunk_fwd_vec): gradients of
 * <dout, out> + <dhT, hT> with respect to q, k, v, a, beta and h0, as for
 * gdr_chunk_bwd, except that a and da are [tokens, H, dk] (one gate input and one
 * gradient per key channel).  It runs the chunked tensor-core form only: bf16,
 * dk = dv = 128, chunk 16, 0 < b <= 5 (GDR_ERR_UNSUPPORTED otherwise); the
 * bounded gate is implied.  Errors, ownership and streams as for gdr_chunk_bwd.
 */
GDR_API gdr_status_t gdr_chunk_bwd_vec(const void *q, const void *k, const void *v, const void *a,
                               const void *beta, const float *h0, const void *dout,
                               const float *dhT, void *dq, void *dk_out, void *dv_out, void *da,
                               void *dbeta, float *dh0, const int32_t *cu_seqlens, int B,
                               int64_t T, int H, int dk, int dv, int chunk, float b,
                               gdr_dtype_t dtype, gdr_stream_t stream);

/* Bias-update rule of the quantile-balancing router (see gdr_router_bias_update). */
typedef enum { GDR_QB_SIGN = 0, GDR_QB_PROPORTIONAL = 1 } gdr_qb_mode_t;

/*
 * Routing step of aux-loss-free quantile balancing ("Deep Dive: The Next
 * Generation of Ultra-Long Context Sparse MoE LLMs", §4.2; "Core Technologies
 * Behind Ultra-Long-Context Sparse MoE Large Models", §3.2): every token t
 * picks the k experts of largest score logits[t, e] + bias[e], the sum taken
 * in binary32; equal scores go to the lower expert index.  The bias only
 * steers the selection: topk_logit returns the unbiased logits.
 *   logits     [T, E] in dtype (bf16 or fp32), 16-byte aligned (device)
 *   bias       [E] fp32 (device)
 *   topk_idx   [T, k] int32, experts in descending score order (device, written)
 *   topk_logit [T, k] fp32 logits of the picked experts, or NULL
 *   load       [E] int64: this call's per-expert counts are ADDED (a window may
 *              span several calls; zero it at the window start), or NULL
 * 1 <= E <= 2048 with E % 4 == 0 and 1 <= k <= min(E, 32): GDR_ERR_UNSUPPORTED
 * otherwise.  NaN logits or biases give an unspecified (but in-bounds)
 * selection.  Outputs must not overlap inputs: GDR_ERR_INVALID_ARG.
 * Asynchronous on `stream`; the counts are exact (integer atomics).
 */
GDR_API gdr_status_t gdr_router_topk(const void *logits, const float *bias, int32_t *topk_idx,
                             float *topk_logit, int64_t *load, int64_t T, int E, int k,
                             gdr_dtype_t dtype, gdr_stream_t stream);

/*
 * Bias step of quantile balancing (the four pages print it in two forms;
 * "Core Technologies ...", §3.2, "How Trillion-Scale Sparse MoE Models Achieve
 * Million-Token Long Context Capabilities", §4.3, "Evaluating Next-Gen Sparse
 * MoE and Long-Context LLMs", §3.2).  Q(q) is the q-quantile of the E loads by
 * linear interpolation between order statistics (sorted x, p = q (E - 1),
 * i = floor p: Q = x_i + (p - i)(x_{i+1} - x_i)), in binary64.
 *   GDR_QB_SIGN:         bias[e] -= eta if load[e] > Q(q_hi), else
 *                        bias[e] += eta if load[e] < Q(q_lo)   (binary32 steps;
 *                        q_lo = q_hi is the single-threshold form)
 *   GDR_QB_PROPORTIONAL: bias[e] += eta (Q(q_hi) - load[e]) / Q(q_hi) in
 *                        binary64, rounded to binary32; no change if Q(q_hi) = 0
 *   load [E] int64 (device), bias [E] fp32 (device, updated in place),
 *   thresholds [2] fp64 = {Q(q_lo), Q(q_hi)} (device, written) or NULL.
 * 1 <= E <= 2048 (GDR_ERR_UNSUPPORTED otherwise); q_lo, q_hi in [0, 1] and eta
 * finite (GDR_ERR_INVALID_ARG otherwise).  Asynchronous on `stream`.
 */
GDR_API gdr_status_t gdr_router_bias_update(const int64_t *load, float *bias, double *thresholds,
                                    int E, gdr_qb_mode_t mode, double q_lo, double q_hi,
                                    float eta, gdr_stream_t stream);

/*
 * The backward pass: gradients of  L = <dout, out> + <dhT, hT>  with respect to
 * q, k, v, a, beta and h0, for the forward of gdr_chunk_fwd_ex on the same
 * inputs (same layouts, dtype, gate, b and cu_seqlens; B is N for varlen).
 * The pages train the layer in bf16 mixed precision ("Core Technologies ...",
 * §2.3; "Deep Dive ...", §3.3) but print no backward; the adjoints here are
 * those of the recurrence H_t = alpha H_{t-1} + beta k (v - alpha H^T k)^T,
 * o = H_t^T q, written out per token:
 *   dout [tokens, H, dv] (dtype) or NULL (zero);  dhT [N, H, dk, dv] fp32 or NULL
 *   dq, dk [tokens, H, dk], dv [tokens, H, dv], da, dbeta [tokens, H]  (dtype, all
 *   written);  dh0 [N, H, dk, dv] fp32 (written when not NULL)
 * `chunk` is validated like the forward's; the pass works on 16-token tiles
 * either way.  bf16 with dk = dv = 128 and the bounded gate with b <= 5 runs
 * the chunked tensor-core form: the states at tile boundaries are stored in
 * bf16, and each tile's gradients come from dense products.  Every other case
 * runs token by token, from fp32 checkpoints every 16 tokens with the tokens
 * between them recomputed.  Device pointers owned
 * by the caller; scratch comes from the internal per-device cache.  Outputs
 * must not alias inputs; dhT and dh0 must be 16-byte aligned (copied as
 * float4), GDR_ERR_INVALID_ARG otherwise.  The result is deterministic (no
 * atomics).  Errors as for gdr_chunk_fwd_ex; asynchronous on `stream`.  The
 * chunked form runs its two state chains (forward and adjoint, independent of
 * each other) concurrently: the adjoint chain on a second stream the library
 * keeps per device (freed by gdr_release), forked from and joined back to
 * `stream` with events, so the call is ordered on `stream` as a whole.  Both
 * chains run on the tcgen05 tensor cores with the state in tensor memory when
 * q, k, v, dout (and a per-channel a) are 16-byte aligned, and on warp-level
 * tensor-core kernels otherwise; their waits are bounded like the forward's
 * (GDR_ERR_TIMEOUT in the status word).
 */
GDR_API gdr_status_t gdr_chunk_bwd(const void *q, const void *k, const void *v, const void *a,
                           const void *beta, const float *h0, const void *dout,
                           const float *dhT, void *dq, void *dk_out, void *dv_out, void *da,
                           void *dbeta, float *dh0, const int32_t *cu_seqlens, int B,
                           int64_t T, int H, int dk, int dv, int chunk, float b,
                           gdr_dtype_t dtype, gdr_gate_t gate, gdr_stream_t stream);

/* Synchronise `stream`, then read and clear the current device's status word.
 * Returns GDR_OK, GDR_ERR_BAD_SEQLENS, GDR_ERR_TIMEOUT or GDR_ERR_CUDA. */
GDR_API gdr_status_t gdr_get_status(gdr_stream_t stream);

/* Static description of a status code (never NULL). */
GDR_API const char *gdr_status_string(gdr_status_t status);

/* Free the internal per-device caches of every device (synchronises them). */
GDR_API void gdr_release(void);

/* Number of kernels this library has launched so far in this process. */
GDR_API uint64_t gdr_launch_count(void);

/*
 * Per-kernel timing.  While enabled, every kernel the library launches is
 * bracketed by a pair of CUDA events recorded on its launch stream.
 * gdr_profile_read synchronises those events, writes for up to `max`
 * distinct kernels its name (a static string), the summed device time in
 * milliseconds and the launch count, returns the number of distinct kernels
 * seen (which may exceed `max`), and clears the record.  Enabling adds two
 * event records per launch and nothing else.
 */
GDR_API void gdr_profile_enable(int on);
GDR_API int gdr_profile_read(const char **names, double *total_ms, int *launches, int max);
/* Restrict the timing to the launches of one kernel, named as gdr_profile_read
 * reports it (NULL or "": every kernel, the default), so that a measurement of
 * that kernel puts no events between the other launches.  The name is copied. */
GDR_API void gdr_profile_select(const char *name);

#ifdef __cplusplus
}
#endif
#endif /* GDR_H_ */
