// gdr_api.cu -- the C ABI: argument checks, per-device state, workspace
// layout and dispatch to the kernel families.  No arithmetic of the method
// lives here; every step of the pass runs in the kernels.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <mutex>
#include <string>
#include <vector>

#include "gdr_internal.cuh"
#include "gdr_tc.cuh"

namespace gdr {

static std::atomic<uint64_t> g_launches{0};
void count_launch(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

#ifdef GDR_DEBUG
namespace {
std::vector<DebugFlagReader> &debug_readers() {
    static std::vector<DebugFlagReader> v;
    return v;
}
std::mutex &debug_mu() {
    static std::mutex m;
    return m;
}
}  // namespace
bool register_debug_flag(DebugFlagReader fn) {
    std::lock_guard<std::mutex> lk(debug_mu());
    debug_readers().push_back(fn);
    return true;
}
#endif

// ---- per-kernel event timing ------------------------------------------------
namespace {
struct ProfRec {
    const char *name;
    cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
std::atomic<bool> g_prof_on{false};
std::string g_prof_only;   // record only launches of this kernel ("" = all); guarded by g_prof_mu
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t prof_event() {
    if (!g_prof_pool.empty()) {
        cudaEvent_t e = g_prof_pool.back();
        g_prof_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}
}  // namespace

ProfScope::ProfScope(cudaStream_t stream, const char *name) : stream_(stream), slot_(-1) {
    if (!g_prof_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_only.empty() && g_prof_only != name) return;
    ProfRec r{name, prof_event(), prof_event()};
    if (!r.start || !r.stop) return;
    cudaEventRecord(r.start, stream_);
    slot_ = (long)g_prof.size();
    g_prof.push_back(r);
}

ProfScope::~ProfScope() {
    if (slot_ < 0) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (slot_ < (long)g_prof.size()) cudaEventRecord(g_prof[slot_].stop, stream_);
}

namespace {

constexpr int kMaxPieces = 8;   // pieces of a pipelined host-buffer call

std::mutex &g_mu_aux() {
    static std::mutex m;
    return m;
}

struct DeviceCtx {
    int *d_status = nullptr;
    int sms = 0;         // streaming multiprocessors of the device
    void *ws = nullptr;  // internal workspace cache
    size_t ws_bytes = 0;
    void *io = nullptr;  // device copies for the host-buffer entry point
    size_t io_bytes = 0;
    // copy streams and per-piece events of the pipelined host-buffer entry point
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_in[kMaxPieces] = {}, ev_comp[kMaxPieces] = {}, ev_out[kMaxPieces] = {};
    // the backward's second stream (its two state chains run concurrently)
    AuxStream aux;
};

// The device's auxiliary stream and fork/join events, created on first use (an
// empty AuxStream, i.e. one stream for everything, if that fails).
AuxStream aux_stream(DeviceCtx *c) {
    std::lock_guard<std::mutex> lk(g_mu_aux());
    if (!c->aux.stream) {
        AuxStream a;
        if (cudaStreamCreateWithFlags(&a.stream, cudaStreamNonBlocking) != cudaSuccess) return AuxStream{};
        if (cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming) != cudaSuccess) {
            if (a.fork) cudaEventDestroy(a.fork);
            cudaStreamDestroy(a.stream);
            return AuxStream{};
        }
        c->aux = a;
    }
    return c->aux;
}

std::mutex g_mu;
// a deque: growing it for a new device keeps every handed-out context in place
std::deque<DeviceCtx> g_ctx;

// The calling thread's current device context, with its status word
// allocated.  Returns nullptr on a CUDA failure.
DeviceCtx *device_ctx() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if ((int)g_ctx.size() <= dev) g_ctx.resize(dev + 1);
    DeviceCtx &c = g_ctx[dev];
    if (!c.d_status) {
        if (cudaMalloc(&c.d_status, sizeof(int)) != cudaSuccess) return nullptr;
        if (cudaMemset(c.d_status, 0, sizeof(int)) != cudaSuccess) return nullptr;
        if (cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
    }
    return &c;
}

// Grow a cached device buffer to at least `bytes` (contents not preserved).
bool grow(void **buf, size_t *have, size_t bytes) {
    if (*have >= bytes) return true;
    if (*buf) {
        cudaDeviceSynchronize();  // the old buffer may still be in use
        cudaFree(*buf);
        *buf = nullptr;
        *have = 0;
    }
    if (bytes == 0) return true;
    if (cudaMalloc(buf, bytes) != cudaSuccess) {
        *buf = nullptr;
        return false;
    }
    *have = bytes;
    return true;
}

// Upper bound on the tiles of all sequences: every dense sequence ends in its
// own partial tile; packed sequences can each add one partial tile.
inline int64_t tile_bound(bool varlen, int B, int64_t T, int chunk) {
    return varlen ? (T + chunk - 1) / chunk + B : (int64_t)B * ((T + chunk - 1) / chunk);
}

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Shape {
    int N, H, dk, dv, C;
    int64_t T_per, T_total;   // tokens per dense sequence / packed total
    bool varlen;
    int64_t max_chunks;       // upper bound on tiles over all sequences
};

// Scratch layout of one call.  Every region is 256-byte aligned.
struct Layout {
    size_t plan = 0, G = 0, W = 0, U = 0, tc = 0, total = 0;
};

// The shape a path runs: the tensor-core path tiles by kTcTile whatever chunk the
// caller named (16, 32 or 64).
Shape run_shape(Shape s, gdr_path_t path) {
    if (path == GDR_PATH_TC && s.C != kTcTile) {
        s.C = kTcTile;
        s.max_chunks = tile_bound(s.varlen, s.N, s.varlen ? s.T_total : s.T_per, kTcTile);
    }
    return s;
}

Layout layout_for(const Shape &s_in, gdr_path_t path) {
    const Shape s = run_shape(s_in, path);
    Layout L;
    size_t off = 0;
    L.plan = off;
    off += align_up(3 * sizeof(int64_t) * (size_t)(s.N + 1));
    L.G = off;
    off += align_up(sizeof(float) * (size_t)s.H * s.T_total);
    if (path == GDR_PATH_TC) {
        L.tc = off;
        off += align_up(tc_workspace_bytes(s.N, s.H, s.T_total, s.C, s.varlen));
    } else {
        L.W = off;
        off += align_up(sizeof(float) * (size_t)s.T_total * s.H * s.dk);
        L.U = off;
        off += align_up(sizeof(float) * (size_t)s.T_total * s.H * s.dv);
    }
    L.total = off;
    return L;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const char *pa = (const char *)a, *pb = (const char *)b;
    return pa < pb + nb && pb < pa + na;
}

// 16-byte alignment (a null pointer counts as aligned): TMA tiles, cp.async and
// the float4 state copies need it.
inline bool al16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Checks shared by every forward entry point.  Fills `s` on success.
gdr_status_t check_args(const void *q, const void *k, const void *v, const void *a,
                        const void *beta, const float *h0, const void *out, const float *hT,
                        const int32_t *cu, int B, int64_t T, int H, int dk, int dv, int chunk,
                        float b, gdr_dtype_t dtype, gdr_gate_t gate, gdr_path_t path,
                        Shape *s) {
    if (dtype != GDR_BF16 && dtype != GDR_F32) return GDR_ERR_INVALID_ARG;
    if (gate != GDR_GATE_BOUNDED && gate != GDR_GATE_SOFTPLUS) return GDR_ERR_INVALID_ARG;
    if (path != GDR_PATH_AUTO && path != GDR_PATH_SIMT && path != GDR_PATH_TC)
        return GDR_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || chunk < 1) return GDR_ERR_INVALID_ARG;
    if (gate == GDR_GATE_BOUNDED && !(b > 0.f && std::isfinite(b))) return GDR_ERR_INVALID_ARG;
    if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return GDR_ERR_UNSUPPORTED;
    if (chunk != 16 && chunk != 32 && chunk != 64) return GDR_ERR_UNSUPPORTED;
    if (T > ((int64_t)1 << 40) || (int64_t)B * T > ((int64_t)1 << 40)) return GDR_ERR_UNSUPPORTED;
    const bool varlen = cu != nullptr;
    const int64_t T_total = varlen ? T : (int64_t)B * T;
    // at most 2^40 (token, head) rows, so that no byte count below wraps
    if (T_total > 0 && (int64_t)H > ((int64_t)1 << 40) / T_total) return GDR_ERR_UNSUPPORTED;
    if (T_total > 0 && (!q || !k || !v || !a || !beta || !out)) return GDR_ERR_INVALID_ARG;
    const size_t es = dtype == GDR_BF16 ? 2 : 4;
    const size_t rows = (size_t)T_total * H;
    const size_t n_state = (size_t)B * H * dk * dv * sizeof(float);
    const void *ins[5] = {q, k, v, a, beta};
    const size_t in_bytes[5] = {rows * dk * es, rows * dk * es, rows * dv * es, rows * es, rows * es};
    const size_t out_bytes = rows * dv * es;
    for (int i = 0; i < 5; ++i) {
        if (overlaps(out, out_bytes, ins[i], in_bytes[i])) return GDR_ERR_INVALID_ARG;
        if (overlaps(hT, n_state, ins[i], in_bytes[i])) return GDR_ERR_INVALID_ARG;
    }
    if (overlaps(out, out_bytes, h0, n_state) || overlaps(out, out_bytes, hT, n_state))
        return GDR_ERR_INVALID_ARG;
    if (hT && h0 && (const void *)hT != (const void *)h0 && overlaps(hT, n_state, h0, n_state))
        return GDR_ERR_INVALID_ARG;
    if (path == GDR_PATH_TC && !tc_supported(dtype, dk, dv, chunk)) return GDR_ERR_UNSUPPORTED;
    s->N = B;
    s->H = H;
    s->dk = dk;
    s->dv = dv;
    s->C = chunk;
    s->T_per = varlen ? 0 : T;
    s->T_total = T_total;
    s->varlen = varlen;
    s->max_chunks = tile_bound(varlen, B, T, chunk);
    return GDR_OK;
}

gdr_path_t resolve_path(gdr_path_t path, gdr_dtype_t dtype, int dk, int dv, int chunk) {
    if (path != GDR_PATH_AUTO) return path;
    return tc_supported(dtype, dk, dv, chunk) ? GDR_PATH_TC : GDR_PATH_SIMT;
}

gdr_status_t run_forward(const void *q, const void *k, const void *v, const void *a,
                         const void *beta, const float *h0, void *out, float *hT,
                         const int32_t *cu, const Shape &s_in, float b, gdr_dtype_t dtype,
                         gdr_gate_t gate, gdr_path_t path, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
    const Shape s = run_shape(s_in, path);
    DeviceCtx *ctx = device_ctx();
    if (!ctx) return GDR_ERR_CUDA;
    const Layout L = layout_for(s, path);
    char *ws = (char *)workspace;
    if (ws) {
        if (workspace_bytes < L.total) return GDR_ERR_NO_WORKSPACE;
    } else {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!grow(&ctx->ws, &ctx->ws_bytes, L.total)) return GDR_ERR_CUDA;
        ws = (char *)ctx->ws;
    }
    int64_t *seq_start = (int64_t *)(ws + L.plan);
    int64_t *chunk_base = seq_start + (s.N + 1);
    int64_t *seg_base = chunk_base + (s.N + 1);
    float *G = (float *)(ws + L.G);
    const int seg_chunks = path == GDR_PATH_TC ? tc_segment_chunks(s.N, s.H, s.T_total, s.C, s.varlen) : (1 << 30);
    Plan plan{s.N, s.C, seg_chunks, seq_start, chunk_base, seg_base};

    cudaError_t err = launch_plan(cu, s.N, s.T_per, s.T_total, s.C, seg_chunks, seq_start,
                                  chunk_base, seg_base, ctx->d_status, stream);
    if (err != cudaSuccess) return GDR_ERR_CUDA;
    err = launch_gate_cumsum(a, beta, dtype, G, nullptr, plan, s.H, s.T_total, s.max_chunks, b, gate,
                             stream);
    if (err != cudaSuccess) return GDR_ERR_CUDA;
    if (path == GDR_PATH_TC) {
        err = launch_tc_forward(q, k, v, G, beta, h0, out, hT, plan, s.H, s.T_total, s.max_chunks,
                                ws + L.tc, ctx->d_status, stream);
    } else {
        float *W = (float *)(ws + L.W);
        float *U = (float *)(ws + L.U);
        err = launch_wy_simt(k, v, beta, G, W, U, dtype, plan, s.H, s.dk, s.dv, s.T_total,
                             s.max_chunks, stream);
        if (err != cudaSuccess) return GDR_ERR_CUDA;
        err = launch_state_out_simt(q, k, W, U, G, h0, out, hT, dtype, plan, s.H, s.dk, s.dv,
                                    s.T_total, stream);
    }
    return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// host-buffer forward, pipelined: the tokens are cut into pieces (dense input:
// tile-aligned ranges of every sequence, the state carried from piece to
// piece; packed input: groups of whole sequences), and piece p runs while
// piece p + 1 is copied in and piece p - 1 is copied out, on two copy streams.
// Device buffers of the pieces are double buffered.
// ---------------------------------------------------------------------------
struct Piece {
    int64_t t0, t1;   // dense: token range of every sequence; packed: token range
    int g0, g1;       // packed: sequence range
};

bool pipe_ready(DeviceCtx *c) {
    if (c->s_in) return true;
    if (cudaStreamCreateWithFlags(&c->s_in, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&c->s_out, cudaStreamNonBlocking) != cudaSuccess) return false;
    for (int i = 0; i < kMaxPieces; ++i)
        if (cudaEventCreateWithFlags(&c->ev_in[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&c->ev_comp[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&c->ev_out[i], cudaEventDisableTiming) != cudaSuccess)
            return false;
    return true;
}

// The pieces of a call, or none (fewer than two) when it is better run whole.
std::vector<Piece> host_pieces(const Shape &s, const int32_t *cu) {
    std::vector<Piece> pcs;
    const int64_t units = s.T_total * s.H;
    if (units < ((int64_t)1 << 21)) return pcs;            // small: one piece
    const int want = (int)std::min<int64_t>(kMaxPieces, std::max<int64_t>(2, units >> 21));
    if (!s.varlen) {
        int64_t step = (s.T_per + want - 1) / want;
        step = (step + s.C - 1) / s.C * s.C;                // tile aligned
        for (int64_t t0 = 0; t0 < s.T_per; t0 += step)
            pcs.push_back({t0, std::min(s.T_per, t0 + step), 0, s.N});
    } else {
        // only well-formed offsets are cut here; anything else runs whole, where
        // the device-side plan reports it
        if (cu[0] != 0 || cu[s.N] != s.T_total) return pcs;
        for (int g = 0; g < s.N; ++g)
            if (cu[g + 1] < cu[g]) return pcs;
        const int64_t target = (s.T_total + want - 1) / want;
        int g0 = 0;
        for (int g = 0; g < s.N; ++g) {
            if (cu[g + 1] - cu[g0] >= target || g == s.N - 1) {
                pcs.push_back({cu[g0], cu[g + 1], g0, g + 1});
                g0 = g + 1;
            }
        }
        if (pcs.size() > (size_t)kMaxPieces) pcs.clear();   // cannot happen; be safe
    }
    if (pcs.size() < 2) pcs.clear();
    return pcs;
}

gdr_status_t fwd_host_pipelined(const void *q, const void *k, const void *v, const void *a,
                                const void *beta, const float *h0, void *out, float *hT,
                                const int32_t *cu, const Shape &s, const std::vector<Piece> &pcs,
                                float b, gdr_dtype_t dtype, gdr_gate_t gate, gdr_path_t path,
                                cudaStream_t stream) {
    DeviceCtx *ctx = device_ctx();
    if (!ctx) return GDR_ERR_CUDA;
    const size_t es = dtype == GDR_BF16 ? 2 : 4;
    const int H = s.H;
    const size_t rk = (size_t)H * s.dk * es, rv = (size_t)H * s.dv * es, r1 = (size_t)H * es;
    const size_t nst1 = (size_t)H * s.dk * s.dv * sizeof(float);   // one sequence's state
    const int np = (int)pcs.size();
    // the largest piece, in token rows and sequences
    int64_t max_rows = 0;
    int max_seq = 0;
    for (const Piece &pc : pcs) {
        const int64_t rows = s.varlen ? pc.t1 - pc.t0 : (int64_t)s.N * (pc.t1 - pc.t0);
        max_rows = std::max(max_rows, rows);
        max_seq = std::max(max_seq, pc.g1 - pc.g0);
    }
    // device layout: 2 x [q k v a beta cu] in, 2 x out, states
    const size_t in_sz[6] = {max_rows * rk, max_rows * rk, max_rows * rv, max_rows * r1,
                             max_rows * r1, sizeof(int32_t) * (size_t)(max_seq + 1)};
    size_t in_off[6], in_tot = 0;
    for (int i = 0; i < 6; ++i) {
        in_off[i] = in_tot;
        in_tot += align_up(in_sz[i]);
    }
    const size_t out_tot = align_up(max_rows * rv);
    const size_t st_tot = align_up((size_t)s.N * nst1);
    // dense: 2 carried states (+ h0); packed: all entering states and all final states
    const size_t tot = 2 * in_tot + 2 * out_tot + 3 * st_tot;
    char *io;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!pipe_ready(ctx)) return GDR_ERR_CUDA;
        if (!grow(&ctx->io, &ctx->io_bytes, tot)) return GDR_ERR_CUDA;
        io = (char *)ctx->io;
    }
    char *IN[2] = {io, io + in_tot};
    char *OUT[2] = {io + 2 * in_tot, io + 2 * in_tot + out_tot};
    float *ST0 = (float *)(io + 2 * in_tot + 2 * out_tot);        // dense: carried state A / packed: h0
    float *ST1 = (float *)((char *)ST0 + st_tot);                 // dense: carried state B / packed: hT
    float *dH0 = (float *)((char *)ST1 + st_tot);                 // dense: h0
    // the workspace of the largest piece, grown once before anything is queued
    {
        Shape ps = s;
        ps.N = s.varlen ? max_seq : s.N;
        ps.T_total = max_rows;
        ps.T_per = s.varlen ? 0 : max_rows / s.N;
        ps.max_chunks = tile_bound(s.varlen, ps.N, s.varlen ? max_rows : ps.T_per, s.C);
        std::lock_guard<std::mutex> lk(g_mu);
        if (!grow(&ctx->ws, &ctx->ws_bytes, layout_for(ps, path).total)) return GDR_ERR_CUDA;
    }
    auto ck = [](cudaError_t e) { return e == cudaSuccess; };
    cudaStream_t si = ctx->s_in, so = ctx->s_out;
    // everything queued before this call on `stream` precedes the copies
    if (!ck(cudaEventRecord(ctx->ev_out[0], stream)) || !ck(cudaStreamWaitEvent(si, ctx->ev_out[0], 0)) ||
        !ck(cudaStreamWaitEvent(so, ctx->ev_out[0], 0)))
        return GDR_ERR_CUDA;
    if (h0 && !ck(cudaMemcpyAsync(s.varlen ? ST0 : dH0, h0, (size_t)s.N * nst1, cudaMemcpyHostToDevice, si)))
        return GDR_ERR_CUDA;
    std::vector<std::vector<int32_t>> cus(np);
    for (int p = 0; p < np; ++p) {
        const Piece &pc = pcs[p];
        char *in = IN[p & 1];
        // ---- copy in (after the compute of piece p - 2 released the buffer)
        if (p >= 2 && !ck(cudaStreamWaitEvent(si, ctx->ev_comp[p - 2], 0))) return GDR_ERR_CUDA;
        const void *src[5] = {q, k, v, a, beta};
        const size_t rb[5] = {rk, rk, rv, r1, r1};
        for (int i = 0; i < 5; ++i) {
            if (s.varlen) {
                if (!ck(cudaMemcpyAsync(in + in_off[i], (const char *)src[i] + pc.t0 * rb[i],
                                        (pc.t1 - pc.t0) * rb[i], cudaMemcpyHostToDevice, si)))
                    return GDR_ERR_CUDA;
            } else {
                const size_t w = (size_t)(pc.t1 - pc.t0) * rb[i];
                if (!ck(cudaMemcpy2DAsync(in + in_off[i], w, (const char *)src[i] + pc.t0 * rb[i],
                                          (size_t)s.T_per * rb[i], w, s.N, cudaMemcpyHostToDevice, si)))
                    return GDR_ERR_CUDA;
            }
        }
        if (s.varlen) {
            cus[p].resize(pc.g1 - pc.g0 + 1);
            for (int g = pc.g0; g <= pc.g1; ++g) cus[p][g - pc.g0] = (int32_t)(cu[g] - cu[pc.g0]);
            if (!ck(cudaMemcpyAsync(in + in_off[5], cus[p].data(), sizeof(int32_t) * cus[p].size(),
                                    cudaMemcpyHostToDevice, si)))
                return GDR_ERR_CUDA;
        }
        if (!ck(cudaEventRecord(ctx->ev_in[p], si))) return GDR_ERR_CUDA;
        // ---- compute (after its copy-in, and after the copy-out of piece p - 2)
        if (!ck(cudaStreamWaitEvent(stream, ctx->ev_in[p], 0))) return GDR_ERR_CUDA;
        if (p >= 2 && !ck(cudaStreamWaitEvent(stream, ctx->ev_out[p - 2], 0))) return GDR_ERR_CUDA;
        Shape ps = s;
        const float *hin;
        float *hout;
        if (s.varlen) {
            ps.N = pc.g1 - pc.g0;
            ps.T_total = pc.t1 - pc.t0;
            ps.T_per = 0;
            ps.max_chunks = tile_bound(true, ps.N, ps.T_total, s.C);
            hin = h0 ? ST0 + (size_t)pc.g0 * (nst1 / sizeof(float)) : nullptr;
            hout = ST1 + (size_t)pc.g0 * (nst1 / sizeof(float));
        } else {
            ps.T_per = pc.t1 - pc.t0;
            ps.T_total = (int64_t)s.N * ps.T_per;
            ps.max_chunks = tile_bound(false, s.N, ps.T_per, s.C);
            hin = p == 0 ? (h0 ? dH0 : nullptr) : ((p - 1) & 1 ? ST1 : ST0);
            hout = (p & 1) ? ST1 : ST0;
        }
        const gdr_status_t st =
            run_forward(in + in_off[0], in + in_off[1], in + in_off[2], in + in_off[3], in + in_off[4],
                        hin, OUT[p & 1], hout, s.varlen ? (const int32_t *)(in + in_off[5]) : nullptr, ps, b,
                        dtype, gate, path, nullptr, 0, stream);
        if (st != GDR_OK) return st;
        if (!ck(cudaEventRecord(ctx->ev_comp[p], stream))) return GDR_ERR_CUDA;
        // ---- copy out
        if (!ck(cudaStreamWaitEvent(so, ctx->ev_comp[p], 0))) return GDR_ERR_CUDA;
        if (s.varlen) {
            if (!ck(cudaMemcpyAsync((char *)out + pc.t0 * rv, OUT[p & 1], (pc.t1 - pc.t0) * rv,
                                    cudaMemcpyDeviceToHost, so)))
                return GDR_ERR_CUDA;
            if (hT && !ck(cudaMemcpyAsync((char *)hT + (size_t)pc.g0 * nst1, hout,
                                          (size_t)(pc.g1 - pc.g0) * nst1, cudaMemcpyDeviceToHost, so)))
                return GDR_ERR_CUDA;
        } else {
            const size_t w = (size_t)(pc.t1 - pc.t0) * rv;
            if (!ck(cudaMemcpy2DAsync((char *)out + pc.t0 * rv, (size_t)s.T_per * rv, OUT[p & 1], w, w,
                                      s.N, cudaMemcpyDeviceToHost, so)))
                return GDR_ERR_CUDA;
            if (p == np - 1 && hT &&
                !ck(cudaMemcpyAsync(hT, hout, (size_t)s.N * nst1, cudaMemcpyDeviceToHost, so)))
                return GDR_ERR_CUDA;
        }
        if (!ck(cudaEventRecord(ctx->ev_out[p], so))) return GDR_ERR_CUDA;
    }
    const bool ok = ck(cudaStreamSynchronize(so)) && ck(cudaStreamSynchronize(stream)) &&
                    ck(cudaStreamSynchronize(si));
    return ok ? GDR_OK : GDR_ERR_CUDA;
}

}  // namespace

gdr_status_t validate_forward(const void *q, const void *k, const void *v, const void *a,
                              const void *beta, const float *h0, const void *out, const float *hT,
                              const int32_t *cu, int B, int64_t T, int H, int dk, int dv,
                              int chunk, float b, gdr_dtype_t dtype, gdr_gate_t gate,
                              gdr_path_t path) {
    Shape s;
    return check_args(q, k, v, a, beta, h0, out, hT, cu, B, T, H, dk, dv, chunk, b, dtype, gate,
                      path, &s);
}

}  // namespace gdr

using namespace gdr;

extern "C" {

gdr_status_t gdr_chunk_fwd_ex(const void *q, const void *k, const void *v, const void *a,
                              const void *beta, const float *h0, void *out, float *hT,
                              const int32_t *cu_seqlens, int B, int64_t T, int H, int dk,
                              int dv, int chunk, float b, gdr_dtype_t dtype, gdr_gate_t gate,
                              gdr_path_t path, void *workspace, size_t workspace_bytes,
                              gdr_stream_t stream) {
    Shape s;
    gdr_status_t st = check_args(q, k, v, a, beta, h0, out, hT, cu_seqlens, B, T, H, dk, dv,
                                 chunk, b, dtype, gate, path, &s);
    if (st != GDR_OK) return st;
    // the tensor-core path reads q, k, v as TMA tiles, which start on 16-byte boundaries
    if (!(al16(q) && al16(k) && al16(v))) {
        if (path == GDR_PATH_TC) return GDR_ERR_UNSUPPORTED;
        path = GDR_PATH_SIMT;
    }
    path = resolve_path(path, dtype, dk, dv, chunk);
    return run_forward(q, k, v, a, beta, h0, out, hT, cu_seqlens, s, b, dtype, gate, path,
                       workspace, workspace_bytes, (cudaStream_t)stream);
}

gdr_status_t gdr_chunk_fwd(const void *q, const void *k, const void *v, const void *a,
                           const void *beta, const float *h0, void *out, float *hT,
                           const int32_t *cu_seqlens, int B, int64_t T, int H, int dk, int dv,
                           int chunk, float b, gdr_stream_t stream) {
    return gdr_chunk_fwd_ex(q, k, v, a, beta, h0, out, hT, cu_seqlens, B, T, H, dk, dv, chunk, b,
                            GDR_BF16, GDR_GATE_BOUNDED, GDR_PATH_AUTO, nullptr, 0, stream);
}

size_t gdr_chunk_fwd_workspace_size(int B, int64_t T, int H, int dk, int dv, int chunk,
                                    gdr_dtype_t dtype, gdr_path_t path) {
    if (B < 1 || H < 1 || T < 0 || (dk != 64 && dk != 128) || (dv != 64 && dv != 128) ||
        (chunk != 16 && chunk != 32 && chunk != 64) || (dtype != GDR_BF16 && dtype != GDR_F32))
        return 0;
    if (path == GDR_PATH_TC && !tc_supported(dtype, dk, dv, chunk)) return 0;
    // AUTO may run either path (unaligned q, k, v take the CUDA-core one): the larger
    // of the two, and of the dense (B*T tokens) and varlen (T tokens) readings of (B, T)
    const gdr_path_t resolved = resolve_path(path, dtype, dk, dv, chunk);
    const gdr_path_t paths[2] = {resolved, path == GDR_PATH_AUTO ? GDR_PATH_SIMT : resolved};
    size_t best = 0;
    for (int pi = 0; pi < 2; ++pi) {
        for (int varlen = 0; varlen < 2; ++varlen) {
            Shape s;
            s.N = B;
            s.H = H;
            s.dk = dk;
            s.dv = dv;
            s.C = chunk;
            s.T_total = varlen ? T : (int64_t)B * T;
            s.T_per = varlen ? 0 : T;
            s.varlen = varlen != 0;
            s.max_chunks = tile_bound(s.varlen, B, T, chunk);
            const size_t n = layout_for(s, paths[pi]).total;
            if (n > best) best = n;
        }
    }
    return best;
}

gdr_status_t gdr_chunk_fwd_host(const void *q, const void *k, const void *v, const void *a,
                                const void *beta, const float *h0, void *out, float *hT,
                                const int32_t *cu_seqlens, int B, int64_t T, int H, int dk,
                                int dv, int chunk, float b, gdr_dtype_t dtype, gdr_gate_t gate,
                                gdr_path_t path, gdr_stream_t stream_) {
    Shape s;
    gdr_status_t st = check_args(q, k, v, a, beta, h0, out, hT, cu_seqlens, B, T, H, dk, dv,
                                 chunk, b, dtype, gate, path, &s);
    if (st != GDR_OK) return st;
    cudaStream_t stream = (cudaStream_t)stream_;
    {
        const std::vector<Piece> pcs = host_pieces(s, cu_seqlens);
        if (!pcs.empty())
            return fwd_host_pipelined(q, k, v, a, beta, h0, out, hT, cu_seqlens, s, pcs, b, dtype,
                                      gate, resolve_path(path, dtype, dk, dv, chunk), stream);
    }
    DeviceCtx *ctx = device_ctx();
    if (!ctx) return GDR_ERR_CUDA;
    const size_t es = dtype == GDR_BF16 ? 2 : 4;
    const size_t rows = (size_t)s.T_total * H;
    const size_t nst = (size_t)B * H * dk * dv * sizeof(float);
    const size_t sz[9] = {rows * dk * es, rows * dk * es, rows * dv * es, rows * es, rows * es,
                          h0 ? nst : 0,   rows * dv * es, hT ? nst : 0,
                          cu_seqlens ? sizeof(int32_t) * (size_t)(B + 1) : 0};
    size_t off[9], tot = 0;
    for (int i = 0; i < 9; ++i) {
        off[i] = tot;
        tot += align_up(sz[i]);
    }
    char *io;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!grow(&ctx->io, &ctx->io_bytes, tot)) return GDR_ERR_CUDA;
        io = (char *)ctx->io;
    }
    const void *src[9] = {q, k, v, a, beta, h0, nullptr, nullptr, cu_seqlens};
    for (int i = 0; i < 9; ++i)
        if (src[i] && sz[i] &&
            cudaMemcpyAsync(io + off[i], src[i], sz[i], cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return GDR_ERR_CUDA;
    path = resolve_path(path, dtype, dk, dv, chunk);
    st = run_forward(io + off[0], io + off[1], io + off[2], io + off[3], io + off[4],
                     h0 ? (const float *)(io + off[5]) : nullptr, io + off[6],
                     hT ? (float *)(io + off[7]) : nullptr,
                     cu_seqlens ? (const int32_t *)(io + off[8]) : nullptr, s, b, dtype, gate,
                     path, nullptr, 0, stream);
    if (st != GDR_OK) return st;
    if (s.T_total > 0 &&
        cudaMemcpyAsync(out, io + off[6], sz[6], cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return GDR_ERR_CUDA;
    if (hT && cudaMemcpyAsync(hT, io + off[7], sz[7], cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return GDR_ERR_CUDA;
    return cudaStreamSynchronize(stream) == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

gdr_status_t gdr_recurrent_fwd(const void *q, const void *k, const void *v, const void *a,
                               const void *beta, float *state, void *out, int N, int64_t T,
                               int H, int dk, int dv, float b, gdr_dtype_t dtype,
                               gdr_gate_t gate, gdr_stream_t stream) {
    if (dtype != GDR_BF16 && dtype != GDR_F32) return GDR_ERR_INVALID_ARG;
    if (gate != GDR_GATE_BOUNDED && gate != GDR_GATE_SOFTPLUS) return GDR_ERR_INVALID_ARG;
    if (N < 1 || H < 1 || T < 0) return GDR_ERR_INVALID_ARG;
    if (gate == GDR_GATE_BOUNDED && !(b > 0.f && std::isfinite(b))) return GDR_ERR_INVALID_ARG;
    if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return GDR_ERR_UNSUPPORTED;
    if (T > ((int64_t)1 << 40) || (int64_t)N * T > ((int64_t)1 << 40)) return GDR_ERR_UNSUPPORTED;
    if (T == 0) return GDR_OK;
    if (!q || !k || !v || !a || !beta || !state || !out) return GDR_ERR_INVALID_ARG;
    if (!al16(state)) return GDR_ERR_INVALID_ARG;   // read and written as float4
    const size_t es = dtype == GDR_BF16 ? 2 : 4;
    const size_t rows = (size_t)N * T * H;
    const size_t out_bytes = rows * dv * es, n_state = (size_t)N * H * dk * dv * sizeof(float);
    const void *ins[5] = {q, k, v, a, beta};
    const size_t in_bytes[5] = {rows * dk * es, rows * dk * es, rows * dv * es, rows * es, rows * es};
    for (int i = 0; i < 5; ++i)
        if (overlaps(out, out_bytes, ins[i], in_bytes[i]) || overlaps(state, n_state, ins[i], in_bytes[i]))
            return GDR_ERR_INVALID_ARG;
    if (overlaps(out, out_bytes, state, n_state)) return GDR_ERR_INVALID_ARG;
    return launch_recurrent(q, k, v, a, beta, state, out, dtype, N, T, H, dk, dv, b, gate,
                            (cudaStream_t)stream) == cudaSuccess
               ? GDR_OK
               : GDR_ERR_CUDA;
}

// GDR_BWD_TOKEN=1 sends every backward call to the token-by-token kernels (the
// parity tests compare the two forms).
static bool bwd_force_token_path() {
    const char *e = std::getenv("GDR_BWD_TOKEN");
    return e && e[0] == '1';
}

// GDR_VEC_MMA=1 runs the per-channel forward on the earlier mma.sync kernel instead
// of the tcgen05 one (for comparisons).
static bool vec_use_mma_sync() {
    const char *e = std::getenv("GDR_VEC_MMA");
    return e && e[0] == '1';
}

static gdr_status_t chunk_bwd_impl(const void *q, const void *k, const void *v, const void *a,
                           const void *beta, const float *h0, const void *dout,
                           const float *dhT, void *dq, void *dk_out, void *dv_out, void *da,
                           void *dbeta, float *dh0, const int32_t *cu_seqlens, int B,
                           int64_t T, int H, int dk, int dv, int chunk, float b,
                           gdr_dtype_t dtype, gdr_gate_t gate, gdr_stream_t stream_,
                           bool per_channel) {
    Shape s;
    // the forward's checks (with dq standing in for out in the aliasing tests)
    gdr_status_t st = check_args(q, k, v, a, beta, h0, dq, nullptr, cu_seqlens, B, T, H, dk, dv,
                                 chunk, b, dtype, gate, GDR_PATH_SIMT, &s);
    if (st != GDR_OK) return st;
    if (s.T_total > 0 && (!dq || !dk_out || !dv_out || !da || !dbeta)) return GDR_ERR_INVALID_ARG;
    // the per-channel form exists as the chunked tensor-core form only
    if (per_channel && (dtype != GDR_BF16 || dk != 128 || dv != 128 || gate != GDR_GATE_BOUNDED ||
                        b > kVecMaxB || chunk != kBwTile))
        return GDR_ERR_UNSUPPORTED;
    const size_t es = dtype == GDR_BF16 ? 2 : 4;
    const size_t rows = (size_t)s.T_total * H;
    const size_t a_b = rows * (per_channel ? dk : 1) * es;   // a and da
    const void *ins[6] = {q, k, v, a, beta, dout};
    const size_t in_b[6] = {rows * dk * es, rows * dk * es, rows * dv * es, a_b, rows * es,
                            rows * dv * es};
    void *outs[5] = {dq, dk_out, dv_out, da, dbeta};
    const size_t out_b[5] = {rows * dk * es, rows * dk * es, rows * dv * es, a_b, rows * es};
    for (int i = 0; i < 5; ++i)
        for (int j = 0; j < 6; ++j)
            if (overlaps(outs[i], out_b[i], ins[j], in_b[j])) return GDR_ERR_INVALID_ARG;
    const size_t nst = (size_t)B * H * dk * dv * sizeof(float);
    if (dh0 && (overlaps(dh0, nst, h0, nst) || overlaps(dh0, nst, dhT, nst))) return GDR_ERR_INVALID_ARG;
    if (!al16(dhT) || !al16(dh0)) return GDR_ERR_INVALID_ARG;   // copied as float4
    if (s.T_total == 0) {   // no tokens: dh0 = dhT
        if (!dh0) return GDR_OK;
        cudaStream_t stream = (cudaStream_t)stream_;
        const cudaError_t e = dhT ? cudaMemcpyAsync(dh0, dhT, nst, cudaMemcpyDeviceToDevice, stream)
                                  : cudaMemsetAsync(dh0, 0, nst, stream);
        return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
    }
    DeviceCtx *ctx = device_ctx();
    if (!ctx) return GDR_ERR_CUDA;
    const int64_t tiles = tile_bound(s.varlen, B, s.varlen ? T : s.T_per, kBwTile);
    const size_t plan_b = align_up(3 * sizeof(int64_t) * (size_t)(B + 1));
    // the chunked tensor-core form takes bf16, d = 128 and the bounded gate (its
    // factored in-tile decays need exp(16 b) < FLT_MAX); the rest runs token by token
    // (the scalar gate's tile kernel moves q, k, v, dout and dv in 16-byte pieces, dq and
    // dk in 4-byte pairs)
    const bool chunked = per_channel || (dtype == GDR_BF16 && dk == 128 && dv == 128 &&
                                         gate == GDR_GATE_BOUNDED && b <= kVecMaxB && al16(q) && al16(k) &&
                                         al16(v) && al16(dout) && al16(dv_out) && al16(dq) && al16(dk_out) &&
                                         !bwd_force_token_path());
    const int seg = chunked ? chunk_bwd_segment_tiles(tiles, H, ctx->sms) : (1 << 30);
    const int64_t segs = s.varlen ? (tiles + seg - 1) / seg + B : (int64_t)B * ((tiles / B + seg - 1) / seg);
    const size_t need = plan_b + (chunked ? chunk_bwd_scratch_bytes(tiles, B, H)
                                          : bwd_scratch_bytes(tiles, s.T_total, H, dk, dv));
    char *ws;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!grow(&ctx->ws, &ctx->ws_bytes, need)) return GDR_ERR_CUDA;
        ws = (char *)ctx->ws;
    }
    cudaStream_t stream = (cudaStream_t)stream_;
    int64_t *seq_start = (int64_t *)ws;
    Plan plan{B, kBwTile, seg, seq_start, seq_start + (B + 1), seq_start + 2 * (B + 1)};
    if (launch_plan(cu_seqlens, B, s.T_per, s.T_total, kBwTile, seg, seq_start, seq_start + (B + 1),
                    seq_start + 2 * (B + 1), ctx->d_status, stream) != cudaSuccess)
        return GDR_ERR_CUDA;
    if (chunked)
        return launch_chunk_bwd(q, k, v, a, beta, h0, dout, dhT, dq, dk_out, dv_out, da, dbeta, dh0,
                                plan, H, s.T_total, tiles, segs, b, per_channel, ws + plan_b,
                                ctx->d_status, stream, aux_stream(ctx)) == cudaSuccess
                   ? GDR_OK
                   : GDR_ERR_CUDA;
    return launch_bwd(q, k, v, a, beta, h0, dout, dhT, dq, dk_out, dv_out, da, dbeta, dh0, dtype,
                      plan, H, dk, dv, s.T_total, tiles, b, gate, ws + plan_b, stream) == cudaSuccess
               ? GDR_OK
               : GDR_ERR_CUDA;
}

gdr_status_t gdr_chunk_bwd(const void *q, const void *k, const void *v, const void *a,
                           const void *beta, const float *h0, const void *dout,
                           const float *dhT, void *dq, void *dk_out, void *dv_out, void *da,
                           void *dbeta, float *dh0, const int32_t *cu_seqlens, int B,
                           int64_t T, int H, int dk, int dv, int chunk, float b,
                           gdr_dtype_t dtype, gdr_gate_t gate, gdr_stream_t stream) {
    return chunk_bwd_impl(q, k, v, a, beta, h0, dout, dhT, dq, dk_out, dv_out, da, dbeta, dh0,
                          cu_seqlens, B, T, H, dk, dv, chunk, b, dtype, gate, stream, false);
}

gdr_status_t gdr_chunk_bwd_vec(const void *q, const void *k, const void *v, const void *a,
                               const void *beta, const float *h0, const void *dout,
                               const float *dhT, void *dq, void *dk_out, void *dv_out, void *da,
                               void *dbeta, float *dh0, const int32_t *cu_seqlens, int B,
                               int64_t T, int H, int dk, int dv, int chunk, float b,
                               gdr_dtype_t dtype, gdr_stream_t stream) {
    return chunk_bwd_impl(q, k, v, a, beta, h0, dout, dhT, dq, dk_out, dv_out, da, dbeta, dh0,
                          cu_seqlens, B, T, H, dk, dv, chunk, b, dtype, GDR_GATE_BOUNDED, stream,
                          true);
}

gdr_status_t gdr_chunk_fwd_vec(const void *q, const void *k, const void *v, const void *a,
                               const void *beta, const float *h0, void *out, float *hT,
                               const int32_t *cu_seqlens, int B, int64_t T, int H, int dk, int dv,
                               int chunk, float b, gdr_dtype_t dtype, gdr_stream_t stream_) {
    Shape s;
    gdr_status_t st = check_args(q, k, v, a, beta, h0, out, hT, cu_seqlens, B, T, H, dk, dv, chunk,
                                 b, dtype, GDR_GATE_BOUNDED, GDR_PATH_SIMT, &s);
    if (st != GDR_OK) return st;
    if (chunk != kVecTile || b > kVecMaxB) return GDR_ERR_UNSUPPORTED;
    // a holds dk gate inputs per (token, head): check it against the outputs too
    const size_t es = dtype == GDR_BF16 ? 2 : 4;
    const size_t rows = (size_t)s.T_total * H;
    const size_t a_bytes = rows * dk * es, out_bytes = rows * dv * es;
    const size_t nst = (size_t)B * H * dk * dv * sizeof(float);
    if (overlaps(out, out_bytes, a, a_bytes) || overlaps(hT, nst, a, a_bytes)) return GDR_ERR_INVALID_ARG;
    cudaStream_t stream = (cudaStream_t)stream_;
    if (s.T_total == 0) {   // no tokens: hT = h0
        if (!hT) return GDR_OK;
        const cudaError_t e = h0 ? cudaMemcpyAsync(hT, h0, nst, cudaMemcpyDeviceToDevice, stream)
                                 : cudaMemsetAsync(hT, 0, nst, stream);
        return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
    }
    DeviceCtx *ctx = device_ctx();
    if (!ctx) return GDR_ERR_CUDA;
    // tensor-core kernel; it reads q, k, v, a and writes out in 16-byte pieces, so an
    // unaligned one of those takes the CUDA-core kernels
    const bool aligned16 = ((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)a |
                            (uintptr_t)out) % 16 == 0;
    const bool fused = dtype == GDR_BF16 && dk == 128 && dv == 128 && aligned16;
    const int64_t tiles = tile_bound(s.varlen, B, T, kVecTile);
    const size_t plan_b = align_up(3 * sizeof(int64_t) * (size_t)(B + 1));
    const int seg = fused ? vec_mma_segment_tiles(tiles, H, ctx->sms) : (1 << 30);
    // segments: at most one partial segment per sequence beyond the full ones
    const int64_t segs = s.varlen ? (tiles + seg - 1) / seg + B : (int64_t)B * ((tiles / B + seg - 1) / seg);
    const size_t need = plan_b + (fused ? vec_mma_scratch_bytes(segs, H)
                                        : vec_scratch_bytes(tiles, s.T_total, H, dk, dv));
    char *ws;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!grow(&ctx->ws, &ctx->ws_bytes, need)) return GDR_ERR_CUDA;
        ws = (char *)ctx->ws;
    }
    int64_t *seq_start = (int64_t *)ws;
    Plan plan{B, kVecTile, seg, seq_start, seq_start + (B + 1), seq_start + 2 * (B + 1)};
    if (launch_plan(cu_seqlens, B, s.T_per, s.T_total, kVecTile, seg, seq_start,
                    seq_start + (B + 1), seq_start + 2 * (B + 1), ctx->d_status, stream) != cudaSuccess)
        return GDR_ERR_CUDA;
    if (fused && vec_use_mma_sync())
        return launch_vec_mma(q, k, v, a, beta, h0, out, hT, plan, H, b, segs, ws + plan_b, stream) ==
                       cudaSuccess
                   ? GDR_OK
                   : GDR_ERR_CUDA;
    if (fused) {   // tcgen05 kernel after the warm-up search
        int *warm = (int *)(ws + plan_b);
        if (launch_vec_warm(a, k, beta, warm, plan, H, b, segs, stream) != cudaSuccess) return GDR_ERR_CUDA;
        return launch_tc_vec(q, k, v, a, beta, h0, out, hT, plan, H, s.T_total, b, segs, warm,
                             ctx->d_status, stream) == cudaSuccess
                   ? GDR_OK
                   : GDR_ERR_CUDA;
    }
    return launch_vec_forward(q, k, v, a, beta, h0, out, hT, dtype, plan, H, dk, dv, s.T_total, tiles,
                              b, ws + plan_b, stream) == cudaSuccess
               ? GDR_OK
               : GDR_ERR_CUDA;
}

gdr_status_t gdr_router_topk(const void *logits, const float *bias, int32_t *topk_idx,
                             float *topk_logit, int64_t *load, int64_t T, int E, int k,
                             gdr_dtype_t dtype, gdr_stream_t stream) {
    if (dtype != GDR_BF16 && dtype != GDR_F32) return GDR_ERR_INVALID_ARG;
    if (T < 0 || E < 1 || k < 1) return GDR_ERR_INVALID_ARG;
    if (E > kRouterMaxE || E % 4 != 0 || k > E || k > kRouterMaxK) return GDR_ERR_UNSUPPORTED;
    if (T > ((int64_t)1 << 40)) return GDR_ERR_UNSUPPORTED;
    if (T == 0) return GDR_OK;
    if (!logits || !bias || !topk_idx) return GDR_ERR_INVALID_ARG;
    if ((uintptr_t)logits % 16 != 0) return GDR_ERR_INVALID_ARG;
    const size_t es = dtype == GDR_BF16 ? 2 : 4;
    const size_t xb = (size_t)T * E * es, bb = sizeof(float) * (size_t)E;
    const size_t ib = sizeof(int32_t) * (size_t)T * k, sb = sizeof(float) * (size_t)T * k;
    const size_t lb = sizeof(int64_t) * (size_t)E;
    const void *outs[3] = {topk_idx, topk_logit, load};
    const size_t ob[3] = {ib, sb, lb};
    for (int i = 0; i < 3; ++i) {
        if (overlaps(outs[i], ob[i], logits, xb) || overlaps(outs[i], ob[i], bias, bb))
            return GDR_ERR_INVALID_ARG;
        for (int j = i + 1; j < 3; ++j)
            if (overlaps(outs[i], ob[i], outs[j], ob[j])) return GDR_ERR_INVALID_ARG;
    }
    return launch_router_topk(logits, bias, topk_idx, topk_logit, load, T, E, k, dtype,
                              (cudaStream_t)stream) == cudaSuccess
               ? GDR_OK
               : GDR_ERR_CUDA;
}

gdr_status_t gdr_router_bias_update(const int64_t *load, float *bias, double *thresholds, int E,
                                    gdr_qb_mode_t mode, double q_lo, double q_hi, float eta,
                                    gdr_stream_t stream) {
    if (E < 1) return GDR_ERR_INVALID_ARG;
    if (E > kRouterMaxE) return GDR_ERR_UNSUPPORTED;
    if (mode != GDR_QB_SIGN && mode != GDR_QB_PROPORTIONAL) return GDR_ERR_INVALID_ARG;
    if (!(q_lo >= 0.0 && q_lo <= 1.0) || !(q_hi >= 0.0 && q_hi <= 1.0) || !std::isfinite(eta))
        return GDR_ERR_INVALID_ARG;
    if (!load || !bias) return GDR_ERR_INVALID_ARG;
    const size_t lb = sizeof(int64_t) * (size_t)E, bb = sizeof(float) * (size_t)E;
    if (overlaps(bias, bb, load, lb) || overlaps(thresholds, 16, load, lb) ||
        overlaps(thresholds, 16, bias, bb))
        return GDR_ERR_INVALID_ARG;
    return launch_router_update(load, bias, thresholds, E, (int)mode, q_lo, q_hi, eta,
                                (cudaStream_t)stream) == cudaSuccess
               ? GDR_OK
               : GDR_ERR_CUDA;
}

gdr_status_t gdr_gate_cumsum(const void *a, float *G, const int32_t *cu_seqlens, int B,
                             int64_t T, int H, int chunk, float b, gdr_dtype_t dtype,
                             gdr_gate_t gate, gdr_stream_t stream) {
    if (dtype != GDR_BF16 && dtype != GDR_F32) return GDR_ERR_INVALID_ARG;
    if (gate != GDR_GATE_BOUNDED && gate != GDR_GATE_SOFTPLUS) return GDR_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || T < 0 || chunk < 1) return GDR_ERR_INVALID_ARG;
    if (gate == GDR_GATE_BOUNDED && !(b > 0.f && std::isfinite(b))) return GDR_ERR_INVALID_ARG;
    if (chunk != 16 && chunk != 32 && chunk != 64) return GDR_ERR_UNSUPPORTED;
    const int64_t T_total = cu_seqlens ? T : (int64_t)B * T;
    if (T_total > 0 && (!a || !G)) return GDR_ERR_INVALID_ARG;
    DeviceCtx *ctx = device_ctx();
    if (!ctx) return GDR_ERR_CUDA;
    const size_t need = align_up(3 * sizeof(int64_t) * (size_t)(B + 1));
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!grow(&ctx->ws, &ctx->ws_bytes, need)) return GDR_ERR_CUDA;
    }
    int64_t *seq_start = (int64_t *)ctx->ws;
    Plan plan{B, chunk, 1 << 30, seq_start, seq_start + (B + 1), seq_start + 2 * (B + 1)};
    cudaStream_t st = (cudaStream_t)stream;
    if (launch_plan(cu_seqlens, B, cu_seqlens ? 0 : T, T_total, chunk, 1 << 30, seq_start,
                    seq_start + (B + 1), seq_start + 2 * (B + 1), ctx->d_status, st) != cudaSuccess)
        return GDR_ERR_CUDA;
    const int64_t max_chunks = tile_bound(cu_seqlens != nullptr, B, T, chunk);
    if (launch_gate_cumsum(a, nullptr, dtype, G, nullptr, plan, H, T_total, max_chunks, b, gate,
                           st) != cudaSuccess)
        return GDR_ERR_CUDA;
    return GDR_OK;
}

gdr_status_t gdr_wy_repr(const void *k, const void *v, const void *beta, const float *G,
                         float *W, float *U, const int32_t *cu_seqlens, int B, int64_t T, int H,
                         int dk, int dv, int chunk, gdr_dtype_t dtype, gdr_stream_t stream) {
    if (dtype != GDR_BF16 && dtype != GDR_F32) return GDR_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || T < 0 || chunk < 1 || dk < 1 || dv < 1) return GDR_ERR_INVALID_ARG;
    if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return GDR_ERR_UNSUPPORTED;
    if (chunk != 16 && chunk != 32 && chunk != 64) return GDR_ERR_UNSUPPORTED;
    const int64_t T_total = cu_seqlens ? T : (int64_t)B * T;
    if (T_total > 0 && (!k || !v || !beta || !G || !W || !U)) return GDR_ERR_INVALID_ARG;
    DeviceCtx *ctx = device_ctx();
    if (!ctx) return GDR_ERR_CUDA;
    const size_t need = align_up(3 * sizeof(int64_t) * (size_t)(B + 1));
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!grow(&ctx->ws, &ctx->ws_bytes, need)) return GDR_ERR_CUDA;
    }
    int64_t *seq_start = (int64_t *)ctx->ws;
    Plan plan{B, chunk, 1 << 30, seq_start, seq_start + (B + 1), seq_start + 2 * (B + 1)};
    cudaStream_t st = (cudaStream_t)stream;
    if (launch_plan(cu_seqlens, B, cu_seqlens ? 0 : T, T_total, chunk, 1 << 30, seq_start,
                    seq_start + (B + 1), seq_start + 2 * (B + 1), ctx->d_status, st) != cudaSuccess)
        return GDR_ERR_CUDA;
    const int64_t max_chunks = tile_bound(cu_seqlens != nullptr, B, T, chunk);
    if (launch_wy_simt(k, v, beta, G, W, U, dtype, plan, H, dk, dv, T_total, max_chunks, st) !=
        cudaSuccess)
        return GDR_ERR_CUDA;
    return GDR_OK;
}

gdr_status_t gdr_get_status(gdr_stream_t stream) {
    DeviceCtx *ctx = device_ctx();
    if (!ctx) return GDR_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDR_ERR_CUDA;
    int code = 0;
    if (cudaMemcpy(&code, ctx->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GDR_ERR_CUDA;
    if (code != 0 && cudaMemset(ctx->d_status, 0, sizeof(int)) != cudaSuccess) return GDR_ERR_CUDA;
#ifdef GDR_DEBUG
    {
        std::lock_guard<std::mutex> lk(debug_mu());
        for (DebugFlagReader fn : debug_readers())
            if (fn() && code == 0) code = GDR_ERR_BOUNDS;
    }
#endif
    return (gdr_status_t)code;
}

const char *gdr_status_string(gdr_status_t status) {
    switch (status) {
        case GDR_OK: return "ok";
        case GDR_ERR_INVALID_ARG: return "invalid argument";
        case GDR_ERR_UNSUPPORTED: return "unsupported size or option";
        case GDR_ERR_CUDA: return "CUDA runtime error";
        case GDR_ERR_TIMEOUT: return "device-side wait timed out";
        case GDR_ERR_NO_WORKSPACE: return "workspace too small";
        case GDR_ERR_BAD_SEQLENS: return "cu_seqlens is not a valid offset list";
        case GDR_ERR_BOUNDS: return "device-side index check failed (checking build)";
    }
    return "unknown status";
}

void gdr_release(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (size_t d = 0; d < g_ctx.size(); ++d) {
        DeviceCtx &c = g_ctx[d];
        if (!c.ws && !c.io && !c.d_status && !c.s_in && !c.aux.stream) continue;
        cudaSetDevice((int)d);
        cudaDeviceSynchronize();
        if (c.ws) cudaFree(c.ws);
        if (c.io) cudaFree(c.io);
        if (c.d_status) cudaFree(c.d_status);
        if (c.s_in) cudaStreamDestroy(c.s_in);
        if (c.s_out) cudaStreamDestroy(c.s_out);
        if (c.aux.stream) cudaStreamDestroy(c.aux.stream);
        if (c.aux.fork) cudaEventDestroy(c.aux.fork);
        if (c.aux.join) cudaEventDestroy(c.aux.join);
        for (int i = 0; i < kMaxPieces; ++i) {
            if (c.ev_in[i]) cudaEventDestroy(c.ev_in[i]);
            if (c.ev_comp[i]) cudaEventDestroy(c.ev_comp[i]);
            if (c.ev_out[i]) cudaEventDestroy(c.ev_out[i]);
        }
        c = DeviceCtx{};
    }
    cudaSetDevice(cur);
}

uint64_t gdr_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void gdr_profile_enable(int on) { g_prof_on.store(on != 0); }

void gdr_profile_select(const char *name) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_only = name ? name : "";
}

int gdr_profile_read(const char **names, double *total_ms, int *launches, int max) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    std::vector<const char *> nm;
    std::vector<double> ms;
    std::vector<int> cnt;
    for (const ProfRec &r : g_prof) {
        float t = 0.f;
        cudaEventSynchronize(r.stop);
        if (cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess) t = 0.f;
        size_t i = 0;
        while (i < nm.size() && std::strcmp(nm[i], r.name) != 0) ++i;
        if (i == nm.size()) {
            nm.push_back(r.name);
            ms.push_back(0.0);
            cnt.push_back(0);
        }
        ms[i] += t;
        cnt[i] += 1;
        g_prof_pool.push_back(r.start);
        g_prof_pool.push_back(r.stop);
    }
    g_prof.clear();
    for (size_t i = 0; i < nm.size() && (int)i < max; ++i) {
        if (names) names[i] = nm[i];
        if (total_ms) total_ms[i] = ms[i];
        if (launches) launches[i] = cnt[i];
    }
    return (int)nm.size();
}

}  // extern "C"
