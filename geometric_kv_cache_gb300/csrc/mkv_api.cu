// C ABI of the compression path (declared in include/mkv.h): host-side
// argument checks, workspace carving and the launch sequence. Nothing here
// allocates device memory or synchronises, except mkv_device_status.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "mkv_internal.h"

namespace mkv {

namespace {

constexpr size_t kAlign = 256;

// Whether mkv_compress may use the single-pass centroid + score kernel
// (mkv_set_single_pass). Off by default: on GB300 the three-kernel path is
// currently faster for every measured shape.
std::atomic<int> g_single_pass_enabled{0};

// Whether mkv_compress may use the head-group kernel (one read of K from
// HBM, global centroids, heads short enough for L2). On by default.
std::atomic<int> g_head_groups_enabled{1};
// Whether the head groups may use the copy-ring kernel where it applies
// (bf16, head dim 128; mkv_set_head_group_ring).
std::atomic<int> g_head_group_ring{0};

// The head-group plan mkv_compress takes: the copy-ring kernel where it
// applies and is allowed, else the register kernel (groups 0: neither).
HeadGroupPlan choose_head_groups(const PieceGeometry &pg, int mode, size_t counters)
{
    if (g_head_group_ring.load(std::memory_order_relaxed)) {
        const HeadGroupPlan r = head_group_ring_plan(pg, mode, counters);
        if (r.groups > 0) return r;
    }
    return head_group_plan(pg, mode, counters);
}
// The fused whole-path kernel (mkv_set_fused): the scorer CTA budget (0: off,
// < 0: automatic) and the selector CTAs of a forced budget.
std::atomic<int> g_fused_scorers{-1};
std::atomic<int> g_fused_selectors{32};

// Scorer and selector budgets of the fused kernel for this shape; scorers 0
// when it is not to run. Automatic: bf16 caches, head dim 128, global
// centroids, 12288 < t_max (<= 20480, the kernel's own limit) and at least
// 64 heads, where it was measured faster than the separate kernels on GB300
// (256 heads x 16K: 0.620 against 0.649 ms; 64 x 16K: 0.187 against 0.204)
// -- not with fewer heads (32 x 16K: 0.119 against 0.113), at 8K tokens
// (512 x 8K: 0.687 against 0.648) nor for E4M3 caches (256 x 16K: 0.558
// against 0.42), whose scoring is decode-bound. There it uses 3/4 of the
// resident grid for scoring and max(16, heads / 16) selector CTAs (fewer
// than 16 made the selects the bottleneck: 1.03 ms with 8).
struct FusedBudget {
    int scorers = 0, selectors = 0;
};
FusedBudget fused_budget(const Geometry &g)
{
    FusedBudget b;
    const int sc = g_fused_scorers.load(std::memory_order_relaxed);
    if (sc > 0) {
        b.scorers = sc;
        b.selectors = g_fused_selectors.load(std::memory_order_relaxed);
    } else if (sc < 0 && g.es == 2 && g.d == kHeadDim && g.pg.nwin_max == 1 && g.t_max > 12288 && g.n_heads >= 64) {
        b.scorers = -1;  // 3/4 of the resident grid (fused_plan)
        b.selectors = (int)std::max<int64_t>(16, (g.n_heads + 15) / 16);
    }
    return b;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// floor(T*(1-ratio) + 0.5) clamped to [0, T]; volatile stops the host
// compiler from fusing the multiply and add, so this rounds like the kernels.
int32_t host_num_keep(int32_t T, double ratio)
{
    if (T <= 0) return 0;
    volatile double one_minus = 1.0 - ratio;
    volatile double prod = (double)T * one_minus;
    volatile double sum = prod + 0.5;
    const double x = floor(sum);
    if (x < 0.0) return 0;
    if (x > (double)T) return T;
    return (int32_t)x;
}

bool ratio_ok(double r) { return r >= 0.0 && r <= 1.0; }  // false for NaN

// Kept tokens of a T-token head when each window keeps its own share.
int64_t host_num_keep_quota(int32_t T, double ratio, int32_t window)
{
    if (T <= 0) return 0;
    if (window <= 0 || window >= T) return host_num_keep(T, ratio);
    const int32_t nw = (int32_t)(((int64_t)T + window - 1) / window);
    return (int64_t)(nw - 1) * host_num_keep(window, ratio) + host_num_keep(T - (nw - 1) * window, ratio);
}

// Shape checks shared by all entry points. Returns MKV_OK or the error.
mkv_status check_shape(const mkv_shape &s)
{
    if (s.batch < 0 || s.heads < 0 || s.t_max < 0 || s.head_dim <= 0) return MKV_ERR_INVALID_ARG;
    if (!supported_head_dim(s.head_dim) || elem_bytes(s.dtype) == 0) return MKV_ERR_UNSUPPORTED;
    if (s.t_max > (1 << 30)) return MKV_ERR_UNSUPPORTED;
    if (s.seq_lens && !aligned(s.seq_lens, 4)) return MKV_ERR_INVALID_ARG;
    return MKV_OK;
}

bool empty(const mkv_shape &s) { return s.batch == 0 || s.heads == 0 || s.t_max == 0; }

Geometry geometry_of(const mkv_shape &s, int32_t window)
{
    return make_geometry(s.batch, s.heads, s.t_max, window, s.head_dim, elem_bytes(s.dtype));
}

mkv_status check_ws(const Layout &L, void *ws, size_t ws_bytes)
{
    if (!ws || !aligned(ws, kAlign) || ws_bytes < L.total) return MKV_ERR_WORKSPACE;
    return MKV_OK;
}

// Workspace needs of the step-wise calls that use no partial sums, centroids
// or scores of their own: the status word and the compaction offsets. This is
// never larger than the full layout of the same shape.
Layout make_step_layout(const Geometry &g)
{
    Layout L;
    L.status = 0;
    L.chunk = kAlign;
    L.total = kAlign + round_up((size_t)g.n_heads * g.nch * sizeof(int2), kAlign);
    return L;
}

template <typename T>
T *region(void *ws, size_t off)
{
    return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

mkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MKV_OK : MKV_ERR_CUDA; }

// mkv_compress_host splits the batch rows into up to this many chunks, so
// that the copies of one chunk overlap the kernels and copies of others.
constexpr int32_t kHostChunks = 16;

// Library-owned copy streams and events of one device (created on first use,
// kept for the life of the process; the mutex serialises enqueueing).
// Keys and values are copied in on two streams (two copy engines move more
// than one), the results out on a third.
struct CopyStreams {
    std::mutex mu;
    cudaStream_t in[2] = {nullptr, nullptr}, out = nullptr;
    cudaEvent_t start = nullptr, out_done = nullptr;
    cudaEvent_t in_done[2][kHostChunks + 1] = {};
    cudaEvent_t comp_done[kHostChunks] = {};
};

CopyStreams *copy_streams()
{
    static std::mutex mu;
    static CopyStreams *table[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (table[dev]) return table[dev];
    CopyStreams *cs = new CopyStreams();
    const unsigned ef = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&cs->in[0], cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&cs->in[1], cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&cs->out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&cs->start, ef) == cudaSuccess &&
              cudaEventCreateWithFlags(&cs->out_done, ef) == cudaSuccess;
    for (int k = 0; k < 2; ++k)
        for (int i = 0; ok && i <= kHostChunks; ++i) ok = cudaEventCreateWithFlags(&cs->in_done[k][i], ef) == cudaSuccess;
    for (int i = 0; ok && i < kHostChunks; ++i) ok = cudaEventCreateWithFlags(&cs->comp_done[i], ef) == cudaSuccess;
    if (!ok) return nullptr;  // (the partial set is leaked; a CUDA error here is not recoverable anyway)
    table[dev] = cs;
    return cs;
}

// Checks of mkv_compact / mkv_compress outputs.
// quota_window > 0: per-window quotas, whose kept count bounds the stride.
mkv_status check_outputs(const mkv_shape &s, double ratio, const int32_t *n_keep, int32_t keep_stride,
                         const void *K, const void *V, const void *K_out, const void *V_out,
                         const int32_t *idx, const int32_t *kept, bool need_kv, int32_t quota_window = 0)
{
    if (!ratio_ok(ratio) || keep_stride < 0) return MKV_ERR_INVALID_ARG;
    if (quota_window > 0) {
        if (keep_stride < host_num_keep_quota(s.t_max, ratio, quota_window)) return MKV_ERR_INVALID_ARG;
    } else if (!n_keep && keep_stride < host_num_keep(s.t_max, ratio)) {
        return MKV_ERR_INVALID_ARG;
    }
    if (n_keep && !aligned(n_keep, 4)) return MKV_ERR_INVALID_ARG;
    if ((K_out == nullptr) != (V_out == nullptr)) return MKV_ERR_INVALID_ARG;
    if (need_kv && !K_out) return MKV_ERR_INVALID_ARG;
    if (K_out && (!K || !V)) return MKV_ERR_INVALID_ARG;
    if (K && !aligned(K, 16)) return MKV_ERR_INVALID_ARG;
    if (V && !aligned(V, 16)) return MKV_ERR_INVALID_ARG;
    if (K_out && (!aligned(K_out, 16) || !aligned(V_out, 16))) return MKV_ERR_INVALID_ARG;
    if (idx && !aligned(idx, 4)) return MKV_ERR_INVALID_ARG;
    if (kept && !aligned(kept, 4)) return MKV_ERR_INVALID_ARG;
    return MKV_OK;
}

// a1 + a2 as mkv_compress runs them: the head-group kernel (global
// centroids whose heads fit in L2, K read from HBM once), the single-pass
// kernel (opt-in), or piece sums + window means + scores. All write the same
// bits to C and S. `mark(i)` records the caller's stage events 1..3.
template <typename Mark>
mkv_status run_centroid_score(const Geometry &g, const Layout &L, const void *K, const mkv_shape &s, mkv_mode mode,
                              void *ws, float *C, float *S, cudaStream_t st, Mark &mark, bool stall_windows)
{
    uint32_t *status = region<uint32_t>(ws, L.status);
    float *partial = region<float>(ws, L.partial);
    cudaError_t e = cudaSuccess;
    const int grid = g.d == kHeadDim && g.es == 2 &&
                             (stall_windows || g_single_pass_enabled.load(std::memory_order_relaxed))
                         ? single_pass_grid((int)mode)
                         : 0;
    bool single = grid > 0 && grid >= g.pg.ppw;
    if (stall_windows && !single) return MKV_ERR_UNSUPPORTED;
    const HeadGroupPlan plan = (!single && g_head_groups_enabled.load(std::memory_order_relaxed))
                                   ? choose_head_groups(g.pg, (int)mode, L.centroid - L.counters)
                                   : HeadGroupPlan{};
    if (plan.groups > 0) {
        e = launch_head_groups(g.pg, plan, K, s.seq_lens, (int)mode, partial, region<uint32_t>(ws, L.counters), C, S,
                               status, st);
        if (e == cudaErrorCooperativeLaunchTooLarge) {  // fewer CTAs fit right now: the three-kernel path
            (void)cudaGetLastError();
            e = cudaSuccess;
        } else {
            if (e != cudaSuccess) return cuda_status(e);
            single = true;
            if (!mark(1) || !mark(2) || !mark(3)) return MKV_ERR_CUDA;
        }
    } else if (single) {
        e = launch_single_pass(g.pg, grid, K, s.seq_lens, (int)mode, partial, region<float>(ws, L.gsum),
                               region<uint32_t>(ws, L.counters), C, S, status, st, stall_windows);
        if (e == cudaErrorCooperativeLaunchTooLarge) {  // fewer CTAs fit right now
            (void)cudaGetLastError();
            single = false;
            e = cudaSuccess;
        } else {
            if (e != cudaSuccess) return cuda_status(e);
            if (!mark(1) || !mark(2) || !mark(3)) return MKV_ERR_CUDA;
        }
    }
    if (!single) {
        if ((e = launch_piece_sums(g.pg, K, s.seq_lens, partial, status, st)) != cudaSuccess) return cuda_status(e);
        if (!mark(1)) return MKV_ERR_CUDA;
        if ((e = launch_window_means(g.pg, partial, s.seq_lens, C, status, st)) != cudaSuccess) return cuda_status(e);
        if (!mark(2)) return MKV_ERR_CUDA;
        if ((e = launch_piece_scores(g.pg, K, C, s.seq_lens, (int)mode, S, status, st)) != cudaSuccess)
            return cuda_status(e);
        if (!mark(3)) return MKV_ERR_CUDA;
    }
    return MKV_OK;
}

// The fused launch sequence; events (optional) bracket every kernel.
mkv_status run_compress(const void *K, const void *V, mkv_shape s, double ratio, const int32_t *n_keep,
                        mkv_mode mode, int32_t window, int32_t keep_stride, void *K_out, void *V_out,
                        int32_t *idx, int32_t *kept, void *ws, size_t ws_bytes, cudaStream_t st,
                        void *const *events, bool stall_windows = false, bool quota = false, bool in_place = false,
                        bool allow_fused = true, int stall_fused = -1)
{
    mkv_status rc = check_shape(s);
    if (rc != MKV_OK) return rc;
    if (!K || !V || window < 0 || (mode != MKV_MODE_L2 && mode != MKV_MODE_COSINE)) return MKV_ERR_INVALID_ARG;
    // per-window quotas; one window per head is the ordinary selection
    quota = quota && window > 0 && window < s.t_max;
    rc = check_outputs(s, ratio, n_keep, keep_stride, K, V, K_out, V_out, idx, kept, false, quota ? window : 0);
    if (rc != MKV_OK) return rc;
    const Geometry g = geometry_of(s, window);
    const Layout L = make_layout(g);
    rc = check_ws(L, ws, ws_bytes);
    if (rc != MKV_OK) return rc;
    if (empty(s)) return MKV_OK;
    uint32_t *status = region<uint32_t>(ws, L.status);
    float *C = region<float>(ws, L.centroid);
    float *S = region<float>(ws, L.score);
    mkv_cut *cut = region<mkv_cut>(ws, L.cut);
    int2 *chunk = region<int2>(ws, L.chunk);
    int32_t *kept_w = kept ? kept : region<int32_t>(ws, L.kept);
    auto mark = [&](int i) -> bool {
        return !events || cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) == cudaSuccess;
    };
    cudaError_t e = cudaSuccess;
    int32_t *idx_w = idx ? idx : region<int32_t>(ws, L.idx);
    const int32_t idx_stride = idx ? keep_stride : g.t_max;
    // the whole path in one launch, when the fused setting and the shape allow
    // it (a stall injection takes it wherever the kernel can run the shape)
    FusedBudget fb = fused_budget(g);
    if (stall_fused >= 0 && fb.scorers == 0) {
        fb.scorers = -1;
        fb.selectors = (int)std::max<int64_t>(16, (g.n_heads + 15) / 16);
    }
    if (fb.scorers != 0 && allow_fused && !events && !stall_windows && !quota && !in_place && K_out &&
        g_head_groups_enabled.load(std::memory_order_relaxed) && !g_single_pass_enabled.load(std::memory_order_relaxed)) {
        const FusedPlan fp = fused_plan(g.pg, (int)mode, L.centroid - L.counters, fb.scorers, fb.selectors);
        if (fp.grid > 0) {
            e = launch_fused(g.pg, fp, (int)mode, K, V, s.seq_lens, region<float>(ws, L.partial),
                             region<uint32_t>(ws, L.counters), C, S, ratio, n_keep, keep_stride, kept_w, idx_w,
                             idx_stride, K_out, V_out, status, st, stall_fused);
            if (e != cudaErrorCooperativeLaunchTooLarge || stall_fused >= 0) return cuda_status(e);
            (void)cudaGetLastError();  // fewer CTAs fit right now: the separate kernels
        }
    }
    if (stall_fused >= 0) return MKV_ERR_UNSUPPORTED;  // the fused kernel cannot run this shape here
    if (!mark(0)) return MKV_ERR_CUDA;
    // a1 + a2 (C and S are workspace regions here)
    rc = run_centroid_score(g, L, K, s, mode, ws, C, S, st, mark, stall_windows);
    if (rc != MKV_OK) return rc;
    // a3 (+ a4 when the head's scores fit shared memory), then a4, a5
    const bool emit = quota || select_emits_indices(g);
    if (quota)
        e = launch_select_quota(g, S, s.seq_lens, ratio, keep_stride, kept_w, idx_w, idx_stride, status, st);
    else
        e = launch_select(g, S, s.seq_lens, ratio, n_keep, keep_stride, cut, emit ? nullptr : chunk, kept_w,
                          emit ? idx_w : nullptr, idx_stride, status, st);
    if (e != cudaSuccess) return cuda_status(e);
    if (!mark(4)) return MKV_ERR_CUDA;
    if (!emit &&
        (e = launch_compact(g, S, cut, chunk, s.seq_lens, keep_stride, idx_w, idx_stride, status, st)) != cudaSuccess)
        return cuda_status(e);
    if (!mark(5)) return MKV_ERR_CUDA;
    if (in_place) {
        if ((e = launch_gather_inplace(g, idx_w, idx_stride, kept_w, s.seq_lens, const_cast<void *>(K),
                                       const_cast<void *>(V), status, st)) != cudaSuccess)
            return cuda_status(e);
    } else if (K_out &&
               (e = launch_gather(g, idx_w, idx_stride, kept_w, keep_stride, K, V, K_out, V_out, status, st,
                                  !quota && emit && select_single_wave(g))) != cudaSuccess) {
        return cuda_status(e);
    }
    if (!mark(6)) return MKV_ERR_CUDA;
    return MKV_OK;
}

constexpr int32_t kCompressStages = 6;

}  // namespace

Geometry make_geometry(int32_t batch, int32_t heads, int32_t t_max, int32_t window, int32_t head_dim, int32_t es)
{
    Geometry g;
    g.d = head_dim;
    g.pg.d = head_dim;
    g.es = es;
    g.pg.es = es;
    g.n_heads = (int64_t)batch * heads;
    g.heads = heads;
    g.t_max = t_max;
    g.nch = (t_max + kCompactChunk - 1) / kCompactChunk;
    PieceGeometry &p = g.pg;
    p.n_heads = g.n_heads;
    p.heads = heads;
    p.t_max = t_max;
    p.window = window;
    const int32_t wl_max = (window <= 0 || window >= t_max) ? t_max : window;
    p.nwin_max = t_max > 0 ? (int32_t)(((int64_t)t_max + wl_max - 1) / wl_max) : 0;
    // pieces of 256 * 2^k tokens: the smallest that keep a window within
    // kMaxPiecesPerWindow pieces (a function of the shape only)
    int32_t rows = kMinPieceRows;
    while (wl_max > 0 && (wl_max + rows - 1) / rows > kMaxPiecesPerWindow && rows < (1 << 24)) rows *= 2;
    p.piece_rows = rows;
    p.ppw = wl_max > 0 ? (wl_max + rows - 1) / rows : 0;
    p.ngroups_max = (p.ppw + kGroupPieces - 1) / kGroupPieces;
    p.n_items = g.n_heads * p.nwin_max * (int64_t)p.ppw;
    return g;
}

Layout make_layout(const Geometry &g)
{
    const PieceGeometry &p = g.pg;
    const size_t wins = (size_t)g.n_heads * p.nwin_max;
    Layout L;
    size_t off = 0;
    L.status = off;
    off += kAlign;
    L.partial = off;
    off += round_up(wins * p.ppw * p.d * sizeof(float), kAlign);
    L.gsum = off;
    off += round_up(wins * p.ngroups_max * p.d * sizeof(float), kAlign);
    L.counters = off;
    off += round_up(wins * (p.ngroups_max + 2) * sizeof(uint32_t), kAlign);
    L.centroid = off;
    off += round_up(wins * p.d * sizeof(float), kAlign);
    L.score = off;
    off += round_up((size_t)g.n_heads * g.t_max * sizeof(float), kAlign);
    L.cut = off;
    off += round_up((size_t)g.n_heads * sizeof(mkv_cut), kAlign);
    L.chunk = off;
    off += round_up((size_t)g.n_heads * g.nch * sizeof(int2), kAlign);
    L.kept = off;
    off += round_up((size_t)g.n_heads * sizeof(int32_t), kAlign);
    L.idx = off;  // kept indices when the caller does not ask for them (row stride t_max)
    off += round_up((size_t)g.n_heads * g.t_max * sizeof(int32_t), kAlign);
    L.total = off;
    return L;
}

}  // namespace mkv

using namespace mkv;

extern "C" {

int32_t mkv_num_keep(int32_t T, double ratio)
{
    if (T < 0 || !ratio_ok(ratio)) return -1;
    return host_num_keep(T, ratio);
}

int32_t mkv_num_windows(int32_t t_max, int32_t window)
{
    if (t_max < 0 || window < 0) return -1;
    return make_geometry(1, 1, t_max, window).pg.nwin_max;
}

size_t mkv_workspace_size(mkv_shape shape, int32_t window)
{
    if (check_shape(shape) != MKV_OK || window < 0) return 0;
    return make_layout(geometry_of(shape, window)).total;
}

mkv_status mkv_centroid(const void *K, mkv_shape shape, int32_t window, float *C, void *workspace,
                        size_t workspace_bytes, mkv_stream_t stream)
{
    mkv_status rc = check_shape(shape);
    if (rc != MKV_OK) return rc;
    if (!K || !C || window < 0 || !aligned(K, 16) || !aligned(C, 16)) return MKV_ERR_INVALID_ARG;
    const Geometry g = geometry_of(shape, window);
    const Layout L = make_layout(g);
    if ((rc = check_ws(L, workspace, workspace_bytes)) != MKV_OK) return rc;
    if (empty(shape)) return MKV_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t *status = region<uint32_t>(workspace, L.status);
    float *partial = region<float>(workspace, L.partial);
    cudaError_t e = launch_piece_sums(g.pg, K, shape.seq_lens, partial, status, st);
    if (e == cudaSuccess) e = launch_window_means(g.pg, partial, shape.seq_lens, C, status, st);
    return cuda_status(e);
}

mkv_status mkv_window_means(const void *X, mkv_shape shape, int32_t window, float *mean, float *radius,
                            void *workspace, size_t workspace_bytes, mkv_stream_t stream)
{
    mkv_status rc = check_shape(shape);
    if (rc != MKV_OK) return rc;
    if (!X || !mean || window < 0 || !aligned(X, 16) || !aligned(mean, 16)) return MKV_ERR_INVALID_ARG;
    if (radius && !aligned(radius, 4)) return MKV_ERR_INVALID_ARG;
    const Geometry g = geometry_of(shape, window);
    const bool small = window > 0 && window <= kSmallWindowMax;
    if (radius && !small) return MKV_ERR_UNSUPPORTED;
    const Layout L = make_layout(g);
    if ((rc = check_ws(L, workspace, workspace_bytes)) != MKV_OK) return rc;
    if (empty(shape)) return MKV_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t *status = region<uint32_t>(workspace, L.status);
    if (small) return cuda_status(launch_small_window_means(g.pg, X, shape.seq_lens, mean, radius, status, st));
    cudaError_t e = launch_piece_sums(g.pg, X, shape.seq_lens, region<float>(workspace, L.partial), status, st);
    if (e == cudaSuccess) e = launch_window_means(g.pg, region<float>(workspace, L.partial), shape.seq_lens, mean, status, st);
    return cuda_status(e);
}

mkv_status mkv_centroid_score(const void *K, mkv_shape shape, int32_t window, mkv_mode mode, float *C, float *S,
                              void *workspace, size_t workspace_bytes, mkv_stream_t stream)
{
    mkv_status rc = check_shape(shape);
    if (rc != MKV_OK) return rc;
    if (!K || !C || !S || window < 0 || !aligned(K, 16) || !aligned(C, 16) || !aligned(S, 4)) return MKV_ERR_INVALID_ARG;
    if (mode != MKV_MODE_L2 && mode != MKV_MODE_COSINE) return MKV_ERR_INVALID_ARG;
    const Geometry g = geometry_of(shape, window);
    const Layout L = make_layout(g);
    if ((rc = check_ws(L, workspace, workspace_bytes)) != MKV_OK) return rc;
    if (empty(shape)) return MKV_OK;
    auto mark = [](int) { return true; };
    return run_centroid_score(g, L, K, shape, mode, workspace, C, S, reinterpret_cast<cudaStream_t>(stream), mark, false);
}

mkv_status mkv_score(const void *K, const float *C, mkv_shape shape, int32_t window, mkv_mode mode, float *S,
                     void *workspace, size_t workspace_bytes, mkv_stream_t stream)
{
    mkv_status rc = check_shape(shape);
    if (rc != MKV_OK) return rc;
    if (!K || !C || !S || window < 0 || !aligned(K, 16) || !aligned(C, 16) || !aligned(S, 4)) return MKV_ERR_INVALID_ARG;
    if (mode != MKV_MODE_L2 && mode != MKV_MODE_COSINE) return MKV_ERR_INVALID_ARG;
    const Geometry g = geometry_of(shape, window);
    const Layout L = make_step_layout(g);
    if ((rc = check_ws(L, workspace, workspace_bytes)) != MKV_OK) return rc;
    if (empty(shape)) return MKV_OK;
    return cuda_status(launch_piece_scores(g.pg, K, C, shape.seq_lens, (int)mode, S,
                                           region<uint32_t>(workspace, L.status), reinterpret_cast<cudaStream_t>(stream)));
}

mkv_status mkv_select_topk(const float *S, mkv_shape shape, double ratio, const int32_t *n_keep, mkv_cut *cut,
                           void *workspace, size_t workspace_bytes, mkv_stream_t stream)
{
    mkv_status rc = check_shape(shape);
    if (rc != MKV_OK) return rc;
    if (!S || !cut || !aligned(S, 4) || !aligned(cut, 8) || !ratio_ok(ratio)) return MKV_ERR_INVALID_ARG;
    if (n_keep && !aligned(n_keep, 4)) return MKV_ERR_INVALID_ARG;
    const Geometry g = geometry_of(shape, 0);
    const Layout L = make_step_layout(g);
    if ((rc = check_ws(L, workspace, workspace_bytes)) != MKV_OK) return rc;
    if (empty(shape)) return MKV_OK;
    return cuda_status(launch_select(g, S, shape.seq_lens, ratio, n_keep, -1, cut, nullptr, nullptr, nullptr, 0,
                                     region<uint32_t>(workspace, L.status), reinterpret_cast<cudaStream_t>(stream)));
}

mkv_status mkv_compact(const float *S, const mkv_cut *cut, const void *K, const void *V, mkv_shape shape,
                       double ratio, const int32_t *n_keep, int32_t keep_stride, int32_t *idx, int32_t *kept,
                       void *K_out, void *V_out, void *workspace, size_t workspace_bytes, mkv_stream_t stream)
{
    mkv_status rc = check_shape(shape);
    if (rc != MKV_OK) return rc;
    if (!S || !cut || !idx || !kept || !aligned(S, 4) || !aligned(cut, 8)) return MKV_ERR_INVALID_ARG;
    rc = check_outputs(shape, ratio, n_keep, keep_stride, K, V, K_out, V_out, idx, kept, false);
    if (rc != MKV_OK) return rc;
    const Geometry g = geometry_of(shape, 0);
    const Layout L = make_step_layout(g);
    if ((rc = check_ws(L, workspace, workspace_bytes)) != MKV_OK) return rc;
    if (empty(shape)) return MKV_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t *status = region<uint32_t>(workspace, L.status);
    int2 *chunk = region<int2>(workspace, L.chunk);
    cudaError_t e = launch_chunk_offsets(g, S, cut, shape.seq_lens, ratio, n_keep, keep_stride, chunk, kept, status, st);
    if (e == cudaSuccess) e = launch_compact(g, S, cut, chunk, shape.seq_lens, keep_stride, idx, keep_stride, status, st);
    if (e == cudaSuccess && K_out)
        e = launch_gather(g, idx, keep_stride, kept, keep_stride, K, V, K_out, V_out, status, st);
    return cuda_status(e);
}

mkv_status mkv_compress(const void *K, const void *V, mkv_shape shape, double ratio, const int32_t *n_keep,
                        mkv_mode mode, int32_t window, int32_t keep_stride, void *K_out, void *V_out, int32_t *idx,
                        int32_t *kept, void *workspace, size_t workspace_bytes, mkv_stream_t stream)
{
    return run_compress(K, V, shape, ratio, n_keep, mode, window, keep_stride, K_out, V_out, idx, kept, workspace,
                        workspace_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

int32_t mkv_num_keep_quota(int32_t T, double ratio, int32_t window)
{
    if (T < 0 || window < 0 || !ratio_ok(ratio)) return -1;
    return (int32_t)host_num_keep_quota(T, ratio, window);
}

mkv_status mkv_select_quota(const float *S, mkv_shape shape, double ratio, int32_t window, int32_t keep_stride,
                            int32_t *idx, int32_t *kept, void *workspace, size_t workspace_bytes,
                            mkv_stream_t stream)
{
    mkv_status rc = check_shape(shape);
    if (rc != MKV_OK) return rc;
    if (!S || !idx || !kept || !aligned(S, 4) || !aligned(idx, 4) || !aligned(kept, 4)) return MKV_ERR_INVALID_ARG;
    if (!ratio_ok(ratio) || window < 0 || keep_stride < host_num_keep_quota(shape.t_max, ratio, window))
        return MKV_ERR_INVALID_ARG;
    const Geometry g = geometry_of(shape, window);
    const Layout L = make_step_layout(g);
    if ((rc = check_ws(L, workspace, workspace_bytes)) != MKV_OK) return rc;
    if (empty(shape)) return MKV_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t *status = region<uint32_t>(workspace, L.status);
    return cuda_status(launch_select_quota(g, S, shape.seq_lens, ratio, keep_stride, kept, idx, keep_stride, status, st));
}

mkv_status mkv_compress_quota(const void *K, const void *V, mkv_shape shape, double ratio, mkv_mode mode,
                              int32_t window, int32_t keep_stride, void *K_out, void *V_out, int32_t *idx,
                              int32_t *kept, void *workspace, size_t workspace_bytes, mkv_stream_t stream)
{
    return run_compress(K, V, shape, ratio, nullptr, mode, window, keep_stride, K_out, V_out, idx, kept, workspace,
                        workspace_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr, false, true);
}

size_t mkv_oja_workspace_size(mkv_shape shape, int32_t n_query)
{
    if (check_shape(shape) != MKV_OK || shape.head_dim != kHeadDim || shape.dtype != MKV_DTYPE_BF16 || n_query < 16 ||
        n_query > 256 || n_query % 16)
        return 0;
    const Geometry g = geometry_of(shape, 0);
    return make_layout(g).total + round_up(oja_operand_bytes(g.n_heads, n_query), kAlign);
}

namespace {

// Checks shared by the OjaKV entry points; on success *g and *L describe the
// problem and the workspace.
mkv_status oja_checks(const void *K, const void *Q, const float *U, const mkv_shape &s, int32_t n_query, int32_t rank,
                      void *ws, size_t ws_bytes, Geometry *g, Layout *L)
{
    mkv_status rc = check_shape(s);
    if (rc != MKV_OK) return rc;
    // the contraction is built for 128 bf16 dims
    if (s.head_dim != kHeadDim || s.dtype != MKV_DTYPE_BF16) return MKV_ERR_UNSUPPORTED;
    if (!K || !Q || (rank > 0 && !U)) return MKV_ERR_INVALID_ARG;
    if (!aligned(K, 16) || !aligned(Q, 16) || (U && !aligned(U, 16))) return MKV_ERR_INVALID_ARG;
    if (n_query < 16 || n_query > 256 || n_query % 16 || rank < 0 || rank > kHeadDim) return MKV_ERR_INVALID_ARG;
    *g = geometry_of(s, 0);
    // TMA row coordinates are 32-bit
    if ((uint64_t)g->n_heads * (uint64_t)s.t_max >= (1ull << 31) ||
        (uint64_t)g->n_heads * 2u * (uint64_t)n_query >= (1ull << 31))
        return MKV_ERR_UNSUPPORTED;
    *L = make_layout(*g);
    if (!ws || !aligned(ws, kAlign) || ws_bytes < L->total + round_up(oja_operand_bytes(g->n_heads, n_query), kAlign))
        return MKV_ERR_WORKSPACE;
    return MKV_OK;
}

}  // namespace

mkv_status mkv_oja_score(const void *K, const void *Q, const float *U, mkv_shape shape, int32_t n_query, int32_t rank,
                         float *S, void *workspace, size_t workspace_bytes, mkv_stream_t stream)
{
    Geometry g;
    Layout L;
    mkv_status rc = oja_checks(K, Q, U, shape, n_query, rank, workspace, workspace_bytes, &g, &L);
    if (rc != MKV_OK) return rc;
    if (!S || !aligned(S, 4)) return MKV_ERR_INVALID_ARG;
    if (empty(shape)) return MKV_OK;
    return cuda_status(launch_oja_scores(g, K, Q, U, shape.seq_lens, n_query, rank, region<void>(workspace, L.total), S,
                                         region<uint32_t>(workspace, L.status), reinterpret_cast<cudaStream_t>(stream)));
}

mkv_status mkv_oja_score_profiled(const void *K, const void *Q, const float *U, mkv_shape shape, int32_t n_query,
                                  int32_t rank, float *S, void *workspace, size_t workspace_bytes, mkv_stream_t stream,
                                  void *const *events, int32_t n_events)
{
    if (!events || n_events < 3 || !events[0] || !events[1] || !events[2]) return MKV_ERR_INVALID_ARG;
    Geometry g;
    Layout L;
    mkv_status rc = oja_checks(K, Q, U, shape, n_query, rank, workspace, workspace_bytes, &g, &L);
    if (rc != MKV_OK) return rc;
    if (!S || !aligned(S, 4)) return MKV_ERR_INVALID_ARG;
    if (empty(shape)) return MKV_OK;
    return cuda_status(launch_oja_scores(g, K, Q, U, shape.seq_lens, n_query, rank, region<void>(workspace, L.total), S,
                                         region<uint32_t>(workspace, L.status), reinterpret_cast<cudaStream_t>(stream),
                                         events));
}

mkv_status mkv_compress_oja(const void *K, const void *V, const void *Q, const float *U, mkv_shape shape,
                            int32_t n_query, int32_t rank, double ratio, const int32_t *n_keep, int32_t keep_stride,
                            void *K_out, void *V_out, int32_t *idx, int32_t *kept, void *workspace,
                            size_t workspace_bytes, mkv_stream_t stream)
{
    Geometry g;
    Layout L;
    mkv_status rc = oja_checks(K, Q, U, shape, n_query, rank, workspace, workspace_bytes, &g, &L);
    if (rc != MKV_OK) return rc;
    if (!V) return MKV_ERR_INVALID_ARG;
    rc = check_outputs(shape, ratio, n_keep, keep_stride, K, V, K_out, V_out, idx, kept, false);
    if (rc != MKV_OK) return rc;
    if (empty(shape)) return MKV_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t *status = region<uint32_t>(workspace, L.status);
    float *S = region<float>(workspace, L.score);
    cudaError_t e = launch_oja_scores(g, K, Q, U, shape.seq_lens, n_query, rank, region<void>(workspace, L.total), S,
                                      status, st);
    if (e != cudaSuccess) return cuda_status(e);
    // the selection back end of mkv_compress on these scores
    int32_t *kept_w = kept ? kept : region<int32_t>(workspace, L.kept);
    int32_t *idx_w = idx ? idx : region<int32_t>(workspace, L.idx);
    const int32_t idx_stride = idx ? keep_stride : g.t_max;
    mkv_cut *cut = region<mkv_cut>(workspace, L.cut);
    int2 *chunk = region<int2>(workspace, L.chunk);
    const bool emit = select_emits_indices(g);
    if ((e = launch_select(g, S, shape.seq_lens, ratio, n_keep, keep_stride, cut, emit ? nullptr : chunk, kept_w,
                           emit ? idx_w : nullptr, idx_stride, status, st)) != cudaSuccess)
        return cuda_status(e);
    if (!emit &&
        (e = launch_compact(g, S, cut, chunk, shape.seq_lens, keep_stride, idx_w, idx_stride, status, st)) != cudaSuccess)
        return cuda_status(e);
    if (K_out && (e = launch_gather(g, idx_w, idx_stride, kept_w, keep_stride, K, V, K_out, V_out, status, st,
                                    emit && select_single_wave(g))) != cudaSuccess)
        return cuda_status(e);
    return MKV_OK;
}

mkv_status mkv_compress_inplace(void *K, void *V, mkv_shape shape, double ratio, const int32_t *n_keep, mkv_mode mode,
                                int32_t window, int32_t *idx, int32_t *kept, void *workspace, size_t workspace_bytes,
                                mkv_stream_t stream)
{
    // the kept rows land at the front of each head's own rows: the output
    // stride is t_max and the outputs are K and V themselves
    return run_compress(K, V, shape, ratio, n_keep, mode, window, shape.t_max, nullptr, nullptr, idx, kept, workspace,
                        workspace_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr, false, false, true);
}

int32_t mkv_compress_num_stages(void) { return kCompressStages; }

int32_t mkv_compress_single_pass(mkv_shape shape, int32_t window, mkv_mode mode)
{
    if (check_shape(shape) != MKV_OK || window < 0 || (mode != MKV_MODE_L2 && mode != MKV_MODE_COSINE)) return -1;
    const Geometry g = geometry_of(shape, window);
    if (g.d == kHeadDim && g.es == 2 && g_single_pass_enabled.load(std::memory_order_relaxed)) {
        const int grid = single_pass_grid((int)mode);
        if (grid <= 0) return -1;
        if (grid >= g.pg.ppw) return 1;
    }
    if (g_head_groups_enabled.load(std::memory_order_relaxed)) {
        const Layout L = make_layout(g);
        const FusedBudget fb = fused_budget(g);
        if (fb.scorers != 0 && fused_plan(g.pg, (int)mode, L.centroid - L.counters, fb.scorers, fb.selectors).grid > 0)
            return 3;
        const HeadGroupPlan hp = choose_head_groups(g.pg, (int)mode, L.centroid - L.counters);
        if (hp.groups > 0) return hp.ring ? 4 : 2;
    }
    return 0;
}

int32_t mkv_head_group_plan(mkv_shape shape, int32_t window, mkv_mode mode, int32_t *plan)
{
    if (!plan || check_shape(shape) != MKV_OK || window < 0 || (mode != MKV_MODE_L2 && mode != MKV_MODE_COSINE))
        return -1;
    const Geometry g = geometry_of(shape, window);
    const Layout L = make_layout(g);
    const HeadGroupPlan hp = choose_head_groups(g.pg, (int)mode, L.centroid - L.counters);
    plan[0] = hp.groups;
    plan[1] = hp.gsize;
    plan[2] = hp.wb;
    plan[3] = hp.ring ? 1 : 0;
    return hp.groups > 0 ? 0 : -1;
}

int32_t mkv_set_oja_pair(int32_t enable)
{
    return oja_set_pair(enable);
}

int32_t mkv_set_head_groups(int32_t enable)
{
    return g_head_groups_enabled.exchange(enable ? 1 : 0);
}

int32_t mkv_set_head_group_ring(int32_t enable)
{
    return g_head_group_ring.exchange(enable ? 1 : 0);
}

int32_t mkv_set_fused(int32_t scorer_ctas, int32_t select_ctas)
{
    if (select_ctas > 0) g_fused_selectors.store(select_ctas);
    return g_fused_scorers.exchange(scorer_ctas > 0 ? scorer_ctas : scorer_ctas < 0 ? -1 : 0);
}

mkv_status mkv_inject_stalled_windows(const void *K, const void *V, mkv_shape shape, double ratio, mkv_mode mode,
                                      int32_t window, int32_t keep_stride, void *K_out, void *V_out, int32_t *idx,
                                      int32_t *kept, void *workspace, size_t workspace_bytes, mkv_stream_t stream)
{
    return run_compress(K, V, shape, ratio, nullptr, mode, window, keep_stride, K_out, V_out, idx, kept, workspace,
                        workspace_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr, true);
}

mkv_status mkv_inject_stalled_fused(const void *K, const void *V, mkv_shape shape, double ratio, mkv_mode mode,
                                    int32_t keep_stride, void *K_out, void *V_out, int32_t *idx, int32_t *kept,
                                    int32_t stage, void *workspace, size_t workspace_bytes, mkv_stream_t stream)
{
    if (stage != 0 && stage != 1) return MKV_ERR_INVALID_ARG;
    if (!K_out || !V_out) return MKV_ERR_INVALID_ARG;
    return run_compress(K, V, shape, ratio, nullptr, mode, 0, keep_stride, K_out, V_out, idx, kept, workspace,
                        workspace_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr, false, false, false, true,
                        stage);
}

int32_t mkv_layer_budgets(const double *sensitivity, int32_t layers, double r, double gamma, int64_t total,
                          const int32_t *cap, int32_t *budget)
{
    if (!sensitivity || !cap || !budget || layers <= 0 || !(r > 0.0) || !(gamma >= 1.0) || total < 0) return -1;
    double smin = sensitivity[0], smax = sensitivity[0];
    int64_t capsum = 0;
    for (int32_t l = 0; l < layers; ++l) {
        if (sensitivity[l] != sensitivity[l] || cap[l] < 0) return -1;
        smin = fmin(smin, sensitivity[l]);
        smax = fmax(smax, sensitivity[l]);
        capsum += cap[l];
    }
    if (total >= capsum) {  // the caps absorb everything
        for (int32_t l = 0; l < layers; ++l) budget[l] = cap[l];
        return total == capsum ? 0 : 1;
    }
    std::vector<double> w(layers), x(layers);
    std::vector<char> full(layers, 0);
    for (int32_t l = 0; l < layers; ++l) {
        const double sn = smax > smin ? (sensitivity[l] - smin) / (smax - smin) : 0.0;
        w[l] = fmin(fmax(pow(r, sn), 1.0 / gamma), gamma);
    }
    // water-filling: budgets proportional to w, layers that reach their cap
    // are fixed there and the rest of the total is shared by the others
    for (;;) {
        double rest = (double)total, wsum = 0.0;
        for (int32_t l = 0; l < layers; ++l) {
            if (full[l]) rest -= cap[l];
            else wsum += w[l];
        }
        const double lambda = rest / wsum;
        bool grew = false;
        for (int32_t l = 0; l < layers; ++l)
            if (!full[l] && lambda * w[l] >= (double)cap[l]) full[l] = 1, grew = true;
        if (!grew) {
            for (int32_t l = 0; l < layers; ++l) x[l] = full[l] ? (double)cap[l] : lambda * w[l];
            break;
        }
    }
    // integers by largest remainder, lower layer first among equal remainders
    int64_t assigned = 0;
    for (int32_t l = 0; l < layers; ++l) {
        budget[l] = (int32_t)floor(x[l]);
        assigned += budget[l];
    }
    std::vector<int32_t> order(layers);
    for (int32_t l = 0; l < layers; ++l) order[l] = l;
    std::stable_sort(order.begin(), order.end(),
                     [&](int32_t a, int32_t b) { return x[a] - budget[a] > x[b] - budget[b]; });
    for (int32_t k = 0; k < layers && assigned < total; ++k) {
        const int32_t l = order[k];
        if (budget[l] < cap[l]) {
            ++budget[l];
            ++assigned;
        }
    }
    return 0;
}

int32_t mkv_set_single_pass(int32_t enable)
{
    return g_single_pass_enabled.exchange(enable ? 1 : 0);
}

mkv_status mkv_compress_profiled(const void *K, const void *V, mkv_shape shape, double ratio,
                                 const int32_t *n_keep, mkv_mode mode, int32_t window, int32_t keep_stride,
                                 void *K_out, void *V_out, int32_t *idx, int32_t *kept, void *workspace,
                                 size_t workspace_bytes, mkv_stream_t stream, void *const *events,
                                 int32_t n_events)
{
    if (!events || n_events < kCompressStages + 1) return MKV_ERR_INVALID_ARG;
    for (int i = 0; i <= kCompressStages; ++i)
        if (!events[i]) return MKV_ERR_INVALID_ARG;
    return run_compress(K, V, shape, ratio, n_keep, mode, window, keep_stride, K_out, V_out, idx, kept, workspace,
                        workspace_bytes, reinterpret_cast<cudaStream_t>(stream), events);
}

mkv_status mkv_compress_host(const void *hK, const void *hV, void *dK, void *dV, mkv_shape shape, double ratio,
                             mkv_mode mode, int32_t window, int32_t keep_stride, void *dK_out, void *dV_out,
                             int32_t *d_idx, int32_t *d_kept, void *hK_out, void *hV_out, int32_t *h_idx,
                             int32_t *h_kept, void *workspace, size_t workspace_bytes, mkv_stream_t stream)
{
    mkv_status rc = check_shape(shape);
    if (rc != MKV_OK) return rc;
    if (!hK || !hV || !dK || !dV || !dK_out || !dV_out || !d_idx || !d_kept) return MKV_ERR_INVALID_ARG;
    rc = check_outputs(shape, ratio, nullptr, keep_stride, dK, dV, dK_out, dV_out, d_idx, d_kept, true);
    if (rc != MKV_OK) return rc;
    if (window < 0 || (mode != MKV_MODE_L2 && mode != MKV_MODE_COSINE)) return MKV_ERR_INVALID_ARG;
    const Geometry g = geometry_of(shape, window);
    if ((rc = check_ws(make_layout(g), workspace, workspace_bytes)) != MKV_OK) return rc;
    if (empty(shape)) return MKV_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    CopyStreams *cs = copy_streams();
    if (!cs) return MKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(cs->mu);
    // rows of the batch per chunk: up to kHostChunks chunks
    const int32_t per = (shape.batch + kHostChunks - 1) / kHostChunks;
    const int32_t chunks = (shape.batch + per - 1) / per;
    const size_t row_bytes = (size_t)shape.head_dim * elem_bytes(shape.dtype);
    const size_t in_row = (size_t)shape.heads * shape.t_max * row_bytes;      // bytes of one batch row of K
    const size_t out_row = (size_t)shape.heads * keep_stride * row_bytes;     // of K_out
    const size_t idx_row = (size_t)shape.heads * keep_stride * sizeof(int32_t);
    const size_t kept_row = (size_t)shape.heads * sizeof(int32_t);
    auto bytes_at = [](const void *p, size_t off) { return static_cast<const uint8_t *>(p) + off; };
    auto wbytes_at = [](void *p, size_t off) { return static_cast<uint8_t *>(p) + off; };
    // Values are only read for the kept rows (the gather): when hV is pinned
    // host memory the device can address, the gather reads those rows
    // straight from it and only they cross the link; otherwise V is copied.
    const uint8_t *v_host_dev = nullptr;
    {
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, hV) == cudaSuccess && attr.type == cudaMemoryTypeHost &&
            attr.devicePointer != nullptr)
            v_host_dev = static_cast<const uint8_t *>(attr.devicePointer);
        else
            (void)cudaGetLastError();
    }
    // the copies wait for earlier work on the caller's stream (earlier users of the buffers)
    if (cudaEventRecord(cs->start, st) != cudaSuccess || cudaStreamWaitEvent(cs->in[0], cs->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(cs->in[1], cs->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(cs->out, cs->start, 0) != cudaSuccess)
        return MKV_ERR_CUDA;
    for (int32_t c = 0; c < chunks; ++c) {
        const int32_t r0 = c * per, rows = std::min(per, shape.batch - r0);
        const size_t ib = (size_t)rows * in_row, io = (size_t)r0 * in_row;
        if (cudaMemcpyAsync(wbytes_at(dK, io), bytes_at(hK, io), ib, cudaMemcpyHostToDevice, cs->in[0]) != cudaSuccess ||
            (!v_host_dev &&
             cudaMemcpyAsync(wbytes_at(dV, io), bytes_at(hV, io), ib, cudaMemcpyHostToDevice, cs->in[1]) != cudaSuccess) ||
            cudaEventRecord(cs->in_done[0][c], cs->in[0]) != cudaSuccess ||
            cudaEventRecord(cs->in_done[1][c], cs->in[1]) != cudaSuccess ||
            cudaStreamWaitEvent(st, cs->in_done[0][c], 0) != cudaSuccess ||
            cudaStreamWaitEvent(st, cs->in_done[1][c], 0) != cudaSuccess)
            return MKV_ERR_CUDA;
        mkv_shape sub = shape;
        sub.batch = rows;
        sub.seq_lens = shape.seq_lens ? shape.seq_lens + r0 : nullptr;
        const size_t oo = (size_t)r0 * out_row;
        int32_t *ci = reinterpret_cast<int32_t *>(wbytes_at(d_idx, (size_t)r0 * idx_row));
        int32_t *ck = reinterpret_cast<int32_t *>(wbytes_at(d_kept, (size_t)r0 * kept_row));
        const void *vsrc = v_host_dev ? static_cast<const void *>(v_host_dev + io) : bytes_at(dV, io);
        // the separate kernels: with the host link as the limit, the fused
        // kernel's overlap of scoring and gathering buys nothing here
        rc = run_compress(bytes_at(dK, io), vsrc, sub, ratio, nullptr, mode, window, keep_stride,
                          wbytes_at(dK_out, oo), wbytes_at(dV_out, oo), ci, ck, workspace, workspace_bytes, st, nullptr,
                          false, false, false, false);
        if (rc != MKV_OK) return rc;
        if (cudaEventRecord(cs->comp_done[c], st) != cudaSuccess || cudaStreamWaitEvent(cs->out, cs->comp_done[c], 0) != cudaSuccess)
            return MKV_ERR_CUDA;
        const size_t ob = (size_t)rows * out_row;
        if (hK_out && ob && cudaMemcpyAsync(wbytes_at(hK_out, oo), wbytes_at(dK_out, oo), ob, cudaMemcpyDeviceToHost, cs->out) != cudaSuccess)
            return MKV_ERR_CUDA;
        if (hV_out && ob && cudaMemcpyAsync(wbytes_at(hV_out, oo), wbytes_at(dV_out, oo), ob, cudaMemcpyDeviceToHost, cs->out) != cudaSuccess)
            return MKV_ERR_CUDA;
        if (h_idx && rows * idx_row &&
            cudaMemcpyAsync(wbytes_at(h_idx, (size_t)r0 * idx_row), ci, (size_t)rows * idx_row, cudaMemcpyDeviceToHost,
                            cs->out) != cudaSuccess)
            return MKV_ERR_CUDA;
        if (h_kept && cudaMemcpyAsync(wbytes_at(h_kept, (size_t)r0 * kept_row), ck, (size_t)rows * kept_row,
                                      cudaMemcpyDeviceToHost, cs->out) != cudaSuccess)
            return MKV_ERR_CUDA;
    }
    // the caller's stream resumes once every copy has landed
    if (cudaEventRecord(cs->out_done, cs->out) != cudaSuccess || cudaStreamWaitEvent(st, cs->out_done, 0) != cudaSuccess)
        return MKV_ERR_CUDA;
    for (int k = 0; k < 2; ++k)
        if (cudaEventRecord(cs->in_done[k][kHostChunks], cs->in[k]) != cudaSuccess ||
            cudaStreamWaitEvent(st, cs->in_done[k][kHostChunks], 0) != cudaSuccess)
            return MKV_ERR_CUDA;
    return MKV_OK;
}

mkv_status mkv_device_status(void *workspace, mkv_stream_t stream, uint32_t *bits)
{
    if (!workspace || !aligned(workspace, kAlign)) return MKV_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MKV_ERR_CUDA;
    if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return MKV_ERR_CUDA;
    if (word && cudaMemset(workspace, 0, sizeof word) != cudaSuccess) return MKV_ERR_CUDA;
    if (bits) *bits = word;
    return word ? MKV_ERR_DEVICE : MKV_OK;
}

const char *mkv_status_string(int32_t status)
{
    switch (status) {
    case MKV_OK: return "MKV_OK";
    case MKV_ERR_INVALID_ARG: return "MKV_ERR_INVALID_ARG: bad argument (null or misaligned pointer, size, ratio, window or stride)";
    case MKV_ERR_UNSUPPORTED:
        return "MKV_ERR_UNSUPPORTED: head_dim must be 64, 128 or 256, dtype bf16 or fp8 E4M3 (bf16 and 128 dims for "
               "the OjaKV scorer) and t_max at most 2^30";
    case MKV_ERR_WORKSPACE: return "MKV_ERR_WORKSPACE: workspace missing, misaligned or smaller than mkv_workspace_size";
    case MKV_ERR_CUDA: return "MKV_ERR_CUDA: a CUDA call or kernel launch failed";
    case MKV_ERR_DEVICE: return "MKV_ERR_DEVICE: a kernel reported bad device-side input (see the status bits)";
    default: return "unknown mkv_status";
    }
}

}  // extern "C"
