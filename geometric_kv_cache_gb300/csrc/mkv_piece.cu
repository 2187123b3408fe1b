// Centroid and score kernels (steps a1 and a2), and the opt-in kernel that
// runs the whole path in one launch (k_fused_path: the head groups' scoring
// followed, through per-head counters, by the select and gather device
// functions of mkv_select.cuh and mkv_gather.cuh).
//
// Method: "ManifoldKV: Training-Free KV Cache Compression via Euclidean
// Outlier Detection" (ICML 2026 poster 62526), abstract: every token is
// ranked by its distance to the key centroid (one global centroid, or one per
// window for WindowedManifoldKV); the KeyDiff-style cosine score is the
// baseline switch.
//
// Work units. A piece is at most g.piece_rows (64 * 2^k) consecutive tokens
// inside one window of one head; items = (head, window, piece), head-major,
// spread over a persistent grid. A CTA streams its piece with 16-byte
// non-coherent loads, kBatch rows per 8-lane group in flight (8 loads per
// thread), so every SM keeps ~100 KB of HBM reads outstanding.
//
// Fixed reduction order, the same in every kernel and for every grid size:
// lane q of the 8-lane group of row slot s (s = tid / 8, 32 slots) adds the
// rows s, s + 32, s + 64, ... of the piece in order; the 4 slots of a warp
// are combined by xor-shuffles (8 then 16); the 8 warps in warp order. A
// window's centroid is the sum over groups of 32 pieces (group order) of the
// group's piece sums (piece order), divided by the window's token count.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "mkv_device.cuh"
#include "mkv_internal.h"
#include "mkv_select.cuh"
#include "mkv_gather.cuh"

namespace mkv {
namespace {

using namespace dev;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowSlots = kThreads / 8;                   // 8 lanes per row

static_assert(kStageRows % kRowSlots == 0, "piece rows must be a multiple of the row slots");

struct Piece {
    int64_t head;
    int w;        // window index
    int p;        // piece index in the window
    int a;        // first token
    int len;      // tokens in this piece
    int wlen;     // tokens in the window
    int npieces;  // pieces in the window
};

// Position in a CTA's item sequence blockIdx.x, +gridDim.x, ...: items are
// (head, r) with r = window * ppw + piece. Stepping by the grid is done with
// precomputed quotient and remainder, and the head's length is re-read only
// when the head changes, so walking the sequence costs a few integer ops.
struct Walker {
    int64_t head;
    int r;
    int T;            // tokens of `head` (0 when done or empty)
    int64_t cached;   // head whose T is cached (-1 none)
};

struct Steps {
    int per_head;     // nwin_max * ppw
    int64_t head_step;
    int r_step;
};

__device__ __forceinline__ Steps make_steps(const PieceGeometry &g)
{
    Steps st;
    st.per_head = g.nwin_max * g.ppw;
    st.head_step = (int64_t)gridDim.x / st.per_head;
    st.r_step = (int)((int64_t)gridDim.x - st.head_step * st.per_head);
    return st;
}

__device__ __forceinline__ void walker_load_T(Walker &wk, const PieceGeometry &g, const int32_t *seq_lens,
                                              uint32_t *status)
{
    if (wk.head >= g.n_heads) {
        wk.T = 0;
    } else if (wk.head != wk.cached) {
        wk.T = head_len(seq_lens, wk.head, g.heads, g.t_max, status, threadIdx.x == 0);
        wk.cached = wk.head;
    }
}

__device__ __forceinline__ void walker_step(Walker &wk, const Steps &st)
{
    wk.r += st.r_step;
    wk.head += st.head_step;
    if (wk.r >= st.per_head) {
        wk.r -= st.per_head;
        ++wk.head;
    }
}

// Decode the walker's current item; false if it holds no token.
__device__ __forceinline__ bool decode_piece(const Walker &wk, const PieceGeometry &g, Piece &pc)
{
    pc.head = wk.head;
    pc.w = wk.r / g.ppw;
    pc.p = wk.r - pc.w * g.ppw;
    if (wk.T == 0) return false;
    const int wl = window_len(wk.T, g.window);
    const int64_t wstart = (int64_t)pc.w * wl;
    if (wstart >= wk.T) return false;
    pc.wlen = (int)min((int64_t)wl, (int64_t)wk.T - wstart);
    const int off = pc.p * g.piece_rows;
    if (off >= pc.wlen) return false;
    pc.a = (int)wstart + off;
    pc.len = min(g.piece_rows, pc.wlen - off);
    pc.npieces = (pc.wlen + g.piece_rows - 1) / g.piece_rows;
    return true;
}

// Move to the first non-empty item at or after the walker (head >= n_heads
// when none is left).
__device__ __forceinline__ void walker_settle(Walker &wk, const Steps &st, const PieceGeometry &g,
                                              const int32_t *seq_lens, uint32_t *status, Piece &pc)
{
    for (;;) {
        walker_load_T(wk, g, seq_lens, status);
        if (wk.head >= g.n_heads) return;
        if (decode_piece(wk, g, pc)) return;
        walker_step(wk, st);
    }
}

__device__ __forceinline__ Walker first_walker(const PieceGeometry &g, const Steps &st)
{
    Walker wk;
    wk.head = (int64_t)blockIdx.x / st.per_head;
    wk.r = (int)((int64_t)blockIdx.x - wk.head * st.per_head);
    wk.T = 0;
    wk.cached = -1;
    return wk;
}

// A CTA's stream of non-empty items.
struct Cursor {
    Walker wk;
    Piece pc;  // the current item (valid while !done)
    bool done;
};

__device__ __forceinline__ Cursor first_cursor(const PieceGeometry &g, const Steps &st, const int32_t *seq_lens,
                                               uint32_t *status)
{
    Cursor c;
    c.wk = first_walker(g, st);
    walker_settle(c.wk, st, g, seq_lens, status, c.pc);
    c.done = c.wk.head >= g.n_heads;
    return c;
}

__device__ __forceinline__ void advance(Cursor &c, const Steps &st, const PieceGeometry &g, const int32_t *seq_lens,
                                        uint32_t *status)
{
    walker_step(c.wk, st);
    walker_settle(c.wk, st, g, seq_lens, status, c.pc);
    c.done = c.wk.head >= g.n_heads;
}

// Item index of the cursor's current piece (for per-piece records).
__device__ __forceinline__ int64_t cursor_item(const Cursor &c, const Steps &st)
{
    return c.wk.head * st.per_head + c.wk.r;
}

// ------------------------------------------------------------ arithmetic --

// Head dims. A row of D = 64 * NB bf16 values is read by the 8 lanes of its
// row group; lane q owns NB blocks of 8 dims, [64k + 8q, 64k + 8q + 8) for
// k < NB, the 16 bytes at byte offset 128k + 16q of the row. Its per-thread
// arrays hold 8 * NB values in that order (block k at [8k, 8k + 8)).

// Combine the per-thread accumulators into the piece sum, written to out[]
// (D floats) by threads 0..D-1. `red` is [kWarps][D] shared scratch; the
// caller synchronises before `red` is reused.
template <int NB = 2>
__device__ __forceinline__ void finish_sum(float acc[8 * NB], float *red, float *out)
{
    constexpr int D = 64 * NB;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, q = threadIdx.x & 7;
#pragma unroll
    for (int j = 0; j < 8 * NB; ++j) {
        acc[j] += __shfl_xor_sync(kFull, acc[j], 8);
        acc[j] += __shfl_xor_sync(kFull, acc[j], 16);
    }
    if (lane < 8) {
#pragma unroll
        for (int k = 0; k < NB; ++k)
#pragma unroll
            for (int j = 0; j < 8; ++j) red[warp * D + 64 * k + q * 8 + j] = acc[8 * k + j];
    }
    __syncthreads();
    if (threadIdx.x < D) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[w * D + threadIdx.x];
        out[threadIdx.x] = s;
    }
}

// Score of one row from the thread's 16 dims f, centroid dims c and the
// centroid norm nc (cosine only). Reduces over the row's 8 lanes, so all 32
// lanes of the warp must call it.
template <int MODE, int NB = 2>
__device__ __forceinline__ float score_of(const float f[8 * NB], const float c[8 * NB], float nc)
{
    if (MODE == MKV_MODE_L2) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 8 * NB; ++j) {
            const float d = f[j] - c[j];
            acc = fmaf(d, d, acc);
        }
        acc += __shfl_xor_sync(kFull, acc, 4);
        acc += __shfl_xor_sync(kFull, acc, 2);
        acc += __shfl_xor_sync(kFull, acc, 1);
        return __fsqrt_rn(acc);
    } else {
        float dot = 0.f, kk = 0.f;
#pragma unroll
        for (int j = 0; j < 8 * NB; ++j) {
            dot = fmaf(f[j], c[j], dot);
            kk = fmaf(f[j], f[j], kk);
        }
        dot += __shfl_xor_sync(kFull, dot, 4);
        kk += __shfl_xor_sync(kFull, kk, 4);
        dot += __shfl_xor_sync(kFull, dot, 2);
        kk += __shfl_xor_sync(kFull, kk, 2);
        dot += __shfl_xor_sync(kFull, dot, 1);
        kk += __shfl_xor_sync(kFull, kk, 1);
        const float den = __fmul_rn(__fsqrt_rn(kk), nc);
        return den == 0.f ? 1.f : __fsub_rn(1.f, __fdiv_rn(dot, den));
    }
}

// Centroid norm for cosine (all 32 lanes call it).
template <int NB = 2>
__device__ __forceinline__ float centroid_norm(const float c[8 * NB])
{
    float cc = 0.f;
#pragma unroll
    for (int j = 0; j < 8 * NB; ++j) cc = fmaf(c[j], c[j], cc);
    cc += __shfl_xor_sync(kFull, cc, 4);
    cc += __shfl_xor_sync(kFull, cc, 2);
    cc += __shfl_xor_sync(kFull, cc, 1);
    return __fsqrt_rn(cc);
}

// The thread's 8 * NB centroid dims from cw (L2 reads: another CTA may have
// written them during this kernel).
template <int NB = 2>
__device__ __forceinline__ void load_centroid(const float *cw, float c[8 * NB])
{
    const int q = threadIdx.x & 7;
#pragma unroll
    for (int k = 0; k < NB; ++k) {
        const float4 a = __ldcg(reinterpret_cast<const float4 *>(cw + 64 * k + q * 8));
        const float4 b = __ldcg(reinterpret_cast<const float4 *>(cw + 64 * k + q * 8 + 4));
        c[8 * k + 0] = a.x; c[8 * k + 1] = a.y; c[8 * k + 2] = a.z; c[8 * k + 3] = a.w;
        c[8 * k + 4] = b.x; c[8 * k + 5] = b.y; c[8 * k + 6] = b.z; c[8 * k + 7] = b.w;
    }
}

// The thread's 8 * NB dims of a row from its NB chunks (ES: element bytes).
template <int NB = 2, int ES = 2>
__device__ __forceinline__ void row_to_f32(const typename Chunk<ES>::raw *v, float f[8 * NB])
{
#pragma unroll
    for (int k = 0; k < NB; ++k) Chunk<ES>::to_f32(v[k], f + 8 * k);
}

// acc += the thread's 8 * NB dims of a row (fp32 adds in dim order).
template <int NB, int ES>
__device__ __forceinline__ void row_accumulate(const typename Chunk<ES>::raw *v, float acc[8 * NB])
{
#pragma unroll
    for (int k = 0; k < NB; ++k) Chunk<ES>::add_to(v[k], acc + 8 * k);
}

// score_of on a row still in its cache encoding. L2 subtracts the centroid
// straight from the encoded elements (the same roundings as widening first).
template <int MODE, int NB, int ES>
__device__ __forceinline__ float score_row(const typename Chunk<ES>::raw *v, const float c[8 * NB], float nc)
{
    if (MODE == MKV_MODE_L2) {
        float d[8 * NB];
#pragma unroll
        for (int k = 0; k < NB; ++k) Chunk<ES>::sub_from(v[k], c + 8 * k, d + 8 * k);
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 8 * NB; ++j) acc = fmaf(d[j], d[j], acc);
        acc += __shfl_xor_sync(kFull, acc, 4);
        acc += __shfl_xor_sync(kFull, acc, 2);
        acc += __shfl_xor_sync(kFull, acc, 1);
        return __fsqrt_rn(acc);
    } else {
        float f[8 * NB];
        row_to_f32<NB, ES>(v, f);
        return score_of<MODE, NB>(f, c, nc);
    }
}

// Sum of n (<= kGroupPieces) consecutive D-float records, record order,
// dim d; loads issued in batches of 8 ahead of their adds.
template <int D = 128>
__device__ __forceinline__ float ordered_sum(const float *first, int n, int d)
{
    float s = 0.f;
    for (int j0 = 0; j0 < n; j0 += 8) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = j0 + j < n ? __ldcg(first + (int64_t)(j0 + j) * D + d) : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j0 + j < n) s += v[j];
    }
    return s;
}

struct Pointers {
    const uint8_t *K;
    const int32_t *seq_lens;
    float *partial;  // [heads, nwin_max, ppw, 128]
    float *C;        // [heads, nwin_max, 128]
    float *S;        // [heads, t_max]
    uint32_t *status;
};

// ------------------------------------------------------------- kernels --

// Rows r = slot + 32 * (i0 + u), u < N, of a piece starting at `base`
// (this thread's NB chunks of 8 elements of ES bytes each, elements 64k + 8q;
// chunk k of row u at v[NB u + k]), loaded before use.
template <int N, int NB = 2, int ES = 2>
__device__ __forceinline__ void load_rows(const uint8_t *base, int len, int i0, typename Chunk<ES>::raw v[NB * N])
{
    const int slot = threadIdx.x >> 3, q = threadIdx.x & 7;
#pragma unroll
    for (int u = 0; u < N; ++u) {
        const int r = slot + (i0 + u) * kRowSlots;
        const uint8_t *row = base + (size_t)(r < len ? r : 0) * (64 * NB * ES);
#pragma unroll
        for (int k = 0; k < NB; ++k) v[NB * u + k] = Chunk<ES>::load(row + (64 * k + 8 * q) * ES);
    }
}

// Rows in flight per lane in the streaming kernels: 128 bytes per lane for
// every head dim and element type (8 / NB rows of bf16, 16 / NB of E4M3), at
// most 8 rows (a 256-token piece gives each row slot 8 rows).
template <int NB, int ES = 2>
__host__ __device__ constexpr int batch_rows() { return 16 / (NB * ES) < 8 ? 16 / (NB * ES) : 8; }

// a1, first half: piece sums. The first batch of the next piece is loaded
// before the current piece's CTA reduction, so the loads stay in flight
// across piece boundaries.
template <int NB, int ES>
__global__ void __launch_bounds__(kThreads, NB > 2 ? 2 : 3)
k_piece_sums(PieceGeometry g, Pointers P)
{
    constexpr int D = 64 * NB, RB = ES * D, B = batch_rows<NB, ES>();
    using Raw = typename Chunk<ES>::raw;
    __shared__ float red[kWarps * D];
    const Steps st = make_steps(g);
    const int slot = threadIdx.x >> 3;
    Cursor cur = first_cursor(g, st, P.seq_lens, P.status);
    Raw v[NB * B];
    if (!cur.done) load_rows<B, NB, ES>(P.K + ((size_t)cur.pc.head * g.t_max + cur.pc.a) * RB, cur.pc.len, 0, v);
    while (!cur.done) {
        const Piece pc = cur.pc;
        const int64_t item = cursor_item(cur, st);
        const uint8_t *base = P.K + ((size_t)pc.head * g.t_max + pc.a) * RB;
        const int nrows = (pc.len + kRowSlots - 1) / kRowSlots;  // rows per slot (upper bound)
        float acc[8 * NB];
#pragma unroll
        for (int j = 0; j < 8 * NB; ++j) acc[j] = 0.f;
        for (int i0 = 0; i0 < nrows; i0 += B) {
#pragma unroll
            for (int u = 0; u < B; ++u) {
                if (slot + (i0 + u) * kRowSlots < pc.len) row_accumulate<NB, ES>(v + NB * u, acc);
            }
            if (i0 + B < nrows) load_rows<B, NB, ES>(base, pc.len, i0 + B, v);
        }
        advance(cur, st, g, P.seq_lens, P.status);
        if (!cur.done) load_rows<B, NB, ES>(P.K + ((size_t)cur.pc.head * g.t_max + cur.pc.a) * RB, cur.pc.len, 0, v);
        finish_sum<NB>(acc, red, P.partial + item * D);
        __syncthreads();  // red is free again
    }
}

// a1, second half: window means. One D-thread CTA per (head, window),
// thread d for dim d: the groups of 32 piece sums in piece order, then the
// groups in group order, divided by the window's token count (the same order
// as the single-pass and head-group kernels).
template <int D>
__global__ void __launch_bounds__(D)
k_window_means(PieceGeometry g, Pointers P)
{
    const int64_t win = blockIdx.x;
    const int64_t head = win / g.nwin_max;
    const int w = (int)(win - head * g.nwin_max);
    const int T = head_len(P.seq_lens, head, g.heads, g.t_max, P.status, false);
    if (T == 0) return;
    const int wl = window_len(T, g.window);
    const int64_t wstart = (int64_t)w * wl;
    if (wstart >= T) return;
    const int wlen = (int)min((int64_t)wl, (int64_t)T - wstart);
    const int np = (wlen + g.piece_rows - 1) / g.piece_rows;
    const int ng = (np + kGroupPieces - 1) / kGroupPieces;
    const float *pw = P.partial + win * (int64_t)g.ppw * D;
    float tot = 0.f;
    for (int gi = 0; gi < ng; ++gi)
        tot += ordered_sum<D>(pw + (int64_t)gi * kGroupPieces * D, min(kGroupPieces, np - gi * kGroupPieces),
                              threadIdx.x);
    P.C[win * D + threadIdx.x] = __fdiv_rn(tot, (float)wlen);
}

// a2: scores of every piece against its window's mean in C. As in
// k_piece_sums, the next piece's first batch is loaded as soon as the current
// piece's last batch is consumed, before the next centroid is read.
template <int MODE, int NB, int ES>
__global__ void __launch_bounds__(kThreads, NB > 2 ? 2 : 3)
k_piece_scores(PieceGeometry g, Pointers P)
{
    constexpr int D = 64 * NB, RB = ES * D, B = batch_rows<NB, ES>();
    using Raw = typename Chunk<ES>::raw;
    const Steps st = make_steps(g);
    const int slot = threadIdx.x >> 3, q = threadIdx.x & 7;
    Cursor cur = first_cursor(g, st, P.seq_lens, P.status);
    Raw v[NB * B];
    if (!cur.done) load_rows<B, NB, ES>(P.K + ((size_t)cur.pc.head * g.t_max + cur.pc.a) * RB, cur.pc.len, 0, v);
    while (!cur.done) {
        const Piece pc = cur.pc;
        const uint8_t *base = P.K + ((size_t)pc.head * g.t_max + pc.a) * RB;
        float *srow = P.S + (size_t)pc.head * g.t_max + pc.a;
        float c[8 * NB];
        load_centroid<NB>(P.C + (pc.head * g.nwin_max + pc.w) * D, c);
        const float nc = MODE == MKV_MODE_COSINE ? centroid_norm<NB>(c) : 0.f;
        const int nrows = (pc.len + kRowSlots - 1) / kRowSlots;
        for (int i0 = 0; i0 < nrows; i0 += B) {
#pragma unroll
            for (int u = 0; u < B; ++u) {
                const int r = slot + (i0 + u) * kRowSlots;
                const float s = score_row<MODE, NB, ES>(v + NB * u, c, nc);
                if (r < pc.len && q == 0) srow[r] = s;
            }
            if (i0 + B < nrows) load_rows<B, NB, ES>(base, pc.len, i0 + B, v);
        }
        // the next piece's first batch goes out before its centroid is read
        advance(cur, st, g, P.seq_lens, P.status);
        if (!cur.done) load_rows<B, NB, ES>(P.K + ((size_t)cur.pc.head * g.t_max + cur.pc.a) * RB, cur.pc.len, 0, v);
    }
}

// ------------------------------------------------- single-pass kernel --
//
// One read of K from HBM for both a1 and a2, with three warp roles:
//  * a producer warp streams the CTA's pieces into a ring of kRing 16 KB
//    shared-memory slots with bulk asynchronous copies (cp.async.bulk,
//    completion on a "full" mbarrier per slot; the slot is refilled once its
//    "empty" mbarrier has seen all 8 compute warps), so HBM reads stay in
//    flight whatever the compute warps are doing;
//  * 8 compute warps add each piece's rows up from shared memory (phase 1)
//    and hand the per-warp sums to the sync warp; kLag pieces later they
//    re-read that older piece's rows with 16-byte loads -- normally L2 hits,
//    the rows were copied in a few microseconds earlier -- and score them
//    against the window mean (phase 2);
//  * a sync warp does all waiting on other CTAs: it publishes each piece sum
//    (global record, release fence, arrival counter; the last arrival of a
//    group of 32 pieces adds the group, the last group adds the window,
//    divides, and raises the window's ready flag) and copies the window mean
//    of each phase-2 piece into shared memory once that flag is up.
// Hand-overs between roles go through double-buffered shared memory guarded
// by mbarriers. The arithmetic is exactly that of k_piece_sums,
// k_window_means and k_piece_scores, so both paths give the same bits.
//
// Progress: the kernel is launched cooperatively (all CTAs resident). A
// window spans at most kMaxPiecesPerWindow consecutive items and every CTA
// takes one item per round, so a window's pieces lie in at most two
// consecutive rounds; the sync warp fetches the mean of round t - kLag
// before publishing round t (or after, when phase 2 has caught up with the
// CTA's own latest piece), so every wait depends only on earlier rounds. All
// waits are still bounded by a timer: running out sets MKV_DEV_TIMEOUT, makes
// every later wait give up at once, and leaves the affected scores unwritten.

constexpr int kLag = 2;
constexpr int kBatch2 = 4;  // phase-2 rows per lane in flight (L2 hits)
constexpr int kRing = 4;
constexpr uint32_t kStageBytes = kStageRows * kRowBytes;  // 16 KB
constexpr int kFusedThreads = kThreads + 64;              // + producer warp + sync warp
constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s bound on every wait

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ bool timed_out(const uint32_t *status)
{
    return (ld_acquire(status) & MKV_DEV_TIMEOUT) != 0u;
}

// Wait (bounded) for completion `parity` of `bar`; on its own timeout it flags
// MKV_DEV_TIMEOUT. An abortable wait (a hand-over between warps of this CTA)
// also gives up at once when some other wait already timed out. Waits on the
// ring's copy barriers are not abortable: a bulk copy always lands, and no
// slot may be reused or abandoned while its copy is in flight.
__device__ __forceinline__ void mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *status, bool abortable = true)
{
    const uint32_t b = smem_addr(bar);
    const uint64_t t0 = global_ns();
    for (uint32_t spin = 0;; ++spin) {
        uint32_t done;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
            : "=r"(done)
            : "r"(b), "r"(parity)
            : "memory");
        if (done) return;
        if ((spin & 63u) == 63u) {
            if (abortable && timed_out(status)) return;
            if (global_ns() - t0 > kWaitNs) {
                atomicOr(status, MKV_DEV_TIMEOUT);
                return;
            }
        }
    }
}

// One thread: expect `bytes` on `bar` and start the copy global -> shared.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Compute warps only (the producer and sync warps never join).
__device__ __forceinline__ void compute_barrier()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}

struct FusedPointers {
    Pointers P;
    float *gsum;    // [heads, nwin_max, ngroups_max, 128]
    uint32_t *cnt;  // [heads, nwin_max, ngroups_max + 2]: group counters, window counter, ready flag
};

struct FusedShared {
    uint8_t ring[kRing][kStageBytes];
    float red[2][kWarps * kHeadDim];
    float cbuf[2][kHeadDim];
    uint64_t full[kRing], empty[kRing];
    uint64_t redfull[2], redempty[2], cfull[2], cempty[2];
};

// Sum of n (<= kGroupPieces) consecutive 128-float records, record order,
// for the four dims 4*lane .. 4*lane + 3 (loads in batches of 4).
__device__ __forceinline__ float4 ordered_sum4(const float *first, int n, int lane)
{
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < n; j0 += 4) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            v[j] = j0 + j < n ? __ldcg(reinterpret_cast<const float4 *>(first + (int64_t)(j0 + j) * kHeadDim) + lane)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (j0 + j < n) {
                s.x += v[j].x;
                s.y += v[j].y;
                s.z += v[j].z;
                s.w += v[j].w;
            }
    }
    return s;
}

// Sync warp: publish piece `pc` (item `item`) from red[b].
__device__ __forceinline__ void publish(const Piece &pc, int64_t item, const PieceGeometry &g, const FusedPointers &F,
                                        FusedShared &sh, int b, uint32_t use)
{
    const int lane = threadIdx.x & 31;
    mbar_wait(&sh.redfull[b], use & 1u, F.P.status);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const float4 r = reinterpret_cast<const float4 *>(sh.red[b] + w * kHeadDim)[lane];
        s.x += r.x;
        s.y += r.y;
        s.z += r.z;
        s.w += r.w;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.redempty[b]);
    const int64_t win = pc.head * g.nwin_max + pc.w;
    float *pw = F.P.partial + win * (int64_t)g.ppw * kHeadDim;
    reinterpret_cast<float4 *>(F.P.partial + item * kHeadDim)[lane] = s;
    __threadfence();
    __syncwarp();
    uint32_t *cnt = F.cnt + win * (g.ngroups_max + 2);
    const int ng = (pc.npieces + kGroupPieces - 1) / kGroupPieces;
    const int gi = pc.p / kGroupPieces;
    const int gsize = min(kGroupPieces, pc.npieces - gi * kGroupPieces);
    uint32_t old = 0;
    if (lane == 0) old = atomicAdd(&cnt[gi], 1u);
    old = __shfl_sync(kFull, old, 0);
    if (old != (uint32_t)(gsize - 1)) return;
    // last piece of its group: the group's sum
    __threadfence();
    float *gw = F.gsum + win * (int64_t)g.ngroups_max * kHeadDim;
    const float4 gs = ordered_sum4(pw + (int64_t)gi * kGroupPieces * kHeadDim, gsize, lane);
    reinterpret_cast<float4 *>(gw + (int64_t)gi * kHeadDim)[lane] = gs;
    __threadfence();
    __syncwarp();
    if (lane == 0) old = atomicAdd(&cnt[g.ngroups_max], 1u);
    old = __shfl_sync(kFull, old, 0);
    if (old != (uint32_t)(ng - 1)) return;
    // last group of its window: the window mean, then the ready flag
    __threadfence();
    const float4 t = ordered_sum4(gw, ng, lane);
    const float n = (float)pc.wlen;
    reinterpret_cast<float4 *>(F.P.C + win * kHeadDim)[lane] =
        make_float4(__fdiv_rn(t.x, n), __fdiv_rn(t.y, n), __fdiv_rn(t.z, n), __fdiv_rn(t.w, n));
    __threadfence();
    __syncwarp();
    if (lane == 0) atomicExch(&cnt[g.ngroups_max + 1], 1u);
}

// Sync warp: wait for the window of `pc`, copy its mean into cbuf[b].
__device__ __forceinline__ void fetch_mean(const Piece &pc, const PieceGeometry &g, const FusedPointers &F,
                                           FusedShared &sh, int b, uint32_t use)
{
    const int lane = threadIdx.x & 31;
    if (use > 0) mbar_wait(&sh.cempty[b], (use - 1) & 1u, F.P.status);
    const int64_t win = pc.head * g.nwin_max + pc.w;
    const uint32_t *ready = F.cnt + win * (g.ngroups_max + 2) + g.ngroups_max + 1;
    if (lane == 0) {
        const uint64_t t0 = global_ns();
        while (ld_acquire(ready) == 0u) {
            if (timed_out(F.P.status)) break;
            if (global_ns() - t0 > kWaitNs) {
                atomicOr(F.P.status, MKV_DEV_TIMEOUT);
                break;
            }
            __nanosleep(64);
        }
    }
    __syncwarp();
    (void)ld_acquire(ready);  // order this lane's reads of the mean after the flag
    reinterpret_cast<float4 *>(sh.cbuf[b])[lane] = __ldcg(reinterpret_cast<const float4 *>(F.P.C + win * kHeadDim) + lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.cfull[b]);
}

// Round structure shared by all roles: in round t the compute warps do
// phase 1 of the CTA's t-th piece (while any is left) and then phase 2 of the
// (t - kLag)-th (or, once phase 1 is exhausted, of the next pending one).
template <int MODE>
__global__ void __launch_bounds__(kFusedThreads, 2)
k_single_pass(PieceGeometry g, FusedPointers F)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    FusedShared &sh = *reinterpret_cast<FusedShared *>(smem_raw);
    const Pointers &P = F.P;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], kWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.redfull[b], 1);
            mbar_init(&sh.redempty[b], 1);
            mbar_init(&sh.cfull[b], 1);
            mbar_init(&sh.cempty[b], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const Steps st = make_steps(g);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == kWarps) {
        // ---- producer: the phase-1 stages of every piece, in order
        Cursor c = first_cursor(g, st, P.seq_lens, P.status);
        uint32_t seq = 0;
        for (; !c.done; advance(c, st, g, P.seq_lens, P.status)) {
            for (int r0 = 0; r0 < c.pc.len; r0 += kStageRows, ++seq) {
                const int s = (int)(seq % kRing);
                if (seq >= kRing) mbar_wait(&sh.empty[s], ((seq / kRing) - 1) & 1u, P.status, false);
                if (lane == 0) {
                    const int rows = min(kStageRows, c.pc.len - r0);
                    bulk_load(sh.ring[s], P.K + ((size_t)c.pc.head * g.t_max + c.pc.a + r0) * kRowBytes,
                              (uint32_t)rows * kRowBytes, &sh.full[s]);
                }
                __syncwarp();
            }
        }
        // stay resident until the copies still in flight have landed
        for (uint32_t k = seq > kRing ? seq - kRing : 0; k < seq; ++k)
            mbar_wait(&sh.full[k % kRing], (k / kRing) & 1u, P.status, false);
        return;
    }

    Cursor c1 = first_cursor(g, st, P.seq_lens, P.status);  // phase-1 stream
    Cursor c2 = c1;                                          // phase-2 stream, kLag behind
    uint32_t u1 = 0, u2 = 0;                                 // pieces through phase 1 / phase 2
    uint32_t seq = 0;                                        // ring stages consumed
    const int slot = threadIdx.x >> 3, q = threadIdx.x & 7;
    for (int t = 0; !c1.done || !c2.done; ++t) {
        const bool do1 = !c1.done;
        Piece p1;
        int64_t item1 = 0;
        if (do1) {
            p1 = c1.pc;
            item1 = cursor_item(c1, st);
            advance(c1, st, g, P.seq_lens, P.status);
        }
        const bool do2 = !c2.done && (t >= kLag || c1.done);
        Piece p2;
        if (do2) p2 = c2.pc;
        if (warp == kWarps + 1) {
            // ---- sync warp. Normally the fetch for the older piece goes
            // first (its window is complete by now). When phase 2 reaches this
            // round's own piece, that piece must be published first.
            if (do1 && do2 && u2 == u1) {
                publish(p1, item1, g, F, sh, (int)(u1 & 1u), u1 >> 1);
                fetch_mean(p2, g, F, sh, (int)(u2 & 1u), u2 >> 1);
            } else {
                if (do2) fetch_mean(p2, g, F, sh, (int)(u2 & 1u), u2 >> 1);
                if (do1) publish(p1, item1, g, F, sh, (int)(u1 & 1u), u1 >> 1);
            }
        } else {
            if (do1) {
                // ---- phase 1: the piece sum from the ring (k_piece_sums order)
                float acc[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] = 0.f;
                for (int r0 = 0; r0 < p1.len; r0 += kStageRows, ++seq) {
                    const int s = (int)(seq % kRing);
                    mbar_wait(&sh.full[s], (seq / kRing) & 1u, P.status, false);
                    const int rows = min(kStageRows, p1.len - r0);
#pragma unroll
                    for (int i = 0; i < kStageRows / kRowSlots; ++i) {
                        const int r = slot + i * kRowSlots;
                        if (r < rows) {
                            const uint8_t *row = sh.ring[s] + r * kRowBytes;
                            float f[16];
                            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(row + q * 16), f);
                            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(row + 128 + q * 16), f + 8);
#pragma unroll
                            for (int j = 0; j < 16; ++j) acc[j] += f[j];
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.empty[s]);
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    acc[j] += __shfl_xor_sync(kFull, acc[j], 8);
                    acc[j] += __shfl_xor_sync(kFull, acc[j], 16);
                }
                const int b = (int)(u1 & 1u);
                if (u1 >= 2) mbar_wait(&sh.redempty[b], ((u1 >> 1) - 1) & 1u, P.status);
                if (lane < 8) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        sh.red[b][warp * kHeadDim + q * 8 + j] = acc[j];
                        sh.red[b][warp * kHeadDim + 64 + q * 8 + j] = acc[8 + j];
                    }
                }
                compute_barrier();
                if (threadIdx.x == 0) mbar_arrive(&sh.redfull[b]);
            }
            if (do2) {
                // ---- phase 2: scores of the older piece against its window mean
                const int b = (int)(u2 & 1u);
                mbar_wait(&sh.cfull[b], (u2 >> 1) & 1u, P.status);
                float c[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    c[j] = sh.cbuf[b][q * 8 + j];
                    c[8 + j] = sh.cbuf[b][64 + q * 8 + j];
                }
                compute_barrier();
                if (threadIdx.x == 0) mbar_arrive(&sh.cempty[b]);
                const float nc = MODE == MKV_MODE_COSINE ? centroid_norm(c) : 0.f;
                if (!timed_out(P.status)) {
                    const uint8_t *base = P.K + ((size_t)p2.head * g.t_max + p2.a) * kRowBytes;
                    float *srow = P.S + (size_t)p2.head * g.t_max + p2.a;
                    const int nrows = (p2.len + kRowSlots - 1) / kRowSlots;
                    for (int i0 = 0; i0 < nrows; i0 += kBatch2) {
                        uint4 v[2 * kBatch2];
                        load_rows<kBatch2>(base, p2.len, i0, v);
#pragma unroll
                        for (int u = 0; u < kBatch2; ++u) {
                            const int r = slot + (i0 + u) * kRowSlots;
                            float f[16];
                            bf16x8_to_f32(v[2 * u], f);
                            bf16x8_to_f32(v[2 * u + 1], f + 8);
                            const float sc = score_of<MODE>(f, c, nc);
                            if (r < p2.len && q == 0) srow[r] = sc;
                        }
                    }
                }
            }
        }
        if (do1) ++u1;
        if (do2) {
            ++u2;
            advance(c2, st, g, P.seq_lens, P.status);
        }
    }
}

// ------------------------------------------------------ head groups --

// Non-coherent load of one chunk (16 bytes of bf16, 8 of E4M3) carrying an
// L2 eviction policy (createpolicy).
template <int ES>
__device__ __forceinline__ typename Chunk<ES>::raw ld_policy(const void *p, uint64_t pol);

template <>
__device__ __forceinline__ uint4 ld_policy<2>(const void *p, uint64_t pol)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p), "l"(pol));
    return r;
}

template <>
__device__ __forceinline__ uint2 ld_policy<1>(const void *p, uint64_t pol)
{
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
        : "=r"(r.x), "=r"(r.y)
        : "l"(p), "l"(pol));
    return r;
}

// load_rows with an L2 eviction policy on every load.
template <int N, int NB, int ES>
__device__ __forceinline__ void load_rows_policy(const uint8_t *base, int len, int i0,
                                                 typename Chunk<ES>::raw v[NB * N], uint64_t pol)
{
    const int slot = threadIdx.x >> 3, q = threadIdx.x & 7;
#pragma unroll
    for (int u = 0; u < N; ++u) {
        const int r = slot + (i0 + u) * kRowSlots;
        const uint8_t *row = base + (size_t)(r < len ? r : 0) * (64 * NB * ES);
#pragma unroll
        for (int k = 0; k < NB; ++k) v[NB * u + k] = ld_policy<ES>(row + (64 * k + 8 * q) * ES, pol);
    }
}
//
// One read of K from HBM for a1 + a2: a group of `gsize` CTAs shares a
// unit -- a block of `wb` consecutive windows of one head (a global
// centroid is one window: the unit is the whole head). Pass 1: each CTA sums
// its piece slots f = rank, rank + gsize, ... (exactly the arithmetic of
// k_piece_sums) and writes the piece sums; the group then meets at a barrier
// (an arrival counter in global memory, polled with a time bound). Each CTA
// forms the unit's window means from all piece sums (exactly k_window_means'
// order) and, in pass 2, re-reads its own pieces and scores them (exactly
// k_piece_scores). Only one unit per group is in flight, so the host picks
// the group count and unit size such that their keys fit in L2 and pass 2
// reads L2, not HBM. The CTAs of one group do the same number of rounds; the kernel is
// launched cooperatively (all CTAs resident), so every arrival comes.
// Pass 1 loads carry an L2 evict-last policy and pass 2 loads evict-first,
// so the rows of the heads in flight stay in L2 until their second read
// (measured: 0.30 ms against 0.33 ms for the three kernels on 256 heads of
// 16K tokens; without the policies pass 2 missed L2 on about a third of its
// rows). Same bits as the three-kernel path.
// Dynamic shared memory of k_head_groups: the pass-1 stash of per-warp piece
// sums, then (same bytes) the unit's means; padded so that at most two CTAs
// share an SM (the grid is then spread over all SMs). A unit holds at most
// kMaxUnitWindows windows.
// Pieces of its own sequence a head-group CTA prefetches into L2 ahead of
// its pass-1 loads (bulk L2 prefetches issued by one thread; the sequence runs
// on into the CTA's next unit, so the prefetches keep HBM busy while the CTA
// waits at the group barrier, forms the means and re-reads the unit from L2).
#ifndef MKV_HG_PREFETCH
#define MKV_HG_PREFETCH 0
#endif
constexpr int kHgPrefetch = MKV_HG_PREFETCH;
// Share of L2 (percent) the head groups' units in flight may take.
#ifndef MKV_HG_L2_BUDGET_PCT
#define MKV_HG_L2_BUDGET_PCT 60
#endif
#ifndef MKV_RING_L2_BUDGET_PCT
#define MKV_RING_L2_BUDGET_PCT 60
#endif
constexpr size_t kGroupSmem = 80 * 1024;
// CTAs per SM of the stand-alone head-group kernel: 2 (kGroupSmem of shared
// memory, 16 / NB rows per lane in flight) or 3 (kGroupSmem3, 8 / NB rows).
#ifndef MKV_HG_CTAS
#define MKV_HG_CTAS 2
#endif
constexpr size_t kGroupSmem3 = 64 * 1024;
constexpr size_t kHgSmem = MKV_HG_CTAS >= 3 ? kGroupSmem3 : kGroupSmem;
constexpr int kMaxUnitWindows = 64;
constexpr int kMaxDim = 256;
static_assert(kMaxUnitWindows * kMaxDim * sizeof(float) <= kGroupSmem3, "means must fit");
// pieces the stash holds for head dim D
__host__ __device__ constexpr int stash_slots(int D) { return (int)(kGroupSmem / sizeof(float)) / (kWarps * D); }
constexpr int kMaxSlots = stash_slots(64);

// L2 prefetch of `bytes` (a multiple of 16) at `p` (16-byte aligned) with a
// cache policy; asynchronous, completes on its own.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes, uint64_t pol)
{
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p), "r"(bytes), "l"(pol)
                 : "memory");
}

// The piece slots f = rank, rank + gsize, ... of a unit that a CTA of rank
// `rank` takes, and their count (slots past the unit's windows excluded).
struct UnitPieces {
    int64_t head;
    int T, wl, w0, nf;
};
__device__ __forceinline__ UnitPieces unit_pieces(const PieceGeometry &g, const Pointers &P, int64_t unit, int wb)
{
    const int upw = (g.nwin_max + wb - 1) / wb;
    UnitPieces u;
    u.head = unit / upw;
    u.w0 = (int)(unit - u.head * upw) * wb;
    u.T = head_len(P.seq_lens, u.head, g.heads, g.t_max, P.status, false);
    u.wl = window_len(u.T, g.window);
    const int nw = u.T > 0 ? (u.T + u.wl - 1) / u.wl : 0;
    u.nf = max(0, min(u.w0 + wb, nw) - u.w0) * g.ppw;
    return u;
}

// Prefetch the piece `ahead` places after slot number i (0-based, the CTA's
// i-th slot of `unit`) in the CTA's sequence of slots, which runs on into
// its later units; nothing when the sequence ends first or the slot lies
// past its window's last piece.
template <int RB>
__device__ __forceinline__ void prefetch_ahead(const PieceGeometry &g, const Pointers &P, int64_t unit, int i,
                                               int ahead, int rank, int gsize, int groups, int wb, int64_t n_units,
                                               uint64_t pol)
{
    int j = i + ahead;
    for (int64_t u = unit; u < n_units; u += groups) {
        const UnitPieces up = unit_pieces(g, P, u, wb);
        const int n = up.nf > rank ? (up.nf - rank - 1) / gsize + 1 : 0;
        if (j < n) {
            const int f = rank + j * gsize;
            const int w = up.w0 + f / g.ppw, p = f - (f / g.ppw) * g.ppw;
            const int wstart = w * up.wl, wlen = min(up.wl, up.T - wstart), off = p * g.piece_rows;
            if (off < wlen)
                prefetch_l2(P.K + ((size_t)up.head * g.t_max + wstart + off) * RB,
                            (uint32_t)min(g.piece_rows, wlen - off) * RB, pol);
            return;
        }
        j -= n;
    }
}

//
// head_groups_run is one CTA's share (group `group` of `groups`, rank `rank`
// in it). With head_done, every CTA of the group adds 1 to head_done[head]
// once the unit's scores it wrote are visible GPU-wide (units are whole heads
// there: a group's count reaches gsize when the head's scores are complete).
//
// A group barrier that runs out (or, with `abortable`, finds that another
// wait of the launch has run out) skips the unit's means and scores, and its
// CTA does not count the head in head_done: a head's count then never
// reaches gsize, so nothing downstream reads its scores. `barrier_extra`
// raises this group's barrier target above its CTA count (failure
// injection: 0 in every ordinary launch).
template <int MODE, int NB, int ES, int BATCH = 16 / NB, size_t SMEM = kGroupSmem>
__device__ __forceinline__ void head_groups_run(const PieceGeometry &g, const Pointers &P, uint32_t *gcnt, int gsize,
                                                int wb, uint32_t stagger_ns, int groups, int group, int rank,
                                                uint32_t *head_done, bool abortable = false,
                                                uint32_t barrier_extra = 0)
{
    constexpr int D = 64 * NB, RB = ES * D;
    using Raw = typename Chunk<ES>::raw;
    constexpr int kBatchG = BATCH;  // rows per lane in flight (16 / NB: 256 bytes per lane for every head dim)
    constexpr int kSlots = (int)(SMEM / sizeof(float)) / (kWarps * D);
    extern __shared__ float dyn[];    // pass 1: stash [kSlots][kWarps][D]; pass 2: means [wb][D]
    float *stash = dyn;
    float *cmean = dyn;
    __shared__ uint32_t s_ok;
    __shared__ int64_t s_off[kMaxSlots];  // partial-sum offset of each stashed piece
    // Every group does the same work per round, so groups that start
    // together stay in phase: all read HBM (pass 1) at once, then all read L2
    // (pass 2). Starting groups (group mod 4) stagger steps late spreads the
    // phases (measured on 256 heads x 16K: 0.313 -> 0.298 ms).
    if (stagger_ns) {
        const uint64_t t0 = global_ns(), wait = (uint64_t)(group & 3) * stagger_ns;
        while (global_ns() - t0 < wait) {
        }
    }
    const int slot = threadIdx.x >> 3, q = threadIdx.x & 7, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // the stash's piece sums: warps in order (finish_sum's order), then free
    auto flush = [&](int ns) {
        __syncthreads();
        for (int e = threadIdx.x; e < ns * D; e += kThreads) {
            const int j = e / D, d = e - j * D;
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) sum += stash[(j * kWarps + w) * D + d];
            P.partial[s_off[j] + d] = sum;
        }
        __threadfence();  // the piece sums are visible GPU-wide before the arrival
        __syncthreads();
    };
    uint64_t keep_l2, drop_l2;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep_l2));
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(drop_l2));
    const int upw = (g.nwin_max + wb - 1) / wb;  // units (blocks of wb windows) per head
    const int64_t n_units = g.n_heads * upw;
    uint32_t round = 0;
    for (int64_t unit = group; unit < n_units; unit += groups, ++round) {
        // the select may start launching once every CTA is on its last unit
        if (unit + groups >= n_units) pdl_trigger();
        const int64_t head = unit / upw;
        const int w0 = (int)(unit - head * upw) * wb;
        const int T = head_len(P.seq_lens, head, g.heads, g.t_max, P.status, threadIdx.x == 0 && rank == 0 && w0 == 0);
        const int wl = window_len(T, g.window);
        const int nw = T > 0 ? (T + wl - 1) / wl : 0;
        const int nwu = max(0, min(w0 + wb, nw) - w0);  // windows of this unit that exist
        const int nf = nwu * g.ppw;                      // piece slots of the unit
        // pass 1: piece sums; piece slot f is window w0 + f / ppw, piece f % ppw.
        // Each warp combines its 4 row slots by shuffles (as finish_sum does)
        // and stashes the result; the CTA adds the warps once per kSlots
        // pieces, so warps only meet at a CTA barrier there.
        int ns = 0;
        if (kHgPrefetch > 0 && threadIdx.x == 0 && round == 0)  // the CTA's first slots
            for (int a = 0; a < kHgPrefetch; ++a)
                prefetch_ahead<RB>(g, P, unit, 0, a, rank, gsize, groups, wb, n_units, keep_l2);
        for (int f = rank, i = 0; f < nf; f += gsize, ++i) {
            if (kHgPrefetch > 0 && threadIdx.x == 0)
                prefetch_ahead<RB>(g, P, unit, i, kHgPrefetch, rank, gsize, groups, wb, n_units, keep_l2);
            const int w = w0 + f / g.ppw, p = f - (f / g.ppw) * g.ppw;
            const int wstart = w * wl, wlen = min(wl, T - wstart), off = p * g.piece_rows;
            if (off >= wlen) continue;  // past the window's last piece (the same for every thread)
            const int len = min(g.piece_rows, wlen - off);
            const uint8_t *base = P.K + ((size_t)head * g.t_max + wstart + off) * RB;
            const int nrows = (len + kRowSlots - 1) / kRowSlots;
            float acc[8 * NB];
#pragma unroll
            for (int j = 0; j < 8 * NB; ++j) acc[j] = 0.f;
            for (int i0 = 0; i0 < nrows; i0 += kBatchG) {
                Raw v[NB * kBatchG];
                load_rows_policy<kBatchG, NB, ES>(base, len, i0, v, keep_l2);
#pragma unroll
                for (int u = 0; u < kBatchG; ++u) {
                    if (slot + (i0 + u) * kRowSlots < len) row_accumulate<NB, ES>(v + NB * u, acc);
                }
            }
#pragma unroll
            for (int j = 0; j < 8 * NB; ++j) {
                acc[j] += __shfl_xor_sync(kFull, acc[j], 8);
                acc[j] += __shfl_xor_sync(kFull, acc[j], 16);
            }
            if (lane < 8) {
#pragma unroll
                for (int k = 0; k < NB; ++k)
#pragma unroll
                    for (int j = 0; j < 8; ++j) stash[(ns * kWarps + warp) * D + 64 * k + q * 8 + j] = acc[8 * k + j];
            }
            if (threadIdx.x == 0) s_off[ns] = ((head * g.nwin_max + w) * (int64_t)g.ppw + p) * D;
            if (++ns == kSlots) {
                flush(ns);
                ns = 0;
            }
        }
        if (ns > 0) flush(ns);
        // the group's barrier for this unit
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(&gcnt[group], 1u);
            const uint32_t target = (round + 1) * (uint32_t)gsize + barrier_extra;
            const uint64_t t0 = global_ns();
            uint32_t ok = 1;
            for (uint32_t spin = 0; ld_acquire(&gcnt[group]) < target; ++spin) {
                if ((spin & 63u) == 63u) {
                    if (abortable && timed_out(P.status)) {
                        ok = 0;
                        break;
                    }
                    if (global_ns() - t0 > kWaitNs) {
                        atomicOr(P.status, MKV_DEV_TIMEOUT);
                        ok = 0;
                        break;
                    }
                }
            }
            s_ok = ok;
        }
        __syncthreads();
        if (s_ok && nwu > 0) {  // the same for every thread
            // window means in k_window_means' order (pieces of a group of 32
            // in order, then the groups), a group's loads in flight at once;
            // threads t, t + D, ... take successive windows
            for (int j = threadIdx.x / D; j < nwu; j += kThreads / D) {
                const int d = threadIdx.x % D;
                const int w = w0 + j;
                const int wlen = min(wl, T - w * wl);
                const int np = (wlen + g.piece_rows - 1) / g.piece_rows;
                const int ng = (np + kGroupPieces - 1) / kGroupPieces;
                const float *pw = P.partial + (head * g.nwin_max + w) * (int64_t)g.ppw * D + d;
                float tot = 0.f;
                for (int gi = 0; gi < ng; ++gi) {
                    const int n = min(kGroupPieces, np - gi * kGroupPieces);
                    float v[kGroupPieces];
#pragma unroll
                    for (int k = 0; k < kGroupPieces; ++k)
                        v[k] = k < n ? __ldcg(pw + (int64_t)(gi * kGroupPieces + k) * D) : 0.f;
                    float gs = 0.f;
#pragma unroll
                    for (int k = 0; k < kGroupPieces; ++k)
                        if (k < n) gs += v[k];
                    tot += gs;
                }
                const float m = __fdiv_rn(tot, (float)wlen);
                cmean[j * D + d] = m;
                if (rank == 0) P.C[(head * g.nwin_max + w) * D + d] = m;
            }
            __syncthreads();
            // pass 2: scores of the same pieces (their rows are L2 hits)
            for (int f = rank; f < nf; f += gsize) {
                const int jw = f / g.ppw, w = w0 + jw, p = f - jw * g.ppw;
                const int wstart = w * wl, wlen = min(wl, T - wstart), off = p * g.piece_rows;
                if (off >= wlen) continue;
                const int len = min(g.piece_rows, wlen - off);
                float c[8 * NB];
#pragma unroll
                for (int k = 0; k < NB; ++k)
#pragma unroll
                    for (int j = 0; j < 8; ++j) c[8 * k + j] = cmean[jw * D + 64 * k + q * 8 + j];
                const float nc = MODE == MKV_MODE_COSINE ? centroid_norm<NB>(c) : 0.f;
                const uint8_t *base = P.K + ((size_t)head * g.t_max + wstart + off) * RB;
                float *srow = P.S + (size_t)head * g.t_max + wstart + off;
                const int nrows = (len + kRowSlots - 1) / kRowSlots;
                for (int i0 = 0; i0 < nrows; i0 += kBatchG) {
                    Raw v[NB * kBatchG];
                    load_rows_policy<kBatchG, NB, ES>(base, len, i0, v, drop_l2);
#pragma unroll
                    for (int u = 0; u < kBatchG; ++u) {
                        const int r = slot + (i0 + u) * kRowSlots;
                        const float sc = score_row<MODE, NB, ES>(v + NB * u, c, nc);
                        if (r < len && q == 0) srow[r] = sc;
                    }
                }
            }
        }
        if (head_done && s_ok) {  // this CTA's scores of the unit are visible before the count
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();  // the publishing thread's own fence: the count releases the CTA's writes
                atomicAdd(&head_done[head], 1u);
            }
        }
        __syncthreads();  // the means are rewritten for the next unit
    }
}

template <int MODE, int NB, int ES>
__global__ void __launch_bounds__(kThreads, MKV_HG_CTAS)
k_head_groups(PieceGeometry g, Pointers P, uint32_t *gcnt, int gsize, int wb, uint32_t stagger_ns)
{
    const int groups = gridDim.x / gsize;
    const int group = blockIdx.x / gsize, rank = blockIdx.x - group * gsize;
    if (group >= groups) return;  // a launch is always a whole number of groups
    head_groups_run<MODE, NB, ES, (MKV_HG_CTAS >= 3 ? 8 : 16) / NB, kHgSmem>(g, P, gcnt, gsize, wb, stagger_ns, groups,
                                                                            group, rank, nullptr);
}

// ------------------------------------------- head groups with a copy ring --
//
// k_head_groups_ring: the head-group kernel (same units, groups, barrier,
// means and pass 2, hence the same bits), with pass 1 fed by a producer warp
// instead of the consumer warps' own loads. The producer streams the CTA's
// pass-1 rows, piece by piece and unit after unit, into a ring of
// kRingStages stages of kRingStageBytes with bulk asynchronous copies
// (cp.async.bulk, an L2 evict-last hint so the rows stay for pass 2; a
// "full" mbarrier per stage completes when its bytes land, an "empty" one
// when all 8 consumer warps have added its rows up). It does not wait for
// the group barrier, so while the consumers sit at the barrier, form the
// means and re-read the unit from L2 in pass 2, the ring already fills with
// the next unit's rows: HBM reads stay in flight through the whole round.
// Consumers read their rows from shared memory with the row-slot mapping of
// the register kernel (lane q of slot s adds rows s, s + 32, ... in order),
// so every sum has the same order.
constexpr int kRingStages = 3;
constexpr uint32_t kRingStageBytes = 32 * 1024;
constexpr int kRingWarps = kWarps + 1;                   // 8 consumer warps + the producer warp
constexpr int kRingThreads = kRingWarps * 32;
constexpr size_t kRingStash = 16 * 1024;                 // per-warp piece sums; then the unit's means
constexpr size_t kRingSmem = kRingStages * kRingStageBytes + kRingStash + 2 * kRingStages * sizeof(uint64_t);
// windows a unit may hold: their means must fit the stash buffer
__host__ __device__ constexpr int ring_unit_windows(int D) { return (int)(kRingStash / (sizeof(float) * D)); }

// One thread: expect `bytes` on `bar` and start the copy global -> shared
// with an L2 cache policy.
__device__ __forceinline__ void bulk_load_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

// The 256 consumer threads only (the producer warp never joins).
__device__ __forceinline__ void consumer_barrier()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}

// Two CTAs per SM: 18 warps spread over the four SM sub-partitions put five
// warps of 9 on some, so a thread may hold at most 96 registers.
template <int MODE, int NB>
__global__ void __launch_bounds__(kRingThreads, 2)
k_head_groups_ring(PieceGeometry g, Pointers P, uint32_t *gcnt, int gsize, int wb, uint32_t stagger_ns)
{
    constexpr int D = 64 * NB, RB = 2 * D;  // bf16 rows
    constexpr int SR = (int)(kRingStageBytes / RB);        // rows per stage
    constexpr int kSlots = (int)(kRingStash / (sizeof(float) * kWarps * D));
    constexpr int kBatchG = 8 / NB;                       // pass-2 rows per lane in flight (96 registers)
    static_assert(SR % kRowSlots == 0, "a stage must hold whole rounds of row slots");
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    float *stash = reinterpret_cast<float *>(smem + kRingStages * kRingStageBytes);
    float *cmean = stash;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kRingStages * kRingStageBytes + kRingStash);
    uint64_t *empty = full + kRingStages;
    __shared__ uint32_t s_ok;
    __shared__ int64_t s_off[kSlots];
    const int groups = gridDim.x / gsize;
    const int group = blockIdx.x / gsize, rank = blockIdx.x - group * gsize;
    if (group >= groups) return;  // a launch is always a whole number of groups
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRingStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (stagger_ns) {  // as in the register kernel: groups start (group mod 4) steps apart
        const uint64_t t0 = global_ns(), wait = (uint64_t)(group & 3) * stagger_ns;
        while (global_ns() - t0 < wait) {
        }
    }
    const int upw = (g.nwin_max + wb - 1) / wb;  // units (blocks of wb windows) per head
    const int64_t n_units = g.n_heads * upw;

    if (warp == kWarps) {
        // ---- producer: every pass-1 stage of the CTA's pieces, unit after unit
        if (lane == 0) {
            uint64_t keep_l2;
            asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep_l2));
            uint32_t seq = 0;
            for (int64_t unit = group; unit < n_units; unit += groups) {
                const int64_t head = unit / upw;
                const int w0 = (int)(unit - head * upw) * wb;
                const int T = head_len(P.seq_lens, head, g.heads, g.t_max, P.status, false);
                const int wl = window_len(T, g.window);
                const int nw = T > 0 ? (T + wl - 1) / wl : 0;
                const int nf = max(0, min(w0 + wb, nw) - w0) * g.ppw;
                for (int f = rank; f < nf; f += gsize) {
                    const int w = w0 + f / g.ppw, p = f - (f / g.ppw) * g.ppw;
                    const int wstart = w * wl, wlen = min(wl, T - wstart), off = p * g.piece_rows;
                    if (off >= wlen) continue;
                    const int len = min(g.piece_rows, wlen - off);
                    const uint8_t *base = P.K + ((size_t)head * g.t_max + wstart + off) * RB;
                    for (int r0 = 0; r0 < len; r0 += SR, ++seq) {
                        const int st = (int)(seq % kRingStages);
                        if (seq >= (uint32_t)kRingStages)
                            mbar_wait(&empty[st], ((seq / kRingStages) - 1) & 1u, P.status, false);
                        bulk_load_hint(ring + (size_t)st * kRingStageBytes, base + (size_t)r0 * RB,
                                       (uint32_t)min(SR, len - r0) * RB, &full[st], keep_l2);
                    }
                }
            }
            // stay until the copies still in flight have landed (they normally
            // have: the consumers wait for every stage)
            for (uint32_t k = seq > (uint32_t)kRingStages ? seq - kRingStages : 0; k < seq; ++k)
                mbar_wait(&full[k % kRingStages], (k / kRingStages) & 1u, P.status, false);
        }
        return;
    }

    // ---- consumers: threads 0..255
    const int slot = threadIdx.x >> 3, q = threadIdx.x & 7;
    auto flush = [&](int ns) {  // the stash's piece sums: warps in order, then free
        consumer_barrier();
        for (int e = threadIdx.x; e < ns * D; e += kThreads) {
            const int j = e / D, d = e - j * D;
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) sum += stash[(j * kWarps + w) * D + d];
            P.partial[s_off[j] + d] = sum;
        }
        __threadfence();  // the piece sums are visible GPU-wide before the arrival
        consumer_barrier();
    };
    uint64_t drop_l2;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(drop_l2));
    uint32_t round = 0, seq = 0;
    for (int64_t unit = group; unit < n_units; unit += groups, ++round) {
        if (unit + groups >= n_units) pdl_trigger();
        const int64_t head = unit / upw;
        const int w0 = (int)(unit - head * upw) * wb;
        const int T = head_len(P.seq_lens, head, g.heads, g.t_max, P.status, threadIdx.x == 0 && rank == 0 && w0 == 0);
        const int wl = window_len(T, g.window);
        const int nw = T > 0 ? (T + wl - 1) / wl : 0;
        const int nwu = max(0, min(w0 + wb, nw) - w0);
        const int nf = nwu * g.ppw;
        // pass 1: piece sums from the ring
        int ns = 0;
        for (int f = rank; f < nf; f += gsize) {
            const int w = w0 + f / g.ppw, p = f - (f / g.ppw) * g.ppw;
            const int wstart = w * wl, wlen = min(wl, T - wstart), off = p * g.piece_rows;
            if (off >= wlen) continue;
            const int len = min(g.piece_rows, wlen - off);
            float acc[8 * NB];
#pragma unroll
            for (int j = 0; j < 8 * NB; ++j) acc[j] = 0.f;
            for (int r0 = 0; r0 < len; r0 += SR, ++seq) {
                const int st = (int)(seq % kRingStages);
                mbar_wait(&full[st], (seq / kRingStages) & 1u, P.status, false);
                const int rows = min(SR, len - r0);
                const uint8_t *stage = ring + (size_t)st * kRingStageBytes;
#pragma unroll
                for (int i = 0; i < SR / kRowSlots; ++i) {
                    const int r = slot + i * kRowSlots;
                    if (r < rows) {
                        uint4 v[NB];
#pragma unroll
                        for (int k = 0; k < NB; ++k)
                            v[k] = *reinterpret_cast<const uint4 *>(stage + (size_t)r * RB + 128 * k + 16 * q);
                        row_accumulate<NB, 2>(v, acc);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
#pragma unroll
            for (int j = 0; j < 8 * NB; ++j) {
                acc[j] += __shfl_xor_sync(kFull, acc[j], 8);
                acc[j] += __shfl_xor_sync(kFull, acc[j], 16);
            }
            if (lane < 8) {
#pragma unroll
                for (int k = 0; k < NB; ++k)
#pragma unroll
                    for (int j = 0; j < 8; ++j) stash[(ns * kWarps + warp) * D + 64 * k + q * 8 + j] = acc[8 * k + j];
            }
            if (threadIdx.x == 0) s_off[ns] = ((head * g.nwin_max + w) * (int64_t)g.ppw + p) * D;
            if (++ns == kSlots) {
                flush(ns);
                ns = 0;
            }
        }
        if (ns > 0) flush(ns);
        // the group's barrier for this unit
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(&gcnt[group], 1u);
            const uint32_t target = (round + 1) * (uint32_t)gsize;
            const uint64_t t0 = global_ns();
            uint32_t ok = 1;
            for (uint32_t spin = 0; ld_acquire(&gcnt[group]) < target; ++spin) {
                if ((spin & 63u) == 63u && global_ns() - t0 > kWaitNs) {
                    atomicOr(P.status, MKV_DEV_TIMEOUT);
                    ok = 0;
                    break;
                }
            }
            s_ok = ok;
        }
        consumer_barrier();
        if (s_ok && nwu > 0) {  // the same for every consumer thread
            // window means in k_window_means' order (the register kernel's code)
            for (int j = threadIdx.x / D; j < nwu; j += kThreads / D) {
                const int d = threadIdx.x % D;
                const int w = w0 + j;
                const int wlen = min(wl, T - w * wl);
                const int np = (wlen + g.piece_rows - 1) / g.piece_rows;
                const int ng = (np + kGroupPieces - 1) / kGroupPieces;
                const float *pw = P.partial + (head * g.nwin_max + w) * (int64_t)g.ppw * D + d;
                float tot = 0.f;
                for (int gi = 0; gi < ng; ++gi) {
                    const int n = min(kGroupPieces, np - gi * kGroupPieces);
                    float v[kGroupPieces];
#pragma unroll
                    for (int k = 0; k < kGroupPieces; ++k)
                        v[k] = k < n ? __ldcg(pw + (int64_t)(gi * kGroupPieces + k) * D) : 0.f;
                    float gs = 0.f;
#pragma unroll
                    for (int k = 0; k < kGroupPieces; ++k)
                        if (k < n) gs += v[k];
                    tot += gs;
                }
                const float m = __fdiv_rn(tot, (float)wlen);
                cmean[j * D + d] = m;
                if (rank == 0) P.C[(head * g.nwin_max + w) * D + d] = m;
            }
            consumer_barrier();
            // pass 2: scores of the same pieces (their rows are L2 hits)
            for (int f = rank; f < nf; f += gsize) {
                const int jw = f / g.ppw, w = w0 + jw, p = f - jw * g.ppw;
                const int wstart = w * wl, wlen = min(wl, T - wstart), off = p * g.piece_rows;
                if (off >= wlen) continue;
                const int len = min(g.piece_rows, wlen - off);
                float c[8 * NB];
#pragma unroll
                for (int k = 0; k < NB; ++k)
#pragma unroll
                    for (int j = 0; j < 8; ++j) c[8 * k + j] = cmean[jw * D + 64 * k + q * 8 + j];
                const float nc = MODE == MKV_MODE_COSINE ? centroid_norm<NB>(c) : 0.f;
                const uint8_t *base = P.K + ((size_t)head * g.t_max + wstart + off) * RB;
                float *srow = P.S + (size_t)head * g.t_max + wstart + off;
                const int nrows = (len + kRowSlots - 1) / kRowSlots;
                for (int i0 = 0; i0 < nrows; i0 += kBatchG) {
                    uint4 v[NB * kBatchG];
                    load_rows_policy<kBatchG, NB, 2>(base, len, i0, v, drop_l2);
#pragma unroll
                    for (int u = 0; u < kBatchG; ++u) {
                        const int r = slot + (i0 + u) * kRowSlots;
                        const float sc = score_row<MODE, NB, 2>(v + NB * u, c, nc);
                        if (r < len && q == 0) srow[r] = sc;
                    }
                }
            }
        }
        consumer_barrier();  // the means are rewritten for the next unit
    }
}

// The whole path in one cooperative launch (global centroids, heads of at
// most kFusedMaxT tokens), in three roles:
//  * scorers, CTAs [0, groups * gsize): the heads' centroids and scores as
//    head groups compute them (units are whole heads; head_done[h] reaches
//    gsize when the scores of head h are complete);
//  * selectors, the last select_ctas CTAs (after their scoring, if they are
//    also scorers): the heads' selects in head order from one ticket
//    counter, each waiting for its head's scores and publishing sel_done[h];
//  * gatherers, every warp of every CTA once its other roles are done: gather
//    items of one warp each (16 output slots for rows of 256 bytes, 8 rows of
//    K and of V in flight per lane) from a second ticket counter, head-major,
//    each waiting for sel_done of its head. A warp claims its next item while
//    it copies the current one and meets no other warp, so many independent
//    item chains per SM hide each other's latency.
// Scorers wait only on their own group, selectors only on scorers, gatherers
// only on selectors, so with every CTA resident each wait ends; each is also
// bounded in time (a wait that runs out sets MKV_DEV_TIMEOUT and its work is
// skipped: the head keeps no rows). The arithmetic is that of the head-group,
// select and gather kernels, so the outputs are the same bits.
constexpr int kFusedMaxT = (int)(kGroupSmem / sizeof(float));  // the select keeps a head's scores in shared memory
// output slots of a warp's gather item: 8 rows of K and 8 of V in flight per
// lane (16 slots for 256-byte rows)
__host__ __device__ constexpr int fused_gather_rows(int row_bytes) { return 8 * 32 * 16 / row_bytes; }

struct TailArgs {
    const uint8_t *V;
    uint8_t *K_out, *V_out;
    const int32_t *n_keep;
    int32_t *kept, *idx;
    uint32_t *head_done, *sel_done, *sel_ticket, *gather_ticket;
    double ratio;
    int keep_stride, idx_stride, bph, select_ctas;
    // failure injection (-1 in every ordinary launch): the scorer group whose
    // barrier target is one above its CTA count, and the head whose select
    // waits for one scorer more than the group has
    int stall_group;
    int64_t stall_head;
};

// One thread waits until *flag >= target (bounded); 1 when it got there. With
// `abortable` it also gives up once any wait of the launch has timed out, so
// that a failure drains in about one wait bound (a timeout bit already set
// when the CTA started is not taken for one of this launch).
__device__ __forceinline__ uint32_t wait_count(const uint32_t *flag, uint32_t target, uint32_t *status, bool abortable)
{
    const uint64_t t0 = global_ns();
    for (uint32_t spin = 0; ld_acquire(flag) < target; ++spin) {
        if ((spin & 63u) == 63u) {
            if (abortable && timed_out(status)) return 0u;
            if (global_ns() - t0 > kWaitNs) {
                atomicOr(status, MKV_DEV_TIMEOUT);
                return 0u;
            }
            __nanosleep(256);
        }
    }
    return 1u;
}

// One warp's item of ROWS output slots (groups of LPR lanes per row, ROWS /
// (32 / LPR) rows of K and of V in flight per lane), for indices and kept
// counts written earlier in the same launch: both are read through L2 only
// (__ldcg), the indices at once with the count (only slots below both
// keep_stride and idx_stride, so every load stays inside the head's index
// row) and then masked by it. No barrier: warps run independent items.
// Whether the fused kernel's gathers load and store with an L2 evict-first
// policy (their rows are not read again in the launch, while the scorers'
// units must stay in L2 between their two passes).
#ifndef MKV_FUSED_GATHER_EVICT_FIRST
#define MKV_FUSED_GATHER_EVICT_FIRST 1
#endif

// 16-byte store carrying an L2 cache policy.
__device__ __forceinline__ void st_policy(void *p, uint4 v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w), "l"(pol)
                 : "memory");
}

template <int LPR, int ROWS>
__device__ __forceinline__ void gather_warp_item(int64_t head, int item, const int32_t *idx, int idx_stride,
                                                 const int32_t *kept, int t_max, int keep_stride,
                                                 const uint8_t *__restrict__ K, const uint8_t *__restrict__ V,
                                                 uint8_t *__restrict__ K_out, uint8_t *__restrict__ V_out,
                                                 uint32_t *status, uint64_t pol)
{
    constexpr int RB = LPR * 16, SL = 32 / LPR, R = ROWS / SL;
    static_assert(R * SL == ROWS, "ROWS must be a multiple of the rows a warp step covers");
    const int lane = threadIdx.x & 31, hw = lane / LPR, lr = lane % LPR;
    const int j0 = item * ROWS;
    const int cap = min(ROWS, min(keep_stride, idx_stride) - j0);
    const int32_t *ih = idx + head * idx_stride + j0;
    int src[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
        const int j = u * SL + hw;
        src[u] = j < cap ? __ldcg(ih + j) : -1;
    }
    const int n = min(cap, __ldcg(kept + head) - j0);
    const size_t in_head = (size_t)head * t_max * RB + lr * 16;
    const size_t out_head = ((size_t)head * keep_stride + j0) * RB + lr * 16;
    uint4 kv[R], vv[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
        if (u * SL + hw >= n) src[u] = -1;
        if (src[u] >= t_max) {
            atomicOr(status, MKV_DEV_INTERNAL);
            src[u] = -1;
        }
        if (src[u] >= 0) {
            const size_t off = in_head + (size_t)src[u] * RB;
            if (MKV_FUSED_GATHER_EVICT_FIRST) {
                kv[u] = ld_policy<2>(K + off, pol);
                vv[u] = ld_policy<2>(V + off, pol);
            } else {
                kv[u] = ld_stream(K + off);
                vv[u] = ld_stream(V + off);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < R; ++u) {
        if (src[u] >= 0) {
            const size_t off = out_head + (size_t)(u * SL + hw) * RB;
            if (MKV_FUSED_GATHER_EVICT_FIRST) {
                st_policy(K_out + off, kv[u], pol);
                st_policy(V_out + off, vv[u], pol);
            } else {
                st_v4(K_out + off, kv[u]);
                st_v4(V_out + off, vv[u]);
            }
        }
    }
}

template <int MODE, int NB, int ES>
__global__ void __launch_bounds__(kThreads, 2)
k_fused_path(PieceGeometry g, Pointers P, uint32_t *gcnt, int gsize, int groups, uint32_t stagger_ns, TailArgs A)
{
    constexpr int LPR = 4 * NB * ES;  // lanes per row: row bytes / 16
    constexpr int ROWS = fused_gather_rows(16 * LPR);
    __shared__ uint32_t s_ticket, s_go, s_abortable;
    if (threadIdx.x == 0) s_abortable = timed_out(P.status) ? 0u : 1u;  // read before any wait of this CTA
    __syncthreads();
    const bool abortable = s_abortable != 0u;
    if ((int)blockIdx.x < groups * gsize) {
        const int group = (int)blockIdx.x / gsize;
        head_groups_run<MODE, NB, ES>(g, P, gcnt, gsize, 1, stagger_ns, groups, group, (int)blockIdx.x % gsize,
                                      A.head_done, abortable, group == A.stall_group ? 1u : 0u);
    }
    const int64_t n_heads = g.n_heads;
    if ((int)blockIdx.x >= (int)gridDim.x - A.select_ctas) {
        for (;;) {
            __syncthreads();  // s_ticket and s_go of the previous select are read; shared memory is free
            if (threadIdx.x == 0) s_ticket = atomicAdd(A.sel_ticket, 1u);
            __syncthreads();
            const int64_t head = s_ticket;
            if (head >= n_heads) break;  // the same for every thread
            if (threadIdx.x == 0)
                s_go = wait_count(A.head_done + head, (uint32_t)gsize + (head == A.stall_head ? 1u : 0u), P.status,
                                  abortable);
            __syncthreads();
            if (s_go)
                select_item<true, false, kThreads>(head, P.S, P.seq_lens, g.heads, g.t_max, A.ratio, A.n_keep,
                                                   A.keep_stride, 0, g.nwin_max, nullptr, nullptr, 0, A.kept, A.idx,
                                                   A.idx_stride, P.status);
            else if (threadIdx.x == 0)
                A.kept[head] = 0;  // its gather items copy nothing
            __threadfence();  // the indices and the kept count are visible before the flag
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();  // the publishing thread's own fence: the flag releases the CTA's writes
                atomicExch(A.sel_done + head, 1u);
            }
        }
    }
    // gatherer: every warp on its own
    const int lane = threadIdx.x & 31;
    uint64_t drop_l2 = 0;
    if (MKV_FUSED_GATHER_EVICT_FIRST) asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(drop_l2));
    const int64_t n_items = n_heads * A.bph;
    uint32_t next = 0;
    if (lane == 0) next = atomicAdd(A.gather_ticket, 1u);
    next = __shfl_sync(kFull, next, 0);
    while ((int64_t)next < n_items) {
        const int64_t t = next, head = t / A.bph;
        const int item = (int)(t - head * A.bph);
        uint32_t claim = 0, go = 0;
        if (lane == 0) {
            claim = atomicAdd(A.gather_ticket, 1u);  // the next item, claimed while this one is copied
            go = wait_count(A.sel_done + head, 1u, P.status, abortable);
        }
        go = __shfl_sync(kFull, go, 0);
        __syncwarp();  // the lanes' reads of the indices come after lane 0's acquire of the flag
        if (go)
            gather_warp_item<LPR, ROWS>(head, item, A.idx, A.idx_stride, A.kept, g.t_max, A.keep_stride, P.K, A.V,
                                        A.K_out, A.V_out, P.status, drop_l2);
        next = __shfl_sync(kFull, claim, 0);
    }
}

Pointers make_pointers(const void *K, const int32_t *seq_lens, float *partial, float *C, float *S, uint32_t *status)
{
    Pointers P;
    P.K = static_cast<const uint8_t *>(K);
    P.seq_lens = seq_lens;
    P.partial = partial;
    P.C = C;
    P.S = S;
    P.status = status;
    return P;
}

}  // namespace

// ------------------------------------------------------------- launchers --

int single_pass_grid(int mode)
{
    const void *fn = mode == MKV_MODE_L2 ? reinterpret_cast<const void *>(k_single_pass<MKV_MODE_L2>)
                                         : reinterpret_cast<const void *>(k_single_pass<MKV_MODE_COSINE>);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(FusedShared)) != cudaSuccess)
        return 0;
    return resident_grid(fn, kFusedThreads, sizeof(FusedShared));
}

cudaError_t launch_single_pass(const PieceGeometry &g, int grid, const void *K, const int32_t *seq_lens, int mode,
                               float *partial, float *gsum, uint32_t *cnt, float *C, float *S, uint32_t *status,
                               cudaStream_t st, bool stall_windows)
{
    if (g.n_items == 0) return cudaSuccess;
    const size_t stride = (size_t)(g.ngroups_max + 2) * sizeof(uint32_t);
    const size_t wins = (size_t)g.n_heads * g.nwin_max;
    cudaError_t e = cudaMemsetAsync(cnt, 0, wins * stride, st);
    if (e != cudaSuccess) return e;
    if (stall_windows) {
        // failure injection: group and window counters start far past any
        // group size, so no window ever completes and every window wait must
        // run out; the ready flags stay 0
        e = cudaMemset2DAsync(cnt, stride, 0x40, (size_t)(g.ngroups_max + 1) * sizeof(uint32_t), wins, st);
        if (e != cudaSuccess) return e;
    }
    FusedPointers F;
    F.P = make_pointers(K, seq_lens, partial, C, S, status);
    F.gsum = gsum;
    F.cnt = cnt;
    PieceGeometry gg = g;
    void *args[] = {&gg, &F};
    const void *fn = mode == MKV_MODE_L2 ? reinterpret_cast<const void *>(k_single_pass<MKV_MODE_L2>)
                                         : reinterpret_cast<const void *>(k_single_pass<MKV_MODE_COSINE>);
    return cudaLaunchCooperativeKernel(fn, dim3((unsigned)grid), dim3(kFusedThreads), args, sizeof(FusedShared), st);
}

namespace {


// The kernel instance for a head dim (64 * NB), element size and mode.
template <int ES>
const void *head_groups_fn_es(int d, int mode)
{
    const bool l2 = mode == MKV_MODE_L2;
    switch (d) {
    case 64: return l2 ? (const void *)k_head_groups<MKV_MODE_L2, 1, ES> : (const void *)k_head_groups<MKV_MODE_COSINE, 1, ES>;
    case 128: return l2 ? (const void *)k_head_groups<MKV_MODE_L2, 2, ES> : (const void *)k_head_groups<MKV_MODE_COSINE, 2, ES>;
    case 256: return l2 ? (const void *)k_head_groups<MKV_MODE_L2, 4, ES> : (const void *)k_head_groups<MKV_MODE_COSINE, 4, ES>;
    default: return nullptr;
    }
}

const void *head_groups_fn(int d, int es, int mode)
{
    return es == 2 ? head_groups_fn_es<2>(d, mode) : es == 1 ? head_groups_fn_es<1>(d, mode) : nullptr;
}

template <int ES>
const void *fused_fn_es(int d, int mode)
{
    const bool l2 = mode == MKV_MODE_L2;
    switch (d) {
    case 64: return l2 ? (const void *)k_fused_path<MKV_MODE_L2, 1, ES> : (const void *)k_fused_path<MKV_MODE_COSINE, 1, ES>;
    case 128: return l2 ? (const void *)k_fused_path<MKV_MODE_L2, 2, ES> : (const void *)k_fused_path<MKV_MODE_COSINE, 2, ES>;
    case 256: return l2 ? (const void *)k_fused_path<MKV_MODE_L2, 4, ES> : (const void *)k_fused_path<MKV_MODE_COSINE, 4, ES>;
    default: return nullptr;
    }
}

const void *fused_fn(int d, int es, int mode)
{
    return es == 2 ? fused_fn_es<2>(d, mode) : es == 1 ? fused_fn_es<1>(d, mode) : nullptr;
}

template <int ES>
const void *piece_scores_fn_es(int d, int mode)
{
    const bool l2 = mode == MKV_MODE_L2;
    switch (d) {
    case 64: return l2 ? (const void *)k_piece_scores<MKV_MODE_L2, 1, ES> : (const void *)k_piece_scores<MKV_MODE_COSINE, 1, ES>;
    case 128: return l2 ? (const void *)k_piece_scores<MKV_MODE_L2, 2, ES> : (const void *)k_piece_scores<MKV_MODE_COSINE, 2, ES>;
    case 256: return l2 ? (const void *)k_piece_scores<MKV_MODE_L2, 4, ES> : (const void *)k_piece_scores<MKV_MODE_COSINE, 4, ES>;
    default: return nullptr;
    }
}

const void *piece_scores_fn(int d, int es, int mode)
{
    return es == 2 ? piece_scores_fn_es<2>(d, mode) : es == 1 ? piece_scores_fn_es<1>(d, mode) : nullptr;
}

template <int ES>
const void *piece_sums_fn_es(int d)
{
    switch (d) {
    case 64: return (const void *)k_piece_sums<1, ES>;
    case 128: return (const void *)k_piece_sums<2, ES>;
    case 256: return (const void *)k_piece_sums<4, ES>;
    default: return nullptr;
    }
}

const void *piece_sums_fn(int d, int es)
{
    return es == 2 ? piece_sums_fn_es<2>(d) : es == 1 ? piece_sums_fn_es<1>(d) : nullptr;
}

const void *window_means_fn(int d)
{
    switch (d) {
    case 64: return (const void *)k_window_means<64>;
    case 128: return (const void *)k_window_means<128>;
    case 256: return (const void *)k_window_means<256>;
    default: return nullptr;
    }
}

}  // namespace

namespace {

// Group count, group size and unit size for `resident` CTAs; `alone` applies
// the comparison with the three-kernel path (the head-group kernel on its
// own), which the fused kernel does not take.
HeadGroupPlan plan_groups(const PieceGeometry &g, int resident, size_t counters, bool alone,
                          int max_unit_windows = kMaxUnitWindows, bool ring = false)
{
    HeadGroupPlan plan;
    int dev = 0, l2 = 0;
    if (resident < 16 || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 <= 0)
        return plan;
    // Units (blocks of wb windows) in flight, one per group, must fit in 60%
    // of L2. Among group sizes of 4..64 CTAs and unit sizes of 1..kMaxUnit
    // windows, take the least modelled time: rounds (units per group) x (the
    // busiest CTA's pieces + 2 for the barrier, the means and the L2 pass),
    // with the groups filling at least 3/4 of the resident grid (else the
    // three-kernel path keeps more SMs busy). Equal costs keep the first
    // found: the fewest windows per unit, then the smallest group (measured:
    // Qwen W = 4096, 76 groups of 4 CTAs with one window 1.196 ms against 38
    // of 8 with two 1.220 ms; Phi-4 W = 8192, 38 of 8 with one window 3.360
    // ms against 19 of 16 with two 3.439 ms).
    const int wl_max = (g.window <= 0 || g.window >= g.t_max) ? g.t_max : g.window;
    if (wl_max < kMinPieceRows) return plan;  // windows shorter than a piece: barrier-bound rounds
    const double window_bytes = (double)wl_max * g.es * g.d;
    const double budget = 0.01 * (ring ? MKV_RING_L2_BUDGET_PCT : MKV_HG_L2_BUDGET_PCT) * (double)l2;
    double best = 0.0;
    for (int wb = 1; wb <= std::min(g.nwin_max, max_unit_windows); ++wb) {
        const int64_t fit = (int64_t)(budget / (window_bytes * wb));
        const int64_t units = g.n_heads * ((g.nwin_max + wb - 1) / wb);
        for (int gsize = 4; gsize <= 64; ++gsize) {
            const int64_t groups = std::min<int64_t>(std::min<int64_t>(fit, resident / gsize), units);
            if (groups < 1 || 4 * groups * gsize < 3 * (int64_t)resident) continue;
            if ((size_t)groups * sizeof(uint32_t) > counters) continue;
            const int64_t rounds = (units + groups - 1) / groups;
            const int ppc = (wb * g.ppw + gsize - 1) / gsize;
            const double cost = (double)rounds * (ppc + 2);
            if (plan.groups == 0 || cost < best) {
                best = cost;
                plan.groups = (int)groups;
                plan.gsize = gsize;
                plan.wb = wb;
            }
        }
    }
    if (plan.groups > 0) {
        const int64_t units = g.n_heads * ((g.nwin_max + plan.wb - 1) / plan.wb);
        const int64_t rounds = (units + plan.groups - 1) / plan.groups;
        // With several rounds per group the work, not the launch count,
        // decides: keep the head groups only if their modelled time is below
        // the three kernels' (every piece read twice over the same CTAs, in
        // the same piece-time units). Measured ratios follow the model up to
        // head dim 128: 0.84 on 256 x 16K global (model 0.83), 0.84 on the
        // Qwen and Phi-4 windowed shapes (0.78, 0.77), 1.07-1.16 on the
        // ragged batch of 2048 heads up to 32K (1.06: two pieces per CTA per
        // round). At head dim 256 the piece kernels keep half the head-group
        // kernel's bytes in flight per lane, so the model does not hold there
        // (64 x 16K: head groups 0.156 ms, three kernels 0.187).
        // E4M3 caches: decoding, not HBM, bounds both passes, so a saved read
        // of K does not pay for the rounds (256 x 16K: head groups 0.250 ms,
        // three kernels 0.243; cosine 0.294 against 0.289).
        const double three = 2.0 * (double)g.n_heads * g.nwin_max * g.ppw / (double)resident;
        if (alone && rounds >= 4 && (g.es == 1 || (g.d <= 128 && best >= three))) return HeadGroupPlan{};
        // the stagger step: a third of the time the units in flight take to
        // stream from HBM (at 6.5 TB/s), when every group has 4 rounds or more
        const double round_ns = (double)plan.groups * plan.wb * window_bytes / 6500.0;  // 6.5 TB/s = 6500 B/ns
        plan.stagger_ns = rounds >= 4 ? (uint32_t)std::min(20000.0, round_ns / 3.0) : 0u;
    }
    return plan;
}

}  // namespace

// The copy-ring head-group kernel of a mode (bf16 caches at head dim 128
// only: other shapes run the register kernel); nullptr where it has none.
const void *head_groups_ring_fn(int d, int es, int mode)
{
    if (d != 128 || es != 2) return nullptr;
    return mode == MKV_MODE_L2 ? (const void *)k_head_groups_ring<MKV_MODE_L2, 2>
                               : (const void *)k_head_groups_ring<MKV_MODE_COSINE, 2>;
}

HeadGroupPlan head_group_ring_plan(const PieceGeometry &g, int mode, size_t counters)
{
    if (g.n_heads == 0 || g.t_max == 0 || g.nwin_max == 0) return HeadGroupPlan{};
    const void *fn = head_groups_ring_fn(g.d, g.es, mode);
    // two CTAs of ~113 KB share an SM only with the whole carveout as shared memory
    if (!fn || cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRingSmem) != cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
            cudaSuccess)
        return HeadGroupPlan{};
    HeadGroupPlan plan = plan_groups(g, resident_grid(fn, kRingThreads, kRingSmem), counters, true,
                                     ring_unit_windows(g.d), true);
    plan.ring = plan.groups > 0;
    return plan;
}

HeadGroupPlan head_group_plan(const PieceGeometry &g, int mode, size_t counters)
{
    if (g.n_heads == 0 || g.t_max == 0 || g.nwin_max == 0) return HeadGroupPlan{};
    const void *fn = head_groups_fn(g.d, g.es, mode);
    if (!fn || cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kHgSmem) != cudaSuccess)
        return HeadGroupPlan{};
    return plan_groups(g, resident_grid(fn, kThreads, kHgSmem), counters, true);
}

FusedPlan fused_plan(const PieceGeometry &g, int mode, size_t counters, int scorer_ctas, int select_ctas)
{
    FusedPlan fp;
    // whole heads as units, and each head's scores fit the select's shared memory
    if (g.n_heads == 0 || g.t_max == 0 || g.nwin_max != 1 || g.t_max > kFusedMaxT || scorer_ctas == 0) return fp;
    const void *fn = fused_fn(g.d, g.es, mode);
    if (!fn || cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGroupSmem) != cudaSuccess)
        return fp;
    const int resident = resident_grid(fn, kThreads, kGroupSmem);
    if (resident < 16) return fp;
    // a negative budget: 3/4 of the resident grid
    const HeadGroupPlan hp = plan_groups(g, scorer_ctas < 0 ? resident * 3 / 4 : std::min(scorer_ctas, resident),
                                         counters, false);
    if (hp.groups == 0 || hp.wb != 1) return fp;
    // counters: the groups' arrivals, head_done, sel_done and the two tickets
    if (((size_t)hp.groups + 2 * (size_t)g.n_heads + 2) * sizeof(uint32_t) > counters) return fp;
    fp.hg = hp;
    fp.grid = resident;
    fp.select_ctas = std::max(1, std::min(select_ctas > 0 ? select_ctas : 32, resident));
    return fp;
}

cudaError_t launch_fused(const PieceGeometry &g, const FusedPlan &fp, int mode, const void *K, const void *V,
                         const int32_t *seq_lens, float *partial, uint32_t *cnt, float *C, float *S, double ratio,
                         const int32_t *n_keep, int32_t keep_stride, int32_t *kept, int32_t *idx, int32_t idx_stride,
                         void *K_out, void *V_out, uint32_t *status, cudaStream_t st, int stall)
{
    const void *fn = fused_fn(g.d, g.es, mode);
    if (!fn || fp.grid <= 0) return cudaErrorInvalidValue;
    const size_t words = (size_t)fp.hg.groups + 2 * (size_t)g.n_heads + 2;
    cudaError_t e = cudaMemsetAsync(cnt, 0, words * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    Pointers P = make_pointers(K, seq_lens, partial, C, S, status);
    TailArgs A;
    A.V = static_cast<const uint8_t *>(V);
    A.K_out = static_cast<uint8_t *>(K_out);
    A.V_out = static_cast<uint8_t *>(V_out);
    A.n_keep = n_keep;
    A.kept = kept;
    A.idx = idx;
    A.head_done = cnt + fp.hg.groups;
    A.sel_done = A.head_done + g.n_heads;
    A.sel_ticket = A.sel_done + g.n_heads;
    A.gather_ticket = A.sel_ticket + 1;
    A.ratio = ratio;
    A.keep_stride = keep_stride;
    A.idx_stride = idx_stride;
    const int rows = fused_gather_rows(g.d * g.es);
    A.bph = (keep_stride + rows - 1) / rows;
    A.select_ctas = fp.select_ctas;
    A.stall_group = stall == 0 ? 0 : -1;
    A.stall_head = stall == 1 ? 0 : -1;
    PieceGeometry gg = g;
    int gsize = fp.hg.gsize, groups = fp.hg.groups;
    uint32_t stagger = fp.hg.stagger_ns;
    void *args[] = {&gg, &P, &cnt, &gsize, &groups, &stagger, &A};
    return cudaLaunchCooperativeKernel(fn, dim3((unsigned)fp.grid), dim3(kThreads), args, kGroupSmem, st);
}

cudaError_t launch_head_groups(const PieceGeometry &g, const HeadGroupPlan &plan, const void *K,
                               const int32_t *seq_lens, int mode, float *partial, uint32_t *cnt, float *C, float *S,
                               uint32_t *status, cudaStream_t st)
{
    const void *fn = plan.ring ? head_groups_ring_fn(g.d, g.es, mode) : head_groups_fn(g.d, g.es, mode);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(cnt, 0, (size_t)plan.groups * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    Pointers P = make_pointers(K, seq_lens, partial, C, S, status);
    PieceGeometry gg = g;
    int gsize = plan.gsize, wb = plan.wb;
    uint32_t stagger = plan.stagger_ns;
    void *args[] = {&gg, &P, &cnt, &gsize, &wb, &stagger};
    return cudaLaunchCooperativeKernel(fn, dim3((unsigned)(plan.groups * plan.gsize)),
                                       dim3(plan.ring ? kRingThreads : kThreads), args,
                                       plan.ring ? kRingSmem : kHgSmem, st);
}

cudaError_t launch_piece_sums(const PieceGeometry &g, const void *K, const int32_t *seq_lens, float *partial,
                              uint32_t *status, cudaStream_t st)
{
    if (g.n_items == 0) return cudaSuccess;
    const void *fn = piece_sums_fn(g.d, g.es);
    if (!fn) return cudaErrorInvalidValue;
    const int grid = grid_for_items(fn, kThreads, 0, g.n_items);
    PieceGeometry gg = g;
    Pointers P = make_pointers(K, seq_lens, partial, nullptr, nullptr, status);
    void *args[] = {&gg, &P};
    return cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(kThreads), args, 0, st);
}

cudaError_t launch_window_means(const PieceGeometry &g, const float *partial, const int32_t *seq_lens, float *C,
                                uint32_t *status, cudaStream_t st)
{
    const int64_t wins = g.n_heads * g.nwin_max;
    if (wins == 0) return cudaSuccess;
    const void *fn = window_means_fn(g.d);
    if (!fn) return cudaErrorInvalidValue;
    PieceGeometry gg = g;
    Pointers P = make_pointers(nullptr, seq_lens, const_cast<float *>(partial), C, nullptr, status);
    void *args[] = {&gg, &P};
    return cudaLaunchKernel(fn, dim3((unsigned)wins), dim3((unsigned)g.d), args, 0, st);
}

cudaError_t launch_piece_scores(const PieceGeometry &g, const void *K, const float *C, const int32_t *seq_lens,
                                int mode, float *S, uint32_t *status, cudaStream_t st)
{
    if (g.n_items == 0) return cudaSuccess;
    const void *fn = piece_scores_fn(g.d, g.es, mode);
    if (!fn) return cudaErrorInvalidValue;
    const int grid = grid_for_items(fn, kThreads, 0, g.n_items);
    PieceGeometry gg = g;
    Pointers P = make_pointers(K, seq_lens, nullptr, const_cast<float *>(C), S, status);
    void *args[] = {&gg, &P};
    return cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(kThreads), args, 0, st);
}

}  // namespace mkv
