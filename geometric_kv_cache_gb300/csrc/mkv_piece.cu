// Centroid and score kernels (steps a1 and a2).
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

#include "mkv_device.cuh"
#include "mkv_internal.h"

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

// Combine the per-thread accumulators into the piece sum, written to out[]
// (128 floats) by threads 0..127. `red` is [kWarps][128] shared scratch; the
// caller synchronises before `red` is reused.
__device__ __forceinline__ void finish_sum(float acc[16], float *red, float *out)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, q = threadIdx.x & 7;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        acc[j] += __shfl_xor_sync(kFull, acc[j], 8);
        acc[j] += __shfl_xor_sync(kFull, acc[j], 16);
    }
    if (lane < 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            red[warp * kHeadDim + q * 8 + j] = acc[j];
            red[warp * kHeadDim + 64 + q * 8 + j] = acc[8 + j];
        }
    }
    __syncthreads();
    if (threadIdx.x < kHeadDim) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[w * kHeadDim + threadIdx.x];
        out[threadIdx.x] = s;
    }
}

// Score of one row from the thread's 16 dims f, centroid dims c and the
// centroid norm nc (cosine only). Reduces over the row's 8 lanes, so all 32
// lanes of the warp must call it.
template <int MODE>
__device__ __forceinline__ float score_of(const float f[16], const float c[16], float nc)
{
    if (MODE == MKV_MODE_L2) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
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
        for (int j = 0; j < 16; ++j) {
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
__device__ __forceinline__ float centroid_norm(const float c[16])
{
    float cc = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) cc = fmaf(c[j], c[j], cc);
    cc += __shfl_xor_sync(kFull, cc, 4);
    cc += __shfl_xor_sync(kFull, cc, 2);
    cc += __shfl_xor_sync(kFull, cc, 1);
    return __fsqrt_rn(cc);
}

// The thread's 16 centroid dims from cw (L2 reads: another CTA may have
// written them during this kernel).
__device__ __forceinline__ void load_centroid(const float *cw, float c[16])
{
    const int q = threadIdx.x & 7;
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(cw + q * 8));
    const float4 b = __ldcg(reinterpret_cast<const float4 *>(cw + q * 8 + 4));
    const float4 d = __ldcg(reinterpret_cast<const float4 *>(cw + 64 + q * 8));
    const float4 e = __ldcg(reinterpret_cast<const float4 *>(cw + 64 + q * 8 + 4));
    c[0] = a.x; c[1] = a.y; c[2] = a.z; c[3] = a.w;
    c[4] = b.x; c[5] = b.y; c[6] = b.z; c[7] = b.w;
    c[8] = d.x; c[9] = d.y; c[10] = d.z; c[11] = d.w;
    c[12] = e.x; c[13] = e.y; c[14] = e.z; c[15] = e.w;
}

// Sum of n (<= kGroupPieces) consecutive 128-float records, record order,
// dim d; all loads issued before the adds.
__device__ __forceinline__ float ordered_sum(const float *first, int n, int d)
{
    float v[kGroupPieces];
#pragma unroll
    for (int j = 0; j < kGroupPieces; ++j) v[j] = j < n ? __ldcg(first + (int64_t)j * kHeadDim + d) : 0.f;
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kGroupPieces; ++j)
        if (j < n) s += v[j];
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

// Rows r = slot + 32 * (i0 + u), u < kBatch, of a piece starting at `base`
// (this thread's two 16-byte chunks of each), loaded before use.
constexpr int kBatch = 4;

__device__ __forceinline__ void load_batch(const uint8_t *base, int len, int i0, uint4 v[2 * kBatch])
{
    const int slot = threadIdx.x >> 3, q = threadIdx.x & 7;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
        const int r = slot + (i0 + u) * kRowSlots;
        const uint8_t *row = base + (size_t)(r < len ? r : 0) * kRowBytes;
        v[2 * u] = ld_stream(row + q * 16);
        v[2 * u + 1] = ld_stream(row + 128 + q * 16);
    }
}

// a1, first half: piece sums. The first batch of the next piece is loaded
// before the current piece's CTA reduction, so the loads stay in flight
// across piece boundaries.
__global__ void __launch_bounds__(kThreads)
k_piece_sums(PieceGeometry g, Pointers P)
{
    __shared__ float red[kWarps * kHeadDim];
    const Steps st = make_steps(g);
    const int slot = threadIdx.x >> 3;
    Cursor cur = first_cursor(g, st, P.seq_lens, P.status);
    uint4 v[2 * kBatch];
    if (!cur.done) load_batch(P.K + ((size_t)cur.pc.head * g.t_max + cur.pc.a) * kRowBytes, cur.pc.len, 0, v);
    while (!cur.done) {
        const Piece pc = cur.pc;
        const int64_t item = cursor_item(cur, st);
        const uint8_t *base = P.K + ((size_t)pc.head * g.t_max + pc.a) * kRowBytes;
        const int nrows = (pc.len + kRowSlots - 1) / kRowSlots;  // rows per slot (upper bound)
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = 0.f;
        for (int i0 = 0; i0 < nrows; i0 += kBatch) {
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (slot + (i0 + u) * kRowSlots < pc.len) {
                    float f[16];
                    bf16x8_to_f32(v[2 * u], f);
                    bf16x8_to_f32(v[2 * u + 1], f + 8);
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] += f[j];
                }
            }
            if (i0 + kBatch < nrows) load_batch(base, pc.len, i0 + kBatch, v);
        }
        advance(cur, st, g, P.seq_lens, P.status);
        if (!cur.done) load_batch(P.K + ((size_t)cur.pc.head * g.t_max + cur.pc.a) * kRowBytes, cur.pc.len, 0, v);
        finish_sum(acc, red, P.partial + item * kHeadDim);
        __syncthreads();  // red is free again
    }
}

// a1, second half: window means, one warp per (head, window): groups of 32
// pieces in piece order, then the groups in group order.
__global__ void __launch_bounds__(256)
k_window_means(PieceGeometry g, Pointers P)
{
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (gw >= g.n_heads * g.nwin_max) return;
    const int64_t head = gw / g.nwin_max;
    const int w = (int)(gw - head * g.nwin_max);
    const int T = head_len(P.seq_lens, head, g.heads, g.t_max, P.status, false);
    if (T == 0) return;
    const int wl = window_len(T, g.window);
    const int64_t wstart = (int64_t)w * wl;
    if (wstart >= T) return;
    const int wlen = (int)min((int64_t)wl, (int64_t)T - wstart);
    const int np = (wlen + g.piece_rows - 1) / g.piece_rows;
    const int ng = (np + kGroupPieces - 1) / kGroupPieces;
    const float *pw = P.partial + ((head * g.nwin_max + w) * (int64_t)g.ppw) * kHeadDim;
    float tot[4] = {0.f, 0.f, 0.f, 0.f};
    for (int gi = 0; gi < ng; ++gi) {
        const int n = min(kGroupPieces, np - gi * kGroupPieces);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            tot[k] += ordered_sum(pw + (int64_t)gi * kGroupPieces * kHeadDim, n, lane * 4 + k);
    }
    float *cw = P.C + (head * g.nwin_max + w) * kHeadDim;
    const float n = (float)wlen;
#pragma unroll
    for (int k = 0; k < 4; ++k) cw[lane * 4 + k] = __fdiv_rn(tot[k], n);
}

// a2: scores of every piece against its window's mean in C.
template <int MODE>
__global__ void __launch_bounds__(kThreads)
k_piece_scores(PieceGeometry g, Pointers P)
{
    const Steps st = make_steps(g);
    const int slot = threadIdx.x >> 3, q = threadIdx.x & 7;
    Cursor cur = first_cursor(g, st, P.seq_lens, P.status);
    while (!cur.done) {
        const Piece &pc = cur.pc;
        const uint8_t *base = P.K + ((size_t)pc.head * g.t_max + pc.a) * kRowBytes;
        float *srow = P.S + (size_t)pc.head * g.t_max + pc.a;
        float c[16];
        load_centroid(P.C + (pc.head * g.nwin_max + pc.w) * kHeadDim, c);
        const float nc = MODE == MKV_MODE_COSINE ? centroid_norm(c) : 0.f;
        const int nrows = (pc.len + kRowSlots - 1) / kRowSlots;
        for (int i0 = 0; i0 < nrows; i0 += kBatch) {
            uint4 v[2 * kBatch];
            load_batch(base, pc.len, i0, v);
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int r = slot + (i0 + u) * kRowSlots;
                float f[16];
                bf16x8_to_f32(v[2 * u], f);
                bf16x8_to_f32(v[2 * u + 1], f + 8);
                const float s = score_of<MODE>(f, c, nc);
                if (r < pc.len && q == 0) srow[r] = s;
            }
        }
        advance(cur, st, g, P.seq_lens, P.status);
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

cudaError_t launch_piece_sums(const PieceGeometry &g, const void *K, const int32_t *seq_lens, float *partial,
                              uint32_t *status, cudaStream_t st)
{
    if (g.n_items == 0) return cudaSuccess;
    const int grid = grid_for_items(reinterpret_cast<const void *>(k_piece_sums), kThreads, 0, g.n_items);
    k_piece_sums<<<grid, kThreads, 0, st>>>(g, make_pointers(K, seq_lens, partial, nullptr, nullptr, status));
    return cudaGetLastError();
}

cudaError_t launch_window_means(const PieceGeometry &g, const float *partial, const int32_t *seq_lens, float *C,
                                uint32_t *status, cudaStream_t st)
{
    const int64_t wins = g.n_heads * g.nwin_max;
    if (wins == 0) return cudaSuccess;
    k_window_means<<<(unsigned)((wins + 7) / 8), 256, 0, st>>>(
        g, make_pointers(nullptr, seq_lens, const_cast<float *>(partial), C, nullptr, status));
    return cudaGetLastError();
}

cudaError_t launch_piece_scores(const PieceGeometry &g, const void *K, const float *C, const int32_t *seq_lens,
                                int mode, float *S, uint32_t *status, cudaStream_t st)
{
    if (g.n_items == 0) return cudaSuccess;
    const Pointers P = make_pointers(K, seq_lens, nullptr, const_cast<float *>(C), S, status);
    if (mode == MKV_MODE_L2) {
        const int grid = grid_for_items(reinterpret_cast<const void *>(k_piece_scores<MKV_MODE_L2>), kThreads, 0,
                                        g.n_items);
        k_piece_scores<MKV_MODE_L2><<<grid, kThreads, 0, st>>>(g, P);
    } else {
        const int grid = grid_for_items(reinterpret_cast<const void *>(k_piece_scores<MKV_MODE_COSINE>), kThreads, 0,
                                        g.n_items);
        k_piece_scores<MKV_MODE_COSINE><<<grid, kThreads, 0, st>>>(g, P);
    }
    return cudaGetLastError();
}

}  // namespace mkv
