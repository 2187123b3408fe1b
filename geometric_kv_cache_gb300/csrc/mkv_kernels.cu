// sm_103a kernels of the ManifoldKV-style compression path.
//
// Method: "ManifoldKV: Training-Free KV Cache Compression via Euclidean
// Outlier Detection" (ICML 2026 poster 62526), abstract and lay summary --
// key centroid (global, or per window for WindowedManifoldKV), Euclidean or
// one-minus-cosine score against it, keep the highest-scoring tokens, gather
// the kept K/V rows.
//
// Every kernel here streams HBM: none of the work is a dense contraction, so
// there are no tensor-core paths. Design rules used throughout:
//  * a 256-byte bf16 key row is read by 16 lanes with one 16-byte load each
//    (a warp covers two rows per load instruction), through the
//    non-coherent path with L1 no-allocate, four rows in flight per lane;
//  * fp32 accumulation in a fixed order (per-lane sequential, then a fixed
//    shared-memory or shuffle tree): results never depend on grid size;
//  * grids are a multiple of the SM count times the resident CTAs per SM and
//    loop over work items (persistent style), so short tails stay small;
//  * no float atomics, no spin waits, no traps: bad device-side inputs set
//    bits in a status word and the head is skipped.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "mkv_internal.h"

namespace mkv {
namespace {

constexpr int kStreamThreads = 256;            // centroid / score / gather CTAs
constexpr int kSlots = kStreamThreads / 16;    // rows per CTA per load step
constexpr int kUnroll = 4;                     // load steps in flight per lane
constexpr int kSelectThreads = 1024;
constexpr unsigned kFull = 0xFFFFFFFFu;

// ---------------------------------------------------------------- helpers --

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v)
{
    *reinterpret_cast<uint4 *>(p) = v;
}

// Eight bf16 values of a 16-byte chunk, widened exactly to fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float f[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Sum over the 16 lanes of a half-warp (all 32 lanes must call it).
__device__ __forceinline__ float half_warp_sum(float v)
{
    v += __shfl_xor_sync(kFull, v, 8);
    v += __shfl_xor_sync(kFull, v, 4);
    v += __shfl_xor_sync(kFull, v, 2);
    v += __shfl_xor_sync(kFull, v, 1);
    return v;
}

// Order-preserving map of fp32 bits to uint32 (larger score -> larger key).
__device__ __forceinline__ uint32_t score_key(float s)
{
    const uint32_t b = __float_as_uint(s);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Tokens of head `head`; a length outside [0, t_max] is reported and the
// head treated as empty.
__device__ __forceinline__ int head_len(const int32_t *seq_lens, int64_t head, int heads, int t_max,
                                        uint32_t *status, bool report)
{
    if (!seq_lens) return t_max;
    const int T = seq_lens[head / heads];
    if (T < 0 || T > t_max) {
        if (report) atomicOr(status, MKV_DEV_BAD_SEQ_LEN);
        return 0;
    }
    return T;
}

__device__ __forceinline__ int window_len(int T, int window)
{
    return (window <= 0 || window >= T) ? T : window;
}

// floor(T*(1-ratio) + 0.5) clamped to [0, T], each operation rounded once
// (no contraction into an FMA), matching the host helper bit for bit.
__device__ __forceinline__ int num_keep_dev(int T, double ratio)
{
    if (T <= 0) return 0;
    const double x = floor(__dadd_rn(__dmul_rn((double)T, __dsub_rn(1.0, ratio)), 0.5));
    if (x < 0.0) return 0;
    if (x > (double)T) return T;
    return (int)x;
}

// Exclusive prefix sum over the CTA in thread order; *total gets the sum.
// Every thread of the CTA must call it; `scratch` holds one word per warp.
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *scratch, uint32_t *total)
{
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < NW ? scratch[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NW) scratch[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    const uint32_t before_warp = warp ? scratch[warp - 1] : 0u;
    if (total) *total = scratch[NW - 1];
    __syncthreads();  // scratch may be reused right after
    return before_warp + x - v;
}

// ---------------------------------------------------------- a1: centroid --

// Partial key sums of one piece (a run of at most g.piece tokens inside one
// window). Item = (head, window, piece), head-major. Each half-warp owns a
// token slot, each lane eight dims; the 16 slot sums are added in slot order.
__global__ void __launch_bounds__(kStreamThreads)
k_centroid_partial(const uint8_t *__restrict__ K, const int32_t *__restrict__ seq_lens, int heads,
                   int t_max, int window, int nwin_max, int piece, int ppw, int64_t n_items,
                   float *__restrict__ partial, uint32_t *status)
{
    __shared__ float4 red[kSlots][kHeadDim / 4];
    const int hw = threadIdx.x >> 4, l16 = threadIdx.x & 15;
    const int64_t per_head = (int64_t)nwin_max * ppw;
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int64_t head = item / per_head;
        const int r = (int)(item - head * per_head);
        const int w = r / ppw, p = r - w * ppw;
        const int T = head_len(seq_lens, head, heads, t_max, status, r == 0 && threadIdx.x == 0);
        const int wl = window_len(T, window);
        if (T == 0) continue;
        const int64_t a64 = (int64_t)w * wl + (int64_t)p * piece;
        const int64_t wend = min((int64_t)(w + 1) * wl, (int64_t)T);
        if (a64 >= wend) continue;
        const int a = (int)a64, b = (int)min(a64 + piece, wend);
        const uint8_t *base = K + ((size_t)head * t_max) * kRowBytes + l16 * 16;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int r0 = a; r0 < b; r0 += kSlots * kUnroll) {
            uint4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int row = r0 + u * kSlots + hw;
                v[u] = row < b ? ld_stream(base + (size_t)row * kRowBytes) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                float f[8];
                bf16x8_to_f32(v[u], f);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] += f[j];
            }
        }
        red[hw][l16 * 2] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        red[hw][l16 * 2 + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        __syncthreads();
        if (threadIdx.x < kHeadDim) {
            const float *redf = reinterpret_cast<const float *>(red);
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < kSlots; ++k) s += redf[k * kHeadDim + threadIdx.x];
            partial[item * kHeadDim + threadIdx.x] = s;
        }
        __syncthreads();
    }
}

// Window means: one warp per (head, window) adds the window's pieces in order
// and divides by the window's token count (IEEE division).
__global__ void __launch_bounds__(256)
k_centroid_finalize(const float *__restrict__ partial, const int32_t *__restrict__ seq_lens, int heads,
                    int t_max, int window, int nwin_max, int piece, int ppw, int64_t n_win_items,
                    float *__restrict__ C, uint32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (gw >= n_win_items) return;
    const int64_t head = gw / nwin_max;
    const int w = (int)(gw - head * nwin_max);
    const int T = head_len(seq_lens, head, heads, t_max, status, false);
    if (T == 0) return;
    const int wl = window_len(T, window);
    const int nwin = (T + wl - 1) / wl;
    if (w >= nwin) return;
    const int len = min(wl, T - w * wl);
    const int np = (len + piece - 1) / piece;
    const float4 *src = reinterpret_cast<const float4 *>(partial + ((head * nwin_max + w) * (int64_t)ppw) * kHeadDim);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = 0; p < np; ++p) {
        const float4 x = src[(int64_t)p * (kHeadDim / 4) + lane];
        s.x += x.x;
        s.y += x.y;
        s.z += x.z;
        s.w += x.w;
    }
    const float n = (float)len;
    reinterpret_cast<float4 *>(C + (head * nwin_max + w) * kHeadDim)[lane] =
        make_float4(__fdiv_rn(s.x, n), __fdiv_rn(s.y, n), __fdiv_rn(s.z, n), __fdiv_rn(s.w, n));
}

// -------------------------------------------------------------- a2: score --

// One score per token: |k - c| (L2) or 1 - k.c/(|k||c|) (cosine, 1 when the
// denominator is 0), c the centroid of the token's window. Item = (head,
// chunk of score_chunk tokens). Loop bounds are CTA-uniform so the shuffles
// always run with the whole warp.
template <int MODE>
__global__ void __launch_bounds__(kStreamThreads)
k_score(const uint8_t *__restrict__ K, const float *__restrict__ C, const int32_t *__restrict__ seq_lens,
        int heads, int t_max, int window, int nwin_max, int chunk, int nch, int64_t n_items,
        float *__restrict__ S, uint32_t *status)
{
    const int hw = threadIdx.x >> 4, l16 = threadIdx.x & 15;
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int64_t head = item / nch;
        const int ch = (int)(item - head * nch);
        const int T = head_len(seq_lens, head, heads, t_max, status, false);
        const int a = ch * chunk;
        if (a >= T) continue;
        const int b = min(a + chunk, T);
        const int wl = window_len(T, window);
        const uint8_t *base = K + ((size_t)head * t_max) * kRowBytes + l16 * 16;
        const float *cbase = C + (size_t)head * nwin_max * kHeadDim + l16 * 8;
        float *srow = S + (size_t)head * t_max;
        int cur_w = -1;
        float c[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float nc = 0.f;
        for (int r0 = a; r0 < b; r0 += kSlots * kUnroll) {
            uint4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int row = r0 + u * kSlots + hw;
                v[u] = row < b ? ld_stream(base + (size_t)row * kRowBytes) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int row = r0 + u * kSlots + hw;
                const bool valid = row < b;
                const int w = valid ? row / wl : cur_w;
                const bool need = w != cur_w;
                if (__any_sync(kFull, need)) {
                    if (need) {
                        const float4 c0 = reinterpret_cast<const float4 *>(cbase + (size_t)w * kHeadDim)[0];
                        const float4 c1 = reinterpret_cast<const float4 *>(cbase + (size_t)w * kHeadDim)[1];
                        c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
                        c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
                        cur_w = w;
                    }
                    if (MODE == MKV_MODE_COSINE) {
                        float cc = 0.f;
#pragma unroll
                        for (int j = 0; j < 8; ++j) cc = fmaf(c[j], c[j], cc);
                        nc = __fsqrt_rn(half_warp_sum(cc));
                    }
                }
                float f[8];
                bf16x8_to_f32(v[u], f);
                float s;
                if (MODE == MKV_MODE_L2) {
                    float acc = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float d = f[j] - c[j];
                        acc = fmaf(d, d, acc);
                    }
                    s = __fsqrt_rn(half_warp_sum(acc));
                } else {
                    float dot = 0.f, kk = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        dot = fmaf(f[j], c[j], dot);
                        kk = fmaf(f[j], f[j], kk);
                    }
                    dot = half_warp_sum(dot);
                    kk = half_warp_sum(kk);
                    const float den = __fmul_rn(__fsqrt_rn(kk), nc);
                    s = den == 0.f ? 1.f : __fsub_rn(1.f, __fdiv_rn(dot, den));
                }
                if (valid && l16 == 0) srow[row] = s;
            }
        }
    }
}

// ------------------------------------------------------ a3: radix select --

// Per-chunk kept counts and their exclusive scan for one head (all threads of
// the 1024-thread CTA call it): chunk_info[c] = {first output slot of chunk c,
// ties at the cut key in chunks before c}; returns the head's kept count.
__device__ int chunk_offsets_block(const float *srow, int T, mkv_cut cut, int nch_max,
                                   int2 *__restrict__ info, uint32_t *s_warp)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nch = (T + kCompactChunk - 1) / kCompactChunk;
    for (int c = warp; c < nch; c += kSelectThreads / 32) {
        const int a = c * kCompactChunk, b = min(a + kCompactChunk, T);
        uint32_t gt = 0, eq = 0;
        for (int t = a + lane; t < b; t += 32) {
            const uint32_t u = score_key(srow[t]);
            gt += u > cut.key;
            eq += u == cut.key;
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            gt += __shfl_xor_sync(kFull, gt, o);
            eq += __shfl_xor_sync(kFull, eq, o);
        }
        if (lane == 0) info[c] = make_int2((int)gt, (int)eq);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int offset = 0, ties_before = 0;
        for (int c = 0; c < nch; ++c) {
            const int2 ge = info[c];
            const int tie_keep = max(0, min(ge.y, cut.ties - ties_before));
            info[c] = make_int2(offset, ties_before);
            offset += ge.x + tie_keep;
            ties_before += ge.y;
        }
        s_warp[0] = (uint32_t)offset;
    }
    __syncthreads();
    const int kept = (int)s_warp[0];
    __syncthreads();
    return kept;
}

// One CTA per head (persistent over heads). Three histogram passes over the
// head's score keys (digits of 11, 11 and 10 bits, most significant first)
// find the n_keep-th largest key and how many of its ties are kept; with
// chunk_info it then computes the compaction offsets (fused path).
__global__ void __launch_bounds__(kSelectThreads, 1)
k_select(const float *__restrict__ S, const int32_t *__restrict__ seq_lens, int heads, int t_max,
         double ratio, const int32_t *__restrict__ n_keep, int keep_stride, int64_t n_heads,
         mkv_cut *__restrict__ cut_out, int2 *__restrict__ chunk_info, int nch_max,
         int32_t *__restrict__ kept_out, uint32_t *status)
{
    __shared__ uint32_t hist[2048];
    __shared__ uint32_t s_warp[32];
    __shared__ uint32_t s_digit, s_above;
    const int lane = threadIdx.x & 31;
    for (int64_t head = blockIdx.x; head < n_heads; head += gridDim.x) {
        const int T = head_len(seq_lens, head, heads, t_max, status, threadIdx.x == 0);
        const int nk = n_keep ? n_keep[head] : num_keep_dev(T, ratio);
        if (nk < 0 || nk > T || (keep_stride >= 0 && nk > keep_stride)) {
            if (threadIdx.x == 0) {
                atomicOr(status, MKV_DEV_BAD_N_KEEP);
                mkv_cut none;
                none.key = kNoneKey;
                none.ties = 0;
                cut_out[head] = none;
                if (kept_out) kept_out[head] = 0;
            }
            if (chunk_info) {
                const int nch = (T + kCompactChunk - 1) / kCompactChunk;
                for (int c = threadIdx.x; c < nch; c += kSelectThreads) chunk_info[head * nch_max + c] = make_int2(-1, -1);
            }
            continue;
        }
        const float *srow = S + (size_t)head * t_max;
        uint32_t prefix = 0, pmask = 0;
        int need = nk;
        if (nk > 0) {
#pragma unroll 1
            for (int pass = 0; pass < 3; ++pass) {
                const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
                const int nb = pass == 2 ? 1024 : 2048;
                for (int i = threadIdx.x; i < nb; i += kSelectThreads) hist[i] = 0;
                __syncthreads();
                for (int base = 0; base < T; base += kSelectThreads) {
                    const int t = base + threadIdx.x;
                    bool v = t < T;
                    uint32_t u = 0;
                    if (v) {
                        u = score_key(srow[t]);
                        v = (u & pmask) == prefix;
                    }
                    const uint32_t dig = v ? ((u >> shift) & (uint32_t)(nb - 1)) : 0xFFFFFFFFu;
                    const uint32_t peers = __match_any_sync(kFull, dig);
                    if (v && lane == __ffs(peers) - 1) atomicAdd(&hist[dig], (uint32_t)__popc(peers));
                }
                __syncthreads();
                // Thread i owns bins in descending order: bpt bins from nb-1-i*bpt down.
                const int bpt = nb / kSelectThreads;
                const int hi = nb - 1 - threadIdx.x * bpt;
                uint32_t local = 0;
                for (int j = 0; j < bpt; ++j) local += hist[hi - j];
                uint32_t above = block_exclusive_scan<kSelectThreads>(local, s_warp, nullptr);
                for (int j = 0; j < bpt; ++j) {
                    const uint32_t h = hist[hi - j];
                    if (above < (uint32_t)need && (uint32_t)need <= above + h) {
                        s_digit = (uint32_t)(hi - j);
                        s_above = above;
                    }
                    above += h;
                }
                __syncthreads();
                prefix |= s_digit << shift;
                pmask |= (uint32_t)(nb - 1) << shift;
                need -= (int)s_above;
                __syncthreads();
            }
        } else {
            prefix = kNoneKey;
            need = 0;
        }
        mkv_cut cut;
        cut.key = prefix;
        cut.ties = need;
        if (threadIdx.x == 0) cut_out[head] = cut;
        if (chunk_info) {
            const int kept = nk > 0 ? chunk_offsets_block(srow, T, cut, nch_max, chunk_info + head * nch_max, s_warp) : 0;
            if (threadIdx.x == 0) {
                if (kept != nk) atomicOr(status, MKV_DEV_INTERNAL);
                if (kept_out) kept_out[head] = kept;
            }
        }
    }
}

// Compaction offsets for a given cut (the step-wise path).
__global__ void __launch_bounds__(kSelectThreads)
k_chunk_offsets(const float *__restrict__ S, const mkv_cut *__restrict__ cuts,
                const int32_t *__restrict__ seq_lens, int heads, int t_max, double ratio,
                const int32_t *__restrict__ n_keep, int keep_stride, int64_t n_heads,
                int2 *__restrict__ chunk_info, int nch_max, int32_t *__restrict__ kept_out,
                uint32_t *status)
{
    __shared__ uint32_t s_warp[32];
    for (int64_t head = blockIdx.x; head < n_heads; head += gridDim.x) {
        const int T = head_len(seq_lens, head, heads, t_max, status, threadIdx.x == 0);
        const int nk = n_keep ? n_keep[head] : num_keep_dev(T, ratio);
        const mkv_cut cut = cuts[head];
        const bool bad = nk < 0 || nk > T || (keep_stride >= 0 && nk > keep_stride);
        int kept = 0;
        if (!bad && cut.key != kNoneKey) {
            kept = chunk_offsets_block(S + (size_t)head * t_max, T, cut, nch_max, chunk_info + head * nch_max, s_warp);
        } else {
            // Mark every chunk of a skipped head so the gather leaves it alone.
            const int nch = (T + kCompactChunk - 1) / kCompactChunk;
            for (int c = threadIdx.x; c < nch; c += kSelectThreads) chunk_info[head * nch_max + c] = make_int2(-1, -1);
        }
        if (threadIdx.x == 0) {
            if (bad) atomicOr(status, MKV_DEV_BAD_N_KEEP);
            else if (kept != nk) atomicOr(status, MKV_DEV_INTERNAL);
            if (kept_out) kept_out[head] = kept;
        }
    }
}

// ------------------------------------------------ a4 + a5: compact, gather --

// Item = (head, chunk of 4096 tokens). Each thread classifies 16 consecutive
// tokens against the cut; two CTA scans give each kept token its tie rank and
// its output slot; kept token ids go to shared memory (and idx), then
// half-warps copy the kept K and V rows, 16 bytes per lane.
__global__ void __launch_bounds__(kStreamThreads)
k_compact_gather(const float *__restrict__ S, const mkv_cut *__restrict__ cuts,
                 const int2 *__restrict__ chunk_info, const int32_t *__restrict__ seq_lens, int heads,
                 int t_max, int nch_max, int keep_stride, int64_t n_items, int32_t *__restrict__ idx,
                 const uint8_t *__restrict__ K, const uint8_t *__restrict__ V, uint8_t *__restrict__ K_out,
                 uint8_t *__restrict__ V_out, uint32_t *status)
{
    __shared__ int32_t tok[kCompactChunk];
    __shared__ uint32_t s_warp[kStreamThreads / 32];
    const int hw = threadIdx.x >> 4, l16 = threadIdx.x & 15;
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int64_t head = item / nch_max;
        const int c = (int)(item - head * nch_max);
        const int T = head_len(seq_lens, head, heads, t_max, status, false);
        const int a = c * kCompactChunk;
        if (a >= T) continue;
        const mkv_cut cut = cuts[head];
        if (cut.key == kNoneKey && cut.ties == 0) continue;
        const int2 info = chunk_info[head * nch_max + c];
        // Offsets of a skipped head are {-1, -1}; anything else outside
        // [0, keep_stride] cannot come from the offsets pass and is refused.
        if (info.x < 0 || info.x > keep_stride || info.y < 0) {
            if (threadIdx.x == 0 && info.x != -1) atomicOr(status, MKV_DEV_INTERNAL);
            continue;
        }
        const float *srow = S + (size_t)head * t_max;
        const int t0 = a + threadIdx.x * 16;
        uint32_t gtm = 0, eqm = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int t = t0 + j;
            if (t < T) {
                const uint32_t u = score_key(srow[t]);
                gtm |= (uint32_t)(u > cut.key) << j;
                eqm |= (uint32_t)(u == cut.key) << j;
            }
        }
        uint32_t rank = (uint32_t)info.y + block_exclusive_scan<kStreamThreads>(__popc(eqm), s_warp, nullptr);
        uint32_t keepm = gtm;
        for (uint32_t m = eqm; m; m &= m - 1) {
            if (rank < (uint32_t)cut.ties) keepm |= m & (~m + 1);
            ++rank;
        }
        uint32_t n_chunk = 0;
        const uint32_t kb = block_exclusive_scan<kStreamThreads>(__popc(keepm), s_warp, &n_chunk);
        int32_t *idx_head = idx ? idx + head * keep_stride : nullptr;
        uint32_t r = kb;
        for (uint32_t m = keepm; m; m &= m - 1, ++r) {
            const int t = t0 + __ffs(m) - 1;
            tok[r] = t;
            const int64_t slot = (int64_t)info.x + r;
            if (slot >= 0 && slot < keep_stride) {
                if (idx_head) idx_head[slot] = t;
            } else {
                atomicOr(status, MKV_DEV_INTERNAL);
            }
        }
        __syncthreads();
        if (K_out) {
            const size_t in_head = (size_t)head * t_max * kRowBytes + l16 * 16;
            const size_t out_head = ((size_t)head * keep_stride + info.x) * kRowBytes + l16 * 16;
            const int n_rows = (int)min((int64_t)n_chunk, (int64_t)keep_stride - info.x);
            for (int j0 = 0; j0 < n_rows; j0 += kSlots * kUnroll) {
                uint4 kv[kUnroll], vv[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int j = j0 + u * kSlots + hw;
                    if (j < n_rows) {
                        const size_t off = in_head + (size_t)tok[j] * kRowBytes;
                        kv[u] = ld_stream(K + off);
                        vv[u] = ld_stream(V + off);
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int j = j0 + u * kSlots + hw;
                    if (j < n_rows) {
                        const size_t off = out_head + (size_t)j * kRowBytes;
                        st_v4(K_out + off, kv[u]);
                        st_v4(V_out + off, vv[u]);
                    }
                }
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------- occupancy --

// Resident CTAs per SM of a kernel on the current device, cached per
// (kernel, device); the grid is that times the SM count (capped by the number
// of work items), and kernels loop over their items.
struct OccEntry {
    const void *fn;
    int dev;
    int per_sm;
};

int resident_per_sm(const void *fn, int threads, int dev)
{
    static std::mutex mu;
    static OccEntry table[64];
    static int used = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (table[i].fn == fn && table[i].dev == dev) return table[i].per_sm;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    if (used < 64) table[used++] = OccEntry{fn, dev, per_sm};
    return per_sm;
}

int sm_count(int dev)
{
    static std::mutex mu;
    static int sms[64] = {0};
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return 1;
    if (sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
        sms[dev] = n;
    }
    return sms[dev];
}

template <typename Kern>
int grid_for(Kern kernel, int threads, int64_t items)
{
    int dev = 0;
    cudaGetDevice(&dev);
    const int64_t full = (int64_t)sm_count(dev) * resident_per_sm(reinterpret_cast<const void *>(kernel), threads, dev);
    return (int)(items < full ? (items > 0 ? items : 1) : full);
}

}  // namespace

// ------------------------------------------------------------- launchers --

cudaError_t launch_centroid_partial(const Geometry &g, const void *K, const int32_t *seq_lens,
                                    float *partial, uint32_t *status, cudaStream_t st)
{
    const int64_t items = g.n_heads * g.nwin_max * (int64_t)g.ppw;
    if (items == 0) return cudaSuccess;
    const int grid = grid_for(k_centroid_partial, kStreamThreads, items);
    k_centroid_partial<<<grid, kStreamThreads, 0, st>>>(static_cast<const uint8_t *>(K), seq_lens, g.heads,
                                                         g.t_max, g.window, g.nwin_max, g.piece, g.ppw,
                                                         items, partial, status);
    return cudaGetLastError();
}

cudaError_t launch_centroid_finalize(const Geometry &g, const float *partial, const int32_t *seq_lens,
                                     float *C, uint32_t *status, cudaStream_t st)
{
    const int64_t items = g.n_heads * g.nwin_max;
    if (items == 0) return cudaSuccess;
    const int64_t blocks = (items + 7) / 8;
    k_centroid_finalize<<<(unsigned)blocks, 256, 0, st>>>(partial, seq_lens, g.heads, g.t_max, g.window,
                                                          g.nwin_max, g.piece, g.ppw, items, C, status);
    return cudaGetLastError();
}

cudaError_t launch_score(const Geometry &g, const void *K, const float *C, const int32_t *seq_lens,
                         int mode, float *S, uint32_t *status, cudaStream_t st)
{
    const int nch = (g.t_max + g.score_chunk - 1) / g.score_chunk;
    const int64_t items = g.n_heads * nch;
    if (items == 0) return cudaSuccess;
    if (mode == MKV_MODE_L2) {
        const int grid = grid_for(k_score<MKV_MODE_L2>, kStreamThreads, items);
        k_score<MKV_MODE_L2><<<grid, kStreamThreads, 0, st>>>(static_cast<const uint8_t *>(K), C, seq_lens,
                                                              g.heads, g.t_max, g.window, g.nwin_max,
                                                              g.score_chunk, nch, items, S, status);
    } else {
        const int grid = grid_for(k_score<MKV_MODE_COSINE>, kStreamThreads, items);
        k_score<MKV_MODE_COSINE><<<grid, kStreamThreads, 0, st>>>(static_cast<const uint8_t *>(K), C,
                                                                  seq_lens, g.heads, g.t_max, g.window,
                                                                  g.nwin_max, g.score_chunk, nch, items, S,
                                                                  status);
    }
    return cudaGetLastError();
}

cudaError_t launch_select(const Geometry &g, const float *S, const int32_t *seq_lens, double ratio,
                          const int32_t *n_keep, int32_t keep_stride, mkv_cut *cut, int2 *chunk_info,
                          int32_t *kept, uint32_t *status, cudaStream_t st)
{
    if (g.n_heads == 0) return cudaSuccess;
    const int grid = grid_for(k_select, kSelectThreads, g.n_heads);
    k_select<<<grid, kSelectThreads, 0, st>>>(S, seq_lens, g.heads, g.t_max, ratio, n_keep, keep_stride,
                                              g.n_heads, cut, chunk_info, g.nch, kept, status);
    return cudaGetLastError();
}

cudaError_t launch_chunk_offsets(const Geometry &g, const float *S, const mkv_cut *cut,
                                 const int32_t *seq_lens, double ratio, const int32_t *n_keep,
                                 int32_t keep_stride, int2 *chunk_info, int32_t *kept,
                                 uint32_t *status, cudaStream_t st)
{
    if (g.n_heads == 0) return cudaSuccess;
    const int grid = grid_for(k_chunk_offsets, kSelectThreads, g.n_heads);
    k_chunk_offsets<<<grid, kSelectThreads, 0, st>>>(S, cut, seq_lens, g.heads, g.t_max, ratio, n_keep,
                                                     keep_stride, g.n_heads, chunk_info, g.nch, kept,
                                                     status);
    return cudaGetLastError();
}

cudaError_t launch_compact_gather(const Geometry &g, const float *S, const mkv_cut *cut,
                                  const int2 *chunk_info, const int32_t *seq_lens, int32_t keep_stride,
                                  int32_t *idx, const void *K, const void *V, void *K_out, void *V_out,
                                  uint32_t *status, cudaStream_t st)
{
    const int64_t items = g.n_heads * g.nch;
    if (items == 0) return cudaSuccess;
    const int grid = grid_for(k_compact_gather, kStreamThreads, items);
    k_compact_gather<<<grid, kStreamThreads, 0, st>>>(
        S, cut, chunk_info, seq_lens, g.heads, g.t_max, g.nch, keep_stride, items, idx,
        static_cast<const uint8_t *>(K), static_cast<const uint8_t *>(V), static_cast<uint8_t *>(K_out),
        static_cast<uint8_t *>(V_out), status);
    return cudaGetLastError();
}

}  // namespace mkv
