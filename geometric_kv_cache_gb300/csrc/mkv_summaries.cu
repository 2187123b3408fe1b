// sm_103a cluster summaries: per-window means of a cache (keys or values,
// bf16 or E4M3) for short windows, with each window's radius.
//
// "RefineKV: Query-Adaptive KV Cache Compression via Attention-Error Bounds"
// (project page), method overview, step 1 (Summarize): the cache is cut
// into contiguous clusters (10 keys in its Figure 2), and each cluster's
// mean key and mean value are cached with metadata. Here the clusters are
// the windows [jW, min((j+1)W, T)), and the radius max_t |x_t - mean|_2 is
// the metadata a query-time bound on logit deviation needs
// (|q.k_t - q.mean| <= |q| radius). Longer windows use the piece kernels of
// the centroid step (mkv_piece.cu) instead.
//
// Layout: one window per 8-lane group. Lane q of a group owns dims
// [64k + 8q, 64k + 8q + 8) of every row for k < d/64 (one 16-byte load per
// 64 bf16 dims, 8-byte for E4M3, each group reading whole lines). Sums run
// per dim in token order in fp32, so no lane talks to another for the mean.
// The radius sums each row's squared offsets per lane, then over the group
// with an xor butterfly (the same bits on every lane). Windows of at most 16
// rows keep their rows in registers from the mean to the radius
// (k_small_window_regs); longer ones re-read them from L1/L2
// (k_small_window_means). Both give the same bits.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mkv_device.cuh"
#include "mkv_internal.h"

namespace mkv {
namespace {

constexpr int kSumThreads = 256;
constexpr int kWindowsPerCta = kSumThreads / 8;
constexpr int kBatchRows = 4;  // rows in flight per lane
using namespace dev;

// This lane's NB chunks of 8 elements of a row (chunk k at element 64k of
// the lane's first chunk).
template <int NB, int ES>
__device__ __forceinline__ void load_row(const uint8_t *row, typename Chunk<ES>::raw (&v)[NB])
{
#pragma unroll
    for (int k = 0; k < NB; ++k) v[k] = Chunk<ES>::load_l1(row + 64 * ES * k);
}

// Lane q of a window's group owns dims [64k + 8q, 64k + 8q + 8), k < NB
// (head dim 64 NB).
template <int NB, int ES>
__global__ void __launch_bounds__(kSumThreads)
k_small_window_means(const uint8_t *__restrict__ X, const int32_t *__restrict__ seq_lens, int heads, int t_max,
                     int window, int nwin_max, int64_t n_items, float *__restrict__ mean,
                     float *__restrict__ radius, uint32_t *status)
{
    constexpr int D = 64 * NB, RB = ES * D;
    using Raw = typename Chunk<ES>::raw;
    const int grp = threadIdx.x >> 3, q = threadIdx.x & 7;
    for (int64_t base = (int64_t)blockIdx.x * kWindowsPerCta; base < n_items;
         base += (int64_t)gridDim.x * kWindowsPerCta) {
        const int64_t item = base + grp;
        int n = 0;
        int64_t head = 0;
        int j = 0;
        if (item < n_items) {
            head = item / nwin_max;
            j = (int)(item - head * nwin_max);
            const int T = head_len(seq_lens, head, heads, t_max, status, q == 0 && j == 0);
            n = min(window, T - j * window);
        }
        const uint8_t *row0 = X + ((size_t)head * t_max + (size_t)j * window) * RB + q * 8 * ES;
        float m[8 * NB] = {0.f};
        if (n > 0) {
            float acc[8 * NB];
#pragma unroll
            for (int i = 0; i < 8 * NB; ++i) acc[i] = 0.f;
            for (int t0 = 0; t0 < n; t0 += kBatchRows) {
                Raw v[kBatchRows][NB];
#pragma unroll
                for (int u = 0; u < kBatchRows; ++u)
                    if (t0 + u < n) load_row<NB, ES>(row0 + (size_t)(t0 + u) * RB, v[u]);
#pragma unroll
                for (int u = 0; u < kBatchRows; ++u) {
                    if (t0 + u < n) {
#pragma unroll
                        for (int k = 0; k < NB; ++k) {
                            float f[8];
                            Chunk<ES>::to_f32(v[u][k], f);
#pragma unroll
                            for (int i = 0; i < 8; ++i) acc[8 * k + i] += f[i];
                        }
                    }
                }
            }
            const float fn = (float)n;
#pragma unroll
            for (int i = 0; i < 8 * NB; ++i) m[i] = __fdiv_rn(acc[i], fn);
            float4 *out = reinterpret_cast<float4 *>(mean + ((size_t)head * nwin_max + j) * D);
#pragma unroll
            for (int k = 0; k < NB; ++k) {
                out[16 * k + 2 * q] = make_float4(m[8 * k], m[8 * k + 1], m[8 * k + 2], m[8 * k + 3]);
                out[16 * k + 2 * q + 1] = make_float4(m[8 * k + 4], m[8 * k + 5], m[8 * k + 6], m[8 * k + 7]);
            }
        }
        if (radius) {
            // every lane of the warp runs the same rows (the butterfly below
            // needs all 32), rows past a group's window count as nothing
            const int n_warp = __reduce_max_sync(kFull, (unsigned)max(n, 0));
            float rmax = 0.f;
            for (int t0 = 0; t0 < n_warp; t0 += kBatchRows) {
                Raw v[kBatchRows][NB];
#pragma unroll
                for (int u = 0; u < kBatchRows; ++u)
                    if (t0 + u < n) load_row<NB, ES>(row0 + (size_t)(t0 + u) * RB, v[u]);
#pragma unroll
                for (int u = 0; u < kBatchRows; ++u) {
                    float ss = 0.f;
                    if (t0 + u < n) {
#pragma unroll
                        for (int k = 0; k < NB; ++k) {
                            float f[8];
                            Chunk<ES>::to_f32(v[u][k], f);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float dlt = f[i] - m[8 * k + i];
                                ss = fmaf(dlt, dlt, ss);
                            }
                        }
                    }
                    ss += __shfl_xor_sync(kFull, ss, 1);
                    ss += __shfl_xor_sync(kFull, ss, 2);
                    ss += __shfl_xor_sync(kFull, ss, 4);
                    if (t0 + u < n) rmax = fmaxf(rmax, sqrtf(ss));
                }
            }
            if (n > 0 && q == 0) radius[(size_t)head * nwin_max + j] = rmax;
        }
    }
}

// The same per window, for windows of at most MR rows: the group issues all
// of its window's row loads at once and keeps the rows in registers for the
// radius, so every row is read once and each window costs one memory round
// trip. Same arithmetic in the same order as k_small_window_means.
template <int NB, int ES, int MR>
__global__ void __launch_bounds__(kSumThreads)
k_small_window_regs(const uint8_t *__restrict__ X, const int32_t *__restrict__ seq_lens, int heads, int t_max,
                    int window, int nwin_max, int64_t n_items, float *__restrict__ mean,
                    float *__restrict__ radius, uint32_t *status)
{
    constexpr int D = 64 * NB, RB = ES * D;
    using Raw = typename Chunk<ES>::raw;
    const int grp = threadIdx.x >> 3, q = threadIdx.x & 7;
    for (int64_t base = (int64_t)blockIdx.x * kWindowsPerCta; base < n_items;
         base += (int64_t)gridDim.x * kWindowsPerCta) {
        const int64_t item = base + grp;
        int n = 0;
        int64_t head = 0;
        int j = 0;
        if (item < n_items) {
            head = item / nwin_max;
            j = (int)(item - head * nwin_max);
            const int T = head_len(seq_lens, head, heads, t_max, status, q == 0 && j == 0);
            n = min(window, T - j * window);
        }
        const uint8_t *row0 = X + ((size_t)head * t_max + (size_t)j * window) * RB + q * 8 * ES;
        Raw v[MR][NB];
#pragma unroll
        for (int u = 0; u < MR; ++u)
            if (u < n) load_row<NB, ES>(row0 + (size_t)u * RB, v[u]);
        float m[8 * NB];
        {
            float acc[8 * NB];
#pragma unroll
            for (int i = 0; i < 8 * NB; ++i) acc[i] = 0.f;
#pragma unroll
            for (int u = 0; u < MR; ++u)
                if (u < n)
#pragma unroll
                    for (int k = 0; k < NB; ++k) Chunk<ES>::add_to(v[u][k], acc + 8 * k);
            const float fn = (float)max(n, 1);
#pragma unroll
            for (int i = 0; i < 8 * NB; ++i) m[i] = __fdiv_rn(acc[i], fn);
        }
        if (n > 0) {
            float4 *out = reinterpret_cast<float4 *>(mean + ((size_t)head * nwin_max + j) * D);
#pragma unroll
            for (int k = 0; k < NB; ++k) {
                out[16 * k + 2 * q] = make_float4(m[8 * k], m[8 * k + 1], m[8 * k + 2], m[8 * k + 3]);
                out[16 * k + 2 * q + 1] = make_float4(m[8 * k + 4], m[8 * k + 5], m[8 * k + 6], m[8 * k + 7]);
            }
        }
        if (radius) {
            // all 32 lanes run every row slot (the butterfly needs them);
            // rows past a group's window count as nothing
            float rmax = 0.f;
#pragma unroll
            for (int u = 0; u < MR; ++u) {
                float ss = 0.f;
                if (u < n) {
#pragma unroll
                    for (int k = 0; k < NB; ++k) {
                        float dlt[8];
                        Chunk<ES>::sub_from(v[u][k], m + 8 * k, dlt);
#pragma unroll
                        for (int i = 0; i < 8; ++i) ss = fmaf(dlt[i], dlt[i], ss);
                    }
                }
                ss += __shfl_xor_sync(kFull, ss, 1);
                ss += __shfl_xor_sync(kFull, ss, 2);
                ss += __shfl_xor_sync(kFull, ss, 4);
                if (u < n) rmax = fmaxf(rmax, sqrtf(ss));
            }
            if (n > 0 && q == 0) radius[(size_t)head * nwin_max + j] = rmax;
        }
    }
}

// Row capacities of the register-resident kernel: the smallest that holds
// the window is taken (10 is RefineKV's cluster size), as long as a lane's
// share of the rows takes at most 128 registers.
template <int NB, int ES, int MR>
constexpr bool regs_fit() { return MR * NB * (ES == 2 ? 4 : 2) <= 128; }

template <int NB, int ES, int MR>
const void *regs_instance()
{
    if constexpr (regs_fit<NB, ES, MR>()) return (const void *)k_small_window_regs<NB, ES, MR>;
    else return nullptr;
}

template <int ES, int MR>
const void *small_window_regs_fn_es(int d)
{
    switch (d) {
    case 64: return regs_instance<1, ES, MR>();
    case 128: return regs_instance<2, ES, MR>();
    case 256: return regs_instance<4, ES, MR>();
    default: return nullptr;
    }
}

template <int MR>
const void *small_window_regs_fn_mr(int d, int es)
{
    return es == 2 ? small_window_regs_fn_es<2, MR>(d) : es == 1 ? small_window_regs_fn_es<1, MR>(d) : nullptr;
}

// The register-resident kernel for windows of at most `window` rows, or null.
const void *small_window_regs_fn(int d, int es, int window)
{
    if (window <= 0) return nullptr;
    if (window <= 8) return small_window_regs_fn_mr<8>(d, es);
    if (window <= 10) return small_window_regs_fn_mr<10>(d, es);
    if (window <= 16) return small_window_regs_fn_mr<16>(d, es);
    return nullptr;
}

template <int ES>
const void *small_window_means_fn_es(int d)
{
    switch (d) {
    case 64: return (const void *)k_small_window_means<1, ES>;
    case 128: return (const void *)k_small_window_means<2, ES>;
    case 256: return (const void *)k_small_window_means<4, ES>;
    default: return nullptr;
    }
}

const void *small_window_means_fn(int d, int es)
{
    return es == 2 ? small_window_means_fn_es<2>(d) : es == 1 ? small_window_means_fn_es<1>(d) : nullptr;
}

}  // namespace

cudaError_t launch_small_window_means(const PieceGeometry &g, const void *X, const int32_t *seq_lens, float *mean,
                                      float *radius, uint32_t *status, cudaStream_t st)
{
    const int64_t items = g.n_heads * g.nwin_max;
    if (items == 0) return cudaSuccess;
    const void *fn = small_window_regs_fn(g.d, g.es, g.window);
    if (!fn) fn = small_window_means_fn(g.d, g.es);
    if (!fn) return cudaErrorInvalidValue;
    const int grid = grid_for_items(fn, kSumThreads, 0, (items + kWindowsPerCta - 1) / kWindowsPerCta);
    const uint8_t *Xb = static_cast<const uint8_t *>(X);
    int heads = g.heads, t_max = g.t_max, window = g.window, nwin_max = g.nwin_max;
    int64_t n_items = items;
    void *args[] = {&Xb, &seq_lens, &heads, &t_max, &window, &nwin_max, &n_items, &mean, &radius, &status};
    return cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(kSumThreads), args, 0, st);
}

}  // namespace mkv
