// sm_103a gather of the kept K/V rows (the last step of the ManifoldKV-style
// compression path: the retained tokens form the compressed cache, "ManifoldKV:
// Training-Free KV Cache Compression via Euclidean Outlier Detection", ICML 2026
// poster 62526, abstract).
//
// K_out[h][j] = K[h][idx[h][j]] and V_out likewise, bit copies. This is the
// path's dominant kernel (8 bytes per kept element of K and V read and
// written), a plain HBM-bound copy: 16-byte non-coherent loads, streaming
// (evict-first) stores, a persistent grid over (head, 64-slot) items.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mkv_device.cuh"
#include "mkv_internal.h"

namespace mkv {
namespace {

constexpr int kStreamThreads = 256;
constexpr int kSlots = kStreamThreads / 16;    // rows per CTA per load step
using namespace dev;

// Item = (head, block of 64 output slots). Half-warps copy rows, 16 bytes per
// lane: K_out[h][j] = K[h][idx[h][j]], V_out likewise, for j < kept[h]; four
// rows of K and of V in flight per lane. No CTA barrier anywhere.
constexpr int kGatherRows = 64;

__global__ void __launch_bounds__(kStreamThreads)
k_gather_rows(const int32_t *__restrict__ idx, int idx_stride, const int32_t *__restrict__ kept, int t_max,
              int keep_stride, int blocks_per_head, int64_t n_items, const uint8_t *__restrict__ K,
              const uint8_t *__restrict__ V, uint8_t *__restrict__ K_out, uint8_t *__restrict__ V_out,
              uint32_t *status)
{
    const int hw = threadIdx.x >> 4, l16 = threadIdx.x & 15;
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int64_t head = item / blocks_per_head;
        const int j0 = (int)(item - head * blocks_per_head) * kGatherRows;
        const int n = min(kGatherRows, min(kept[head], keep_stride) - j0);
        if (n <= 0) continue;
        const int32_t *ih = idx + head * idx_stride + j0;
        const size_t in_head = (size_t)head * t_max * kRowBytes + l16 * 16;
        const size_t out_head = ((size_t)head * keep_stride + j0) * kRowBytes + l16 * 16;
        uint4 kv[kGatherRows / kSlots], vv[kGatherRows / kSlots];
        int src[kGatherRows / kSlots];
#pragma unroll
        for (int u = 0; u < kGatherRows / kSlots; ++u) {
            const int j = u * kSlots + hw;
            src[u] = j < n ? ih[j] : -1;
            if (src[u] >= t_max) {
                atomicOr(status, MKV_DEV_INTERNAL);
                src[u] = -1;
            }
        }
#pragma unroll
        for (int u = 0; u < kGatherRows / kSlots; ++u) {
            if (src[u] >= 0) {
                const size_t off = in_head + (size_t)src[u] * kRowBytes;
                kv[u] = ld_stream(K + off);
                vv[u] = ld_stream(V + off);
            }
        }
#pragma unroll
        for (int u = 0; u < kGatherRows / kSlots; ++u) {
            if (src[u] >= 0) {
                const size_t off = out_head + (size_t)(u * kSlots + hw) * kRowBytes;
                st_stream(K_out + off, kv[u]);
                st_stream(V_out + off, vv[u]);
            }
        }
    }
}

}  // namespace

cudaError_t launch_gather(const Geometry &g, const int32_t *idx, int32_t idx_stride, const int32_t *kept,
                          int32_t keep_stride, const void *K, const void *V, void *K_out, void *V_out,
                          uint32_t *status, cudaStream_t st)
{
    const int bph = (keep_stride + kGatherRows - 1) / kGatherRows;
    const int64_t items = g.n_heads * bph;
    if (items == 0) return cudaSuccess;
    const int grid = grid_for_items(reinterpret_cast<const void *>(k_gather_rows), kStreamThreads, 0, items);
    k_gather_rows<<<grid, kStreamThreads, 0, st>>>(idx, idx_stride, kept, g.t_max, keep_stride, bph, items,
                                                   static_cast<const uint8_t *>(K), static_cast<const uint8_t *>(V),
                                                   static_cast<uint8_t *>(K_out), static_cast<uint8_t *>(V_out),
                                                   status);
    return cudaGetLastError();
}

}  // namespace mkv
