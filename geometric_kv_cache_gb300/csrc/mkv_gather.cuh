// One item of the K/V row gather (a5) as a device function, called by the
// gather kernel and by the fused whole-path kernel: K_out[h][j] =
// K[h][idx[h][j]] and V_out likewise, bit copies.
//
// Method: "ManifoldKV: Training-Free KV Cache Compression via Euclidean
// Outlier Detection" (ICML 2026 poster 62526), abstract -- the retained
// tokens form the compressed cache.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "mkv_device.cuh"
#include "mkv_internal.h"

namespace mkv {
namespace {

constexpr int kGatherThreads = 256;  // threads of a CTA that runs gather items
using namespace dev;

// Item = (head, block of 64 output slots). Groups of LPR lanes (LPR = row
// bytes / 16: 16 bytes per lane) copy rows: K_out[h][j] = K[h][idx[h][j]], V_out
// likewise, for j < kept[h]; 64 / (256 / LPR) rows of K and of V in flight
// per lane. No CTA barrier anywhere.
constexpr int kGatherRows = 64;

// One item of ROWS output slots; COHERENT reads the indices and kept counts
// through L2 only (__ldcg), for indices written earlier in the same launch.
template <int LPR, bool COHERENT, int ROWS = kGatherRows>
__device__ __forceinline__ void gather_item(int64_t item, const int32_t *idx, int idx_stride, const int32_t *kept,
                                            int t_max, int keep_stride, int blocks_per_head,
                                            const uint8_t *__restrict__ K, const uint8_t *__restrict__ V,
                                            uint8_t *__restrict__ K_out, uint8_t *__restrict__ V_out, uint32_t *status)
{
    constexpr int RB = LPR * 16;                 // row bytes
    constexpr int SLOTS = kGatherThreads / LPR;  // rows per CTA per load step
    constexpr int R = ROWS / SLOTS;       // rows per lane group
    const int hw = threadIdx.x / LPR, lr = threadIdx.x % LPR;
    {
        const int64_t head = item / blocks_per_head;
        const int j0 = (int)(item - head * blocks_per_head) * ROWS;
        const int kh = COHERENT ? __ldcg(kept + head) : kept[head];
        const int n = min(ROWS, min(kh, keep_stride) - j0);
        if (n <= 0) return;
        const int32_t *ih = idx + head * idx_stride + j0;
        const size_t in_head = (size_t)head * t_max * RB + lr * 16;
        const size_t out_head = ((size_t)head * keep_stride + j0) * RB + lr * 16;
        uint4 kv[R], vv[R];
        int src[R];
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const int j = u * SLOTS + hw;
            src[u] = j < n ? (COHERENT ? __ldcg(ih + j) : ih[j]) : -1;
            if (src[u] >= t_max) {
                atomicOr(status, MKV_DEV_INTERNAL);
                src[u] = -1;
            }
        }
#pragma unroll
        for (int u = 0; u < R; ++u) {
            if (src[u] >= 0) {
                const size_t off = in_head + (size_t)src[u] * RB;
                kv[u] = ld_stream(K + off);
                vv[u] = ld_stream(V + off);
            }
        }
#pragma unroll
        for (int u = 0; u < R; ++u) {
            if (src[u] >= 0) {
                const size_t off = out_head + (size_t)(u * SLOTS + hw) * RB;
                st_v4(K_out + off, kv[u]);
                st_v4(V_out + off, vv[u]);
            }
        }
    }
}

}  // namespace
}  // namespace mkv
