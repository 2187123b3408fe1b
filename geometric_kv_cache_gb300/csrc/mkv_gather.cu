// sm_103a gather of the kept K/V rows (the last step of the ManifoldKV-style
// compression path: the retained tokens form the compressed cache, "ManifoldKV:
// Training-Free KV Cache Compression via Euclidean Outlier Detection", ICML 2026
// poster 62526, abstract).
//
// K_out[h][j] = K[h][idx[h][j]] and V_out likewise, bit copies. This is the
// path's dominant kernel (8 bytes per kept element of K and V read and
// written), a plain HBM-bound copy: 16-byte non-coherent loads, plain
// 16-byte stores (measured 1.5% faster here than evict-first streaming
// stores), a persistent grid over (head, 64-slot) items.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mkv_device.cuh"
#include "mkv_internal.h"

namespace mkv {
namespace {

constexpr int kStreamThreads = 256;
using namespace dev;

// Item = (head, block of 64 output slots). Groups of LPR lanes (LPR = row
// bytes / 16: 16 bytes per lane) copy rows: K_out[h][j] = K[h][idx[h][j]], V_out
// likewise, for j < kept[h]; 64 / (256 / LPR) rows of K and of V in flight
// per lane. No CTA barrier anywhere.
constexpr int kGatherRows = 64;

template <int LPR>
__global__ void __launch_bounds__(kStreamThreads)
k_gather_rows(const int32_t *__restrict__ idx, int idx_stride, const int32_t *__restrict__ kept, int t_max,
              int keep_stride, int blocks_per_head, int64_t n_items, const uint8_t *__restrict__ K,
              const uint8_t *__restrict__ V, uint8_t *__restrict__ K_out, uint8_t *__restrict__ V_out,
              uint32_t *status)
{
    constexpr int RB = LPR * 16;                 // row bytes
    constexpr int SLOTS = kStreamThreads / LPR;  // rows per CTA per load step
    constexpr int R = kGatherRows / SLOTS;       // rows per lane group
    const int hw = threadIdx.x / LPR, lr = threadIdx.x % LPR;
    pdl_wait();  // the indices of the previous kernel are complete
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int64_t head = item / blocks_per_head;
        const int j0 = (int)(item - head * blocks_per_head) * kGatherRows;
        const int n = min(kGatherRows, min(kept[head], keep_stride) - j0);
        if (n <= 0) continue;
        const int32_t *ih = idx + head * idx_stride + j0;
        const size_t in_head = (size_t)head * t_max * RB + lr * 16;
        const size_t out_head = ((size_t)head * keep_stride + j0) * RB + lr * 16;
        uint4 kv[R], vv[R];
        int src[R];
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const int j = u * SLOTS + hw;
            src[u] = j < n ? ih[j] : -1;
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

// The kernel for a row of `row_bytes` bytes (head dim x element size).
const void *gather_fn(int row_bytes)
{
    switch (row_bytes) {
    case 64: return (const void *)k_gather_rows<4>;
    case 128: return (const void *)k_gather_rows<8>;
    case 256: return (const void *)k_gather_rows<16>;
    case 512: return (const void *)k_gather_rows<32>;
    default: return nullptr;
    }
}

}  // namespace

cudaError_t launch_gather(const Geometry &g, const int32_t *idx, int32_t idx_stride, const int32_t *kept,
                          int32_t keep_stride, const void *K, const void *V, void *K_out, void *V_out,
                          uint32_t *status, cudaStream_t st, bool pdl)
{
    const int bph = (keep_stride + kGatherRows - 1) / kGatherRows;
    const int64_t items = g.n_heads * bph;
    if (items == 0) return cudaSuccess;
    const void *fn = gather_fn(g.d * g.es);
    if (!fn) return cudaErrorInvalidValue;
    const int grid = grid_for_items(fn, kStreamThreads, 0, items);
    int t_max = g.t_max;
    int64_t n_items = items;
    int bph_arg = bph;
    const uint8_t *Kb = static_cast<const uint8_t *>(K), *Vb = static_cast<const uint8_t *>(V);
    uint8_t *Ko = static_cast<uint8_t *>(K_out), *Vo = static_cast<uint8_t *>(V_out);
    void *args[] = {&idx, &idx_stride, &kept, &t_max, &keep_stride, &bph_arg, &n_items, &Kb, &Vb, &Ko, &Vo, &status};
    // with pdl: launched as a programmatic dependent of a one-wave select
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kStreamThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace mkv
