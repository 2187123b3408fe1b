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
#include "mkv_gather.cuh"

namespace mkv {
namespace {

constexpr int kStreamThreads = kGatherThreads;
using namespace dev;

// gather_item (one (head, 64-slot) item) is in mkv_gather.cuh.
template <int LPR>
__global__ void __launch_bounds__(kStreamThreads)
k_gather_rows(const int32_t *__restrict__ idx, int idx_stride, const int32_t *__restrict__ kept, int t_max,
              int keep_stride, int blocks_per_head, int64_t n_items, const uint8_t *__restrict__ K,
              const uint8_t *__restrict__ V, uint8_t *__restrict__ K_out, uint8_t *__restrict__ V_out,
              uint32_t *status)
{
    pdl_wait();  // the indices of the previous kernel are complete
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x)
        gather_item<LPR, false>(item, idx, idx_stride, kept, t_max, keep_stride, blocks_per_head, K, V, K_out, V_out,
                                status);
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
