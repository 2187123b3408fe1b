// sm_103a in-place compaction: the kept K/V rows of every head are moved to
// the front of the head's own rows (the memory-saving form of the gather
// that ends the ManifoldKV-style path: the retained tokens form the
// compressed cache, "ManifoldKV: Training-Free KV Cache Compression via
// Euclidean Outlier Detection", ICML 2026 poster 62526, abstract).
#include <cuda_runtime.h>
#include <stdint.h>

#include "mkv_device.cuh"
#include "mkv_internal.h"

namespace mkv {
namespace {

constexpr int kStreamThreads = 256;
using namespace dev;

// ----------------------------------------------------------- in place --

// 16-byte load through L2 only: the rows read here are written by the same
// kernel, so the non-coherent (read-only) path must not be used.
__device__ __forceinline__ uint4 ld_cg(const void *p)
{
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p)
                 : "memory");
    return r;
}

constexpr int kInplaceRows = 64;  // output slots per chunk

// One chunk of a lane group's rows: R rows of K and V, their destinations.
template <int R>
struct MoveChunk {
    uint4 k[R], v[R];
    int dst[R];  // destination row, or -1 (no slot, or the row is already in place)
};

// Groups of LPR lanes (16 bytes each) cover a row of RB = 16 LPR bytes.
template <int LPR>
__device__ __forceinline__ void inplace_load(MoveChunk<kInplaceRows * LPR / kStreamThreads> &c, int chunk, int n, int T,
                                             const int32_t *ih, const uint8_t *Kh, const uint8_t *Vh, int hw,
                                             uint32_t *status)
{
    constexpr int RB = LPR * 16, SLOTS = kStreamThreads / LPR, R = kInplaceRows / SLOTS;
#pragma unroll
    for (int u = 0; u < R; ++u) {
        const int j = chunk * kInplaceRows + u * SLOTS + hw;
        c.dst[u] = -1;
        if (j < n) {
            const int src = ih[j];
            if (src < j || src >= T) {
                atomicOr(status, MKV_DEV_INTERNAL);  // not an ascending index list: the move would be unsafe
            } else if (src != j) {
                c.dst[u] = j;
                c.k[u] = ld_cg(Kh + (size_t)src * RB);
                c.v[u] = ld_cg(Vh + (size_t)src * RB);
            }
        }
    }
}

template <int LPR>
__device__ __forceinline__ void inplace_store(const MoveChunk<kInplaceRows * LPR / kStreamThreads> &c, uint8_t *Kh,
                                              uint8_t *Vh)
{
    constexpr int RB = LPR * 16, R = kInplaceRows * LPR / kStreamThreads;
#pragma unroll
    for (int u = 0; u < R; ++u) {
        if (c.dst[u] >= 0) {
            st_stream(Kh + (size_t)c.dst[u] * RB, c.k[u]);
            st_stream(Vh + (size_t)c.dst[u] * RB, c.v[u]);
        }
    }
}

// In-place compaction: row j of each head becomes row idx[j] (j < kept), in
// the head's own K and V rows. Row r is read by at most one slot j <= r
// (idx ascends from 0, so idx[j] >= j) and written by slot r, so walking the
// slots in chunks of 64 in ascending order is safe when chunk c's loads are
// performed before chunk c's stores (a CTA barrier between them): every
// earlier reader of a row chunk c overwrites sits in chunk c or before. The
// loads of chunk c+1 read rows at or beyond its own slots, which no earlier
// chunk writes, so they are issued before chunk c's stores (two chunks in
// flight). One CTA walks one head; heads are spread over the persistent grid.
template <int LPR>
__global__ void __launch_bounds__(kStreamThreads)
k_gather_inplace(const int32_t *__restrict__ idx, int idx_stride, const int32_t *__restrict__ kept,
                 const int32_t *__restrict__ seq_lens, int heads, int t_max, int64_t n_heads, uint8_t *K, uint8_t *V,
                 uint32_t *status)
{
    constexpr int RB = LPR * 16, R = kInplaceRows * LPR / kStreamThreads;
    const int hw = threadIdx.x / LPR, lr = threadIdx.x % LPR;
    for (int64_t head = blockIdx.x; head < n_heads; head += gridDim.x) {
        const int T = head_len(seq_lens, head, heads, t_max, status, false);
        const int n = min(kept[head], T);
        if (n <= 0) continue;  // the same for every thread
        const int32_t *ih = idx + head * idx_stride;
        uint8_t *Kh = K + (size_t)head * t_max * RB + lr * 16;
        uint8_t *Vh = V + (size_t)head * t_max * RB + lr * 16;
        const int nch = (n + kInplaceRows - 1) / kInplaceRows;
        MoveChunk<R> a, b;
        inplace_load<LPR>(a, 0, n, T, ih, Kh, Vh, hw, status);
        for (int c = 0; c < nch; c += 2) {
            __syncthreads();  // chunk c's loads are performed CTA-wide
            if (c + 1 < nch) inplace_load<LPR>(b, c + 1, n, T, ih, Kh, Vh, hw, status);
            inplace_store<LPR>(a, Kh, Vh);
            if (c + 1 >= nch) break;
            __syncthreads();  // chunk c+1's loads are performed CTA-wide
            if (c + 2 < nch) inplace_load<LPR>(a, c + 2, n, T, ih, Kh, Vh, hw, status);
            inplace_store<LPR>(b, Kh, Vh);
        }
        __syncthreads();  // the next head starts with every store of this one issued
    }
}

// The kernel for a row of `row_bytes` bytes (head dim x element size).
const void *inplace_fn(int row_bytes)
{
    switch (row_bytes) {
    case 64: return (const void *)k_gather_inplace<4>;
    case 128: return (const void *)k_gather_inplace<8>;
    case 256: return (const void *)k_gather_inplace<16>;
    case 512: return (const void *)k_gather_inplace<32>;
    default: return nullptr;
    }
}

}  // namespace

cudaError_t launch_gather_inplace(const Geometry &g, const int32_t *idx, int32_t idx_stride, const int32_t *kept,
                                  const int32_t *seq_lens, void *K, void *V, uint32_t *status, cudaStream_t st)
{
    if (g.n_heads == 0) return cudaSuccess;
    const void *fn = inplace_fn(g.d * g.es);
    if (!fn) return cudaErrorInvalidValue;
    const int grid = grid_for_items(fn, kStreamThreads, 0, g.n_heads);
    int heads = g.heads, t_max = g.t_max;
    int64_t n_heads = g.n_heads;
    uint8_t *Kb = static_cast<uint8_t *>(K), *Vb = static_cast<uint8_t *>(V);
    void *args[] = {&idx, &idx_stride, &kept, &seq_lens, &heads, &t_max, &n_heads, &Kb, &Vb, &status};
    return cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(kStreamThreads), args, 0, st);
}

}  // namespace mkv
