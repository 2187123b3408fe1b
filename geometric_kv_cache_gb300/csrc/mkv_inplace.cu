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

constexpr int kMoveRows = 4;  // rows of K and of V per lane group and chunk

// One chunk of a lane group's rows: R rows of K and V, their destinations.
template <int R>
struct MoveChunk {
    uint4 k[R], v[R];
    int dst[R];  // destination row, or -1 (no slot, or the row is already in place)
};

// Groups of LPR lanes (16 bytes each) cover a row of RB = 16 LPR bytes; a
// chunk is CR = (256 / LPR) x 4 output slots (32 KB of K and V rows for
// every row size). Lane group hw takes slots u * SLOTS + hw, u < 4.
template <int LPR>
struct MoveShape {
    static constexpr int RB = LPR * 16, SLOTS = kStreamThreads / LPR, CR = SLOTS * kMoveRows;
};

// The sources of chunk c's slots for this lane group (-1 past the kept count).
template <int LPR>
__device__ __forceinline__ void move_sources(int c, int n, const int32_t *ih, int hw, int (&s)[kMoveRows])
{
    using M = MoveShape<LPR>;
#pragma unroll
    for (int u = 0; u < kMoveRows; ++u) {
        const int j = c * M::CR + u * M::SLOTS + hw;
        s[u] = j < n ? __ldcg(ih + j) : -1;
    }
}

// Loads of chunk c's rows from the sources s (read earlier).
template <int LPR>
__device__ __forceinline__ void move_load(MoveChunk<kMoveRows> &m, int c, int n, int T, const int (&s)[kMoveRows],
                                          const uint8_t *Kh, const uint8_t *Vh, int hw, uint32_t *status)
{
    using M = MoveShape<LPR>;
#pragma unroll
    for (int u = 0; u < kMoveRows; ++u) {
        const int j = c * M::CR + u * M::SLOTS + hw;
        m.dst[u] = -1;
        if (j < n) {
            const int src = s[u];
            if (src < j || src >= T) {
                atomicOr(status, MKV_DEV_INTERNAL);  // not an ascending index list: the move would be unsafe
            } else if (src != j) {
                m.dst[u] = j;
                m.k[u] = ld_cg(Kh + (size_t)src * M::RB);
                m.v[u] = ld_cg(Vh + (size_t)src * M::RB);
            }
        }
    }
}

template <int LPR>
__device__ __forceinline__ void move_store(const MoveChunk<kMoveRows> &m, uint8_t *Kh, uint8_t *Vh)
{
    using M = MoveShape<LPR>;
#pragma unroll
    for (int u = 0; u < kMoveRows; ++u) {
        if (m.dst[u] >= 0) {
            st_stream(Kh + (size_t)m.dst[u] * M::RB, m.k[u]);
            st_stream(Vh + (size_t)m.dst[u] * M::RB, m.v[u]);
        }
    }
}

// In-place compaction: row j of each head becomes row idx[j] (j < kept), in
// the head's own K and V rows. Row r is read by at most one slot j <= r
// (idx ascends from 0, so idx[j] >= j) and written by slot r, so walking the
// slots in chunks in ascending order is safe when chunk c's stores come
// after a CTA barrier that follows the loads of chunks <= c: every earlier
// reader of a row chunk c overwrites sits in chunk c or before. The loads of
// chunk c + 2 read rows at or beyond its own slots, which no chunk <= c + 1
// writes, so they are issued before chunk c's stores: three chunks of rows
// are in flight, and each chunk's indices are read three steps ahead of its
// row loads (the index read would otherwise put one memory round trip on
// every step). One CTA walks one head; heads are spread over the
// persistent grid.
template <int LPR>
__global__ void __launch_bounds__(kStreamThreads, 2)
k_gather_inplace(const int32_t *__restrict__ idx, int idx_stride, const int32_t *__restrict__ kept,
                 const int32_t *__restrict__ seq_lens, int heads, int t_max, int64_t n_heads, uint8_t *K, uint8_t *V,
                 uint32_t *status)
{
    using M = MoveShape<LPR>;
    const int hw = threadIdx.x / LPR, lr = threadIdx.x % LPR;
    for (int64_t head = blockIdx.x; head < n_heads; head += gridDim.x) {
        const int T = head_len(seq_lens, head, heads, t_max, status, false);
        const int n = min(kept[head], T);
        if (n <= 0) continue;  // the same for every thread
        const int32_t *ih = idx + head * idx_stride;
        uint8_t *Kh = K + (size_t)head * t_max * M::RB + lr * 16;
        uint8_t *Vh = V + (size_t)head * t_max * M::RB + lr * 16;
        const int nch = (n + M::CR - 1) / M::CR;
        MoveChunk<kMoveRows> m0, m1, m2;
        int s0[kMoveRows], s1[kMoveRows], s2[kMoveRows];
        move_sources<LPR>(0, n, ih, hw, s0);
        move_sources<LPR>(1, n, ih, hw, s1);
        move_load<LPR>(m0, 0, n, T, s0, Kh, Vh, hw, status);
        move_load<LPR>(m1, 1, n, T, s1, Kh, Vh, hw, status);
        move_sources<LPR>(2, n, ih, hw, s0);
        move_sources<LPR>(3, n, ih, hw, s1);
        move_sources<LPR>(4, n, ih, hw, s2);
        // step c: chunk c's rows in a, chunk c + 2's sources in sc (read three
        // steps earlier); chunk c + 2's rows go into the third buffer and
        // chunk c + 5's sources into sc
        auto step = [&](int c, MoveChunk<kMoveRows> &a, MoveChunk<kMoveRows> &nx, int (&sc)[kMoveRows]) {
            __syncthreads();  // the loads of chunks <= c are performed CTA-wide
            move_load<LPR>(nx, c + 2, n, T, sc, Kh, Vh, hw, status);
            move_sources<LPR>(c + 5, n, ih, hw, sc);
            move_store<LPR>(a, Kh, Vh);
        };
        for (int c = 0; c < nch; c += 3) {
            step(c, m0, m2, s0);
            if (c + 1 >= nch) break;
            step(c + 1, m1, m0, s1);
            if (c + 2 >= nch) break;
            step(c + 2, m2, m1, s2);
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
