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

#include "mkv_device.cuh"
#include "mkv_internal.h"
#include "mkv_select.cuh"

namespace mkv {
namespace {

constexpr int kStreamThreads = 256;            // compaction CTAs
constexpr int kSelectThreads = 512;    // select CTAs whose head's scores sit in shared memory (two per SM)
constexpr int kSelectThreadsL2 = 1024; // select CTAs that pass over the scores in L2 (one per SM)
constexpr int kSelectSmemScores = 40960;  // heads up to this many tokens are selected from shared memory
using namespace dev;

// ------------------------------------------------------ a3: radix select --

// chunk_offsets_block and select_item (one head's select) are in mkv_select.cuh.
template <bool IN_SMEM, bool QUOTA, int NT>
__global__ void __launch_bounds__(NT, NT > 512 ? 1 : 2)
k_select(const float *__restrict__ S, const int32_t *__restrict__ seq_lens, int heads, int t_max,
         double ratio, const int32_t *__restrict__ n_keep, int keep_stride, int64_t n_items, int window,
         int nwin_max, mkv_cut *__restrict__ cut_out, int2 *__restrict__ chunk_info, int nch_max,
         int32_t *__restrict__ kept_out, int32_t *__restrict__ idx, int idx_stride, uint32_t *status)
{
    pdl_wait();  // the scores of the previous kernel are complete
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        // the gather may start launching once every CTA is on its last item
        // (earlier, its waiting CTAs would slow a select of many rounds)
        if (item + gridDim.x >= n_items) pdl_trigger();
        select_item<IN_SMEM, QUOTA, NT>(item, S, seq_lens, heads, t_max, ratio, n_keep, keep_stride, window, nwin_max,
                                        cut_out, chunk_info, nch_max, kept_out, idx, idx_stride, status);
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
            kept = chunk_offsets_block<kSelectThreads>(S + (size_t)head * t_max, T, cut, nch_max, chunk_info + head * nch_max, s_warp);
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

// ------------------------------------------------------- a4: compaction --

// Item = (head, chunk of 4096 tokens). Each thread classifies 16 consecutive
// tokens against the cut; a CTA scan gives each kept token its output slot
// (a first scan its tie rank, in the chunks that hold tokens equal to the
// cut); the kept token ids go, in ascending order, to shared memory and from
// there, coalesced, to idx[head * idx_stride + slot]. The next item's scores
// are loaded while the current item's scans and stores run.
__global__ void __launch_bounds__(kStreamThreads)
k_compact(const float *__restrict__ S, const mkv_cut *__restrict__ cuts, const int2 *__restrict__ chunk_info,
          const int32_t *__restrict__ seq_lens, int heads, int t_max, int nch_max, int keep_stride, int64_t n_items,
          int32_t *__restrict__ idx, int idx_stride, uint32_t *status)
{
    __shared__ uint32_t s_warp[kStreamThreads / 32];
    __shared__ int32_t s_idx[kCompactChunk];
    // the thread's 16 scores of `item` (tokens past the head's end: not read)
    auto load16 = [&](int64_t item, float v[16]) {
        const int64_t head = item / nch_max;
        const int c = (int)(item - head * nch_max);
        const int T = head_len(seq_lens, head, heads, t_max, status, false);
        const float *srow = S + (size_t)head * t_max;
        const int t0 = c * kCompactChunk + threadIdx.x * 16;
        if (t0 + 16 <= T && (reinterpret_cast<uintptr_t>(srow + t0) & 15) == 0) {
            const float4 *s4 = reinterpret_cast<const float4 *>(srow + t0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 x = s4[i];
                v[4 * i] = x.x;
                v[4 * i + 1] = x.y;
                v[4 * i + 2] = x.z;
                v[4 * i + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = t0 + j < T ? srow[t0 + j] : 0.f;
        }
    };
    float nxt[16];
    if ((int64_t)blockIdx.x < n_items) load16(blockIdx.x, nxt);
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = nxt[j];
        if (item + gridDim.x < n_items) load16(item + gridDim.x, nxt);
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
        const int t0 = a + threadIdx.x * 16;
        uint32_t gtm = 0, eqm = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (t0 + j < T) {
                const uint32_t u = score_key(v[j]);
                gtm |= (uint32_t)(u > cut.key) << j;
                eqm |= (uint32_t)(u == cut.key) << j;
            }
        }
        uint32_t keepm = gtm;
        if (__syncthreads_or(eqm != 0u)) {
            uint32_t rank = (uint32_t)info.y + block_exclusive_scan<kStreamThreads>(__popc(eqm), s_warp, nullptr);
            for (uint32_t m = eqm; m; m &= m - 1) {
                if (rank < (uint32_t)cut.ties) keepm |= m & (~m + 1);
                ++rank;
            }
        }
        uint32_t nk = 0;
        uint32_t r = block_exclusive_scan<kStreamThreads>(__popc(keepm), s_warp, &nk);
        for (uint32_t m = keepm; m; m &= m - 1, ++r) s_idx[r] = t0 + __ffs(m) - 1;
        __syncthreads();
        int32_t *idx_head = idx + head * idx_stride;
        for (uint32_t i = threadIdx.x; i < nk; i += kStreamThreads) {
            const int64_t slot = (int64_t)info.x + i;
            if (slot < keep_stride) idx_head[slot] = s_idx[i];
            else atomicOr(status, MKV_DEV_INTERNAL);
        }
        __syncthreads();  // s_idx is rewritten by the next item
    }
}

}  // namespace

// ------------------------------------------------------------- occupancy --

namespace {

struct OccEntry {
    const void *fn;
    int dev;
    int threads;
    size_t smem;
    int per_sm;
};

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

// Resident CTAs per SM of a kernel on a device, cached.
int resident_per_sm(const void *fn, int threads, size_t smem, int dev)
{
    static std::mutex mu;
    static OccEntry table[128];
    static int used = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (table[i].fn == fn && table[i].dev == dev && table[i].threads == threads && table[i].smem == smem)
            return table[i].per_sm;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess || per_sm < 0)
        per_sm = 0;
    if (used < 128) table[used++] = OccEntry{fn, dev, threads, smem, per_sm};
    return per_sm;
}

}  // namespace

int resident_grid(const void *fn, int threads, size_t dyn_smem)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    return sm_count(dev) * resident_per_sm(fn, threads, dyn_smem, dev);
}

int grid_for_items(const void *fn, int threads, size_t dyn_smem, int64_t items)
{
    int64_t full = resident_grid(fn, threads, dyn_smem);
    if (full < 1) full = 1;
    return (int)(items < full ? (items > 0 ? items : 1) : full);
}

template <typename Kern>
int grid_for(Kern kernel, int threads, int64_t items)
{
    return grid_for_items(reinterpret_cast<const void *>(kernel), threads, 0, items);
}

// ------------------------------------------------------------- launchers --

bool select_emits_indices(const Geometry &g) { return g.t_max <= kSelectSmemScores; }

bool select_single_wave(const Geometry &g)
{
    if (g.n_heads == 0 || g.t_max > kSelectSmemScores) return false;
    auto *kern = k_select<true, false, kSelectThreads>;
    const size_t smem = (size_t)g.t_max * sizeof(float);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return grid_for_items(reinterpret_cast<const void *>(kern), kSelectThreads, smem, g.n_heads) >= g.n_heads;
}

cudaError_t launch_select(const Geometry &g, const float *S, const int32_t *seq_lens, double ratio,
                          const int32_t *n_keep, int32_t keep_stride, mkv_cut *cut, int2 *chunk_info,
                          int32_t *kept, int32_t *idx, int32_t idx_stride, uint32_t *status, cudaStream_t st)
{
    if (g.n_heads == 0) return cudaSuccess;
    const size_t smem = (size_t)g.t_max * sizeof(float);
    if (g.t_max <= kSelectSmemScores) {
        auto *kern = k_select<true, false, kSelectThreads>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        const int grid = grid_for_items(reinterpret_cast<const void *>(kern), kSelectThreads, smem, g.n_heads);
        // launched as a programmatic dependent of the score kernel
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kSelectThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = grid >= g.n_heads ? 1 : 0;  // one wave only (select_single_wave)
        e = cudaLaunchKernelEx(&cfg, kern, S, seq_lens, (int)g.heads, (int)g.t_max, ratio, n_keep, (int)keep_stride,
                               (int64_t)g.n_heads, 0, 1, cut, chunk_info, (int)g.nch, kept, idx, (int)idx_stride, status);
        if (e != cudaSuccess) return e;
    } else {
        auto *kern = k_select<false, false, kSelectThreadsL2>;
        const int grid = grid_for(kern, kSelectThreadsL2, g.n_heads);
        kern<<<grid, kSelectThreadsL2, 0, st>>>(S, seq_lens, g.heads, g.t_max, ratio, n_keep, keep_stride, g.n_heads, 0,
                                              1, cut, chunk_info, g.nch, kept, idx, idx_stride, status);
    }
    return cudaGetLastError();
}

cudaError_t launch_select_quota(const Geometry &g, const float *S, const int32_t *seq_lens, double ratio,
                                int32_t keep_stride, int32_t *kept, int32_t *idx, int32_t idx_stride,
                                uint32_t *status, cudaStream_t st)
{
    const PieceGeometry &p = g.pg;
    const int64_t items = g.n_heads * p.nwin_max;
    if (items == 0) return cudaSuccess;
    // one window per head (window 0 or >= t_max) is the ordinary selection
    const int wl = (p.window <= 0 || p.window >= g.t_max) ? g.t_max : p.window;
    if (wl <= kSelectSmemScores) {
        auto *kern = k_select<true, true, kSelectThreads>;
        const size_t smem = (size_t)wl * sizeof(float);
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        const int grid = grid_for_items(reinterpret_cast<const void *>(kern), kSelectThreads, smem, items);
        kern<<<grid, kSelectThreads, smem, st>>>(S, seq_lens, g.heads, g.t_max, ratio, nullptr, keep_stride, items,
                                                 wl, p.nwin_max, nullptr, nullptr, 0, kept, idx, idx_stride, status);
    } else {
        auto *kern = k_select<false, true, kSelectThreadsL2>;
        const int grid = grid_for(kern, kSelectThreadsL2, items);
        kern<<<grid, kSelectThreadsL2, 0, st>>>(S, seq_lens, g.heads, g.t_max, ratio, nullptr, keep_stride, items,
                                              wl, p.nwin_max, nullptr, nullptr, 0, kept, idx, idx_stride, status);
    }
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

cudaError_t launch_compact(const Geometry &g, const float *S, const mkv_cut *cut, const int2 *chunk_info,
                           const int32_t *seq_lens, int32_t keep_stride, int32_t *idx, int32_t idx_stride,
                           uint32_t *status, cudaStream_t st)
{
    const int64_t items = g.n_heads * g.nch;
    if (items == 0) return cudaSuccess;
    const int grid = grid_for(k_compact, kStreamThreads, items);
    k_compact<<<grid, kStreamThreads, 0, st>>>(S, cut, chunk_info, seq_lens, g.heads, g.t_max, g.nch, keep_stride,
                                               items, idx, idx_stride, status);
    return cudaGetLastError();
}

}  // namespace mkv
