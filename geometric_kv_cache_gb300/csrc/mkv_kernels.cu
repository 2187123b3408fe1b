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

namespace mkv {
namespace {

constexpr int kStreamThreads = 256;            // compaction CTAs
constexpr int kSelectThreads = 512;    // select CTAs whose head's scores sit in shared memory (two per SM)
constexpr int kSelectThreadsL2 = 1024; // select CTAs that pass over the scores in L2 (one per SM)
constexpr int kSelectCandidates = 1024; // keys a radix pass may collect for the later passes
constexpr int kSelectSmemScores = 40960;  // heads up to this many tokens are selected from shared memory
using namespace dev;

// ------------------------------------------------------ a3: radix select --

// Per-chunk kept counts and their exclusive scan for one head (all NT threads
// of the CTA call it): chunk_info[c] = {first output slot of chunk c, ties at
// the cut key in chunks before c}; returns the head's kept count.
template <int NT>
__device__ int chunk_offsets_block(const float *srow, int T, mkv_cut cut, int nch_max,
                                   int2 *__restrict__ info, uint32_t *s_warp)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nch = (T + kCompactChunk - 1) / kCompactChunk;
    for (int c = warp; c < nch; c += NT / 32) {
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

// One CTA per head (persistent over heads). Histogram passes over the head's
// score keys (digits of up to 11 bits, most significant first, starting at
// the highest bit where the head's smallest and largest keys differ) find
// the n_keep-th largest key and how many of its ties are kept; with
// chunk_info it then computes the compaction offsets (fused path). When the
// launch gives dynamic shared memory for t_max scores (IN_SMEM), the head's
// scores are copied there once and every pass reads shared memory; otherwise
// the passes read global memory (L2), four loads in flight per thread.
//
// QUOTA (the per-window-quota selection): the item is a (head, window) pair
// instead of a head; each window of W tokens keeps its own share
// n_keep(|w|, ratio) of its tokens, selected among them alone, and writes
// its indices at slot w * n_keep(W, ratio) of the head's row (every window
// before the last is full, so the offset has this closed form). The CTA of
// window 0 writes the head's kept count. idx is required, cut_out and
// chunk_info unused.
template <bool IN_SMEM, bool QUOTA, int NT>
__global__ void __launch_bounds__(NT, NT > 512 ? 1 : 2)
k_select(const float *__restrict__ S, const int32_t *__restrict__ seq_lens, int heads, int t_max,
         double ratio, const int32_t *__restrict__ n_keep, int keep_stride, int64_t n_items, int window,
         int nwin_max, mkv_cut *__restrict__ cut_out, int2 *__restrict__ chunk_info, int nch_max,
         int32_t *__restrict__ kept_out, int32_t *__restrict__ idx, int idx_stride, uint32_t *status)
{
    extern __shared__ __align__(16) float s_scores[];
    __shared__ uint32_t hist[2048];
    __shared__ uint32_t s_warp[32];
    __shared__ uint32_t s_digit, s_above, s_count, s_ncand;
    __shared__ uint32_t s_min[NT / 32], s_max[NT / 32];
    __shared__ uint32_t s_cand[kSelectCandidates];
    const int lane = threadIdx.x & 31;
    constexpr int kUnroll = 4;
    pdl_wait();  // the scores of the previous kernel are complete
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        // the gather may start launching once every CTA is on its last item
        // (earlier, its waiting CTAs would slow a select of many rounds)
        if (item + gridDim.x >= n_items) pdl_trigger();
        int64_t head = item;
        int T, nk, seg = 0;  // segment [seg, seg + T) of the head's tokens
        int32_t *idx_head = nullptr;
        if (QUOTA) {
            head = item / nwin_max;
            const int w = (int)(item - head * nwin_max);
            const int Th = head_len(seq_lens, head, heads, t_max, status, threadIdx.x == 0 && w == 0);
            const int nw = (Th + window - 1) / window;
            const int q_full = num_keep_dev(window, ratio);
            const int total = nw > 0 ? (nw - 1) * q_full + num_keep_dev(Th - (nw - 1) * window, ratio) : 0;
            if (w == 0 && threadIdx.x == 0) {
                if (total > keep_stride) atomicOr(status, MKV_DEV_BAD_N_KEEP);
                if (kept_out) kept_out[head] = total > keep_stride ? 0 : total;
            }
            seg = w * window;
            if (seg >= Th || total > keep_stride) continue;  // the same for every thread
            T = min(window, Th - seg);
            nk = num_keep_dev(T, ratio);
            idx_head = idx + head * idx_stride + (int64_t)w * q_full;
        } else {
            T = head_len(seq_lens, head, heads, t_max, status, threadIdx.x == 0);
            nk = n_keep ? n_keep[head] : num_keep_dev(T, ratio);
            if (idx) idx_head = idx + head * idx_stride;
        }
        // output slots this segment may use
        const int cap = QUOTA ? nk : keep_stride;
        if (!QUOTA && (nk < 0 || nk > T || (keep_stride >= 0 && nk > keep_stride))) {
            if (threadIdx.x == 0) {
                atomicOr(status, MKV_DEV_BAD_N_KEEP);
                mkv_cut none;
                none.key = kNoneKey;
                none.ties = 0;
                if (cut_out) cut_out[head] = none;
                if (kept_out) kept_out[head] = 0;
            }
            if (chunk_info) {
                const int nch = (T + kCompactChunk - 1) / kCompactChunk;
                for (int c = threadIdx.x; c < nch; c += NT) chunk_info[head * nch_max + c] = make_int2(-1, -1);
            }
            continue;
        }
        const float *grow = S + (size_t)head * t_max + seg;
        const float *srow = grow;
        // Smallest and largest key of the head: bits above their highest
        // differing bit are common to every key, so the digits start there
        // and the first pass spreads over all its bins. Taken while the
        // scores are copied to shared memory, else in a pass of their own.
        uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
        auto see = [&](float v) {
            const uint32_t u = score_key(v);
            kmin = min(kmin, u);
            kmax = max(kmax, u);
        };
        if (IN_SMEM) {
            if ((reinterpret_cast<uintptr_t>(grow) & 15) == 0) {  // 16-byte aligned segment
                const float4 *g4 = reinterpret_cast<const float4 *>(grow);
                float4 *s4 = reinterpret_cast<float4 *>(s_scores);
                for (int i = threadIdx.x; i < T / 4; i += NT) {
                    const float4 v = __ldcg(g4 + i);
                    s4[i] = v;
                    see(v.x);
                    see(v.y);
                    see(v.z);
                    see(v.w);
                }
                for (int i = (T & ~3) + threadIdx.x; i < T; i += NT) {
                    const float v = __ldcg(grow + i);
                    s_scores[i] = v;
                    see(v);
                }
            } else {
                for (int i = threadIdx.x; i < T; i += NT) {
                    const float v = __ldcg(grow + i);
                    s_scores[i] = v;
                    see(v);
                }
            }
            __syncthreads();
            srow = s_scores;
        }
        uint32_t prefix = 0, pmask = 0;
        int need = nk;
        if (nk > 0) {
            if (!IN_SMEM)
                for (int t = threadIdx.x; t < T; t += NT) see(srow[t]);
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
                kmax = max(kmax, __shfl_xor_sync(kFull, kmax, o));
            }
            if (lane == 0) {
                s_min[threadIdx.x >> 5] = kmin;
                s_max[threadIdx.x >> 5] = kmax;
            }
            __syncthreads();
            kmin = s_min[0];
            kmax = s_max[0];
            for (int w = 1; w < NT / 32; ++w) {
                kmin = min(kmin, s_min[w]);
                kmax = max(kmax, s_max[w]);
            }
            __syncthreads();
            if (kmin == kmax) {  // every key equal: the cut is that key, the first nk tokens are kept
                prefix = kmin;
            } else {
                const int hb = 31 - __clz(kmin ^ kmax);  // highest differing bit
                pmask = hb == 31 ? 0u : ~((2u << hb) - 1u);
                prefix = kmin & pmask;
                // Keys that match the prefix so far: once there are at most
                // kSelectCandidates of them (the count of the previous pass's
                // chosen bin), a full pass also copies them into s_cand and
                // the later passes scan that list instead of all T keys.
                uint32_t match = (uint32_t)T;
                bool listed = false;
                int ncand = 0;
#pragma unroll 1
                for (int lo = hb + 1; lo > 0;) {
                    const int width = min(11, lo);
                    const int shift = lo - width;
                    const int nb = 1 << width;
                    const bool build = !listed && shift > 0 && match <= (uint32_t)kSelectCandidates;
                    for (int i = threadIdx.x; i < nb; i += NT) hist[i] = 0;
                    if (threadIdx.x == 0) s_ncand = 0;
                    __syncthreads();
                    if (listed) {
                        for (int i = threadIdx.x; i < ncand; i += NT) {
                            const uint32_t u = s_cand[i];
                            if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & (uint32_t)(nb - 1)], 1u);
                        }
                    } else {
                        for (int base = 0; base < T; base += NT * kUnroll) {
                            uint32_t u[kUnroll];
#pragma unroll
                            for (int k = 0; k < kUnroll; ++k) {
                                const int t = base + k * NT + threadIdx.x;
                                u[k] = t < T ? score_key(srow[t]) : 0u;
                            }
#pragma unroll
                            for (int k = 0; k < kUnroll; ++k) {
                                const int t = base + k * NT + threadIdx.x;
                                if (t < T && (u[k] & pmask) == prefix) {
                                    atomicAdd(&hist[(u[k] >> shift) & (uint32_t)(nb - 1)], 1u);
                                    if (build) {
                                        const uint32_t c = atomicAdd(&s_ncand, 1u);
                                        if (c < (uint32_t)kSelectCandidates) s_cand[c] = u[k];
                                    }
                                }
                            }
                        }
                    }
                    __syncthreads();
                    // Thread i owns bpt bins in descending order from nb-1-i*bpt.
                    const int bpt = nb > NT ? nb / NT : 1;
                    const int hi = nb - 1 - (int)threadIdx.x * bpt;
                    uint32_t local = 0;
                    if (hi >= 0)
                        for (int j = 0; j < bpt; ++j) local += hist[hi - j];
                    uint32_t above = block_exclusive_scan<NT>(local, s_warp, nullptr);
                    if (hi >= 0) {
                        for (int j = 0; j < bpt; ++j) {
                            const uint32_t h = hist[hi - j];
                            if (above < (uint32_t)need && (uint32_t)need <= above + h) {
                                s_digit = (uint32_t)(hi - j);
                                s_above = above;
                                s_count = h;
                            }
                            above += h;
                        }
                    }
                    __syncthreads();
                    prefix |= s_digit << shift;
                    pmask |= (uint32_t)(nb - 1) << shift;
                    need -= (int)s_above;
                    match = s_count;
                    if (build && s_ncand <= (uint32_t)kSelectCandidates) {  // (always: the count was known)
                        listed = true;
                        ncand = (int)s_ncand;
                    }
                    __syncthreads();
                    lo = shift;
                }
            }
        } else {
            prefix = kNoneKey;
            need = 0;
        }
        mkv_cut cut;
        cut.key = prefix;
        cut.ties = need;
        if (threadIdx.x == 0 && cut_out) cut_out[head] = cut;
        if (idx_head) {
            // Emit the kept indices in ascending order straight from the
            // scores in hand. A round covers 16 * NT tokens; warp w takes 16
            // steps of 32 consecutive tokens from a + 512 w (lane l reads
            // token step + l: no bank conflicts). Counts of keys above and at
            // the cut per warp, scanned over the warps, give each warp's
            // first tie rank and first output slot; within the warp,
            // ballots and popcounts place every kept token, so consecutive
            // kept tokens land in consecutive slots (coalesced stores).
            // Counts are carried across rounds.
            const int warp = threadIdx.x >> 5;
            const uint32_t lt = (1u << lane) - 1u;
            uint32_t kept = 0, ties_before = 0;
            for (int a = 0; a < T && nk > 0; a += NT * 16) {
                const int wb = a + warp * 512;
                uint32_t ngt = 0, neq = 0;
#pragma unroll 4
                for (int j = 0; j < 16; ++j) {
                    const int t = wb + j * 32 + lane;
                    const uint32_t u = t < T ? score_key(srow[t]) : 0u;
                    ngt += __popc(__ballot_sync(kFull, t < T && u > cut.key));
                    neq += __popc(__ballot_sync(kFull, t < T && u == cut.key));
                }
                if (lane == 0) {
                    s_warp[warp] = neq;
                    s_min[warp] = ngt;  // reused as per-warp scratch
                }
                __syncthreads();
                uint32_t tie_base = ties_before, eq_total = 0;
                for (int w = 0; w < NT / 32; ++w) {
                    const uint32_t e = s_warp[w];
                    if (w < warp) tie_base += e;
                    eq_total += e;
                }
                // ties of this warp that are kept, then the warp's first slot
                const uint32_t keep_ties_w =
                    (uint32_t)min(max((int)cut.ties - (int)tie_base, 0), (int)neq);
                __syncthreads();
                if (lane == 0) s_max[warp] = s_min[warp] + keep_ties_w;
                __syncthreads();
                uint32_t slot = kept, k_total = 0;
                for (int w = 0; w < NT / 32; ++w) {
                    const uint32_t k = s_max[w];
                    if (w < warp) slot += k;
                    k_total += k;
                }
                uint32_t rank = tie_base;
#pragma unroll 4
                for (int j = 0; j < 16; ++j) {
                    const int t = wb + j * 32 + lane;
                    const uint32_t u = t < T ? score_key(srow[t]) : 0u;
                    const bool gt = t < T && u > cut.key, eq = t < T && u == cut.key;
                    const uint32_t eqb = __ballot_sync(kFull, eq);
                    const bool keep = gt || (eq && rank + __popc(eqb & lt) < (uint32_t)cut.ties);
                    const uint32_t kb = __ballot_sync(kFull, keep);
                    if (keep) {
                        const uint32_t sl = slot + __popc(kb & lt);
                        if (sl < (uint32_t)cap) idx_head[sl] = seg + t;
                        else atomicOr(status, MKV_DEV_INTERNAL);
                    }
                    rank += __popc(eqb);
                    slot += __popc(kb);
                }
                __syncthreads();  // s_warp, s_min and s_max are rewritten next round
                kept += k_total;
                ties_before += eq_total;
            }
            if (threadIdx.x == 0) {
                if ((int)kept != nk) atomicOr(status, MKV_DEV_INTERNAL);
                if (!QUOTA && kept_out) kept_out[head] = (int32_t)kept;
            }
        } else if (chunk_info) {
            const int kept = nk > 0 ? chunk_offsets_block<NT>(srow, T, cut, nch_max, chunk_info + head * nch_max, s_warp) : 0;
            if (threadIdx.x == 0) {
                if (kept != nk) atomicOr(status, MKV_DEV_INTERNAL);
                if (kept_out) kept_out[head] = kept;
            }
        }
        if (IN_SMEM) __syncthreads();  // s_scores is reused by the next head
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
// tokens against the cut; two CTA scans give each kept token its tie rank
// and its output slot; each thread then writes its kept token ids, in
// ascending order, to idx[head * idx_stride + slot].
__global__ void __launch_bounds__(kStreamThreads)
k_compact(const float *__restrict__ S, const mkv_cut *__restrict__ cuts, const int2 *__restrict__ chunk_info,
          const int32_t *__restrict__ seq_lens, int heads, int t_max, int nch_max, int keep_stride, int64_t n_items,
          int32_t *__restrict__ idx, int idx_stride, uint32_t *status)
{
    __shared__ uint32_t s_warp[kStreamThreads / 32];
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
        const uint32_t kb = block_exclusive_scan<kStreamThreads>(__popc(keepm), s_warp, nullptr);
        int32_t *idx_head = idx + head * idx_stride;
        uint32_t r = kb;
        for (uint32_t m = keepm; m; m &= m - 1, ++r) {
            const int64_t slot = (int64_t)info.x + r;
            if (slot >= 0 && slot < keep_stride) idx_head[slot] = t0 + __ffs(m) - 1;
            else atomicOr(status, MKV_DEV_INTERNAL);
        }
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
