// One head's top-k select (a3) and its ascending kept indices (a4), as device
// functions that every select kernel of the library calls: the step kernel
// k_select and the fused whole-path kernel.
//
// Method: "ManifoldKV: Training-Free KV Cache Compression via Euclidean
// Outlier Detection" (ICML 2026 poster 62526), abstract -- the tokens farthest
// from the key centroid are kept; ties at the cut go to the lower index.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "mkv_device.cuh"
#include "mkv_internal.h"

namespace mkv {
namespace {

constexpr int kSelectCandidates = 1024;  // keys a radix pass may collect for the later passes
using namespace dev;

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
//
// select_item is one item's work (all NT threads of the CTA call it); the
// fused kernel calls it too, on scores written earlier in the same launch,
// which it reads through L2 only (__ldcg) and only with IN_SMEM.
template <bool IN_SMEM, bool QUOTA, int NT>
__device__ __forceinline__ void
select_item(int64_t item, const float *__restrict__ S, const int32_t *__restrict__ seq_lens, int heads, int t_max,
            double ratio, const int32_t *__restrict__ n_keep, int keep_stride, int window, int nwin_max,
            mkv_cut *__restrict__ cut_out, int2 *__restrict__ chunk_info, int nch_max,
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
    {
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
            if (seg >= Th || total > keep_stride) return;  // the same for every thread
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
            return;
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
        // scores in L2 (not in shared memory) are read as 16-byte vectors
        // when the head's row allows it, kUnroll of them in flight per thread
        const bool vec = !IN_SMEM && (reinterpret_cast<uintptr_t>(grow) & 15) == 0;
        const int n4 = vec ? T / 4 : 0;
        const float4 *g4 = reinterpret_cast<const float4 *>(grow);
        if (nk > 0) {
            if (!IN_SMEM) {
                for (int i = threadIdx.x; i < n4; i += NT * kUnroll) {
                    float4 v[kUnroll];
#pragma unroll
                    for (int k = 0; k < kUnroll; ++k)
                        if (i + k * NT < n4) v[k] = g4[i + k * NT];
#pragma unroll
                    for (int k = 0; k < kUnroll; ++k)
                        if (i + k * NT < n4) {
                            see(v[k].x);
                            see(v[k].y);
                            see(v[k].z);
                            see(v[k].w);
                        }
                }
                for (int t = 4 * n4 + threadIdx.x; t < T; t += NT) see(srow[t]);
            }
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
                    } else if (!IN_SMEM) {
                        auto visit = [&](float x) {
                            const uint32_t u = score_key(x);
                            if ((u & pmask) == prefix) {
                                atomicAdd(&hist[(u >> shift) & (uint32_t)(nb - 1)], 1u);
                                if (build) {
                                    const uint32_t c = atomicAdd(&s_ncand, 1u);
                                    if (c < (uint32_t)kSelectCandidates) s_cand[c] = u;
                                }
                            }
                        };
                        for (int i = threadIdx.x; i < n4; i += NT * kUnroll) {
                            float4 v[kUnroll];
#pragma unroll
                            for (int k = 0; k < kUnroll; ++k)
                                if (i + k * NT < n4) v[k] = g4[i + k * NT];
#pragma unroll
                            for (int k = 0; k < kUnroll; ++k)
                                if (i + k * NT < n4) {
                                    visit(v[k].x);
                                    visit(v[k].y);
                                    visit(v[k].z);
                                    visit(v[k].w);
                                }
                        }
                        for (int t = 4 * n4 + threadIdx.x; t < T; t += NT) visit(srow[t]);
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

}  // namespace
}  // namespace mkv
