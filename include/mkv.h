/*
 * mkv.h -- C ABI of a GB300 (sm_103a) implementation of ManifoldKV-style
 * KV-cache compression.
 *
 * The method ("ManifoldKV: Training-Free KV Cache Compression via Euclidean
 * Outlier Detection", ICML 2026 poster 62526, abstract and lay summary): for
 * every head of the key cache, take the key centroid (one global mean, or one
 * mean per non-overlapping window for WindowedManifoldKV), score every token
 * by its Euclidean distance to its centroid (or, as the KeyDiff-style
 * baseline the abstract compares against, by one minus its cosine similarity
 * to the centroid), keep the highest-scoring tokens -- those far from the
 * centroid -- and gather the kept key and value rows into a compacted cache.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Cache layout. A cache is [batch, heads, t_max, head_dim] of bf16 or of
 *   fp8 E4M3 codes (shape.dtype), head_dim innermost and contiguous (one row
 *   of head_dim elements per token: 128, 256 or 512 bytes at head_dim 64,
 *   128, 256 in bf16, half that in E4M3). Keys and values share the type;
 *   centroids, scores and summaries are fp32 on the decoded values (E4M3
 *   decodes exactly). A per-tensor scale that the caller keeps beside an
 *   E4M3 cache changes no kept set: l2 scores scale with it and cosine scores
 *   do not change; C, S and means come out in stored units.
 *   "batch" counts (layer, sequence) rows: callers fold layers into it, so a
 *   "head" is one (layer, sequence, KV head) triple, and every head is
 *   processed independently. Head h = b*heads + j covers tokens
 *   [0, T_b) with T_b = seq_lens[b] (or t_max when seq_lens is NULL); rows at
 *   or past T_b are never read.
 * Windows. window = 0, or window >= T_b, means one global centroid per head;
 *   otherwise the windows are [jW, min((j+1)W, T_b)), the last one holding the
 *   remainder, and every token is scored against its own window's centroid.
 *   Selection is one top-n_keep per head over all its tokens.
 * Kept count. n_keep(T, ratio) = floor(T*(1-ratio) + 0.5) clamped to [0, T]
 *   (ratio is the share removed: 20% compression of 4096 tokens keeps 3277),
 *   unless a per-head array n_keep[batch*heads] is passed.
 * Ties. Among equal scores the lower token index is kept. Kept indices are
 *   emitted in ascending token order.
 * Memory. Every pointer except the host-pointer arguments of
 *   mkv_compress_host is a device pointer owned by the caller. The library
 *   allocates and frees nothing and never synchronises, except
 *   mkv_device_status (which synchronises the stream). Cache and output row
 *   pointers must be 16-byte aligned; float / int32 arrays 4-byte aligned; the
 *   workspace 256-byte aligned.
 * Streams. All work is enqueued on `stream` (NULL = the legacy default
 *   stream); results are valid in stream order. Inside a call some kernels
 *   start as programmatic dependent launches of the previous one, and some
 *   kernels allow the next launch on the stream to start early; a kernel the
 *   caller launches right after a call with programmatic stream
 *   serialization must wait for its dependency (cudaGridDependencySynchronize)
 *   before it reads the call's outputs, as it must after any kernel.
 * Errors. Arguments are checked on the host before anything is enqueued; a
 *   bad argument returns a status and enqueues nothing. A failed launch
 *   returns MKV_ERR_CUDA. Problems only the GPU can see (a seq_lens entry
 *   outside [0, t_max], an n_keep entry outside [0, min(T_b, keep_stride)])
 *   set bits in a status word at the start of the workspace; the affected
 *   head is skipped (nothing written for it). Read and clear the word with
 *   mkv_device_status. No kernel traps or asserts.
 * Workspace. mkv_workspace_size() bytes are enough for every entry point on
 *   that shape and window. The status word must be zero before the first
 *   call (allocate the workspace zeroed, or call mkv_device_status once).
 *   Calls that share a workspace must not overlap on the GPU.
 * Supported. head_dim 64, 128 or 256 and dtype bf16 or E4M3 (else
 *   MKV_ERR_UNSUPPORTED; the OjaKV scorer needs 128 and bf16); t_max <= 2^30.
 *   Scores must not be NaN (inputs with NaN/Inf are outside the contract).
 */
#ifndef MKV_H_
#define MKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *mkv_stream_t;

typedef enum {
    MKV_OK = 0,
    MKV_ERR_INVALID_ARG = 1, /* null / misaligned pointer, negative size, ratio outside [0,1], ... */
    MKV_ERR_UNSUPPORTED = 2, /* head_dim other than 64/128/256, an unknown dtype (OjaKV: 128, bf16), t_max above 2^30 */
    MKV_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned or smaller than required */
    MKV_ERR_CUDA = 4,        /* a CUDA call or launch failed */
    MKV_ERR_DEVICE = 5       /* mkv_device_status only: the status word is nonzero */
} mkv_status;

/* Bits of the device status word. */
#define MKV_DEV_BAD_SEQ_LEN 0x1u  /* a seq_lens entry outside [0, t_max] */
#define MKV_DEV_BAD_N_KEEP 0x2u   /* an n_keep entry outside [0, min(T_b, keep_stride)] */
#define MKV_DEV_INTERNAL 0x4u     /* a kept count disagreed with n_keep (a library bug) */
#define MKV_DEV_TIMEOUT 0x8u      /* a bounded wait between CTAs ran out; the scores it guarded are missing */

typedef enum {
    MKV_MODE_L2 = 0,     /* s_t = |k_t - c| (ManifoldKV, abstract) */
    MKV_MODE_COSINE = 1  /* s_t = 1 - cos(k_t, c); 1 when |k_t||c| = 0 (the cosine baseline, abstract) */
} mkv_mode;

/* Element type of a cache. */
typedef enum {
    MKV_DTYPE_BF16 = 0,     /* bfloat16 */
    MKV_DTYPE_FP8_E4M3 = 1  /* OCP 8-bit floating point E4M3 (torch.float8_e4m3fn): the method runs on the
                               decoded values, which fp32 holds exactly; the NaN codes are outside the contract */
} mkv_dtype;

/* Shape of a cache. dtype: an mkv_dtype (0 = bf16). seq_lens: device int32
 * [batch], or NULL for all t_max. */
typedef struct {
    int32_t batch;
    int32_t heads;
    int32_t t_max;
    int32_t head_dim;
    int32_t dtype;
    const int32_t *seq_lens;
} mkv_shape;

/* Result of selection for one head: keep every token whose score key is
 * above `key`, and the first `ties` tokens (in index order) whose key equals
 * it. The key is the order-preserving map of the fp32 score bits:
 * bits ^ 0x80000000 for a nonnegative score, ~bits for a negative one.
 * n_keep = 0 is encoded as {0xFFFFFFFF, 0}. */
typedef struct {
    uint32_t key;
    int32_t ties;
} mkv_cut;

/* Kept tokens out of T at compression `ratio` (host helper; same rounding as
 * the kernels). Returns -1 for T < 0 or ratio outside [0, 1].
 * Source: the ManifoldKV abstract quotes its results "at 20% compression" and
 * "at 50% compression"; the percentage is read as the share of tokens
 * removed, so n_keep = round(T * (1 - ratio)), halves rounding up (the
 * workload text fixes 3277 kept of 4096 at 20%). */
int32_t mkv_num_keep(int32_t T, double ratio);

/* Windows per head of t_max tokens (0 if t_max = 0). */
int32_t mkv_num_windows(int32_t t_max, int32_t window);

/* Bytes of workspace any entry point needs for this shape and window
 * (0 on a bad shape). */
size_t mkv_workspace_size(mkv_shape shape, int32_t window);

/* Key centroids (abstract: the key centroid; per-window centroids for
 * WindowedManifoldKV). K: key cache. C: fp32 [batch, heads, nw, head_dim]
 * with nw = mkv_num_windows(t_max, window); window j of head h gets the mean
 * of its keys, accumulated in fp32 in a fixed order (the result does not
 * depend on the GPU or the grid). Windows a short head does not have are not
 * written. */
mkv_status mkv_centroid(const void *K, mkv_shape shape, int32_t window, float *C,
                        void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* Cluster summaries ("RefineKV: Query-Adaptive KV Cache Compression via
 * Attention-Error Bounds", project page, method overview step 1, Summarize:
 * contiguous clusters, their mean keys and mean values, and metadata). X is
 * a cache -- keys or values -- in the cache layout; the clusters are the
 * windows of `window` tokens (the last one holding the rest; window 0 or
 * >= t_max is one cluster per head). mean: fp32 [batch, heads, nw,
 * head_dim] with nw = mkv_num_windows(t_max, window); mean[h][j] is the
 * window's mean row, summed in fp32 in token order for windows of at most
 * 128 tokens and as mkv_centroid sums for longer ones (then bit-identical
 * to mkv_centroid). radius (NULL, or fp32 [batch, heads, nw]; windows of at
 * most 128 tokens only, else MKV_ERR_UNSUPPORTED): radius[h][j] =
 * max over the window's rows of |x_t - mean[h][j]|_2, the metadata behind a
 * bound on how far a member's logit can drift from the mean's
 * (|q.x_t - q.mean| <= |q| radius). Windows a short head does not have are
 * not written. */
mkv_status mkv_window_means(const void *X, mkv_shape shape, int32_t window, float *mean, float *radius,
                            void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* Steps a1 and a2 together, as mkv_compress runs them (the head-group, the
 * single-pass or the three-kernel path; see mkv_compress_single_pass):
 * C and S as written by mkv_centroid and mkv_score, the same bits. */
mkv_status mkv_centroid_score(const void *K, mkv_shape shape, int32_t window, mkv_mode mode, float *C, float *S,
                              void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* Scores (abstract: Euclidean distance to the key centroid; cosine baseline).
 * C as written by mkv_centroid. S: fp32 [batch, heads, t_max]; S[h][t] for
 * t < T_b is the score of token t against its window's centroid (fp32,
 * correctly rounded sqrt); entries at t >= T_b are not written. */
mkv_status mkv_score(const void *K, const float *C, mkv_shape shape, int32_t window, mkv_mode mode,
                     float *S, void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* Top-n_keep selection per head (abstract: which past tokens to retain; lay
 * summary: the far ones). S: fp32 scores as above. n_keep: device int32
 * [batch*heads] or NULL to use `ratio`. cut: [batch*heads] (see mkv_cut). An
 * exact radix select over the score keys; ties go to the lower index. */
mkv_status mkv_select_topk(const float *S, mkv_shape shape, double ratio, const int32_t *n_keep,
                           mkv_cut *cut, void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* Compaction and gather (abstract: the method decides which past tokens
 * the cache retains; lay summary: the retained far-from-ordinary tokens form
 * the smaller cache). From S and cut, emit per head the kept token indices
 * in ascending order into idx [batch*heads, keep_stride] and their count into
 * kept [batch*heads], and copy the kept rows bit for bit: K_out[h][j] =
 * K[h][idx[h][j]], V_out likewise, both [batch, heads, keep_stride,
 * head_dim] of the cache's type. Slots at or past kept[h] are not written. K_out and V_out may be
 * NULL together (indices only); then K and V may be NULL too. With n_keep
 * NULL, keep_stride must be at least mkv_num_keep(t_max, ratio). */
mkv_status mkv_compact(const float *S, const mkv_cut *cut, const void *K, const void *V,
                       mkv_shape shape, double ratio, const int32_t *n_keep, int32_t keep_stride,
                       int32_t *idx, int32_t *kept, void *K_out, void *V_out,
                       void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* The whole path (centroid -> score -> select -> compact + gather) in one
 * call, intermediates in the workspace (abstract: rank the cached keys by
 * their distance to the key centroid -- per window for WindowedManifoldKV --
 * and keep the most distant share; the cosine-to-centroid scorer is the
 * baseline switch; lay summary: only the unusual, far-away tokens stay in
 * the compressed cache). Outputs as for mkv_compact; idx and kept may be
 * NULL (not returned). */
mkv_status mkv_compress(const void *K, const void *V, mkv_shape shape, double ratio,
                        const int32_t *n_keep, mkv_mode mode, int32_t window, int32_t keep_stride,
                        void *K_out, void *V_out, int32_t *idx, int32_t *kept,
                        void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* Per-window-quota variant of WindowedManifoldKV (a reading of the
 * abstract, which makes the centroid per window and says nothing more about
 * the selection): instead of one top-n_keep per head, every window keeps its
 * own share n_keep(|w|, ratio) of its tokens, the highest-scoring within it
 * (ties to the lower index). mkv_num_keep_quota gives a T-token head's kept
 * count, (nw-1)*n_keep(W, ratio) + n_keep(T-(nw-1)W, ratio); -1 on a bad
 * argument. With window 0 or >= T it equals mkv_num_keep. */
int32_t mkv_num_keep_quota(int32_t T, double ratio, int32_t window);

/* Selection with per-window quotas, from scores S (as written by mkv_score
 * with the same window): the kept indices of head h, ascending, into
 * idx[h * keep_stride + slot] (window j's at slots from j * n_keep(W,
 * ratio)), their count into kept[h]. keep_stride must be at least
 * mkv_num_keep_quota(t_max, ratio, window). Needs the workspace's status
 * word only. */
mkv_status mkv_select_quota(const float *S, mkv_shape shape, double ratio, int32_t window, int32_t keep_stride,
                            int32_t *idx, int32_t *kept, void *workspace, size_t workspace_bytes,
                            mkv_stream_t stream);

/* mkv_compress with per-window quotas: same centroids and scores, the
 * selection of mkv_select_quota, then the row gather. Outputs as for
 * mkv_compress (idx and kept may be NULL); keep_stride as for
 * mkv_select_quota. */
mkv_status mkv_compress_quota(const void *K, const void *V, mkv_shape shape, double ratio, mkv_mode mode,
                              int32_t window, int32_t keep_stride, void *K_out, void *V_out, int32_t *idx,
                              int32_t *kept, void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* OjaKV-style reconstruction-error scores ("OjaKV: Context-Aware Online
 * Low-Rank KV Cache Compression", deep notes of the ACL 2026 Findings paper,
 * method details, error-based token selection for the hybrid storage):
 *     e_t = (1/M) sum_m |q_m . (k_t - U U^T k_t)| / sqrt(head_dim),
 * the error the low-rank basis U leaves in key t, weighed by the M rows q_m
 * of the recent query window of the query heads that read this KV head.
 * K: bf16 cache. Q: bf16 [batch, heads, n_query, head_dim], the window's
 * query rows per KV head (group heads x recent positions, flattened; any
 * order). U: fp32 [batch, heads, head_dim, rank], row-major (column j is
 * basis vector j), 16-byte aligned; it need not be orthonormal (the formula
 * is used as is); may be NULL when rank = 0. n_query: a multiple of 16 in [16, 256]; rank in
 * [0, head_dim]. S: fp32 [batch, heads, t_max], written for t < T_b.
 * Computed as (P q_m) . k_t with P = I - U U^T: P q_m in fp32, split into
 * two bf16 operands (hi + lo, about 2^-17 relative), contracted with the
 * keys on the tensor cores in fp32. The workspace must hold
 * mkv_oja_workspace_size(shape, n_query) bytes. MKV_ERR_UNSUPPORTED when
 * batch*heads*t_max or batch*heads*2*n_query reaches 2^31 (32-bit TMA
 * coordinates). */
size_t mkv_oja_workspace_size(mkv_shape shape, int32_t n_query);
mkv_status mkv_oja_score(const void *K, const void *Q, const float *U, mkv_shape shape, int32_t n_query,
                         int32_t rank, float *S, void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* Choose, process-wide, how the OjaKV contraction runs for n_query <= 128;
 * returns the previous setting. 0 (the default): one CTA per SM, 128 tokens
 * per tensor-core MMA. 1: pairs of CTAs on two SMs (a thread-block cluster
 * of two, tcgen05.mma with cta_group::2), 256 tokens per MMA, each SM
 * holding half of the projected query rows (the hi split on one, the lo
 * split on the other). Same scores either way; larger n_query always runs on
 * one CTA per SM. */
int32_t mkv_set_oja_pair(int32_t enable);

/* mkv_oja_score recording caller-created CUDA events (cudaEvent_t as void*)
 * on `stream`: events[0] before the query projection kernel, events[1]
 * between it and the tensor-core contraction, events[2] after; n_events >= 3.
 * Nothing is recorded for an empty shape. */
mkv_status mkv_oja_score_profiled(const void *K, const void *Q, const float *U, mkv_shape shape, int32_t n_query,
                                  int32_t rank, float *S, void *workspace, size_t workspace_bytes,
                                  mkv_stream_t stream, void *const *events, int32_t n_events);

/* OjaKV's full-rank selection: the scores of mkv_oja_score, then the
 * top-n_keep selection, compaction and gather of mkv_compress (keep the
 * largest errors; ties to the lower index; outputs as for mkv_compress). */
mkv_status mkv_compress_oja(const void *K, const void *V, const void *Q, const float *U, mkv_shape shape,
                            int32_t n_query, int32_t rank, double ratio, const int32_t *n_keep,
                            int32_t keep_stride, void *K_out, void *V_out, int32_t *idx, int32_t *kept,
                            void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* mkv_compress that writes the compacted cache over the input (the
 * memory-saving form: no output buffers). After the call, rows
 * [0, kept[h]) of head h in K and V hold K/V[h][idx[h][j]], j < kept[h], in
 * ascending token order; rows from kept[h] on are unchanged. idx
 * [batch*heads, t_max] and kept [batch*heads] may be NULL (not returned).
 * Scores and selection are those of mkv_compress; the move runs one CTA per
 * head through chunks of 64 rows in ascending order (a row is always read
 * before it is overwritten, as idx[j] >= j). */
mkv_status mkv_compress_inplace(void *K, void *V, mkv_shape shape, double ratio, const int32_t *n_keep,
                                mkv_mode mode, int32_t window, int32_t *idx, int32_t *kept, void *workspace,
                                size_t workspace_bytes, mkv_stream_t stream);

/* Number of stages mkv_compress_profiled brackets with events: 6, one per
 * kernel -- piece sums (a1), window means (a1), scores (a2), top-k select
 * (a3; also emits the kept indices when a head's scores fit in shared
 * memory, t_max <= 40960), compaction into ascending indices (a4; empty when
 * select emitted them), row gather of K and V (a5). When the single-pass or
 * the head-group kernel is in use, stage 0 is that kernel and stages 1-2 are
 * empty. */
int32_t mkv_compress_num_stages(void);

/* Which a1 + a2 path mkv_compress takes on the current device for this
 * shape, window and mode: 1 the single-pass kernel (opt-in, K read once),
 * 4 the head-group kernel with its pass 1 fed through a copy ring (see
 * mkv_set_head_group_ring), 2 the head-group kernel (the default when a unit of windows fits in L2
 * and, with several rounds per group, the cache is bf16 and, for head dims up
 * to 128, its modelled cost is below the three kernels': K read from HBM
 * once, the second read hits L2), 3 the fused whole-path kernel (every step
 * in one launch; see mkv_set_fused), 0 the three-kernel path (K read twice);
 * -1 on a bad argument or CUDA error.
 * All give bit-identical results. */
int32_t mkv_compress_single_pass(mkv_shape shape, int32_t window, mkv_mode mode);

/* Allow (1, the default) or forbid (0) the head-group kernel in
 * mkv_compress, process-wide; returns the previous setting. With a global
 * centroid, groups of CTAs share a head: they sum its pieces, meet at a
 * bounded arrival barrier, form the mean and score the pieces again while
 * their rows are still in L2 -- one HBM read of K instead of two. */
int32_t mkv_set_head_groups(int32_t enable);

/* The head-group plan mkv_centroid_score and mkv_compress's separate
 * kernels would take on the current device (a diagnostic): plan[0] groups,
 * plan[1] CTAs per group, plan[2] windows per unit, plan[3] 1 for the
 * copy-ring kernel. Returns 0, or -1 (plan zeroed) when head groups do not
 * apply or on a bad argument (plan untouched when it is NULL). */
int32_t mkv_head_group_plan(mkv_shape shape, int32_t window, mkv_mode mode, int32_t *plan);

/* Allow (1) or forbid (0) the copy-ring form of the head-group kernel,
 * process-wide; returns the previous setting. It applies to bf16 caches at
 * head dim 128 wherever head groups run (on their own, not inside the fused
 * kernel): the same units, group barrier, means and L2 pass, but pass 1 is
 * streamed into shared memory by a producer warp with bulk asynchronous
 * copies, a ring of three 32 KB stages per CTA, which keeps running into the
 * next unit while the other warps wait at the group barrier and re-read the
 * unit from L2. The results are the same bits. */
int32_t mkv_set_head_group_ring(int32_t enable);

/* Choose, process-wide, when mkv_compress runs the fused whole-path kernel;
 * returns the previous scorer setting. scorer_ctas < 0 (the default): on its
 * own rule -- bf16 caches, head dim 128, global centroids, 12288 < t_max
 * <= 20480 and at least 64 heads (batch * heads), the shapes where it was
 * measured faster than the separate kernels on GB300 -- with 3/4 of the
 * resident grid scoring and max(16,
 * heads / 16) selector CTAs. scorer_ctas > 0: wherever it applies, with that
 * scorer budget and select_ctas selector CTAs (select_ctas <= 0 keeps the
 * current value, 32 at start). scorer_ctas == 0: never. It applies to global
 * centroids (window 0 or >= t_max) with t_max <= 20480, without per-window
 * quotas, in-place compaction or caller events, and when head groups are
 * allowed and the single-pass kernel is not. One cooperative launch then
 * runs every step: head groups score the heads (K read from HBM once), the
 * selector CTAs run the selects in head order, and every warp then copies
 * gather items on its own, each step waiting (bounded; a wait that runs out
 * sets MKV_DEV_TIMEOUT in the status word and that head keeps no rows) for
 * the one it depends on. The outputs are the same bits as the separate
 * kernels'. When the whole grid cannot be resident at launch, mkv_compress
 * runs the separate kernels instead. mkv_compress_host always runs the
 * separate kernels (the host link, not the kernels, bounds it). */
int32_t mkv_set_fused(int32_t scorer_ctas, int32_t select_ctas);

/* Per-layer kept-token budgets for the n_keep array (host helper). The
 * budget mapping of "RippleKV" (gist.science explainer of arXiv 2608.08684),
 * Methodology section 2, Sensitivity-Guided Budget Allocation: the layer
 * sensitivities are normalised to [0, 1] (all equal -> 0), mapped to
 * multipliers w = r^s, clipped to [1/gamma, gamma], and scaled so that the
 * budgets add up to `total`. Readings where that text is silent: layer l
 * cannot keep more than cap[l] tokens (allocation min(cap, lambda * w) with
 * lambda meeting the total, i.e. water-filling); real budgets become integers
 * by largest remainder, lower layer first among equal remainders. Writes
 * budget[layers]; returns 0, 1 when the caps cannot absorb the total (every
 * layer then gets its cap), -1 on bad input (r <= 0, gamma < 1, NaN,
 * negative cap or total). The profiling that yields the sensitivities needs
 * a model and is not part of this library. */
int32_t mkv_layer_budgets(const double *sensitivity, int32_t layers, double r, double gamma, int64_t total,
                          const int32_t *cap, int32_t *budget);

/* Allow (1) or forbid (0, the default) the single-pass centroid + score
 * kernel in mkv_compress, process-wide; returns the previous setting. The
 * single-pass kernel reads K from HBM once instead of twice but waits on
 * other CTAs for every window's mean; on GB300 it is currently slower than
 * the three-kernel path, so it is off unless asked for. */
int32_t mkv_set_single_pass(int32_t enable);

/* mkv_compress, recording caller-created CUDA events (cudaEvent_t handles
 * passed as void*) on `stream`: events[i] right before stage i and
 * events[n_stages] after the last, so the caller can time every stage
 * inside the real call. n_events must be at least n_stages + 1. */
mkv_status mkv_compress_profiled(const void *K, const void *V, mkv_shape shape, double ratio,
                                 const int32_t *n_keep, mkv_mode mode, int32_t window,
                                 int32_t keep_stride, void *K_out, void *V_out, int32_t *idx,
                                 int32_t *kept, void *workspace, size_t workspace_bytes,
                                 mkv_stream_t stream, void *const *events, int32_t n_events);

/* mkv_compress for a cache held in host memory (e.g. offloaded to CPU RAM):
 * copies hK, hV (host, pinned for asynchrony) into the caller's device
 * buffers dK, dV, runs mkv_compress, and copies the results back into host
 * buffers hK_out, hV_out [batch, heads, keep_stride, head_dim] and h_idx,
 * h_kept [batch*heads(, keep_stride)]; any of the four host outputs may be
 * NULL. Device output buffers dK_out, dV_out, d_idx, d_kept are required.
 * The batch rows are processed in up to 16 chunks: chunk c's host-to-device
 * copies run on two library-owned copy-in streams (keys on one, values on
 * the other), its kernels on `stream`, its device-to-host copies on a
 * copy-out stream, so copies of different chunks overlap each other and the
 * kernels. Values are read only for the kept rows: when hV is pinned host
 * memory the device can address (cudaHostAlloc / cudaHostRegister), the
 * gather reads the kept value rows straight from it and dV is not used, so
 * only those rows cross the host link. The copy streams first wait for
 * the work already on `stream`, and `stream` waits for every copy before
 * anything enqueued after this call, so the call behaves as if it were all on
 * `stream`. The three streams and their events are created on a device's first
 * call and kept until the process exits. Every copy is one cudaMemcpyAsync;
 * nothing synchronises the host. */
mkv_status mkv_compress_host(const void *hK, const void *hV, void *dK, void *dV, mkv_shape shape,
                             double ratio, mkv_mode mode, int32_t window, int32_t keep_stride,
                             void *dK_out, void *dV_out, int32_t *d_idx, int32_t *d_kept,
                             void *hK_out, void *hV_out, int32_t *h_idx, int32_t *h_kept,
                             void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* Failure injection for tests of the fused whole-path kernel's bounded waits
 * (no counterpart in the paper). Runs mkv_compress through the fused kernel
 * (global centroids; with the automatic budgets when its own rule would not
 * take the shape) with one wait that cannot end: stage 0 raises the
 * barrier target of scorer group 0 above its CTA count, stage 1 makes the
 * select of head 0 wait for one scorer more than its group has. The wait
 * runs out after its bound (about 1 s) and sets MKV_DEV_TIMEOUT; every other
 * wait of the launch then gives up at once, so the launch ends in about one
 * bound and the context stays usable. A head whose scoring or select did not
 * complete keeps no rows (kept = 0): no select runs on stale scores. The
 * other outputs are not meaningful. MKV_ERR_INVALID_ARG for another stage or
 * without K_out/V_out; MKV_ERR_UNSUPPORTED when the fused kernel cannot run
 * the shape (window is 0 here). */
mkv_status mkv_inject_stalled_fused(const void *K, const void *V, mkv_shape shape, double ratio, mkv_mode mode,
                                    int32_t keep_stride, void *K_out, void *V_out, int32_t *idx, int32_t *kept,
                                    int32_t stage, void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* Size of the library-owned scratch array used by mkv_compress_noalloc. */
#define MKV_NOALLOC_SCRATCH_BYTES (32u << 20)

/* mkv_compress for callers that cannot allocate device memory. The paper has
 * no counterpart: this is an engineering entry point. Some callers get only
 * input and output pointers and a stream: a custom operator behind an inference
 * engine's C plugin interface, a server whose memory planner reserves all
 * device memory up front and forbids allocations while it serves, or a
 * latency-critical path that cannot afford cudaMalloc's implicit device
 * synchronisation. This call therefore needs no workspace. It uses a fixed
 * scratch array of MKV_NOALLOC_SCRATCH_BYTES (32 MiB) in the library's device
 * image. Every GPU that loads the library holds that array until the process
 * exits, whether or not this call is used.
 *   Limits: the problem must fit, i.e. mkv_workspace_size(shape, window) <=
 *   MKV_NOALLOC_SCRATCH_BYTES. At head dim 128 and window 0 the workspace
 *   takes about 10 bytes per token row (heads x t_max: scores, fallback
 *   indices, partial sums, compaction offsets), so one call holds about
 *   3.3M token rows at t_max 4K-16K (202 heads of 16384 tokens) and about
 *   3.9M at 64K-128K (30 heads of 131072). Larger problems return
 *   MKV_ERR_UNSUPPORTED and enqueue nothing; split them into several calls
 *   over groups of heads, sized with mkv_workspace_size.
 *   Set-up: the first call on a device, with that device current, looks up the
 *   array's device address once (cudaGetSymbolAddress) and keeps it for the
 *   life of the process. Make that first call before any stream capture. Do
 *   not call this entry point again on a device after cudaDeviceReset there:
 *   the kept address would be stale.
 *   Sharing: every call uses the same array, and it keeps the last call's
 *   contents. Calls that can overlap on the GPU (different streams, or
 *   different host threads, on one device) race on it and corrupt each
 *   other's results. Serialise them.
 *   Outputs and arguments: as for mkv_compress. status_out (device, nullable)
 *   receives the device status word of this call (MKV_DEV_* bits); the call
 *   then resets the word to zero. With status_out NULL those bits are
 *   discarded (there is no workspace to query afterwards), including
 *   MKV_DEV_TIMEOUT: callers that need device-side error detection must pass
 *   status_out. After MKV_ERR_CUDA the call still tries to
 *   reset it (best effort: the failed call's bits are not reported, and a
 *   sticky CUDA error can prevent the reset). The call allocates and frees
 *   nothing. */
mkv_status mkv_compress_noalloc(const void *K, const void *V, mkv_shape shape, double ratio,
                                const int32_t *n_keep, mkv_mode mode, int32_t window, int32_t keep_stride,
                                void *K_out, void *V_out, int32_t *idx, int32_t *kept, uint32_t *status_out,
                                mkv_stream_t stream);

/* Failure injection for tests of the single-pass kernel's bounded waits (no
 * counterpart in the paper). Runs mkv_compress with the single-pass centroid
 * + score kernel, but with every window's arrival counters started past any
 * group size, so no window mean is ever published: each wait between CTAs
 * runs out after its time bound (about 1 s), MKV_DEV_TIMEOUT is set in the
 * status word, the remaining waits give up at once, the kernels finish and
 * the context stays usable. The outputs are not meaningful. Returns
 * MKV_ERR_UNSUPPORTED when the single-pass kernel cannot run this shape. */
mkv_status mkv_inject_stalled_windows(const void *K, const void *V, mkv_shape shape, double ratio, mkv_mode mode,
                                      int32_t window, int32_t keep_stride, void *K_out, void *V_out, int32_t *idx,
                                      int32_t *kept, void *workspace, size_t workspace_bytes, mkv_stream_t stream);

/* Synchronise `stream`, read the status word of `workspace` into *bits (may
 * be NULL) and reset it to zero. MKV_OK if it was zero, MKV_ERR_DEVICE if
 * not, MKV_ERR_CUDA if the synchronisation or copy failed. */
mkv_status mkv_device_status(void *workspace, mkv_stream_t stream, uint32_t *bits);

/* Static, human-readable name of a status code. */
const char *mkv_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* MKV_H_ */
