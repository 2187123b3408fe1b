// Internal declarations shared by the kernels (mkv_kernels.cu) and the C ABI
// (mkv_api.cu). Not installed; callers use include/mkv.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mkv.h"

namespace mkv {

constexpr int kHeadDim = 128;          // the head dim of the single-pass and OjaKV kernels
constexpr int kRowBytes = kHeadDim * 2;  // one bf16 row at that head dim
// head dims the streaming kernels support (rows of 128, 256, 512 bytes)
constexpr bool supported_head_dim(int d) { return d == 64 || d == 128 || d == 256; }
// bytes per cache element of an mkv_dtype (0: not a supported type)
constexpr int elem_bytes(int32_t dtype) { return dtype == MKV_DTYPE_BF16 ? 2 : dtype == MKV_DTYPE_FP8_E4M3 ? 1 : 0; }
constexpr int kCompactChunk = 4096;    // tokens per compaction CTA (256 threads x 16)
constexpr int kStageRows = 64;         // piece lengths are multiples of this
constexpr int kMinPieceRows = 256;     // pieces are 256 * 2^k tokens (a window shorter than that is one piece) ...
constexpr int kMaxPiecesPerWindow = 64;  // ... the fewest that keep a window within this many pieces
constexpr int kGroupPieces = 32;       // pieces per first-level group of a window's sum
constexpr uint32_t kNoneKey = 0xFFFFFFFFu;  // mkv_cut.key meaning "keep nothing"
constexpr int kSmallWindowMax = 128;   // cluster summaries of windows up to this long run one group per window

// Piece decomposition of the centroid / score work: item = (head, window,
// piece), head-major. Depends only on the shape and the window (never on
// the GPU), so results are the same on every device and grid size.
struct PieceGeometry {
    int64_t n_heads = 0;   // batch * heads
    int64_t n_items = 0;   // n_heads * nwin_max * ppw
    int32_t heads = 0;
    int32_t t_max = 0;
    int32_t window = 0;    // 0 = global
    int32_t d = kHeadDim;  // head dim (64, 128 or 256)
    int32_t es = 2;        // bytes per cache element (2 bf16, 1 E4M3)
    int32_t nwin_max = 0;  // windows of a head of t_max tokens
    int32_t piece_rows = 0;  // tokens per piece (256 * 2^k)
    int32_t ppw = 0;       // pieces per window (upper bound)
    int32_t ngroups_max = 0;
};

struct Geometry {
    PieceGeometry pg;
    int64_t n_heads = 0;
    int32_t heads = 0;
    int32_t t_max = 0;
    int32_t nch = 0;       // compaction chunks per head (upper bound)
    int32_t d = kHeadDim;  // head dim
    int32_t es = 2;        // bytes per cache element
};

// Byte offsets of the workspace regions (each 256-byte aligned).
struct Layout {
    size_t status = 0, partial = 0, gsum = 0, counters = 0, centroid = 0, score = 0, cut = 0, chunk = 0, kept = 0,
           idx = 0, total = 0;
};

Geometry make_geometry(int32_t batch, int32_t heads, int32_t t_max, int32_t window, int32_t head_dim = kHeadDim,
                       int32_t es = 2);
Layout make_layout(const Geometry &g);

// Occupancy helpers (kernels loop over their items, persistent style).
int resident_grid(const void *fn, int threads, size_t dyn_smem);              // SMs x resident CTAs per SM
int grid_for_items(const void *fn, int threads, size_t dyn_smem, int64_t items);

// Kernel launchers: each enqueues its kernel(s) on `st` and returns the
// launch error (cudaSuccess when fine).
cudaError_t launch_piece_sums(const PieceGeometry &g, const void *K, const int32_t *seq_lens, float *partial,
                              uint32_t *status, cudaStream_t st);
cudaError_t launch_window_means(const PieceGeometry &g, const float *partial, const int32_t *seq_lens, float *C,
                                uint32_t *status, cudaStream_t st);
cudaError_t launch_piece_scores(const PieceGeometry &g, const void *K, const float *C, const int32_t *seq_lens,
                                int mode, float *S, uint32_t *status, cudaStream_t st);
// CTAs the single-pass centroid + score kernel runs with on the current
// device (0 on error); it is usable when this is at least g.ppw.
int single_pass_grid(int mode);
// Clears the arrival counters, then launches the single-pass kernel
// cooperatively with `grid` CTAs.
// With stall_windows (failure injection) no window ever becomes ready.
cudaError_t launch_single_pass(const PieceGeometry &g, int grid, const void *K, const int32_t *seq_lens, int mode,
                               float *partial, float *gsum, uint32_t *cnt, float *C, float *S, uint32_t *status,
                               cudaStream_t st, bool stall_windows = false);
// Head groups (one read of K from HBM for a1 + a2): the plan has groups = 0
// when the shape does not qualify (a global centroid over a head too long
// for L2, too few resident CTAs, or too little counter space).
struct HeadGroupPlan {
    int groups = 0;
    int gsize = 0;  // CTAs per group
    int wb = 0;     // windows per unit
    uint32_t stagger_ns = 0;  // start delay step: group g waits (g mod 4) steps
    bool ring = false;        // the copy-ring kernel (pass 1 streamed by a producer warp)
};
HeadGroupPlan head_group_plan(const PieceGeometry &g, int mode, size_t counter_bytes);
// The plan of the copy-ring head-group kernel (bf16, head dim 128); groups 0
// when it does not apply.
HeadGroupPlan head_group_ring_plan(const PieceGeometry &g, int mode, size_t counter_bytes);
// The fused whole-path kernel (global centroids, heads of at most 20480
// tokens): scorer head groups within `scorer_ctas` CTAs (< 0: 3/4 of the
// resident grid), `select_ctas`
// selector CTAs, every warp a gatherer afterwards; grid 0 when it does not
// apply. launch_fused's `stall` injects a wait that cannot end (failure
// tests only): 0 the barrier of scorer group 0, 1 the select of head 0; -1
// none.
struct FusedPlan {
    HeadGroupPlan hg;
    int grid = 0;         // resident CTAs of the launch
    int select_ctas = 0;  // CTAs that run the selects
};
FusedPlan fused_plan(const PieceGeometry &g, int mode, size_t counter_bytes, int scorer_ctas, int select_ctas);
cudaError_t launch_fused(const PieceGeometry &g, const FusedPlan &fp, int mode, const void *K, const void *V,
                         const int32_t *seq_lens, float *partial, uint32_t *cnt, float *C, float *S, double ratio,
                         const int32_t *n_keep, int32_t keep_stride, int32_t *kept, int32_t *idx, int32_t idx_stride,
                         void *K_out, void *V_out, uint32_t *status, cudaStream_t st, int stall = -1);
cudaError_t launch_head_groups(const PieceGeometry &g, const HeadGroupPlan &plan, const void *K,
                               const int32_t *seq_lens, int mode, float *partial, uint32_t *cnt, float *C, float *S,
                               uint32_t *status, cudaStream_t st);
// Radix select. With idx (only when select_emits_indices(g): the head's
// scores fit in shared memory) it also writes the ascending kept indices to
// idx[head * idx_stride + slot] and the kept counts (no compaction kernel
// needed); else with chunk_info it computes the per-chunk output offsets and
// the kept counts for k_compact (the fused path's fourth pass).
bool select_emits_indices(const Geometry &g);
// True when the shared-memory select gives every head a CTA at once (one
// wave): then it and the gather after it run as programmatic dependent
// launches (measured to hide the launch gaps there, and to slow down a
// select of many rounds).
bool select_single_wave(const Geometry &g);
cudaError_t launch_select(const Geometry &g, const float *S, const int32_t *seq_lens, double ratio,
                          const int32_t *n_keep, int32_t keep_stride, mkv_cut *cut, int2 *chunk_info,
                          int32_t *kept, int32_t *idx, int32_t idx_stride, uint32_t *status, cudaStream_t st);
// Per-window-quota selection: every window keeps n_keep(|w|, ratio) of its
// own tokens (window 0 or >= t_max: one window, the ordinary selection);
// writes the ascending kept indices to idx[head * idx_stride + slot] and the
// kept counts.
cudaError_t launch_select_quota(const Geometry &g, const float *S, const int32_t *seq_lens, double ratio,
                                int32_t keep_stride, int32_t *kept, int32_t *idx, int32_t idx_stride,
                                uint32_t *status, cudaStream_t st);
// Means (and, with radius, the largest distance of a member to its mean) of
// the windows of a bf16 tensor, 0 < window <= kSmallWindowMax.
cudaError_t launch_small_window_means(const PieceGeometry &g, const void *X, const int32_t *seq_lens, float *mean,
                                      float *radius, uint32_t *status, cudaStream_t st);
// In place: K/V rows [head][j] = K/V[head][idx[head * idx_stride + j]] for
// j < kept[head], inside the head's own rows (idx ascending).
cudaError_t launch_gather_inplace(const Geometry &g, const int32_t *idx, int32_t idx_stride, const int32_t *kept,
                                  const int32_t *seq_lens, void *K, void *V, uint32_t *status, cudaStream_t st);
// OjaKV-style reconstruction-error scores (mkv_oja.cu): the projected query
// rows (hi + lo bf16, oja_operand_bytes in `qhl`), then the tcgen05
// contraction writing S[head * t_max + t] for t < T_head.
size_t oja_operand_bytes(int64_t n_heads, int32_t n_query);
int oja_stages(int32_t n_query);
// the CTA-pair contraction: the setting (returns the previous one) and whether it runs for n_query
int oja_set_pair(int enable);
bool oja_uses_pair(int32_t n_query);
cudaError_t launch_oja_scores(const Geometry &g, const void *K, const void *Q, const float *U, const int32_t *seq_lens,
                              int32_t n_query, int32_t rank, void *qhl, float *S, uint32_t *status, cudaStream_t st,
                              void *const *events = nullptr);
cudaError_t launch_chunk_offsets(const Geometry &g, const float *S, const mkv_cut *cut,
                                 const int32_t *seq_lens, double ratio, const int32_t *n_keep,
                                 int32_t keep_stride, int2 *chunk_info, int32_t *kept,
                                 uint32_t *status, cudaStream_t st);
// Ascending kept indices into idx[head * idx_stride + slot], slot < keep_stride.
cudaError_t launch_compact(const Geometry &g, const float *S, const mkv_cut *cut, const int2 *chunk_info,
                           const int32_t *seq_lens, int32_t keep_stride, int32_t *idx, int32_t idx_stride,
                           uint32_t *status, cudaStream_t st);
// K_out/V_out rows [head][j] = K/V[head][idx[head * idx_stride + j]] for j < kept[head].
cudaError_t launch_gather(const Geometry &g, const int32_t *idx, int32_t idx_stride, const int32_t *kept,
                          int32_t keep_stride, const void *K, const void *V, void *K_out, void *V_out,
                          uint32_t *status, cudaStream_t st, bool pdl = false);

}  // namespace mkv
