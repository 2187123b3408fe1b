/*
 * mkv_oracle.c -- the fp64 CPU oracle for ManifoldKV-style KV-cache
 * compression.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, plain reference that the
 * CUDA library is checked against. Only the test suite, the smoke check and
 * the bench's CPU-baseline / reference leg may load it; the library never
 * does, and it shares no code, header, table or helper with the library.
 *
 * What it computes (per head = one (layer, sequence, KV head) triple), from
 * "ManifoldKV: Training-Free KV Cache Compression via Euclidean Outlier
 * Detection" (ICML 2026 poster 62526), abstract and lay summary:
 *   1. the key centroid -- the mean key of the head; the windowed variant
 *      (WindowedManifoldKV, abstract) uses one mean per non-overlapping
 *      window of W tokens instead of one global mean;
 *   2. a score per token: its Euclidean distance to its centroid (the
 *      ManifoldKV scorer, abstract), or, as the switchable baseline, one
 *      minus its cosine similarity to the centroid (the KeyDiff-style scorer
 *      the abstract compares against);
 *   3. the tokens that sit farthest from the centroid are the ones retained
 *      (lay summary): keep the n_keep highest scores, where the compression
 *      percentage is the fraction of tokens removed (abstract: "20%
 *      compression" at 95.7% accuracy);
 *   4. the kept key and value rows, in ascending token order, form the
 *      compacted cache.
 * Readings where the pages are silent (each one is also listed in the design
 * notes): ties at the cut go to the lower token index; n_keep =
 * floor(T*(1-ratio) + 0.5) clamped to [0, T]; the last window holds the
 * remaining T mod W tokens; a cosine score with a zero key or zero centroid
 * is 1; the selection is one global top-n_keep per head even when the
 * centroids are per window.
 *
 * Everything is fp64, summed in token order, with no blocking or reordering.
 * Keys arrive as raw bfloat16 bit patterns (uint16); decoding them to double
 * is exact. fp8 (E4M3) caches are widened exactly to bfloat16 first
 * (oracle_e4m3_to_bf16) and their kept rows are copied as bytes
 * (oracle_gather_bytes). Compile with -ffp-contract=off so every operation
 * rounds once.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MODE_L2 0
#define ORACLE_MODE_COSINE 1

/* bfloat16 is the upper half of an IEEE binary32: shifting the 16 bits into
 * the top of a 32-bit word gives the float exactly; float -> double is exact. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* fp8 caches hold OCP 8-bit floating point E4M3 codes (the "OCP 8-bit
 * Floating Point Specification (OFP8)", E4M3 encoding; torch's
 * float8_e4m3fn): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent field 0 is subnormal, m * 2^-9; no infinities; S.1111.111 is NaN.
 * The method runs on the decoded values, which this returns exactly (NaN
 * for the NaN codes, which are outside the contract). */
double oracle_e4m3_to_double(uint8_t code)
{
    int neg = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + (double)m, e - 10); /* (1 + m/8) 2^(e-7) */
    return neg ? -v : v;
}

/* Every finite E4M3 value is a bfloat16 value (3 mantissa bits fit in 7, and
 * 2^-9 .. 448 lies inside bf16's normal range), so an fp8 cache widens to a
 * bf16 cache exactly and every step below runs on it unchanged. Writes the
 * bf16 bit patterns of n codes; returns -1 (nothing defined) on a NaN code. */
int oracle_e4m3_to_bf16(const uint8_t *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) {
        double v = oracle_e4m3_to_double(x[i]);
        if (v != v) return -1;
        float f = (float)v; /* exact */
        uint32_t w;
        memcpy(&w, &f, sizeof w);
        if (w & 0xFFFFu) return -1; /* cannot happen for a finite E4M3 value */
        out[i] = (uint16_t)(w >> 16);
    }
    return 0;
}

/* Step 4 for caches of any element type: row idx[j] of X (row_bytes bytes
 * per row) copied to row j of out. */
void oracle_gather_bytes(const uint8_t *X, int64_t row_bytes, const int32_t *idx, int64_t n, uint8_t *out)
{
    for (int64_t j = 0; j < n; ++j) memcpy(out + j * row_bytes, X + (int64_t)idx[j] * row_bytes, (size_t)row_bytes);
}

/* Step 3, reading of "% compression": the percentage is the share removed,
 * so round(T * (1 - ratio)) tokens stay; halves round up. */
int64_t oracle_num_keep(int64_t T, double ratio)
{
    if (T <= 0) return 0;
    double keep = floor((double)T * (1.0 - ratio) + 0.5);
    if (keep < 0.0) return 0;
    if (keep > (double)T) return T;
    return (int64_t)keep;
}

/* Window tiling of step 1: window <= 0 or window >= T means one global
 * window; otherwise non-overlapping windows [jW, min((j+1)W, T)). */
int64_t oracle_window_len(int64_t T, int64_t window)
{
    if (window <= 0 || window >= T) return T;
    return window;
}

int64_t oracle_num_windows(int64_t T, int64_t window)
{
    if (T <= 0) return 0;
    int64_t w = oracle_window_len(T, window);
    return (T + w - 1) / w;
}

/* Step 1: C[j][i] = (1/|w_j|) * sum_{t in w_j} K[t][i], summed in token order.
 * K: T x d bf16 bits, row-major. C: num_windows x d doubles. */
void oracle_centroids(const uint16_t *K, int64_t T, int64_t d, int64_t window, double *C)
{
    int64_t wl = oracle_window_len(T, window);
    int64_t nw = oracle_num_windows(T, window);
    for (int64_t j = 0; j < nw; ++j) {
        int64_t a = j * wl;
        int64_t b = a + wl < T ? a + wl : T;
        for (int64_t i = 0; i < d; ++i) {
            double sum = 0.0;
            for (int64_t t = a; t < b; ++t) sum += oracle_bf16_to_double(K[t * d + i]);
            C[j * d + i] = sum / (double)(b - a);
        }
    }
}

/* Step 2: each token is scored against the centroid of its own window.
 *   L2:     s_t = sqrt( sum_i (k_ti - c_i)^2 )
 *   cosine: s_t = 1 - (k_t . c) / (|k_t| |c|), and 1 when |k_t| |c| = 0. */
void oracle_scores(const uint16_t *K, int64_t T, int64_t d, int64_t window, int mode,
                   const double *C, double *S)
{
    int64_t wl = oracle_window_len(T, window);
    for (int64_t t = 0; t < T; ++t) {
        const double *c = C + (t / wl) * d;
        if (mode == ORACLE_MODE_L2) {
            double ss = 0.0;
            for (int64_t i = 0; i < d; ++i) {
                double diff = oracle_bf16_to_double(K[t * d + i]) - c[i];
                ss += diff * diff;
            }
            S[t] = sqrt(ss);
        } else {
            double dot = 0.0, kk = 0.0, cc = 0.0;
            for (int64_t i = 0; i < d; ++i) {
                double k = oracle_bf16_to_double(K[t * d + i]);
                dot += k * c[i];
                kk += k * k;
                cc += c[i] * c[i];
            }
            double denom = sqrt(kk) * sqrt(cc);
            S[t] = denom == 0.0 ? 1.0 : 1.0 - dot / denom;
        }
    }
}

typedef struct {
    double score;
    int64_t token;
} oracle_ranked;

/* Order by score descending, then token index ascending (ties at the cut go
 * to the lower index). The order is total, so qsort's instability is moot. */
static int oracle_rank_cmp(const void *pa, const void *pb)
{
    const oracle_ranked *a = (const oracle_ranked *)pa, *b = (const oracle_ranked *)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->token > b->token) - (a->token < b->token);
}

static int oracle_index_cmp(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/* Step 3: full sort of (score desc, index asc); the first n_keep tokens are
 * retained; their indices are emitted in ascending order (step 4's order).
 * Returns 0, or -1 if a score is NaN or memory runs out. */
int oracle_select(const double *S, int64_t T, int64_t n_keep, int32_t *idx)
{
    if (n_keep < 0 || n_keep > T) return -1;
    oracle_ranked *r = (oracle_ranked *)malloc((size_t)(T > 0 ? T : 1) * sizeof *r);
    if (!r) return -1;
    for (int64_t t = 0; t < T; ++t) {
        if (isnan(S[t])) { free(r); return -1; }
        r[t].score = S[t];
        r[t].token = t;
    }
    qsort(r, (size_t)T, sizeof *r, oracle_rank_cmp);
    for (int64_t j = 0; j < n_keep; ++j) idx[j] = (int32_t)r[j].token;
    free(r);
    qsort(idx, (size_t)n_keep, sizeof *idx, oracle_index_cmp);
    return 0;
}

/* Step 4: out[j] = X[idx[j]], whole rows of d bf16 values, bit for bit. */
void oracle_gather(const uint16_t *X, int64_t d, const int32_t *idx, int64_t n, uint16_t *out)
{
    for (int64_t j = 0; j < n; ++j)
        memcpy(out + j * d, X + (int64_t)idx[j] * d, (size_t)d * sizeof *X);
}

/* Steps 1-4 for one head. C (num_windows x d) and S (T) are caller scratch;
 * idx, K_out, V_out receive n_keep entries / rows. Returns n_keep or -1. */
int64_t oracle_compress_head(const uint16_t *K, const uint16_t *V, int64_t T, int64_t d,
                             double ratio, int mode, int64_t window,
                             double *C, double *S, int32_t *idx, uint16_t *K_out, uint16_t *V_out)
{
    int64_t n_keep = oracle_num_keep(T, ratio);
    oracle_centroids(K, T, d, window, C);
    oracle_scores(K, T, d, window, mode, C, S);
    if (oracle_select(S, T, n_keep, idx) != 0) return -1;
    if (K_out) oracle_gather(K, d, idx, n_keep, K_out);
    if (V_out) oracle_gather(V, d, idx, n_keep, V_out);
    return n_keep;
}

/* The same for n_heads heads laid out back to back with row stride t_stride
 * (a [heads, t_stride, d] cache); head h has lens[h] tokens. Outputs use row
 * stride keep_stride per head. The plain loop over heads is what the bench's
 * CPU baseline times. Returns 0, or -1 on the first failing head. */
int oracle_compress_heads(const uint16_t *K, const uint16_t *V, int64_t n_heads, int64_t t_stride,
                          int64_t d, const int32_t *lens, double ratio, int mode, int64_t window,
                          int64_t keep_stride, int32_t *idx, int32_t *kept,
                          uint16_t *K_out, uint16_t *V_out)
{
    double *C = (double *)malloc((size_t)(t_stride > 0 ? t_stride : 1) * (size_t)d * sizeof(double));
    double *S = (double *)malloc((size_t)(t_stride > 0 ? t_stride : 1) * sizeof(double));
    if (!C || !S) { free(C); free(S); return -1; }
    int rc = 0;
    for (int64_t h = 0; h < n_heads && rc == 0; ++h) {
        int64_t T = lens[h];
        if (T < 0 || T > t_stride || oracle_num_keep(T, ratio) > keep_stride) { rc = -1; break; }
        int64_t n = oracle_compress_head(K + h * t_stride * d, V + h * t_stride * d, T, d, ratio,
                                         mode, window, C, S, idx + h * keep_stride,
                                         K_out ? K_out + h * keep_stride * d : NULL,
                                         V_out ? V_out + h * keep_stride * d : NULL);
        if (n < 0) rc = -1;
        else kept[h] = (int32_t)n;
    }
    free(C);
    free(S);
    return rc;
}

/* Per-layer kept-token budgets, "RippleKV" (gist.science explainer of arXiv
 * 2608.08684), Methodology section 2, Sensitivity-Guided Budget Allocation:
 * layer sensitivities are normalised to [0, 1], mapped to multipliers
 * w = r^s, clipped to [1/gamma, gamma], and scaled so that the layer budgets
 * add up to the global budget. Readings where the text is silent: all-equal
 * sensitivities normalise to 0; a layer's budget cannot exceed its tokens
 * cap[l] -- the allocation is min(cap, lambda * w) with lambda chosen so the
 * total is met (found here by bisection); real budgets become integers by
 * largest remainder (ties to the lower layer). Returns 0, 1 when the caps
 * cannot absorb the total (every layer gets its cap), -1 on bad input. */
static double oracle_alloc_sum(const double *w, const int32_t *cap, int32_t L, double lam)
{
    double sum = 0.0;
    for (int32_t l = 0; l < L; ++l) {
        double x = lam * w[l];
        sum += x < (double)cap[l] ? x : (double)cap[l];
    }
    return sum;
}

int oracle_layer_budgets(const double *sens, int32_t L, double r, double gamma, int64_t total,
                         const int32_t *cap, int32_t *budget)
{
    if (L <= 0 || !(r > 0.0) || !(gamma >= 1.0) || total < 0) return -1;
    double smin = sens[0], smax = sens[0];
    int64_t capsum = 0;
    for (int32_t l = 0; l < L; ++l) {
        if (isnan(sens[l]) || cap[l] < 0) return -1;
        if (sens[l] < smin) smin = sens[l];
        if (sens[l] > smax) smax = sens[l];
        capsum += cap[l];
    }
    if (total >= capsum) {
        for (int32_t l = 0; l < L; ++l) budget[l] = cap[l];
        return total == capsum ? 0 : 1;
    }
    double *w = (double *)malloc((size_t)L * sizeof(double));
    double *x = (double *)malloc((size_t)L * sizeof(double));
    if (!w || !x) { free(w); free(x); return -1; }
    for (int32_t l = 0; l < L; ++l) {
        double s = smax > smin ? (sens[l] - smin) / (smax - smin) : 0.0;
        double m = pow(r, s);
        if (m < 1.0 / gamma) m = 1.0 / gamma;
        if (m > gamma) m = gamma;
        w[l] = m;
    }
    /* lambda by bisection: the allocated sum is nondecreasing in lambda */
    double lo = 0.0, hi = 1.0;
    while (oracle_alloc_sum(w, cap, L, hi) < (double)total) hi *= 2.0;
    for (int it = 0; it < 200; ++it) {
        double mid = 0.5 * (lo + hi);
        if (oracle_alloc_sum(w, cap, L, mid) < (double)total) lo = mid; else hi = mid;
    }
    int64_t assigned = 0;
    for (int32_t l = 0; l < L; ++l) {
        double v = hi * w[l];
        x[l] = v < (double)cap[l] ? v : (double)cap[l];
        budget[l] = (int32_t)floor(x[l]);
        assigned += budget[l];
    }
    /* largest remainder: one more token to the layers with the largest
     * fractional part, lower index first among equals */
    while (assigned < total) {
        int32_t best = -1;
        double bestf = -1.0;
        for (int32_t l = 0; l < L; ++l) {
            double f = x[l] - (double)budget[l];
            if (budget[l] < cap[l] && f > bestf) { bestf = f; best = l; }
        }
        if (best < 0) break;
        budget[best] += 1;
        x[best] = (double)budget[best];  /* its remainder is used */
        assigned += 1;
    }
    free(w);
    free(x);
    return 0;
}

/* Steps 1-4 for one head with an explicit kept count (per-layer budgets). */
int64_t oracle_compress_head_n(const uint16_t *K, const uint16_t *V, int64_t T, int64_t d, int64_t n_keep,
                               int mode, int64_t window, double *C, double *S, int32_t *idx,
                               uint16_t *K_out, uint16_t *V_out)
{
    if (n_keep < 0 || n_keep > T) return -1;
    oracle_centroids(K, T, d, window, C);
    oracle_scores(K, T, d, window, mode, C, S);
    if (oracle_select(S, T, n_keep, idx) != 0) return -1;
    if (K_out) oracle_gather(K, d, idx, n_keep, K_out);
    if (V_out) oracle_gather(V, d, idx, n_keep, V_out);
    return n_keep;
}

/* Cluster summaries, "RefineKV: Query-Adaptive KV Cache Compression via
 * Attention-Error Bounds" (project page), method overview, step 1
 * (Summarize): the cache is cut into contiguous clusters, and each cluster's
 * mean key, mean value and some metadata are cached. The clusters here are
 * the windows of step 1 (W tokens each, the last one holding the rest), and
 * the mean is the one oracle_centroids computes, applied to whichever tensor
 * X is passed (keys or values). The metadata taken here (a reading; the page
 * does not list it) is the cluster's size, implied by the tiling, and
 * radius[j] = max over t in window j of |X_t - mean_j|_2. That is what a
 * query-time bound on how far a member's logit can drift from the mean's
 * needs (|q.k_t - q.mean| <= |q| * radius, Cauchy-Schwarz; Figure 2's
 * logit-deviation bound). radius may be NULL. */
void oracle_window_means(const uint16_t *X, int64_t T, int64_t d, int64_t window, double *mean, double *radius)
{
    oracle_centroids(X, T, d, window, mean);
    if (!radius) return;
    int64_t wl = oracle_window_len(T, window);
    int64_t nw = oracle_num_windows(T, window);
    for (int64_t j = 0; j < nw; ++j) {
        int64_t a = j * wl;
        int64_t b = a + wl < T ? a + wl : T;
        double rmax = 0.0;
        for (int64_t t = a; t < b; ++t) {
            double ss = 0.0;
            for (int64_t i = 0; i < d; ++i) {
                double diff = oracle_bf16_to_double(X[t * d + i]) - mean[j * d + i];
                ss += diff * diff;
            }
            double r = sqrt(ss);
            if (r > rmax) rmax = r;
        }
        radius[j] = rmax;
    }
}

/* Per-window quota variant of WindowedManifoldKV (a reading of the abstract,
 * which replaces the global centroid by per-window centroids and says
 * nothing more about the selection): every window keeps its own share
 * oracle_num_keep(|w|, ratio) of its tokens, the highest-scoring ones within
 * it (ties to the lower index), instead of one top-n over the whole head.
 * Total kept tokens of a head of T tokens: */
int64_t oracle_num_keep_quota(int64_t T, double ratio, int64_t window)
{
    int64_t wl = oracle_window_len(T, window);
    int64_t nw = oracle_num_windows(T, window);
    int64_t total = 0;
    for (int64_t j = 0; j < nw; ++j) {
        int64_t a = j * wl;
        int64_t b = a + wl < T ? a + wl : T;
        total += oracle_num_keep(b - a, ratio);
    }
    return total;
}

/* Selection with a per-window quota: oracle_select on each window's scores,
 * indices shifted to head positions and concatenated in window order (so
 * they ascend). Returns the number kept, or -1. */
int64_t oracle_select_quota(const double *S, int64_t T, int64_t window, double ratio, int32_t *idx)
{
    int64_t wl = oracle_window_len(T, window);
    int64_t nw = oracle_num_windows(T, window);
    int64_t n = 0;
    for (int64_t j = 0; j < nw; ++j) {
        int64_t a = j * wl;
        int64_t b = a + wl < T ? a + wl : T;
        int64_t q = oracle_num_keep(b - a, ratio);
        if (oracle_select(S + a, b - a, q, idx + n) != 0) return -1;
        for (int64_t k = 0; k < q; ++k) idx[n + k] += (int32_t)a;
        n += q;
    }
    return n;
}

/* Steps 1-4 for one head with per-window quotas. Returns the kept count or -1. */
int64_t oracle_compress_head_quota(const uint16_t *K, const uint16_t *V, int64_t T, int64_t d, double ratio,
                                   int mode, int64_t window, double *C, double *S, int32_t *idx,
                                   uint16_t *K_out, uint16_t *V_out)
{
    oracle_centroids(K, T, d, window, C);
    oracle_scores(K, T, d, window, mode, C, S);
    int64_t n = oracle_select_quota(S, T, window, ratio, idx);
    if (n < 0) return -1;
    if (K_out) oracle_gather(K, d, idx, n, K_out);
    if (V_out) oracle_gather(V, d, idx, n, V_out);
    return n;
}

/* OjaKV reconstruction-error score, "OjaKV: Context-Aware Online Low-Rank
 * KV Cache Compression" (deep notes of the ACL 2026 Findings paper), method
 * details, error-based token selection for the hybrid storage: the residual
 * r_t = k_t - U U^T k_t is the part of key t its low-rank reconstruction
 * misses, and
 *     e_t = (1/|W|) * sum over (head h, query q) in W of |q_{h,q}^T r_t / sqrt(d)|
 * weighs it by the recent query window W of every query head that reads
 * this KV head. The tokens with the largest errors stay at full rank (the
 * top-k of the normalised errors; a per-head normaliser does not change the
 * order, so the selection is the top-n_keep of e itself).
 * K: T x d bf16 bits; Q: M x d bf16 bits, the window's query rows (group
 * heads x recent positions, flattened, |W| = M); U: d x r doubles,
 * row-major (column j is basis vector j). E: T doubles. */
void oracle_oja_scores(const uint16_t *K, int64_t T, int64_t d, const uint16_t *Q, int64_t M,
                       const double *U, int64_t r, double *E)
{
    double *k = (double *)malloc((size_t)d * sizeof(double));
    double *y = (double *)malloc((size_t)(r > 0 ? r : 1) * sizeof(double));
    double *res = (double *)malloc((size_t)d * sizeof(double));
    if (!k || !y || !res) { free(k); free(y); free(res); return; }
    double sqrt_d = sqrt((double)d);
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t i = 0; i < d; ++i) k[i] = oracle_bf16_to_double(K[t * d + i]);
        for (int64_t j = 0; j < r; ++j) {          /* y = U^T k */
            double s = 0.0;
            for (int64_t i = 0; i < d; ++i) s += U[i * r + j] * k[i];
            y[j] = s;
        }
        for (int64_t i = 0; i < d; ++i) {          /* r_t = k - U y */
            double s = 0.0;
            for (int64_t j = 0; j < r; ++j) s += U[i * r + j] * y[j];
            res[i] = k[i] - s;
        }
        double acc = 0.0;
        for (int64_t m = 0; m < M; ++m) {
            double dot = 0.0;
            for (int64_t i = 0; i < d; ++i) dot += oracle_bf16_to_double(Q[m * d + i]) * res[i];
            acc += fabs(dot / sqrt_d);
        }
        E[t] = M > 0 ? acc / (double)M : 0.0;
    }
    free(k);
    free(y);
    free(res);
}

/* OjaKV's full-rank selection for one head: errors, top-n_keep (ties to the
 * lower index, ascending), and the kept K/V rows. Returns n_keep or -1. */
int64_t oracle_compress_head_oja(const uint16_t *K, const uint16_t *V, int64_t T, int64_t d, const uint16_t *Q,
                                 int64_t M, const double *U, int64_t r, int64_t n_keep, double *E, int32_t *idx,
                                 uint16_t *K_out, uint16_t *V_out)
{
    if (n_keep < 0 || n_keep > T) return -1;
    oracle_oja_scores(K, T, d, Q, M, U, r, E);
    if (oracle_select(E, T, n_keep, idx) != 0) return -1;
    if (K_out) oracle_gather(K, d, idx, n_keep, K_out);
    if (V_out) oracle_gather(V, d, idx, n_keep, V_out);
    return n_keep;
}

/* In-place compaction (the memory-saving form of step 4): the kept rows are
 * moved to the front of the head's own rows, X[j] = X[idx[j]] for j < n;
 * rows from n on keep their contents. Done one row at a time in ascending j,
 * which is safe because idx ascends from 0, so idx[j] >= j: every source row
 * is read before anything overwrites it. Returns 0, or -1 if idx is not
 * strictly ascending or leaves [0, T). */
int oracle_compact_in_place(uint16_t *X, int64_t T, int64_t d, const int32_t *idx, int64_t n)
{
    for (int64_t j = 0; j < n; ++j)
        if (idx[j] < 0 || idx[j] >= T || (j > 0 && idx[j] <= idx[j - 1])) return -1;
    for (int64_t j = 0; j < n; ++j)
        if (idx[j] != j) memcpy(X + j * d, X + (int64_t)idx[j] * d, (size_t)d * sizeof *X);
    return 0;
}
