"""Pins of the fp64 oracle to things other than itself.

Each test ties one oracle function to a hand-worked case, a closed form, an
invariant of the definitions, a library routine computing the same quantity a
different way, or brute force on tiny inputs. Together they are chosen so
that a plausible slip anywhere in the oracle (a dropped term, a wrong sign,
divisor or window index, an inverted ranking or tie rule, a transposed
operand, a wrong rounding of the kept count) fails at least one of them.

Definitions followed: "ManifoldKV: Training-Free KV Cache Compression via
Euclidean Outlier Detection" (ICML 2026 poster 62526), abstract and lay
summary.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.spatial.distance import cdist

import oracle
import synthkv


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "hand_cases.json")) as f:
        return json.load(f)


def _bf16(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _f64(K):
    return K.to(torch.float64).numpy()


# --- decoding ------------------------------------------------------------------

def test_bf16_decode_matches_torch_for_every_finite_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    lib = oracle._load()
    got = np.array([lib.oracle_bf16_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isinf(got), np.isinf(ref))


# --- kept count ----------------------------------------------------------------

def test_num_keep_table(golden_dir):
    for T, r, want, _why in _golden(golden_dir)["num_keep"]:
        assert oracle.num_keep(T, r) == want, (T, r)


def test_num_keep_is_nearest_integer_and_clamped():
    rng = np.random.default_rng(1)
    for _ in range(2000):
        T = int(rng.integers(0, 200000))
        r = float(rng.random())
        x = T * (1.0 - r)
        k = oracle.num_keep(T, r)
        assert 0 <= k <= T
        assert abs(k - x) <= 0.5 + 1e-9


# --- hand-worked cases ----------------------------------------------------------

@pytest.mark.parametrize("case_ix", range(5))
def test_hand_cases(golden_dir, case_ix):
    case = _golden(golden_dir)["cases"][case_ix]
    K = _bf16(case["keys"])
    w, mode = case["window"], case["mode"]
    C = oracle.centroids(K, w)
    np.testing.assert_array_equal(C, np.array(case["centroids"], dtype=np.float64))
    S = oracle.scores(K, C, w, mode)
    if "scores_squared" in case:
        np.testing.assert_allclose(S ** 2, case["scores_squared"], rtol=1e-14, atol=0)
    else:
        want = [eval(e, {"sqrt": math.sqrt}) for e in case["scores_closed_form"]]
        np.testing.assert_allclose(S, want, rtol=0, atol=1e-14)
    for r, idx in case["keep"].items():
        n = oracle.num_keep(len(case["keys"]), float(r))
        assert n == len(idx)
        assert oracle.select(S, n).tolist() == idx, (case["name"], r)
        full = oracle.compress_head(K, K, float(r), mode, w)
        assert full["idx"].tolist() == idx


# --- centroid -----------------------------------------------------------------

@pytest.mark.parametrize("T,window", [(1000, 0), (1000, 1000), (1000, 128), (1001, 100), (37, 5), (64, 1)])
def test_centroid_equals_library_mean(T, window):
    rng = np.random.default_rng(T + window)
    K = _bf16(rng.normal(size=(T, 64)) * 3 + 0.5)
    C = oracle.centroids(K, window)
    k = _f64(K)
    wl = T if window <= 0 or window >= T else window
    want = np.stack([k[a:a + wl].mean(axis=0) for a in range(0, T, wl)])
    assert C.shape == want.shape
    np.testing.assert_allclose(C, want, rtol=1e-13, atol=1e-13)


def test_centroid_closed_form_sum_of_squares():
    # I9: sum_t |k_t - c|^2 = sum_t |k_t|^2 - T |c|^2, and c minimises it.
    rng = np.random.default_rng(7)
    K = _bf16(rng.normal(size=(4096, 128)) * np.exp(0.5 * rng.normal(size=(4096, 1))))
    C = oracle.centroids(K, 0)
    S = oracle.scores(K, C, 0, "l2")
    k = _f64(K)
    lhs = np.sum(S ** 2)
    rhs = np.sum(k * k) - k.shape[0] * np.sum(C[0] ** 2)
    assert abs(lhs - rhs) <= 1e-12 * abs(rhs)
    for _ in range(4):
        c2 = C + rng.normal(size=C.shape) * 1e-3
        assert np.sum(oracle.scores(K, c2, 0, "l2") ** 2) > lhs


# --- scores -------------------------------------------------------------------

@pytest.mark.parametrize("window", [0, 256, 100])
def test_l2_scores_equal_library_distance(window):
    rng = np.random.default_rng(3)
    K = _bf16(rng.normal(size=(1000, 128)) * 2 - 1)
    C = oracle.centroids(K, window)
    S = oracle.scores(K, C, window, "l2")
    k = _f64(K)
    wl = oracle.window_len(1000, window)
    want = np.array([cdist(k[t:t + 1], C[t // wl][None], "euclidean")[0, 0] for t in range(1000)])
    np.testing.assert_allclose(S, want, rtol=1e-13, atol=0)


@pytest.mark.parametrize("window", [0, 300])
def test_cosine_scores_equal_library_cosine_distance(window):
    rng = np.random.default_rng(4)
    K = _bf16(rng.normal(size=(900, 128)) + 0.3)
    C = oracle.centroids(K, window)
    S = oracle.scores(K, C, window, "cosine")
    k = _f64(K)
    wl = oracle.window_len(900, window)
    want = np.array([cdist(k[t:t + 1], C[t // wl][None], "cosine")[0, 0] for t in range(900)])
    np.testing.assert_allclose(S, want, rtol=0, atol=1e-13)
    assert S.min() >= -1e-15 and S.max() <= 2 + 1e-15


def test_l2_translation_invariance_exact():
    # I3: integer keys, power-of-two T: every fp64 sum is exact, so shifting all
    # keys by v leaves the scores bit for bit unchanged.
    rng = np.random.default_rng(5)
    base = rng.integers(-20, 20, size=(256, 128)).astype(np.float32)
    v = rng.integers(-50, 50, size=(1, 128)).astype(np.float32)
    K1, K2 = _bf16(base), _bf16(base + v)
    for window in (0, 64):
        S1 = oracle.scores(K1, oracle.centroids(K1, window), window, "l2")
        S2 = oracle.scores(K2, oracle.centroids(K2, window), window, "l2")
        np.testing.assert_array_equal(S1, S2)


def test_cosine_scale_invariance():
    # I4: a global alpha > 0 leaves cosine scores unchanged (exact for powers of
    # two); a per-token alpha_t against a fixed centroid also does.
    rng = np.random.default_rng(6)
    base = rng.normal(size=(512, 128)).astype(np.float32)
    K1 = _bf16(base)
    K2 = _bf16(base.astype(np.float64) * 8.0)
    S1 = oracle.scores(K1, oracle.centroids(K1, 0), 0, "cosine")
    S2 = oracle.scores(K2, oracle.centroids(K2, 0), 0, "cosine")
    np.testing.assert_array_equal(S1, S2)
    alpha = 2.0 ** rng.integers(-3, 4, size=(512, 1))
    K3 = _bf16(K1.to(torch.float64).numpy() * alpha)
    C = oracle.centroids(K1, 0)
    np.testing.assert_allclose(oracle.scores(K3, C, 0, "cosine"), S1, rtol=0, atol=1e-15)
    # l2 is not scale invariant: the pin above would not pass for it
    assert not np.allclose(oracle.scores(K2, oracle.centroids(K2, 0), 0, "l2"),
                           oracle.scores(K1, oracle.centroids(K1, 0), 0, "l2"))


@pytest.mark.parametrize("mode", ["l2", "cosine"])
def test_window_at_least_T_equals_global(mode):
    # I5
    rng = np.random.default_rng(8)
    K = _bf16(rng.normal(size=(300, 128)))
    ref = oracle.compress_head(K, K, 0.3, mode, 0)
    for w in (300, 301, 10 ** 6):
        got = oracle.compress_head(K, K, 0.3, mode, w)
        np.testing.assert_array_equal(got["S"], ref["S"])
        np.testing.assert_array_equal(got["idx"], ref["idx"])


def test_window_one_gives_zero_scores_and_lowest_indices():
    # I6: every token is its own centroid, all l2 scores are 0, ties keep the
    # lowest indices.
    rng = np.random.default_rng(9)
    K = _bf16(rng.normal(size=(100, 128)))
    out = oracle.compress_head(K, K, 0.37, "l2", 1)
    assert np.all(out["S"] == 0.0)
    assert out["idx"].tolist() == list(range(oracle.num_keep(100, 0.37)))


# --- selection ------------------------------------------------------------------

def test_select_brute_force_tiny():
    # I2: the kept set is the unique subset of size n in which every kept token
    # beats every dropped one by (score higher, or equal score and lower index).
    rng = np.random.default_rng(10)
    for trial in range(300):
        T = int(rng.integers(1, 9))
        S = rng.integers(0, 4, size=T).astype(np.float64) * 0.5
        n = int(rng.integers(0, T + 1))
        winners = []
        for subset in itertools.combinations(range(T), n):
            kept = set(subset)
            ok = all((S[i] > S[j]) or (S[i] == S[j] and i < j)
                     for i in kept for j in range(T) if j not in kept)
            if ok:
                winners.append(list(subset))
        assert len(winners) == 1
        assert oracle.select(S, n).tolist() == winners[0], (S, n)


def test_select_matches_stable_library_sort():
    rng = np.random.default_rng(11)
    for T in (1, 17, 1000, 4097):
        S = rng.integers(0, 50, size=T).astype(np.float64)
        n = int(rng.integers(0, T + 1))
        order = np.lexsort((np.arange(T), -S))
        assert oracle.select(S, n).tolist() == sorted(order[:n].tolist())


@pytest.mark.parametrize("T,ratio", [(1, 0.5), (2, 0.5), (513, 0.5), (1000, 0.0), (1000, 1.0), (4096, 0.2)])
def test_kept_count_exact_including_all_tied(T, ratio):
    # I8
    K = _bf16(np.ones((T, 128)))
    for mode in ("l2", "cosine"):
        out = oracle.compress_head(K, K, ratio, mode, 0)
        assert len(out["idx"]) == oracle.num_keep(T, ratio)
        assert out["idx"].tolist() == list(range(len(out["idx"])))


def test_gathered_rows_and_ascending_indices():
    # I10
    rng = np.random.default_rng(12)
    K = _bf16(rng.normal(size=(777, 128)))
    V = _bf16(rng.normal(size=(777, 128)))
    out = oracle.compress_head(K, V, 0.45, "l2", 100)
    idx = out["idx"]
    assert np.all(np.diff(idx) > 0)
    kb = K.view(torch.int16).numpy().view(np.uint16)
    vb = V.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(out["K_out"], kb[idx])
    np.testing.assert_array_equal(out["V_out"], vb[idx])


def test_planted_outliers_always_retained():
    # I7, on the single-layer 8-head 4096-token workload (seed 0): the tokens
    # planted at 4x the median norm sit far from the centroid and are kept, with
    # a wide margin over the cut.
    w = synthkv.WORKLOADS["single-layer-h8-t4096"]
    K, V, lens, planted = synthkv.make_kv(w, seed=0, with_planted=True)
    Kf = K.reshape(w.n_heads, w.t_max, w.head_dim)
    mode, window, ratio = w.runs[0]
    for h in range(w.n_heads):
        out = oracle.compress_head(Kf[h], Kf[h], ratio, mode, window)
        kept = set(out["idx"].tolist())
        assert len(kept) == 3277
        assert set(planted[h].tolist()) <= kept
        cut = np.sort(out["S"])[::-1][len(kept) - 1]
        assert out["S"][planted[h].numpy()].min() > 1.5 * cut


def test_compress_heads_matches_per_head_on_ragged_lengths():
    w = synthkv.WORKLOADS["ragged-b8-llama-kv-t8k-32k"].scaled(
        "ragged-small", layers=1, batch=3, heads=2, t_max=700, t_min=1, planted=4)
    K, V, lens = synthkv.make_kv(w, seed=3)
    Kf = K.reshape(w.n_heads, w.t_max, 128)
    Vf = V.reshape(w.n_heads, w.t_max, 128)
    hl = lens.repeat_interleave(w.heads)
    for mode, window, ratio in (("l2", 0, 0.5), ("cosine", 64, 0.2)):
        stride = oracle.num_keep(w.t_max, ratio)
        idx, kept, ko, vo = oracle.compress_heads(Kf, Vf, hl, ratio, mode, window, stride)
        for h in range(w.n_heads):
            T = int(hl[h])
            ref = oracle.compress_head(Kf[h, :T], Vf[h, :T], ratio, mode, window)
            assert kept[h] == len(ref["idx"])
            np.testing.assert_array_equal(idx[h, :kept[h]], ref["idx"])
            np.testing.assert_array_equal(ko[h, :kept[h]], ref["K_out"])
            np.testing.assert_array_equal(vo[h, :kept[h]], ref["V_out"])


def test_empty_head():
    K = _bf16(np.zeros((0, 128)))
    out = oracle.compress_head(K, K, 0.5, "l2", 0)
    assert len(out["idx"]) == 0 and len(out["S"]) == 0


# --- per-layer budgets ------------------------------------------------------------

def _budget_cases(golden_dir):
    with open(os.path.join(golden_dir, "budget_cases.json")) as f:
        return json.load(f)["cases"]


def test_layer_budgets_hand_cases(golden_dir):
    for c in _budget_cases(golden_dir):
        st, b = oracle.layer_budgets(c["s"], c["r"], c["gamma"], c["total"], c["cap"])
        assert st == c.get("status", 0), c
        assert b.tolist() == c["budget"], c


def test_layer_budgets_invariants():
    rng = np.random.default_rng(21)
    for _ in range(300):
        L = int(rng.integers(1, 40))
        s = rng.normal(size=L)
        r = float(np.exp(rng.normal()))
        gamma = float(1 + rng.exponential(3))
        cap = rng.integers(0, 5000, size=L)
        total = int(rng.integers(0, max(1, cap.sum())))
        st, b = oracle.layer_budgets(s, r, gamma, total, cap)
        assert st == 0
        assert int(b.sum()) == total
        assert np.all(b >= 0) and np.all(b <= cap)
    # no caps in the way: the allocation follows w within rounding
    s = rng.normal(size=16)
    st, b = oracle.layer_budgets(s, 3.0, 2.5, 160000, np.full(16, 10 ** 6))
    sn = (s - s.min()) / (s.max() - s.min())
    w = np.clip(3.0 ** sn, 1 / 2.5, 2.5)
    np.testing.assert_allclose(b, 160000 * w / w.sum(), atol=1.0)
    assert b.max() / b.min() <= 2.5 ** 2 + 1e-6
    # r = 1 is uniform; r > 1 gives more to more sensitive layers
    st, b = oracle.layer_budgets(s, 1.0, 10.0, 1600, np.full(16, 10 ** 6))
    assert b.max() - b.min() <= 1
    st, b = oracle.layer_budgets(s, 5.0, 100.0, 160000, np.full(16, 10 ** 6))
    order = np.argsort(s)
    assert np.all(np.diff(b[order]) >= -1)


def test_compress_head_n_matches_the_ratio_form():
    rng = np.random.default_rng(22)
    K = _bf16(rng.normal(size=(500, 128)))
    for r in (0.0, 0.3, 0.5, 1.0):
        a = oracle.compress_head(K, K, r, "l2", 0)
        b = oracle.compress_head_n(K, K, oracle.num_keep(500, r), "l2", 0)
        np.testing.assert_array_equal(a["idx"], b["idx"])


# ---- cluster summaries ("RefineKV" project page, method overview step 1) ----

def test_window_means_hand_case():
    # rows (0,0),(2,0) | (1,1),(3,3) | (5,-1), clusters of 2: means (1,0),
    # (2,2), (5,-1); radii: |(2,0)-(1,0)| = 1, |(3,3)-(2,2)| = sqrt 2, 0
    X = _bf16([[0, 0], [2, 0], [1, 1], [3, 3], [5, -1]])
    M, R = oracle.window_means(X, 2)
    assert M.tolist() == [[1.0, 0.0], [2.0, 2.0], [5.0, -1.0]]
    assert R[0] == 1.0 and R[1] == math.sqrt(2.0) and R[2] == 0.0


@pytest.mark.parametrize("window", [1, 3, 10, 64, 0])
def test_window_means_equal_library_mean_and_max_distance(window):
    g = torch.Generator().manual_seed(11 + window)
    T, d = 157, 16
    X = (torch.randn(T, d, generator=g) * 3).to(torch.bfloat16)
    M, R = oracle.window_means(X, window)
    x = _f64(X)
    wl = T if window <= 0 or window >= T else window
    starts = list(range(0, T, wl))
    assert M.shape == (len(starts), d) and R.shape == (len(starts),)
    for j, a in enumerate(starts):
        rows = x[a:a + wl]
        mean = np.mean(rows, axis=0)
        np.testing.assert_allclose(M[j], mean, rtol=1e-12, atol=1e-12)
        assert R[j] == pytest.approx(cdist(rows, mean[None, :]).max(), rel=1e-12, abs=1e-12)


def test_window_means_translation_exact():
    # small integers: every sum is exact, so adding v to every row shifts each
    # mean by exactly v and leaves every radius unchanged
    g = torch.Generator().manual_seed(5)
    X = torch.randint(-20, 20, (40, 8), generator=g).to(torch.float32)
    v = torch.randint(-50, 50, (8,), generator=g).to(torch.float32)
    M0, R0 = oracle.window_means(X.to(torch.bfloat16), 8)
    M1, R1 = oracle.window_means((X + v).to(torch.bfloat16), 8)
    np.testing.assert_array_equal(M1, M0 + v.numpy().astype(np.float64))
    np.testing.assert_array_equal(R1, R0)


def test_radius_bounds_every_members_logit_deviation():
    # the reading behind the radius: |q.x_t - q.mean| <= |q| * radius for
    # every member t and any query q, with equality for q along the farthest
    # member's offset
    g = torch.Generator().manual_seed(8)
    X = torch.randn(50, 32, generator=g).to(torch.bfloat16)
    M, R = oracle.window_means(X, 10)
    x = _f64(X)
    q = np.random.default_rng(0).normal(size=(20, 32))
    for j in range(5):
        dev = np.abs((x[10 * j:10 * j + 10] - M[j]) @ q.T)
        assert np.all(dev <= np.linalg.norm(q, axis=1) * R[j] * (1 + 1e-12))
        off = x[10 * j:10 * j + 10] - M[j]
        far = off[np.argmax(np.linalg.norm(off, axis=1))]
        assert abs(far @ far) / np.linalg.norm(far) == pytest.approx(R[j], rel=1e-12)


def test_window_means_without_radius():
    X = _bf16([[1, 2], [3, 4], [5, 6]])
    M, R = oracle.window_means(X, 2, radius=False)
    assert R is None and M.tolist() == [[2.0, 3.0], [5.0, 6.0]]


# ---- per-window quota (a reading of WindowedManifoldKV's selection) ----

def test_select_quota_hand_cases():
    # two windows of 4, keep 2 each: (5,1,3,3) keeps 0 and the lower of the
    # tied 3s (2); (2,9,0,4) keeps 5 and 7
    assert oracle.select_quota(np.array([5, 1, 3, 3, 2, 9, 0, 4.0]), 4, 0.5).tolist() == [0, 2, 5, 7]
    # windows (1,2), (3,4), (5): floor(2*0.5+0.5) = 1 and floor(1*0.5+0.5) = 1
    # each, so the higher of each pair and the lone last token
    assert oracle.select_quota(np.array([1, 2, 3, 4, 5.0]), 2, 0.5).tolist() == [1, 3, 4]
    assert oracle.num_keep_quota(5, 0.5, 2) == 3
    # the same scores under one global top-3 keep the three largest instead
    assert oracle.select(np.array([1, 2, 3, 4, 5.0]), 3).tolist() == [2, 3, 4]


def test_select_quota_brute_force():
    rng = np.random.default_rng(3)
    for trial in range(200):
        T = int(rng.integers(0, 40))
        W = int(rng.integers(1, 12))
        r = float(rng.choice([0.0, 0.25, 0.5, 0.7, 1.0]))
        s = rng.integers(0, 5, size=T).astype(np.float64)  # many ties
        want = []
        for a in range(0, T, W):
            seg = s[a:a + W]
            q = math.floor(len(seg) * (1 - r) + 0.5)
            order = sorted(range(len(seg)), key=lambda t: (-seg[t], t))
            want += sorted(a + t for t in order[:q])
        assert oracle.select_quota(s, W, r).tolist() == want, (T, W, r)


@pytest.mark.parametrize("T", [1, 7, 100, 4096, 5000])
@pytest.mark.parametrize("W", [1, 3, 256, 4096])
@pytest.mark.parametrize("r", [0.2, 0.5, 0.75])
def test_num_keep_quota_closed_form(T, W, r):
    q = lambda n: min(max(math.floor(n * (1 - r) + 0.5), 0), n)
    nw = -(-T // W)
    assert oracle.num_keep_quota(T, r, W) == (nw - 1) * q(W) + q(T - (nw - 1) * W)


def test_select_quota_special_cases():
    rng = np.random.default_rng(4)
    s = rng.normal(size=300)
    # a window covering the head is the global selection
    for W in (300, 301, 0):
        np.testing.assert_array_equal(oracle.select_quota(s, W, 0.3), oracle.select(s, oracle.num_keep(300, 0.3)))
    # one-token windows keep every token for r <= 1/2 and none above
    assert oracle.select_quota(s, 1, 0.5).tolist() == list(range(300))
    assert oracle.select_quota(s, 1, 0.51).size == 0


def test_compress_head_quota_rows_and_counts():
    w = synthkv.WORKLOADS["single-layer-h8-t4096"]
    K, V, _ = synthkv.make_kv(w, seed=2, device="cpu", heads=[1])
    K, V = K[0, :3001], V[0, :3001]
    out = oracle.compress_head_quota(K, V, 0.4, "l2", 512)
    idx = out["idx"]
    assert idx.shape[0] == oracle.num_keep_quota(3001, 0.4, 512)
    assert np.all(np.diff(idx) > 0)
    for a in range(0, 3001, 512):
        n = min(512, 3001 - a)
        assert int(((idx >= a) & (idx < a + n)).sum()) == oracle.num_keep(n, 0.4)
    kb = K.contiguous().view(torch.int16).numpy().view(np.uint16)
    vb = V.contiguous().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(out["K_out"], kb[idx])
    np.testing.assert_array_equal(out["V_out"], vb[idx])
    # the scores are the windowed ones; only the selection differs
    np.testing.assert_array_equal(out["S"], oracle.scores(K, oracle.centroids(K, 512), 512, "l2"))


# ---- OjaKV reconstruction-error score (OjaKV deep notes, method details) ----

def _orthonormal(d, r, seed):
    a = np.random.default_rng(seed).normal(size=(d, max(r, 1)))
    q, _ = np.linalg.qr(a)
    return q[:, :r]


def _oja_inputs(T=60, M=12, d=32, seed=0):
    g = torch.Generator().manual_seed(seed)
    K = (torch.randn(T, d, generator=g) * 2).to(torch.bfloat16)
    Q = torch.randn(M, d, generator=g).to(torch.bfloat16)
    return K, Q


def test_oja_hand_case():
    # U spans the first axis: k = (3,4) leaves r = (0,4); queries (1,2) and
    # (0,-1) give |8| and |-4|, mean 6, over sqrt 2; k = (1,0) lies in the
    # span (error 0); k = (0,2) gives |4|, |-2|, mean 3, over sqrt 2
    E = oracle.oja_scores(_bf16([[3, 4], [1, 0], [0, 2]]), _bf16([[1, 2], [0, -1]]), np.array([[1.0], [0.0]]))
    assert E[0] == pytest.approx(6 / math.sqrt(2), rel=1e-15)
    assert E[1] == 0.0
    assert E[2] == pytest.approx(3 / math.sqrt(2), rel=1e-15)


def test_oja_without_a_basis_is_the_mean_absolute_attention_logit():
    # r = 0: nothing is reconstructed, e_t = mean_q |q.k_t| / sqrt(d)
    K, Q = _oja_inputs()
    E = oracle.oja_scores(K, Q, np.zeros((32, 0)))
    want = np.abs(_f64(Q) @ _f64(K).T).mean(axis=0) / math.sqrt(32)
    np.testing.assert_allclose(E, want, rtol=1e-12)


def test_oja_full_rank_basis_leaves_no_error():
    K, Q = _oja_inputs()
    E = oracle.oja_scores(K, Q, _orthonormal(32, 32, 1))
    scale = np.abs(_f64(Q)).sum(axis=1).mean() * np.abs(_f64(K)).max() / math.sqrt(32)
    assert np.all(E <= 1e-12 * scale)


def test_oja_keys_inside_and_outside_the_span():
    # U = the first 8 standard axes: keys zero beyond dim 8 are reconstructed
    # exactly (error exactly 0); keys zero in dims < 8 are untouched
    K, Q = _oja_inputs()
    U = np.eye(32)[:, :8]
    k = _f64(K)
    inside = torch.from_numpy(np.where(np.arange(32) < 8, k, 0.0)).to(torch.bfloat16)
    outside = torch.from_numpy(np.where(np.arange(32) >= 8, k, 0.0)).to(torch.bfloat16)
    assert np.all(oracle.oja_scores(inside, Q, U) == 0.0)
    want = np.abs(_f64(Q) @ _f64(outside).T).mean(axis=0) / math.sqrt(32)
    np.testing.assert_allclose(oracle.oja_scores(outside, Q, U), want, rtol=1e-12)


def test_oja_depends_on_the_span_only():
    # U and U R (R orthogonal r x r) span the same space: same errors; a
    # transposed or half-applied projector would break this
    K, Q = _oja_inputs(seed=2)
    U = _orthonormal(32, 10, 3)
    R = _orthonormal(10, 10, 4)
    np.testing.assert_allclose(oracle.oja_scores(K, Q, U @ R), oracle.oja_scores(K, Q, U), rtol=1e-10, atol=1e-13)


def test_oja_symmetries():
    K, Q = _oja_inputs(seed=5)
    U = _orthonormal(32, 6, 6)
    E = oracle.oja_scores(K, Q, U)
    # the sign of a query does not matter; doubling every key doubles the
    # errors exactly (powers of two scale every fp64 operation exactly)
    np.testing.assert_array_equal(oracle.oja_scores(K, (-Q.float()).to(torch.bfloat16), U), E)
    np.testing.assert_array_equal(oracle.oja_scores((K.float() * 2).to(torch.bfloat16), Q, U), 2 * E)
    # the order of the window's queries does not matter (a mean)
    perm = torch.randperm(Q.shape[0], generator=torch.Generator().manual_seed(0))
    np.testing.assert_allclose(oracle.oja_scores(K, Q[perm], U), E, rtol=1e-13)


def test_oja_equals_the_projected_query_form():
    # q.(k - U U^T k) = (q - U U^T q).k because U U^T is symmetric (for any U,
    # orthonormal or not): the form the GPU computes
    K, Q = _oja_inputs(seed=7)
    U = np.random.default_rng(8).normal(size=(32, 5)) * 0.3
    P = np.eye(32) - U @ U.T
    want = np.abs((_f64(Q) @ P) @ _f64(K).T).mean(axis=0) / math.sqrt(32)
    np.testing.assert_allclose(oracle.oja_scores(K, Q, U), want, rtol=1e-10, atol=1e-12)


def test_oja_selection_keeps_the_largest_errors():
    K, Q = _oja_inputs(T=200, seed=9)
    V = (K.float() + 1).to(torch.bfloat16)
    U = _orthonormal(32, 8, 10)
    out = oracle.compress_head_oja(K, V, Q, U, 50)
    E = oracle.oja_scores(K, Q, U)
    np.testing.assert_array_equal(out["S"], E)
    order = sorted(range(200), key=lambda t: (-E[t], t))
    assert out["idx"].tolist() == sorted(order[:50])
    kb = K.contiguous().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(out["K_out"], kb[out["idx"]])


# ---- in-place compaction (the memory-saving form of the gather) ----

def test_compact_in_place_hand_case():
    X = np.arange(12, dtype=np.uint16).reshape(6, 2)  # rows (0,1) (2,3) ... (10,11)
    out = oracle.compact_in_place(X, [1, 2, 4])
    assert out.tolist() == [[2, 3], [4, 5], [8, 9], [6, 7], [8, 9], [10, 11]]
    # the input is not modified
    assert X[0].tolist() == [0, 1]


def test_compact_in_place_equals_gather_then_tail():
    rng = np.random.default_rng(12)
    for _ in range(100):
        T = int(rng.integers(0, 60))
        n = int(rng.integers(0, T + 1))
        idx = np.sort(rng.choice(T, size=n, replace=False)).astype(np.int32)
        X = rng.integers(0, 65535, size=(T, 8)).astype(np.uint16)
        out = oracle.compact_in_place(X, idx)
        np.testing.assert_array_equal(out[:n], oracle.gather(X, idx))
        np.testing.assert_array_equal(out[n:], X[n:])


def test_compact_in_place_rejects_unordered_indices():
    X = np.zeros((4, 2), dtype=np.uint16)
    for bad in ([2, 1], [0, 0], [4], [-1]):
        with pytest.raises(ValueError):
            oracle.compact_in_place(X, bad)


# --- fp8 (E4M3) caches ---------------------------------------------------------
# Decoding follows the OCP 8-bit floating point specification (OFP8), E4M3:
# 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, subnormals m * 2^-9 at
# exponent field 0, no infinities, S.1111.111 = NaN.

E4M3_TABLE = [  # code, value, why
    (0x00, 0.0, "zero"),
    (0x01, 2.0 ** -9, "smallest subnormal: m = 1 at exponent field 0"),
    (0x07, 7 * 2.0 ** -9, "largest subnormal"),
    (0x08, 2.0 ** -6, "smallest normal: exponent field 1, 2^(1-7)"),
    (0x38, 1.0, "exponent field 7 = bias"),
    (0x3F, 1.875, "1 + 7/8"),
    (0x40, 2.0, "exponent field 8"),
    (0x77, 240.0, "1.875 * 2^7"),
    (0x7E, 448.0, "largest finite: 1.75 * 2^8 (1.875 * 2^8 is the NaN code)"),
    (0x80, -0.0, "negative zero"),
    (0xB8, -1.0, "sign bit"),
    (0xFE, -448.0, "most negative finite"),
]


def test_e4m3_decode_table():
    for code, value, why in E4M3_TABLE:
        got = oracle.e4m3_to_double(code)
        assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value), (hex(code), why)
    assert math.isnan(oracle.e4m3_to_double(0x7F)) and math.isnan(oracle.e4m3_to_double(0xFF))


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    finite = np.isfinite(ref)
    assert finite.sum() == 254
    assert np.array_equal(got[finite], ref[finite])
    assert np.isnan(got[~finite]).all()


def test_e4m3_widening_to_bf16_is_exact():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    bits = oracle.e4m3_to_bf16_bits(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.bfloat16)
    assert np.array_equal(bits.view(np.int16), ref.view(torch.int16).numpy())
    with pytest.raises(ValueError):
        oracle.e4m3_to_bf16_bits(np.array([0x7F], dtype=np.uint8))


def _fp8(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn)


def test_fp8_hand_case():
    # keys (0,0), (2,0), (0,2), (6,6) are exact in E4M3: centroid (2,2),
    # distances sqrt(8), 2, 2, sqrt(32); r = 0.25 keeps {0, 1, 3} (the tie
    # between tokens 1 and 2 goes to the lower index)
    K = _fp8([[0, 0], [2, 0], [0, 2], [6, 6]])
    V = _fp8([[1, -1], [2, -2], [3, -3], [4, -4]])
    res = oracle.compress_head(K, V, 0.25, "l2", 0)
    assert np.array_equal(res["C"], [[2.0, 2.0]])
    assert np.array_equal(res["S"], [math.sqrt(8), 2.0, 2.0, math.sqrt(32)])
    assert res["idx"].tolist() == [0, 1, 3]
    codes = V.view(torch.uint8).numpy()
    assert res["V_out"].dtype == np.uint8 and np.array_equal(res["V_out"], codes[[0, 1, 3]])


@pytest.mark.parametrize("mode,window", [("l2", 0), ("cosine", 0), ("l2", 37), ("cosine", 100)])
def test_fp8_head_equals_its_bf16_widening(mode, window):
    # the method runs on the decoded values: an fp8 head and its exact bf16
    # widening give the same centroids, scores and kept set, and the kept
    # rows are the fp8 rows at those indices
    g = torch.Generator().manual_seed(5)
    K = (torch.randn(301, 16, generator=g) * 3).clamp(-448, 448).to(torch.float8_e4m3fn)
    V = (torch.randn(301, 16, generator=g) * 3).clamp(-448, 448).to(torch.float8_e4m3fn)
    a = oracle.compress_head(K, V, 0.4, mode, window)
    b = oracle.compress_head(K.to(torch.bfloat16), V.to(torch.bfloat16), 0.4, mode, window)
    assert np.array_equal(a["C"], b["C"]) and np.array_equal(a["S"], b["S"]) and np.array_equal(a["idx"], b["idx"])
    kc = K.view(torch.uint8).numpy()
    assert np.array_equal(a["K_out"], kc[a["idx"]])
    # batched form and the in-place form agree with the per-head one
    idx, kept, ko, vo = oracle.compress_heads(K[None], V[None], [301], 0.4, mode, window)
    assert int(kept[0]) == len(a["idx"]) and np.array_equal(idx[0, :kept[0]], a["idx"])
    assert np.array_equal(ko[0, :kept[0]], a["K_out"]) and np.array_equal(vo[0, :kept[0]], a["V_out"])
    x = oracle.compact_in_place(V, a["idx"])
    n = len(a["idx"])
    assert np.array_equal(x[:n], a["V_out"]) and np.array_equal(x[n:], V.view(torch.uint8).numpy()[n:])
