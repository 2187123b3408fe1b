"""GPU parity of the cluster summaries (mkv_window_means) and of the
per-window-quota selection (mkv_select_quota, mkv_compress_quota) against
the fp64 oracle.

Tolerances, derived from the fp32 arithmetic (u = 2^-24):
* window mean of n rows, per dim: the GPU sums in fp32 (in token order, or
  in a fixed tree for windows over 128 tokens) and divides once, so
  |mean_gpu - mean| <= (n + 1) u sum_t |x_t| / n;
* radius max_t |x_t - mean|_2: moving the mean by d moves every distance by
  at most |d|_2, and the fp32 differences, fused square-sums over 16 dims,
  the 8-lane sum and the sqrt add at most about 12u relative, so
  |radius_gpu - radius| <= 1.01 |mean bound|_2 + 32 u radius;
* quota selection: per window, exactly as the global selection per head
  (scores 1e-5 relative, kept sets exact but for tokens within 1e-5 of the
  window's own cut, rows bit-exact, and the GPU's choice exactly the top of
  its own fp32 scores).
"""
import numpy as np
import pytest
import torch

import geometric_kv_cache_gb300 as mkv
import oracle
import synthkv
from parity_util import bits, compare_head, report

pytestmark = pytest.mark.gpu

DEV = "cuda"
U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mkv.load()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _ragged_cache(seed=3, t_max=3001, rows=3, heads=2):
    w = synthkv.WORKLOADS["ragged-b8-llama-kv-t8k-32k"].scaled(
        "ragged-summaries", layers=1, batch=rows, heads=heads, t_max=t_max, t_min=1)
    return synthkv.make_kv(w, seed=seed, device=DEV)


def _check_means(name, X, lens, window, mean, radius):
    """Every head of X [B, H, T, D] against the oracle."""
    B, H, T, D = X.shape
    Xc = X.reshape(B * H, T, D).cpu()
    Mc = mean.reshape(B * H, -1, D).cpu().numpy().astype(np.float64)
    Rc = radius.reshape(B * H, -1).cpu().numpy().astype(np.float64) if radius is not None else None
    lens_c = lens.cpu().numpy()
    worst_m, worst_r = 0.0, 0.0
    for h in range(B * H):
        Th = int(lens_c[h // H])
        M_o, R_o = oracle.window_means(Xc[h, :Th], window, radius=radius is not None)
        nw = M_o.shape[0]
        if nw == 0:
            continue
        x = np.abs(Xc[h, :Th].to(torch.float64).numpy())
        wl = Th if window <= 0 or window >= Th else window
        tol = np.empty_like(M_o)
        for j in range(nw):
            rows = x[j * wl:(j + 1) * wl]
            n = rows.shape[0]
            tol[j] = (n + 1) * U * rows.sum(axis=0) / n + 1e-30
        err = np.abs(Mc[h, :nw] - M_o)
        worst_m = max(worst_m, float((err / tol).max()))
        assert np.all(err <= tol), f"{name}: head {h} mean error {float((err / tol).max())} x tolerance"
        if Rc is not None:
            rtol = 1.01 * np.linalg.norm(tol, axis=1) + 32 * U * R_o + 1e-30
            rerr = np.abs(Rc[h, :nw] - R_o)
            worst_r = max(worst_r, float((rerr / rtol).max()))
            assert np.all(rerr <= rtol), f"{name}: head {h} radius error {float((rerr / rtol).max())} x tolerance"
    report(name, window=window, mean_max_err_over_tol=worst_m, radius_max_err_over_tol=worst_r)


@pytest.mark.parametrize("window", [1, 3, 10, 64, 128])
def test_short_window_means_and_radii_match_the_oracle(window):
    K, V, lens = _ragged_cache()
    B, H, T, D = K.shape
    nw = mkv.mkv_num_windows(T, window)
    ws = mkv.workspace_for(K, window, lens)
    for X, tag in ((K, "K"), (V, "V")):
        mean = torch.full((B, H, nw, D), float("nan"), device=DEV)
        radius = torch.full((B, H, nw), float("nan"), device=DEV)
        mkv.mkv_window_means(X, window, mean, ws, radius=radius, seq_lens=lens)
        assert mkv.mkv_device_status(ws) == 0
        _check_means(f"window-means-{tag}-w{window}", X, lens, window, mean, radius)
        # windows a short head does not have are not written
        lens_c = lens.cpu().numpy()
        for b in range(B):
            have = -(-int(lens_c[b]) // window)
            assert torch.isnan(mean[b, :, have:]).all() and torch.isnan(radius[b, :, have:]).all()
        # without radius: the same means
        mean2 = torch.zeros_like(mean)
        mkv.mkv_window_means(X, window, mean2, ws, seq_lens=lens)
        m = ~torch.isnan(mean)
        assert torch.equal(mean2[m], mean[m])


@pytest.mark.parametrize("window", [129, 500, 4096, 0])
def test_long_window_means_are_the_centroids(window):
    K, V, lens = _ragged_cache(seed=4, t_max=9000)
    B, H, T, D = K.shape
    nw = mkv.mkv_num_windows(T, window)
    ws = mkv.workspace_for(K, window, lens)
    C = torch.zeros((B, H, nw, D), device=DEV)
    mkv.mkv_centroid(K, window, C, ws, lens)
    for X, tag in ((K, "K"), (V, "V")):
        mean = torch.zeros((B, H, nw, D), device=DEV)
        mkv.mkv_window_means(X, window, mean, ws, seq_lens=lens)
        assert mkv.mkv_device_status(ws) == 0
        if tag == "K":
            assert torch.equal(mean, C)
        _check_means(f"window-means-{tag}-w{window}", X, lens, window, mean, None)


def test_window_means_full_size_llama_clusters_of_ten():
    w = synthkv.WORKLOADS["llama3.1-8b-kv-t16k"]
    torch.cuda.empty_cache()
    K, V, lens = synthkv.make_kv(w, seed=0, device=DEV)
    n, T, window = w.n_heads, w.t_max, 10
    nw = mkv.mkv_num_windows(T, window)
    ws = mkv.workspace_for(K, window, lens)
    rng = np.random.default_rng(1)
    heads = sorted(set([0, n - 1] + rng.integers(0, n, size=4).tolist()))
    for X, tag in ((K, "K"), (V, "V")):
        mean = torch.empty((w.rows, w.heads, nw, 128), device=DEV)
        radius = torch.empty((w.rows, w.heads, nw), device=DEV)
        mkv.mkv_window_means(X, window, mean, ws, radius=radius, seq_lens=lens)
        assert mkv.mkv_device_status(ws) == 0
        # every head: the mean lies within the window's per-dim range, the
        # radius is finite and nonnegative (fp32 torch on the GPU)
        Xw = X.reshape(n, T, 128)[:, : (T // window) * window].reshape(n, T // window, window, 128).float()
        m = mean.reshape(n, nw, 128)[:, : T // window]
        assert torch.all(m >= Xw.amin(dim=2)) and torch.all(m <= Xw.amax(dim=2))
        assert torch.all(torch.isfinite(radius)) and torch.all(radius >= 0)
        del Xw, m
        # sampled heads against the oracle
        sub = torch.tensor(heads, device=DEV)
        Xs = X.reshape(n, 1, T, 128)[sub]
        _check_means(f"window-means-{tag}-w10-full", Xs, torch.full((len(heads),), T, dtype=torch.int32),
                     window, mean.reshape(n, 1, nw, 128)[sub], radius.reshape(n, 1, nw)[sub])
        del mean, radius
    del K, V
    torch.cuda.empty_cache()


# ------------------------------------------------------------ quota selection --

def _quota_step(K, V, lens, ratio, mode, window):
    """Step-wise: centroids, scores, quota selection; then the fused call."""
    B, H, T, D = K.shape
    nw = max(mkv.mkv_num_windows(T, window), 1)
    ks = mkv.mkv_num_keep_quota(T, ratio, window)
    shape = mkv.shape_of(K, lens)
    ws = mkv.workspace_for(K, window, lens)
    C = torch.zeros((B, H, nw, D), device=DEV)
    S = torch.zeros((B, H, T), device=DEV)
    idx = torch.full((B, H, max(ks, 1)), -7, dtype=torch.int32, device=DEV)
    kept = torch.full((B, H), -7, dtype=torch.int32, device=DEV)
    mkv.mkv_centroid(K, window, C, ws, lens)
    mkv.mkv_score(K, C, window, mode, S, ws, lens)
    mkv.mkv_select_quota(S, shape, ratio, window, ks, idx, kept, ws)
    assert mkv.mkv_device_status(ws) == 0
    Ko = torch.zeros((B, H, max(ks, 1), D), dtype=torch.bfloat16, device=DEV)
    Vo = torch.zeros_like(Ko)
    idx2 = torch.full_like(idx, -7)
    kept2 = torch.full_like(kept, -7)
    mkv.mkv_compress_quota(K, V, ratio, mode, window, ks, Ko, Vo, idx2, kept2, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    return C, S, idx, kept, Ko, Vo, idx2, kept2


def _check_quota(name, K, V, lens, ratio, mode, window):
    B, H, T, D = K.shape
    n = B * H
    C, S, idx, kept, Ko, Vo, idx2, kept2 = _quota_step(K, V, lens, ratio, mode, window)
    # the fused call makes the same choice from the same scores
    assert torch.equal(kept, kept2)
    live = torch.arange(idx.shape[2], device=DEV)[None, None, :] < kept[..., None]
    assert torch.equal(torch.where(live, idx, 0), torch.where(live, idx2, 0))
    Kc, Vc = K.reshape(n, T, D).cpu(), V.reshape(n, T, D).cpu()
    Sc, Cc = S.reshape(n, T).cpu().numpy(), C.reshape(n, -1, D).cpu().numpy()
    ic, kc = idx.reshape(n, -1).cpu().numpy(), kept.reshape(n).cpu().numpy()
    Kob, Vob = bits(Ko).reshape(n, -1, D), bits(Vo).reshape(n, -1, D)
    lens_c = lens.cpu().numpy()
    near = 0
    for h in range(n):
        Th = int(lens_c[h // H])
        ora = oracle.compress_head_quota(Kc[h, :Th], Vc[h, :Th], ratio, mode, window)
        assert int(kc[h]) == len(ora["idx"]) == oracle.num_keep_quota(Th, ratio, window)
        if Th == 0:
            continue
        scale = float(Kc[h, :Th].float().abs().mean())
        compare_head({"S": ora["S"], "C": ora["C"], "idx": np.zeros(0, np.int32)}, Th, S_gpu=Sc[h],
                     C_gpu=Cc[h, :len(ora["C"])], key_scale=scale, mode=mode)
        wl = Th if window <= 0 or window >= Th else window
        q_full = oracle.num_keep(wl, ratio)
        for j, a in enumerate(range(0, Th, wl)):
            b = min(a + wl, Th)
            q = oracle.num_keep(b - a, ratio)
            off = j * q_full
            sub = {"S": ora["S"][a:b], "idx": ora["idx"][off:off + q] - a,
                   "K_out": ora["K_out"][off:off + q], "V_out": ora["V_out"][off:off + q]}
            res = compare_head(sub, b - a, S_gpu=Sc[h, a:b], idx_gpu=ic[h, off:off + q] - a,
                               K_head=Kc[h, a:b], V_head=Vc[h, a:b], Kout_gpu=Kob[h, off:off + q],
                               Vout_gpu=Vob[h, off:off + q], mode=mode)
            near += res["near_cut_exceptions"]
    report(name, mode=mode, window=window, ratio=ratio, near_cut_exceptions=near)


@pytest.mark.parametrize("window", [1, 7, 100, 512, 4096, 0, 10000])
@pytest.mark.parametrize("mode", ["l2", "cosine"])
def test_quota_selection_matches_the_oracle_per_window(window, mode):
    # one-token windows make one oracle call per token: a shorter cache
    K, V, lens = _ragged_cache(seed=5, t_max=9001 if window >= 8 else 1500)
    for ratio in (0.25, 0.5, 0.8):
        _check_quota(f"quota-{mode}-w{window}-r{ratio}", K, V, lens, ratio, mode, window)


def test_quota_with_one_window_is_the_global_selection():
    K, V, lens = _ragged_cache(seed=6, t_max=5000)
    ratio = 0.4
    _, _, idx_q, kept_q, Ko_q, _, _, _ = _quota_step(K, V, lens, ratio, "l2", 0)
    ks = mkv.mkv_num_keep(K.shape[2], ratio)
    Ko, Vo, idx, kept = mkv.compress(K, V, ratio, "l2", 0, seq_lens=lens, keep_stride=ks)
    assert torch.equal(kept, kept_q)
    live = torch.arange(ks, device=DEV)[None, None, :] < kept[..., None]
    assert torch.equal(torch.where(live, idx, 0), torch.where(live, idx_q[..., :ks], 0))
    assert torch.equal(torch.where(live[..., None], Ko, 0), torch.where(live[..., None], Ko_q[:, :, :ks], 0))


def test_quota_full_size_qwen_windows():
    w = synthkv.WORKLOADS["qwen3-8b-kv-t64k-w4096"]
    torch.cuda.empty_cache()
    K, V, lens = synthkv.make_kv(w, seed=0, device=DEV)
    mode, window, ratio = w.runs[0]
    n, T = w.n_heads, w.t_max
    ks = mkv.mkv_num_keep_quota(T, ratio, window)
    Ko = torch.empty((w.rows, w.heads, ks, 128), dtype=torch.bfloat16, device=DEV)
    Vo = torch.empty_like(Ko)
    idx = torch.full((w.rows, w.heads, ks), -1, dtype=torch.int32, device=DEV)
    kept = torch.zeros((w.rows, w.heads), dtype=torch.int32, device=DEV)
    ws = mkv.workspace_for(K, window, lens)
    mkv.mkv_compress_quota(K, V, ratio, mode, window, ks, Ko, Vo, idx, kept, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    assert torch.all(kept == ks)
    # every head: each window holds exactly its share, indices ascend, rows equal K/V[idx]
    ii = idx.long()
    assert torch.all(ii[..., 1:] > ii[..., :-1])
    q = mkv.mkv_num_keep(window, ratio)
    win = ii.reshape(w.rows, w.heads, T // window, q) // window
    assert torch.equal(win, torch.arange(T // window, device=DEV)[None, None, :, None].expand_as(win))
    for r in range(w.rows):
        gi = ii[r][..., None].expand(-1, -1, 128)
        assert torch.equal(torch.gather(K[r], 1, gi), Ko[r])
        assert torch.equal(torch.gather(V[r], 1, gi), Vo[r])
    # sampled heads against the oracle, window by window
    rng = np.random.default_rng(2)
    heads = sorted(set([0, n - 1] + rng.integers(0, n, size=2).tolist()))
    Kf, Vf = K.reshape(n, T, 128), V.reshape(n, T, 128)
    near = 0
    for h in heads:
        ora = oracle.compress_head_quota(Kf[h].cpu(), Vf[h].cpu(), ratio, mode, window)
        b, hh = divmod(h, w.heads)
        g = idx[b, hh].cpu().numpy()
        Kc, Vc = Kf[h].cpu(), Vf[h].cpu()
        Kob, Vob = bits(Ko[b, hh]), bits(Vo[b, hh])
        for j in range(T // window):
            a, off = j * window, j * q
            sub = {"S": ora["S"][a:a + window], "idx": ora["idx"][off:off + q] - a,
                   "K_out": ora["K_out"][off:off + q], "V_out": ora["V_out"][off:off + q]}
            res = compare_head(sub, window, idx_gpu=g[off:off + q] - a, K_head=Kc[a:a + window],
                               V_head=Vc[a:a + window], Kout_gpu=Kob[off:off + q], Vout_gpu=Vob[off:off + q],
                               mode=mode)
            near += res["near_cut_exceptions"]
    report(f"{w.name}:quota:full", heads_sampled=len(heads), near_cut_exceptions=near, heads_property_checked=n)
    del K, V, Ko, Vo, idx, kept, ws
    torch.cuda.empty_cache()
