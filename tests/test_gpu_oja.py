"""GPU parity of the OjaKV-style reconstruction-error scorer (the tcgen05
contraction) and of its full-rank selection against the fp64 oracle.

Tolerance of a score, derived from the arithmetic (u = 2^-24; per head, P =
I - U U^T, p_m = P q_m, e_t = (1/(M sqrt d)) sum_m |p_m . k_t|):
* p_m in fp32: |dp_mi| <= u |p_mi| + (r + d + 1) u sum_j |U_ij| sum_l |U_lj| |q_ml|
  (the two fp32 sums of length d and r, then the subtraction);
* the bf16 split hi + lo of p_m: |p - hi - lo| <= 2^-18 |p|;
* the tensor-core contraction: bf16 x bf16 products are exact in fp32; the
  accumulation over 2 x 128 terms is allowed 2 d u sum_i |p_mi k_ti|;
* the epilogue: M fp32 additions of |x|, the scale and its product: (M + 3) u e_t.
So |e_gpu - e| <= (1/(M sqrt d)) sum_i w_i |k_ti| + (M + 3) u e_t with
w_i = sum_m [(r + d + 1) u B_mi + (u + 2^-18 + 2 d u) |p_mi|], B = (|Q| |U|) |U|^T.
Kept sets: a token may differ from the oracle's choice only when its oracle
score is within twice the head's largest tolerance of the oracle's cut; the
GPU's choice must be exactly the top-n_keep of its own fp32 scores; rows are
bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import geometric_kv_cache_gb300 as mkv
import oracle
import synthkv
from parity_util import bits, gpu_topk_consistent, report

pytestmark = pytest.mark.gpu

DEV = "cuda"
U32 = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mkv.load()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def score_tolerance(K_head, Q_head, U_head, E):
    """Per-token bound on |e_gpu - e_oracle| for one head (float64 [T])."""
    k = np.abs(K_head.to(torch.float64).cpu().numpy())
    q = Q_head.to(torch.float64).cpu().numpy()
    U = U_head.to(torch.float64).cpu().numpy()
    M, d = q.shape
    r = U.shape[1]
    P = q - (q @ U) @ U.T
    B = (np.abs(q) @ np.abs(U)) @ np.abs(U).T
    W = (r + d + 1) * U32 * B + (U32 + 2.0 ** -18 + 2 * d * U32) * np.abs(P)
    return (k @ W.sum(axis=0)) / (M * math.sqrt(d)) + (M + 3) * U32 * np.abs(E) + 1e-30


def _case(rows=3, heads=2, t_max=3001, n_query=128, rank=64, seed=0, t_min=1):
    w = synthkv.WORKLOADS["ragged-b8-llama-kv-t8k-32k"].scaled(
        "oja-small", layers=1, batch=rows, heads=heads, t_max=t_max, t_min=t_min)
    K, V, lens = synthkv.make_kv(w, seed=seed, device=DEV)
    Q, U = synthkv.make_oja_inputs(w, seed, n_query, rank, device=DEV)
    return K, V, lens, Q, U


def _check(name, K, V, lens, Q, U, ratio, sample=None):
    B, H, T, D = K.shape
    n = B * H
    M = Q.shape[2]
    ws = mkv.oja_workspace_for(K, M, lens)
    S = torch.full((B, H, T), float("nan"), device=DEV)
    mkv.mkv_oja_score(K, Q, U, S, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    ks = mkv.mkv_num_keep(T, ratio)
    Ko = torch.zeros((B, H, max(ks, 1), D), dtype=torch.bfloat16, device=DEV)
    Vo = torch.zeros_like(Ko)
    idx = torch.full((B, H, max(ks, 1)), -7, dtype=torch.int32, device=DEV)
    kept = torch.full((B, H), -7, dtype=torch.int32, device=DEV)
    mkv.mkv_compress_oja(K, V, Q, U, ratio, ks, Ko, Vo, idx, kept, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    lens_c = lens.cpu().numpy()
    Sc = S.reshape(n, T).cpu().numpy()
    ic, kc = idx.reshape(n, -1).cpu().numpy(), kept.reshape(n).cpu().numpy()
    Kob, Vob = bits(Ko).reshape(n, -1, D), bits(Vo).reshape(n, -1, D)
    Kf, Vf, Qf, Uf = K.reshape(n, T, D), V.reshape(n, T, D), Q.reshape(n, M, D), U.reshape(n, D, -1)
    heads = range(n) if sample is None else sample
    worst, near = 0.0, 0
    for h in heads:
        Th = int(lens_c[h // H])
        # scores past the head's length are not written
        assert np.isnan(Sc[h, Th:]).all()
        nk = mkv.mkv_num_keep(Th, ratio)
        assert int(kc[h]) == nk
        if Th == 0:
            continue
        Kc, Vc, Qc, Uc = Kf[h, :Th].cpu(), Vf[h, :Th].cpu(), Qf[h].cpu(), Uf[h].cpu()
        ora = oracle.compress_head_oja(Kc, Vc, Qc, Uc.numpy(), nk)
        E = ora["S"]
        tol = score_tolerance(Kc, Qc, Uc, E)
        err = np.abs(Sc[h, :Th].astype(np.float64) - E)
        worst = max(worst, float((err / tol).max()))
        assert np.all(err <= tol), f"{name}: head {h}: {int((err > tol).sum())} scores outside the bound " \
                                   f"(max err/tol {float((err / tol).max()):.3g})"
        g = ic[h, :nk].astype(np.int64)
        assert np.all(np.diff(g) > 0) and (g.size == 0 or (g[0] >= 0 and g[-1] < Th))
        assert gpu_topk_consistent(Sc[h, :Th], g, nk), "GPU selection is not the top-n_keep of its own scores"
        diff = np.setxor1d(g, ora["idx"])
        if diff.size:
            cut = np.sort(E)[::-1][nk - 1]
            ok = np.abs(E[diff] - cut) <= 2 * tol.max()
            assert ok.all(), f"{name}: head {h}: kept-set differences away from the cut"
            near += int(diff.size)
        kb, vb = bits(Kc), bits(Vc)
        assert np.array_equal(Kob[h, :nk], kb[g]) and np.array_equal(Vob[h, :nk], vb[g])
    report(name, n_query=M, rank=U.shape[-1], ratio=ratio, score_max_err_over_tol=worst,
           near_cut_exceptions=near, heads_checked=len(list(heads)))
    return S, idx, kept


@pytest.mark.parametrize("n_query,rank", [(128, 64), (16, 0), (48, 16), (256, 96), (128, 1), (64, 127)])
def test_oja_scores_and_selection_match_the_oracle(n_query, rank):
    K, V, lens, Q, U = _case(n_query=n_query, rank=rank, seed=n_query + rank)
    _check(f"oja-M{n_query}-r{rank}", K, V, lens, Q, U, 0.5)


@pytest.mark.parametrize("T", [1, 127, 128, 129, 1000, 4097])
def test_oja_ragged_tails(T):
    K, V, lens, Q, U = _case(rows=1, heads=3, t_max=T, n_query=32, rank=32, seed=T, t_min=T)
    for ratio in (0.0, 0.3, 1.0):
        _check(f"oja-tail-T{T}", K, V, lens, Q, U, ratio)


def test_oja_non_orthonormal_basis_and_large_queries():
    # the formula is used as given, orthonormal or not
    K, V, lens, Q, U = _case(n_query=64, rank=24, seed=9)
    U = (U * 1.7 + 0.05).contiguous()
    Q = (Q.float() * 8).to(torch.bfloat16)
    _check("oja-nonorthonormal", K, V, lens, Q, U, 0.25)


def test_oja_zero_basis_gives_the_mean_absolute_logit():
    K, V, lens, Q, U = _case(rows=1, heads=2, t_max=2000, n_query=32, rank=8, seed=3, t_min=2000)
    S0 = torch.zeros(K.shape[:3], device=DEV)
    ws = mkv.oja_workspace_for(K, 32, lens)
    mkv.mkv_oja_score(K, Q, torch.zeros_like(U), S0, ws, lens)
    S1 = torch.zeros_like(S0)
    mkv.mkv_oja_score(K, Q, U[..., :0].contiguous(), S1, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    assert torch.equal(S0, S1)
    # U = 0 (or rank 0): e_t = mean_m |q_m . k_t| / sqrt(d), by torch in fp64
    want = ((Q.double() @ K.double().transpose(-1, -2)).abs().mean(dim=2) / math.sqrt(128)).cpu().numpy()
    got = S0.double().cpu().numpy()
    for h in range(2):
        tol = score_tolerance(K[0, h], Q[0, h], U[0, h, :, :0], want[0, h])
        assert np.all(np.abs(got[0, h] - want[0, h]) <= tol)


def test_oja_full_rank_basis_leaves_only_rounding():
    # rank = d with an orthonormal basis: every residual is 0, so every
    # score must lie within its rounding bound of 0 (a selection among such
    # scores ranks rounding noise and is not compared)
    K, V, lens, Q, U = _case(rows=2, heads=2, t_max=1500, n_query=64, rank=128, seed=4)
    ws = mkv.oja_workspace_for(K, 64, lens)
    S = torch.zeros(K.shape[:3], device=DEV)
    mkv.mkv_oja_score(K, Q, U, S, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    lens_c = lens.cpu().numpy()
    for b in range(2):
        for h in range(2):
            Th = int(lens_c[b])
            E = oracle.oja_scores(K[b, h, :Th].cpu(), Q[b, h].cpu(), U[b, h].cpu().numpy())
            tol = score_tolerance(K[b, h, :Th], Q[b, h], U[b, h], E)
            assert np.all(np.abs(S[b, h, :Th].double().cpu().numpy() - E) <= tol)
            assert np.all(np.abs(S[b, h, :Th].double().cpu().numpy()) <= 2 * tol)


def test_oja_is_deterministic():
    K, V, lens, Q, U = _case(seed=11)
    ws = mkv.oja_workspace_for(K, 128, lens)
    a = torch.zeros(K.shape[:3], device=DEV)
    b = torch.zeros_like(a)
    mkv.mkv_oja_score(K, Q, U, a, ws, lens)
    mkv.mkv_oja_score(K, Q, U, b, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    live = torch.arange(K.shape[2], device=DEV)[None, None] < lens[:, None, None]
    assert torch.equal(a[live.expand_as(a)], b[live.expand_as(b)])


def test_oja_full_size_llama():
    w = synthkv.WORKLOADS["llama3.1-8b-kv-t16k"]
    torch.cuda.empty_cache()
    K, V, lens = synthkv.make_kv(w, seed=0, device=DEV)
    Q, U = synthkv.make_oja_inputs(w, 0, 128, 64, device=DEV)
    rng = np.random.default_rng(3)
    n = w.n_heads
    sample = sorted(set([0, n - 1] + rng.integers(0, n, size=3).tolist()))
    S, idx, kept = _check("oja-full-llama3.1-8b-kv-t16k", K, V, lens, Q, U, 0.5, sample=sample)
    # every head: kept count, ascending indices in range
    assert torch.all(kept == w.t_max // 2)
    assert torch.all(idx[..., 1:] > idx[..., :-1]) and torch.all(idx >= 0) and torch.all(idx < w.t_max)
    assert torch.all(torch.isfinite(S)) and torch.all(S >= 0)
    del K, V, Q, U, S, idx, kept
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n_query", [16, 48, 64, 128])
def test_pair_kernel_gives_the_one_cta_kernels_bits(n_query):
    """The contraction on pairs of CTAs (tcgen05 cta_group::2, 256 tokens per
    MMA, the hi and lo operand rows split over the two SMs) writes exactly the
    scores of the one-CTA kernel: ragged heads, a head shorter than one pair
    tile, rank 0 and a non-orthonormal-sized rank."""
    for rows, heads, t_max, t_min, rank, seed in ((1, 1, 200, None, 64, 61), (3, 2, 3001, 1, 64, 62),
                                                  (2, 3, 5000, 600, 0, 63)):
        K, V, lens, Q, U = _case(rows=rows, heads=heads, t_max=t_max, n_query=n_query, rank=rank, seed=seed,
                                 t_min=t_min)
        B, H, T, D = K.shape
        ws = mkv.oja_workspace_for(K, n_query, lens)
        out = []
        for pair in (False, True):
            prev = mkv.mkv_set_oja_pair(pair)
            try:
                S = torch.full((B, H, T), float("nan"), device=DEV)
                mkv.mkv_oja_score(K, Q, U, S, ws, lens)
                assert mkv.mkv_device_status(ws) == 0
            finally:
                mkv.mkv_set_oja_pair(prev)
            out.append(S)
        assert torch.equal(out[0].nan_to_num(-1.0), out[1].nan_to_num(-1.0))
        lens_c = lens.cpu().numpy()
        for r in range(B):  # every score below T_b written, none past it
            assert not torch.isnan(out[1][r, :, :int(lens_c[r])]).any()
            assert torch.isnan(out[1][r, :, int(lens_c[r]):]).all()


def test_pair_setting_keeps_large_windows_on_one_cta():
    """n_query above 128 (hi and lo in separate MMAs) always runs the
    one-CTA kernel; the pair setting changes nothing there."""
    K, V, lens, Q, U = _case(rows=2, heads=2, t_max=1500, n_query=192, rank=32, seed=64)
    B, H, T, D = K.shape
    ws = mkv.oja_workspace_for(K, 192, lens)
    out = []
    for pair in (False, True):
        prev = mkv.mkv_set_oja_pair(pair)
        try:
            S = torch.zeros((B, H, T), device=DEV)
            mkv.mkv_oja_score(K, Q, U, S, ws, lens)
            assert mkv.mkv_device_status(ws) == 0
        finally:
            mkv.mkv_set_oja_pair(prev)
        out.append(S)
    assert torch.equal(out[0], out[1])
