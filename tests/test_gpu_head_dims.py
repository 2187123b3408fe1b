"""GPU parity at head dims 64 and 256 (the streaming kernels are templated on
the head dim; 128 is covered everywhere else): the fused and step-wise paths
against the fp64 oracle on every head, the head-group kernel against the
three-kernel path bit for bit, cluster summaries, in-place compaction and the
per-window quota. Tolerances as in parity_util and test_gpu_summaries_quota.
"""
import numpy as np
import pytest
import torch

import geometric_kv_cache_gb300 as mkv
import oracle
import synthkv
from parity_util import StepBuffers, bits, check_in_place_vs_oracle, compare_head, oracle_heads, report

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


def _cache(d, seed, rows=3, heads=2, t_max=5001, t_min=1):
    w = synthkv.WORKLOADS["ragged-b8-llama-kv-t8k-32k"].scaled(
        f"d{d}", layers=1, batch=rows, heads=heads, t_max=t_max, t_min=t_min, head_dim=d)
    return synthkv.make_kv(w, seed=seed, device=DEV)


def _fused(K, V, ratio, mode, window, lens):
    B, H, T, D = K.shape
    ks = mkv.mkv_num_keep(T, ratio)
    Ko = torch.zeros((B, H, max(ks, 1), D), dtype=torch.bfloat16, device=DEV)
    Vo = torch.zeros_like(Ko)
    idx = torch.full((B, H, max(ks, 1)), -7, dtype=torch.int32, device=DEV)
    kept = torch.full((B, H), -7, dtype=torch.int32, device=DEV)
    ws = mkv.workspace_for(K, window, lens)
    mkv.mkv_compress(K, V, ratio, mode, window, ks, Ko, Vo, idx, kept, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    return Ko, Vo, idx, kept


@pytest.mark.parametrize("d", [64, 256])
@pytest.mark.parametrize("mode,window,ratio", [("l2", 0, 0.5), ("cosine", 0, 0.2), ("l2", 1000, 0.3),
                                               ("cosine", 777, 0.6)])
def test_path_matches_the_oracle(d, mode, window, ratio):
    K, V, lens = _cache(d, seed=d + int(ratio * 10))
    B, H, T, D = K.shape
    n = B * H
    ora = oracle_heads(K, V, lens.cpu().numpy(), H, range(n), ratio, mode, window)
    Ko, Vo, idx, kept = _fused(K, V, ratio, mode, window, lens)
    # step-wise calls: centroids and scores to compare, then select + compact
    sb = StepBuffers(K, window, ratio, lens)
    mkv.mkv_centroid(K, window, sb.C, sb.ws, lens)
    mkv.mkv_score(K, sb.C, window, mode, sb.S, sb.ws, lens)
    mkv.mkv_select_topk(sb.S, sb.shape, ratio, sb.cut, sb.ws)
    mkv.mkv_compact(sb.S, sb.cut, K, V, sb.shape, ratio, sb.keep_stride, sb.idx, sb.kept, sb.K_out, sb.V_out, sb.ws)
    assert mkv.mkv_device_status(sb.ws) == 0
    S = sb.S.cpu().numpy().reshape(n, T)
    C = sb.C.cpu().numpy().reshape(n, sb.nw, D)
    Kob, Vob = bits(Ko).reshape(n, -1, D), bits(Vo).reshape(n, -1, D)
    idxc, keptc = idx.cpu().numpy().reshape(n, -1), kept.cpu().numpy().reshape(n)
    lens_c = lens.cpu().numpy()
    near = 0
    for h in range(n):
        Th = int(lens_c[h // H])
        res = compare_head(ora[h], Th, S_gpu=S[h], idx_gpu=idxc[h], kept_gpu=keptc[h], K_head=K.reshape(n, T, D)[h],
                           V_head=V.reshape(n, T, D)[h], Kout_gpu=Kob[h], Vout_gpu=Vob[h],
                           C_gpu=C[h, :len(ora[h]["C"])],
                           key_scale=float(K.reshape(n, T, D)[h, :Th].float().abs().mean()) if Th else 1.0, mode=mode)
        near += res.get("near_cut_exceptions", 0)
        # the step-wise path gives the fused path's selection
        k = int(keptc[h])
        assert np.array_equal(sb.idx.cpu().numpy().reshape(n, -1)[h, :k], idxc[h, :k])
    report(f"d{d}-{mode}-w{window}-r{ratio}", near_cut_exceptions=near)


@pytest.mark.parametrize("d", [64, 256])
@pytest.mark.parametrize("window", [0, 2048])
def test_head_groups_equal_three_kernels(d, window):
    K, V, lens = _cache(d, seed=40 + d, rows=4, heads=4, t_max=12000)
    B, H, T, D = K.shape
    nw = mkv.mkv_num_windows(T, window)
    out = []
    for enable in (True, False):
        prev = mkv.mkv_set_head_groups(enable)
        try:
            used = mkv.mkv_compress_single_pass(mkv.shape_of(K, lens), window, "l2")
            ws = mkv.workspace_for(K, window, lens)
            C = torch.zeros((B, H, nw, D), device=DEV)
            S = torch.full((B, H, T), float("nan"), device=DEV)
            mkv.mkv_centroid_score(K, window, "l2", C, S, ws, lens)
            assert mkv.mkv_device_status(ws) == 0
            out.append((used, S))
        finally:
            mkv.mkv_set_head_groups(prev)
    assert out[0][0] == 2 and out[1][0] == 0
    live = (torch.arange(T, device=DEV)[None, None, :] < lens[:, None, None]).expand_as(out[0][1])
    assert torch.equal(out[0][1][live], out[1][1][live])


@pytest.mark.parametrize("d", [64, 256])
def test_cluster_summaries(d):
    K, V, lens = _cache(d, seed=50 + d)
    B, H, T, D = K.shape
    for window in (10, 500):
        nw = mkv.mkv_num_windows(T, window)
        ws = mkv.workspace_for(K, window, lens)
        mean = torch.full((B, H, nw, D), float("nan"), device=DEV)
        radius = torch.full((B, H, nw), float("nan"), device=DEV) if window <= 128 else None
        mkv.mkv_window_means(V, window, mean, ws, radius=radius, seq_lens=lens)
        assert mkv.mkv_device_status(ws) == 0
        Vc = V.reshape(B * H, T, D).cpu()
        lens_c = lens.cpu().numpy()
        for h in range(B * H):
            Th = int(lens_c[h // H])
            M_o, R_o = oracle.window_means(Vc[h, :Th], window, radius=radius is not None)
            if M_o.shape[0] == 0:
                continue
            x = np.abs(Vc[h, :Th].to(torch.float64).numpy())
            wl = Th if window >= Th else window
            tol = np.stack([(min(wl, Th - j * wl) + 1) * U * x[j * wl:(j + 1) * wl].sum(0) / min(wl, Th - j * wl)
                            for j in range(M_o.shape[0])]) + 1e-30
            Mg = mean.reshape(B * H, nw, D)[h, :M_o.shape[0]].double().cpu().numpy()
            assert np.all(np.abs(Mg - M_o) <= tol)
            if radius is not None:
                Rg = radius.reshape(B * H, nw)[h, :M_o.shape[0]].double().cpu().numpy()
                rtol = 1.01 * np.linalg.norm(tol, axis=1) + 32 * U * R_o + 1e-30
                assert np.all(np.abs(Rg - R_o) <= rtol)


@pytest.mark.parametrize("d", [64, 256])
def test_in_place_and_quota(d):
    K, V, lens = _cache(d, seed=60 + d)
    B, H, T, D = K.shape
    ratio = 0.4
    Ko, Vo, idx, kept = _fused(K, V, ratio, "l2", 0, lens)
    Ki, Vi = K.clone(), V.clone()
    ws = mkv.workspace_for(K, 0, lens)
    kept_i = torch.zeros_like(kept)
    idx_i = torch.full((B, H, T), -7, dtype=torch.int32, device=DEV)
    mkv.mkv_compress_inplace(Ki, Vi, ratio, "l2", 0, ws, idx=idx_i, kept=kept_i, seq_lens=lens)
    assert mkv.mkv_device_status(ws) == 0
    assert torch.equal(kept_i, kept)
    # every head against the oracle's in-place move (rows past kept untouched)
    check_in_place_vs_oracle(K, V, Ki, Vi, kept_i, lens.cpu().numpy(), ratio, "l2", 0, idx_i=idx_i)
    ks = idx.shape[2]
    front = (torch.arange(ks, device=DEV)[None, None, :] < kept[..., None])[..., None].expand(-1, -1, -1, D)
    assert torch.equal(Ki[..., :ks, :][front], Ko[front]) and torch.equal(Vi[..., :ks, :][front], Vo[front])
    rest = torch.ones_like(Ki, dtype=torch.bool)
    rest[..., :ks, :] = ~front
    assert torch.equal(Ki[rest], K[rest])
    # per-window quota against the oracle
    window = 700
    kq = mkv.mkv_num_keep_quota(T, ratio, window)
    Kq = torch.zeros((B, H, kq, D), dtype=torch.bfloat16, device=DEV)
    Vq = torch.zeros_like(Kq)
    iq = torch.full((B, H, kq), -1, dtype=torch.int32, device=DEV)
    kpq = torch.zeros((B, H), dtype=torch.int32, device=DEV)
    wsq = mkv.workspace_for(K, window, lens)
    mkv.mkv_compress_quota(K, V, ratio, "l2", window, kq, Kq, Vq, iq, kpq, wsq, lens)
    assert mkv.mkv_device_status(wsq) == 0
    lens_c = lens.cpu().numpy()
    for h in range(B * H):
        b, hh = divmod(h, H)
        Th = int(lens_c[b])
        ora = oracle.compress_head_quota(K[b, hh, :Th].cpu(), V[b, hh, :Th].cpu(), ratio, "l2", window)
        n = len(ora["idx"])
        assert int(kpq[b, hh]) == n
        g = iq[b, hh, :n].cpu().numpy()
        # window by window, a token may differ only within 1e-5 of its
        # window's cut (the scores agree to 1e-5 relative)
        wl = Th if window >= Th else window
        q_full = oracle.num_keep(wl, ratio)
        for j, a in enumerate(range(0, Th, wl)):
            e = min(a + wl, Th)
            q = oracle.num_keep(e - a, ratio)
            off = j * q_full
            diff = np.setxor1d(g[off:off + q], ora["idx"][off:off + q])
            if diff.size:
                Sw = ora["S"][a:e]
                cut = np.sort(Sw)[::-1][q - 1]
                assert np.all(np.abs(ora["S"][diff] - cut) <= 1e-5 * abs(cut))
        assert np.array_equal(bits(Kq[b, hh, :n]), bits(K[b, hh])[g])


@pytest.mark.parametrize("d", [64, 256])
def test_larger_cache(d):
    # 64 heads of 16384 tokens: head groups at full occupancy
    w = synthkv.WORKLOADS["llama3.1-8b-kv-t16k"].scaled(f"d{d}-big", layers=8, head_dim=d)
    K, V, lens = synthkv.make_kv(w, seed=70, device=DEV)
    assert mkv.mkv_compress_single_pass(mkv.shape_of(K, lens), 0, "l2") == 2
    Ko, Vo, idx, kept = _fused(K, V, 0.5, "l2", 0, lens)
    assert torch.all(kept == w.t_max // 2)
    ii = idx.long()
    assert torch.all(ii[..., 1:] > ii[..., :-1])
    for r in range(w.rows):
        gi = ii[r][..., None].expand(-1, -1, d)
        assert torch.equal(torch.gather(K[r], 1, gi), Ko[r]) and torch.equal(torch.gather(V[r], 1, gi), Vo[r])
    n = w.n_heads
    for h in (0, n // 2, n - 1):
        b, hh = divmod(h, w.heads)
        ora = oracle.compress_head(K[b, hh].cpu(), V[b, hh].cpu(), 0.5, "l2", 0)
        res = compare_head(ora, w.t_max, idx_gpu=idx[b, hh].cpu().numpy(), kept_gpu=int(kept[b, hh]),
                           K_head=K[b, hh], V_head=V[b, hh], Kout_gpu=bits(Ko[b, hh]), Vout_gpu=bits(Vo[b, hh]))
        report(f"d{d}-big-head{h}", near_cut_exceptions=res["near_cut_exceptions"])
