"""GPU parity for fp8 (E4M3) caches at head dims 64, 128 and 256.

E4M3 codes (OCP 8-bit floating point, E4M3 encoding) decode exactly to fp32,
and every E4M3 value is a bf16 value, so:
* against the fp64 oracle, the same tolerances as for bf16 caches hold
  (parity_util: scores 1e-5 relative, indices exact but for near-cut ties,
  kept rows byte-exact);
* against the library's own bf16 path on the exactly widened cache, the
  results are bit-identical: each lane takes the same 8-element chunks in
  both types and every sum keeps its order, so the centroids and scores have
  the same bits and the kept indices are the same; the kept rows are the fp8
  rows at those indices.
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
F8 = torch.float8_e4m3fn


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mkv.load()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _cache(d, seed, rows=3, heads=2, t_max=5001, t_min=1, dtype=F8):
    w = synthkv.WORKLOADS["ragged-b8-llama-kv-t8k-32k"].scaled(
        f"f8-d{d}", layers=1, batch=rows, heads=heads, t_max=t_max, t_min=t_min, head_dim=d)
    return synthkv.make_kv(w, seed=seed, device=DEV, dtype=dtype)


def _fused(K, V, ratio, mode, window, lens):
    B, H, T, D = K.shape
    ks = mkv.mkv_num_keep(T, ratio)
    Ko = torch.zeros((B, H, max(ks, 1), D), dtype=K.dtype, device=DEV)
    Vo = torch.zeros_like(Ko)
    idx = torch.full((B, H, max(ks, 1)), -7, dtype=torch.int32, device=DEV)
    kept = torch.full((B, H), -7, dtype=torch.int32, device=DEV)
    ws = mkv.workspace_for(K, window, lens)
    mkv.mkv_compress(K, V, ratio, mode, window, ks, Ko, Vo, idx, kept, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    return Ko, Vo, idx, kept


def _centroid_score(K, window, mode, lens):
    B, H, T, D = K.shape
    nw = mkv.mkv_num_windows(T, window)
    ws = mkv.workspace_for(K, window, lens)
    C = torch.full((B, H, nw, D), float("nan"), device=DEV)
    S = torch.full((B, H, T), float("nan"), device=DEV)
    mkv.mkv_centroid_score(K, window, mode, C, S, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    return C, S


def _live(lens, T):
    return torch.arange(T, device=DEV)[None, None, :] < lens[:, None, None]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("mode,window,ratio", [("l2", 0, 0.5), ("cosine", 0, 0.2), ("l2", 1000, 0.3),
                                               ("cosine", 777, 0.6)])
def test_fp8_path_matches_the_oracle(d, mode, window, ratio):
    K, V, lens = _cache(d, seed=d + int(ratio * 10))
    B, H, T, D = K.shape
    n = B * H
    ora = oracle_heads(K, V, lens.cpu().numpy(), H, range(n), ratio, mode, window)
    Ko, Vo, idx, kept = _fused(K, V, ratio, mode, window, lens)
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
    Kf, Vf = K.reshape(n, T, D), V.reshape(n, T, D)
    near = 0
    for h in range(n):
        Th = int(lens_c[h // H])
        scale = float(Kf[h, :Th].float().abs().mean()) if Th else 1.0
        res = compare_head(ora[h], Th, S_gpu=S[h], idx_gpu=idxc[h], kept_gpu=keptc[h], K_head=Kf[h], V_head=Vf[h],
                           Kout_gpu=Kob[h], Vout_gpu=Vob[h], C_gpu=C[h, :len(ora[h]["C"])], key_scale=scale,
                           mode=mode)
        near += res.get("near_cut_exceptions", 0)
        k = int(keptc[h])
        assert np.array_equal(sb.idx.cpu().numpy().reshape(n, -1)[h, :k], idxc[h, :k])
        assert np.array_equal(bits(sb.K_out).reshape(n, -1, D)[h, :k], Kob[h, :k])
    report(f"fp8-d{d}-{mode}-w{window}-r{ratio}", near_cut_exceptions=near)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("mode,window", [("l2", 0), ("cosine", 0), ("l2", 700), ("cosine", 3000)])
def test_fp8_equals_the_bf16_path_on_the_widened_cache(d, mode, window):
    K8, V8, lens = _cache(d, seed=20 + d, rows=2, heads=3, t_max=9000)
    Kw, Vw = K8.to(torch.bfloat16), V8.to(torch.bfloat16)  # exact
    assert torch.equal(Kw.float(), K8.float())
    T = K8.shape[2]
    C8, S8 = _centroid_score(K8, window, mode, lens)
    Cw, Sw = _centroid_score(Kw, window, mode, lens)
    live = _live(lens, T).expand_as(S8)
    assert torch.equal(S8[live], Sw[live])
    nw = C8.shape[2]
    wl = torch.where((window <= 0) | (window >= lens), lens, torch.full_like(lens, max(window, 1)))
    nwin = (lens + wl - 1) // wl.clamp(min=1)  # windows per batch row (0 for an empty row)
    wlive = (torch.arange(nw, device=DEV)[None, :] < nwin[:, None])[:, None, :]
    assert torch.equal(C8[wlive.expand(C8.shape[:3])], Cw[wlive.expand(Cw.shape[:3])])
    Ko8, Vo8, i8, k8 = _fused(K8, V8, 0.45, mode, window, lens)
    Kow, Vow, iw, kw = _fused(Kw, Vw, 0.45, mode, window, lens)
    assert torch.equal(k8, kw)
    slot = torch.arange(i8.shape[2], device=DEV)[None, None, :] < k8[..., None]
    assert torch.equal(i8[slot], iw[slot])
    rows = slot[..., None].expand(Ko8.shape)
    assert torch.equal(Ko8.view(torch.uint8)[rows], K8.view(torch.uint8).gather(
        2, i8.clamp(min=0).long()[..., None].expand(Ko8.shape))[rows])
    assert torch.equal(Ko8.float()[rows], Kow.float()[rows]) and torch.equal(Vo8.float()[rows], Vow.float()[rows])


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("window", [0, 2048])
def test_fp8_head_groups_equal_three_kernels(d, window):
    K, V, lens = _cache(d, seed=40 + d, rows=4, heads=4, t_max=12000)
    out = []
    for enable in (True, False):
        prev = mkv.mkv_set_head_groups(enable)
        try:
            used = mkv.mkv_compress_single_pass(mkv.shape_of(K, lens), window, "l2")
            out.append((used, _centroid_score(K, window, "l2", lens)[1]))
        finally:
            mkv.mkv_set_head_groups(prev)
    assert out[0][0] == 2 and out[1][0] == 0
    live = _live(lens, K.shape[2]).expand_as(out[0][1])
    assert torch.equal(out[0][1][live], out[1][1][live])


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp8_summaries_in_place_and_quota(d):
    K, V, lens = _cache(d, seed=50 + d)
    B, H, T, D = K.shape
    Kw, Vw = K.to(torch.bfloat16), V.to(torch.bfloat16)
    # cluster summaries of the values: the bf16 path's bits on the widened cache
    for window in (10, 500):
        nw = mkv.mkv_num_windows(T, window)
        res = []
        for X in (V, Vw):
            ws = mkv.workspace_for(X, window, lens)
            mean = torch.full((B, H, nw, D), float("nan"), device=DEV)
            radius = torch.full((B, H, nw), float("nan"), device=DEV) if window <= 128 else None
            mkv.mkv_window_means(X, window, mean, ws, radius=radius, seq_lens=lens)
            assert mkv.mkv_device_status(ws) == 0
            res.append((mean, radius))
        assert torch.equal(torch.nan_to_num(res[0][0], 7.0), torch.nan_to_num(res[1][0], 7.0))
        if window <= 128:
            assert torch.equal(torch.nan_to_num(res[0][1], 7.0), torch.nan_to_num(res[1][1], 7.0))
        # and against the oracle, window by window, for one head: a mean of n
        # fp32-summed terms is within (n + 1) u sum|x| / n of the exact one
        Th = int(lens[0])
        Vc = V.reshape(B * H, T, D)[0, :Th].cpu()
        M_o, _ = oracle.window_means(Vc, window, radius=False)
        x = np.abs(Vc.to(torch.float64).numpy())
        wl = Th if window >= Th else window
        U = 2.0 ** -24
        tol = np.stack([(min(wl, Th - j * wl) + 1) * U * x[j * wl:(j + 1) * wl].sum(0) / min(wl, Th - j * wl)
                        for j in range(M_o.shape[0])]) + 1e-30
        Mg = res[0][0].reshape(B * H, nw, D)[0, :M_o.shape[0]].double().cpu().numpy()
        assert np.all(np.abs(Mg - M_o) <= tol)
    # in-place compaction: the same rows as the out-of-place gather
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
    u8 = lambda t: t.view(torch.uint8)
    assert torch.equal(u8(Ki)[..., :ks, :][front], u8(Ko)[front])
    assert torch.equal(u8(Vi)[..., :ks, :][front], u8(Vo)[front])
    rest = torch.ones(Ki.shape, dtype=torch.bool, device=DEV)
    rest[..., :ks, :] = ~front
    assert torch.equal(u8(Ki)[rest], u8(K)[rest])
    # per-window quota: the widened cache's kept indices
    window = 700
    kq = mkv.mkv_num_keep_quota(T, ratio, window)
    outs = []
    for KK, VV in ((K, V), (Kw, Vw)):
        Kq = torch.zeros((B, H, kq, D), dtype=KK.dtype, device=DEV)
        Vq = torch.zeros_like(Kq)
        iq = torch.full((B, H, kq), -1, dtype=torch.int32, device=DEV)
        kpq = torch.zeros((B, H), dtype=torch.int32, device=DEV)
        wsq = mkv.workspace_for(KK, window, lens)
        mkv.mkv_compress_quota(KK, VV, ratio, "l2", window, kq, Kq, Vq, iq, kpq, wsq, lens)
        assert mkv.mkv_device_status(wsq) == 0
        outs.append((iq, kpq, Kq))
    assert torch.equal(outs[0][1], outs[1][1]) and torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][2].float(), outs[1][2].float())


def test_fp8_host_path():
    w = synthkv.WORKLOADS["ragged-b8-llama-kv-t8k-32k"].scaled("f8-host", layers=1, batch=5, heads=2, t_max=4000,
                                                                 t_min=100)
    K, V, lens = synthkv.make_kv(w, seed=3, device=DEV, dtype=F8)
    ratio, mode, window = 0.4, "l2", 0
    ks = mkv.mkv_num_keep(w.t_max, ratio)
    Ko, Vo, idx, kept = _fused(K, V, ratio, mode, window, lens)
    dK, dV = torch.empty_like(K), torch.empty_like(V)
    dKo = torch.empty((5, 2, ks, 128), dtype=F8, device=DEV)
    dVo = torch.empty_like(dKo)
    didx = torch.empty((5, 2, ks), dtype=torch.int32, device=DEV)
    dkept = torch.empty((5, 2), dtype=torch.int32, device=DEV)
    ws = mkv.workspace_for(K, window, lens)
    hK, hV = K.cpu().pin_memory(), V.cpu().pin_memory()
    hKo = torch.zeros(dKo.shape, dtype=F8).pin_memory()
    hVo = torch.zeros(dKo.shape, dtype=F8).pin_memory()
    hidx = torch.zeros(didx.shape, dtype=torch.int32).pin_memory()
    hkept = torch.zeros(dkept.shape, dtype=torch.int32).pin_memory()
    mkv.mkv_compress_host(hK, hV, dK, dV, ratio, mode, window, ks, dKo, dVo, didx, dkept, hKo, hVo, hidx, hkept,
                          ws, lens)
    torch.cuda.synchronize()
    assert mkv.mkv_device_status(ws) == 0
    kk = kept.cpu()
    assert torch.equal(hkept, kk)
    live = torch.arange(ks)[None, None, :] < kk[..., None]
    assert torch.equal(hidx[live], idx.cpu()[live])
    rows = live[..., None].expand(hKo.shape)
    assert torch.equal(hKo.view(torch.uint8)[rows], Ko.cpu().view(torch.uint8)[rows])
    assert torch.equal(hVo.view(torch.uint8)[rows], Vo.cpu().view(torch.uint8)[rows])


def test_fp8_full_size_llama():
    w = synthkv.WORKLOADS["llama3.1-8b-kv-t16k"]
    torch.cuda.empty_cache()
    K, V, lens = synthkv.make_kv(w, seed=0, device=DEV, dtype=F8)
    # E4M3 caches with several rounds per head group take the three kernels
    assert mkv.mkv_compress_single_pass(mkv.shape_of(K, lens), 0, "l2") == 0
    Ko, Vo, idx, kept = _fused(K, V, 0.5, "l2", 0, lens)
    assert torch.all(kept == w.t_max // 2)
    ii = idx.long()
    assert torch.all(ii[..., 1:] > ii[..., :-1])
    n = w.n_heads
    for h in (0, n // 2, n - 1):
        b, hh = divmod(h, w.heads)
        ora = oracle.compress_head(K[b, hh].cpu(), V[b, hh].cpu(), 0.5, "l2", 0)
        res = compare_head(ora, w.t_max, idx_gpu=idx[b, hh].cpu().numpy(), kept_gpu=int(kept[b, hh]),
                           K_head=K[b, hh], V_head=V[b, hh], Kout_gpu=bits(Ko[b, hh]), Vout_gpu=bits(Vo[b, hh]))
        report(f"fp8-full-head{h}", near_cut_exceptions=res["near_cut_exceptions"])
    for r in range(0, w.rows, 7):
        gi = ii[r][..., None].expand(-1, -1, w.head_dim)
        assert torch.equal(torch.gather(K[r].view(torch.uint8), 1, gi), Ko[r].view(torch.uint8))
        assert torch.equal(torch.gather(V[r].view(torch.uint8), 1, gi), Vo[r].view(torch.uint8))
    del K, V, Ko, Vo
    torch.cuda.empty_cache()
