"""GPU parity of the copy-ring head-group kernel (mkv_set_head_group_ring):
its pass 1 streams K into shared memory through bulk asynchronous copies fed
by a producer warp, and its sums keep the register kernel's order, so its
centroids and scores must be the same bits as the register head-group kernel's
and the three kernels' on every live token -- global and windowed centroids,
both score modes, ragged lengths with empty and sub-piece heads, pieces longer
than a copy stage (long global heads) -- and a small case is checked against
the fp64 oracle."""
import numpy as np
import pytest
import torch

import geometric_kv_cache_gb300 as mkv
import synthkv
from parity_util import compare_head, oracle_heads

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mkv.load()
    prev = mkv.mkv_set_head_group_ring(False)
    prev_fused = mkv.mkv_set_fused(0)  # the path query then names the a1 + a2 kernel mkv_centroid_score runs
    yield
    mkv.mkv_set_fused(prev_fused)
    mkv.mkv_set_head_group_ring(prev)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _centroid_score(K, window, mode, lens):
    B, H, T, D = K.shape
    nw = max(mkv.mkv_num_windows(T, window), 1)
    C = torch.zeros((B, H, nw, D), dtype=torch.float32, device=DEV)
    S = torch.zeros((B, H, T), dtype=torch.float32, device=DEV)
    ws = mkv.workspace_for(K, window, lens)
    mkv.mkv_centroid_score(K, window, mode, C, S, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    return C, S


def _three_ways(K, window, mode, lens):
    """(path, C, S) for the ring kernel, the register head groups and the three kernels."""
    out = []
    shape = mkv.shape_of(K, lens)
    for ring, groups in ((True, True), (False, True), (False, False)):
        pr = mkv.mkv_set_head_group_ring(ring)
        pg = mkv.mkv_set_head_groups(groups)
        try:
            out.append((mkv.mkv_compress_single_pass(shape, window, mode),) + _centroid_score(K, window, mode, lens))
        finally:
            mkv.mkv_set_head_group_ring(pr)
            mkv.mkv_set_head_groups(pg)
    return out


def _live(lens, B, H, T):
    Th = (lens if lens is not None else torch.full((B,), T, device=DEV)).long()
    return torch.arange(T, device=DEV)[None, None, :] < Th.repeat_interleave(H).reshape(B, H)[..., None]


def _same_bits(K, window, mode, lens):
    B, H, T, D = K.shape
    (p0, C0, S0), (p1, C1, S1), (p2, C2, S2) = _three_ways(K, window, mode, lens)
    assert p0 == 4, f"the ring kernel is not taken (path {p0})"
    live = _live(lens, B, H, T)
    assert torch.equal(S0[live], S1[live]), "ring and register head groups give different scores"
    assert torch.equal(S0[live], S2[live]), "ring head groups and the three kernels give different scores"
    nwin = torch.tensor([[mkv.mkv_num_windows(int(t), window) if t > 0 else 0] * H
                         for t in (lens.cpu().tolist() if lens is not None else [T] * B)], device=DEV)
    wlive = torch.arange(C0.shape[2], device=DEV)[None, None, :] < nwin[..., None]
    assert torch.equal(C0[wlive], C2[wlive]), "ring head groups and the three kernels give different centroids"
    return S0


@pytest.mark.parametrize("mode", ["l2", "cosine"])
def test_ring_global_llama_shape(mode):
    w = synthkv.WORKLOADS["llama3.1-8b-kv-t16k"].scaled("ring-llama", layers=8)
    K, V, lens = synthkv.make_kv(w, seed=41, device=DEV)
    _same_bits(K, 0, mode, None)


@pytest.mark.parametrize("mode,window", [("l2", 4096), ("cosine", 8192), ("l2", 3000)])
def test_ring_windowed(mode, window):
    w = synthkv.WORKLOADS["qwen3-8b-kv-t64k-w4096"].scaled("ring-qwen", layers=2)
    K, V, lens = synthkv.make_kv(w, seed=42, device=DEV)
    _same_bits(K, window, mode, None)


def test_ring_phi4_windowed_shape():
    w = synthkv.WORKLOADS["phi4-kv-t128k"].scaled("ring-phi4", layers=3)
    K, V, lens = synthkv.make_kv(w, seed=43, device=DEV)
    _same_bits(K, 8192, "l2", None)


def test_ring_long_global_pieces():
    # 40000-token global heads: 1024-row pieces, several copy stages each
    w = synthkv.WORKLOADS["llama3.1-8b-kv-t16k"].scaled("ring-long", layers=1, heads=6, t_max=40000)
    K, V, lens = synthkv.make_kv(w, seed=44, device=DEV)
    _same_bits(K, 0, "l2", None)


@pytest.mark.parametrize("mode,window", [("l2", 0), ("cosine", 0), ("l2", 2048)])
def test_ring_ragged_with_empty_and_short_heads(mode, window):
    w = synthkv.WORKLOADS["ragged-b8-llama-kv-t8k-32k"].scaled("ring-ragged", layers=2, batch=6, heads=4,
                                                                t_max=12000, t_min=0)
    K, V, lens = synthkv.make_kv(w, seed=45, device=DEV)
    lens[0] = 0      # an empty head row
    lens[1] = 100    # shorter than a piece and than a copy stage
    lens[2] = 12000  # the full length
    _same_bits(K, window, mode, lens)


def test_ring_against_the_oracle():
    w = synthkv.WORKLOADS["llama3.1-8b-kv-t16k"].scaled("ring-oracle", layers=1, heads=8, t_max=9000)
    K, V, lens = synthkv.make_kv(w, seed=46, device=DEV)
    for mode, window in (("l2", 0), ("cosine", 2500)):
        S = _same_bits(K, window, mode, None)
        ora = oracle_heads(K, V, [w.t_max], w.heads, list(range(w.heads)), 0.5, mode, window)
        for h in range(w.heads):
            compare_head(ora[h], w.t_max, S_gpu=S[0, h].cpu().numpy(), mode=mode)
