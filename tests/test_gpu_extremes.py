"""GPU parity at the edges of the shape space, every head against the fp64
oracle: a few very long heads (two million tokens: 8 MB pieces, the select
passes over L2, compaction chunks) and very many tiny heads (hundreds of
thousands of heads of a few tokens: grid striding, empty and one-token
heads)."""
import numpy as np
import pytest
import torch

import geometric_kv_cache_gb300 as mkv
import synthkv
from parity_util import bits, compare_head, oracle_heads, report

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mkv.load()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _compress_and_check(name, K, V, lens, ratio, mode, window, heads=None):
    B, H, T, D = K.shape
    n = B * H
    ks = mkv.mkv_num_keep(T, ratio)
    Ko = torch.zeros((B, H, max(ks, 1), D), dtype=K.dtype, device=DEV)
    Vo = torch.zeros_like(Ko)
    idx = torch.full((B, H, max(ks, 1)), -7, dtype=torch.int32, device=DEV)
    kept = torch.full((B, H), -7, dtype=torch.int32, device=DEV)
    ws = mkv.workspace_for(K, window, lens)
    mkv.mkv_compress(K, V, ratio, mode, window, ks, Ko, Vo, idx, kept, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    heads = range(n) if heads is None else heads
    lens_c = lens.cpu().numpy()
    ora = oracle_heads(K, V, lens_c, H, heads, ratio, mode, window)
    Kob, Vob = bits(Ko).reshape(n, -1, D), bits(Vo).reshape(n, -1, D)
    idxc, keptc = idx.cpu().numpy().reshape(n, -1), kept.cpu().numpy().reshape(n)
    Kf, Vf = K.reshape(n, T, D), V.reshape(n, T, D)
    near = 0
    for h in heads:
        Th = int(lens_c[h // H])
        res = compare_head(ora[h], Th, idx_gpu=idxc[h], kept_gpu=keptc[h], K_head=Kf[h], V_head=Vf[h],
                           Kout_gpu=Kob[h], Vout_gpu=Vob[h], mode=mode)
        near += res.get("near_cut_exceptions", 0)
    report(name, shape=[B, H, T], mode=mode, window=window, ratio=ratio, heads_checked=len(heads),
           near_cut_exceptions=near)


@pytest.mark.parametrize("mode,window,ratio", [("l2", 0, 0.5), ("cosine", 700001, 0.3)])
def test_two_million_token_heads(mode, window, ratio):
    # 2 rows x 1 head, T = 2^21 (the second row 1.5M tokens): pieces of
    # 32768 rows, scores beyond shared memory, ragged last window
    w = synthkv.WORKLOADS["phi4-kv-t128k"].scaled("long", layers=1, batch=2, heads=1, t_max=1 << 21)
    K, V, _ = synthkv.make_kv(w, seed=51, device=DEV)
    lens = torch.tensor([1 << 21, 3 << 19], dtype=torch.int32, device=DEV)
    _compress_and_check(f"long-{mode}-w{window}", K, V, lens, ratio, mode, window)
    del K, V
    torch.cuda.empty_cache()


def test_many_tiny_heads():
    # 16384 rows x 8 heads = 131072 heads of 0..5 tokens (keys and values
    # N(0, 1) in bf16, drawn in one call: the per-head generator is too slow
    # for this many heads); a sample of heads against the oracle
    rows, H, T = 16384, 8, 5
    g = torch.Generator().manual_seed(52)
    K = torch.randn(rows, H, T, 128, generator=g).to(torch.bfloat16).to(DEV)
    V = torch.randn(rows, H, T, 128, generator=g).to(torch.bfloat16).to(DEV)
    lens = torch.randint(0, T + 1, (rows,), generator=g, dtype=torch.int32).to(DEV)
    rng = np.random.default_rng(52)
    heads = sorted(set(rng.integers(0, rows * H, size=600).tolist()) | {0, rows * H - 1})
    for mode, window, ratio in (("l2", 0, 0.5), ("cosine", 2, 0.2)):
        _compress_and_check(f"tiny-{mode}-w{window}", K, V, lens, ratio, mode, window, heads=heads)


@pytest.mark.parametrize("mode,window,ratio", [("l2", 0, 0.5), ("cosine", 7001, 0.3)])
def test_long_heads_with_unaligned_score_rows(mode, window, ratio):
    # t_max = 45001 (above the 40960 scores a select keeps in shared memory):
    # the select's passes and the compaction read the scores from L2, as
    # 16-byte vectors where a head's row of scores starts on a 16-byte
    # boundary (head 0, 4, ...) and one score at a time elsewhere; the
    # lengths leave tails of 1, 0 and 3 scores past the last full vector
    w = synthkv.WORKLOADS["phi4-kv-t128k"].scaled("odd", layers=1, batch=3, heads=2, t_max=45001)
    K, V, _ = synthkv.make_kv(w, seed=53, device=DEV)
    lens = torch.tensor([45001, 45000, 41003], dtype=torch.int32, device=DEV)
    _compress_and_check(f"odd-{mode}-w{window}", K, V, lens, ratio, mode, window)
    del K, V
    torch.cuda.empty_cache()
