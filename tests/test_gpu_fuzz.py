"""Randomised GPU parity sweep: seeded random shapes, head dims, modes,
windows, ratios and ragged lengths through mkv_compress (whichever centroid +
score path the library picks), every head against the fp64 oracle with the
tolerances of parity_util."""
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


@pytest.mark.parametrize("case", range(24))
def test_random_configuration(case):
    rng = np.random.default_rng(1000 + case)
    d = int(rng.choice([64, 128, 256]))
    rows, heads = int(rng.integers(1, 4)), int(rng.integers(1, 4))
    t_max = int(rng.choice([1, 17, 300, 1000, 4097, 9000]))
    t_min = int(rng.integers(0, t_max + 1))
    mode = str(rng.choice(["l2", "cosine"]))
    window = int(rng.choice([0, 0, 1, 64, 256, 1000, 5000]))
    ratio = float(rng.choice([0.0, 0.1, 0.25, 0.5, 0.9, 1.0]))
    w = synthkv.WORKLOADS["ragged-b8-llama-kv-t8k-32k"].scaled(
        "fuzz", layers=1, batch=rows, heads=heads, t_max=t_max, t_min=t_min, head_dim=d)
    K, V, lens = synthkv.make_kv(w, seed=case, device=DEV)
    B, H, T, D = K.shape
    ks = mkv.mkv_num_keep(T, ratio)
    Ko = torch.zeros((B, H, max(ks, 1), D), dtype=torch.bfloat16, device=DEV)
    Vo = torch.zeros_like(Ko)
    idx = torch.full((B, H, max(ks, 1)), -7, dtype=torch.int32, device=DEV)
    kept = torch.full((B, H), -7, dtype=torch.int32, device=DEV)
    ws = mkv.workspace_for(K, window, lens)
    mkv.mkv_compress(K, V, ratio, mode, window, ks, Ko, Vo, idx, kept, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    n = B * H
    lens_c = lens.cpu().numpy()
    ora = oracle_heads(K, V, lens_c, H, range(n), ratio, mode, window)
    Kob, Vob = bits(Ko).reshape(n, -1, D), bits(Vo).reshape(n, -1, D)
    idxc, keptc = idx.cpu().numpy().reshape(n, -1), kept.cpu().numpy().reshape(n)
    near = 0
    for h in range(n):
        Th = int(lens_c[h // H])
        res = compare_head(ora[h], Th, idx_gpu=idxc[h], kept_gpu=keptc[h], K_head=K.reshape(n, T, D)[h],
                           V_head=V.reshape(n, T, D)[h], Kout_gpu=Kob[h], Vout_gpu=Vob[h], mode=mode)
        near += res.get("near_cut_exceptions", 0)
    report(f"fuzz{case}", d=d, shape=[rows, heads, t_max, t_min], mode=mode, window=window, ratio=ratio,
           path=mkv.mkv_compress_single_pass(mkv.shape_of(K, lens), window, mode), near_cut_exceptions=near)
