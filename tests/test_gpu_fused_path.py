"""GPU parity of the fused whole-path kernel: one cooperative launch whose
scorer head groups, selector CTAs and gatherer warps hand work over through
bounded waits. mkv_compress takes it by default under its own shape rule
(bf16, head dim 128, global centroids, 12288 < t_max <= 20480, at least 64
heads);
mkv_set_fused forces scorer/selector budgets wherever it applies, or turns
it off (this module turns it off and forces it per test, then restores the
previous setting). Its outputs must be the separate kernels' bits
(every head, every output row) on bf16 and E4M3 caches, head dims 64 / 128 /
256, ragged lengths with empty and sub-piece heads, a per-head n_keep array,
both score modes, the largest t_max it takes, and small and large scorer
and selector budgets; a small case is also checked head by head against
the fp64 oracle. Its bounded waits are made to run out on purpose (a
host-side injection, no fault): the launch must drain in about one wait
bound, report MKV_DEV_TIMEOUT, keep no rows for the heads it could not
finish, and leave the context usable."""
import time

import numpy as np
import pytest
import torch

import geometric_kv_cache_gb300 as mkv
import synthkv
from parity_util import bits, compare_head, oracle_heads

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mkv.load()
    prev = mkv.mkv_set_fused(0)
    yield
    mkv.mkv_set_fused(prev)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _compress(K, V, lens, ratio, mode, keep_stride, n_keep=None):
    B, H, T, D = K.shape
    Ko = torch.zeros((B, H, max(keep_stride, 1), D), dtype=K.dtype, device=DEV)
    Vo = torch.zeros_like(Ko)
    idx = torch.full((B, H, max(keep_stride, 1)), -7, dtype=torch.int32, device=DEV)
    kept = torch.full((B, H), -7, dtype=torch.int32, device=DEV)
    ws = mkv.workspace_for(K, 0, lens)
    mkv.mkv_compress(K, V, ratio, mode, 0, keep_stride, Ko, Vo, idx, kept, ws, lens, n_keep)
    status = mkv.mkv_device_status(ws)
    u8 = (lambda x: x.view(torch.uint8)) if K.dtype == torch.float8_e4m3fn else (lambda x: x)
    return status, (kept, idx, u8(Ko), u8(Vo))


def _both(K, V, lens, ratio, mode, keep_stride, n_keep=None, scorers=152, selectors=32):
    """(separate kernels, fused kernel) outputs; asserts the fused path was taken."""
    mkv.mkv_set_fused(0)
    st0, a = _compress(K, V, lens, ratio, mode, keep_stride, n_keep)
    mkv.mkv_set_fused(scorers, selectors)
    try:
        assert mkv.mkv_compress_single_pass(mkv.shape_of(K, lens), 0, mode) == 3
        st1, b = _compress(K, V, lens, ratio, mode, keep_stride, n_keep)
    finally:
        mkv.mkv_set_fused(0)
    assert st0 == 0 and st1 == 0
    return a, b


def _same(a, b):
    for name, x, y in zip(("kept", "idx", "K_out", "V_out"), a, b):
        assert torch.equal(x, y), f"{name} differs between the fused and the separate kernels"


def _cache(name, seed, dtype=torch.bfloat16, **changes):
    w = synthkv.WORKLOADS["llama3.1-8b-kv-t16k"].scaled(name, **changes)
    return synthkv.make_kv(w, seed=seed, device=DEV, dtype=dtype)


@pytest.mark.parametrize("mode,ratio", [("l2", 0.5), ("cosine", 0.2)])
def test_fused_equals_separate_kernels_llama_shape(mode, ratio):
    K, V, lens = _cache("fused-llama", 0, layers=8)
    a, b = _both(K, V, None, ratio, mode, mkv.mkv_num_keep(K.shape[2], ratio))
    _same(a, b)


@pytest.mark.parametrize("scorers,selectors", [(16, 1), (96, 7), (288, 400)])
def test_fused_scorer_and_selector_budgets(scorers, selectors):
    K, V, lens = _cache("fused-budget", 1, layers=4, t_max=9000)
    a, b = _both(K, V, None, 0.4, "l2", mkv.mkv_num_keep(K.shape[2], 0.4), scorers=scorers, selectors=selectors)
    _same(a, b)


def test_fused_ragged_with_empty_and_short_heads():
    w = synthkv.WORKLOADS["ragged-b8-llama-kv-t8k-32k"].scaled("fused-ragged", layers=2, batch=4, t_max=16384, t_min=1)
    K, V, lens = synthkv.make_kv(w, seed=3, device=DEV)
    lens[0], lens[1], lens[2] = 0, 255, 256
    a, b = _both(K, V, lens, 0.2, "cosine", mkv.mkv_num_keep(K.shape[2], 0.2))
    _same(a, b)
    assert int(a[0][0].sum()) == 0  # the empty row keeps nothing


def test_fused_per_head_n_keep():
    w = synthkv.WORKLOADS["ragged-b8-llama-kv-t8k-32k"].scaled("fused-nkeep", layers=2, batch=2, t_max=12000, t_min=1)
    K, V, lens = synthkv.make_kv(w, seed=5, device=DEV)
    g = torch.Generator().manual_seed(5)
    T = lens.long().repeat_interleave(w.heads).cpu()
    nk = (torch.rand(T.shape, generator=g) * (T + 1).float()).long().clamp(max=T).to(torch.int32).to(DEV)
    a, b = _both(K, V, lens, 0.5, "l2", K.shape[2], n_keep=nk)
    _same(a, b)
    assert torch.equal(a[0].flatten().cpu(), nk.cpu())


@pytest.mark.parametrize("d,dtype", [(64, torch.bfloat16), (256, torch.bfloat16), (128, torch.float8_e4m3fn)])
def test_fused_head_dims_and_fp8(d, dtype):
    K, V, lens = _cache(f"fused-d{d}", 2, dtype=dtype, layers=2, head_dim=d, t_max=10000)
    for mode in ("l2", "cosine"):
        a, b = _both(K, V, None, 0.5, mode, mkv.mkv_num_keep(K.shape[2], 0.5))
        _same(a, b)


def test_fused_largest_t_max_and_the_fallback_above_it():
    K, V, lens = _cache("fused-tmax", 4, layers=1, heads=4, t_max=20480)
    a, b = _both(K, V, None, 0.3, "l2", mkv.mkv_num_keep(20480, 0.3))
    _same(a, b)
    K, V, lens = _cache("fused-tmax1", 4, layers=1, heads=4, t_max=20481)
    mkv.mkv_set_fused(152)
    try:
        assert mkv.mkv_compress_single_pass(mkv.shape_of(K), 0, "l2") != 3  # not taken: the separate kernels
    finally:
        mkv.mkv_set_fused(0)


def test_fused_small_case_against_the_oracle():
    """Two heads (fewer than the selector CTAs): the fused outputs head by head
    against the fp64 oracle, under the same tolerances as the other paths."""
    K, V, lens = _cache("fused-oracle", 6, layers=1, heads=2, t_max=3000)
    ratio, mode = 0.3, "l2"
    ks = mkv.mkv_num_keep(3000, ratio)
    mkv.mkv_set_fused(152, 48)
    try:
        assert mkv.mkv_compress_single_pass(mkv.shape_of(K), 0, mode) == 3
        st, (kept, idx, Ko, Vo) = _compress(K, V, None, ratio, mode, ks)
    finally:
        mkv.mkv_set_fused(0)
    assert st == 0
    H = K.shape[1]
    ora = oracle_heads(K, V, np.full(K.shape[0], 3000), H, range(H), ratio, mode, 0)
    Kf, Vf = K.reshape(-1, 3000, K.shape[3]), V.reshape(-1, 3000, V.shape[3])
    kf, vf = Ko.reshape(H, ks, -1), Vo.reshape(H, ks, -1)
    for h in range(H):
        compare_head(ora[h], 3000, idx_gpu=idx.reshape(H, -1)[h].cpu().numpy(), kept_gpu=kept.flatten()[h].item(),
                     K_head=Kf[h], V_head=Vf[h], Kout_gpu=bits(kf[h]), Vout_gpu=bits(vf[h]), mode=mode)


def test_fused_kernel_own_rule():
    """The default setting runs the fused kernel where it was measured faster:
    bf16, head dim 128, global centroids, 12288 < t_max <= 20480, at least 64
    heads."""
    prev = mkv.mkv_set_fused(-1)
    try:
        q = mkv.mkv_compress_single_pass
        assert q(mkv.MkvShape(32, 8, 16384, 128, 0, None), 0, "l2") == 3
        assert q(mkv.MkvShape(32, 8, 16384, 128, 0, None), 0, "cosine") == 3
        assert q(mkv.MkvShape(8, 8, 20480, 128, 0, None), 0, "l2") == 3
        assert q(mkv.MkvShape(8, 8, 20480, 128, 0, None), 20480, "l2") == 3     # one window covers the head
        assert q(mkv.MkvShape(64, 8, 8192, 128, 0, None), 0, "l2") != 3          # 8K tokens
        assert q(mkv.MkvShape(32, 8, 16384, 128, 0, None), 4096, "l2") == 2      # windows
        assert q(mkv.MkvShape(8, 8, 20481, 128, 0, None), 0, "l2") != 3          # above the kernel's limit
        assert q(mkv.MkvShape(8, 8, 16384, 64, 0, None), 0, "l2") != 3           # other head dims
        assert q(mkv.MkvShape(32, 8, 16384, 128, 1, None), 0, "l2") != 3         # E4M3 caches
        assert q(mkv.MkvShape(4, 8, 16384, 128, 0, None), 0, "l2") != 3          # 32 heads
        assert q(mkv.MkvShape(8, 8, 16384, 128, 0, None), 0, "l2") == 3          # 64 heads
    finally:
        mkv.mkv_set_fused(prev)
    K, V, lens = _cache("fused-rule", 7, layers=8)
    prev = mkv.mkv_set_fused(-1)
    try:
        assert mkv.mkv_compress_single_pass(mkv.shape_of(K), 0, "l2") == 3
        st1, b = _compress(K, V, None, 0.5, "l2", mkv.mkv_num_keep(K.shape[2], 0.5))
    finally:
        mkv.mkv_set_fused(0)
    st0, a = _compress(K, V, None, 0.5, "l2", mkv.mkv_num_keep(K.shape[2], 0.5))
    assert st0 == 0 and st1 == 0
    _same(a, b)


@pytest.mark.parametrize("stage", [0, 1])
def test_fused_stalled_wait_times_out_and_drains(stage):
    # One wait that cannot end: stage 0 raises scorer group 0's barrier
    # target above its CTA count (head 0 is group 0's first unit), stage 1
    # makes head 0's select wait for one scorer more than its group has.
    K, V, lens = _cache("fused-stall", 3, layers=4)  # 32 heads x 16384 tokens
    ratio, mode = 0.5, "l2"
    B, H, T, D = K.shape
    ks = mkv.mkv_num_keep(T, ratio)
    ref_status, ref = _compress(K, V, lens, ratio, mode, ks)  # separate kernels (fused off in this module)
    assert ref_status == 0
    Ko = torch.zeros((B, H, ks, D), dtype=K.dtype, device=DEV)
    Vo = torch.zeros_like(Ko)
    idx = torch.full((B, H, ks), -7, dtype=torch.int32, device=DEV)
    kept = torch.full((B, H), -7, dtype=torch.int32, device=DEV)
    ws = mkv.workspace_for(K, 0, lens)
    assert mkv.mkv_device_status(ws) == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    mkv.mkv_inject_stalled_fused(K, V, ratio, mode, ks, Ko, Vo, idx, kept, stage, ws, lens)
    status = mkv.mkv_device_status(ws)  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert status & mkv.MKV_DEV_TIMEOUT
    # one wait bound (1 s), not one per wait: the other waits gave up at once
    assert elapsed < 2.5, f"the stalled launch took {elapsed:.2f} s"
    kc = kept.reshape(-1).cpu()
    assert int(kc[0]) == 0, "the stalled head kept rows"
    assert bool(torch.all((kc == 0) | (kc == ks))), "a head kept a partial count"
    # a head that kept rows was selected on its complete scores: its indices
    # are the separate kernels' (no select ran on stale or partial scores)
    done = torch.nonzero(kc == ks).flatten().tolist()
    ref_idx = ref[1].reshape(B * H, ks)
    got_idx = idx.reshape(B * H, ks)
    for h in done:
        assert torch.equal(got_idx[h], ref_idx[h]), f"head {h} kept other rows than the separate kernels"
    if stage == 1:  # only head 0's select waited: every other head completed
        assert len(done) == B * H - 1
    # the context is still usable: an ordinary fused call on the same
    # workspace gives the separate kernels' bits
    a, b = _both(K, V, lens, ratio, mode, ks)
    _same(a, b)
