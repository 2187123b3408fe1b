"""Host-side checks of the C ABI (no GPU needed): the library builds for
sm_103a and loads, exports every symbol include/mkv.h declares, and rejects
bad arguments on the host before anything is enqueued."""
import ctypes
import os
import re

import pytest
import torch

import geometric_kv_cache_gb300 as mkv
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mkv.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mkv_[a-z0-9_]+)\s*\(", text)))


def test_library_loads_and_exports_every_declared_symbol():
    lib = mkv.load()
    declared = _declared_functions()
    assert declared, "no functions parsed from the header"
    assert sorted(mkv.EXPORTED) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_num_keep_matches_the_oracle_rounding():
    for T in list(range(0, 40)) + [4096, 16384, 32767, 65536, 131072, 8193, 24577]:
        for r in (0.0, 0.1, 0.2, 0.25, 1 / 3, 0.5, 0.75, 0.9, 1.0, 0.26, 0.24, 0.125):
            assert mkv.mkv_num_keep(T, r) == oracle.num_keep(T, r), (T, r)
    assert mkv.mkv_num_keep(4096, 0.2) == 3277
    assert mkv.mkv_num_keep(10, -0.1) == -1
    assert mkv.mkv_num_keep(10, 1.5) == -1
    assert mkv.mkv_num_keep(-1, 0.5) == -1
    assert mkv.mkv_num_keep(10, float("nan")) == -1


def test_num_windows_matches_the_oracle_tiling():
    for T in (0, 1, 5, 4096, 65536, 65537):
        for w in (0, 1, 3, 4096, 8192, 10 ** 6):
            assert mkv.mkv_num_windows(T, w) == oracle.num_windows(T, w), (T, w)


def _shape(batch=2, heads=8, t_max=1024, head_dim=128, seq_lens=None, dtype=0):
    return mkv.MkvShape(batch, heads, t_max, head_dim, dtype, seq_lens)


def test_workspace_size_grows_with_the_problem():
    small = mkv.mkv_workspace_size(_shape(t_max=1024))
    big = mkv.mkv_workspace_size(_shape(t_max=65536))
    assert 256 < small < big
    # scores alone need 4 bytes per token
    assert big >= 2 * 8 * 65536 * 4
    assert mkv.mkv_workspace_size(_shape(head_dim=96)) == 0
    assert mkv.mkv_workspace_size(_shape(batch=-1)) == 0


# Fake, aligned device addresses: every call below must fail its host checks
# and so never touch them.
A = 1 << 20


def _compress(shape, ratio=0.5, mode=0, window=0, keep_stride=512, K=A, V=A, Ko=A, Vo=A, idx=A, kept=A,
              ws=A, ws_bytes=1 << 40, n_keep=None):
    lib = mkv.load()
    vp = ctypes.c_void_p
    return lib.mkv_compress(vp(K), vp(V), shape, ratio, vp(n_keep) if n_keep else None, mode, window, keep_stride,
                            vp(Ko) if Ko else None, vp(Vo) if Vo else None, vp(idx) if idx else None,
                            vp(kept) if kept else None, vp(ws) if ws else None, ws_bytes, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(shape=_shape(head_dim=96)), mkv.MKV_ERR_UNSUPPORTED),
    (dict(shape=_shape(t_max=(1 << 30) + 1)), mkv.MKV_ERR_UNSUPPORTED),
    (dict(shape=_shape(heads=-1)), mkv.MKV_ERR_INVALID_ARG),
    (dict(shape=_shape(), ratio=1.5), mkv.MKV_ERR_INVALID_ARG),
    (dict(shape=_shape(), ratio=-0.1), mkv.MKV_ERR_INVALID_ARG),
    (dict(shape=_shape(), ratio=float("nan")), mkv.MKV_ERR_INVALID_ARG),
    (dict(shape=_shape(), mode=7), mkv.MKV_ERR_INVALID_ARG),
    (dict(shape=_shape(), window=-3), mkv.MKV_ERR_INVALID_ARG),
    (dict(shape=_shape(), keep_stride=511), mkv.MKV_ERR_INVALID_ARG),
    (dict(shape=_shape(), K=0), mkv.MKV_ERR_INVALID_ARG),
    (dict(shape=_shape(), K=A + 8), mkv.MKV_ERR_INVALID_ARG),
    (dict(shape=_shape(), Ko=A + 4), mkv.MKV_ERR_INVALID_ARG),
    (dict(shape=_shape(), Vo=0), mkv.MKV_ERR_INVALID_ARG),
    (dict(shape=_shape(), idx=A + 2), mkv.MKV_ERR_INVALID_ARG),
    (dict(shape=_shape(), ws=0), mkv.MKV_ERR_WORKSPACE),
    (dict(shape=_shape(), ws=A + 16), mkv.MKV_ERR_WORKSPACE),
    (dict(shape=_shape(), ws_bytes=1024), mkv.MKV_ERR_WORKSPACE),
])
def test_compress_rejects_bad_arguments_on_the_host(kwargs, status):
    assert _compress(**kwargs) == status


def test_empty_problems_enqueue_nothing_and_succeed():
    for shp, stride in ((_shape(batch=0), 512), (_shape(heads=0), 512), (_shape(t_max=0), 0)):
        assert _compress(shp, keep_stride=stride) == mkv.MKV_OK


def test_step_calls_reject_bad_arguments():
    lib = mkv.load()
    vp = ctypes.c_void_p
    shp = _shape()
    big = 1 << 40
    assert lib.mkv_centroid(vp(A), shp, -1, vp(A), vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_centroid(vp(A), shp, 0, vp(A), vp(A), 16, None) == mkv.MKV_ERR_WORKSPACE
    assert lib.mkv_score(vp(A), vp(A), shp, 0, 5, vp(A), vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_score(vp(A), None, shp, 0, 0, vp(A), vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_select_topk(vp(A), shp, 2.0, None, vp(A), vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_select_topk(vp(A), shp, 0.5, None, vp(A + 4), vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_compact(vp(A), vp(A), vp(A), vp(A), shp, 0.5, None, 10, vp(A), vp(A), vp(A), vp(A), vp(A), big,
                           None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_compact(vp(A), vp(A), None, None, shp, 0.5, None, 512, vp(A), vp(A), vp(A), None, vp(A), big,
                           None) == mkv.MKV_ERR_INVALID_ARG
    events = (ctypes.c_void_p * 2)(vp(A), vp(A))
    assert lib.mkv_compress_profiled(vp(A), vp(A), shp, 0.5, None, 0, 0, 512, vp(A), vp(A), None, None, vp(A), big,
                                     None, events, 2) == mkv.MKV_ERR_INVALID_ARG
    assert mkv.mkv_compress_num_stages() == 6


def test_status_strings():
    for s in range(6):
        assert mkv.mkv_status_string(s).startswith("MKV_")
    assert "unknown" in mkv.mkv_status_string(99)


def test_layer_budgets_match_the_oracle():
    import json
    import numpy as np
    with open(os.path.join(ROOT, "tests", "golden", "budget_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        st, b = mkv.mkv_layer_budgets(c["s"], c["r"], c["gamma"], c["total"], c["cap"])
        assert (st, b) == (c.get("status", 0), c["budget"]), c
    rng = np.random.default_rng(23)
    for _ in range(300):
        L = int(rng.integers(1, 40))
        s = rng.normal(size=L)
        r, gamma = float(np.exp(rng.normal())), float(1 + rng.exponential(3))
        cap = rng.integers(0, 5000, size=L)
        total = int(rng.integers(0, max(1, cap.sum()) + 100))
        st, b = mkv.mkv_layer_budgets(s, r, gamma, total, cap)
        st_o, b_o = oracle.layer_budgets(s, r, gamma, total, cap)
        assert st == st_o and b == b_o.tolist()
    for bad in ((0.0, 2.0), (2.0, 0.5), (float("nan"), 2.0)):
        with pytest.raises(mkv.MKVError):
            mkv.mkv_layer_budgets([0, 1], bad[0], bad[1], 10, [10, 10])


def test_num_keep_quota_matches_the_oracle():
    for T in (0, 1, 2, 7, 100, 1023, 4096, 5000):
        for W in (0, 1, 3, 10, 256, 4096, 10000):
            for r in (0.0, 0.2, 0.5, 0.75, 1.0):
                assert mkv.mkv_num_keep_quota(T, r, W) == oracle.num_keep_quota(T, r, W), (T, W, r)
    assert mkv.mkv_num_keep_quota(-1, 0.5, 4) == -1
    assert mkv.mkv_num_keep_quota(10, 0.5, -4) == -1
    assert mkv.mkv_num_keep_quota(10, 2.0, 4) == -1


def test_window_means_and_quota_calls_reject_bad_arguments():
    lib = mkv.load()
    vp = ctypes.c_void_p
    shp = _shape()
    big = 1 << 40
    # radius only for windows of at most 128 tokens
    assert lib.mkv_window_means(vp(A), shp, 129, vp(A), vp(A), vp(A), big, None) == mkv.MKV_ERR_UNSUPPORTED
    assert lib.mkv_window_means(vp(A), shp, 0, vp(A), vp(A), vp(A), big, None) == mkv.MKV_ERR_UNSUPPORTED
    assert lib.mkv_window_means(vp(A), shp, -1, vp(A), None, vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_window_means(vp(A + 8), shp, 10, vp(A), None, vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_window_means(vp(A), shp, 10, vp(A + 4), None, vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_window_means(vp(A), shp, 10, vp(A), vp(A + 2), vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_window_means(vp(A), shp, 10, vp(A), None, vp(A), 16, None) == mkv.MKV_ERR_WORKSPACE
    assert lib.mkv_window_means(vp(A), _shape(head_dim=96), 10, vp(A), None, vp(A), big, None) == \
        mkv.MKV_ERR_UNSUPPORTED
    # the quota selection needs room for every window's share
    need = mkv.mkv_num_keep_quota(shp.t_max, 0.5, 3)
    assert need > mkv.mkv_num_keep(shp.t_max, 0.5)
    assert lib.mkv_select_quota(vp(A), shp, 0.5, 3, need - 1, vp(A), vp(A), vp(A), big, None) == \
        mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_select_quota(vp(A), shp, 0.5, 3, need, None, vp(A), vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_select_quota(vp(A), shp, 0.5, -3, need, vp(A), vp(A), vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_compress_quota(vp(A), vp(A), shp, 0.5, 0, 3, need - 1, vp(A), vp(A), None, None, vp(A), big,
                                  None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_compress_quota(vp(A), vp(A), shp, 0.5, 0, 3, need, vp(A), vp(A), None, None, vp(A), 1024,
                                  None) == mkv.MKV_ERR_WORKSPACE
    assert lib.mkv_compress_quota(vp(A), vp(A), _shape(batch=0), 0.5, 0, 3, need, vp(A), vp(A), None, None, vp(A),
                                  big, None) == mkv.MKV_OK


def test_quota_stride_bound_is_the_quota_total():
    # one-token windows at ratio 0.8 keep nothing: a zero stride is enough,
    # though the global selection of the same shape would need 205 slots
    lib = mkv.load()
    vp = ctypes.c_void_p
    shp = _shape(batch=0)
    assert mkv.mkv_num_keep_quota(shp.t_max, 0.8, 1) == 0
    assert lib.mkv_compress_quota(vp(A), vp(A), shp, 0.8, 0, 1, 0, vp(A), vp(A), None, None, vp(A), 1 << 40,
                                  None) == mkv.MKV_OK
    assert _compress(shp, ratio=0.8, keep_stride=0) == mkv.MKV_ERR_INVALID_ARG


def test_oja_calls_reject_bad_arguments():
    lib = mkv.load()
    vp = ctypes.c_void_p
    shp = _shape()
    big = 1 << 40
    ws_need = mkv.mkv_oja_workspace_size(shp, 128)
    assert ws_need > mkv.mkv_workspace_size(shp)
    assert mkv.mkv_oja_workspace_size(shp, 100) == 0 and mkv.mkv_oja_workspace_size(shp, 512) == 0

    def score(K=A, Q=A, U=A, shape=shp, n_query=128, rank=64, S=A, ws=A, ws_bytes=big):
        return lib.mkv_oja_score(vp(K) if K else None, vp(Q) if Q else None, vp(U) if U else None, shape, n_query,
                                 rank, vp(S) if S else None, vp(ws) if ws else None, ws_bytes, None)

    assert score(n_query=100) == mkv.MKV_ERR_INVALID_ARG
    assert score(n_query=0) == mkv.MKV_ERR_INVALID_ARG
    assert score(n_query=272) == mkv.MKV_ERR_INVALID_ARG
    assert score(rank=129) == mkv.MKV_ERR_INVALID_ARG
    assert score(rank=-1) == mkv.MKV_ERR_INVALID_ARG
    assert score(U=0) == mkv.MKV_ERR_INVALID_ARG
    assert score(U=0, rank=0, shape=_shape(batch=0)) == mkv.MKV_OK
    assert score(K=A + 8) == mkv.MKV_ERR_INVALID_ARG
    assert score(Q=A + 8) == mkv.MKV_ERR_INVALID_ARG
    assert score(S=0) == mkv.MKV_ERR_INVALID_ARG
    assert score(ws_bytes=ws_need - 1) == mkv.MKV_ERR_WORKSPACE
    assert score(ws=A + 16) == mkv.MKV_ERR_WORKSPACE
    assert score(shape=_shape(head_dim=96)) == mkv.MKV_ERR_UNSUPPORTED
    # 32-bit TMA row coordinates
    assert score(shape=_shape(batch=1024, heads=64, t_max=32768)) == mkv.MKV_ERR_UNSUPPORTED
    assert lib.mkv_compress_oja(vp(A), None, vp(A), vp(A), shp, 128, 64, 0.5, None, 512, vp(A), vp(A), None, None,
                                vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert lib.mkv_compress_oja(vp(A), vp(A), vp(A), vp(A), shp, 128, 64, 0.5, None, 100, vp(A), vp(A), None, None,
                                vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG


def test_in_place_compress_rejects_bad_arguments():
    lib = mkv.load()
    vp = ctypes.c_void_p
    shp = _shape()
    big = 1 << 40
    f = lib.mkv_compress_inplace
    assert f(None, vp(A), shp, 0.5, None, 0, 0, None, None, vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert f(vp(A + 8), vp(A), shp, 0.5, None, 0, 0, None, None, vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert f(vp(A), vp(A), shp, 1.5, None, 0, 0, None, None, vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert f(vp(A), vp(A), shp, 0.5, None, 9, 0, None, None, vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert f(vp(A), vp(A), shp, 0.5, None, 0, 0, vp(A + 2), None, vp(A), big, None) == mkv.MKV_ERR_INVALID_ARG
    assert f(vp(A), vp(A), shp, 0.5, None, 0, 0, None, None, vp(A), 64, None) == mkv.MKV_ERR_WORKSPACE
    assert f(vp(A), vp(A), _shape(batch=0), 0.5, None, 0, 0, None, None, vp(A), big, None) == mkv.MKV_OK


def test_head_dims():
    # 64, 128 and 256 are supported by the streaming path (workspace grows
    # with d); other dims are refused; the OjaKV scorer is built for 128
    sizes = [mkv.mkv_workspace_size(_shape(head_dim=d)) for d in (64, 128, 256)]
    assert 0 < sizes[0] < sizes[1] < sizes[2]
    for d in (0, 32, 96, 192, 512):
        assert mkv.mkv_workspace_size(_shape(head_dim=d)) == 0
        assert _compress(_shape(head_dim=d)) in (mkv.MKV_ERR_UNSUPPORTED, mkv.MKV_ERR_INVALID_ARG)
    lib = mkv.load()
    vp = ctypes.c_void_p
    assert lib.mkv_oja_score(vp(A), vp(A), vp(A), _shape(head_dim=64), 128, 8, vp(A), vp(A), 1 << 40, None) == \
        mkv.MKV_ERR_UNSUPPORTED
    assert _compress(_shape(head_dim=64, batch=0)) == mkv.MKV_OK
    assert _compress(_shape(head_dim=256, batch=0)) == mkv.MKV_OK


def test_cache_dtypes():
    # bf16 (0) and E4M3 (1) caches share one workspace layout; other types are unsupported
    assert mkv.mkv_workspace_size(_shape(dtype=1)) == mkv.mkv_workspace_size(_shape(dtype=0)) > 0
    for bad in (2, -1, 7):
        assert mkv.mkv_workspace_size(_shape(dtype=bad)) == 0
        assert mkv.load().mkv_centroid(None, _shape(dtype=bad), 0, None, None, 0, None) == mkv.MKV_ERR_UNSUPPORTED
    # the OjaKV scorer is bf16 only
    assert mkv.mkv_oja_workspace_size(_shape(dtype=1), 128) == 0
    assert mkv.mkv_oja_workspace_size(_shape(dtype=0), 128) > 0
    assert mkv.load().mkv_oja_score(None, None, None, _shape(dtype=1), 128, 8, None, None, 0, None) == \
        mkv.MKV_ERR_UNSUPPORTED
    # the binding maps torch dtypes and refuses mixed caches
    K = torch.zeros((1, 2, 8, 64), dtype=torch.float8_e4m3fn)
    assert mkv.shape_of(K).dtype == 1 and mkv.shape_of(K.to(torch.bfloat16)).dtype == 0
    with pytest.raises(ValueError):
        mkv.shape_of(K.float())
    with pytest.raises(ValueError):
        mkv._cache_types(K, K.to(torch.bfloat16))
