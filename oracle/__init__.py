"""fp64 CPU oracle for ManifoldKV-style KV-cache compression (test
infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline and
reference legs may import this package. The CUDA library never does: it must
fail loudly instead of falling back to anything here. The arithmetic lives in
``mkv_oracle.c`` (plain C, fp64, token-order sums); this module compiles it
with gcc and marshals numpy arrays into it.

Parity pins: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (hand-computed cases, closed forms, invariants,
library routines and brute force on tiny inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmkv_oracle.so")

MODE_L2 = 0
MODE_COSINE = 1
_MODES = {"l2": MODE_L2, "cosine": MODE_COSINE, MODE_L2: MODE_L2, MODE_COSINE: MODE_COSINE}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library with gcc; return its path.

    -ffp-contract=off keeps every multiply and add separately rounded (no
    fused multiply-add), so the fp64 arithmetic is exactly what the source
    says on x86 and on Arm alike."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, f64, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        lib.oracle_bf16_to_double.restype = f64
        lib.oracle_e4m3_to_double.restype = f64
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_bf16.restype = i32
        lib.oracle_e4m3_to_bf16.argtypes = [vp, i64, vp]
        lib.oracle_gather_bytes.argtypes = [vp, i64, vp, i64, vp]
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_num_keep.restype = i64
        lib.oracle_num_keep.argtypes = [i64, f64]
        lib.oracle_window_len.restype = i64
        lib.oracle_window_len.argtypes = [i64, i64]
        lib.oracle_num_windows.restype = i64
        lib.oracle_num_windows.argtypes = [i64, i64]
        lib.oracle_centroids.restype = None
        lib.oracle_centroids.argtypes = [vp, i64, i64, i64, vp]
        lib.oracle_scores.restype = None
        lib.oracle_scores.argtypes = [vp, i64, i64, i64, i32, vp, vp]
        lib.oracle_select.restype = i32
        lib.oracle_select.argtypes = [vp, i64, i64, vp]
        lib.oracle_gather.restype = None
        lib.oracle_gather.argtypes = [vp, i64, vp, i64, vp]
        lib.oracle_compress_head.restype = i64
        lib.oracle_compress_head.argtypes = [vp, vp, i64, i64, f64, i32, i64, vp, vp, vp, vp, vp]
        lib.oracle_compress_heads.restype = i32
        lib.oracle_compress_heads.argtypes = [vp, vp, i64, i64, i64, vp, f64, i32, i64, i64,
                                              vp, vp, vp, vp]
        lib.oracle_layer_budgets.restype = i32
        lib.oracle_layer_budgets.argtypes = [vp, i32, f64, f64, i64, vp, vp]
        lib.oracle_compress_head_n.restype = i64
        lib.oracle_compress_head_n.argtypes = [vp, vp, i64, i64, i64, i32, i64, vp, vp, vp, vp, vp]
        lib.oracle_window_means.restype = None
        lib.oracle_window_means.argtypes = [vp, i64, i64, i64, vp, vp]
        lib.oracle_num_keep_quota.restype = i64
        lib.oracle_num_keep_quota.argtypes = [i64, f64, i64]
        lib.oracle_select_quota.restype = i64
        lib.oracle_select_quota.argtypes = [vp, i64, i64, f64, vp]
        lib.oracle_compress_head_quota.restype = i64
        lib.oracle_compress_head_quota.argtypes = [vp, vp, i64, i64, f64, i32, i64, vp, vp, vp, vp, vp]
        lib.oracle_oja_scores.restype = None
        lib.oracle_oja_scores.argtypes = [vp, i64, i64, vp, i64, vp, i64, vp]
        lib.oracle_compress_head_oja.restype = i64
        lib.oracle_compress_head_oja.argtypes = [vp, vp, i64, i64, vp, i64, vp, i64, i64, vp, vp, vp, vp]
        lib.oracle_compact_in_place.restype = i32
        lib.oracle_compact_in_place.argtypes = [vp, i64, i64, vp, i64]
        _lib = lib
        return lib


def _is_fp8(x) -> bool:
    return hasattr(x, "dtype") and str(x.dtype) == "torch.float8_e4m3fn"


def _codes(x) -> np.ndarray:
    """The E4M3 codes of a torch float8_e4m3fn tensor as a C-contiguous uint8 array."""
    import torch
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.uint8).numpy())


def e4m3_to_double(code: int) -> float:
    return _load().oracle_e4m3_to_double(int(code) & 0xFF)


def e4m3_to_bf16_bits(codes) -> np.ndarray:
    """Exact widening of E4M3 codes (uint8 array) to bf16 bit patterns."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(c.shape, dtype=np.uint16)
    if _load().oracle_e4m3_to_bf16(_ptr(c), c.size, _ptr(out)) != 0:
        raise ValueError("NaN E4M3 code (outside the contract)")
    return out


def _bits(x) -> np.ndarray:
    """bf16 data as a C-contiguous uint16 array of raw bit patterns.

    Accepts a numpy uint16/int16 array or a torch bfloat16 tensor (on the
    CPU); a torch float8_e4m3fn tensor is widened exactly to bf16 first."""
    if _is_fp8(x):
        return e4m3_to_bf16_bits(_codes(x))
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(x)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bits as uint16, got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _fp8_rows(res: dict, K, V) -> dict:
    """For fp8 inputs, replace the kept rows (computed on the exact bf16
    widening) by byte copies of the fp8 rows at the same indices."""
    if not _is_fp8(K):
        return res
    res = dict(res)
    res["K_out"] = gather_bytes(_codes(K), res["idx"])
    res["V_out"] = gather_bytes(_codes(V), res["idx"])
    return res


def gather_bytes(X: np.ndarray, idx) -> np.ndarray:
    """Rows X[idx] of a uint8 [T, row_bytes] array (any element type)."""
    x = np.ascontiguousarray(X, dtype=np.uint8)
    i = np.ascontiguousarray(idx, dtype=np.int32)
    out = np.zeros((i.shape[0], x.shape[1]), dtype=np.uint8)
    _load().oracle_gather_bytes(_ptr(x), x.shape[1], _ptr(i), i.shape[0], _ptr(out))
    return out


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits) & 0xFFFF)


def num_keep(T: int, ratio: float) -> int:
    """Tokens kept out of T at compression ``ratio`` (the share removed)."""
    return int(_load().oracle_num_keep(int(T), float(ratio)))


def window_len(T: int, window: int) -> int:
    return int(_load().oracle_window_len(int(T), int(window)))


def num_windows(T: int, window: int) -> int:
    return int(_load().oracle_num_windows(int(T), int(window)))


def centroids(K, window: int = 0) -> np.ndarray:
    """Per-window mean keys of one head: K [T, d] bf16 -> float64 [n_windows, d]."""
    k = _bits(K)
    T, d = k.shape
    C = np.zeros((max(num_windows(T, window), 0), d), dtype=np.float64)
    _load().oracle_centroids(_ptr(k), T, d, int(window), _ptr(C))
    return C


def scores(K, C: np.ndarray, window: int = 0, mode="l2") -> np.ndarray:
    """Per-token scores of one head against the centroids C: float64 [T]."""
    k = _bits(K)
    T, d = k.shape
    c = np.ascontiguousarray(C, dtype=np.float64)
    if c.shape != (num_windows(T, window), d):
        raise ValueError(f"centroid shape {c.shape} does not match T={T}, window={window}")
    S = np.zeros(T, dtype=np.float64)
    _load().oracle_scores(_ptr(k), T, d, int(window), _MODES[mode], _ptr(c), _ptr(S))
    return S


def select(S, n_keep: int) -> np.ndarray:
    """Indices (ascending, int32) of the n_keep highest scores; ties at the
    cut go to the lower index."""
    s = np.ascontiguousarray(S, dtype=np.float64)
    idx = np.zeros(max(int(n_keep), 0), dtype=np.int32)
    if _load().oracle_select(_ptr(s), s.shape[0], int(n_keep), _ptr(idx)) != 0:
        raise ValueError("oracle_select: bad n_keep or NaN score")
    return idx


def gather(X, idx) -> np.ndarray:
    """Rows X[idx] of a bf16 [T, d] array, as uint16 bits [len(idx), d]."""
    x = _bits(X)
    i = np.ascontiguousarray(idx, dtype=np.int32)
    out = np.zeros((i.shape[0], x.shape[1]), dtype=np.uint16)
    _load().oracle_gather(_ptr(x), x.shape[1], _ptr(i), i.shape[0], _ptr(out))
    return out


def compress_head(K, V, ratio: float, mode="l2", window: int = 0):
    """All steps for one head. Returns dict(C, S, idx, K_out, V_out)."""
    k, v = _bits(K), _bits(V)
    T, d = k.shape
    C = np.zeros((max(num_windows(T, window), 1), d), dtype=np.float64)
    S = np.zeros(max(T, 1), dtype=np.float64)
    n = num_keep(T, ratio)
    idx = np.zeros(max(n, 1), dtype=np.int32)
    ko = np.zeros((max(n, 1), d), dtype=np.uint16)
    vo = np.zeros((max(n, 1), d), dtype=np.uint16)
    got = _load().oracle_compress_head(_ptr(k), _ptr(v), T, d, float(ratio), _MODES[mode], int(window),
                                       _ptr(C), _ptr(S), _ptr(idx), _ptr(ko), _ptr(vo))
    if got != n:
        raise ValueError("oracle_compress_head failed")
    return _fp8_rows({"C": C[: num_windows(T, window)], "S": S[:T], "idx": idx[:n], "K_out": ko[:n],
                      "V_out": vo[:n]}, K, V)


def compress_heads(K, V, lens, ratio: float, mode="l2", window: int = 0, keep_stride=None):
    """All steps for a [n_heads, t_stride, d] cache with per-head lengths.

    Returns (idx int32 [n, keep_stride], kept int32 [n], K_out, V_out uint16
    [n, keep_stride, d], or uint8 codes for float8_e4m3fn inputs); entries
    past a head's kept count are zero."""
    k, v = _bits(K), _bits(V)
    n_heads, t_stride, d = k.shape
    ln = np.ascontiguousarray(lens, dtype=np.int32).reshape(-1)
    if ln.shape[0] != n_heads:
        raise ValueError("one length per head is required")
    if keep_stride is None:
        keep_stride = num_keep(t_stride, ratio)
    idx = np.zeros((n_heads, max(keep_stride, 1)), dtype=np.int32)
    kept = np.zeros(n_heads, dtype=np.int32)
    ko = np.zeros((n_heads, max(keep_stride, 1), d), dtype=np.uint16)
    vo = np.zeros_like(ko)
    rc = _load().oracle_compress_heads(_ptr(k), _ptr(v), n_heads, t_stride, d, _ptr(ln), float(ratio),
                                       _MODES[mode], int(window), int(max(keep_stride, 1)),
                                       _ptr(idx), _ptr(kept), _ptr(ko), _ptr(vo))
    if rc != 0:
        raise ValueError("oracle_compress_heads failed")
    if _is_fp8(K):  # the kept rows as fp8 bytes at the same indices
        kc, vc = _codes(K), _codes(V)
        ko = np.zeros((n_heads, max(keep_stride, 1), d), dtype=np.uint8)
        vo = np.zeros_like(ko)
        for h in range(n_heads):
            n = int(kept[h])
            ko[h, :n] = gather_bytes(kc[h], idx[h, :n])
            vo[h, :n] = gather_bytes(vc[h], idx[h, :n])
    return idx[:, :keep_stride], kept, ko[:, :keep_stride], vo[:, :keep_stride]


def layer_budgets(sensitivity, r: float, gamma: float, total: int, cap):
    """Per-layer kept-token budgets (RippleKV budget mapping). Returns
    (status, budgets int32 [L]); status 1 means the caps absorb the total."""
    sv = np.ascontiguousarray(sensitivity, dtype=np.float64)
    cp = np.ascontiguousarray(cap, dtype=np.int32)
    out = np.zeros(sv.shape[0], dtype=np.int32)
    st = _load().oracle_layer_budgets(_ptr(sv), sv.shape[0], float(r), float(gamma), int(total), _ptr(cp), _ptr(out))
    if st < 0:
        raise ValueError("oracle_layer_budgets: bad input")
    return int(st), out


def compress_head_n(K, V, n_keep: int, mode="l2", window: int = 0):
    """All steps for one head keeping exactly n_keep tokens."""
    k, v = _bits(K), _bits(V)
    T, d = k.shape
    C = np.zeros((max(num_windows(T, window), 1), d), dtype=np.float64)
    S = np.zeros(max(T, 1), dtype=np.float64)
    n = int(n_keep)
    idx = np.zeros(max(n, 1), dtype=np.int32)
    ko = np.zeros((max(n, 1), d), dtype=np.uint16)
    vo = np.zeros((max(n, 1), d), dtype=np.uint16)
    got = _load().oracle_compress_head_n(_ptr(k), _ptr(v), T, d, n, _MODES[mode], int(window), _ptr(C), _ptr(S),
                                         _ptr(idx), _ptr(ko), _ptr(vo))
    if got != n:
        raise ValueError("oracle_compress_head_n failed")
    return _fp8_rows({"C": C[: num_windows(T, window)], "S": S[:T], "idx": idx[:n], "K_out": ko[:n],
                      "V_out": vo[:n]}, K, V)


def window_means(X, window: int, radius: bool = True):
    """Cluster summaries of one head's bf16 rows X [T, d] (keys or values):
    per-window means float64 [n_windows, d] and, when asked, each window's
    radius max_t |x_t - mean|_2 float64 [n_windows] (else None)."""
    x = _bits(X)
    T, d = x.shape
    nw = max(num_windows(T, window), 0)
    M = np.zeros((max(nw, 1), d), dtype=np.float64)
    R = np.zeros(max(nw, 1), dtype=np.float64)
    _load().oracle_window_means(_ptr(x), T, d, int(window), _ptr(M), _ptr(R) if radius else None)
    return M[:nw], (R[:nw] if radius else None)


def num_keep_quota(T: int, ratio: float, window: int) -> int:
    """Kept tokens of a T-token head when every window keeps its own share."""
    return int(_load().oracle_num_keep_quota(int(T), float(ratio), int(window)))


def select_quota(S, window: int, ratio: float) -> np.ndarray:
    """Per-window-quota selection: ascending int32 indices."""
    s = np.ascontiguousarray(S, dtype=np.float64)
    n = num_keep_quota(s.shape[0], ratio, window)
    idx = np.zeros(max(n, 1), dtype=np.int32)
    got = _load().oracle_select_quota(_ptr(s), s.shape[0], int(window), float(ratio), _ptr(idx))
    if got != n:
        raise ValueError("oracle_select_quota: NaN score")
    return idx[:n]


def compress_head_quota(K, V, ratio: float, mode="l2", window: int = 0):
    """All steps for one head with per-window quotas. Returns dict(C, S, idx, K_out, V_out)."""
    k, v = _bits(K), _bits(V)
    T, d = k.shape
    C = np.zeros((max(num_windows(T, window), 1), d), dtype=np.float64)
    S = np.zeros(max(T, 1), dtype=np.float64)
    n = num_keep_quota(T, ratio, window)
    idx = np.zeros(max(n, 1), dtype=np.int32)
    ko = np.zeros((max(n, 1), d), dtype=np.uint16)
    vo = np.zeros((max(n, 1), d), dtype=np.uint16)
    got = _load().oracle_compress_head_quota(_ptr(k), _ptr(v), T, d, float(ratio), _MODES[mode], int(window),
                                             _ptr(C), _ptr(S), _ptr(idx), _ptr(ko), _ptr(vo))
    if got != n:
        raise ValueError("oracle_compress_head_quota failed")
    return _fp8_rows({"C": C[: num_windows(T, window)], "S": S[:T], "idx": idx[:n], "K_out": ko[:n],
                      "V_out": vo[:n]}, K, V)


def oja_scores(K, Q, U) -> np.ndarray:
    """OjaKV reconstruction-error scores of one head: K [T, d] bf16 keys,
    Q [M, d] bf16 query-window rows, U [d, r] basis (float; fp32 values are
    used exactly). Returns float64 [T]."""
    k, q = _bits(K), _bits(Q)
    T, d = k.shape
    u = np.ascontiguousarray(np.asarray(U, dtype=np.float64).reshape(d, -1))
    if q.shape[1] != d:
        raise ValueError("Q and K must share the head dim")
    E = np.zeros(max(T, 1), dtype=np.float64)
    _load().oracle_oja_scores(_ptr(k), T, d, _ptr(q), q.shape[0], _ptr(u), u.shape[1], _ptr(E))
    return E[:T]


def compress_head_oja(K, V, Q, U, n_keep: int):
    """OjaKV full-rank selection of one head: dict(S, idx, K_out, V_out)."""
    k, v, q = _bits(K), _bits(V), _bits(Q)
    T, d = k.shape
    u = np.ascontiguousarray(np.asarray(U, dtype=np.float64).reshape(d, -1))
    E = np.zeros(max(T, 1), dtype=np.float64)
    n = int(n_keep)
    idx = np.zeros(max(n, 1), dtype=np.int32)
    ko = np.zeros((max(n, 1), d), dtype=np.uint16)
    vo = np.zeros((max(n, 1), d), dtype=np.uint16)
    got = _load().oracle_compress_head_oja(_ptr(k), _ptr(v), T, d, _ptr(q), q.shape[0], _ptr(u), u.shape[1], n,
                                           _ptr(E), _ptr(idx), _ptr(ko), _ptr(vo))
    if got != n:
        raise ValueError("oracle_compress_head_oja failed")
    return {"S": E[:T], "idx": idx[:n], "K_out": ko[:n], "V_out": vo[:n]}


def compact_in_place(X, idx) -> np.ndarray:
    """In-place compaction of a bf16 [T, d] head: a copy of X (uint16 bits)
    with rows [0, len(idx)) replaced by X[idx] and the rest unchanged. For a
    float8_e4m3fn head the result is uint8 codes: rows are moved whole, so
    each row's bytes are moved as d / 2 uint16 pairs."""
    if _is_fp8(X):
        c = _codes(X)
        x = np.ascontiguousarray(c).view(np.uint16).copy()
        i = np.ascontiguousarray(idx, dtype=np.int32)
        if _load().oracle_compact_in_place(_ptr(x), x.shape[0], x.shape[1], _ptr(i), i.shape[0]) != 0:
            raise ValueError("oracle_compact_in_place: indices not strictly ascending in [0, T)")
        return x.view(np.uint8)
    x = _bits(X).copy()
    i = np.ascontiguousarray(idx, dtype=np.int32)
    if _load().oracle_compact_in_place(_ptr(x), x.shape[0], x.shape[1], _ptr(i), i.shape[0]) != 0:
        raise ValueError("oracle_compact_in_place: indices not strictly ascending in [0, T)")
    return x
