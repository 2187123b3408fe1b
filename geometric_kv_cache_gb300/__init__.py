"""Python binding of the GB300 ManifoldKV-style KV-cache compressor.

Thin ctypes marshalling over the C ABI in ``include/mkv.h`` (``libmkv.so``,
built in-tree by ``geometric_kv_cache_gb300.build``). Every step of the path
runs in the library's CUDA kernels; this module only turns torch tensors into
pointers and sizes, passes the current CUDA stream, and raises on a non-OK
status. There is no CPU fallback: without the compiled library, or without a
CUDA device, the calls raise.

Functions carry the C names (``mkv_centroid``, ``mkv_score``,
``mkv_select_topk``, ``mkv_compact``, ``mkv_compress``, ...). ``compress`` is
a convenience wrapper that allocates the outputs and the workspace with torch.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

MKV_OK = 0
MKV_ERR_INVALID_ARG = 1
MKV_ERR_UNSUPPORTED = 2
MKV_ERR_WORKSPACE = 3
MKV_ERR_CUDA = 4
MKV_ERR_DEVICE = 5

MKV_DEV_BAD_SEQ_LEN = 0x1
MKV_DEV_BAD_N_KEEP = 0x2
MKV_DEV_INTERNAL = 0x4
MKV_DEV_TIMEOUT = 0x8

MKV_MODE_L2 = 0
MKV_MODE_COSINE = 1
_MODES = {"l2": MKV_MODE_L2, "cosine": MKV_MODE_COSINE, MKV_MODE_L2: MKV_MODE_L2, MKV_MODE_COSINE: MKV_MODE_COSINE}

HEAD_DIM = 128

# Every symbol include/mkv.h declares (checked by the tests).
EXPORTED = (
    "mkv_num_keep", "mkv_num_windows", "mkv_workspace_size", "mkv_centroid", "mkv_score",
    "mkv_select_topk", "mkv_compact", "mkv_compress", "mkv_compress_num_stages",
    "mkv_compress_profiled", "mkv_compress_host", "mkv_device_status", "mkv_status_string",
    "mkv_compress_noalloc", "mkv_compress_single_pass", "mkv_set_single_pass", "mkv_layer_budgets",
    "mkv_inject_stalled_windows", "mkv_window_means", "mkv_num_keep_quota", "mkv_select_quota",
    "mkv_compress_quota", "mkv_oja_workspace_size", "mkv_oja_score", "mkv_compress_oja", "mkv_oja_score_profiled",
    "mkv_compress_inplace", "mkv_set_head_groups", "mkv_set_fused", "mkv_centroid_score",
    "mkv_inject_stalled_fused", "mkv_set_head_group_ring", "mkv_head_group_plan", "mkv_set_oja_pair",
)


class MkvShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32), ("t_max", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32), ("seq_lens", ctypes.c_void_p)]


# mkv_dtype of each supported cache element type
DTYPES = {torch.bfloat16: 0, torch.float8_e4m3fn: 1}


class MKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {mkv_status_string(status)}")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True):
    """Load libmkv.so (building it first if it is missing and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"{path} is missing: run geometric_kv_cache_gb300.build.build_library()")
            _build.build_library()
        lib = ctypes.CDLL(path)
        i32, u32, f64, vp, sz = ctypes.c_int32, ctypes.c_uint32, ctypes.c_double, ctypes.c_void_p, ctypes.c_size_t
        sig = {
            "mkv_num_keep": (i32, [i32, f64]),
            "mkv_num_windows": (i32, [i32, i32]),
            "mkv_workspace_size": (sz, [MkvShape, i32]),
            "mkv_centroid": (i32, [vp, MkvShape, i32, vp, vp, sz, vp]),
            "mkv_score": (i32, [vp, vp, MkvShape, i32, i32, vp, vp, sz, vp]),
            "mkv_select_topk": (i32, [vp, MkvShape, f64, vp, vp, vp, sz, vp]),
            "mkv_compact": (i32, [vp, vp, vp, vp, MkvShape, f64, vp, i32, vp, vp, vp, vp, vp, sz, vp]),
            "mkv_compress": (i32, [vp, vp, MkvShape, f64, vp, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]),
            "mkv_compress_num_stages": (i32, []),
            "mkv_compress_single_pass": (i32, [MkvShape, i32, i32]),
            "mkv_set_single_pass": (i32, [i32]),
            "mkv_set_head_groups": (i32, [i32]),
            "mkv_set_head_group_ring": (i32, [i32]),
            "mkv_head_group_plan": (i32, [MkvShape, i32, i32, ctypes.POINTER(i32)]),
            "mkv_set_fused": (i32, [i32, i32]),
            "mkv_set_oja_pair": (i32, [i32]),
            "mkv_centroid_score": (i32, [vp, MkvShape, i32, i32, vp, vp, vp, sz, vp]),
            "mkv_layer_budgets": (i32, [vp, i32, f64, f64, ctypes.c_int64, vp, vp]),
            "mkv_inject_stalled_windows": (i32, [vp, vp, MkvShape, f64, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]),
            "mkv_inject_stalled_fused": (i32, [vp, vp, MkvShape, f64, i32, i32, vp, vp, vp, vp, i32, vp, sz, vp]),
            "mkv_compress_profiled": (i32, [vp, vp, MkvShape, f64, vp, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp,
                                            ctypes.POINTER(vp), i32]),
            "mkv_compress_host": (i32, [vp, vp, vp, vp, MkvShape, f64, i32, i32, i32, vp, vp, vp, vp,
                                        vp, vp, vp, vp, vp, sz, vp]),
            "mkv_device_status": (i32, [vp, vp, ctypes.POINTER(u32)]),
            "mkv_compress_noalloc": (i32, [vp, vp, MkvShape, f64, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp]),
            "mkv_status_string": (ctypes.c_char_p, [i32]),
            "mkv_window_means": (i32, [vp, MkvShape, i32, vp, vp, vp, sz, vp]),
            "mkv_oja_workspace_size": (sz, [MkvShape, i32]),
            "mkv_compress_inplace": (i32, [vp, vp, MkvShape, f64, vp, i32, i32, vp, vp, vp, sz, vp]),
            "mkv_oja_score": (i32, [vp, vp, vp, MkvShape, i32, i32, vp, vp, sz, vp]),
            "mkv_oja_score_profiled": (i32, [vp, vp, vp, MkvShape, i32, i32, vp, vp, sz, vp, ctypes.POINTER(vp), i32]),
            "mkv_compress_oja": (i32, [vp, vp, vp, vp, MkvShape, i32, i32, f64, vp, i32, vp, vp, vp, vp, vp, sz,
                                       vp]),
            "mkv_num_keep_quota": (i32, [i32, f64, i32]),
            "mkv_select_quota": (i32, [vp, MkvShape, f64, i32, i32, vp, vp, vp, sz, vp]),
            "mkv_compress_quota": (i32, [vp, vp, MkvShape, f64, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


# ------------------------------------------------------------------ helpers --

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != MKV_OK:
        raise MKVError(status, where)


def _cache_types(*ts):
    """The cache tensors of one call (K, V and the compacted outputs) share one
    element type: the library reads them all with the shape's dtype."""
    types = {t.dtype for t in ts if t is not None}
    if len(types) > 1 or not types <= set(DTYPES):
        raise ValueError("K, V and the output caches must share one dtype: bf16 or float8_e4m3fn")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors passed to the CUDA library must live on a CUDA device")
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors passed to the CUDA library must be contiguous")


def shape_of(K: torch.Tensor, seq_lens: Optional[torch.Tensor] = None) -> MkvShape:
    """mkv_shape of a [batch, heads, t_max, head_dim] bf16 or float8_e4m3fn cache."""
    if K.dim() != 4 or K.dtype not in DTYPES:
        raise ValueError("K must be a bf16 or float8_e4m3fn tensor [batch, heads, t_max, head_dim]")
    if seq_lens is not None and (seq_lens.dtype != torch.int32 or seq_lens.numel() != K.shape[0]):
        raise ValueError("seq_lens must be int32 [batch]")
    b, h, t, d = K.shape
    return MkvShape(b, h, t, d, DTYPES[K.dtype], None if seq_lens is None else seq_lens.data_ptr())


def mkv_status_string(status: int) -> str:
    return load().mkv_status_string(int(status)).decode()


def mkv_num_keep(T: int, ratio: float) -> int:
    return int(load().mkv_num_keep(int(T), float(ratio)))


def mkv_num_windows(t_max: int, window: int) -> int:
    return int(load().mkv_num_windows(int(t_max), int(window)))


def mkv_workspace_size(shape: MkvShape, window: int = 0) -> int:
    return int(load().mkv_workspace_size(shape, int(window)))


def mkv_compress_num_stages() -> int:
    return int(load().mkv_compress_num_stages())


def mkv_compress_single_pass(shape: MkvShape, window: int = 0, mode="l2") -> int:
    """1 if mkv_compress reads K once for this shape on the current device."""
    return int(load().mkv_compress_single_pass(shape, int(window), _MODES[mode]))


def mkv_set_single_pass(enable: bool) -> bool:
    """Allow or forbid the single-pass centroid + score kernel; returns the
    previous setting."""
    return bool(load().mkv_set_single_pass(1 if enable else 0))


def mkv_set_head_groups(enable: bool) -> bool:
    """Allow or forbid the head-group kernel; returns the previous setting."""
    return bool(load().mkv_set_head_groups(1 if enable else 0))


def mkv_set_head_group_ring(enable: bool) -> bool:
    """Allow or forbid the copy-ring form of the head-group kernel (bf16,
    head dim 128); returns the previous setting."""
    return bool(load().mkv_set_head_group_ring(1 if enable else 0))


def mkv_head_group_plan(shape, window: int, mode) -> Optional[dict]:
    """The head-group plan on the current device (groups, CTAs per group,
    windows per unit, copy ring), or None when head groups do not apply."""
    out = (ctypes.c_int32 * 4)()
    if load().mkv_head_group_plan(shape, int(window), _MODES[mode], out) != 0:
        return None
    return {"groups": out[0], "gsize": out[1], "windows_per_unit": out[2], "ring": bool(out[3])}


def mkv_set_oja_pair(enable: bool) -> bool:
    """Run the OjaKV contraction (n_query <= 128) on pairs of CTAs (tcgen05
    cta_group::2, 256 tokens per MMA) or on one CTA per SM; returns the
    previous setting."""
    return bool(load().mkv_set_oja_pair(1 if enable else 0))


def mkv_set_fused(scorer_ctas: int, select_ctas: int = 0) -> int:
    """When mkv_compress runs the fused whole-path kernel: scorer_ctas < 0 on
    its own shape rule (the default), > 0 wherever it applies with that scorer
    budget (select_ctas > 0 sets the selector CTAs), 0 never. Returns the
    previous scorer setting."""
    return int(load().mkv_set_fused(int(scorer_ctas), int(select_ctas)))


def mkv_layer_budgets(sensitivity, r: float, gamma: float, total: int, cap):
    """Per-layer kept-token budgets (host helper). Returns (status, budgets)
    with budgets an int32 list of one entry per layer; status 1 means the caps
    absorb the whole total."""
    import array
    sv = array.array("d", [float(x) for x in sensitivity])
    cp = array.array("i", [int(x) for x in cap])
    out = array.array("i", [0] * len(sv))
    if len(cp) != len(sv):
        raise ValueError("one cap per layer is required")
    st = load().mkv_layer_budgets(ctypes.c_void_p(sv.buffer_info()[0]), len(sv), float(r), float(gamma), int(total),
                                  ctypes.c_void_p(cp.buffer_info()[0]), ctypes.c_void_p(out.buffer_info()[0]))
    if st < 0:
        raise MKVError(MKV_ERR_INVALID_ARG, "mkv_layer_budgets")
    return int(st), list(out)


def workspace_for(K: torch.Tensor, window: int = 0, seq_lens=None) -> torch.Tensor:
    """A zeroed workspace (uint8, 256-byte aligned by the caching allocator)."""
    n = mkv_workspace_size(shape_of(K, seq_lens), window)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=K.device)


# -------------------------------------------------------------- entry points --

def mkv_centroid(K, window, C, workspace, seq_lens=None, stream=None):
    _need_cuda(K, C, workspace, seq_lens)
    _check(load().mkv_centroid(_ptr(K), shape_of(K, seq_lens), int(window), _ptr(C), _ptr(workspace),
                               workspace.numel(), _stream(stream)), "mkv_centroid")


def mkv_window_means(X, window, mean, workspace, radius=None, seq_lens=None, stream=None):
    """Cluster summaries of a bf16 cache X (keys or values): fp32 window means
    [batch, heads, nw, 128] and, optionally, fp32 radii [batch, heads, nw]."""
    _need_cuda(X, mean, radius, workspace, seq_lens)
    _check(load().mkv_window_means(_ptr(X), shape_of(X, seq_lens), int(window), _ptr(mean), _ptr(radius),
                                   _ptr(workspace), workspace.numel(), _stream(stream)), "mkv_window_means")


def mkv_centroid_score(K, window, mode, C, S, workspace, seq_lens=None, stream=None):
    """Steps a1 + a2 as mkv_compress runs them (C and S as mkv_centroid / mkv_score write them)."""
    _need_cuda(K, C, S, workspace, seq_lens)
    _check(load().mkv_centroid_score(_ptr(K), shape_of(K, seq_lens), int(window), _MODES[mode], _ptr(C), _ptr(S),
                                     _ptr(workspace), workspace.numel(), _stream(stream)), "mkv_centroid_score")


def mkv_score(K, C, window, mode, S, workspace, seq_lens=None, stream=None):
    _need_cuda(K, C, S, workspace, seq_lens)
    _check(load().mkv_score(_ptr(K), _ptr(C), shape_of(K, seq_lens), int(window), _MODES[mode], _ptr(S),
                            _ptr(workspace), workspace.numel(), _stream(stream)), "mkv_score")


def mkv_select_topk(S, shape: MkvShape, ratio, cut, workspace, n_keep=None, stream=None):
    _need_cuda(S, cut, workspace, n_keep)
    _check(load().mkv_select_topk(_ptr(S), shape, float(ratio), _ptr(n_keep), _ptr(cut), _ptr(workspace),
                                  workspace.numel(), _stream(stream)), "mkv_select_topk")


def mkv_compact(S, cut, K, V, shape: MkvShape, ratio, keep_stride, idx, kept, K_out, V_out, workspace,
                n_keep=None, stream=None):
    _need_cuda(S, cut, K, V, idx, kept, K_out, V_out, workspace, n_keep)
    _cache_types(K, V, K_out, V_out)
    _check(load().mkv_compact(_ptr(S), _ptr(cut), _ptr(K), _ptr(V), shape, float(ratio), _ptr(n_keep),
                              int(keep_stride), _ptr(idx), _ptr(kept), _ptr(K_out), _ptr(V_out), _ptr(workspace),
                              workspace.numel(), _stream(stream)), "mkv_compact")


def mkv_compress(K, V, ratio, mode, window, keep_stride, K_out, V_out, idx, kept, workspace, seq_lens=None,
                 n_keep=None, stream=None):
    _need_cuda(K, V, K_out, V_out, idx, kept, workspace, seq_lens, n_keep)
    _cache_types(K, V, K_out, V_out)
    _check(load().mkv_compress(_ptr(K), _ptr(V), shape_of(K, seq_lens), float(ratio), _ptr(n_keep), _MODES[mode],
                               int(window), int(keep_stride), _ptr(K_out), _ptr(V_out), _ptr(idx), _ptr(kept),
                               _ptr(workspace), workspace.numel(), _stream(stream)), "mkv_compress")


def mkv_num_keep_quota(T: int, ratio: float, window: int) -> int:
    return int(load().mkv_num_keep_quota(int(T), float(ratio), int(window)))


def mkv_select_quota(S, shape: MkvShape, ratio, window, keep_stride, idx, kept, workspace, stream=None):
    _need_cuda(S, idx, kept, workspace)
    _check(load().mkv_select_quota(_ptr(S), shape, float(ratio), int(window), int(keep_stride), _ptr(idx),
                                   _ptr(kept), _ptr(workspace), workspace.numel(), _stream(stream)),
           "mkv_select_quota")


def mkv_compress_quota(K, V, ratio, mode, window, keep_stride, K_out, V_out, idx, kept, workspace, seq_lens=None,
                       stream=None):
    _need_cuda(K, V, K_out, V_out, idx, kept, workspace, seq_lens)
    _cache_types(K, V, K_out, V_out)
    _check(load().mkv_compress_quota(_ptr(K), _ptr(V), shape_of(K, seq_lens), float(ratio), _MODES[mode],
                                     int(window), int(keep_stride), _ptr(K_out), _ptr(V_out), _ptr(idx),
                                     _ptr(kept), _ptr(workspace), workspace.numel(), _stream(stream)),
           "mkv_compress_quota")


def mkv_oja_workspace_size(shape: MkvShape, n_query: int) -> int:
    return int(load().mkv_oja_workspace_size(shape, int(n_query)))


def oja_workspace_for(K: torch.Tensor, n_query: int, seq_lens=None) -> torch.Tensor:
    n = mkv_oja_workspace_size(shape_of(K, seq_lens), n_query)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=K.device)


def mkv_oja_score(K, Q, U, S, workspace, seq_lens=None, stream=None):
    """OjaKV-style reconstruction-error scores: K [B, H, T, 128] bf16,
    Q [B, H, n_query, 128] bf16, U [B, H, 128, rank] fp32 -> S [B, H, T]."""
    _need_cuda(K, Q, U, S, workspace, seq_lens)
    _check(load().mkv_oja_score(_ptr(K), _ptr(Q), _ptr(U), shape_of(K, seq_lens), int(Q.shape[-2]),
                                int(U.shape[-1]), _ptr(S), _ptr(workspace), workspace.numel(), _stream(stream)),
           "mkv_oja_score")


def mkv_oja_score_profiled(K, Q, U, S, workspace, events, seq_lens=None, stream=None):
    """mkv_oja_score with three torch.cuda.Event objects recorded around its
    two kernels (query projection, contraction)."""
    _need_cuda(K, Q, U, S, workspace, seq_lens)
    s = torch.cuda.current_stream() if stream is None else stream
    for e in events:
        e.record(s)  # creates the event handles lazily; re-recorded below
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(load().mkv_oja_score_profiled(_ptr(K), _ptr(Q), _ptr(U), shape_of(K, seq_lens), int(Q.shape[-2]),
                                         int(U.shape[-1]), _ptr(S), _ptr(workspace), workspace.numel(),
                                         _stream(s), arr, len(events)), "mkv_oja_score_profiled")


def mkv_compress_oja(K, V, Q, U, ratio, keep_stride, K_out, V_out, idx, kept, workspace, seq_lens=None, n_keep=None,
                     stream=None):
    _need_cuda(K, V, Q, U, K_out, V_out, idx, kept, workspace, seq_lens, n_keep)
    _check(load().mkv_compress_oja(_ptr(K), _ptr(V), _ptr(Q), _ptr(U), shape_of(K, seq_lens), int(Q.shape[-2]),
                                   int(U.shape[-1]), float(ratio), _ptr(n_keep), int(keep_stride), _ptr(K_out),
                                   _ptr(V_out), _ptr(idx), _ptr(kept), _ptr(workspace), workspace.numel(),
                                   _stream(stream)), "mkv_compress_oja")


def mkv_compress_inplace(K, V, ratio, mode, window, workspace, idx=None, kept=None, seq_lens=None, n_keep=None,
                         stream=None):
    """Compress K and V in place: rows [0, kept) of every head become the
    kept rows; idx [B, H, t_max] and kept [B, H] are optional outputs."""
    _need_cuda(K, V, idx, kept, workspace, seq_lens, n_keep)
    _cache_types(K, V)
    _check(load().mkv_compress_inplace(_ptr(K), _ptr(V), shape_of(K, seq_lens), float(ratio), _ptr(n_keep),
                                       _MODES[mode], int(window), _ptr(idx), _ptr(kept), _ptr(workspace),
                                       workspace.numel(), _stream(stream)), "mkv_compress_inplace")


def mkv_compress_profiled(K, V, ratio, mode, window, keep_stride, K_out, V_out, idx, kept, workspace, events,
                          seq_lens=None, n_keep=None, stream=None):
    """mkv_compress with torch.cuda.Event objects recorded around each kernel."""
    _need_cuda(K, V, K_out, V_out, idx, kept, workspace, seq_lens, n_keep)
    _cache_types(K, V, K_out, V_out)
    st = torch.cuda.current_stream() if stream is None else stream
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on its first record
            e.record(st)
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(load().mkv_compress_profiled(_ptr(K), _ptr(V), shape_of(K, seq_lens), float(ratio), _ptr(n_keep),
                                        _MODES[mode], int(window), int(keep_stride), _ptr(K_out), _ptr(V_out),
                                        _ptr(idx), _ptr(kept), _ptr(workspace), workspace.numel(), _stream(stream),
                                        arr, len(events)), "mkv_compress_profiled")


def mkv_compress_host(hK, hV, dK, dV, ratio, mode, window, keep_stride, dK_out, dV_out, d_idx, d_kept,
                      hK_out, hV_out, h_idx, h_kept, workspace, seq_lens=None, stream=None):
    """Host-resident cache: H2D copies, compress and D2H copies in one call."""
    _need_cuda(dK, dV, dK_out, dV_out, d_idx, d_kept, workspace, seq_lens)
    _cache_types(hK, hV, dK, dV, dK_out, dV_out, hK_out, hV_out)
    for t in (hK, hV, hK_out, hV_out, h_idx, h_kept):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("host buffers must be contiguous CPU tensors (pinned for asynchrony)")
    _check(load().mkv_compress_host(_ptr(hK), _ptr(hV), _ptr(dK), _ptr(dV), shape_of(dK, seq_lens), float(ratio),
                                    _MODES[mode], int(window), int(keep_stride), _ptr(dK_out), _ptr(dV_out),
                                    _ptr(d_idx), _ptr(d_kept), _ptr(hK_out), _ptr(hV_out), _ptr(h_idx),
                                    _ptr(h_kept), _ptr(workspace), workspace.numel(), _stream(stream)),
           "mkv_compress_host")


def mkv_compress_noalloc(K, V, ratio, mode, window, keep_stride, K_out, V_out, idx, kept, status_out=None,
                         seq_lens=None, n_keep=None, stream=None):
    """mkv_compress without a workspace, for callers that cannot allocate
    device memory: the library uses its own fixed 32 MiB scratch array, so
    problems needing more scratch than that raise MKV_ERR_UNSUPPORTED, and
    calls must not overlap on the GPU. ``status_out`` (int32/uint32 [1] on
    the device, optional) receives the call's device status bits."""
    _need_cuda(K, V, K_out, V_out, idx, kept, status_out, seq_lens, n_keep)
    _cache_types(K, V, K_out, V_out)
    _check(load().mkv_compress_noalloc(_ptr(K), _ptr(V), shape_of(K, seq_lens), float(ratio), _ptr(n_keep),
                                       _MODES[mode], int(window), int(keep_stride), _ptr(K_out), _ptr(V_out),
                                       _ptr(idx), _ptr(kept), _ptr(status_out), _stream(stream)),
           "mkv_compress_noalloc")


def mkv_inject_stalled_windows(K, V, ratio, mode, window, keep_stride, K_out, V_out, idx, kept, workspace,
                               seq_lens=None, stream=None):
    """Failure injection: the single-pass kernel with no window ever
    completing; every wait between CTAs must run out (MKV_DEV_TIMEOUT)."""
    _need_cuda(K, V, K_out, V_out, idx, kept, workspace, seq_lens)
    _cache_types(K, V, K_out, V_out)
    _check(load().mkv_inject_stalled_windows(_ptr(K), _ptr(V), shape_of(K, seq_lens), float(ratio), _MODES[mode],
                                             int(window), int(keep_stride), _ptr(K_out), _ptr(V_out), _ptr(idx),
                                             _ptr(kept), _ptr(workspace), workspace.numel(), _stream(stream)),
           "mkv_inject_stalled_windows")


def mkv_inject_stalled_fused(K, V, ratio, mode, keep_stride, K_out, V_out, idx, kept, stage, workspace,
                             seq_lens=None, stream=None):
    """Failure injection: the fused whole-path kernel with one wait that
    cannot end (stage 0: scorer group 0's barrier; stage 1: head 0's select);
    it must run out (MKV_DEV_TIMEOUT) and the rest of the launch drain."""
    _need_cuda(K, V, K_out, V_out, idx, kept, workspace, seq_lens)
    _cache_types(K, V, K_out, V_out)
    _check(load().mkv_inject_stalled_fused(_ptr(K), _ptr(V), shape_of(K, seq_lens), float(ratio), _MODES[mode],
                                           int(keep_stride), _ptr(K_out), _ptr(V_out), _ptr(idx), _ptr(kept),
                                           int(stage), _ptr(workspace), workspace.numel(), _stream(stream)),
           "mkv_inject_stalled_fused")


def mkv_device_status(workspace, stream=None) -> int:
    """Synchronise, return the status bits of ``workspace`` and clear them."""
    bits = ctypes.c_uint32(0)
    st = load().mkv_device_status(_ptr(workspace), _stream(stream), ctypes.byref(bits))
    if st not in (MKV_OK, MKV_ERR_DEVICE):
        raise MKVError(st, "mkv_device_status")
    return int(bits.value)


# ---------------------------------------------------------------- convenience --

def compress(K, V, ratio: float, mode="l2", window: int = 0, seq_lens=None, n_keep=None,
             keep_stride: Optional[int] = None, workspace=None, stream=None):
    """Compress a bf16 cache [batch, heads, t_max, 128]; returns
    (K_out, V_out, idx, kept) with K_out/V_out [batch, heads, keep_stride, 128]."""
    if keep_stride is None:
        keep_stride = mkv_num_keep(K.shape[2], ratio) if n_keep is None else int(n_keep.max().item())
    b, h = K.shape[0], K.shape[1]
    K_out = torch.empty((b, h, keep_stride, K.shape[3]), dtype=K.dtype, device=K.device)
    V_out = torch.empty_like(K_out)
    idx = torch.empty((b, h, keep_stride), dtype=torch.int32, device=K.device)
    kept = torch.empty((b, h), dtype=torch.int32, device=K.device)
    ws = workspace if workspace is not None else workspace_for(K, window, seq_lens)
    mkv_compress(K, V, ratio, mode, window, keep_stride, K_out, V_out, idx, kept, ws, seq_lens, n_keep, stream)
    return K_out, V_out, idx, kept
