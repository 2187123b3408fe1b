"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding and compare it head by head with the fp64 oracle.

Tolerances (the scorer's stated bar, 1e-5 relative, made precise per mode):
* L2 scores: |s_gpu - s_oracle| <= 1e-5 * |s_oracle| (fp32 against fp64);
* cosine scores s = 1 - q with q = k.c/(|k||c|): the fp32 rounding errors
  of q and of the subtraction are relative to |q| as well as to |s|, so the
  bound is 1e-5 * (|s_oracle| + |1 - s_oracle|); as s -> 0 (a key parallel to
  its centroid) a pure relative bound on s would demand more than fp32 holds;
  scores that meet this bound but not the plain 1e-5 * |s_oracle| are
  counted per test ("cosine_relaxed") and reported beside the near-cut
  exceptions;
* kept indices: exact, except tokens whose oracle score lies within 1e-5
  (relative) of the oracle's cut score; such tokens are counted and reported;
* kept count: exactly n_keep; compacted K and V rows: bit-exact copies of the
  input rows at the GPU's own kept indices;
* the GPU's selection is also checked against its own fp32 scores: it must be
  exactly the top n_keep by (score desc, index asc) -- there the decision is
  taken in one precision on both sides, so no exception is allowed.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import geometric_kv_cache_gb300 as mkv
import oracle

SCORE_RTOL = 1e-5
CUT_RTOL = 1e-5

_REPORT = os.environ.get("MKV_PARITY_REPORT")

# Tallies of every compare_head call, per (test, score mode): heads and
# scores compared, near-cut exceptions and cosine scores that needed the
# relaxed bound. tests/conftest.py prints and saves them at the end of the
# session; `current_test` is set per test by its autouse fixture.
TALLY: dict = {}
current_test = "?"
CASES: list = []


def _tally(mode: str, **counts):
    rec = TALLY.setdefault((current_test, mode), {"test": current_test, "mode": mode, "heads": 0, "scores": 0,
                                                  "near_cut_exceptions": 0, "cosine_relaxed": 0})
    for k, v in counts.items():
        rec[k] += int(v)


def report(name: str, **fields):
    """Record one named case (kept for the session summary); also append it
    as a JSON line to $MKV_PARITY_REPORT when that is set."""
    CASES.append({"case": name, **fields})
    if not _REPORT:
        return
    os.makedirs(os.path.dirname(os.path.abspath(_REPORT)), exist_ok=True)
    with open(_REPORT, "a") as f:
        f.write(json.dumps({"case": name, **fields}) + "\n")


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw element bits: uint16 for bf16, the uint8 codes for float8_e4m3fn."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def score_tol(S: np.ndarray, mode: str) -> np.ndarray:
    """Allowed |s_gpu - s_oracle| for oracle scores S."""
    S = np.asarray(S, dtype=np.float64)
    if mode == "cosine":
        return SCORE_RTOL * (np.abs(S) + np.abs(1.0 - S))
    return SCORE_RTOL * np.maximum(np.abs(S), 1e-30)


def gpu_topk_consistent(S_gpu: np.ndarray, idx: np.ndarray, n_keep: int) -> bool:
    """Is idx exactly the top n_keep of the fp32 scores by (desc, lower index)?"""
    T = S_gpu.shape[0]
    order = np.lexsort((np.arange(T), -S_gpu.astype(np.float64)))
    return np.array_equal(np.sort(order[:n_keep]), idx)


def compare_head(ora: dict, T: int, S_gpu=None, idx_gpu=None, kept_gpu=None, K_head=None, V_head=None,
                 Kout_gpu=None, Vout_gpu=None, C_gpu=None, key_scale=None, mode="l2") -> dict:
    """Compare one head; raises AssertionError on a parity failure and returns
    the counters (near-cut exceptions etc.)."""
    out = {"T": T, "near_cut_exceptions": 0, "cosine_relaxed": 0}
    S_o = ora["S"]
    n_keep = len(ora["idx"])
    if C_gpu is not None:
        C_o = ora["C"]
        scale = key_scale if key_scale is not None else max(1e-30, float(np.abs(C_o).max()))
        err = float(np.abs(C_gpu.astype(np.float64) - C_o).max()) if C_o.size else 0.0
        out["centroid_max_abs_err"] = err
        assert err <= 1e-5 * scale, f"centroid error {err} above 1e-5 * {scale}"
    if S_gpu is not None and T:
        s = S_gpu[:T].astype(np.float64)
        tol = score_tol(S_o, mode)
        err = np.abs(s - S_o)
        bad = err > tol
        out["score_max_err_over_tol"] = float(np.max(err / tol))
        assert not bad.any(), (f"{int(bad.sum())} scores outside the tolerance (max error/tol "
                               f"{out['score_max_err_over_tol']})")
        if mode == "cosine":  # within the cosine bound but not the plain relative one
            out["cosine_relaxed"] = int(np.count_nonzero(err > SCORE_RTOL * np.maximum(np.abs(S_o), 1e-30)))
    if kept_gpu is not None:
        assert int(kept_gpu) == n_keep, f"kept {int(kept_gpu)} != n_keep {n_keep}"
    if idx_gpu is not None:
        g = np.asarray(idx_gpu[:n_keep], dtype=np.int64)
        assert np.all(np.diff(g) > 0), "GPU indices are not strictly ascending"
        assert g.size == 0 or (g[0] >= 0 and g[-1] < T), "GPU index out of range"
        o = ora["idx"].astype(np.int64)
        diff = np.setxor1d(g, o)
        near = 0
        if diff.size:
            cut = np.sort(S_o)[::-1][n_keep - 1]
            near_mask = np.abs(S_o[diff] - cut) <= score_tol(np.array([cut]), mode)[0] * (CUT_RTOL / SCORE_RTOL)
            near = int(diff.size)
            assert near_mask.all(), (f"{int((~near_mask).sum())} kept-set differences away from the cut "
                                     f"(cut {cut}, scores {S_o[diff[~near_mask]][:8]})")
        out["near_cut_exceptions"] = near
        if S_gpu is not None:
            assert gpu_topk_consistent(S_gpu[:T], g, n_keep), "GPU selection is not the top-n_keep of its own scores"
        if Kout_gpu is not None:
            kb, vb = bits(K_head)[:T], bits(V_head)[:T]
            assert np.array_equal(Kout_gpu[:n_keep], kb[g]), "gathered K rows differ from K[idx]"
            assert np.array_equal(Vout_gpu[:n_keep], vb[g]), "gathered V rows differ from V[idx]"
            if near == 0:
                assert np.array_equal(Kout_gpu[:n_keep], ora["K_out"]), "compacted K differs from the oracle's"
                assert np.array_equal(Vout_gpu[:n_keep], ora["V_out"]), "compacted V differs from the oracle's"
    _tally(mode, heads=1, scores=T if S_gpu is not None else 0, near_cut_exceptions=out["near_cut_exceptions"],
           cosine_relaxed=out["cosine_relaxed"])
    return out


class StepBuffers:
    """Device buffers of the step-wise API for a cache K [B, H, T, D] (bf16 or E4M3)."""

    def __init__(self, K, window, ratio, seq_lens=None, keep_stride=None):
        B, H, T, D = K.shape
        dev = K.device
        self.shape = mkv.shape_of(K, seq_lens)
        self.nw = max(mkv.mkv_num_windows(T, window), 1)
        self.C = torch.zeros((B, H, self.nw, D), dtype=torch.float32, device=dev)
        self.S = torch.zeros((B, H, T), dtype=torch.float32, device=dev)
        self.cut = torch.zeros((B * H, 2), dtype=torch.int32, device=dev)
        self.keep_stride = mkv.mkv_num_keep(T, ratio) if keep_stride is None else keep_stride
        self.idx = torch.full((B, H, max(self.keep_stride, 1)), -7, dtype=torch.int32, device=dev)
        self.kept = torch.full((B, H), -7, dtype=torch.int32, device=dev)
        self.K_out = torch.zeros((B, H, max(self.keep_stride, 1), D), dtype=K.dtype, device=dev)
        self.V_out = torch.zeros_like(self.K_out)
        self.ws = mkv.workspace_for(K, window, seq_lens)


def oracle_heads(K, V, lens_per_row, heads_per_row, head_ids, ratio, mode, window):
    """Run the oracle on the listed flat heads of a [B, H, T, D] cache."""
    Kf = K.reshape(-1, K.shape[2], K.shape[3])
    Vf = V.reshape(-1, V.shape[2], V.shape[3])
    res = {}
    for h in head_ids:
        T = int(lens_per_row[h // heads_per_row])
        res[h] = oracle.compress_head(Kf[h, :T].cpu(), Vf[h, :T].cpu(), ratio, mode, window)
    return res


def check_in_place_vs_oracle(K, V, Ki, Vi, kept_i, lens_per_row, ratio, mode, window, heads=None, idx_i=None):
    """In-place compaction against the oracle, head by head: the oracle
    selects on the head's own T_b tokens, then oracle.compact_in_place moves
    the kept rows of the head's whole t_max-row block, and the GPU's rows
    (K_i, V_i after mkv_compress_inplace on copies of K, V) must equal that
    bit for bit, the untouched tail included. Where a near-cut exception
    makes the GPU keep another set, the move is checked with the GPU's own
    indices (from idx_i, else the kept rows' positions are not known and the
    head is compared on the kept count only). Returns the near-cut count."""
    B, H, T, D = K.shape
    Kc, Vc = K.reshape(B * H, T, D).cpu(), V.reshape(B * H, T, D).cpu()
    Kic, Vic = bits(Ki.reshape(B * H, T, D)), bits(Vi.reshape(B * H, T, D))
    kept_c = kept_i.reshape(-1).cpu().numpy()
    idx_c = idx_i.reshape(B * H, -1).cpu().numpy() if idx_i is not None else None
    near = 0
    for h in (range(B * H) if heads is None else heads):
        Th = int(lens_per_row[h // H])
        ora = oracle.compress_head(Kc[h, :Th], Vc[h, :Th], ratio, mode, window)
        n = int(kept_c[h])
        res = compare_head(ora, Th, idx_gpu=None if idx_c is None else idx_c[h, :n], kept_gpu=n, mode=mode)
        use = ora["idx"]
        if res["near_cut_exceptions"]:
            near += res["near_cut_exceptions"]
            use = idx_c[h, :n]
        assert np.array_equal(Kic[h], oracle.compact_in_place(Kc[h], use)), f"head {h}: in-place K differs from the oracle's"
        assert np.array_equal(Vic[h], oracle.compact_in_place(Vc[h], use)), f"head {h}: in-place V differs from the oracle's"
    return near
