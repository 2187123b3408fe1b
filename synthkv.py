"""Seeded synthetic key/value caches shaped like the models that ManifoldKV is
evaluated on (Llama-3.1-8B, Qwen3-8B and Phi-4 KV shapes, 4K-131K context).

This module is shared by the CUDA path's tests and bench and by the oracle's
tests. It draws random inputs only: it computes no centroid, no score, no
selection and no compaction, so it holds none of the method's arithmetic.

Key recipe for one head (a (layer, sequence, KV-head) triple) of T rows:

* z_t ~ N(0, I_d);
* ``outlier_channels`` channel indices (drawn per head) of z are multiplied
  by ``outlier_scale`` (the heavy channels that real keys show);
* a per-token magnitude s_t ~ LogNormal(0, sigma);
* ``planted`` token positions (drawn per head without replacement) get
  s_t := ``planted_norm`` (4x the median token magnitude);
* a slowly drifting mean: mu_0 = 0 and mu_{j+1} = mu_j + N(0, drift_std^2 I)
  at every ``drift_every`` tokens;
* k_t = s_t * z_t + mu_{t // drift_every};
* values v_t ~ N(0, I_d);
* both are rounded to bfloat16 (round to nearest even, by torch).

Rows at or beyond a ragged sequence's length are filled with ``pad_value`` so
that any kernel that reads past a sequence's end visibly changes its result.

The cache layout is [L*B, H, T_max, d]: layers are folded into the batch
dimension, layer-major (row index l*B + b), and every layer of sequence b has
the same length T_b.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class KVWorkload:
    """One synthetic workload: the cache shape, the key distribution and the
    compression settings that run on it."""

    name: str
    layers: int
    batch: int
    heads: int
    t_max: int
    head_dim: int = 128
    t_min: Optional[int] = None          # ragged: T_b ~ U{t_min..t_max} per sequence
    sigma: float = 0.5                   # lognormal token-magnitude spread
    outlier_channels: int = 0
    outlier_scale: float = 10.0
    planted: int = 0                     # planted outlier tokens per head
    planted_norm: float = 4.0
    drift_every: int = 0                 # 0 = no mean drift
    drift_std: float = 0.25
    runs: tuple = ()                     # ((mode, window, ratio), ...): mode in {"l2", "cosine"}, window 0 = global
    model: str = ""                      # the model whose KV shape this follows

    @property
    def rows(self) -> int:
        """Number of (layer, sequence) rows of the cache: L*B."""
        return self.layers * self.batch

    @property
    def n_heads(self) -> int:
        """Number of independent heads: L*B*H."""
        return self.layers * self.batch * self.heads

    def scaled(self, name: str, **changes) -> "KVWorkload":
        """A copy with some fields replaced (used for CI-sized variants)."""
        return dataclasses.replace(self, name=name, **changes)


# The five workloads: shapes and key distributions follow the model KV shapes
# the ManifoldKV abstract evaluates on (Llama-3.1-8B, Qwen3-8B, Phi-4) at the
# context lengths it reports (4K-131K), with the compression levels it reports.
WORKLOADS = {
    "single-layer-h8-t4096": KVWorkload(
        name="single-layer-h8-t4096", layers=1, batch=1, heads=8, t_max=4096,
        sigma=0.5, planted=16, runs=(("l2", 0, 0.2),), model=""),
    "llama3.1-8b-kv-t16k": KVWorkload(
        name="llama3.1-8b-kv-t16k", layers=32, batch=1, heads=8, t_max=16384,
        sigma=0.5, outlier_channels=4, runs=(("l2", 0, 0.5),), model="Llama-3.1-8B"),
    "qwen3-8b-kv-t64k-w4096": KVWorkload(
        name="qwen3-8b-kv-t64k-w4096", layers=36, batch=1, heads=8, t_max=65536,
        sigma=0.5, outlier_channels=4, drift_every=8192,
        runs=(("l2", 4096, 0.25),), model="Qwen3-8B"),
    "ragged-b8-llama-kv-t8k-32k": KVWorkload(
        name="ragged-b8-llama-kv-t8k-32k", layers=32, batch=8, heads=8,
        t_max=32768, t_min=8192, sigma=0.5, planted=32,
        runs=(("l2", 0, 0.2), ("l2", 0, 0.5), ("cosine", 0, 0.2), ("cosine", 0, 0.5)), model="Llama-3.1-8B"),
    "phi4-kv-t128k": KVWorkload(
        name="phi4-kv-t128k", layers=40, batch=1, heads=10, t_max=131072,
        sigma=0.7, outlier_channels=4, drift_every=16384,
        runs=(("l2", 8192, 0.5), ("l2", 0, 0.5), ("cosine", 0, 0.5)), model="Phi-4"),
}

# The workload whose throughput the bench reports by default: the largest
# one, Phi-4-shaped at 131072 tokens (where the windowed centroids matter).
BENCH_WORKLOAD = "phi4-kv-t128k"
# The workload the widened paths (OjaKV, summaries, in-place) run on by default.
SECONDARY_WORKLOAD = "llama3.1-8b-kv-t16k"


def describe(w: KVWorkload) -> str:
    """One line naming the workload's shape and key distribution."""
    T = f"T={w.t_max}" if w.t_min is None else f"T~U{{{w.t_min}..{w.t_max}}} per sequence"
    parts = [f"N(0,1) keys", f"lognormal(0,{w.sigma}) token norms"]
    if w.outlier_channels:
        parts.append(f"{w.outlier_channels} outlier channels x{w.outlier_scale:g}")
    if w.planted:
        parts.append(f"{w.planted} planted tokens per head at norm {w.planted_norm:g}")
    if w.drift_every:
        parts.append(f"mean drift every {w.drift_every} tokens")
    shape = f"{w.layers} layers x {w.batch} seq x {w.heads} KV heads, d={w.head_dim}, {T}"
    kind = f"{w.model}-shaped KV cache" if w.model else "KV cache"
    return f"synthetic (seeded; {kind}: {shape}; " + ", ".join(parts) + "; V ~ N(0,1))"


def _mix(seed: int, *keys: int) -> int:
    """Derive a 63-bit sub-seed from a seed and integer keys (splitmix64 finaliser)."""
    x = (seed * 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
    for k in keys:
        x = (x ^ ((k + 0x632BE59BD9B4E019) & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
        x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        x ^= x >> 30
        x = (x * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        x ^= x >> 27
        x = (x * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        x ^= x >> 31
    return x & 0x7FFFFFFFFFFFFFFF


def seq_lengths(w: KVWorkload, seed: int) -> torch.Tensor:
    """Per-(layer, sequence) lengths, int32 [L*B] on the CPU, layer-major.

    Uniform workloads give t_max everywhere; ragged ones draw T_b uniformly
    from {t_min..t_max} once per sequence and repeat it for every layer."""
    if w.t_min is None:
        return torch.full((w.rows,), w.t_max, dtype=torch.int32)
    g = torch.Generator().manual_seed(_mix(seed, 0x5EC))
    per_seq = torch.randint(w.t_min, w.t_max + 1, (w.batch,), generator=g, dtype=torch.int64)
    return per_seq.repeat(w.layers).to(torch.int32)


def _head_kv(w: KVWorkload, seed: int, head: int, t_len: int, device, pad_value: float):
    """Keys and values of one head as bf16 [t_max, d] plus planted positions."""
    d, T = w.head_dim, w.t_max
    g = torch.Generator(device=device).manual_seed(_mix(seed, head))
    z = torch.randn(T, d, generator=g, device=device, dtype=torch.float32)
    if w.outlier_channels:
        ch = torch.randperm(d, generator=g, device=device)[: w.outlier_channels]
        z[:, ch] *= w.outlier_scale
    s = torch.exp(w.sigma * torch.randn(T, generator=g, device=device, dtype=torch.float32))
    planted = torch.empty(0, dtype=torch.int64, device=device)
    if w.planted and t_len > 0:
        planted = torch.randperm(t_len, generator=g, device=device)[: min(w.planted, t_len)]
        s[planted] = w.planted_norm
    k = s[:, None] * z
    if w.drift_every:
        n_seg = (T + w.drift_every - 1) // w.drift_every
        steps = w.drift_std * torch.randn(n_seg, d, generator=g, device=device, dtype=torch.float32)
        steps[0].zero_()
        mu = torch.cumsum(steps, dim=0)
        seg = torch.arange(T, device=device) // w.drift_every
        k += mu[seg]
    v = torch.randn(T, d, generator=g, device=device, dtype=torch.float32)
    if t_len < T:
        k[t_len:] = pad_value
        v[t_len:] = pad_value
    return k.to(torch.bfloat16), v.to(torch.bfloat16), torch.sort(planted).values


# Largest finite magnitude of float8_e4m3fn; torch's cast turns anything
# beyond it into NaN, so fp8 caches are clamped to it first.
E4M3_MAX = 448.0


def make_kv(w: KVWorkload, seed: int = 0, device="cpu", pad_value: float = 300.0,
            heads: Optional[Sequence[int]] = None, with_planted: bool = False, dtype=torch.bfloat16):
    """Generate the cache of a workload.

    Returns (K, V, seq_lens) with K, V [L*B, H, t_max, d] on ``device`` and
    seq_lens int32 [L*B] on ``device``. K and V are bf16, or, with ``dtype``
    torch.float8_e4m3fn, the same values clamped to +-448 and rounded to
    E4M3 by torch's cast. With ``heads`` (flat head indices in [0, L*B*H)),
    only those heads are generated and K, V have shape [len(heads), t_max,
    d]; each head's data does not depend on which other heads are generated.
    With ``with_planted`` a list of the planted token positions per
    generated head is returned as a fourth element."""
    lens = seq_lengths(w, seed)
    ids = list(range(w.n_heads)) if heads is None else list(heads)
    fp8 = dtype == torch.float8_e4m3fn
    if dtype not in (torch.bfloat16, torch.float8_e4m3fn):
        raise ValueError(f"unsupported cache dtype {dtype}")
    K = torch.empty((len(ids), w.t_max, w.head_dim), dtype=dtype, device=device)
    V = torch.empty_like(K)
    planted = []
    for j, h in enumerate(ids):
        t_len = int(lens[h // w.heads])
        k, v, p = _head_kv(w, seed, h, t_len, device, pad_value)
        if fp8:
            k = k.float().clamp(-E4M3_MAX, E4M3_MAX)
            v = v.float().clamp(-E4M3_MAX, E4M3_MAX)
        K[j].copy_(k)
        V[j].copy_(v)
        planted.append(p.cpu())
    if heads is None:
        K = K.view(w.rows, w.heads, w.t_max, w.head_dim)
        V = V.view(w.rows, w.heads, w.t_max, w.head_dim)
    out = (K, V, lens.to(device))
    return out + (planted,) if with_planted else out


def random_scores(n_heads: int, t: int, seed: int, tie_fraction: float = 0.0,
                  levels: int = 0, device="cpu") -> torch.Tensor:
    """Seeded fp32 score rows [n_heads, t] for exercising selection alone.

    Scores are nonnegative, as distances and 1 - cos are. ``levels`` > 0 draws
    from that many distinct values only (heavy ties); ``tie_fraction`` copies
    one value onto that fraction of each row."""
    g = torch.Generator(device=device).manual_seed(_mix(seed, 0x5C0))
    if levels:
        s = torch.randint(0, levels, (n_heads, t), generator=g, device=device).to(torch.float32) * 0.125
    else:
        s = torch.exp(torch.randn(n_heads, t, generator=g, device=device, dtype=torch.float32)) * 8.0
    if tie_fraction > 0 and t > 0:
        n = max(1, int(math.floor(tie_fraction * t)))
        for h in range(n_heads):
            pos = torch.randperm(t, generator=g, device=device)[:n]
            s[h, pos] = float(s[h, pos[0]].item())
    return s


def make_oja_inputs(w: KVWorkload, seed: int, n_query: int, rank: int, device="cpu",
                    heads: Optional[Sequence[int]] = None, query_scale: float = 1.0):
    """Query windows and low-rank bases for the OjaKV-style scorer.

    Returns (Q, U): Q bf16 [L*B, H, n_query, d] (the recent query rows of the
    query heads that read each KV head, N(0, query_scale^2)), and U fp32
    [L*B, H, d, rank] with orthonormal columns (a QR factor of a Gaussian
    matrix, drawn on the CPU so both sides see the same basis). With
    ``heads``, only those flat heads: [len(heads), n_query, d] and
    [len(heads), d, rank]."""
    ids = list(range(w.n_heads)) if heads is None else list(heads)
    d = w.head_dim
    Q = torch.empty((len(ids), n_query, d), dtype=torch.bfloat16, device=device)
    U = torch.empty((len(ids), d, rank), dtype=torch.float32)
    for j, h in enumerate(ids):
        g = torch.Generator(device=device).manual_seed(_mix(seed, 0x0A, h))
        Q[j].copy_((query_scale * torch.randn(n_query, d, generator=g, device=device)).to(torch.bfloat16))
        if rank:
            gc = torch.Generator().manual_seed(_mix(seed, 0x0B, h))
            a = torch.randn(d, rank, generator=gc, dtype=torch.float64)
            U[j].copy_(torch.linalg.qr(a).Q.to(torch.float32))
    U = U.to(device)
    if heads is None:
        Q = Q.view(w.rows, w.heads, n_query, d)
        U = U.view(w.rows, w.heads, d, rank)
    return Q, U
