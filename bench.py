"""Throughput of the ManifoldKV-style compression path on GB300.

One step = one mkv_compress over the whole synthetic cache of the bench
workload: centroid, score, top-k select, compaction and K/V gather for every
head. By default that is the largest workload, Phi-4-shaped KV (40 layers x
10 KV heads, d=128, T=131072, bf16: 400 heads, 26.8 GB of K and V) with its
first run, WindowedManifoldKV (L2 distance to per-window centroids of 8192
tokens) at 50% compression. ``--workload`` and ``--run`` pick any workload
and any of its runs (mode, window, ratio); ``--mode``, ``--window`` and
``--ratio`` override single fields.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--run I] [--mode l2|cosine] [--window W] [--ratio R]

Prints one JSON line (rank 0). ``value`` is KV token rows (one per layer,
KV head and position) scored and compacted per second over all ranks, inputs
resident in HBM. ``e2e`` is the same metric through mkv_compress_host with
the cache in pinned host memory (H2D of K and V, compress, D2H of the
compacted cache, indices and counts inside the timed region). ``roofline`` is
for the kernel with the largest share of the step, timed with CUDA events on
the launching stream inside the real call. ``cpu_baseline`` is the fp64
oracle on the host cores on a sample of the same cache.

``--impl reference`` times the oracle (the only reference implementation of
this path) on the host cores on a sample of the same workload and prints the
same JSON line with ``"impl": "reference"``. Both CPU legs time the oracle
the same way (oracle_sample_rate): a step runs the sample's heads split into
one contiguous batch per host thread.

Under torchrun (N > 1) every rank compresses its own cache of the same shape
(heads are independent; no collective touches the data path); the step time
is the max over ranks and ``value`` counts all ranks' tokens.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthkv  # noqa: E402

METRIC = "KV tokens scored+compacted/sec and achieved HBM GB/s vs ~8 TB/s peak"
UNIT = "tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
CACHE_DTYPE_NAMES = ("bf16", "fp8")  # --dtype: bf16, or E4M3 codes (torch.float8_e4m3fn)
STAGES = ["piece_sums", "window_means", "piece_scores", "select", "compact", "gather"]


# ----------------------------------------------------------------- helpers --

def workload_run(name: str, layers: int = 0, run: int = 0, mode=None, window=None, ratio=None):
    """The workload and its run number ``run`` (mode, window, ratio), each
    field replaced when given; ``layers`` > 0 keeps the shape of each layer
    but changes the layer count (a smaller case for profiler captures)."""
    w = synthkv.WORKLOADS[name]
    if layers and layers != w.layers:
        w = w.scaled(f"{w.name}-{layers}layers", layers=layers)
    if not 0 <= run < len(w.runs):
        raise SystemExit(f"--run {run}: {w.name} has runs 0..{len(w.runs) - 1}: {list(w.runs)}")
    m, wd, r = w.runs[run]
    return w, (m if mode is None else mode), (wd if window is None else window), (r if ratio is None else ratio)


def keep_count(T: int, ratio: float) -> int:
    """Same rounding as the library's mkv_num_keep (used for byte counts only)."""
    import geometric_kv_cache_gb300 as mkv
    return mkv.mkv_num_keep(T, ratio)


def path_bytes(lens, heads: int, ratio: float, d: int = 128, k_reads: int = 2, es: int = 2) -> dict:
    """Algorithmic bytes of one step as the metric defines them: K read twice
    (centroid, score) plus the kept K and V rows read and written (es bytes
    per element: 2 for bf16, 1 for E4M3). Per kernel: the bytes each must
    move -- piece sums read K, scores read K and write 4 B per token, the
    gather reads and writes the kept K and V rows (with k_reads == 1, the
    single-pass kernel in stage 0 reads K once and writes the scores)."""
    tok = sum(int(t) for t in lens) * heads
    keep = sum(keep_count(int(t), ratio) for t in lens) * heads
    k_read = es * tok * d
    return {
        "tokens": tok,
        "kept": keep,
        "path": 2 * k_read + 4 * es * keep * d,
        "piece_sums": k_read + (4 * tok if k_reads == 1 else 0),
        "window_means": 0,
        "piece_scores": 0 if k_reads == 1 else k_read + 4 * tok,
        "select": 0,
        "compact": 0,
        "gather": 4 * es * keep * d,
    }


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.25)
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        if not self.lines:
            return None
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_seed(seed: int, rank: int) -> int:
    """Each rank compresses its own cache: seeds differ per rank."""
    return seed + 1000003 * rank


def max_over_ranks(x: float, group=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def sum_over_ranks(x: float, group=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


# ----------------------------------------------------------- CPU oracle leg --

def oracle_sample_rate(Kf, Vf, hl, ratio, mode, window, threads, steps=None, warmup=1, budget_s=None):
    """Time the oracle, as it stands, on one sample of heads: Kf, Vf [m, T, d]
    host tensors, hl their lengths. A step runs the m heads split into one
    contiguous batch per host thread (``threads`` at most; each batch is one
    call into the C oracle, which releases the interpreter lock) and waits
    for all of them. After ``warmup`` untimed steps it times ``steps`` steps,
    or, with ``budget_s``, steps until that much time has passed (at least 3).
    Returns (token rows per second over the mean step time, threads used,
    list of step seconds)."""
    import concurrent.futures as cf

    import numpy as np

    import oracle
    m = Kf.shape[0]
    hl = np.asarray(hl, dtype=np.int32)
    stride = keep_count(int(Kf.shape[1]), ratio)
    bounds = np.linspace(0, m, min(max(1, threads), m) + 1).astype(int)
    batches = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]

    def run(ab):
        a, b = ab
        oracle.compress_heads(Kf[a:b], Vf[a:b], hl[a:b], ratio, mode, window, stride)

    times = []
    with cf.ThreadPoolExecutor(max_workers=len(batches)) as pool:
        for _ in range(warmup):
            list(pool.map(run, batches))
        t_all = time.perf_counter()
        while True:
            t0 = time.perf_counter()
            list(pool.map(run, batches))
            times.append(time.perf_counter() - t0)
            if steps is not None and len(times) >= steps:
                break
            if steps is None and len(times) >= 3 and time.perf_counter() - t_all >= (budget_s or 0.0):
                break
    tok = int(hl.sum())
    return tok / (sum(times) / len(times)), len(batches), times


def oracle_sample_size(t_head_s: float, threads: int, target_step_s: float, n_heads: int) -> int:
    """Heads in a sample whose step (one batch per thread) takes about
    ``target_step_s``, given one head's single-thread time; a multiple of the
    thread count where the workload allows."""
    per = max(1, int(round(target_step_s / max(t_head_s, 1e-9))))
    return max(1, min(n_heads, per * threads))


def cpu_baseline_leg(K, V, lens_list, w, ratio, mode, window, budget_s):
    """The cpu_baseline object: the oracle, as it stands, on the host cores
    on a sample of the first heads of the same (device) cache, timed by
    oracle_sample_rate on every host thread, with the single-thread rate
    beside it. The sample is sized so that one step takes about half a
    second; a third of ``budget_s`` goes to the single-thread figure."""
    import numpy as np

    import oracle
    n, T, D = w.n_heads, K.shape[2], K.shape[3]
    Kd, Vd = K.reshape(n, T, D), V.reshape(n, T, D)
    hl_all = np.repeat(np.asarray(lens_list, dtype=np.int32), w.heads)
    nt = host_threads()
    K0, V0 = Kd[:1].cpu(), Vd[:1].cpu()
    t0 = time.perf_counter()
    oracle.compress_heads(K0, V0, hl_all[:1], ratio, mode, window, keep_count(T, ratio))
    t_head = max(time.perf_counter() - t0, 1e-6)
    m = oracle_sample_size(t_head, nt, 0.5, n)
    Kh, Vh = Kd[:m].cpu(), Vd[:m].cpu()
    m1 = max(1, min(m, int(round(0.5 / t_head))))
    tps1, _, times1 = oracle_sample_rate(Kh[:m1], Vh[:m1], hl_all[:m1], ratio, mode, window, 1, budget_s=budget_s / 3)
    tps, used, times = oracle_sample_rate(Kh, Vh, hl_all[:m], ratio, mode, window, nt, budget_s=2 * budget_s / 3)
    tok = int(hl_all[:m].sum())
    return {"value": tps, "unit": UNIT, "cores": used, "cpu_model": host_cpu_model(), "kind": "oracle",
            "sample": f"the first {m} of {n} heads ({tok} token rows) per step, split into {used} batches, one host "
                      f"thread each; {len(times)} steps of {statistics.mean(times):.3f} s (mean), fp64 C oracle",
            "single_thread": {"value": tps1, "cores": 1,
                              "sample": f"the first {m1} heads per step, {len(times1)} steps of "
                                        f"{statistics.mean(times1):.3f} s (mean)"}}


def host_cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def host_threads():
    """Host cores this process may use."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


# ------------------------------------------------------------------ our arm --

def run_ours(args):
    import torch
    import torch.distributed as dist

    import geometric_kv_cache_gb300 as mkv

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    mkv.load()
    if args.no_head_groups:
        mkv.mkv_set_head_groups(False)
    if args.ring is not None:
        mkv.mkv_set_head_group_ring(bool(args.ring))
    w, mode, window, ratio = workload_run(args.workload, args.layers, args.run, args.mode, args.window, args.ratio)
    cache_dtype = {"bf16": torch.bfloat16, "fp8": torch.float8_e4m3fn}[args.dtype]
    K, V, lens = synthkv.make_kv(w, seed=rank_seed(args.seed, rank), device=dev, dtype=cache_dtype)
    es = K.element_size()
    T = w.t_max
    ks = mkv.mkv_num_keep(T, ratio)
    K_out = torch.empty((w.rows, w.heads, ks, w.head_dim), dtype=cache_dtype, device=dev)
    V_out = torch.empty_like(K_out)
    idx = torch.empty((w.rows, w.heads, ks), dtype=torch.int32, device=dev)
    kept = torch.empty((w.rows, w.heads), dtype=torch.int32, device=dev)
    ws = mkv.workspace_for(K, window, lens)
    stream = torch.cuda.current_stream(dev)
    lens_list = lens.cpu().tolist()
    if args.fused is not None:
        mkv.mkv_set_fused(args.fused, args.fused_selectors)
    single = mkv.mkv_compress_single_pass(mkv.shape_of(K, lens), window, mode)
    hg_plan = mkv.mkv_head_group_plan(mkv.shape_of(K, lens), window, mode)
    if args.fused is not None and args.fused > 0 and single != 3:
        raise SystemExit("--fused: the fused kernel does not apply to this workload (global centroids, t <= 20480)")
    select_emits = T <= 40960  # select writes the kept indices itself (no compaction kernel)
    nbytes = path_bytes(lens_list, w.heads, ratio, w.head_dim, k_reads=1 if single in (1, 2, 3, 4) else 2, es=es)

    def step():
        mkv.mkv_compress(K, V, ratio, mode, window, ks, K_out, V_out, idx, kept, ws, lens, stream=stream)

    # warm-up, then a correctness guard on the status word
    for _ in range(max(args.warmup, 3)):
        step()
    if mkv.mkv_device_status(ws, stream) != 0:
        raise RuntimeError("device status nonzero after warm-up")

    # main timed region: exactly K steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    ms_local = ev0.elapsed_time(ev1) / args.steps
    ms = max_over_ranks(ms_local)
    tokens_all = sum_over_ranks(float(nbytes["tokens"]))
    value = tokens_all / (ms / 1e3)

    # per-kernel durations inside the real call (events on the launching stream);
    # the profiled call runs the separate kernels, so with --fused the one
    # kernel's time is the step's (one launch after a counter reset)
    ns = mkv.mkv_compress_num_stages()
    prof_steps = max(10, min(args.steps, 200))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(ns + 1)] for _ in range(prof_steps)]
    torch.cuda.synchronize(dev)
    for i in range(prof_steps):
        mkv.mkv_compress_profiled(K, V, ratio, mode, window, ks, K_out, V_out, idx, kept, ws, evs[i], lens,
                                  stream=stream)
    torch.cuda.synchronize(dev)
    stage_ms = [sum(e[j].elapsed_time(e[j + 1]) for e in evs) / prof_steps for j in range(ns)]
    # the dominant kernel among those that move the metric's bytes
    dom = max((j for j in range(ns) if nbytes[STAGES[j]] > 0), key=lambda j: stage_ms[j])
    peaks = measured_peaks()
    dom_name = STAGES[dom]
    dom_bytes, dom_ms = nbytes[dom_name], stage_ms[dom]
    if single == 3:  # the one kernel moves K once, writes the scores, and gathers
        dom_name, dom_bytes, dom_ms = "fused_path", nbytes["piece_sums"] + nbytes["gather"], ms_local
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    traffic = args.traffic.get(dom_name) if args.traffic else None

    # end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e:
        hK = K.cpu().pin_memory()
        hV = V.cpu().pin_memory()
        hKo = torch.empty(K_out.shape, dtype=cache_dtype).pin_memory()
        hVo = torch.empty_like(hKo).pin_memory()
        hidx = torch.empty(idx.shape, dtype=torch.int32).pin_memory()
        hkept = torch.empty(kept.shape, dtype=torch.int32).pin_memory()
        dK, dV = torch.empty_like(K), torch.empty_like(V)

        def e2e_step():
            mkv.mkv_compress_host(hK, hV, dK, dV, ratio, mode, window, ks, K_out, V_out, idx, kept, hKo, hVo, hidx,
                                  hkept, ws, lens, stream=stream)
        for _ in range(2):
            e2e_step()
        e2e_steps = max(3, min(args.steps, args.e2e_steps))
        barrier()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_ms = max_over_ranks(ev0.elapsed_time(ev1) / e2e_steps)
        # keys cross the link in full; values only for the kept rows (the
        # gather reads them from the pinned host buffer)
        h2d = hK.numel() * es + nbytes["kept"] * w.head_dim * es
        d2h = hKo.numel() * es + hVo.numel() * es + hidx.numel() * 4 + hkept.numel() * 4
        e2e = {"value": tokens_all / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps}
        if mkv.mkv_device_status(ws, stream) != 0:
            raise RuntimeError("device status nonzero after the e2e steps")

    # CPU baseline: the oracle on a bounded sample of the same cache (rank 0, N=1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(K, V, lens_list, w, ratio, mode, window, args.cpu_budget)

    hbm_gbs = nbytes["path"] * (world) / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        # value counts token rows (layer x KV head x position); the same per
        # sequence position, every layer and KV head of it compressed
        "sequence_tokens_per_s": value / (w.layers * w.heads),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "io_dtype": args.dtype if args.dtype == "bf16" else "fp8_e4m3",
        "data": synthkv.describe(w),
        "config": {"workload": w.name, "run": args.run, "layers": w.layers, "batch": w.batch, "kv_heads": w.heads,
                   "cache_dtype": args.dtype if args.dtype == "bf16" else "fp8_e4m3",
                   "heads_total": w.n_heads, "t": T, "head_dim": w.head_dim, "mode": mode,
                   "window": window, "ratio": ratio, "keep_per_head": ks,
                   "centroid_score_path": {0: "three kernels (K read twice)", 1: "single pass (K read once)",
                                           2: "head groups (K read from HBM once, again from L2)",
                                           4: "head groups with a copy ring (K read from HBM once by bulk "
                                              "copies, again from L2)",
                                           3: "fused whole path (one launch: head groups, selects, gathers; "
                                              + ("the library's own rule" if args.fused is None else
                                                 f"scorer budget {args.fused}, {args.fused_selectors} selector CTAs")
                                              + ")"}.get(single, "?"),
                   "head_group_plan": hg_plan,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "no flush: K+V (%.1f GB) exceed the 129 MB L2" % (2 * K.numel() * es / 1e9)},
        "hbm": {"path_bytes_per_step": nbytes["path"], "achieved_gbs": hbm_gbs,
                "frac_of_nominal_8000": hbm_gbs / world / NOMINAL_HBM_GBS,
                "frac_of_measured": hbm_gbs / world / peaks["hbm_gbs"]},
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"],
                     "traffic": traffic, "algorithmic_bytes_per_launch": dom_bytes,
                     "ms_per_launch": dom_ms},
        "stages_ms": dict(zip(STAGES, stage_ms)),
        "cpu_baseline": cpu,
        "e2e": e2e,
        # per step: a1 + a2 (one kernel, or piece sums + window means + scores),
        # select, compaction when select did not emit the indices, gather
        "gpu_launches": args.steps * (1 if single == 3 else
                                      (1 if single in (1, 2, 4) else 3) + 1 + (0 if select_emits else 1) + 1),
        "clocks": clocks.summary(),
    }
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------ reference arm --

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np

    import oracle
    w, mode, window, ratio = workload_run(args.workload, args.layers, args.run, args.mode, args.window, args.ratio)
    lens = synthkv.seq_lengths(w, args.seed).tolist()
    oracle.build()
    # one head sizes the sample, so that the whole run takes about ref_budget
    K1, V1, _ = synthkv.make_kv(w, seed=args.seed, heads=[0])
    t0 = time.perf_counter()
    oracle.compress_heads(K1, V1, np.array([lens[0]], np.int32), ratio, mode, window)
    t_head = max(time.perf_counter() - t0, 1e-6)
    nt = host_threads()
    per_step = oracle_sample_size(t_head, nt, args.ref_budget / max(1, args.steps + args.warmup), w.n_heads)
    ids = list(range(per_step))
    K, V, _ = synthkv.make_kv(w, seed=args.seed, heads=ids)
    hl = np.array([lens[h // w.heads] for h in ids], np.int32)
    value, used, times = oracle_sample_rate(K, V, hl, ratio, mode, window, nt, steps=args.steps, warmup=args.warmup)
    sec = sum(times) / len(times)
    tok = int(hl.sum())
    sample = (f"the first {per_step} of {w.n_heads} heads ({tok} token rows) per step, split into {used} batches, "
              f"one host thread each, fp64 C oracle")
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64",
        "data": synthkv.describe(w) + "; the same recipe drawn on the CPU",
        "config": {"workload": w.name, "run": args.run, "heads_total": w.n_heads, "t": w.t_max,
                   "head_dim": w.head_dim, "mode": mode, "window": window, "ratio": ratio,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "cpu_model": host_cpu_model(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------ the widened paths (NEXT) --

def _timed(fn, steps, stream, torch):
    """Mean ms of fn() over `steps` calls, CUDA events on the launching stream."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_secondary(args):
    """One JSON line for a widened path (rank 0, one GPU): the OjaKV scorer
    and its selection, the cluster summaries, or the per-window quota."""
    import torch

    import geometric_kv_cache_gb300 as mkv

    world, rank, local = dist_env()
    if rank != 0:
        return
    dev = torch.device("cuda", torch.cuda.current_device())
    mkv.load()
    stream = torch.cuda.current_stream(dev)
    peaks = measured_peaks()
    hbm = peaks["hbm_gbs"]
    steps = args.steps
    if args.path == "oja":
        w = workload_run(args.workload, args.layers)[0]
        K, V, lens = synthkv.make_kv(w, seed=args.seed, device=dev)
        M, r, ratio = args.oja_queries, args.oja_rank, 0.5
        Q, U = synthkv.make_oja_inputs(w, args.seed, M, r, device=dev)
        T = w.t_max
        ks = mkv.mkv_num_keep(T, ratio)
        ws = mkv.oja_workspace_for(K, M, lens)
        S = torch.empty(K.shape[:3], device=dev)
        Ko = torch.empty((w.rows, w.heads, ks, 128), dtype=torch.bfloat16, device=dev)
        Vo = torch.empty_like(Ko)
        idx = torch.empty((w.rows, w.heads, ks), dtype=torch.int32, device=dev)
        kept = torch.empty((w.rows, w.heads), dtype=torch.int32, device=dev)

        def step():
            mkv.mkv_compress_oja(K, V, Q, U, ratio, ks, Ko, Vo, idx, kept, ws, lens, stream=stream)

        def score():
            mkv.mkv_oja_score(K, Q, U, S, ws, lens, stream=stream)
        for _ in range(max(3, args.warmup)):
            step()
            score()
        with ClockSampler(dev.index or 0) as clocks:
            ms = _timed(step, steps, stream, torch)
        ms_score = _timed(score, steps, stream, torch)
        if mkv.mkv_device_status(ws, stream) != 0:
            raise RuntimeError("device status nonzero")
        tokens = w.n_heads * T
        kbytes = tokens * (256 + 4)
        flops = 2.0 * 2 * M * 128 * tokens
        achieved = kbytes / (ms_score / 1e3) / 1e9
        tflops = flops / (ms_score / 1e3) / 1e12
        line = {"metric": "OjaKV-style full-rank selection: KV tokens scored (reconstruction error over the query "
                          "window) + selected + compacted per second",
                "value": tokens / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": steps, "warmup": args.warmup,
                "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16 x bf16 -> f32 (tcgen05), f32",
                "data": "synthetic (seeded)",
                "config": {"workload": w.name, "heads_total": w.n_heads, "t": T, "n_query": M, "rank": r,
                           "ratio": ratio, "keep_per_head": ks},
                "roofline": {"bound": "hbm", "kernel": "oja_score (k_oja_project + k_oja_scores)",
                             "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                             "peak_source": peaks["source"], "ms_per_launch": ms_score,
                             "algorithmic_bytes_per_launch": kbytes,
                             "tensor": {"achieved_tflops": tflops, "flops_per_launch": flops,
                                        "note": "2 x 2 x n_query x 128 flop per token (hi and lo operand rows)"}},
                "clocks": clocks.summary(), "gpu_launches": steps * 4}
    elif args.path == "summaries":
        w = workload_run(args.workload, args.layers)[0]
        K, V, lens = synthkv.make_kv(w, seed=args.seed, device=dev)
        W = args.cluster
        nw = mkv.mkv_num_windows(w.t_max, W)
        ws = mkv.workspace_for(K, W, lens)
        Km = torch.empty((w.rows, w.heads, nw, 128), device=dev)
        Vm = torch.empty_like(Km)
        Kr = torch.empty((w.rows, w.heads, nw), device=dev)

        def step():
            mkv.mkv_window_means(K, W, Km, ws, radius=Kr, seq_lens=lens, stream=stream)
            mkv.mkv_window_means(V, W, Vm, ws, seq_lens=lens, stream=stream)
        for _ in range(max(3, args.warmup)):
            step()
        with ClockSampler(dev.index or 0) as clocks:
            ms = _timed(step, steps, stream, torch)
        if mkv.mkv_device_status(ws, stream) != 0:
            raise RuntimeError("device status nonzero")
        tokens = w.n_heads * w.t_max
        nbytes = 2 * tokens * 256 + w.n_heads * nw * (2 * 512 + 4)
        achieved = nbytes / (ms / 1e3) / 1e9
        line = {"metric": "cluster summaries (mean K, mean V, K radius per cluster): KV tokens summarised per second",
                "value": tokens / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": steps, "warmup": args.warmup,
                "ms_per_step": ms, "higher_is_better": True, "dtype": "f32", "data": "synthetic (seeded)",
                "config": {"workload": w.name, "heads_total": w.n_heads, "t": w.t_max, "cluster": W},
                "roofline": {"bound": "hbm", "kernel": "k_small_window_regs (K with radius, then V; clusters of at most 16 rows)" if args.cluster <= 16 else "k_small_window_means (K with radius, then V)",
                             "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                             "peak_source": peaks["source"], "algorithmic_bytes_per_launch": nbytes},
                "clocks": clocks.summary(), "gpu_launches": steps * 2}
    elif args.path == "inplace":
        w, mode, window, ratio = workload_run(args.workload, args.layers)
        K0, V0, lens = synthkv.make_kv(w, seed=args.seed, device=dev)
        K, V = K0.clone(), V0.clone()
        ws = mkv.workspace_for(K, window, lens)
        kept = torch.empty((w.rows, w.heads), dtype=torch.int32, device=dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]

        def step(i=None):
            if i is not None:
                evs[i][0].record(stream)
            mkv.mkv_compress_inplace(K, V, ratio, mode, window, ws, kept=kept, seq_lens=lens, stream=stream)
            if i is not None:
                evs[i][1].record(stream)
        for _ in range(max(3, args.warmup)):
            K.copy_(K0), V.copy_(V0)
            step()
        torch.cuda.synchronize()
        with ClockSampler(dev.index or 0) as clocks:
            # every step compresses a fresh copy of the cache; the restore
            # copies run between the event pairs, outside the timed spans
            for i in range(steps):
                K.copy_(K0), V.copy_(V0)
                step(i)
            torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in evs) / steps
        if mkv.mkv_device_status(ws, stream) != 0:
            raise RuntimeError("device status nonzero")
        lens_list = lens.cpu().tolist()
        nb = path_bytes(lens_list, w.heads, ratio, w.head_dim)
        achieved = nb["path"] / (ms / 1e3) / 1e9
        line = {"metric": "in-place ManifoldKV compression: KV tokens scored+compacted per second (no output buffers)",
                "value": nb["tokens"] / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": steps, "warmup": args.warmup,
                "ms_per_step": ms, "higher_is_better": True, "dtype": "f32", "data": "synthetic (seeded)",
                "config": {"workload": w.name, "heads_total": w.n_heads, "t": w.t_max, "mode": mode,
                           "window": window, "ratio": ratio},
                "hbm": {"path_bytes_per_step": nb["path"], "achieved_gbs": achieved,
                        "frac_of_measured": achieved / hbm, "frac_of_nominal_8000": achieved / NOMINAL_HBM_GBS},
                "clocks": clocks.summary(),
                # a1 + a2 (one kernel or three), select, in-place move
                "gpu_launches": steps * ((1 if mkv.mkv_compress_single_pass(mkv.shape_of(K, lens), window, mode)
                                          in (1, 2, 4) else 3) + 2)}
    else:  # quota
        w = workload_run(args.workload, args.layers)[0]
        K, V, lens = synthkv.make_kv(w, seed=args.seed, device=dev)
        mode, window, ratio = w.runs[0]
        window = window or 4096
        ks = mkv.mkv_num_keep_quota(w.t_max, ratio, window)
        ws = mkv.workspace_for(K, window, lens)
        Ko = torch.empty((w.rows, w.heads, ks, 128), dtype=torch.bfloat16, device=dev)
        Vo = torch.empty_like(Ko)
        idx = torch.empty((w.rows, w.heads, ks), dtype=torch.int32, device=dev)
        kept = torch.empty((w.rows, w.heads), dtype=torch.int32, device=dev)

        def step():
            mkv.mkv_compress_quota(K, V, ratio, mode, window, ks, Ko, Vo, idx, kept, ws, lens, stream=stream)
        for _ in range(max(3, args.warmup)):
            step()
        with ClockSampler(dev.index or 0) as clocks:
            ms = _timed(step, steps, stream, torch)
        if mkv.mkv_device_status(ws, stream) != 0:
            raise RuntimeError("device status nonzero")
        tokens = w.n_heads * w.t_max
        nbytes = 4 * tokens * 128 + 8 * w.n_heads * ks * 128
        achieved = nbytes / (ms / 1e3) / 1e9
        line = {"metric": "WindowedManifoldKV with per-window quotas: KV tokens scored+compacted per second",
                "value": tokens / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": steps, "warmup": args.warmup,
                "ms_per_step": ms, "higher_is_better": True, "dtype": "f32", "data": "synthetic (seeded)",
                "config": {"workload": w.name, "heads_total": w.n_heads, "t": w.t_max, "mode": mode,
                           "window": window, "ratio": ratio, "keep_per_head": ks},
                "hbm": {"path_bytes_per_step": nbytes, "achieved_gbs": achieved, "frac_of_measured": achieved / hbm,
                        "frac_of_nominal_8000": achieved / NOMINAL_HBM_GBS},
                "clocks": clocks.summary(),
                # a1 + a2 (one kernel or three), quota select, gather
                "gpu_launches": steps * ((1 if mkv.mkv_compress_single_pass(mkv.shape_of(K, lens), window, mode)
                                          in (1, 2, 4) else 3) + 2)}
    line["path"] = args.path
    print(json.dumps(line), flush=True)


def load_traffic(path, workload, layers, dtype, run=None, root=ROOT):
    """Per-kernel DRAM bytes per launch from an ncu record (profiles/traffic.json),
    for the bench's own workload, run (mode, window, ratio), layer count and
    cache type only. The record holds one entry per captured (workload, run,
    cache type); a kernel's figure counts only while its source files are
    unchanged: the sha256 of those files, concatenated in the listed order,
    must match the record. Returns {kernel: bytes} (possibly empty), or None
    without a matching entry."""
    if not path or not os.path.exists(path) or layers:
        return None
    with open(path) as f:
        t = json.load(f)
    for rec in t.get("records", []):
        if rec.get("workload") != workload or rec.get("cache_dtype", "bf16") != dtype:
            continue
        if run is not None and rec.get("run") is not None and list(rec["run"]) != list(run):
            continue
        out = {}
        for name, k in rec.get("kernels", {}).items():
            srcs = [os.path.join(root, x) for x in k.get("sources", [])]
            if not srcs or not all(os.path.exists(x) for x in srcs):
                continue
            h = hashlib.sha256()
            for src in srcs:
                with open(src, "rb") as f:
                    h.update(f.read())
            if h.hexdigest()[:16] == k.get("sha256_16"):
                out[name] = k.get("bytes_per_launch")
        return out
    return None


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, choices=sorted(synthkv.WORKLOADS),
                    help=f"default: {synthkv.BENCH_WORKLOAD} (ManifoldKV path), {synthkv.SECONDARY_WORKLOAD} "
                         "(--path oja/summaries/inplace), qwen3-8b-kv-t64k-w4096 (--path quota)")
    ap.add_argument("--run", type=int, default=0, help="which of the workload's runs (mode, window, ratio)")
    ap.add_argument("--mode", choices=["l2", "cosine"], default=None, help="override the run's score mode")
    ap.add_argument("--window", type=int, default=None, help="override the run's window (0 = global)")
    ap.add_argument("--ratio", type=float, default=None, help="override the run's compression ratio")
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count (profiling)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=60.0, help="seconds of oracle time for --impl reference")
    ap.add_argument("--no-head-groups", action="store_true",
                    help="three-kernel centroid + score path instead of head groups (A/B)")
    ap.add_argument("--ring", type=int, choices=[0, 1], default=None,
                    help="copy-ring head-group kernel on (1) or off (0); default: the library's setting")
    ap.add_argument("--path", choices=["manifold", "oja", "summaries", "quota", "inplace"], default="manifold",
                    help="manifold: the headline path; the others time a widened path (one GPU, own JSON line)")
    ap.add_argument("--oja-queries", type=int, default=128, help="query-window rows per KV head (--path oja)")
    ap.add_argument("--oja-rank", type=int, default=64, help="basis rank (--path oja)")
    ap.add_argument("--cluster", type=int, default=10, help="cluster length (--path summaries)")
    ap.add_argument("--dtype", choices=sorted(CACHE_DTYPE_NAMES), default="bf16",
                    help="cache element type: bf16, or fp8 (E4M3 codes; the ManifoldKV path only)")
    ap.add_argument("--fused", type=int, default=None,
                    help="fused whole-path kernel: N > 0 with N scorer CTAs, 0 never (the separate kernels); "
                         "default: the library's own shape rule")
    ap.add_argument("--fused-selectors", type=int, default=32, help="CTAs that run the selects (--fused N > 0)")
    ap.add_argument("--traffic-json", default=os.path.join(ROOT, "profiles", "traffic.json"),
                    help="per-kernel DRAM bytes per launch from an ncu capture (null when absent)")
    args = ap.parse_args(argv)
    if args.workload is None:
        args.workload = (synthkv.BENCH_WORKLOAD if args.path == "manifold" else
                         "qwen3-8b-kv-t64k-w4096" if args.path == "quota" else synthkv.SECONDARY_WORKLOAD)
    if args.path == "manifold":
        _, m, wd, r = workload_run(args.workload, 0, args.run, args.mode, args.window, args.ratio)
        args.traffic = load_traffic(args.traffic_json, args.workload, args.layers, args.dtype, run=(m, wd, r))
    else:
        args.traffic = None
    if args.dtype != "bf16" and (args.impl == "reference" or args.path != "manifold"):
        ap.error("--dtype fp8 applies to the ManifoldKV path of our arm only")
    if args.impl == "reference":
        run_reference(args)
    elif args.path != "manifold":
        run_secondary(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
