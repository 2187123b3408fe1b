"""The bench's ncu traffic record: a kernel's DRAM bytes are reported only for
the recorded workload, run and cache type, and only while the kernel's source
files hash to the recorded value (so a changed kernel reports null)."""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _record(tmp_path, sources, sha, workload="w", dtype="bf16", run=("l2", 0, 0.5)):
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps({"records": [{"workload": workload, "run": list(run), "cache_dtype": dtype,
                                          "kernels": {"k": {"sources": sources, "sha256_16": sha,
                                                            "bytes_per_launch": 123}}}]}))
    return str(p)


def test_traffic_counts_only_for_unchanged_sources(tmp_path):
    a, b = tmp_path / "a.cu", tmp_path / "b.cuh"
    a.write_bytes(b"kernel a\n")
    b.write_bytes(b"header b\n")
    sha = hashlib.sha256(b"kernel a\nheader b\n").hexdigest()[:16]
    rec = _record(tmp_path, ["a.cu", "b.cuh"], sha)
    run = ("l2", 0, 0.5)
    assert bench.load_traffic(rec, "w", 0, "bf16", run, root=str(tmp_path)) == {"k": 123}
    assert bench.load_traffic(rec, "other", 0, "bf16", run, root=str(tmp_path)) is None
    assert bench.load_traffic(rec, "w", 8, "bf16", run, root=str(tmp_path)) is None      # --layers changes the workload
    assert bench.load_traffic(rec, "w", 0, "fp8", run, root=str(tmp_path)) is None
    assert bench.load_traffic(rec, "w", 0, "bf16", ("cosine", 0, 0.5), root=str(tmp_path)) is None
    b.write_bytes(b"header b, changed\n")
    assert bench.load_traffic(rec, "w", 0, "bf16", run, root=str(tmp_path)) == {}
    assert bench.load_traffic(str(tmp_path / "missing.json"), "w", 0, "bf16", run) is None


def test_committed_record_matches_the_gather_sources():
    rec = os.path.join(ROOT, "profiles", "traffic.json")
    got = bench.load_traffic(rec, "llama3.1-8b-kv-t16k", 0, "bf16", ("l2", 0, 0.5))
    assert got is not None and got.get("gather", 0) > 0
    # the Llama workload's default step is the fused kernel: its record must match its sources too
    assert got.get("fused_path", 0) > 0
    # the default bench line (the Phi-4 workload's windowed run) has a record too
    import synthkv
    w, mode, window, ratio = bench.workload_run(synthkv.BENCH_WORKLOAD)
    got = bench.load_traffic(rec, synthkv.BENCH_WORKLOAD, 0, "bf16", (mode, window, ratio))
    assert got is not None and got.get("gather", 0) > 0


def test_every_configured_run_resolves():
    import synthkv
    for name, w in synthkv.WORKLOADS.items():
        for i, run in enumerate(w.runs):
            assert bench.workload_run(name, 0, i)[1:] == tuple(run)
    w, mode, window, ratio = bench.workload_run("phi4-kv-t128k", 0, 2, window=4096)
    assert (mode, window, ratio) == ("cosine", 4096, 0.5)
