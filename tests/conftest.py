import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); runs the CUDA path against the oracle")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


# Parity tallies (tests/parity_util.py): every GPU comparison with the oracle
# counts its heads, near-cut exceptions and relaxed cosine scores per test and
# score mode. The totals are printed at the end of the session and written,
# with one record per test, to profiles/parity_exceptions.json (or to
# $MKV_PARITY_SUMMARY), so they are kept with the other measurements.

@pytest.fixture(autouse=True)
def _parity_test_name(request):
    import parity_util
    parity_util.current_test = request.node.nodeid
    yield


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    pu = sys.modules.get("parity_util")
    if pu is None or not pu.TALLY:
        return
    import json
    import platform
    import time
    recs = sorted(pu.TALLY.values(), key=lambda r: (r["test"], r["mode"]))
    tot = {k: sum(r[k] for r in recs) for k in ("heads", "scores", "near_cut_exceptions", "cosine_relaxed")}
    by_mode = {}
    for r in recs:
        m = by_mode.setdefault(r["mode"], {"heads": 0, "near_cut_exceptions": 0, "cosine_relaxed": 0})
        for k in m:
            m[k] += r[k]
    gpu = "?"
    try:
        import torch
        if torch.cuda.is_available():
            gpu = torch.cuda.get_device_name(0)
    except Exception:  # noqa: BLE001 - the summary must not fail the session
        pass
    out = {"when": time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime()), "gpu": gpu, "host": platform.machine(),
           "exit_status": int(exitstatus), "totals": tot, "by_mode": by_mode, "tests": recs, "cases": pu.CASES}
    path = os.environ.get("MKV_PARITY_SUMMARY") or os.path.join(ROOT, "profiles", "parity_exceptions.json")
    try:
        with open(path, "w") as f:
            json.dump(out, f, indent=1)
            f.write("\n")
    except OSError:
        path = "(not written)"
    terminalreporter.write_line(
        f"parity vs oracle: {tot['heads']} heads, {tot['scores']} scores compared; near-cut exceptions "
        f"{tot['near_cut_exceptions']} (" + ", ".join(f"{m} {v['near_cut_exceptions']}" for m, v in by_mode.items())
        + f"); cosine scores needing the relaxed bound {tot['cosine_relaxed']}; per test in {path}")
