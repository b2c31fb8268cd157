import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def repo_root():
    return ROOT


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The errors the parity checks measured: the worst of each kind of tensor, and the mask
    comparisons with their exempt (near-threshold) entries."""
    try:
        from tests.gpu_util import PARITY_LOG
    except Exception:
        return
    if not PARITY_LOG:
        return
    tr = terminalreporter
    tr.section("parity: measured errors")
    worst = {}
    for r in PARITY_LOG:
        if r["kind"] != "tensor":
            continue
        key = r["name"].split()[-1] if r["name"].split() else r["name"]
        w = worst.setdefault(key, {"n": 0, "max_abs": 0.0, "over": 0.0, "mean_rel": 0.0, "at": ""})
        w["n"] += 1
        if r["worst_over_bound"] > w["over"]:
            w["over"], w["at"] = r["worst_over_bound"], r["name"]
        w["max_abs"] = max(w["max_abs"], r["max_abs"])
        w["mean_rel"] = max(w["mean_rel"], r["mean_rel"])
    for key, w in sorted(worst.items()):
        tr.write_line(f"{key:>10}: {w['n']:4d} checks, max|d| {w['max_abs']:.3e}, worst |d|/bound {w['over']:.3f} "
                      f"({w['at']}), worst mean rel {w['mean_rel']:.3e}")
    masks = [r for r in PARITY_LOG if r["kind"] == "mask"]
    if masks:
        rows = sum(r["rows"] for r in masks)
        ex = sum(r["exempt_entries"] for r in masks)
        amb = sum(r["ambiguous_cut_rows"] for r in masks)
        dp = max(r["max_pbar_delta"] for r in masks)
        tr.write_line(f"      mask: {len(masks)} comparisons, {rows} rows, {ex} exempt near-threshold entries, "
                      f"{amb} rows with an ambiguous Top-p cut, max |dP-bar| {dp:.2e}")
        for r in masks:
            if r["exempt_entries"]:
                tr.write_line(f"            {r['name']}: exempt {r['exempt'][:4]}")
