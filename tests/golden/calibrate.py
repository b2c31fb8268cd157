"""Calibrate the mask parameters (k, p) of the large workloads to a target block sparsity.

The pages report 95 % attention sparsity (thelatestinai.com page, Tables 4 and 5) but give
no k or p.  This script picks them on the oracle's pooled map of the seeded inputs and
writes ``calibration.json`` beside it.  It calls only ``oracle/`` and ``workload/``.

Rule: start at p = 0.9; if Top-p alone keeps more than half the target density, bisect p
down until it keeps half; then take the largest k whose hybrid density does not exceed the
target, and finally bisect p upward until the density is within 0.1 percentage point of
the target (k alone moves in steps of 1/Tk per row).  Sparsity = fraction of
(query-block, key-block) tiles that are skipped.

Usage: python tests/golden/calibrate.py [config ...]
"""
import json
import math
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
from workload import CONFIGS, make_inputs  # noqa: E402

TARGETS = {2: [0.95], 3: [0.95], 4: [0.80, 0.90, 0.95, 0.97], 5: [0.95]}


def sorted_pooled(cfg, threads=8):
    x = make_inputs(cfg, tensors=("q", "k"), threads=threads)
    rows = []
    for b in range(cfg.B):
        for h in range(cfg.H):
            P = O.build_mask_head(O.to_f64(x["q"][b, h]), O.to_f64(x["k"][b, h]),
                                  cfg.bq, cfg.bk, 0.0, 0.0)["P"]
            rows.append(np.take_along_axis(P, O.row_order(P), axis=1))
    return np.concatenate(rows, axis=0)


def density(sP, k, p):
    Tk = sP.shape[1]
    L = np.maximum(O.topk_count(k, Tk), O.topp_count(sP, p))
    return float(L.sum()) / sP.size


def calibrate(sP, target_sparsity, tol=1e-3):
    dens = 1.0 - target_sparsity
    Tk = sP.shape[1]
    p = 0.9
    if density(sP, 0.0, p) > dens / 2:
        lo, hi = 0.0, p
        for _ in range(50):
            mid = 0.5 * (lo + hi)
            if density(sP, 0.0, mid) > dens / 2:
                hi = mid
            else:
                lo = mid
        p = lo
    # largest K (k = K/Tk) whose density does not exceed the target
    K = 0
    while K < Tk and density(sP, (K + 1) / Tk, p) <= dens:
        K += 1
    k = (K - 0.5) / Tk if K > 0 else 0.0  # ceil(k*Tk) = K with margin for fp32 rounding of k
    lo, hi = p, 1.0
    for _ in range(60):
        if abs(density(sP, k, p) - dens) <= tol:
            break
        mid = 0.5 * (lo + hi)
        if density(sP, k, mid) > dens:
            hi = mid
        else:
            lo = mid
            p = mid
    k, p = float(np.float32(k)), float(np.float32(p))  # the library takes float32 k and p
    return k, p, 1.0 - density(sP, k, p)


def main(argv):
    cfgs = [int(a) for a in argv] or sorted(TARGETS)
    path = os.path.join(HERE, "calibration.json")
    out = json.load(open(path)) if os.path.exists(path) else {}
    out["about"] = ("(k, p) per workload and target block sparsity, chosen on the fp64 oracle's "
                    "pooled map of the seeded inputs (seed 0) by tests/golden/calibrate.py")
    for c in cfgs:
        cfg = CONFIGS[c]
        t0 = time.time()
        sP = sorted_pooled(cfg)
        entry = {}
        for t in TARGETS[c]:
            k, p, s = calibrate(sP, t)
            entry[f"{t:.2f}"] = {"k": k, "p": p, "sparsity": s,
                                 "topk_only_sparsity": 1.0 - density(sP, k, 0.0),
                                 "topp_only_sparsity": 1.0 - density(sP, 0.0, p)}
            print(c, cfg.name, t, entry[f"{t:.2f}"], flush=True)
        out[str(c)] = {"name": cfg.name, "targets": entry}
        print(f"config {c}: {time.time() - t0:.1f} s", flush=True)
    with open(path, "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)
        f.write("\n")


if __name__ == "__main__":
    main(sys.argv[1:])
