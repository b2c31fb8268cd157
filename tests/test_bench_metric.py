"""The benchmark's work count: the kept (query, key) token pairs behind every TFLOP/s figure
equal, for ragged shapes, the number of allowed entries of the oracle's token-level mask
(gist.science explainer, section 2.C: tiles are kept or skipped whole, and tokens past N do
not exist)."""
import os
import sys

import numpy as np
import pytest

import oracle as O
from workload.gen import WorkloadConfig

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


@pytest.mark.parametrize("N,bq,bk", [(1000, 128, 64), (777, 64, 64), (130, 128, 64), (1, 128, 64), (4096, 128, 64)])
def test_kept_pairs_count_the_token_mask(N, bq, bk):
    cfg = WorkloadConfig(index=200, name="count", B=2, H=3, grid=(1, 1, N), d=64, dtype="bf16", bq=bq, bk=bk)
    rng = np.random.default_rng(N)
    mask = (rng.random((cfg.B, cfg.H, cfg.Tq, cfg.Tk)) < 0.3).astype(np.uint8)
    mask[0, 0, -1, -1] = 1  # the ragged corner tile
    want = sum(int(O.token_mask(mask[b, h], N, bq, bk).sum()) for b in range(cfg.B) for h in range(cfg.H))
    assert bench.kept_pairs(cfg, mask) == want


def test_dense_mask_counts_every_pair():
    cfg = WorkloadConfig(index=201, name="dense", B=1, H=2, grid=(1, 1, 1000), d=64, dtype="bf16", bq=128, bk=64)
    mask = np.ones((1, 2, cfg.Tq, cfg.Tk), dtype=np.uint8)
    assert bench.kept_pairs(cfg, mask) == 2 * 1000 * 1000


def test_dkdv_traffic_is_reported_only_for_the_captured_workload():
    import dataclasses
    from workload import CONFIGS
    wan14 = CONFIGS[3]
    full = bench.dkdv_traffic(wan14, 0.95)
    assert full is not None and full > 0
    four = bench.dkdv_traffic(dataclasses.replace(wan14, H=4), 0.95)
    assert four == pytest.approx(full * 4 / wan14.H)  # heads are independent and equal in work
    assert bench.dkdv_traffic(wan14, 0.9) is None
    assert bench.dkdv_traffic(CONFIGS[2], 0.95) is None


def test_roofline_accounting_credits_only_algorithmic_work():
    """The dQ kernel is credited with its dQ GEMM only (2 d per kept pair), the dK/dV kernel with
    S, dP, dV, dK (8 d): together the backward's 10 d.  Fractions use the burst bf16 peak, and
    each phase's time includes its conversions and preprocessing."""
    pairs, d, steps = 1.0e9, 128, 2
    prof = {"attn_fwd": (2, 4.0), "attn_bwd_dkdv": (2, 10.0), "attn_bwd_dq": (2, 6.0), "to_f16": (6, 1.5),
            "bwd_preprocess": (2, 1.0), "bwd_pair_union": (2, 0.2), "pool": (2, 0.6)}
    peaks = {"bf16_tflops": 1000.0, "bf16_tflops_sustained": 800.0, "hbm_gbs": 7000.0, "source": "test"}
    ph = bench.phase_rooflines(prof, steps, pairs, d, peaks["bf16_tflops"])
    assert ph["forward"]["ms"] == pytest.approx(2.0 + 0.25)
    assert ph["backward"]["ms"] == pytest.approx(5.0 + 3.0 + 0.5 + 0.1 + 0.5)
    assert ph["backward"]["algorithmic_tflop"] == pytest.approx(10 * d * pairs / 1e12)
    assert ph["backward"]["frac_of_bf16_burst"] == pytest.approx(10 * d * pairs / (9.1e-3) / 1e12 / 1000.0)
    roof = bench.dominant_roofline(prof, pairs, d, peaks)
    assert roof["kernel"] == "attn_bwd_dkdv" and roof["peak"] == 1000.0
    assert roof["achieved"] == pytest.approx(8 * d * pairs / 5e-3 / 1e12)
    dq_only = {"attn_bwd_dq": (1, 3.0)}
    assert bench.dominant_roofline(dq_only, pairs, d, peaks)["achieved"] == pytest.approx(2 * d * pairs / 3e-3 / 1e12)
