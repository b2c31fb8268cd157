"""Mask diagnostics (block_sparse_attention_sa2_gb300/diagnostics.py) on CPU tensors.

The statistics match the oracle's selection: the kept counts equal its L, and the kept mass
equals its pooled mass over kept blocks.  On the mask-probe workload (heads 0-3 flat, heads
4-7 dominated by one sink block) they reproduce the failure analysis of the two rules
(gist.science explainer, section 1):
- Top-k alone keeps little of a flat row's mass;
- Top-p alone keeps a single block on sink rows;
- the hybrid keeps mass >= p on the flat rows and at least K blocks on the sink rows."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_attention_sa2_gb300 import BlockMask
from block_sparse_attention_sa2_gb300.diagnostics import head_histograms, mask_diagnostics
from workload import CONFIGS, make_inputs


@pytest.fixture(scope="module")
def probe():
    cfg = CONFIGS[1]
    return cfg, make_inputs(cfg, tensors=("q", "k"))


def _blockmask(res, cfg):
    B, H = res["mask"].shape[:2]
    bm = BlockMask.empty(B, H, cfg.Tq, cfg.Tk, "cpu", mask=True, pooled=True)
    bm.row_cnt.copy_(torch.from_numpy(res["mask"].sum(axis=-1).astype(np.int32)))
    bm.mask.copy_(torch.from_numpy(res["mask"]))
    bm.pooled_p.copy_(torch.from_numpy(res["P"].astype(np.float32)))
    return bm


def test_statistics_match_the_oracle_selection(probe):
    cfg, x = probe
    res = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, 0.05, 0.9)
    d = mask_diagnostics(_blockmask(res, cfg), bins=8)
    for h in range(cfg.H):
        sel = res["sel"][(0, h)]
        assert np.array_equal(d["kept"][0, h].numpy(), sel.L)
        want_mass = np.array([sel.sorted_P[i, :sel.L[i]].sum() for i in range(cfg.Tq)])
        np.testing.assert_allclose(d["kept_mass"][0, h].numpy(), want_mass, atol=1e-6)
    assert (d["kept_frac_hist"].sum(-1) == cfg.Tq).all()
    assert (d["kept_mass_hist"].sum(-1) == cfg.Tq).all()


def test_failure_modes_of_the_single_rules_and_the_hybrid(probe):
    cfg, x = probe
    k, p = 0.05, 0.9
    K = math.ceil(k * cfg.Tk - 1e-9)
    flat, sink = slice(0, 4), slice(4, 8)
    topk = mask_diagnostics(_blockmask(O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, k, 0.0), cfg))
    assert (topk["kept"] == K).all()
    assert topk["kept_mass"][0, flat].median() < 0.5  # a flat row's mass is spread: K blocks miss most
    topp = mask_diagnostics(_blockmask(O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, 0.0, p), cfg))
    assert (topp["kept"][0, sink] == 1).all()  # the sink block alone reaches p
    assert (topp["kept_mass"][0, sink] >= p).all()
    hyb = mask_diagnostics(_blockmask(O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, k, p), cfg))
    assert (hyb["kept_mass"][0, flat] >= p - 1e-6).all()
    assert (hyb["kept"][0, sink] >= K).all()


def test_histogram_bins_and_edges():
    v = torch.tensor([[0.0, 0.05, 0.1, 0.55, 0.999, 1.0, 1.2, -0.1]])
    assert head_histograms(v, bins=10).tolist() == [[3, 1, 0, 0, 0, 1, 0, 0, 0, 3]]
    with pytest.raises(ValueError):
        head_histograms(v, bins=0)
