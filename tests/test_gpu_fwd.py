"""GPU parity of sa2_attn_fwd against the fp64 oracle.

The CUDA forward runs on the oracle's own block mask (handed over as compact lists), so
the comparison isolates the attention.  Bar: max |d| <= 2e-2 and sum|d| / sum|ref| <= 5e-3
on O; LSE within 2e-2 where finite, and -inf exactly where the row keeps nothing.

fp32 inputs are held to the same bar against the oracle on the exact fp32 inputs: the
library forms their scores as the split fp16 product Qhi Khi^T + Qhi Klo^T + Qlo Khi^T
(about 22 bits) and only P and V take a single fp16 rounding (include/sa2.h)."""
import json
import os

import numpy as np
import pytest

import oracle as O
from tests.gpu_util import assert_close, blockmask_from_oracle, to_device, to_f64
from workload import CONFIGS, make_inputs
from workload.gen import small_case

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def sa2():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_attention_sa2_gb300 as m
    m.load_library()
    return m


def _run_fwd(sa2, cfg, x, mask, scale=None):
    q, k, v = (to_device(x[t]) for t in ("q", "k", "v"))
    bm = blockmask_from_oracle(mask)
    o, lse = sa2.attn_fwd(q, k, v, bm, bq=cfg.bq, bk=cfg.bk, scale=scale)
    sa2.check_device()
    return to_f64(o), lse.cpu().numpy().astype(np.float64)


def _check_head(name, o, lse, ro, rlse, lse_tol=2e-2, **tol):
    assert_close(name + " O", o, ro, **tol)
    fin = np.isfinite(rlse)
    assert (np.isneginf(lse) == ~fin).all(), name + ": -inf LSE pattern differs"
    if fin.any():
        assert np.abs(lse[fin] - rlse[fin]).max() <= lse_tol, name + f" LSE {np.abs(lse[fin] - rlse[fin]).max():.3e}"


def _full_check(sa2, cfg, x, mask, scale=None):
    o, lse = _run_fwd(sa2, cfg, x, mask, scale)
    ro, rlse = O.attn_fwd(x["q"], x["k"], x["v"], mask, cfg.bq, cfg.bk, scale)
    for b in range(cfg.B):
        for h in range(cfg.H):
            _check_head(f"{cfg.name} b{b}h{h}", o[b, h], lse[b, h], ro[b, h], rlse[b, h])


def test_fwd_tiny_fp32_config(sa2):
    cfg = CONFIGS[0]
    x = make_inputs(cfg)
    mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, cfg.topk, cfg.topp)["mask"]
    _full_check(sa2, cfg, x, mask)


@pytest.mark.parametrize("N,d,bq,dtype", [(1000, 128, 128, "bf16"), (777, 64, 64, "bf16"), (1000, 64, 128, "fp32"),
                                          (1100, 128, 64, "fp32"), (130, 128, 128, "bf16"), (1, 64, 128, "bf16")])
def test_fwd_ragged_small_cases(sa2, N, d, bq, dtype):
    cfg, x = small_case(f"ragged-{N}", 2, 2, N, d, dtype, bq, 64, seed=5)
    for topk, topp in ((0.2, 0.6), (1.0, 0.0), (0.0, 0.3)):
        mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, topk, topp)["mask"]
        _full_check(sa2, cfg, x, mask)


def test_fwd_random_masks_with_empty_rows_and_scale(sa2):
    cfg, x = small_case("random-mask", 1, 3, 700, 128, "bf16", 128, 64, seed=7)
    rng = np.random.default_rng(0)
    mask = (rng.random((1, 3, cfg.Tq, cfg.Tk)) < 0.3).astype(np.uint8)
    mask[0, 0, 2] = 0  # an empty row: O = 0, LSE = -inf
    mask[0, 1] = 0  # a head that keeps nothing
    _full_check(sa2, cfg, x, mask)
    _full_check(sa2, cfg, x, mask, scale=0.05)


def test_fwd_mask_probe_config_sampled_rows(sa2):
    cfg = CONFIGS[1]
    x = make_inputs(cfg)
    for topk, topp in ((0.05, 0.9), (0.02, 0.5)):
        mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, topk, topp)["mask"]
        o, lse = _run_fwd(sa2, cfg, x, mask)
        rows = np.concatenate([np.arange(0, 130), np.arange(4000, 4100), np.arange(cfg.N - 130, cfg.N)])
        for h in (0, 3, 4, 7):
            ro, rlse = O.attn_fwd_head(O.to_f64(x["q"][0, h]), O.to_f64(x["k"][0, h]), O.to_f64(x["v"][0, h]),
                                       mask[0, h], cfg.bq, cfg.bk, rows=rows)
            _check_head(f"probe h{h}", o[0, h, rows], lse[0, h, rows], ro, rlse)


def test_fwd_longest_sequence_sampled_rows(sa2):
    """The longest sequence the library accepts (N = 491520 tokens, 7680 key blocks), d = 64,
    Top-k-only mask of 39 blocks per row; sampled rows (first, middle, last blocks)."""
    cfg, x = small_case("longest", 1, 1, 7680 * 64, 64, "bf16", 128, 64, seed=53, tensors=("q", "k", "v"))
    mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, 0.005, 0.0)["mask"]
    o, lse = _run_fwd(sa2, cfg, x, mask)
    rows = np.concatenate([np.arange(0, 64), np.arange(cfg.N // 2, cfg.N // 2 + 64), np.arange(cfg.N - 100, cfg.N)])
    ro, rlse = O.attn_fwd_head(O.to_f64(x["q"][0, 0]), O.to_f64(x["k"][0, 0]), O.to_f64(x["v"][0, 0]),
                               mask[0, 0], cfg.bq, cfg.bk, rows=rows)
    _check_head("longest", o[0, 0, rows], lse[0, 0, rows], ro, rlse)


def test_fwd_end_to_end_from_gpu_mask(sa2):
    """GPU mask -> GPU forward, against the oracle on the oracle's mask (rows whose masks
    agree; the masks differ at most in near-threshold entries)."""
    cfg, x = small_case("e2e", 1, 2, 2000, 128, "bf16", 128, 64, seed=9)
    q, k, v = (to_device(x[t]) for t in ("q", "k", "v"))
    bm = sa2.build_mask(q, k, 0.1, 0.7, bq=cfg.bq, bk=cfg.bk)
    o, lse = sa2.attn_fwd(q, k, v, bm, bq=cfg.bq, bk=cfg.bk)
    sa2.check_device()
    ref = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, 0.1, 0.7)["mask"]
    gm = bm.mask.cpu().numpy()
    ro, rlse = O.attn_fwd(x["q"], x["k"], x["v"], ref, cfg.bq, cfg.bk)
    o, lse = to_f64(o), lse.cpu().numpy()
    for h in range(cfg.H):
        same = np.all(gm[0, h] == ref[0, h], axis=1)
        rows = np.nonzero(np.repeat(same, cfg.bq)[: cfg.N])[0]
        assert rows.size >= cfg.N // 2
        _check_head(f"e2e h{h}", o[0, h, rows], lse[0, h, rows], ro[0, h, rows], rlse[0, h, rows])
