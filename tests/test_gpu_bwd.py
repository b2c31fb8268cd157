"""GPU parity of sa2_attn_bwd against the fp64 oracle.

Forward then backward run on the CUDA path with the oracle's mask; the oracle computes
dQ, dK, dV from the same inputs.  Bar on each gradient: max |d| <= 2e-2 and
sum|d| / sum|ref| <= 5e-3, fp32 inputs included: the reference is the oracle on the exact
inputs (the library forms fp32 scores as a split fp16 product, include/sa2.h)."""
import json
import os

import numpy as np
import pytest
import torch

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


def _run(sa2, cfg, x, mask, scale=None):
    q, k, v, do = (to_device(x[t]) for t in ("q", "k", "v", "do"))
    bm = blockmask_from_oracle(mask)
    o_lo = torch.empty_like(q) if q.dtype == torch.bfloat16 else None
    o, lse = sa2.attn_fwd(q, k, v, bm, bq=cfg.bq, bk=cfg.bk, scale=scale, o_lo=o_lo)
    dq, dk, dv = sa2.attn_bwd(q, k, v, o, lse, do, bm, bq=cfg.bq, bk=cfg.bk, scale=scale, o_lo=o_lo)
    sa2.check_device()
    return to_f64(dq), to_f64(dk), to_f64(dv)


def _full_check(sa2, cfg, x, mask, scale=None):
    g = _run(sa2, cfg, x, mask, scale)
    ref = O.attn_bwd(x["q"], x["k"], x["v"], x["do"], mask, cfg.bq, cfg.bk, scale)
    for name, got, want in zip(("dQ", "dK", "dV"), g, ref):
        for b in range(cfg.B):
            for h in range(cfg.H):
                assert_close(f"{cfg.name} b{b}h{h} {name}", got[b, h], want[b, h])
    return g


def test_bwd_tiny_fp32_config(sa2):
    cfg = CONFIGS[0]
    x = make_inputs(cfg)
    mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, cfg.topk, cfg.topp)["mask"]
    _full_check(sa2, cfg, x, mask)


@pytest.mark.parametrize("N,d,bq,dtype", [(1000, 128, 128, "bf16"), (777, 64, 64, "bf16"), (1000, 64, 128, "fp32"),
                                          (1100, 128, 64, "fp32"), (130, 128, 128, "bf16"), (1, 64, 128, "bf16")])
def test_bwd_ragged_small_cases(sa2, N, d, bq, dtype):
    cfg, x = small_case(f"ragged-{N}", 2, 2, N, d, dtype, bq, 64, seed=5)
    for topk, topp in ((0.2, 0.6), (1.0, 0.0), (0.0, 0.3)):
        mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, topk, topp)["mask"]
        _full_check(sa2, cfg, x, mask)


def test_bwd_random_masks_empty_rows_unused_keys_and_scale(sa2):
    cfg, x = small_case("random-mask", 1, 3, 700, 128, "bf16", 128, 64, seed=7)
    rng = np.random.default_rng(1)
    mask = (rng.random((1, 3, cfg.Tq, cfg.Tk)) < 0.3).astype(np.uint8)
    mask[0, 0, 2] = 0  # a query block that keeps nothing
    mask[0, 2, :, 4] = 0  # a key block kept by nobody: dK = dV = 0
    mask[0, 1] = 0
    g = _full_check(sa2, cfg, x, mask)
    assert not g[1][0, 2, 4 * 64:5 * 64].any() and not g[2][0, 2, 4 * 64:5 * 64].any()
    _full_check(sa2, cfg, x, mask, scale=0.05)


@pytest.mark.parametrize("d,bq,dtype", [(64, 128, "bf16"), (128, 64, "bf16"), (64, 128, "fp32")])
def test_bwd_many_items_per_persistent_cta(sa2, d, bq, dtype):
    """The dK/dV and dQ kernels keep one CTA per SM and take key-block pairs / query blocks
    from a counter.  48 short heads give 480 pairs and 480 or 912 query blocks, several per
    CTA, so barrier phases run across items.  Empty items sit between full ones: a head
    keeping nothing, a whole unused key-block pair, a query block keeping nothing, and a
    dense head with long lists.  Every gradient element is checked, and a second call must
    repeat the first bit for bit (the counter is reset per call, and each item is computed
    by one CTA whatever the assignment)."""
    cfg, x = small_case(f"many-items-d{d}-bq{bq}-{dtype}", 2, 24, 1200, d, dtype, bq, 64, seed=61)
    assert cfg.B * cfg.H * ((cfg.Tk + 1) // 2) == 480 and cfg.B * cfg.H * cfg.Tq >= 480
    rng = np.random.default_rng(17)
    mask = (rng.random((cfg.B, cfg.H, cfg.Tq, cfg.Tk)) < 0.2).astype(np.uint8)
    mask[0, 3] = 0              # a head keeping nothing
    mask[1, 5, :, 4:6] = 0      # key-block pair 2 unused: an empty dK/dV item
    mask[0, 7, 3] = 0           # a query block keeping nothing: an empty dQ item
    mask[1, 11] = 1             # a dense head: the longest lists
    g = _full_check(sa2, cfg, x, mask)
    assert not g[0][0, 3].any() and not g[1][0, 3].any() and not g[2][0, 3].any()
    assert not g[1][1, 5, 4 * 64:6 * 64].any() and not g[2][1, 5, 4 * 64:6 * 64].any()
    assert not g[0][0, 7, 3 * bq:4 * bq].any()
    g2 = _run(sa2, cfg, x, mask)
    for a, b in zip(g, g2):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_bwd_with_forward_workspace_is_bit_identical(sa2, dtype):
    """sa2_attn_bwd_with_fwd_ws takes the forward's fp16 copy of v (and of q, k for fp32
    inputs) instead of converting again: the gradients must equal sa2_attn_bwd's bit for bit."""
    cfg, x = small_case(f"fwd-ws-{dtype}", 1, 3, 1500, 128, dtype, 128, 64, seed=67)
    mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, 0.2, 0.6)["mask"]
    q, k, v, do = (to_device(x[t]) for t in ("q", "k", "v", "do"))
    bm = blockmask_from_oracle(mask)
    lib = sa2.load_library()
    import ctypes
    shp = sa2.make_shape(q, cfg.bq, cfg.bk)
    ws_f = sa2.workspace(lib.sa2_fwd_workspace_size(ctypes.byref(shp)), q.device)
    o_lo = torch.empty_like(q) if q.dtype == torch.bfloat16 else None
    o, lse = sa2.attn_fwd(q, k, v, bm, bq=cfg.bq, bk=cfg.bk, o_lo=o_lo, ws=ws_f)
    plain = sa2.attn_bwd(q, k, v, o, lse, do, bm, bq=cfg.bq, bk=cfg.bk, o_lo=o_lo)
    reused = sa2.attn_bwd(q, k, v, o, lse, do, bm, bq=cfg.bq, bk=cfg.bk, o_lo=o_lo, fwd_ws=ws_f)
    sa2.check_device()
    for name, a, b in zip(("dQ", "dK", "dV"), plain, reused):
        assert torch.equal(a, b), name


def test_bwd_gradient_invariants_on_gpu(sa2):
    """Every row of dS sums to zero and every row of P to one: the keys' dK sum to ~0 and
    the keys' dV sum to the queries' dO (rows that keep something)."""
    cfg, x = small_case("invariants", 1, 2, 1024, 128, "bf16", 128, 64, seed=13)
    mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, 0.25, 0.5)["mask"]
    dq, dk, dv = _run(sa2, cfg, x, mask)
    do = O.to_f64(x["do"])
    for h in range(cfg.H):
        assert np.abs(dk[0, h].sum(axis=0)).max() < 0.1
        np.testing.assert_allclose(dv[0, h].sum(axis=0), do[0, h].sum(axis=0), atol=0.25, rtol=2e-2)


def _sampled_check(sa2, cfg, x, mask, heads, rows, key_blocks):
    dq, dk, dv = _run(sa2, cfg, x, mask)
    for (b, h) in heads:
        q, k, v, do = (O.to_f64(x[t][b, h]) for t in ("q", "k", "v", "do"))
        rdq = O.attn_bwd_dq_rows(q, k, v, do, mask[b, h], cfg.bq, cfg.bk, rows)
        assert_close(f"{cfg.name} h{h} dQ rows", dq[b, h, rows], rdq)
        cols = np.concatenate([np.arange(j * cfg.bk, min(cfg.N, (j + 1) * cfg.bk)) for j in key_blocks])
        rdk, rdv = O.attn_bwd_dkdv_cols(q, k, v, do, mask[b, h], cfg.bq, cfg.bk, cols)
        assert_close(f"{cfg.name} h{h} dK cols", dk[b, h, cols], rdk)
        assert_close(f"{cfg.name} h{h} dV cols", dv[b, h, cols], rdv)


def test_bwd_mask_probe_config_sampled(sa2):
    cfg = CONFIGS[1]
    x = make_inputs(cfg)
    mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, 0.05, 0.9)["mask"]
    rows = np.concatenate([np.arange(0, 130), np.arange(cfg.N - 130, cfg.N)])
    _sampled_check(sa2, cfg, x, mask, [(0, 0), (0, 5)], rows, [0, 1, 63, cfg.Tk - 1])


def test_bwd_longest_sequence_sampled(sa2):
    """The longest sequence the library accepts (N = 491520 tokens: 3840 query blocks, 7680
    key blocks), d = 64, with a Top-k-only mask of 39 blocks per row: long lists, the largest
    pair-union bitmaps and 64-bit offsets.  Sampled query rows, and two key blocks away from
    the sink (whose column holds every row), recomputed by the oracle."""
    cfg, x = small_case("longest", 1, 1, 7680 * 64, 64, "bf16", 128, 64, seed=53)
    mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, 0.005, 0.0)["mask"]
    assert int(mask[0, 0].sum(axis=1).max()) == 39
    rows = np.concatenate([np.arange(0, 64), np.arange(cfg.N // 2, cfg.N // 2 + 32), np.arange(cfg.N - 64, cfg.N)])
    _sampled_check(sa2, cfg, x, mask, [(0, 0)], rows, [cfg.Tk // 2, cfg.Tk - 1])


@pytest.mark.parametrize("ci", [None, 1])
def test_bwd_without_forward_residual(sa2, ci):
    """sa2_attn_bwd with o_lo = NULL (the call a caller makes with only O from the forward)
    must meet the same bar: on ragged small cases and on every row of the mask-probe sink
    heads, where one block holds > 90 % of each row's mass and dS = P (dP - D) cancels."""
    if ci is None:
        cfg, x = small_case("no-residual", 1, 2, 1000, 128, "bf16", 128, 64, seed=71)
        mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, 0.2, 0.6)["mask"]
        heads = [(0, 0), (0, 1)]
    else:
        cfg = CONFIGS[ci]
        x = make_inputs(cfg)
        mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, 0.05, 0.9)["mask"]
        heads = [(0, 4), (0, 6)]
    q, k, v, do = (to_device(x[t]) for t in ("q", "k", "v", "do"))
    bm = blockmask_from_oracle(mask)
    o, lse = sa2.attn_fwd(q, k, v, bm, bq=cfg.bq, bk=cfg.bk)
    dq, dk, dv = sa2.attn_bwd(q, k, v, o, lse, do, bm, bq=cfg.bq, bk=cfg.bk)
    sa2.check_device()
    g = (to_f64(dq), to_f64(dk), to_f64(dv))
    for (b, h) in heads:
        hx = {t: x[t][b:b + 1, h:h + 1] for t in x}
        ref = O.attn_bwd(hx["q"], hx["k"], hx["v"], hx["do"], mask[b:b + 1, h:h + 1], cfg.bq, cfg.bk)
        for name, got, want in zip(("dQ", "dK", "dV"), g, ref):
            assert_close(f"{cfg.name} no o_lo h{h} {name}", got[b, h], want[0, 0])
