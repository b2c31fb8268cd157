"""Failure detection of the CUDA path, tested without faulting the GPU.

* Timeouts: every wait inside the attention kernels is bounded.  A test hook
  (sa2_debug_set_wait_limit) lowers the limit to 2 ms and makes the row warps of each
  kernel's first CTA sleep 200 ms, so the waits on them expire: the CTA must leave its loops,
  drain what it issued, free its tensor memory and report SA2_ERR_TIMEOUT -- and the context
  must stay usable: the same call repeated with the default limit is correct.
* Corrupted block lists (an index or a count out of range, made on the host): the kernels
  clamp what they read, report SA2_ERR_DEVICE_BOUNDS and produce finite outputs.
* An input beyond the fp16 range: saturated and reported as SA2_ERR_RANGE."""
import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_util import assert_close, blockmask_from_oracle, to_device, to_f64
from workload.gen import small_case

pytestmark = pytest.mark.gpu

TIMEOUT, BOUNDS, RANGE = 6, 7, 8


@pytest.fixture(scope="module")
def sa2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_attention_sa2_gb300 as m
    m.load_library()
    m.device_status()  # start from a clear status word
    yield m
    m.debug_set_wait_limit(0, 0)


@pytest.fixture(scope="module")
def case():
    cfg, x = small_case("failure", 1, 4, 1000, 128, "bf16", 128, 64, seed=81)
    mask = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, 0.3, 0.6)["mask"]
    return cfg, x, mask


def _fwd_bwd(sa2, cfg, dev, bm):
    o_lo = torch.empty_like(dev["q"])
    o, lse = sa2.attn_fwd(dev["q"], dev["k"], dev["v"], bm, bq=cfg.bq, bk=cfg.bk, o_lo=o_lo)
    g = sa2.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], bm, bq=cfg.bq, bk=cfg.bk, o_lo=o_lo)
    return o, lse, g


def _parity(cfg, x, mask, o, g):
    ro, _ = O.attn_fwd(x["q"], x["k"], x["v"], mask, cfg.bq, cfg.bk)
    rg = O.attn_bwd(x["q"], x["k"], x["v"], x["do"], mask, cfg.bq, cfg.bk)
    assert_close("after failure O", to_f64(o), ro)
    for name, got, want in zip(("dQ", "dK", "dV"), g, rg):
        assert_close(f"after failure {name}", to_f64(got), want)


@pytest.mark.parametrize("which", ["fwd", "bwd"])
def test_expired_wait_reports_timeout_and_the_context_survives(sa2, case, which):
    cfg, x, mask = case
    dev = {t: to_device(x[t]) for t in x}
    bm = blockmask_from_oracle(mask)
    if which == "bwd":
        o_lo = torch.empty_like(dev["q"])
        o, lse = sa2.attn_fwd(dev["q"], dev["k"], dev["v"], bm, bq=cfg.bq, bk=cfg.bk, o_lo=o_lo)
        assert sa2.device_status() == 0
    sa2.debug_set_wait_limit(2_000_000, 200_000_000)
    try:
        if which == "fwd":
            sa2.attn_fwd(dev["q"], dev["k"], dev["v"], bm, bq=cfg.bq, bk=cfg.bk)
        else:
            sa2.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], bm, bq=cfg.bq, bk=cfg.bk, o_lo=o_lo)
        status = sa2.device_status()
    finally:
        sa2.debug_set_wait_limit(0, 0)
    assert status == TIMEOUT, f"status {status} after an expired wait"
    # the context is usable and the same calls are correct again
    o, lse, g = _fwd_bwd(sa2, cfg, dev, bm)
    assert sa2.device_status() == 0
    _parity(cfg, x, mask, o, g)


def test_out_of_range_block_lists_are_clamped_and_reported(sa2, case):
    cfg, x, mask = case
    dev = {t: to_device(x[t]) for t in x}
    lists = O.mask_to_lists(mask)
    for field, where, value in (("row_idx", (0, 1, 2, 0), cfg.Tk + 5), ("row_idx", (0, 2, 0, 1), -3),
                                ("row_cnt", (0, 3, 1), cfg.Tk + 7), ("col_idx", (0, 0, 3, 0), cfg.Tq + 2),
                                ("col_cnt", (0, 1, 5), -4)):
        bad = {k: v.copy() for k, v in lists.items()}
        bad[field][where] = value
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        bm = sa2.BlockMask(t(bad["row_cnt"]), t(bad["row_idx"]), t(bad["col_cnt"]), t(bad["col_idx"]))
        o, lse, g = _fwd_bwd(sa2, cfg, dev, bm)
        status = sa2.device_status()
        assert status == BOUNDS, f"{field}{where} = {value}: status {status}"
        for name, tns in (("O", o), ("dQ", g[0]), ("dK", g[1]), ("dV", g[2])):
            assert torch.isfinite(tns.float()).all(), f"{field}: {name} not finite"
    # untouched lists: no error, and the results are right
    o, lse, g = _fwd_bwd(sa2, cfg, dev, blockmask_from_oracle(mask))
    assert sa2.device_status() == 0
    _parity(cfg, x, mask, o, g)


def test_input_beyond_fp16_range_is_saturated_and_reported(sa2, case):
    cfg, x, mask = case
    dev = {t: to_device(x[t]) for t in x}
    dev["v"][0, 1, 17, 5] = 1.0e5  # representable in bf16, not in fp16
    o, _ = sa2.attn_fwd(dev["q"], dev["k"], dev["v"], blockmask_from_oracle(mask), bq=cfg.bq, bk=cfg.bk)
    assert sa2.device_status() == RANGE
    assert torch.isfinite(o.float()).all()
