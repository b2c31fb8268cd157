"""Helpers of the GPU parity tests: uploading the seeded inputs, handing the oracle's mask
to the CUDA path, and the error metrics of the parity bar."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

# Parity bar for bf16 attention outputs and gradients: max |delta| <= 2e-2 at unit scale,
# i.e. |delta| <= 2e-2 * max(1, |ref|) element by element (a bf16 result of magnitude >= 8
# is 0.03-0.06 per ulp, so a flat 2e-2 cannot hold there), and sum|delta| / sum|ref| <= 5e-3.
MAX_ABS = 2e-2
MEAN_REL = 5e-3
# Pooled probabilities within this distance of a row's selection threshold may be decided
# either way by two correct floating-point implementations.
NEAR_THRESHOLD = 1e-6


def to_device(x: np.ndarray, device="cuda") -> torch.Tensor:
    """Storage array (uint16 bf16 bits or float32) -> torch tensor on the device."""
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def blockmask_from_oracle(mask: np.ndarray, device="cuda"):
    """The oracle's u8 mask [B, H, Tq, Tk] as the compact lists the CUDA path reads."""
    from block_sparse_attention_sa2_gb300 import BlockMask
    lists = O.mask_to_lists(mask)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
    return BlockMask(t(lists["row_cnt"]), t(lists["row_idx"]), t(lists["col_cnt"]), t(lists["col_idx"]),
                     t(mask.astype(np.uint8)))


def errors(got: np.ndarray, ref: np.ndarray):
    """(max |d| / max(1, |ref|), sum|d| / sum|ref|)."""
    d = np.abs(got - ref)
    denom = np.abs(ref).sum()
    scaled = d / np.maximum(1.0, np.abs(ref))
    return float(scaled.max()) if d.size else 0.0, float(d.sum() / denom) if denom > 0 else float(d.sum())


def assert_close(name: str, got: np.ndarray, ref: np.ndarray, max_abs=MAX_ABS, mean_rel=MEAN_REL):
    mx, mr = errors(got, ref)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    assert mx <= max_abs and mr <= mean_rel, \
        f"{name}: max|d|/max(1,|ref|) {mx:.3e} (<= {max_abs}), mean rel {mr:.3e} (<= {mean_rel})"
    return mx, mr


def check_lists_consistent(bm, B, H, Tq, Tk):
    """The CUDA path's CSR / CSC lists must list exactly its own u8 mask, ascending."""
    mask = bm.mask.cpu().numpy().astype(bool)
    rc = bm.row_cnt.cpu().numpy()
    ri = bm.row_idx.cpu().numpy()
    cc = bm.col_cnt.cpu().numpy()
    ci = bm.col_idx.cpu().numpy()
    assert (rc == mask.sum(-1)).all()
    assert (cc == mask.sum(-2)).all()
    for b in range(B):
        for h in range(H):
            for i in range(Tq):
                n = rc[b, h, i]
                assert (ri[b, h, i, :n] == np.nonzero(mask[b, h, i])[0]).all()
            for j in range(Tk):
                n = cc[b, h, j]
                assert (ci[b, h, j, :n] == np.nonzero(mask[b, h, :, j])[0]).all()
