"""Diagnostics of a built block mask, off the attention path: per-row kept block counts and
kept pooled mass, and their per-head histograms.

They show the two failure modes that motivate the hybrid rule (gist.science explainer,
section 1; the Top-k-only and Top-p-only rows of the ablation, thelatestinai.com page,
Table 6). Top-k keeps a fixed share of the blocks, so on a flat pooled row it keeps little of
the row's mass. Top-p keeps the smallest set that reaches mass p, so on a row dominated by a
sink block it keeps very few blocks. The kept mass needs a mask built with
``want_mask=True, want_pooled=True``.

These are plain PyTorch reductions over the mask's own tensors, on whatever device they live.
"""
from typing import Dict

import torch

from .sa2 import BlockMask


def head_histograms(values: torch.Tensor, bins: int = 10) -> torch.Tensor:
    """Counts of [..., R] values in [0, 1] over `bins` equal bins per leading index.

    Bin i holds [i / bins, (i + 1) / bins); the last bin also holds 1.  Values outside
    [0, 1] are clamped into the end bins.  Returns [..., bins] int64."""
    if bins < 1:
        raise ValueError("bins must be >= 1")
    idx = torch.clamp(torch.floor(values.to(torch.float64) * bins).to(torch.int64), 0, bins - 1)
    counts = torch.zeros(values.shape[:-1] + (bins,), dtype=torch.int64, device=values.device)
    counts.scatter_add_(-1, idx, torch.ones_like(idx))
    return counts


def mask_diagnostics(mask: BlockMask, bins: int = 10) -> Dict[str, torch.Tensor]:
    """Per-row statistics of a block mask and their per-head histograms.

    Returns:
      kept            [B, H, Tq] int64    kept key blocks per query block (row_cnt)
      kept_frac       [B, H, Tq] float64  kept / Tk
      kept_frac_hist  [B, H, bins] int64
    and, when the mask carries its u8 mask and pooled probabilities:
      kept_mass       [B, H, Tq] float64  sum of the pooled probabilities of the kept blocks
      kept_mass_hist  [B, H, bins] int64
    """
    Tk = mask.row_idx.shape[-1]
    kept = mask.row_cnt.to(torch.int64)
    out = {"kept": kept, "kept_frac": kept.to(torch.float64) / Tk}
    out["kept_frac_hist"] = head_histograms(out["kept_frac"], bins)
    if mask.mask is not None and mask.pooled_p is not None:
        out["kept_mass"] = (mask.pooled_p.to(torch.float64) * mask.mask.to(torch.float64)).sum(-1)
        out["kept_mass_hist"] = head_histograms(out["kept_mass"], bins)
    return out
