"""Helpers of the GPU parity tests: uploading the seeded inputs, handing the oracle's mask
to the CUDA path, the parity bar, and the record of the errors every check measured.

Parity bar for attention outputs and gradients (bf16 results of an fp64 reference):
  * element-wise |delta| <= 2e-2 wherever |ref| < 8;
  * where |ref| >= 8, |delta| <= max(2e-2, one bf16 ulp of |ref|), i.e. 2^(floor(log2|ref|) - 7):
    a bf16 output of magnitude in [8, 16) is stored with spacing 1/16, so its rounding alone
    is up to 1/32 > 2e-2 and the flat bound cannot hold there;
  * sum|delta| / sum|ref| <= 5e-3 per tensor (the mean relative error, read as a ratio of
    sums so that entries near zero do not dominate).
Every check records its measured max |delta|, the worst ratio |delta| / bound and the mean
relative error; the session prints them (tests/conftest.py)."""
from __future__ import annotations

import json
import os
from typing import List, Optional, Sequence

import numpy as np
import torch

import oracle as O

MAX_ABS = 2e-2
MEAN_REL = 5e-3
ULP_FROM = 8.0  # |ref| from which one bf16 ulp exceeds the flat bound's reach
# Pooled probabilities within this distance of a row's selection threshold may be decided
# either way by two correct floating-point implementations.
NEAR_THRESHOLD = 1e-6
# A row's Top-p cut is ambiguous between two exact implementations only when the prefix
# mass at the cut lies this close to p (fp64 prefix sums of fp32 values against the
# library's 2^-60 fixed-point sums).
CUT_MASS_TOL = 1e-12

PARITY_LOG: List[dict] = []


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


def bound(ref: np.ndarray, max_abs: float = MAX_ABS) -> np.ndarray:
    """Element-wise bound on |delta|: max_abs below |ref| = 8, above it max(max_abs, one bf16
    ulp of |ref|)."""
    a = np.abs(ref)
    ulp = np.exp2(np.floor(np.log2(np.maximum(a, ULP_FROM))) - 7.0)
    return np.where(a < ULP_FROM, max_abs, np.maximum(max_abs, ulp))


def errors(got: np.ndarray, ref: np.ndarray, max_abs: float = MAX_ABS):
    """(max |delta|, max |delta| / bound, sum|delta| / sum|ref|)."""
    if got.size == 0:
        return 0.0, 0.0, 0.0
    d = np.abs(got - ref)
    denom = np.abs(ref).sum()
    return (float(d.max()), float((d / bound(ref, max_abs)).max()),
            float(d.sum() / denom) if denom > 0 else float(d.sum()))


def record(kind: str, name: str, **values):
    PARITY_LOG.append(dict(kind=kind, name=name, **values))
    path = os.environ.get("SA2_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(PARITY_LOG[-1]) + "\n")


def assert_close(name: str, got: np.ndarray, ref: np.ndarray, max_abs=MAX_ABS, mean_rel=MEAN_REL):
    mx, ratio, mr = errors(got, ref, max_abs)
    record("tensor", name, max_abs=mx, worst_over_bound=ratio, mean_rel=mr, bar_max_abs=max_abs,
           bar_mean_rel=mean_rel)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    assert ratio <= 1.0 and mr <= mean_rel, \
        f"{name}: max|d| {mx:.3e} ({ratio:.2f} of the bound {max_abs} / one bf16 ulp past |ref| 8), " \
        f"mean rel {mr:.3e} (<= {mean_rel})"
    return mx, mr


def check_lists_consistent(bm, B, H, Tq, Tk, heads: Optional[Sequence] = None):
    """The CUDA path's CSR / CSC lists must list exactly its own u8 mask, ascending."""
    mask = bm.mask.cpu().numpy().astype(bool)
    rc = bm.row_cnt.cpu().numpy()
    ri = bm.row_idx.cpu().numpy()
    cc = bm.col_cnt.cpu().numpy()
    ci = bm.col_idx.cpu().numpy()
    assert (rc == mask.sum(-1)).all()
    assert (cc == mask.sum(-2)).all()
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for (b, h) in todo:
        for i in range(Tq):
            n = rc[b, h, i]
            assert (ri[b, h, i, :n] == np.nonzero(mask[b, h, i])[0]).all()
        for j in range(Tk):
            n = cc[b, h, j]
            assert (ci[b, h, j, :n] == np.nonzero(mask[b, h, :, j])[0]).all()


def selection_under_own_probs(gP: np.ndarray, gmask: np.ndarray, topk: float, topp: float):
    """Checks that every row of the GPU's mask of one head is the hybrid selection of the
    GPU's OWN pooled probabilities: the oracle's selection rule applied to gP (fp32 values
    widened to fp64) must give the same row, bit for bit.  Kept count = max(K, m'), a prefix
    of gP's (descending, index-ascending) order, m' the shortest prefix whose mass reaches p.

    The only allowed difference: a row whose prefix mass at the Top-p cut lies within
    CUT_MASS_TOL of p, where m' may differ by one.  Returns (bad rows, ambiguous rows)."""
    P = np.asarray(gP, dtype=np.float32).astype(np.float64)
    sel = O.hybrid_select(P, float(np.float32(topk)), float(np.float32(topp)))
    diff = np.nonzero((sel.mask.astype(bool) != gmask.astype(bool)).any(axis=1))[0]
    bad, ambiguous = [], []
    cs = np.cumsum(sel.sorted_P, axis=1)
    Tk = P.shape[1]
    for i in diff.tolist():
        m = int(sel.m[i])
        near = any(0 <= c < Tk and abs(cs[i, c] - float(np.float32(topp))) <= CUT_MASS_TOL for c in (m - 2, m - 1, m))
        g = gmask[i].astype(bool)
        kept = np.nonzero(g)[0]
        # the GPU row must still be a prefix of gP's order, of length within one of L
        order = sel.order[i]
        prefix_ok = g[order[: kept.size]].all()
        if near and prefix_ok and abs(kept.size - int(sel.L[i])) <= 1:
            ambiguous.append(i)
        else:
            bad.append(i)
    return bad, ambiguous


def compare_masks(bm, ref, heads, topk: float, topp: float, label: str):
    """Mask parity of the GPU mask `bm` (with pooled_p) against the oracle's result `ref`
    on the listed heads:
      * P-bar within 5e-6 of the oracle's (fp32 accuracy);
      * every entry equal to the oracle's, except entries whose oracle P-bar lies within
        NEAR_THRESHOLD of the oracle row's threshold (exempt, logged);
      * every row -- exempt or not -- the exact hybrid selection of the GPU's own P-bar.
    Returns the exempt entries [(b, h, row, j, P_j, smallest kept, largest dropped)]."""
    gmask = bm.mask.cpu().numpy()
    gP = bm.pooled_p.cpu().numpy()
    exempt_all, n_rows, n_amb = [], 0, 0
    worst_p = 0.0
    for (b, h) in heads:
        P = ref["P"][b, h]
        dp = float(np.abs(gP[b, h] - P).max())
        worst_p = max(worst_p, dp)
        assert dp <= 5e-6, f"{label} head {(b, h)}: pooled probabilities differ by {dp:.2e}"
        exempt, bad = O.compare_mask_head(P, ref["sel"][(b, h)], gmask[b, h], NEAR_THRESHOLD)
        assert not bad, f"{label} head {(b, h)}: mask entries differ away from the threshold: {bad[:5]}"
        vbad, amb = selection_under_own_probs(gP[b, h], gmask[b, h], topk, topp)
        assert not vbad, f"{label} head {(b, h)}: rows {vbad[:8]} are not the hybrid selection of the GPU's own P-bar"
        n_amb += len(amb)
        n_rows += P.shape[0]
        exempt_all.extend([(b, h) + tuple(e) for e in exempt])
    record("mask", label, heads=len(heads), rows=n_rows, exempt_entries=len(exempt_all), ambiguous_cut_rows=n_amb,
           max_pbar_delta=worst_p, exempt=[list(map(float, e)) for e in exempt_all[:20]])
    # every exempt entry sits at its row's threshold, and such entries stay rare
    for e in exempt_all:
        _, _, _, _, pj, lo, hi = e
        assert (np.isfinite(lo) and abs(pj - lo) <= NEAR_THRESHOLD) or (np.isfinite(hi) and abs(pj - hi) <= NEAR_THRESHOLD)
    assert len(exempt_all) <= max(4, n_rows // 100), f"{label}: {len(exempt_all)} exempt entries in {n_rows} rows"
    return exempt_all


def sample_rows(cfg, n=64):
    """Query rows of the first, a middle and the (ragged) last query block."""
    mid = (cfg.Tq // 2) * cfg.bq
    return np.unique(np.concatenate([np.arange(0, n), np.arange(mid, mid + n),
                                     np.arange(max(0, cfg.N - n), cfg.N)]))


def _head_rows(t, b, h, idx):
    """Rows `idx` of head (b, h) of a device tensor [B, H, N(, d)] as float64 on the host."""
    x = t[b, h][torch.as_tensor(idx, device=t.device)]
    return x.double().cpu().numpy()


def sampled_attention_parity(cfg, x, mask, got, heads, rows, key_blocks, label, dkdv_heads=None):
    """O, LSE and dQ of the listed query rows, and dK, dV of the listed key blocks, of the
    listed heads, recomputed by the oracle one row / key at a time on `mask` (the mask the
    CUDA path ran with) and compared at the parity bar.  `got` holds the CUDA results as
    device tensors: o, lse, dq, dk, dv (any of them may be missing)."""
    cols = np.concatenate([np.arange(j * cfg.bk, min(cfg.N, (j + 1) * cfg.bk)) for j in key_blocks])
    for (b, h) in heads:
        q, k, v = (O.to_f64(x[t][b, h]) for t in ("q", "k", "v"))
        tag = f"{label} h{h}"
        if "o" in got:
            ro, rlse = O.attn_fwd_head(q, k, v, mask[b, h], cfg.bq, cfg.bk, rows=rows)
            assert_close(f"{tag} rows O", _head_rows(got["o"], b, h, rows), ro)
            lse = _head_rows(got["lse"], b, h, rows)
            fin = np.isfinite(rlse)
            assert (np.isneginf(lse) == ~fin).all(), f"{tag}: -inf LSE pattern differs"
            dl = float(np.abs(lse[fin] - rlse[fin]).max()) if fin.any() else 0.0
            record("tensor", f"{tag} rows LSE", max_abs=dl, worst_over_bound=dl / MAX_ABS, mean_rel=0.0,
                   bar_max_abs=MAX_ABS, bar_mean_rel=MEAN_REL)
            assert dl <= MAX_ABS, f"{tag} LSE {dl:.3e}"
        if "dq" not in got:
            continue
        do = O.to_f64(x["do"][b, h])
        rdq = O.attn_bwd_dq_rows(q, k, v, do, mask[b, h], cfg.bq, cfg.bk, rows)
        assert_close(f"{tag} rows dQ", _head_rows(got["dq"], b, h, rows), rdq)
        if dkdv_heads is not None and (b, h) not in dkdv_heads:
            continue
        rdk, rdv = O.attn_bwd_dkdv_cols(q, k, v, do, mask[b, h], cfg.bq, cfg.bk, cols)
        assert_close(f"{tag} cols dK", _head_rows(got["dk"], b, h, cols), rdk)
        assert_close(f"{tag} cols dV", _head_rows(got["dv"], b, h, cols), rdv)


def run_step_on_own_mask(sa2, cfg, dev, topk, topp, with_bwd=True, o_lo=True):
    """Mask, forward and backward on the GPU the way the benchmark runs them (the backward
    reusing the forward's workspace); returns (mask, dict of device results)."""
    import ctypes
    bm = sa2.build_mask(dev["q"], dev["k"], topk, topp, bq=cfg.bq, bk=cfg.bk, want_pooled=True)
    shp = sa2.make_shape(dev["q"], cfg.bq, cfg.bk)
    ws_f = sa2.workspace(sa2.load_library().sa2_fwd_workspace_size(ctypes.byref(shp)), dev["q"].device)
    lo = torch.empty_like(dev["q"]) if (o_lo and dev["q"].dtype == torch.bfloat16) else None
    o, lse = sa2.attn_fwd(dev["q"], dev["k"], dev["v"], bm, bq=cfg.bq, bk=cfg.bk, o_lo=lo, ws=ws_f)
    out = {"o": o, "lse": lse}
    if with_bwd:
        dq, dk, dv = sa2.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], bm, bq=cfg.bq, bk=cfg.bk,
                                  o_lo=lo, fwd_ws=ws_f)
        out.update(dq=dq, dk=dk, dv=dv)
    sa2.check_device()
    return bm, out
