"""fp64 CPU oracle of the SpargeAttention2 hot path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline (its ``cpu_baseline`` leg and ``--impl reference`` arm) may import or run this
module.  The product path (the CUDA library under ``block_sparse_attention_sa2_gb300`` and
its Python binding) never imports it, and this module imports nothing from the product.
The two share only the seeded input generator in ``workload/``.

What it computes, and from where (pages on "SpargeAttention2: Trainable Sparse Attention
via Hybrid Top-k+Top-p Masking and Distillation Fine-Tuning", arXiv 2602.13515):

* gist.science explainer, section 2.A "Hybride Top-k + Top-p Maskierung": each row of the
  block-pooled attention map P-bar is masked; block j of row i is kept iff j is in the
  Top-k% set OR in the Top-p% set of that row (the union formula of that section).
* gist.science explainer, section 1 (problem statement): Top-k keeps the k largest
  entries; Top-p keeps the smallest set whose cumulative probability reaches p.
* gist.science explainer, section 2.C "Effiziente Kernel-Implementierung": the attention
  is FlashAttention-style block-sparse attention; masked blocks are skipped whole (their
  matmul and softmax are not computed), which equals dense softmax attention with the
  dropped blocks' scores at -inf.
* abstract (shd-paper.top, fugumt.com and thelatestinai.com pages), contribution (ii):
  the sparse attention is trainable, i.e. it has a backward pass; the backward below is
  the gradient of the masked softmax attention with the mask held fixed.
* gist.science explainer, section 2.B: the distillation loss, the squared L2 distance
  between sparse and full-attention outputs (a toy step on one attention block).

Readings where the pages are silent:

* pooling is the mean over the valid tokens of a block (the last block may be partial);
* pooled scores and token scores use the scale 1/sqrt(d) (token scale overridable);
* k is a fraction of the number of key blocks Tk: K = ceil(k*Tk - 1e-9), clamped to [0, Tk];
* the row order is P-bar descending, ties broken by the lower block index; Top-k and
  Top-p are both prefixes of that order, so their union is the prefix of length max(K, m);
* Top-p: m = the smallest m whose sorted prefix sum (fp64) is >= p; p <= 0 gives m = 0,
  p >= 1 gives m = Tk, and a prefix sum that never reaches p (rounding) gives m = Tk;
* attention is non-causal; a row with no kept block has O = 0, LSE = -inf and zero
  gradients; the mask receives no gradient.

Everything is numpy float64.  Functions take one head at a time ([N, d] arrays) unless
their name says otherwise; library primitives used as steps: matmul, exp/log, argsort
(stable), cumsum.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, Optional, Sequence

import numpy as np

TOPK_EPS = 1e-9


# ----------------------------------------------------------------------------- inputs

def to_f64(x: np.ndarray) -> np.ndarray:
    """Storage values -> float64.  uint16 arrays are bf16 bit patterns (widened exactly)."""
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def num_blocks(N: int, b: int) -> int:
    """Number of blocks of b tokens covering N tokens (the last one may be partial)."""
    return -(-N // b)


# ----------------------------------------------------------------------------- masker

def pool_blocks(x: np.ndarray, b: int) -> np.ndarray:
    """Block pooling (gist.science explainer, section 2.A): mean of each block of b tokens.

    x: [N, d] float64.  Returns [ceil(N/b), d]; the last block averages its valid tokens."""
    N, d = x.shape
    T = num_blocks(N, b)
    out = np.empty((T, d), dtype=np.float64)
    full = N // b
    if full:
        out[:full] = x[: full * b].reshape(full, b, d).mean(axis=1)
    if full < T:
        out[full] = x[full * b:].mean(axis=0)
    return out


def pooled_probs(qbar: np.ndarray, kbar: np.ndarray) -> np.ndarray:
    """P-bar = row softmax of qbar kbar^T / sqrt(d) (gist.science explainer, section 2.A)."""
    d = qbar.shape[1]
    s = (qbar @ kbar.T) / math.sqrt(d)
    s = s - s.max(axis=1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=1, keepdims=True)


def topk_count(topk: float, Tk: int) -> int:
    """K = ceil(k*Tk) for k a fraction of the key blocks ("Top-k%"), clamped to [0, Tk]."""
    K = math.ceil(float(topk) * Tk - TOPK_EPS)
    return int(min(max(K, 0), Tk))


def row_order(P: np.ndarray) -> np.ndarray:
    """Indices of each row sorted by P descending, equal values by ascending index."""
    return np.argsort(-P, axis=-1, kind="stable")


def topp_count(sorted_P: np.ndarray, topp: float) -> np.ndarray:
    """m = smallest prefix length of the sorted row whose mass reaches p (gist.science
    explainer, section 1: 'smallest set whose cumulative probability reaches p').

    sorted_P: [..., Tk] rows sorted descending.  Returns int64 [...]."""
    Tk = sorted_P.shape[-1]
    p = float(topp)
    if p <= 0.0:
        return np.zeros(sorted_P.shape[:-1], dtype=np.int64)
    if p >= 1.0:
        return np.full(sorted_P.shape[:-1], Tk, dtype=np.int64)
    cs = np.cumsum(sorted_P, axis=-1)
    below = (cs < p).sum(axis=-1)  # prefixes whose mass is still short of p
    return np.minimum(below + 1, Tk).astype(np.int64)


@dataclass
class RowSelection:
    order: np.ndarray  # [R, Tk] sorted order
    sorted_P: np.ndarray  # [R, Tk]
    K: int
    m: np.ndarray  # [R]
    L: np.ndarray  # [R] kept count = max(K, m)
    mask: np.ndarray  # [R, Tk] uint8


def hybrid_select(P: np.ndarray, topk: float, topp: float) -> RowSelection:
    """Hybrid mask of each row (gist.science explainer, section 2.A):
    M_ij = 1 iff j in Top-k(P_i, k%) U Top-p(P_i, p%).

    Both sets are prefixes of the same order, so the union is the prefix of length
    max(K, m)."""
    P = np.atleast_2d(P)
    R, Tk = P.shape
    order = row_order(P)
    sP = np.take_along_axis(P, order, axis=1)
    K = topk_count(topk, Tk)
    m = topp_count(sP, topp)
    L = np.maximum(K, m)
    mask = np.zeros((R, Tk), dtype=np.uint8)
    ranks = np.arange(Tk)[None, :]
    keep_sorted = ranks < L[:, None]
    np.put_along_axis(mask, order, keep_sorted.astype(np.uint8), axis=1)
    return RowSelection(order=order, sorted_P=sP, K=K, m=m, L=L, mask=mask)


def build_mask_head(q: np.ndarray, k: np.ndarray, bq: int, bk: int, topk: float,
                    topp: float) -> Dict[str, np.ndarray]:
    """Mask of one head: pooled P-bar, the hybrid selection and the kept-block mask."""
    qbar = pool_blocks(q, bq)
    kbar = pool_blocks(k, bk)
    P = pooled_probs(qbar, kbar)
    sel = hybrid_select(P, topk, topp)
    return {"qbar": qbar, "kbar": kbar, "P": P, "sel": sel, "mask": sel.mask}


def build_mask(q: np.ndarray, k: np.ndarray, bq: int, bk: int, topk: float, topp: float,
               heads: Optional[Sequence] = None) -> Dict[str, object]:
    """Masks of [B, H, N, d] inputs (storage form or float64).

    Returns the uint8 mask [B, H, Tq, Tk], P-bar [B, H, Tq, Tk] and the per-head
    selections; heads not listed in ``heads`` are left empty."""
    B, H, N, _ = q.shape
    Tq, Tk = num_blocks(N, bq), num_blocks(N, bk)
    mask = np.zeros((B, H, Tq, Tk), dtype=np.uint8)
    P = np.zeros((B, H, Tq, Tk), dtype=np.float64)
    sels = {}
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for (b, h) in todo:
        r = build_mask_head(to_f64(q[b, h]), to_f64(k[b, h]), bq, bk, topk, topp)
        mask[b, h] = r["mask"]
        P[b, h] = r["P"]
        sels[(b, h)] = r["sel"]
    return {"mask": mask, "P": P, "sel": sels}


def mask_to_lists(mask: np.ndarray) -> Dict[str, np.ndarray]:
    """Compact lists of a block mask [..., Tq, Tk]: row counts / ascending kept key blocks
    (CSR, padded with -1 to Tk) and column counts / ascending query blocks (CSC, padded to
    Tq).  Used to hand the oracle's mask to the CUDA path."""
    Tq, Tk = mask.shape[-2:]
    lead = mask.shape[:-2]
    m2 = mask.reshape(-1, Tq, Tk).astype(bool)
    row_cnt = m2.sum(axis=2).astype(np.int32)
    col_cnt = m2.sum(axis=1).astype(np.int32)
    row_idx = np.full((m2.shape[0], Tq, Tk), -1, dtype=np.int32)
    col_idx = np.full((m2.shape[0], Tk, Tq), -1, dtype=np.int32)
    for g in range(m2.shape[0]):
        for i in range(Tq):
            js = np.nonzero(m2[g, i])[0]
            row_idx[g, i, : js.size] = js
        for j in range(Tk):
            is_ = np.nonzero(m2[g, :, j])[0]
            col_idx[g, j, : is_.size] = is_
    return {"row_cnt": row_cnt.reshape(*lead, Tq), "row_idx": row_idx.reshape(*lead, Tq, Tk),
            "col_cnt": col_cnt.reshape(*lead, Tk), "col_idx": col_idx.reshape(*lead, Tk, Tq)}


# -------------------------------------------------------------------------- attention

def token_mask(block_mask: np.ndarray, N: int, bq: int, bk: int,
               rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Token-level allowed[a, c] = block_mask[a // bq, c // bk] (blocks kept or skipped whole,
    gist.science explainer, section 2.C)."""
    a = np.arange(N) if rows is None else np.asarray(rows)
    c = np.arange(N)
    return block_mask[a // bq][:, c // bk].astype(bool)


def _masked_softmax_rows(s: np.ndarray, allowed: np.ndarray):
    """Row softmax over allowed entries; returns (P, LSE).  Rows with nothing allowed get
    P = 0 and LSE = -inf."""
    s = np.where(allowed, s, -np.inf)
    mx = s.max(axis=1)
    has = np.isfinite(mx)
    mx_safe = np.where(has, mx, 0.0)
    e = np.where(allowed, np.exp(s - mx_safe[:, None]), 0.0)
    z = e.sum(axis=1)
    lse = np.where(has, mx_safe + np.log(np.where(has, z, 1.0)), -np.inf)
    P = np.where(has[:, None], e / np.where(has, z, 1.0)[:, None], 0.0)
    return P, lse


def attn_fwd_head(q, k, v, block_mask, bq, bk, scale=None, rows=None):
    """Block-sparse attention forward of one head (gist.science explainer, section 2.C):
    O_a = sum over allowed c of softmax_c(q_a . k_c * scale) v_c, LSE_a = log sum exp.

    q, k, v: [N, d] float64; block_mask: [Tq, Tk].  ``rows`` limits the query rows.
    Returns (O [R, d], LSE [R])."""
    N, d = k.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    qa = q if rows is None else q[np.asarray(rows)]
    allowed = token_mask(block_mask, N, bq, bk, rows)
    s = (qa @ k.T) * scale
    P, lse = _masked_softmax_rows(s, allowed)
    return P @ v, lse


def attn_bwd_head(q, k, v, do, block_mask, bq, bk, scale=None):
    """Gradient of the block-sparse attention of one head, mask held fixed.

    With P = softmax of the masked scores: dV = P^T dO, dP = dO V^T, D_a = dO_a . O_a,
    dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q.  Returns (dQ, dK, dV)."""
    N, d = k.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    allowed = token_mask(block_mask, N, bq, bk)
    P, _ = _masked_softmax_rows((q @ k.T) * scale, allowed)
    o = P @ v
    dV = P.T @ do
    dP = do @ v.T
    D = (do * o).sum(axis=1)
    dS = P * (dP - D[:, None])
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q)
    return dQ, dK, dV


def _kept_keys(block_mask_row: np.ndarray, N: int, bk: int) -> np.ndarray:
    """Token indices of the key blocks one query block keeps (ascending)."""
    blocks = np.nonzero(block_mask_row)[0]
    if blocks.size == 0:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([np.arange(j * bk, min(N, (j + 1) * bk)) for j in blocks])


def _row_block_grads(q, k, v, do, keys, rows, scale):
    """Softmax, D and dS of the query rows of one query block over its kept keys only.

    Entries of dropped blocks have P = 0 in the masked softmax (gist.science explainer,
    section 2.C: skipped tiles are not computed), so restricting each row to its kept keys
    gives the same P, O, D and dS as masking the full row.  Returns (P, dS) over ``keys``."""
    s = (q[rows] @ k[keys].T) * scale
    P, _ = _masked_softmax_rows(s, np.ones_like(s, dtype=bool))
    o = P @ v[keys]
    D = (do[rows] * o).sum(axis=1)
    dS = P * (do[rows] @ v[keys].T - D[:, None])
    return P, dS


def attn_bwd_dq_rows(q, k, v, do, block_mask, bq, bk, rows, scale=None):
    """dQ of the listed query rows only (same definition as ``attn_bwd_head``), each row
    computed over the key blocks its query block keeps."""
    N, d = k.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rows = np.asarray(rows)
    dQ = np.zeros((rows.size, d))
    for i in np.unique(rows // bq):
        sel = np.nonzero(rows // bq == i)[0]
        keys = _kept_keys(block_mask[i], N, bk)
        if keys.size == 0:
            continue  # a row that keeps nothing has zero gradients
        _, dS = _row_block_grads(q, k, v, do, keys, rows[sel], scale)
        dQ[sel] = scale * (dS @ k[keys])
    return dQ


def attn_bwd_rows(q, k, v, do, block_mask, bq, bk, rows, scale=None):
    """The backward restricted to the listed query rows: their dQ rows, and their
    contributions to dK and dV (the gradient is a sum over query rows, so contributions of
    a partition of the rows add up to the full dK, dV).  Returns (dQ_rows, dK_part, dV_part)."""
    N, d = k.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rows = np.asarray(rows)
    allowed = token_mask(block_mask, N, bq, bk, rows)
    P, _ = _masked_softmax_rows((q[rows] @ k.T) * scale, allowed)
    o = P @ v
    dP = do[rows] @ v.T
    D = (do[rows] * o).sum(axis=1)
    dS = P * (dP - D[:, None])
    return scale * (dS @ k), scale * (dS.T @ q[rows]), P.T @ do[rows]


def attn_bwd_dkdv_cols(q, k, v, do, block_mask, bq, bk, cols, scale=None):
    """dK and dV of the listed key tokens only: the sum over every query block that keeps
    one of these keys, each block's rows computed over the key blocks it keeps."""
    N, d = k.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    cols = np.asarray(cols)
    dK = np.zeros((cols.size, d))
    dV = np.zeros((cols.size, d))
    col_blocks = np.unique(cols // bk)
    for i in np.nonzero(block_mask[:, col_blocks].any(axis=1))[0]:
        rows = np.arange(i * bq, min(N, (i + 1) * bq))
        keys = _kept_keys(block_mask[i], N, bk)
        P, dS = _row_block_grads(q, k, v, do, keys, rows, scale)
        pos = np.searchsorted(keys, cols)  # where each listed key sits among the kept ones
        hit = (pos < keys.size) & (keys[np.minimum(pos, keys.size - 1)] == cols)
        if not hit.any():
            continue
        Pc, dSc = P[:, pos[hit]], dS[:, pos[hit]]
        dV[hit] += Pc.T @ do[rows]
        dK[hit] += scale * (dSc.T @ q[rows])
    return dK, dV


def attn_fwd(q, k, v, block_mask, bq, bk, scale=None):
    """Forward over [B, H, N, d] inputs; returns (O, LSE) as float64 arrays."""
    B, H, N, d = q.shape
    O = np.zeros((B, H, N, d))
    LSE = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            O[b, h], LSE[b, h] = attn_fwd_head(to_f64(q[b, h]), to_f64(k[b, h]), to_f64(v[b, h]),
                                               block_mask[b, h], bq, bk, scale)
    return O, LSE


def attn_bwd(q, k, v, do, block_mask, bq, bk, scale=None):
    """Backward over [B, H, N, d] inputs; returns (dQ, dK, dV) as float64 arrays."""
    B, H, N, d = q.shape
    out = [np.zeros((B, H, N, d)) for _ in range(3)]
    for b in range(B):
        for h in range(H):
            g = attn_bwd_head(to_f64(q[b, h]), to_f64(k[b, h]), to_f64(v[b, h]),
                              to_f64(do[b, h]), block_mask[b, h], bq, bk, scale)
            for t, x in zip(out, g):
                t[b, h] = x
    return tuple(out)


# ---------------------------------------------------------------- distillation (toy)

def vd_loss(o_student, o_teacher):
    """Velocity-distillation loss of one attention block and its gradient.

    gist.science explainer, section 2.B "Geschwindigkeits-Destillation": the fine-tuning
    loss is the squared L2 distance between the velocity predicted by the sparse model and
    by the frozen full-attention model.  On a single attention block the block's output
    stands in for the velocity:
        L = sum over all elements of (O_s - O_t)^2,    dL/dO_s = 2 (O_s - O_t),
    with the teacher O_t held fixed.  Returns (L, dL/dO_s) in float64."""
    diff = to_f64(o_student) - to_f64(o_teacher)
    return float(np.sum(diff * diff)), 2.0 * diff


def distill_step(q, k, v, student_mask, teacher_mask, bq, bk, scale=None):
    """One toy distillation step: teacher forward (full attention, or any mask), student
    forward under the sparse mask, the loss above, and the student's backward with
    dO = dL/dO_s.  Returns (L, dO, dQ, dK, dV) in float64."""
    o_t, _ = attn_fwd(q, k, v, teacher_mask, bq, bk, scale)
    o_s, _ = attn_fwd(q, k, v, student_mask, bq, bk, scale)
    loss, do = vd_loss(o_s, o_t)
    dq, dk, dv = attn_bwd(q, k, v, do, student_mask, bq, bk, scale)
    return loss, do, dq, dk, dv


# --------------------------------------------------------------------- mask comparison

def compare_mask_head(P: np.ndarray, sel: RowSelection, other: np.ndarray, tol: float = 1e-6):
    """Compare another implementation's mask of one head ([Tq, Tk]) with the oracle's.

    A differing entry is exempt when its pooled probability lies within ``tol`` of the
    oracle row's selection threshold (the smallest kept or the largest dropped value):
    there two correct floating-point implementations may decide either way.
    Returns (exempt, bad): lists of (row, j, P_j, smallest_kept, largest_dropped)."""
    exempt, bad = [], []
    diff_rows, diff_cols = np.nonzero(other.astype(bool) != sel.mask.astype(bool))
    Tk = P.shape[1]
    for i, j in zip(diff_rows.tolist(), diff_cols.tolist()):
        L = int(sel.L[i])
        lo = float(sel.sorted_P[i, L - 1]) if L > 0 else float("nan")
        hi = float(sel.sorted_P[i, L]) if L < Tk else float("nan")
        pj = float(P[i, j])
        near = (L > 0 and abs(pj - lo) <= tol) or (L < Tk and abs(pj - hi) <= tol)
        (exempt if near else bad).append((i, j, pj, lo, hi))
    return exempt, bad
