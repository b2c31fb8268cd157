"""Planted mistakes in the oracle (on the CPU) must each fail at least one pin.

Every mutation below is a plausible slip: a dropped term, a wrong comparison, a swapped
index.  The test patches the oracle with the mistake, runs the pins that should catch
it, and requires one of them to fail."""
import math

import numpy as np
import pytest

import oracle
import oracle.sa2_oracle as S
from tests import test_oracle_attn as TA
from tests import test_oracle_mask as TM


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(S, name, fn)
    monkeypatch.setattr(oracle, name, fn)


def _fails(*pins):
    for pin in pins:
        try:
            pin()
        except AssertionError:
            return True
    return False


def _pool_divides_by_block_size(x, b):
    N, d = x.shape
    T = S.num_blocks(N, b)
    pad = np.zeros((T * b, d))
    pad[:N] = x
    return pad.reshape(T, b, d).sum(axis=1) / b


def _probs_without_scale(qbar, kbar):
    s = qbar @ kbar.T
    e = np.exp(s - s.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def _probs_without_normalisation(qbar, kbar):
    s = (qbar @ kbar.T) / math.sqrt(qbar.shape[1])
    return np.exp(s - s.max(axis=1, keepdims=True))


def _order_ties_high_index_first(P):
    Tk = P.shape[-1]
    rev = np.argsort(-P[..., ::-1], axis=-1, kind="stable")
    return Tk - 1 - rev


def _topp_strict(sorted_P, topp):
    Tk = sorted_P.shape[-1]
    if topp <= 0:
        return np.zeros(sorted_P.shape[:-1], dtype=np.int64)
    if topp >= 1:
        return np.full(sorted_P.shape[:-1], Tk, dtype=np.int64)
    cs = np.cumsum(sorted_P, axis=-1)
    return np.minimum((cs <= topp).sum(axis=-1) + 1, Tk)


def _topk_floor(topk, Tk):
    return int(min(max(math.floor(topk * Tk), 0), Tk))


def _hybrid_intersection(P, topk, topp):
    sel = S.RowSelection.__new__(S.RowSelection)
    P = np.atleast_2d(P)
    order = S.row_order(P)
    sP = np.take_along_axis(P, order, axis=1)
    K = S.topk_count(topk, P.shape[1])
    m = S.topp_count(sP, topp)
    L = np.minimum(K, m)
    mask = np.zeros(P.shape, dtype=np.uint8)
    np.put_along_axis(mask, order, (np.arange(P.shape[1])[None] < L[:, None]).astype(np.uint8), axis=1)
    sel.__init__(order=order, sorted_P=sP, K=K, m=m, L=L, mask=mask)
    return sel


def _token_mask_transposed(block_mask, N, bq, bk, rows=None):
    a = np.arange(N) if rows is None else np.asarray(rows)
    c = np.arange(N)
    bm = np.zeros((max(block_mask.shape) + 1,) * 2, dtype=block_mask.dtype)
    bm[: block_mask.shape[1], : block_mask.shape[0]] = block_mask.T
    return bm[a // bk][:, c // bq].astype(bool)


def _bwd_factory(kind):
    def bwd(q, k, v, do, block_mask, bq, bk, scale=None):
        N, d = k.shape
        scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
        allowed = S.token_mask(block_mask, N, bq, bk)
        P, _ = S._masked_softmax_rows((q @ k.T) * scale, allowed)
        o = P @ v
        dV = P.T @ do
        dP = do @ v.T
        D = (do * o).sum(axis=1)
        if kind == "no-D":
            dS = P * dP
        elif kind == "sign":
            dS = P * (D[:, None] - dP)
        else:
            dS = P * (dP - D[:, None])
        dQ = scale * (dS @ k)
        dK = (dS.T @ q) if kind == "dk-no-scale" else scale * (dS.T @ q)
        if kind == "dv-transposed":
            dV = (P @ do) if P.shape[0] == P.shape[1] else dV * 0
        return dQ, dK, dV
    return bwd


MASK_PINS = [TM.test_pool_linear_ramp_is_block_midpoint_with_partial_tail,
             TM.test_pool_tail_divides_by_valid_count,
             TM.test_pooled_probs_are_distributions,
             TM.test_pooled_scores_use_inverse_sqrt_d,
             TM.test_golden_hand_worked_rows,
             TM.test_union_of_independent_topk_and_topp_by_brute_force,
             TM.test_build_mask_on_inputs_and_lists_roundtrip]


@pytest.mark.parametrize("name,fn", [
    ("pool_blocks", _pool_divides_by_block_size),
    ("pooled_probs", _probs_without_scale),
    ("pooled_probs", _probs_without_normalisation),
    ("row_order", _order_ties_high_index_first),
    ("topp_count", _topp_strict),
    ("topk_count", _topk_floor),
    ("hybrid_select", _hybrid_intersection),
])
def test_masker_mutation_is_caught(monkeypatch, name, fn):
    _patch(monkeypatch, name, fn)
    assert _fails(*MASK_PINS, lambda: TM.test_topk_count_is_ceil_of_fraction(0.1, 16, 2))


def test_transposed_token_mask_is_caught(monkeypatch):
    _patch(monkeypatch, "token_mask", _token_mask_transposed)
    assert _fails(lambda: TA.test_forward_matches_brute_force_loops(1, 20, 8, 4),
                  TA.test_forward_matches_torch_sdpa_fp64)


@pytest.mark.parametrize("kind", ["no-D", "sign", "dk-no-scale", "dv-transposed"])
def test_backward_mutation_is_caught(monkeypatch, kind):
    _patch(monkeypatch, "attn_bwd_head", _bwd_factory(kind))
    assert _fails(TA.test_backward_matches_torch_autograd_fp64, TA.test_backward_invariants)


def _vd_loss_factory(kind):
    def vd_loss(o_student, o_teacher):
        diff = S.to_f64(o_student) - S.to_f64(o_teacher)
        if kind == "no-factor-2":
            return float(np.sum(diff * diff)), diff
        if kind == "sign":
            return float(np.sum(diff * diff)), -2.0 * diff
        return float(np.sum(np.abs(diff))), 2.0 * diff  # "l1-loss"
    return vd_loss


@pytest.mark.parametrize("kind", ["no-factor-2", "sign", "l1-loss"])
def test_distillation_mutation_is_caught(monkeypatch, kind):
    from tests import test_oracle_distill as TD
    _patch(monkeypatch, "vd_loss", _vd_loss_factory(kind))
    assert _fails(TD.test_loss_gradient_matches_central_differences,
                  TD.test_chain_matches_central_differences_with_teacher_frozen)


# ---- the sampled backward variants (full-size parity checks recompute chosen rows / keys)

def _kept_keys_ignoring_mask(block_mask_row, N, bk):
    return np.arange(N)


def _row_block_grads_without_D(q, k, v, do, keys, rows, scale):
    s = (q[rows] @ k[keys].T) * scale
    P, _ = S._masked_softmax_rows(s, np.ones_like(s, dtype=bool))
    return P, P * (do[rows] @ v[keys].T)


def _row_block_grads_unscaled(q, k, v, do, keys, rows, scale):
    s = q[rows] @ k[keys].T
    P, _ = S._masked_softmax_rows(s, np.ones_like(s, dtype=bool))
    o = P @ v[keys]
    D = (do[rows] * o).sum(axis=1)
    return P, P * (do[rows] @ v[keys].T - D[:, None])


@pytest.mark.parametrize("name,fn", [
    ("_kept_keys", _kept_keys_ignoring_mask),
    ("_row_block_grads", _row_block_grads_without_D),
    ("_row_block_grads", _row_block_grads_unscaled),
])
def test_sampled_backward_mutation_is_caught(monkeypatch, name, fn):
    monkeypatch.setattr(S, name, fn)
    assert _fails(TA.test_row_and_column_sampled_versions_equal_the_full_computation)


def _bwd_rows_without_D(q, k, v, do, block_mask, bq, bk, rows, scale=None):
    N, d = k.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rows = np.asarray(rows)
    allowed = S.token_mask(block_mask, N, bq, bk, rows)
    P, _ = S._masked_softmax_rows((q[rows] @ k.T) * scale, allowed)
    dS = P * (do[rows] @ v.T)
    return scale * (dS @ k), scale * (dS.T @ q[rows]), P.T @ do[rows]


def test_row_partition_mutation_is_caught(monkeypatch):
    _patch(monkeypatch, "attn_bwd_rows", _bwd_rows_without_D)
    assert _fails(TA.test_row_partition_of_the_backward_adds_up)
