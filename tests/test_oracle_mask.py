"""Pins of the oracle's masker (pooling, pooled softmax, hybrid Top-k U Top-p selection).

Each test checks the oracle against something other than itself: hand-worked rows,
closed forms, brute force over subsets, or an independent library routine."""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------------------ pooling

def test_pool_identical_tokens_pool_to_the_token():
    rng = np.random.default_rng(1)
    tok = rng.standard_normal((5, 7))
    x = np.repeat(tok, 4, axis=0)  # 5 blocks of 4 identical tokens
    np.testing.assert_allclose(O.pool_blocks(x, 4), tok, rtol=0, atol=1e-15)


def test_pool_linear_ramp_is_block_midpoint_with_partial_tail():
    N, b, d = 23, 5, 3  # blocks [0,5) ... [20,23): the last block holds 3 tokens
    alpha = np.array([0.5, -2.0, 3.25])
    beta = np.array([1.0, 0.0, -4.0])
    x = np.arange(N)[:, None] * alpha[None, :] + beta[None, :]
    got = O.pool_blocks(x, b)
    assert got.shape == (5, 3)
    for i in range(5):
        lo, hi = i * b, min(N, (i + 1) * b)
        mid = (lo + hi - 1) / 2.0  # mean index of the valid tokens only
        np.testing.assert_allclose(got[i], alpha * mid + beta, rtol=0, atol=1e-12)


def test_pool_tail_divides_by_valid_count():
    x = np.ones((10, 2))
    x[8:] = 3.0  # last block of b=4 holds tokens 8, 9 only
    got = O.pool_blocks(x, 4)
    np.testing.assert_allclose(got[2], [3.0, 3.0], rtol=0, atol=0)


# ----------------------------------------------------------------------- pooled softmax

def test_pooled_probs_are_distributions():
    rng = np.random.default_rng(2)
    P = O.pooled_probs(rng.standard_normal((9, 16)) * 3, rng.standard_normal((13, 16)) * 3)
    assert P.shape == (9, 13)
    assert (P >= 0).all()
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_pooled_probs_match_library_softmax():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    qb, kb = rng.standard_normal((6, 32)), rng.standard_normal((11, 32))
    ref = torch.softmax(torch.from_numpy(qb) @ torch.from_numpy(kb).T / math.sqrt(32), dim=1)
    np.testing.assert_allclose(O.pooled_probs(qb, kb), ref.numpy(), rtol=1e-12, atol=1e-15)


def test_pooled_probs_invariant_to_common_key_shift():
    # Adding one vector c to every pooled key adds q_i.c/sqrt(d) to a whole row of scores.
    rng = np.random.default_rng(4)
    qb, kb = rng.standard_normal((5, 8)), rng.standard_normal((7, 8))
    c = rng.standard_normal(8) * 10
    np.testing.assert_allclose(O.pooled_probs(qb, kb + c), O.pooled_probs(qb, kb), rtol=1e-9, atol=1e-14)


def test_pooled_scores_use_inverse_sqrt_d():
    # Two keys whose pooled scores differ by delta*sqrt(d)/sqrt(d) = delta: P ratio = e^delta.
    d = 16
    qb = np.zeros((1, d)); qb[0, 0] = 1.0
    kb = np.zeros((2, d)); kb[0, 0] = 2.0 * math.sqrt(d)
    P = O.pooled_probs(qb, kb)
    assert P[0, 0] / P[0, 1] == pytest.approx(math.exp(2.0), rel=1e-12)


# ------------------------------------------------------------------------- selection

def test_golden_hand_worked_rows():
    rows = json.load(open(os.path.join(GOLDEN, "hybrid_rows.json")))["rows"]
    for r in rows:
        P = np.array([r["P"]], dtype=np.float64)
        sel = O.hybrid_select(P, r["k"], r["p"])
        assert sel.K == r["K"], r["name"]
        assert int(sel.m[0]) == r["m"], r["name"]
        assert sel.mask[0].tolist() == r["mask"], r["name"]


@pytest.mark.parametrize("k,Tk,K", [(0.1, 16, 2), (0.05, 128, 7), (0.02, 128, 3), (0.25, 16, 4),
                                    (0.0, 16, 0), (1.0, 16, 16), (0.3, 10, 3), (0.05, 1182, 60),
                                    (0.02, 512, 11), (1.5, 8, 8), (-0.5, 8, 0)])
def test_topk_count_is_ceil_of_fraction(k, Tk, K):
    assert O.topk_count(k, Tk) == K


def _brute_rank(P):
    """rank_j = number of entries ordered before j (larger, or equal with a lower index)."""
    n = len(P)
    return np.array([sum(1 for i in range(n) if P[i] > P[j] or (P[i] == P[j] and i < j))
                     for j in range(n)])


def _brute_topp_size(P, p):
    """Smallest cardinality of any subset whose mass reaches p (enumerates all subsets)."""
    n = len(P)
    if p <= 0:
        return 0
    if p >= 1:
        return n
    for size in range(1, n + 1):
        best = max(math.fsum(P[list(c)]) for c in itertools.combinations(range(n), size))
        if best >= p:
            return size
    return n


def _rows_for_bruteforce(rng, n_rows, Tk):
    out = []
    for r in range(n_rows):
        if r % 3 == 0:  # ties: values drawn from a small set
            e = rng.integers(1, 4, size=Tk).astype(np.float64)
        else:
            e = np.exp(rng.standard_normal(Tk) * (1 + r % 4))
        out.append(e / e.sum())
    return out


def test_union_of_independent_topk_and_topp_by_brute_force():
    rng = np.random.default_rng(5)
    checked = 0
    for Tk in (1, 2, 5, 8, 10):
        for P in _rows_for_bruteforce(rng, 12, Tk):
            for k in (0.0, 0.1, 0.3, 0.5):
                for p in (0.0, 0.3, 0.61, 0.9, 0.97):
                    sel = O.hybrid_select(P[None, :], k, p)
                    rank = _brute_rank(P)
                    K = O.topk_count(k, Tk)
                    topk_set = set(np.nonzero(rank < K)[0].tolist())
                    m = _brute_topp_size(P, p)
                    topp_set = set(np.nonzero(rank < m)[0].tolist())
                    assert int(sel.m[0]) == m
                    assert set(np.nonzero(sel.mask[0])[0].tolist()) == topk_set | topp_set
                    assert int(sel.mask[0].sum()) == max(K, m)
                    checked += 1
    assert checked > 1000


def test_topp_mass_reaches_p_and_is_minimal():
    rng = np.random.default_rng(6)
    P = np.exp(rng.standard_normal((200, 64)) * 2)
    P /= P.sum(axis=1, keepdims=True)
    for p in (0.3, 0.5, 0.9, 0.99):
        sel = O.hybrid_select(P, 0.0, p)
        for i in range(P.shape[0]):
            kept = P[i, sel.mask[i].astype(bool)]
            assert kept.sum() >= p - 1e-12
            # dropping the smallest kept entry falls below p
            assert kept.sum() - kept.min() < p


def test_k_one_keeps_every_block_and_p_one_keeps_every_block():
    rng = np.random.default_rng(7)
    P = np.exp(rng.standard_normal((20, 33)) * 4)
    P /= P.sum(axis=1, keepdims=True)
    assert O.hybrid_select(P, 1.0, 0.0).mask.all()
    assert O.hybrid_select(P, 0.0, 1.0).mask.all()


@pytest.mark.parametrize("Tk,k,p,s0", [(16, 0.1, 0.9, 9.0), (128, 0.05, 0.5, 12.0), (128, 0.02, 0.9, 8.0)])
def test_sink_row_closed_form(Tk, k, p, s0):
    # One block with logit s0 against Tk-1 zeros: P0 = e^s0 / (e^s0 + Tk - 1).
    qb = np.zeros((1, 4)); qb[0, 0] = 1.0
    kb = np.zeros((Tk, 4)); kb[0, 0] = s0 * 2.0  # sqrt(d) = 2
    P = O.pooled_probs(qb, kb)
    P0 = math.exp(s0) / (math.exp(s0) + Tk - 1)
    assert P[0, 0] == pytest.approx(P0, rel=1e-12)
    assert P0 >= p
    sel = O.hybrid_select(P, k, p)
    K = O.topk_count(k, Tk)
    assert int(sel.m[0]) == 1
    # kept = the sink plus, by the index tie-break among the equal zeros, blocks 1..K-1
    assert np.nonzero(sel.mask[0])[0].tolist() == list(range(max(K, 1)))


@pytest.mark.parametrize("Tk,p", [(16, 0.9), (128, 0.5), (128, 0.9), (50, 0.33), (1182, 0.61)])
def test_flat_row_closed_form(Tk, p):
    qb = np.zeros((3, 8))  # Q == 0: every pooled score is 0, P = 1/Tk exactly
    kb = np.random.default_rng(8).standard_normal((Tk, 8))
    P = O.pooled_probs(qb, kb)
    assert np.all(P == P[0, 0])
    m = math.ceil(p * Tk - 1e-9)  # smallest m with m/Tk >= p (p chosen off the grid of 1/Tk)
    for k in (0.0, 0.02, 0.2):
        sel = O.hybrid_select(P, k, p)
        L = max(O.topk_count(k, Tk), m)
        assert (sel.m == m).all()
        for i in range(3):
            assert np.nonzero(sel.mask[i])[0].tolist() == list(range(L))


def test_build_mask_on_inputs_and_lists_roundtrip():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 2, 300, 16))
    k = rng.standard_normal((1, 2, 300, 16))
    r = O.build_mask(q, k, 64, 32, 0.2, 0.6)
    assert r["mask"].shape == (1, 2, 5, 10)
    lists = O.mask_to_lists(r["mask"])
    for h in range(2):
        for i in range(5):
            n = lists["row_cnt"][0, h, i]
            assert lists["row_idx"][0, h, i, :n].tolist() == np.nonzero(r["mask"][0, h, i])[0].tolist()
            assert (lists["row_idx"][0, h, i, n:] == -1).all()
        for j in range(10):
            n = lists["col_cnt"][0, h, j]
            assert lists["col_idx"][0, h, j, :n].tolist() == np.nonzero(r["mask"][0, h, :, j])[0].tolist()
    # each head computed independently from its own pooled blocks
    one = O.build_mask_head(q[0, 1], k[0, 1], 64, 32, 0.2, 0.6)
    assert (one["mask"] == r["mask"][0, 1]).all()


def test_compare_mask_exempts_only_near_threshold_entries():
    P = np.array([[0.4, 0.3, 0.2000004, 0.1 - 0.0000004]])
    sel = O.hybrid_select(P, 0.0, 0.65)  # keeps {0, 1}; threshold values 0.3 and 0.2000004
    near = sel.mask.copy(); near[0, 2] = 1  # 0.2000004 is the largest dropped value
    ex, bad = O.compare_mask_head(P, sel, near)
    assert len(ex) == 1 and not bad
    far = sel.mask.copy(); far[0, 3] = 1  # 0.0999996 is 0.1 away from both thresholds
    ex, bad = O.compare_mask_head(P, sel, far)
    assert len(bad) == 1 and not ex
