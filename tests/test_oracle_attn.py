"""Pins of the oracle's block-sparse attention forward and backward.

The forward is pinned by brute-force loops, per-block dense attention under a
block-diagonal mask, and torch's fp64 scaled-dot-product attention; the backward by
central finite differences, torch autograd in fp64 and two exact invariants."""
import math

import numpy as np
import pytest

import oracle as O


def _rand_case(seed, N=24, d=8, bq=8, bk=4, density=0.5, nonempty=True):
    rng = np.random.default_rng(seed)
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    Tq, Tk = O.num_blocks(N, bq), O.num_blocks(N, bk)
    mask = (rng.random((Tq, Tk)) < density).astype(np.uint8)
    if nonempty:
        for i in range(Tq):
            if not mask[i].any():
                mask[i, rng.integers(Tk)] = 1
    return q, k, v, do, mask


def _brute_fwd(q, k, v, mask, bq, bk, scale):
    N, d = q.shape
    O_ = np.zeros((N, d))
    lse = np.full(N, -np.inf)
    for a in range(N):
        logits = []
        for c in range(N):
            if mask[a // bq, c // bk]:
                logits.append((c, scale * sum(q[a, t] * k[c, t] for t in range(d))))
        if not logits:
            continue
        mx = max(s for _, s in logits)
        z = sum(math.exp(s - mx) for _, s in logits)
        lse[a] = mx + math.log(z)
        for c, s in logits:
            w = math.exp(s - lse[a])
            for t in range(d):
                O_[a, t] += w * v[c, t]
    return O_, lse


@pytest.mark.parametrize("seed,N,bq,bk", [(0, 13, 4, 3), (1, 20, 8, 4), (2, 17, 5, 5)])
def test_forward_matches_brute_force_loops(seed, N, bq, bk):
    q, k, v, _, mask = _rand_case(seed, N=N, d=5, bq=bq, bk=bk, nonempty=False)
    scale = 0.37
    o, lse = O.attn_fwd_head(q, k, v, mask, bq, bk, scale)
    ob, lseb = _brute_fwd(q, k, v, mask, bq, bk, scale)
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-12)
    fin = np.isfinite(lseb)
    assert (np.isfinite(lse) == fin).all()
    np.testing.assert_allclose(lse[fin], lseb[fin], rtol=1e-12, atol=1e-12)


def test_forward_block_diagonal_mask_is_per_block_dense_attention():
    N, d, b = 32, 6, 8
    q, k, v, _, _ = _rand_case(3, N=N, d=d, bq=b, bk=b)
    mask = np.eye(N // b, dtype=np.uint8)
    o, lse = O.attn_fwd_head(q, k, v, mask, b, b)
    for i in range(N // b):
        sl = slice(i * b, (i + 1) * b)
        s = q[sl] @ k[sl].T / math.sqrt(d)
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        np.testing.assert_allclose(o[sl], p @ v[sl], rtol=1e-12, atol=1e-13)


def test_forward_matches_torch_sdpa_fp64():
    torch = pytest.importorskip("torch")
    q, k, v, _, mask = _rand_case(4, N=40, d=16, bq=8, bk=4)
    o, lse = O.attn_fwd_head(q, k, v, mask, 8, 4)
    allowed = torch.from_numpy(O.token_mask(mask, 40, 8, 4))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=allowed[None])[0]
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-11, atol=1e-12)
    s = (torch.from_numpy(q) @ torch.from_numpy(k).T / 4.0).masked_fill(~allowed, -math.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=1).numpy(), rtol=1e-12, atol=1e-12)


def test_k_one_mask_is_dense_attention():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((1, 1, 50, 8)) for _ in range(3))
    mask = O.build_mask(q, k, 16, 8, 1.0, 0.0)["mask"]
    assert mask.all()
    o, _ = O.attn_fwd(q, k, v, mask, 16, 8)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v))
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-11, atol=1e-12)


def _loss(q, k, v, do, mask, bq, bk, scale):
    o, _ = O.attn_fwd_head(q, k, v, mask, bq, bk, scale)
    return float((o * do).sum())


def test_backward_matches_central_finite_differences():
    h = 1e-6
    for seed in (6, 7):  # two heads
        q, k, v, do, mask = _rand_case(seed, N=20, d=6, bq=8, bk=4, density=0.6)
        scale = 1 / math.sqrt(6)
        dq, dk, dv = O.attn_bwd_head(q, k, v, do, mask, 8, 4, scale)
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                x0 = x[idx]
                x[idx] = x0 + h
                lp = _loss(q, k, v, do, mask, 8, 4, scale)
                x[idx] = x0 - h
                lm = _loss(q, k, v, do, mask, 8, 4, scale)
                x[idx] = x0
                fd[idx] = (lp - lm) / (2 * h)
            err = np.abs(fd - g) / np.maximum(1.0, np.abs(g))
            assert err.max() <= 1e-6, (name, err.max())


def test_backward_matches_torch_autograd_fp64():
    torch = pytest.importorskip("torch")
    q, k, v, do, mask = _rand_case(8, N=36, d=8, bq=12, bk=6, density=0.4)
    dq, dk, dv = O.attn_bwd_head(q, k, v, do, mask, 12, 6)
    tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
    allowed = torch.from_numpy(O.token_mask(mask, 36, 12, 6))
    out = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None], attn_mask=allowed[None])[0]
    out.backward(torch.from_numpy(do))
    for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(mine, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_backward_invariants():
    q, k, v, do, mask = _rand_case(9, N=48, d=8, bq=16, bk=8, density=0.5)
    dq, dk, dv = O.attn_bwd_head(q, k, v, do, mask, 16, 8)
    # every row of dS sums to zero -> the keys' dK sum to zero
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    # every row of P sums to one -> the keys' dV sum to the queries' dO
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), rtol=1e-12, atol=1e-12)


def test_empty_rows_give_zero_output_minus_inf_lse_and_zero_gradients():
    q, k, v, do, _ = _rand_case(10, N=16, d=4, bq=8, bk=8)
    mask = np.array([[0, 0], [1, 0]], dtype=np.uint8)  # query block 0 keeps nothing
    o, lse = O.attn_fwd_head(q, k, v, mask, 8, 8)
    assert (o[:8] == 0).all() and np.isneginf(lse[:8]).all() and np.isfinite(lse[8:]).all()
    dq, dk, dv = O.attn_bwd_head(q, k, v, do, mask, 8, 8)
    assert (dq[:8] == 0).all()
    assert (dk[8:] == 0).all() and (dv[8:] == 0).all()  # key block 1 is kept by nobody
    # an all-empty mask (k = 0, p = 0) gives zeros everywhere
    m0 = O.hybrid_select(np.full((2, 2), 0.5), 0.0, 0.0).mask
    assert not m0.any()
    dq, dk, dv = O.attn_bwd_head(q, k, v, do, m0, 8, 8)
    assert not dq.any() and not dk.any() and not dv.any()


def test_row_and_column_sampled_versions_equal_the_full_computation():
    q, k, v, do, mask = _rand_case(11, N=45, d=8, bq=16, bk=8, density=0.4)
    o, lse = O.attn_fwd_head(q, k, v, mask, 16, 8)
    dq, dk, dv = O.attn_bwd_head(q, k, v, do, mask, 16, 8)
    rows = np.array([0, 7, 16, 31, 44])
    o_r, lse_r = O.attn_fwd_head(q, k, v, mask, 16, 8, rows=rows)
    np.testing.assert_allclose(o_r, o[rows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse_r, lse[rows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(O.attn_bwd_dq_rows(q, k, v, do, mask, 16, 8, rows), dq[rows],
                               rtol=1e-12, atol=1e-13)
    cols = np.array([0, 9, 10, 40, 44])
    dk_c, dv_c = O.attn_bwd_dkdv_cols(q, k, v, do, mask, 16, 8, cols)
    np.testing.assert_allclose(dk_c, dk[cols], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv_c, dv[cols], rtol=1e-12, atol=1e-13)
    # a query block that keeps nothing and a key block kept by nobody
    m2 = mask.copy()
    m2[1, :] = 0
    m2[:, 2] = 0
    dq2, dk2, dv2 = O.attn_bwd_head(q, k, v, do, m2, 16, 8)
    np.testing.assert_allclose(O.attn_bwd_dq_rows(q, k, v, do, m2, 16, 8, rows), dq2[rows],
                               rtol=1e-12, atol=1e-13)
    assert not O.attn_bwd_dq_rows(q, k, v, do, m2, 16, 8, np.arange(16, 32)).any()
    cols2 = np.array([0, 16, 23, 40])  # key block 2 (tokens 16..23) is kept by nobody
    dk_c2, dv_c2 = O.attn_bwd_dkdv_cols(q, k, v, do, m2, 16, 8, cols2)
    np.testing.assert_allclose(dk_c2, dk2[cols2], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv_c2, dv2[cols2], rtol=1e-12, atol=1e-13)
    assert not dk_c2[1:3].any() and not dv_c2[1:3].any()


def test_row_partition_of_the_backward_adds_up():
    q, k, v, do, mask = _rand_case(14, N=50, d=8, bq=16, bk=8, density=0.5)
    dq, dk, dv = O.attn_bwd_head(q, k, v, do, mask, 16, 8)
    parts = [np.arange(0, 16), np.arange(16, 40), np.arange(40, 50)]
    dk_sum, dv_sum = np.zeros_like(dk), np.zeros_like(dv)
    for rows in parts:
        dq_r, dk_p, dv_p = O.attn_bwd_rows(q, k, v, do, mask, 16, 8, rows)
        np.testing.assert_allclose(dq_r, dq[rows], rtol=1e-12, atol=1e-13)
        dk_sum += dk_p
        dv_sum += dv_p
    np.testing.assert_allclose(dk_sum, dk, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv_sum, dv, rtol=1e-12, atol=1e-13)


def test_batched_wrappers_and_bf16_widening():
    from workload import bf16_round_bits
    rng = np.random.default_rng(12)
    x = rng.standard_normal((1, 2, 30, 8)).astype(np.float32)
    bits = bf16_round_bits(x)
    wide = O.to_f64(bits)
    assert np.abs(wide - x).max() <= np.abs(x).max() * 2 ** -8
    mask = np.ones((1, 2, 2, 4), dtype=np.uint8)
    o, lse = O.attn_fwd(bits, bits, bits, mask, 16, 8)
    o1, _ = O.attn_fwd_head(wide[0, 1], wide[0, 1], wide[0, 1], mask[0, 1], 16, 8)
    np.testing.assert_allclose(o[0, 1], o1, rtol=0, atol=0)
