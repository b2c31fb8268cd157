"""Pins of the oracle's toy distillation step (gist.science explainer, section 2.B: the loss
is the squared L2 distance between the sparse and the full-attention output).

- a student whose mask equals the teacher's has loss 0 and zero gradients;
- dL/dO_s = 2 (O_s - O_t) agrees with central differences of L (exact for a quadratic);
- the whole chain (sparse forward -> loss -> sparse backward) agrees with central
  differences of L with respect to q, k and v, the teacher's output held fixed (the
  teacher is frozen in distillation)."""
import numpy as np

import oracle as O

BQ = BK = 8


def _tiny(seed=3, B=1, H=1, N=40, d=8):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((B, H, N, d)) for _ in range(3)]


def _masks(N):
    T = O.num_blocks(N, BQ)
    dense = np.ones((1, 1, T, T), dtype=np.uint8)
    rng = np.random.default_rng(11)
    sparse = (rng.random((1, 1, T, T)) < 0.5).astype(np.uint8)
    sparse[..., np.arange(T), np.arange(T)] = 1  # every row keeps its diagonal block
    return dense, sparse


def test_matching_student_has_zero_loss_and_gradients():
    q, k, v = _tiny()
    dense, _ = _masks(q.shape[2])
    loss, do, dq, dk, dv = O.distill_step(q, k, v, dense, dense, BQ, BK)
    assert loss == 0.0
    for g in (do, dq, dk, dv):
        assert np.abs(g).max() == 0.0


def test_loss_gradient_matches_central_differences():
    rng = np.random.default_rng(5)
    o_s, o_t = rng.standard_normal((2, 3, 4)), rng.standard_normal((2, 3, 4))
    _, g = O.vd_loss(o_s, o_t)
    h = 1e-3
    for idx in [(0, 0, 0), (1, 2, 3), (0, 1, 2)]:
        p, m = o_s.copy(), o_s.copy()
        p[idx] += h
        m[idx] -= h
        fd = (O.vd_loss(p, o_t)[0] - O.vd_loss(m, o_t)[0]) / (2 * h)
        assert abs(fd - g[idx]) < 1e-9
    assert O.vd_loss(o_s, o_t)[0] > 0


def test_chain_matches_central_differences_with_teacher_frozen():
    q, k, v = _tiny()
    N = q.shape[2]
    dense, sparse = _masks(N)
    assert 0 < sparse.sum() < dense.sum()
    loss, _, dq, dk, dv = O.distill_step(q, k, v, sparse, dense, BQ, BK)
    assert loss > 0
    o_t, _ = O.attn_fwd(q, k, v, dense, BQ, BK)  # frozen teacher

    def L(qq, kk, vv):
        o_s, _ = O.attn_fwd(qq, kk, vv, sparse, BQ, BK)
        return O.vd_loss(o_s, o_t)[0]

    h = 1e-6
    rng = np.random.default_rng(7)
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(4):
            idx = (0, 0, int(rng.integers(N)), int(rng.integers(q.shape[3])))
            args_p = [x.copy() for x in (q, k, v)]
            args_m = [x.copy() for x in (q, k, v)]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            fd = (L(*args_p) - L(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx, fd, grad[idx])
