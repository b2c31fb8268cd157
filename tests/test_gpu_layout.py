"""Token tensors in the token-major layout [B, N, H, d] (the layout of a model's projection
output, read with no copy) against the same data in the contiguous [B, H, N, d] layout.

sa2_shape carries one stride set for every token tensor, and no kernel's arithmetic depends
on the strides, so the mask, O, LSE, dQ, dK and dV of the two runs must agree bit for bit.
The contiguous run itself is held to the oracle by the other GPU tests."""
import numpy as np
import pytest

from tests.gpu_util import to_device
from workload.gen import small_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa2():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_attention_sa2_gb300 as m
    m.load_library()
    return m


def _token_major(t):
    """The same values stored as [B, N, H, d], viewed as [B, H, N, d]."""
    return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)


def _run(sa2, cfg, q, k, v, do, topk, topp):
    import torch
    bm = sa2.build_mask(q, k, topk, topp, bq=cfg.bq, bk=cfg.bk, want_pooled=True)
    o_lo = torch.empty_like(q) if q.dtype == torch.bfloat16 else None
    o, lse = sa2.attn_fwd(q, k, v, bm, bq=cfg.bq, bk=cfg.bk, o_lo=o_lo)
    dq, dk, dv = sa2.attn_bwd(q, k, v, o, lse, do, bm, bq=cfg.bq, bk=cfg.bk, o_lo=o_lo)
    sa2.check_device()
    torch.cuda.synchronize()
    return bm, {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


@pytest.mark.parametrize("N,d,bq,dtype", [(1000, 128, 128, "bf16"), (777, 64, 64, "fp32")])
def test_token_major_layout_is_bit_identical(sa2, N, d, bq, dtype):
    import torch
    cfg, x = small_case(f"layout-{N}", 2, 3, N, d, dtype, bq, 64, seed=31)
    base = {t: to_device(x[t]) for t in ("q", "k", "v", "do")}
    tm = {t: _token_major(a) for t, a in base.items()}
    assert tm["q"].stride() == (N * 3 * d, d, 3 * d, 1)  # [B, N, H, d] storage
    m1, r1 = _run(sa2, cfg, base["q"], base["k"], base["v"], base["do"], 0.2, 0.6)
    m2, r2 = _run(sa2, cfg, tm["q"], tm["k"], tm["v"], tm["do"], 0.2, 0.6)
    for name in ("row_cnt", "col_cnt", "mask"):
        assert torch.equal(getattr(m1, name), getattr(m2, name)), name
    rc = m1.row_cnt.cpu().numpy()
    ra, rb = m1.row_idx.cpu().numpy(), m2.row_idx.cpu().numpy()
    for g in np.ndindex(rc.shape):
        assert (ra[g][: rc[g]] == rb[g][: rc[g]]).all()
    assert torch.equal(m1.pooled_p, m2.pooled_p)
    for name in ("o", "dq", "dk", "dv"):  # outputs were written in place, token-major
        assert r2[name].stride() == tm["q"].stride(), name
    for name in r1:
        assert torch.equal(r1[name].contiguous(), r2[name].contiguous()), name
