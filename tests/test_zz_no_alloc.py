"""sa2_build_mask_noalloc, the mask builder for callers that cannot allocate device memory
(code under another runtime's memory pool, plugins that only receive tensors, paths where
an allocation would synchronize): it keeps its scratch in a static device array of the
library instead of a caller workspace.

Called through the C ABI twice in a row on different workloads, its outputs must equal
those of sa2_build_mask on the same inputs (integer outputs bit for bit, pooled
probabilities within the mask tests' 5e-6).  Collected last on purpose."""
import ctypes

import numpy as np
import pytest

from tests.gpu_util import to_device
from workload import CONFIGS, make_inputs
from workload.gen import small_case

pytestmark = pytest.mark.gpu

SA2_ERR_WORKSPACE = 4


@pytest.fixture(scope="module")
def sa2():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_attention_sa2_gb300 as m
    lib = m.load_library()
    lib.sa2_build_mask_noalloc.restype = ctypes.c_int
    lib.sa2_build_mask_noalloc.argtypes = [ctypes.POINTER(m.sa2.Shape), ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_float, ctypes.c_float, ctypes.POINTER(m.sa2.BlockMaskStruct),
                                           ctypes.c_void_p]
    return m


def _noalloc(sa2, q, k, topk, topp, bq, bk):
    import torch
    B, H, N, _ = q.shape
    out = sa2.BlockMask.empty(B, H, -(-N // bq), -(-N // bk), q.device, mask=True, pooled=True)
    shp = sa2.make_shape(q, bq, bk)
    st = sa2.load_library().sa2_build_mask_noalloc(ctypes.byref(shp), q.data_ptr(), k.data_ptr(), float(topk),
                                                    float(topp), ctypes.byref(out.struct()),
                                                    torch.cuda.current_stream().cuda_stream)
    assert st == 0, f"sa2_build_mask_noalloc returned {st}"
    return out


def _same(a, b):
    rc = a.row_cnt.cpu().numpy()
    assert (rc == b.row_cnt.cpu().numpy()).all()
    assert (a.col_cnt.cpu().numpy() == b.col_cnt.cpu().numpy()).all()
    assert (a.mask.cpu().numpy() == b.mask.cpu().numpy()).all()
    ra, rb = a.row_idx.cpu().numpy(), b.row_idx.cpu().numpy()
    ca, cb, cc = a.col_idx.cpu().numpy(), b.col_idx.cpu().numpy(), a.col_cnt.cpu().numpy()
    for g in np.ndindex(rc.shape):
        assert (ra[g][: rc[g]] == rb[g][: rc[g]]).all()
    for g in np.ndindex(cc.shape):
        assert (ca[g][: cc[g]] == cb[g][: cc[g]]).all()
    assert np.abs(a.pooled_p.cpu().numpy() - b.pooled_p.cpu().numpy()).max() <= 5e-6


def test_noalloc_matches_build_mask_on_two_calls_in_a_row(sa2):
    import torch
    cfg1 = CONFIGS[1]
    x1 = make_inputs(cfg1, tensors=("q", "k"))
    cfg2, x2 = small_case("noalloc-ragged", 2, 3, 1000, 64, "bf16", 64, 64, seed=21)
    cases = [(cfg1, x1, 0.05, 0.9), (cfg2, x2, 0.2, 0.5)]
    for cfg, x, topk, topp in cases:  # two calls in a row, different shapes and data
        q, k = to_device(x["q"]), to_device(x["k"])
        got = _noalloc(sa2, q, k, topk, topp, cfg.bq, cfg.bk)
        ref = sa2.build_mask(q, k, topk, topp, bq=cfg.bq, bk=cfg.bk, want_pooled=True)
        sa2.check_device()
        torch.cuda.synchronize()
        _same(got, ref)


def test_noalloc_rejects_shapes_beyond_its_scratch(sa2):
    import torch
    # 2*B*H*d*(Tq+Tk)*4 bytes of pooled TF32 pairs alone: 2*1*40*128*(591+1182)*4 = 73 MB > 16 MB.
    # The size check runs before anything is launched, so the tensors are never read.
    q = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    shp = sa2.sa2.Shape(1, 40, 75600, 128, 128, 64, 0, 0, 40 * 75600 * 128, 75600 * 128, 128)
    out = sa2.BlockMask.empty(1, 1, 1, 1, q.device)
    st = sa2.load_library().sa2_build_mask_noalloc(ctypes.byref(shp), q.data_ptr(), q.data_ptr(), 0.1, 0.5,
                                                    ctypes.byref(out.struct()), torch.cuda.current_stream().cuda_stream)
    assert st == SA2_ERR_WORKSPACE
