"""GPU parity of sa2_build_mask against the fp64 oracle.

Masks must match bit for bit except entries whose pooled probability lies within 1e-6 of
the oracle row's selection threshold; those are logged.  The compact lists must list the
CUDA path's own mask exactly, and P-bar must agree with the oracle's to fp32 accuracy."""
import json
import os

import numpy as np
import pytest

import oracle as O
from tests.gpu_util import check_lists_consistent, compare_masks, to_device
from workload import CONFIGS, make_inputs
from workload.gen import small_case

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def sa2():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_attention_sa2_gb300 as m
    m.load_library()
    return m


def _compare(sa2, cfg, x, topk, topp, heads=None, log=None, check_lists=True, label=None):
    """Builds the mask on the GPU and compares it with the oracle's on `heads` (all by
    default): P-bar, the entries (near-threshold ones exempt and logged), and every row as
    the hybrid selection of the GPU's own P-bar.  Returns (mask, oracle result, exempt)."""
    torch = pytest.importorskip("torch")
    q, k = to_device(x["q"]), to_device(x["k"])
    bm = sa2.build_mask(q, k, topk, topp, bq=cfg.bq, bk=cfg.bk, want_pooled=True)
    sa2.check_device()
    torch.cuda.synchronize()
    ref = O.build_mask(x["q"], x["k"], cfg.bq, cfg.bk, topk, topp, heads=heads)
    todo = heads or [(b, h) for b in range(cfg.B) for h in range(cfg.H)]
    exempt = compare_masks(bm, ref, todo, topk, topp, label or f"{cfg.name} k={topk} p={topp}")
    if log is not None:
        log.extend(exempt)
    if check_lists:
        check_lists_consistent(bm, cfg.B, cfg.H, cfg.Tq, cfg.Tk)
    return bm, ref, exempt


def test_mask_tiny_fp32_config(sa2):
    cfg = CONFIGS[0]
    x = make_inputs(cfg, tensors=("q", "k"))
    _compare(sa2, cfg, x, cfg.topk, cfg.topp)


@pytest.mark.parametrize("N,d,bq,dtype", [(1000, 128, 128, "bf16"), (777, 64, 64, "bf16"), (1000, 64, 128, "fp32"),
                                          (64, 128, 128, "bf16"), (1, 128, 128, "bf16")])
def test_mask_ragged_small_cases(sa2, N, d, bq, dtype):
    cfg, x = small_case(f"ragged-{N}", 2, 3, N, d, dtype, bq, 64, seed=3)
    for topk, topp in ((0.1, 0.5), (0.0, 0.9), (0.3, 0.0), (0.0, 0.0), (1.0, 0.3), (0.05, 1.0)):
        _compare(sa2, cfg, x, topk, topp)


@pytest.mark.parametrize("Tk", [1400, 7680])
def test_mask_long_rows(sa2, Tk):
    """Rows of more than 1280 key blocks take the scoring kernel's shared-memory selection
    path (shorter rows keep their keys in registers); 7680 key blocks is the longest row the
    builder accepts (N = 491520 tokens)."""
    cfg, x = small_case(f"long-rows-{Tk}", 1, 1, Tk * 64, 64, "bf16", 128, 64, seed=51, tensors=("q", "k"))
    assert cfg.Tk == Tk
    _compare(sa2, cfg, x, 0.02, 0.5)


def test_mask_failure_probe_sweep(sa2):
    """Mask-failure probe (flat heads 0-3, sink heads 4-7): Top-k-only, Top-p-only, hybrid."""
    cfg = CONFIGS[1]
    x = make_inputs(cfg, tensors=("q", "k"))
    log = []
    summary = {}
    for topk, topp in cfg.sweep:
        K = O.topk_count(topk, cfg.Tk)
        cnt = {}
        for mode, (kk, pp) in (("topk", (topk, 0.0)), ("topp", (0.0, topp)), ("hybrid", (topk, topp))):
            bm, _, _ = _compare(sa2, cfg, x, kk, pp, log=log)
            cnt[mode] = bm.row_cnt.cpu().numpy()[0]  # [H, Tq]
            summary[f"k={topk} p={topp} {mode}"] = [round(float(v), 2) for v in cnt[mode].mean(axis=1)]
        assert (cnt["topk"] == K).all()
        assert (cnt["topp"][4:] == 1).all()  # sink heads: one block already holds > 90 %
        flat = cnt["topp"][:4].mean()
        assert abs(flat - topp * cfg.Tk) <= 0.1 * topp * cfg.Tk + 1  # flat heads keep about p*Tk
        assert (cnt["hybrid"] == np.maximum(cnt["topk"], cnt["topp"])).all()
    # every exempt entry was checked to sit at its row's threshold (compare_masks)
    assert len(log) <= 8, f"{len(log)} exempt entries on the probe sweep: {log[:8]}"
    print(json.dumps(summary, indent=0))


@pytest.mark.parametrize("ci", [2, 3])
def test_mask_full_size_wan_shapes(sa2, ci):
    """Full-size Wan-shaped workloads at the calibrated 95 % sparsity, in the launch
    configuration the benchmark times: the oracle checks every head (P-bar, the entries, the
    selection of the GPU's own P-bar) and the lists of three heads are checked entry by entry."""
    cfg = CONFIGS[ci]
    cal = json.load(open(os.path.join(GOLDEN, "calibration.json")))[str(ci)]["targets"]["0.95"]
    heads = [(0, h) for h in range(cfg.H)]
    x = make_inputs(cfg, tensors=("q", "k"), threads=16)
    bm, ref, exempt = _compare(sa2, cfg, x, cal["k"], cal["p"], heads=heads, check_lists=False)
    n_exempt = len(exempt)
    kept = bm.row_cnt.sum().item() / (cfg.B * cfg.H * cfg.Tq * cfg.Tk)
    assert abs((1 - kept) - 0.95) < 0.01
    # lists of three heads checked entry by entry
    mask = bm.mask.cpu().numpy().astype(bool)
    rc, cc = bm.row_cnt.cpu().numpy(), bm.col_cnt.cpu().numpy()
    assert (rc == mask.sum(-1)).all() and (cc == mask.sum(-2)).all()
    ri, ci_ = bm.row_idx.cpu().numpy(), bm.col_idx.cpu().numpy()
    for (b, h) in (heads[0], heads[len(heads) // 2], heads[-1]):
        for i in range(cfg.Tq):
            assert (ri[b, h, i, :rc[b, h, i]] == np.nonzero(mask[b, h, i])[0]).all()
        for j in range(cfg.Tk):
            assert (ci_[b, h, j, :cc[b, h, j]] == np.nonzero(mask[b, h, :, j])[0]).all()
    print(f"config {ci}: sparsity {1 - kept:.4f}, exempt {n_exempt}")


def test_mask_lists_without_the_optional_outputs(sa2):
    """The u8 mask and P-bar are optional outputs: without them the lists (which the column
    lists build from the rows' kept bits, not from the u8 mask) are the same, bit for bit."""
    import torch
    cfg = CONFIGS[1]
    x = make_inputs(cfg, tensors=("q", "k"))
    q, k = to_device(x["q"]), to_device(x["k"])
    full = sa2.build_mask(q, k, 0.05, 0.9, bq=cfg.bq, bk=cfg.bk, want_pooled=True)
    bare = sa2.build_mask(q, k, 0.05, 0.9, bq=cfg.bq, bk=cfg.bk, want_mask=False, want_pooled=False)
    sa2.check_device()
    torch.cuda.synchronize()
    assert bare.mask is None and bare.pooled_p is None
    for name in ("row_cnt", "col_cnt"):
        assert torch.equal(getattr(full, name), getattr(bare, name)), name
    rc, cc = full.row_cnt.cpu().numpy(), full.col_cnt.cpu().numpy()
    ri, ci = full.row_idx.cpu().numpy(), full.col_idx.cpu().numpy()
    bri, bci = bare.row_idx.cpu().numpy(), bare.col_idx.cpu().numpy()
    for b in range(cfg.B):
        for h in range(cfg.H):
            for i in range(cfg.Tq):
                assert (ri[b, h, i, :rc[b, h, i]] == bri[b, h, i, :rc[b, h, i]]).all()
            for j in range(cfg.Tk):
                assert (ci[b, h, j, :cc[b, h, j]] == bci[b, h, j, :cc[b, h, j]]).all()


def test_mask_rejects_bad_arguments(sa2):
    torch = pytest.importorskip("torch")
    q = torch.zeros((1, 1, 128, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sa2.Sa2Error):
        sa2.build_mask(q, q, 1.5, 0.5)
    with pytest.raises(sa2.Sa2Error):
        sa2.build_mask(q, q, 0.1, float("nan"))
    with pytest.raises(sa2.Sa2Error):
        sa2.build_mask(q, q, 0.1, 0.5, bk=32)


def test_mask_diagnostics_on_gpu_masks(sa2):
    """The diagnostics (per-row kept counts, kept pooled mass, per-head histograms) computed
    on the device from masks the GPU built for the mask-probe workload: kept counts equal the
    oracle's max(K, m) and kept masses its pooled mass over the kept blocks (rows holding a
    logged near-threshold entry aside), and they show the failure modes of the single rules
    (gist.science explainer, section 1; thelatestinai.com Table 6, Top-k-only / Top-p-only)."""
    torch = pytest.importorskip("torch")
    from block_sparse_attention_sa2_gb300.diagnostics import mask_diagnostics
    cfg = CONFIGS[1]
    x = make_inputs(cfg, tensors=("q", "k"))
    k, p = 0.05, 0.9
    K = O.topk_count(k, cfg.Tk)
    flat, sink = slice(0, 4), slice(4, 8)
    stats = {}
    for mode, (kk, pp) in (("topk", (k, 0.0)), ("topp", (0.0, p)), ("hybrid", (k, p))):
        bm, ref, exempt = _compare(sa2, cfg, x, kk, pp, label=f"diagnostics {mode}")
        d = mask_diagnostics(bm, bins=8)
        assert d["kept"].is_cuda and d["kept_mass"].is_cuda
        kept, mass = d["kept"].cpu().numpy()[0], d["kept_mass"].cpu().numpy()[0]
        for h in range(cfg.H):
            sel = ref["sel"][(0, h)]
            skip = {e[2] for e in exempt if e[1] == h}
            rows = [i for i in range(cfg.Tq) if i not in skip]
            assert (kept[h, rows] == sel.L[rows]).all(), f"{mode} head {h}: kept counts"
            want = np.array([sel.sorted_P[i, :sel.L[i]].sum() for i in rows])
            assert np.abs(mass[h, rows] - want).max() <= 1e-5, f"{mode} head {h}: kept mass"
        assert (d["kept_frac_hist"].sum(-1) == cfg.Tq).all() and (d["kept_mass_hist"].sum(-1) == cfg.Tq).all()
        stats[mode] = (torch.as_tensor(kept), torch.as_tensor(mass))
    kept, mass = stats["topk"]
    assert (kept == K).all() and mass[flat].median() < 0.5  # Top-k alone misses a flat row's mass
    kept, mass = stats["topp"]
    assert (kept[sink] == 1).all() and (mass[sink] >= p).all()  # Top-p alone: the sink block only
    kept, mass = stats["hybrid"]
    assert (mass[flat] >= p - 1e-6).all() and (kept[sink] >= K).all()  # the hybrid covers both
