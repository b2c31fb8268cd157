"""The seeded generator: determinism, per-head independence, bf16 rounding, and the
structure each workload is meant to have (checked through the oracle's pooled map)."""
import numpy as np
import pytest

import oracle as O
from workload import CONFIGS, bf16_bits_to_f32, bf16_round_bits, make_head, make_inputs


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.0e-3], dtype=np.float32)
    got = bf16_bits_to_f32(bf16_round_bits(x))
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa -> 1; 1 + 3*2^-8 -> 1 + 2^-6
    assert got.tolist()[:4] == [1.0, 1.0, 1.0 + 2 ** -6, 1.0]
    assert got[4] == -2.5
    assert abs(got[5] - 3.0e-3) <= 3.0e-3 * 2 ** -8


def test_generation_is_deterministic_and_per_head():
    cfg = CONFIGS[1]
    a = make_inputs(cfg, heads=[(0, 2), (0, 5)])
    b = make_inputs(cfg, heads=[(0, 5), (0, 2)], threads=4)
    for t in a:
        assert (a[t] == b[t]).all()
    one = bf16_round_bits(make_head(cfg, 0, 5, "k"))
    assert (one == a["k"][0, 5]).all()
    assert not (a["q"][0, 2] == a["q"][0, 5]).all()


def test_shapes_and_dtypes_of_every_config():
    expect = {0: (1, 2, 1024, 64, 16, 16), 1: (1, 8, 8192, 128, 64, 128),
              2: (1, 12, 32760, 128, 256, 512), 3: (1, 40, 75600, 128, 591, 1182),
              4: (1, 12, 32760, 128, 256, 512), 5: (1, 24, 32760, 64, 256, 512)}
    for i, (B, H, N, d, Tq, Tk) in expect.items():
        c = CONFIGS[i]
        assert (c.B, c.H, c.N, c.d, c.Tq, c.Tk) == (B, H, N, d, Tq, Tk)
    assert CONFIGS[0].dtype == "fp32" and all(CONFIGS[i].dtype == "bf16" for i in (1, 2, 3, 4, 5))
    assert CONFIGS[5].H * CONFIGS[5].d == CONFIGS[2].H * CONFIGS[2].d  # the same model width


def _pooled(cfg, h):
    x = make_inputs(cfg, tensors=("q", "k"), heads=[(0, h)])
    return O.build_mask_head(O.to_f64(x["q"][0, h]), O.to_f64(x["k"][0, h]), cfg.bq, cfg.bk, 0.0, 0.5)


def test_mask_probe_heads_are_flat_or_sink_dominated():
    cfg = CONFIGS[1]
    flat = _pooled(cfg, 0)["P"]
    assert flat.max() < 2.0 / cfg.Tk  # noise-only head: no block holds twice its share
    for h in (4, 7):
        P = _pooled(cfg, h)["P"]
        assert (P[:, 0] > 0.9).all()  # sink block 0 holds > 90 % of every row's pooled mass


@pytest.mark.slow
def test_wan_shaped_heads_have_sinks_and_locality():
    cfg = CONFIGS[2]
    r = _pooled(cfg, 0)
    P = r["P"]
    sink = P[:, list(cfg.sink_blocks)].sum(axis=1)
    assert 0.2 <= sink.mean() <= 0.6  # sinks draw a large share of the pooled mass
    # locality: the key blocks within +-3 of the diagonal hold far more than their share
    diag = np.array([P[i, max(0, 2 * i - 2): 2 * i + 5].sum() for i in range(cfg.Tq)])
    assert diag.mean() > 10 * 7 / cfg.Tk
