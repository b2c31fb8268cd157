"""Seeded synthetic attention inputs shaped like the video-DiT layers the method targets.

The pages on SpargeAttention2 (arXiv 2602.13515) evaluate on Wan2.1 1.3B at 480p and
Wan2.1 14B at 720p (thelatestinai.com page, Tables 4 and 5).  No weights, prompts or
videos are used here: every tensor is drawn from a seeded generator with the shapes of
those attention layers and a structure that exercises the block mask:

* i.i.d. N(0, 1) noise in every channel;
* for Q and K, a smooth positional term over the (t, y, x) latent grid,
  ``amp * cos(2*pi * f_c . (t, y, x) + phi_c)`` with a per-channel frequency vector
  ``f_c ~ N(0, diag(sigma_t^2, sigma_y^2, sigma_x^2))`` and phase ``phi_c ~ U[0, 2*pi)``,
  which makes the similarity of two tokens decay with their grid distance (locality);
* optional "attention sinks": a per-head unit vector ``u`` is added as ``a*u`` to every
  query and as ``s*u`` to every token of the sink key blocks, so that those blocks draw
  a large share of every row's pooled mass.

V and dO are plain N(0, 1).  Values are generated in float64, cast to float32 and, for
bf16 workloads, rounded to bf16 (round to nearest, ties to even); the rounded bits are
the canonical input of both the CUDA path and the oracle.

Every (config, batch, head, tensor) has its own PCG64 stream keyed by
``SeedSequence([seed, config_index, b*H + h, tensor_id])``, so a single head can be
regenerated without the others and heads can be generated in parallel.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Dict, Iterable, Optional, Sequence, Tuple

import numpy as np

TENSOR_IDS = {"q": 0, "k": 1, "v": 2, "do": 3, "aux": 4}


@dataclass(frozen=True)
class WorkloadConfig:
    index: int
    name: str
    B: int
    H: int
    grid: Tuple[int, int, int]  # (T, Y, X) latent grid; N = T*Y*X tokens in raster order
    d: int
    dtype: str  # "bf16" or "fp32"
    bq: int
    bk: int
    pos_amp: float = 0.0
    pos_sigma: Tuple[float, float, float] = (0.0, 0.0, 0.0)  # cycles per grid step
    sink_blocks: Tuple[int, ...] = ()
    sink_s: float = 0.0
    sink_a: float = 0.0
    flat_heads: Tuple[int, ...] = ()  # heads with noise only (no positional term, no sink)
    sink_only_heads: Tuple[int, ...] = ()  # heads with noise + sink, no positional term
    topk: Optional[float] = None  # default mask parameters, where the config fixes them
    topp: Optional[float] = None
    sweep: Tuple[Tuple[float, float], ...] = field(default_factory=tuple)

    @property
    def N(self) -> int:
        return self.grid[0] * self.grid[1] * self.grid[2]

    @property
    def Tq(self) -> int:
        return -(-self.N // self.bq)

    @property
    def Tk(self) -> int:
        return -(-self.N // self.bk)


_WAN_SIGMA = (0.15, 0.06, 0.004)

CONFIGS: Dict[int, WorkloadConfig] = {
    # Tiny correctness case: 4x16x16 grid, fp32, 64x64 blocks, one sink at key block 0.
    0: WorkloadConfig(
        index=0, name="tiny-fp32-1024", B=1, H=2, grid=(4, 16, 16), d=64, dtype="fp32",
        bq=64, bk=64, pos_amp=2.0, pos_sigma=(0.25, 0.25, 0.25), sink_blocks=(0,),
        sink_s=6.0, sink_a=1.0, topk=0.1, topp=0.9),
    # Mask-failure probe: heads 0-3 flat (noise only), heads 4-7 dominated by one sink block.
    1: WorkloadConfig(
        index=1, name="mask-probe-8192", B=1, H=8, grid=(8, 32, 32), d=128, dtype="bf16",
        bq=128, bk=64, sink_blocks=(0,), sink_s=32.0, sink_a=3.0,
        flat_heads=(0, 1, 2, 3), sink_only_heads=(4, 5, 6, 7),
        sweep=((0.02, 0.5), (0.02, 0.9), (0.05, 0.5), (0.05, 0.9))),
    # Wan2.1-1.3B-480p self-attention shape: latent 21x30x52, 12 heads of 128.
    2: WorkloadConfig(
        index=2, name="wan2.1-1.3b-480p", B=1, H=12, grid=(21, 30, 52), d=128, dtype="bf16",
        bq=128, bk=64, pos_amp=1.0, pos_sigma=_WAN_SIGMA, sink_blocks=(0, 1),
        sink_s=30.0, sink_a=2.0),
    # Wan2.1-14B-720p self-attention shape: latent 21x45x80, 40 heads of 128.
    3: WorkloadConfig(
        index=3, name="wan2.1-14b-720p", B=1, H=40, grid=(21, 45, 80), d=128, dtype="bf16",
        bq=128, bk=64, pos_amp=1.0, pos_sigma=_WAN_SIGMA, sink_blocks=(0, 1),
        sink_s=30.0, sink_a=2.0),
    # Sparsity sweep on the 1.3B-480p shape (targets 0/80/90/95/97 % and a dense run).
    4: WorkloadConfig(
        index=4, name="wan2.1-1.3b-480p-sweep", B=1, H=12, grid=(21, 30, 52), d=128,
        dtype="bf16", bq=128, bk=64, pos_amp=1.0, pos_sigma=_WAN_SIGMA, sink_blocks=(0, 1),
        sink_s=30.0, sink_a=2.0),
    # The same latent and model width (1536) split into 24 heads of 64 channels: the d = 64
    # form of the Wan2.1 drop-in.
    5: WorkloadConfig(
        index=5, name="wan2.1-1.3b-480p-d64", B=1, H=24, grid=(21, 30, 52), d=64,
        dtype="bf16", bq=128, bk=64, pos_amp=1.0, pos_sigma=_WAN_SIGMA, sink_blocks=(0, 1),
        sink_s=30.0, sink_a=2.0),
}


def token_coords(grid: Tuple[int, int, int]) -> np.ndarray:
    """(t, y, x) coordinates of each token of a raster-ordered T x Y x X grid, [N, 3] float64."""
    T, Y, X = grid
    n = np.arange(T * Y * X, dtype=np.int64)
    t = n // (Y * X)
    y = (n // X) % Y
    x = n % X
    return np.stack([t, y, x], axis=1).astype(np.float64)


def bf16_round_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even.

    Inputs here are finite, so no NaN handling is needed."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF)
    r += (u >> np.uint32(16)) & np.uint32(1)
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, cfg: WorkloadConfig, bh: int, tensor: str) -> np.random.Generator:
    return np.random.Generator(
        np.random.PCG64(np.random.SeedSequence([seed, cfg.index, bh, TENSOR_IDS[tensor]])))


def _head_aux(seed: int, cfg: WorkloadConfig, bh: int):
    """Per-head positional frequencies/phases and the sink direction."""
    rng = _rng(seed, cfg, bh, "aux")
    f = rng.standard_normal((cfg.d, 3)) * np.asarray(cfg.pos_sigma, dtype=np.float64)
    phi = rng.uniform(0.0, 2.0 * math.pi, size=cfg.d)
    u = rng.standard_normal(cfg.d)
    u /= np.linalg.norm(u)
    return f, phi, u


def make_head(cfg: WorkloadConfig, b: int, h: int, tensor: str, seed: int = 0) -> np.ndarray:
    """One head of one tensor as float32 [N, d], before any bf16 rounding."""
    bh = b * cfg.H + h
    rng = _rng(seed, cfg, bh, tensor)
    x = rng.standard_normal((cfg.N, cfg.d), dtype=np.float32)
    if tensor not in ("q", "k"):
        return x
    flat = h in cfg.flat_heads
    sink_only = h in cfg.sink_only_heads
    if flat:
        return x
    f, phi, u = _head_aux(seed, cfg, bh)
    acc = x.astype(np.float64)
    if cfg.pos_amp != 0.0 and not sink_only:
        coords = token_coords(cfg.grid)
        acc += cfg.pos_amp * np.cos(2.0 * math.pi * (coords @ f.T) + phi[None, :])
    if cfg.sink_blocks:
        if tensor == "q" and cfg.sink_a != 0.0:
            acc += cfg.sink_a * u[None, :]
        if tensor == "k" and cfg.sink_s != 0.0:
            for j in cfg.sink_blocks:
                lo, hi = j * cfg.bk, min(cfg.N, (j + 1) * cfg.bk)
                acc[lo:hi] += cfg.sink_s * u[None, :]
    return acc.astype(np.float32)


def _stored(cfg: WorkloadConfig, x: np.ndarray) -> np.ndarray:
    return bf16_round_bits(x) if cfg.dtype == "bf16" else x


def make_inputs(cfg: WorkloadConfig, seed: int = 0,
                tensors: Sequence[str] = ("q", "k", "v", "do"),
                heads: Optional[Iterable[Tuple[int, int]]] = None,
                threads: int = 0) -> Dict[str, np.ndarray]:
    """Inputs in storage form: uint16 bf16 bits or float32, shape [B, H, N, d].

    ``heads`` restricts generation to the listed (b, h) pairs (the others stay zero), which
    keeps host-side checks of a few heads of the large workloads cheap.  ``threads`` > 1
    generates heads in parallel; the result does not depend on it."""
    dt = np.uint16 if cfg.dtype == "bf16" else np.float32
    if heads is None:
        heads = [(b, h) for b in range(cfg.B) for h in range(cfg.H)]
    heads = list(heads)
    out = {t: np.zeros((cfg.B, cfg.H, cfg.N, cfg.d), dtype=dt) for t in tensors}

    def work(job):
        t, b, h = job
        out[t][b, h] = _stored(cfg, make_head(cfg, b, h, t, seed))

    jobs = [(t, b, h) for t in tensors for (b, h) in heads]
    if threads and threads > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, jobs))
    else:
        for j in jobs:
            work(j)
    return out


def small_case(name: str, B: int, H: int, N: int, d: int, dtype: str, bq: int, bk: int,
               seed: int = 0, sink: bool = True,
               tensors: Tuple[str, ...] = ("q", "k", "v", "do")) -> Tuple[WorkloadConfig, Dict[str, np.ndarray]]:
    """A small ragged case (N need not be a multiple of the blocks) for parity tests.

    The grid is 1 x 1 x N, so the positional term varies along the token index only."""
    cfg = WorkloadConfig(index=100 + N % 97, name=name, B=B, H=H, grid=(1, 1, N), d=d,
                         dtype=dtype, bq=bq, bk=bk, pos_amp=1.0,
                         pos_sigma=(0.0, 0.0, 1.0 / max(bk, 1)),
                         sink_blocks=(0,) if sink else (), sink_s=8.0 if sink else 0.0,
                         sink_a=1.0 if sink else 0.0)
    return cfg, make_inputs(cfg, tensors=tensors, seed=seed)
