"""Benchmark of the SpargeAttention2 hot path on GB300.

One step = the whole hot path over one batch of synthetic input: the hybrid Top-k + Top-p
block mask (sa2_build_mask), the block-sparse forward (sa2_attn_fwd) and the backward
(sa2_attn_bwd_with_fwd_ws: sa2_attn_bwd taking the forward's fp16 copy of V), on a
Wan2.1-14B-720p-shaped attention layer (B=1, H=40, N=75600 tokens of
a 21x45x80 latent, d=128, bf16, 128x64 blocks) at the calibrated 95 % block sparsity.

Metric: kept-tile TFLOP/s of forward + backward (4 + 10 flops per kept query-key pair per
channel, over valid tokens only), whole job over all ranks.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

--impl reference times the fp64 CPU oracle (the only reference this method has) on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workload import CONFIGS, make_inputs  # noqa: E402

FWD_FLOPS, BWD_FLOPS = 4, 10  # per kept (query, key) pair and channel

# DRAM bytes (read + write) of one attn_bwd_dkdv launch per head of the Wan2.1-14B-720p
# workload at its calibrated 95 % sparsity: an ncu capture of the 4-head case (776.9 MB read
# + 141.7 MB written, profiles/) divided by its heads, the heads being independent.  Set to
# None whenever the kernel changes until it has been captured again.
BWD_TRAFFIC_PER_HEAD = (776.931840e6 + 141.679616e6) / 4
BWD_TRAFFIC_WORKLOAD = ("wan2.1-14b-720p", 0.95)


def dkdv_traffic(cfg, sparsity: float):
    """Captured DRAM bytes of one dK/dV launch, scaled to the heads processed; None for a
    workload other than the captured one."""
    if BWD_TRAFFIC_PER_HEAD is None or (cfg.name, sparsity) != BWD_TRAFFIC_WORKLOAD:
        return None
    return BWD_TRAFFIC_PER_HEAD * cfg.B * cfg.H


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--sparsity", type=float, default=0.95,
                    help="calibrated target block sparsity of the config (0 = dense)")
    ap.add_argument("--e2e-steps", type=int, default=0,
                    help="steps of the end-to-end leg (0: the same as --steps)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager steps instead of replays of a CUDA graph of the step")
    ap.add_argument("--cpu-qblocks", type=int, default=4, help="query blocks of the oracle sample")
    ap.add_argument("--heads", type=int, default=0,
                    help="heads of the workload (default: all); a smaller case for profiler captures")
    ap.add_argument("--shard", choices=("heads", "replicas"), default="heads",
                    help="with several ranks: split the heads of the layer over them (strong scaling, "
                         "default) or run a whole layer on every rank (weak scaling)")
    a = ap.parse_args()
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.steps < 1 or a.e2e_steps < 0:
        ap.error("--steps must be >= 1 and --e2e-steps >= 0")
    return a


METRIC_DETAIL = ("TFLOP/s over kept tiles of the whole hot path (mask build + forward + backward) per step; "
                 "per-kernel ms and roofline fractions in 'kernels' / 'roofline'")


def metric_name(sparsity: float) -> str:
    """The benchmark's metric; the default run is the 95 %-sparsity one."""
    tail = "dense (k=1)" if sparsity == 0.0 else f"{round(100 * sparsity)}% sparsity"
    return f"block-sparse attn fwd+bwd ms and TFLOPS (kept tiles) vs bf16 TC peak at {tail}"


def calibration(ci: int, sparsity: float):
    if sparsity == 0.0:
        return 1.0, 1.0  # dense: every block kept
    path = os.path.join(ROOT, "tests", "golden", "calibration.json")
    cal = json.load(open(path))
    entry = cal[str(ci)]["targets"][f"{sparsity:.2f}"]
    return float(entry["k"]), float(entry["p"])


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def cpu_threads() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


# ------------------------------------------------------------------- ranks and timing

def shard_range(total: int, world: int, rank: int):
    """The contiguous share [lo, hi) of `total` independent (batch, head) items that rank
    `rank` of `world` takes: sizes differ by at most one, the first total % world ranks take
    the larger share.  Every (b, h) is independent through the mask, the forward and the
    backward, so the ranks need no exchange."""
    base, extra = divmod(total, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def reduce_sum_over_ranks(value: float, device) -> float:
    """Sum of one scalar over the ranks (the kept work of every rank's heads)."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def local_inputs(cfg, lo: int, hi: int):
    """The seeded inputs of the flat (batch, head) items [lo, hi) of the workload, laid out as
    one batch of hi - lo heads (each item keeps the stream of its global (b, h))."""
    from workload.gen import _stored, make_head
    n = hi - lo
    dt = np.uint16 if cfg.dtype == "bf16" else np.float32
    out = {t: np.zeros((1, n, cfg.N, cfg.d), dtype=dt) for t in ("q", "k", "v", "do")}
    for i, bh in enumerate(range(lo, hi)):
        for t in out:
            out[t][0, i] = _stored(cfg, make_head(cfg, bh // cfg.H, bh % cfg.H, t))
    return out


def reduce_max_over_ranks(value: float, device) -> float:
    """The slowest rank's time: every rank contributes its own and gets the maximum back
    (a reduction of one scalar for timing only; the data path has no collective)."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------- kept work

def tile_sizes(cfg):
    rq = np.minimum(cfg.bq, cfg.N - np.arange(cfg.Tq) * cfg.bq).astype(np.float64)
    rk = np.minimum(cfg.bk, cfg.N - np.arange(cfg.Tk) * cfg.bk).astype(np.float64)
    return rq, rk


def kept_pairs(cfg, mask_u8) -> float:
    """Sum over kept tiles of (valid query rows x valid key columns)."""
    rq, rk = tile_sizes(cfg)
    m = mask_u8.reshape(-1, cfg.Tq, cfg.Tk).astype(np.float64)
    return float(np.einsum("gij,i,j->", m, rq, rk))


# --------------------------------------------------------------------- CPU oracle leg

def oracle_sample(cfg, x, topk, topp, qblocks):
    """The oracle on a bounded sample of the workload: the mask of head 0 (pooling, pooled
    softmax, selection over all its rows), then forward and backward of the listed query
    blocks of head 0.  Returns (seconds, kept flops of the sampled rows, description)."""
    import oracle as O
    t0 = time.perf_counter()
    q, k, v, do = (O.to_f64(x[t][0, 0]) for t in ("q", "k", "v", "do"))
    r = O.build_mask_head(q, k, cfg.bq, cfg.bk, topk, topp)
    mask = r["mask"]
    rq, rk = tile_sizes(cfg)
    flops = 0.0
    for i in qblocks:
        rows = np.arange(i * cfg.bq, min(cfg.N, (i + 1) * cfg.bq))
        O.attn_fwd_head(q, k, v, mask, cfg.bq, cfg.bk, rows=rows)
        O.attn_bwd_rows(q, k, v, do, mask, cfg.bq, cfg.bk, rows)
        flops += (FWD_FLOPS + BWD_FLOPS) * cfg.d * rq[i] * float((mask[i] * rk).sum())
    dt = time.perf_counter() - t0
    desc = (f"oracle (numpy fp64) mask of head 0 + forward/backward of query blocks {list(qblocks)} of head 0 "
            f"({len(qblocks) * cfg.bq} query rows against all {cfg.N} keys)")
    return dt, flops, desc


def spread_qblocks(cfg, n):
    return sorted(set(int(round(v)) for v in np.linspace(0, cfg.Tq - 1, n)))


# ---------------------------------------------------------------------- clock sampler

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms during the timed region."""

    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id):
        self.bus_id = (bus_id or "").lower()
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        lines = [ln.strip() for ln in open(self.f.name) if ln.strip()]
        os.unlink(self.f.name)
        rows = [[c.strip() for c in ln.split(",")] for ln in lines]
        mine = [r for r in rows if len(r) >= 10 and (not self.bus_id or self.bus_id[-12:] in r[1].lower())]
        if not mine:
            mine = [r for r in rows if len(r) >= 10 and r[0] == "0"]
        sm = [float(r[2]) for r in mine if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in mine if r[3].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in mine for i in range(4) if r[6 + i].lower().startswith("active")})
        # samples under load: the upper half of the observed clocks (the bench keeps the GPU busy)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(sm)}


# ------------------------------------------------------------------- roofline accounting

MASK_KERNELS = ("pool", "score_tc", "select", "csc")
# Per kept (query, key) pair and channel, the algorithmic flops each attention kernel is
# credited with: the forward's two GEMMs (S, P V); the dK/dV kernel's S, dP, dV, dK; the dQ
# kernel's dQ GEMM only -- its recomputed S and dP are not algorithmic work.
KERNEL_FLOPS = {"attn_fwd": 4, "attn_bwd_dkdv": 8, "attn_bwd_dq": 2}


def phase_rooflines(prof, steps, pairs, d, peak_tflops):
    """Per-phase time and fraction of the bf16 peak, each phase with everything it launches.

    forward  = attn_fwd + its fp16 copy of V (one of the step's three to_f16 launches) + its
               launch order (one item_order pass);
    backward = attn_bwd_dkdv + attn_bwd_dq + bwd_preprocess + bwd_pair_union + the fp16
               copies of Q and K (two of the three to_f16 launches) + the dQ kernel's own launch
               order when it builds one (a backward given the forward's workspace reuses the
               forward's);
    algorithmic work 4 d (forward) and 10 d (backward) flops per kept pair."""
    def ms(name, share=1.0):
        return prof.get(name, (0, 0.0))[1] * share / steps

    conv = prof.get("to_f16", (0, 0.0))
    per_conv = conv[1] / conv[0] if conv[0] else 0.0  # the three copies are the same size
    passes = prof.get("item_order", (0, 0.0))[0] / steps  # item_order passes per step
    order_pass = ms("item_order") / passes if passes else 0.0  # the passes are the same size
    fwd_ms = ms("attn_fwd") + per_conv * (conv[0] / steps / 3.0 if conv[0] else 0.0) + order_pass
    bwd_ms = (ms("attn_bwd_dkdv") + ms("attn_bwd_dq") + ms("bwd_preprocess") + ms("bwd_pair_union")
              + per_conv * (2.0 * conv[0] / steps / 3.0 if conv[0] else 0.0) + ms("item_order") - order_pass)
    out = {}
    for name, t, f in (("forward", fwd_ms, FWD_FLOPS), ("backward", bwd_ms, BWD_FLOPS)):
        tf = f * d * pairs / (t * 1e-3) / 1e12 if t > 0 else None
        out[name] = {"ms": t, "algorithmic_tflop": f * d * pairs / 1e12, "tflops": tf,
                     "frac_of_bf16_burst": tf / peak_tflops if tf else None}
    return out


def dominant_roofline(prof, pairs, d, peaks):
    """The `roofline` object of the kernel with the largest device time: algorithmic flops of
    one launch (KERNEL_FLOPS x kept pairs) over its average launch time, against the measured
    dense bf16 peak as a burst (the kernels run in steps of tens of milliseconds at full clock;
    fp16 MMAs have the same nominal rate); the sustained figure is given beside it."""
    dom = max(prof.items(), key=lambda kv: kv[1][1])[0]
    c, m = prof[dom]
    if dom in KERNEL_FLOPS and c > 0 and m > 0:
        algo = KERNEL_FLOPS[dom] * d * pairs
        achieved = algo / ((m / c) * 1e-3) / 1e12
        return {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"], "traffic": None,
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                "peak_source": f"{peaks['source']} dense bf16, burst (fp16 MMAs: same nominal rate)",
                "algorithmic_flops_per_launch": algo}
    return {"kernel": dom, "bound": "hbm", "achieved": None, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": None, "traffic": None}


# ---------------------------------------------------------------------------- native

def run_native(a, rank, world):
    import torch
    import block_sparse_attention_sa2_gb300 as sa2
    from block_sparse_attention_sa2_gb300 import build_lib

    if not build_lib.up_to_date():
        if rank == 0:
            build_lib.build()
        if world > 1:
            torch.distributed.barrier()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg = CONFIGS[a.config]
    if a.heads:
        import dataclasses
        cfg = dataclasses.replace(cfg, H=a.heads)
    topk, topp = calibration(a.config, a.sparsity)
    sharded = world > 1 and a.shard == "heads"
    cfg_job = cfg  # the whole layer (sharded runs split its heads)
    if sharded:
        import dataclasses
        lo, hi = shard_range(cfg.B * cfg.H, world, rank)
        x = local_inputs(cfg, lo, hi)
        cfg = dataclasses.replace(cfg, B=1, H=hi - lo)
    else:
        x = make_inputs(cfg, threads=os.cpu_count() or 8)

    def pinned(arr):
        t = torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()

    host = {t: pinned(x[t]) for t in ("q", "k", "v", "do")}
    d = {t: host[t].to(dev) for t in host}
    stream = torch.cuda.current_stream()
    B, H, N, D = d["q"].shape
    bm = sa2.BlockMask.empty(B, H, cfg.Tq, cfg.Tk, dev, mask=True)
    lib = sa2.load_library()
    shp = sa2.make_shape(d["q"], cfg.bq, cfg.bk)
    import ctypes
    ws_m = sa2.workspace(lib.sa2_mask_workspace_size(ctypes.byref(shp)), dev)
    ws_f = sa2.workspace(lib.sa2_fwd_workspace_size(ctypes.byref(shp)), dev)
    ws_b = sa2.workspace(lib.sa2_bwd_workspace_size(ctypes.byref(shp)), dev)
    o, o_lo = torch.empty_like(d["q"]), torch.empty_like(d["q"])
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])

    def step(src, out=None):
        out = out or {"o": o, "dq": dq, "dk": dk, "dv": dv}
        sa2.build_mask(src["q"], src["k"], topk, topp, bq=cfg.bq, bk=cfg.bk, out=bm, ws=ws_m)
        sa2.attn_fwd(src["q"], src["k"], src["v"], bm, bq=cfg.bq, bk=cfg.bk, o=out["o"], lse=lse, o_lo=o_lo,
                     ws=ws_f)
        sa2.attn_bwd(src["q"], src["k"], src["v"], out["o"], lse, src["do"], bm, bq=cfg.bq, bk=cfg.bk,
                     o_lo=o_lo, dq=out["dq"], dk=out["dk"], dv=out["dv"], ws=ws_b, fwd_ws=ws_f)

    for _ in range(a.warmup):
        step(d)
    sa2.check_device()
    torch.cuda.synchronize()
    mask_np = bm.mask.cpu().numpy()
    pairs = kept_pairs(cfg, mask_np)
    sparsity = 1.0 - float(bm.row_cnt.sum().item()) / (B * H * cfg.Tq * cfg.Tk)
    flops_step = (FWD_FLOPS + BWD_FLOPS) * D * pairs
    # the work of the whole job per step: every rank's heads (sharded), or N whole layers
    job_flops_step = reduce_sum_over_ranks(flops_step, dev) if world > 1 else flops_step

    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    # The timed leg replays one CUDA graph of the whole step (its launches, memsets and the
    # mask builder's cross-stream waits, exactly the eager step's work) K times; --no-graph
    # times K eager steps instead.  Per-kernel device times come from a separate leg of K
    # eager steps under the library's launch profiler, whose events would otherwise sit
    # inside the timed region.
    graph = None
    if not a.no_graph:
        torch.cuda.synchronize()
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step(d)
            graph.replay()
            torch.cuda.synchronize()
        except Exception as err:  # a capture this driver refuses: time eager steps instead
            print(f"bench: CUDA graph capture failed ({err}); timing eager steps", file=sys.stderr)
            graph = None
            torch.cuda.synchronize()
        sa2.check_device()

    def timed(run):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(a.steps):
            run()
        t1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return reduce_max_over_ranks(t0.elapsed_time(t1), dev)

    clocks = ClockSampler(bus)
    if rank == 0:
        clocks.start()
    clocks.mark(True)
    ms_max = timed(graph.replay if graph is not None else (lambda: step(d)))
    clocks.mark(False)
    clk = clocks.stop() if rank == 0 else None
    sa2.check_device()
    eager_ms = timed(lambda: step(d)) if graph is not None else ms_max
    sa2.profiler_enable(True)
    sa2.profiler_collect()
    timed(lambda: step(d))
    sa2.profiler_enable(False)
    prof = sa2.profiler_collect()
    sa2.check_device()

    # ---- the mask builder timed on its own: wall time of sa2_build_mask on the stream (its
    # pooling and its second stream's scoring / selection overlap), inputs larger than L2
    mb_reps = max(5, a.steps)
    torch.cuda.synchronize()
    m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    m0.record(stream)
    for _ in range(mb_reps):
        sa2.build_mask(d["q"], d["k"], topk, topp, bq=cfg.bq, bk=cfg.bk, out=bm, ws=ws_m)
    m1.record(stream)
    torch.cuda.synchronize()
    mask_wall_ms = reduce_max_over_ranks(m0.elapsed_time(m1), dev) / mb_reps
    sa2.check_device()

    # ---- end to end through the public API with host buffers.  Every step uploads its
    # inputs from pinned host memory and reads all four results back; the uploads of step
    # i+1 and the read-back of step i-1 run on their own streams while step i computes
    # (inputs and outputs double-buffered on the device, ordered by events).
    # as many steps as the device-timed leg, so that the first upload and the last read-back,
    # which no compute can hide, weigh as they do in a run of that length
    e2e_steps = a.e2e_steps if a.e2e_steps > 0 else a.steps
    outs = ("o", "dq", "dk", "dv")
    hout = {n: torch.empty_like(host["q"]).pin_memory() for n in outs}
    dins = [{t: torch.empty_like(d[t]) for t in d} for _ in range(2)]
    douts = [{n: torch.empty_like(d["q"]) for n in outs} for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "used", "done", "read")}
    h2d = sum(host[t].numel() * host[t].element_size() for t in host)
    d2h = sum(hout[n].numel() * hout[n].element_size() for n in hout)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(e2e_steps):
        b = i & 1
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev["used"][b])  # step i-2 is done with this input buffer
            for t in host:
                dins[b][t].copy_(host[t], non_blocking=True)
            ev["in"][b].record(s_in)
        stream.wait_event(ev["in"][b])
        if i >= 2:
            stream.wait_event(ev["read"][b])  # the read-back of step i-2 has left this buffer
        step(dins[b], douts[b])
        ev["used"][b].record(stream)
        ev["done"][b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["done"][b])
            for n in outs:
                hout[n].copy_(douts[b][n], non_blocking=True)
            ev["read"][b].record(s_out)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max_over_ranks(e0.elapsed_time(e1), dev) / e2e_steps
    sa2.check_device()

    if rank != 0:
        return None
    peaks = measured_peaks()
    value = job_flops_step * a.steps / (ms_max * 1e-3) / 1e12
    kernels = {n: {"launches": c, "ms_per_launch": (m / c if c else 0.0), "total_ms": m} for n, (c, m) in prof.items()}
    # kernels per profiled launch range: a launch order is two kernels (and a memset)
    launches = sum(c * (2 if n == "item_order" else 1) for n, (c, _) in prof.items())
    ph = phase_rooflines(prof, a.steps, pairs, D, peaks["bf16_tflops"])
    roof = dominant_roofline(prof, pairs, D, peaks)
    if roof.get("kernel") == "attn_bwd_dkdv":
        roof["traffic"] = dkdv_traffic(cfg, a.sparsity)
    # mask builder against HBM: it reads Q and K once and writes the mask and lists
    qk_bytes = 2 * B * H * N * D * 2
    out_bytes = B * H * cfg.Tq * cfg.Tk + 4 * 2 * float(bm.row_cnt.sum().item()) + 4 * B * H * (cfg.Tq + cfg.Tk)
    mask_kernel_ms = sum(prof[k][1] for k in MASK_KERNELS if k in prof) / a.steps
    mask_ms = mask_wall_ms
    mask_gbs = (qk_bytes + out_bytes) / (mask_ms * 1e-3) / 1e9 if mask_ms > 0 else None
    fwd_ms, bwd_ms = ph["forward"]["ms"], ph["backward"]["ms"]
    step_frac = flops_step / (ms_max / a.steps * 1e-3) / 1e12 / peaks["bf16_tflops"]
    line = {
        "metric": metric_name(a.sparsity), "metric_detail": METRIC_DETAIL,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": ms_max / a.steps, "higher_is_better": True,
        "timing": (f"{a.steps} replays of one CUDA graph of the step (eager steps: {eager_ms / a.steps:.4f} ms); "
                   if graph is not None else f"{a.steps} eager steps; ")
                  + "per-kernel times from a separate profiled eager leg",
        "scaling": "strong" if sharded else "weak", "vs_baseline": None,
        "dtype": "bf16 in/out; tcgen05 MMAs bf16 (S) and fp16 (P, dS), fp32 accumulate", "data": "synthetic",
        "config": {"workload": f"{cfg.name} attention layer: B={cfg_job.B}, H={cfg_job.H}, N={N} (latent {'x'.join(map(str, cfg.grid))}), d={D}, bf16, "
                               f"blocks {cfg.bq}x{cfg.bk}",
                   "block_sparsity": sparsity, "topk": topk, "topp": topp, "seed": 0,
                   "l2": "inputs larger than L2 (Q,K,V,dO = %.1f GB per step); no flush" % (4 * B * H * N * D * 2 / 1e9),
                   "step": "sa2_build_mask + sa2_attn_fwd + sa2_attn_bwd_with_fwd_ws (the forward's fp16 copy of V reused)", "parallelism": (f"heads sharded over {world} ranks, {H} per rank (no collective)" if sharded
                                   else f"replicas x{world}")},
        "kept_tflop_per_step": flops_step / 1e12,
        "dense_equiv_tflops": (1 if sharded else world) * (FWD_FLOPS + BWD_FLOPS) * D * float(N) * N
                              * cfg_job.B * cfg_job.H * a.steps / (ms_max * 1e-3) / 1e12,
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "mask_ms": mask_ms,
        "fwd_tflops": ph["forward"]["tflops"], "bwd_tflops": ph["backward"]["tflops"],
        "phases": ph,
        "step_frac_of_bf16_burst": step_frac,
        "mask_builder": {"ms": mask_ms, "achieved_gbs": mask_gbs, "peak_gbs": peaks["hbm_gbs"],
                         "frac": mask_gbs / peaks["hbm_gbs"] if mask_gbs else None, "bytes": qk_bytes + out_bytes,
                         "timing": f"wall time of sa2_build_mask alone, mean of {mb_reps} calls (CUDA events)",
                         "sum_of_kernel_ms_in_step": mask_kernel_ms},
        "roofline": roof,
        "e2e": {"value": job_flops_step / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "kernels": kernels,
        "clocks": clk,
    }
    if world == 1 and not a.no_cpu_baseline:
        secs, cflops, desc = oracle_sample(cfg, x, topk, topp, spread_qblocks(cfg, a.cpu_qblocks))
        line["cpu_baseline"] = {"value": cflops / secs / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(),
                                "kind": "oracle", "sample": desc, "seconds": secs}
    return line


# ------------------------------------------------------------------------- reference

def run_reference(a, rank, world):
    if rank != 0:
        return None
    cfg = CONFIGS[a.config]
    topk, topp = calibration(a.config, a.sparsity)
    x = make_inputs(cfg, tensors=("q", "k", "v", "do"), heads=[(0, 0)])
    qb = spread_qblocks(cfg, 2)
    for _ in range(a.warmup):
        oracle_sample(cfg, x, topk, topp, qb)
    t0 = time.perf_counter()
    flops = 0.0
    desc = ""
    for _ in range(a.steps):
        _, f, desc = oracle_sample(cfg, x, topk, topp, qb)
        flops += f
    secs = time.perf_counter() - t0
    value = flops / secs / 1e12
    return {
        "impl": "reference",
        "metric": metric_name(a.sparsity), "metric_detail": METRIC_DETAIL,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": secs * 1e3 / a.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{cfg.name} attention layer (bounded oracle sample per step)",
                   "topk": topk, "topp": topp, "seed": 0},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    a = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        backend = "nccl" if a.impl == "native" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group(backend)
    line = run_reference(a, rank, world) if a.impl == "reference" else run_native(a, rank, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
