"""The benchmark's multi-rank plumbing on CPU with gloo, world size 2: the timing reduction
returns the slowest rank's time on every rank, and under torchrun only rank 0 prints the
JSON line of the reference arm."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    got = bench.reduce_max_over_ranks(10.0 + 5.0 * rank, "cpu")
    q.put((rank, got))
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get() for _ in range(2))
    assert res == {0: 15.0, 1: 15.0}


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_one_line():
    port = 30500 + os.getpid() % 1000
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["e2e"]["h2d_bytes_per_step"] == 0


def test_head_shards_cover_the_layer_once_and_balance():
    sys.path.insert(0, ROOT)
    import bench
    for total in (1, 7, 12, 40, 41):
        for world in (1, 2, 3, 8):
            spans = [bench.shard_range(total, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == total
            assert all(spans[r][1] == spans[r + 1][0] for r in range(world - 1))
            sizes = [hi - lo for lo, hi in spans]
            assert max(sizes) - min(sizes) <= 1


def test_local_inputs_keep_each_heads_own_stream():
    """A rank's inputs for items [lo, hi) equal those heads of the whole workload."""
    sys.path.insert(0, ROOT)
    import bench
    from workload import CONFIGS, make_inputs
    cfg = CONFIGS[1]
    full = make_inputs(cfg, heads=[(0, 3), (0, 4), (0, 5)])
    part = bench.local_inputs(cfg, 3, 6)
    for t in ("q", "k", "v", "do"):
        assert (part[t][0] == full[t][0, 3:6]).all()


def _sum_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    lo, hi = bench.shard_range(40, world, rank)
    q.put((rank, bench.reduce_sum_over_ranks(float(hi - lo), "cpu")))
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_work_sums_to_the_whole_layer_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 31500 + os.getpid() % 1000
    procs = [ctx.Process(target=_sum_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get() for _ in range(2))
    assert res == {0: 40.0, 1: 40.0}
