"""Host-side logic of bench.py without a GPU: the max-over-ranks step time and
the whole-job value on a two-rank gloo group, and the reference arm (the CPU
oracle) launched on two ranks, where rank 0 alone prints its line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier()
        t = bench.max_over_ranks(0.001 * (rank + 1))
        out[rank] = (t, bench.job_value(1e6, world, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, free_port(), out), nprocs=world, join=True)
        res = dict(out)
    # Both ranks see the slowest rank's time; the value counts both ranks' bytes.
    for rank in range(world):
        t, v = res[rank]
        assert t == pytest.approx(0.002)
        assert v == pytest.approx(2 * 1e6 / 0.002 / 1e9)


def test_max_over_ranks_without_group_is_local():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(0.5) == 0.5
    assert bench.job_value(2e9, 1, 1.0) == pytest.approx(2.0)


def test_reference_arm_on_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    for key in ("metric", "unit", "steps", "warmup", "ms_per_step", "higher_is_better", "config",
                "cpu_baseline", "e2e"):
        assert key in d
