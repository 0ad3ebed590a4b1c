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


def test_algorithmic_bytes():
    """Bytes the bench charges per weight and per activation: 0.5 B codes +
    2/128 B scales per weight; bf16 x and y; the quantiser reads bf16 W."""
    sys.path.insert(0, ROOT)
    import bench

    N, K, M = 2560, 9216, 8
    assert bench.gemm_bytes(M, N, K) == N * K * 0.515625 + 2 * M * K + 2 * M * N
    assert bench.quant_bytes(N, K) == N * K * (2 + 0.515625)
    assert bench.affine_bytes(M, N, K, 128, False) == bench.gemm_bytes(M, N, K)
    assert bench.affine_bytes(M, N, K, 32, True) == N * K // 2 + N * (K // 32) * 3 + 2 * M * K + 2 * M * N


def test_profiles_are_reproducible_summaries():
    """Every committed profile summary gives the command that made it and holds
    no raw report; every traffic record parses."""
    pdir = os.path.join(ROOT, "profiles")
    names = sorted(os.listdir(pdir))
    assert any(n.startswith("launches_") for n in names)
    for n in names:
        path = os.path.join(pdir, n)
        assert n.endswith((".md", ".txt")), n
        assert os.path.getsize(path) < 16 * 1024, n
        text = open(path).read()
        if n.endswith(".md"):
            assert "```" in text and ("ncu " in text), n
            assert "--clock-control none" in text, n
    for line in open(os.path.join(pdir, "traffic.txt")):
        if line.startswith("#") or not line.strip():
            continue
        parts = line.split()
        fields = dict(p.split("=", 1) for p in parts[2:])
        assert int(fields["read"]) + int(fields["write"]) == int(fields["bytes_per_launch"])
        assert len(fields["source"]) == 12


def test_oracle_pool_splits_rows_and_runs():
    """The CPU baseline's process pool (spawned workers, the oracle unchanged)
    covers every row once per pass and returns a positive wall time."""
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    from gemm_rtn_sym_gb300 import workloads as wl

    W = wl.bits(wl.random_bf16((10, 256), 0.02, seed=3))
    x = wl.bits(wl.random_bf16((2, 256), 1.0, seed=4))
    pool = bench.OraclePool(3, W, x, 256)
    try:
        assert pool.run(1) > 0 and pool.run(2) > 0
    finally:
        pool.close()
    # The row split used by run(): contiguous, disjoint, complete.
    w = min(pool.workers, pool.rows)
    bounds = [pool.rows * i // w for i in range(w + 1)]
    assert bounds[0] == 0 and bounds[-1] == 10 and all(a < b for a, b in zip(bounds, bounds[1:]))
    assert np.array_equal(np.concatenate([W[a:b] for a, b in zip(bounds, bounds[1:])]), W)


def test_compact_configs_line_is_short():
    """The per-workload summary printed on the result line names every
    workload and stays short enough for a log tail."""
    sys.path.insert(0, ROOT)
    import bench

    pk = {"hbm_gbs": 6773.9, "bf16_tflops": 1872.3, "bf16_tflops_sustained": 1705.0, "source": "measured"}
    one = {"us": 6.6, "frac": 0.27, "bound": "hbm"}
    tc = {"us": 283.0, "frac": 0.67, "bound": "tensor"}
    sub = {"ffn_m1": one, "outlier_m8": one, "quant_ffn": one,
           "layer27b": {f"M{m}": one for m in (1, 5, 7, 13)},
           "layer27b_grouped": {f"M{m}": one for m in (1, 5, 7, 13)},
           "layer70b": {"M208": tc}, "layer70b_grouped": {"M208": tc},
           "stack4b": {f"M{m}": one for m in (1, 2, 4, 8, 16, 32, 64, 128)},
           "stack4b_grouped": {f"M{m}": one for m in (1, 2, 4, 8, 16, 32, 64, 128)}}
    c = bench.compact_configs(sub, pk)
    for label in ("1_ffn", "2_outlier", "3_layer27b", "3_layer27b_grouped", "4_layer70b", "4_layer70b_grouped",
                  "5_stack4b", "5_stack4b_grouped", "quant_ffn"):
        assert label in c
    assert c["4_layer70b_grouped"]["M208"][2] == "tc"
    assert len(json.dumps(c, separators=(",", ":"))) < 1200
