"""Run one small, self-checking case of a single kernel, for a profiler.

    python -m gemm_rtn_sym_gb300.profile_case quantize --workload outlier
    python -m gemm_rtn_sym_gb300.profile_case quantize_scaled --workload outlier
    python -m gemm_rtn_sym_gb300.profile_case gemm --workload outlier --M 8
    python -m gemm_rtn_sym_gb300.profile_case gemm --workload layer70b --matrix 2 --M 208
    python -m gemm_rtn_sym_gb300.profile_case grouped --workload layer27b --M 1
    python -m gemm_rtn_sym_gb300.profile_case grouped --workload layer27b --M 1 --group 128 --asym
    python -m gemm_rtn_sym_gb300.profile_case quantize --workload outlier --group 32 --asym
    python -m gemm_rtn_sym_gb300.profile_case gemm --workload outlier --M 8 --group 32 --asym
    python -m gemm_rtn_sym_gb300.profile_case gptq --workload ffn

The inputs are the seeded synthetic matrices of ``workloads``.  For ``gemm`` the
weights are quantised first (one quantiser launch), then the matmul runs
``--launches`` times on the same inputs.  ``grouped`` quantises every matrix
of the workload and runs one grouped plan over all of them.  ``--group`` and
``--asym`` select the affine formats (w4_quantize_rtn / w4_quantize_rtn_asym at
that group size, w4_gemm_affine).  ``gptq`` factors a seeded synthetic
calibration statistic once and runs the GPTQ quantiser ``--launches`` times.  The case checks the device status
word at the end and exits non-zero if any wait timed out.  It times nothing:
numbers taken under a profiler are not benchmark results.
"""
from __future__ import annotations

import argparse
import sys

import torch

from . import W4_PATH_AUTO, W4_PATH_SMALL_M, W4_PATH_TENSOR
from . import load, w4_gemm_ex, w4_gemm_grouped, w4_grouped_plan, w4_last_device_status, w4_quantize_rtn
from . import w4_gemm_affine, w4_gptq_factor, w4_gptq_quantize, w4_quantize_rtn_asym, w4_quantize_rtn_scaled
from . import workloads as wl

PATHS = {"auto": W4_PATH_AUTO, "small": W4_PATH_SMALL_M, "tensor": W4_PATH_TENSOR}


def main(argv=None) -> int:
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("kernel", choices=["quantize", "quantize_scaled", "gemm", "grouped", "gptq"])
    p.add_argument("--workload", default="outlier", choices=sorted(wl.SHAPES))
    p.add_argument("--matrix", type=int, default=0, help="index into the workload's matrices")
    p.add_argument("--M", type=int, default=8, help="token rows of x (gemm)")
    p.add_argument("--path", default="auto", choices=sorted(PATHS))
    p.add_argument("--launches", type=int, default=3)
    p.add_argument("--group", type=int, default=128, choices=[32, 64, 128])
    p.add_argument("--asym", action="store_true", help="asymmetric codes with zero points")
    a = p.parse_args(argv)

    load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if a.kernel == "grouped":
        problems, zeros = [], []
        for i, (N, K) in enumerate(wl.SHAPES[a.workload]):
            W = wl.weight(a.workload, i, device=dev)
            if a.asym:
                packed, scales, z = w4_quantize_rtn_asym(W, a.group)
                zeros.append(z)
            else:
                packed, scales = w4_quantize_rtn(W, a.group)
            del W
            x = wl.activations(a.workload, a.M, K, i, device=dev)
            problems.append((x, packed, scales, torch.empty((a.M, N), dtype=torch.bfloat16, device=dev)))
        plan = w4_grouped_plan(problems, group=a.group, zeros=zeros if a.asym else None)
        for _ in range(a.launches):
            w4_gemm_grouped(plan)
        torch.cuda.synchronize()
        status = w4_last_device_status(dev)
        print(f"grouped {a.workload} M={a.M}: {len(problems)} problems, {plan.items} items, "
              f"{a.launches} launches, device status {status}")
        return 0 if status == 0 else 1
    N, K = wl.SHAPES[a.workload][a.matrix]
    W = wl.weight(a.workload, a.matrix, device=dev)
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((N, K // a.group), dtype=torch.bfloat16, device=dev)
    zeros = torch.empty((N, K // a.group), dtype=torch.int8, device=dev) if a.asym else None
    affine = a.asym or a.group != 128
    fmt = f" g{a.group} {'asym' if a.asym else 'sym'}"

    def quantize():
        if a.asym:
            w4_quantize_rtn_asym(W, a.group, packed=packed, scales=scales, zeros=zeros)
        else:
            w4_quantize_rtn(W, a.group, packed=packed, scales=scales)
    if a.kernel == "quantize":
        for _ in range(a.launches):
            quantize()
        what = f"quantize {a.workload}[{a.matrix}] {N}x{K}{fmt}"
    elif a.kernel == "gptq":
        H = wl.calibration_hessian(K, 4096, seed=wl.seed_for(a.workload, a.matrix, 4), device=dev)
        U = w4_gptq_factor(H)
        for _ in range(a.launches):
            w4_gptq_quantize(W, U, a.group, packed=packed, scales=scales)
        what = f"gptq {a.workload}[{a.matrix}] {N}x{K} g{a.group}"
    elif a.kernel == "quantize_scaled":
        s = wl.workload_channel_scales(a.workload, a.matrix, device=dev)
        for _ in range(a.launches):
            w4_quantize_rtn_scaled(W, s, packed=packed, scales=scales)
        what = f"quantize_scaled {a.workload}[{a.matrix}] {N}x{K}"
    else:
        quantize()
        del W
        x = wl.activations(a.workload, a.M, K, a.matrix, device=dev)
        y = torch.empty((a.M, N), dtype=torch.bfloat16, device=dev)
        for _ in range(a.launches):
            if affine:
                w4_gemm_affine(x, packed, scales, zeros, group=a.group, out=y, path=PATHS[a.path])
            else:
                w4_gemm_ex(x, packed, scales, out=y, path=PATHS[a.path])
        what = f"gemm {a.workload}[{a.matrix}] M={a.M} N={N} K={K} path={a.path}{fmt}"
    torch.cuda.synchronize()
    status = w4_last_device_status(dev)
    print(f"{what}: {a.launches} launches, device status {status}")
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
