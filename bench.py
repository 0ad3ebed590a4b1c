#!/usr/bin/env python3
"""Benchmark of the W4A16 group-128 RTN path on GB300.

One step = one pass of the whole path over one synthetic matrix: RTN-quantise a
bf16 weight matrix (w4_quantize_rtn) and run the decode matmul (w4_gemm) on a
quantised matrix.  The headline workload is the 2560×9216 FFN matrix with 1 %
outlier input channels and M = 8 token rows (a speculative-verify pass of 7
drafts + 1).  Inputs rotate over enough distinct copies that every step reads
its inputs from HBM (the rotation set exceeds 4× the L2 size); the matmul of
step i reads the copy quantised R/2 steps earlier, so its packed weights are
not L2-resident either.

Timing: the K timed steps are captured once into a CUDA graph and replayed
between CUDA events on the launch stream; per-kernel durations come from
graphs holding only that kernel's K launches, replayed right after.
Sub-benchmarks (M = 1, M = 8, the 27B-class layer at M ∈ {1,5,7,13}, the
70B-class layer at M = 208, the 4B-class 200-matrix stack sweep, quantiser
alone, the AWQ-style channel-scaled quantiser and activation scaling, the
asymmetric and group-32/64 formats, GPTQ) are reported under "sub".

`--impl reference` times the CPU oracle (the only other program here that
computes the same thing) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "outlier"
HEADLINE_M = 8
METRIC = "W4A16 g128 GEMV/GEMM HBM GB/s (% of peak) at M=1,8,208; RTN quant GB/s"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--no-sub", action="store_true", help="skip the sub-benchmarks")
    p.add_argument("--no-sweep", action="store_true", help="skip the 200-matrix stack sweep")
    p.add_argument("--only", default="", help="comma list of sub-benchmarks to run")
    return p.parse_args()


# ----------------------------------------------------------------- bytes / flops
def gemm_bytes(M, N, K):
    """Algorithmic bytes of one matmul: packed codes + scales + x + y."""
    return N * K // 2 + N * (K // 128) * 2 + 2 * M * K + 2 * M * N


def quant_bytes(N, K):
    """Algorithmic bytes of one quantisation: read W, write codes + scales."""
    return 2 * N * K + N * K // 2 + N * (K // 128) * 2


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def tensor_peak(pk):
    """bf16 tensor peak the tensor-bound sub-benchmarks are graded against: the
    measured burst figure (cuBLAS timed alone), because each sub-benchmark times
    a short replay of one graph, i.e. a kernel timed in isolation.  The
    fraction of the sustained figure (cuBLAS back to back for seconds) is
    reported beside it."""
    return pk["bf16_tflops"]


HBM_NOMINAL_GBS = 7900.0  # GB300 HBM3e, nominal (context beside the measured copy peak)


def source_hash(name):
    with open(os.path.join(ROOT, "gemm_rtn_sym_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:12]


def traffic_record(kernel_file, kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    summary is missing or the kernel's source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    h = source_hash(kernel_file)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
                fields = dict(p.split("=", 1) for p in parts[2:] if "=" in p)
                if fields.get("source") == h:
                    return float(fields["bytes_per_launch"])
    return None


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        rows = [[c.strip() for c in l.split(",")] for l in self.lines if l.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())}


# ----------------------------------------------------------------- GPU arm
class Timer:
    """CUDA-event timing of a callable replayed on the current stream."""

    def __init__(self, torch):
        self.torch = torch

    def time(self, fn, reps=1):
        torch = self.torch
        s = torch.cuda.current_stream()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(s)
        for _ in range(reps):
            fn()
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / reps  # seconds per call


def capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # one eager run on the capture stream before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    g.replay()  # upload
    torch.cuda.synchronize()
    return g


def n_copies(torch, bytes_per_copy, minimum=4):
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    return max(minimum, math.ceil(4 * l2 / bytes_per_copy)), l2


def headline(torch, w4, wl, steps, warmup, pk):
    """The timed step: quantise copy i, matmul copy i - R/2 (M = 8)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    N, K = wl.SHAPES[HEADLINE][0]
    M = HEADLINE_M
    W0 = wl.weight(HEADLINE, device=dev)
    x0 = wl.activations(HEADLINE, M, K, device=dev)
    per_copy = 2 * N * K + N * K // 2 + N * K // 64 + 2 * M * K + 2 * M * N
    R, l2 = n_copies(torch, per_copy, minimum=8)
    Ws = [W0.clone() for _ in range(R)]
    xs = [x0.clone() for _ in range(R)]
    Ps = [torch.empty((N, K // 2), dtype=torch.uint8, device=dev) for _ in range(R)]
    Ss = [torch.empty((N, K // 128), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    Ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    for r in range(R):
        w4.w4_quantize_rtn(Ws[r], packed=Ps[r], scales=Ss[r])
    passes = (M + 15) // 16 if w4.w4_gemm_path_for(M, N, K) == w4.W4_PATH_SMALL_M else 1

    def step(i):
        a = i % R
        b = (i + R // 2) % R
        w4.w4_quantize_rtn(Ws[a], packed=Ps[a], scales=Ss[a])
        w4.w4_gemm(xs[b], Ps[b], Ss[b], out=Ys[b])

    for i in range(max(3, warmup)):
        step(i)
    torch.cuda.synchronize()
    g_all = capture(torch, lambda: [step(i) for i in range(steps)])
    g_q = capture(torch, lambda: [w4.w4_quantize_rtn(Ws[i % R], packed=Ps[i % R], scales=Ss[i % R])
                                  for i in range(steps)])
    g_g = capture(torch, lambda: [w4.w4_gemm(xs[(i + R // 2) % R], Ps[(i + R // 2) % R],
                                             Ss[(i + R // 2) % R], out=Ys[(i + R // 2) % R])
                                  for i in range(steps)])
    T = Timer(torch)
    with ClockSampler(dev.index) as clk:
        t_end = time.time() + 1.0
        while time.time() < t_end:  # untimed soak so the clock record spans the load
            g_all.replay()
        torch.cuda.synchronize()
        rank_barrier()
        t_step = T.time(g_all.replay) / steps
        rank_barrier()
    t_q = T.time(g_q.replay) / steps
    t_g = T.time(g_g.replay) / steps
    torch.cuda.synchronize()
    assert w4.w4_last_device_status() == 0

    qb, gb = quant_bytes(N, K), gemm_bytes(M, N, K)
    bytes_step = qb + gb
    dominant = ("quantize_rtn_kernel", "w4_quantize.cu", qb, t_q) if t_q >= t_g else \
        ("gemv_w4_kernel", "w4_gemv.cu", gb, t_g)
    name, src, dbytes, dt = dominant
    achieved = dbytes / dt / 1e9
    traffic = traffic_record(src, name, f"{HEADLINE}-{N}x{K}-M{M}")
    res = {
        "value": bytes_step / t_step / 1e9,
        "ms_per_step": t_step * 1e3,
        "roofline": {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                     "algorithmic_bytes": dbytes, "peak_source": f"{pk['source']} hbm_gbs (burst copy)"},
        "kernels": {
            "quantize": {"us": t_q * 1e6, "GB/s": qb / t_q / 1e9, "frac": qb / t_q / 1e9 / pk["hbm_gbs"]},
            "gemm_m8": {"us": t_g * 1e6, "GB/s": gb / t_g / 1e9, "frac": gb / t_g / 1e9 / pk["hbm_gbs"],
                        "tok/s": M / t_g},
        },
        "clocks": clk.summary(),
        "gpu_launches": steps * (1 + passes),
        "rotation": {"copies": R, "bytes_per_copy": per_copy, "l2_bytes": l2},
    }
    # end to end through the public API with host buffers
    Wh = W0.cpu().pin_memory()
    xh = x0.cpu().pin_memory()
    ph = torch.empty((N, K // 2), dtype=torch.uint8).pin_memory()
    sh = torch.empty((N, K // 128), dtype=torch.bfloat16).pin_memory()
    yh = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()

    # Three streams: uploads, kernels, read-backs.  Step i's upload overlaps
    # step i-1's kernels and step i-2's read-back; every step still moves its
    # own inputs in and its results out.  A device copy is overwritten only
    # after the kernels and read-back that last used it have finished.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_k = torch.cuda.current_stream()
    done_k = [None] * R    # kernels of the step that last used copy r
    done_out = [None] * R  # read-back of the step that last used copy r

    def e2e_step(i):
        a = i % R
        b = (i + R // 2) % R
        with torch.cuda.stream(s_in):
            for r in (a, b):
                if done_k[r] is not None:
                    s_in.wait_event(done_k[r])
            Ws[a].copy_(Wh, non_blocking=True)
            xs[b].copy_(xh, non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
        s_k.wait_event(ev_in)
        for r in (a, b):
            if done_out[r] is not None:
                s_k.wait_event(done_out[r])
        w4.w4_quantize_rtn(Ws[a], packed=Ps[a], scales=Ss[a])
        w4.w4_gemm(xs[b], Ps[b], Ss[b], out=Ys[b])
        ev_k = torch.cuda.Event()
        ev_k.record(s_k)
        done_k[a] = done_k[b] = ev_k
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_k)
            ph.copy_(Ps[a], non_blocking=True)
            sh.copy_(Ss[a], non_blocking=True)
            yh.copy_(Ys[b], non_blocking=True)
            ev_out = torch.cuda.Event()
            ev_out.record(s_out)
        done_out[a] = done_out[b] = ev_out

    def e2e_run(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(s_k)
        s_in.wait_event(start)
        for i in range(n):
            e2e_step(i)
        s_k.wait_stream(s_in)
        s_k.wait_stream(s_out)
        end.record(s_k)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / 1e3 / n

    e2e_run(3)
    t_e2e = e2e_run(steps)
    res["e2e"] = {"value": bytes_step / t_e2e / 1e9, "unit": "GB/s",
                  "h2d_bytes_per_step": 2 * N * K + 2 * M * K,
                  "d2h_bytes_per_step": N * K // 2 + N * (K // 128) * 2 + 2 * M * N,
                  "ms_per_step": t_e2e * 1e3,
                  "overlap": "uploads, kernels and read-backs of consecutive steps on three streams"}
    del Ws, xs, Ps, Ss, Ys
    torch.cuda.empty_cache()
    return res


def gemm_set(torch, w4, wl, workload, Ms, pk, reps=20, path=None, grouped=False, fmt=None):
    """Matmul over every matrix of a workload (one launch per matrix, or one
    grouped launch over all of them), per M.  Matrices that fit in L2 several
    times are rotated over copies.  fmt = (group, asym) selects an affine
    format (grouped launches only): codes from w4_quantize_rtn_asym (asym) or
    w4_quantize_rtn at that group size."""
    dev = torch.device("cuda", torch.cuda.current_device())
    mats = []
    shapes = wl.SHAPES[workload]
    total_packed = sum(n * k // 2 for n, k in shapes)
    copies = 1 if total_packed > 4 * 126e6 else n_copies(torch, total_packed)[0]
    cache = {}
    zeros_of = {}
    group, asym = fmt if fmt else (128, False)
    for i, (N, K) in enumerate(shapes):
        key = (N, K) if workload == "stack4b" else i
        if key not in cache:
            W = wl.weight(workload, i, device=dev)
            if asym:
                p_, s_, z_ = w4.w4_quantize_rtn_asym(W, group)
                cache[key] = (p_, s_)
                zeros_of[key] = z_
            else:
                cache[key] = w4.w4_quantize_rtn(W, group)
            del W
        for c in range(copies):
            p, s = cache[key]
            mats.append((N, K, p.clone() if (copies > 1 or workload == "stack4b") else p,
                         s.clone() if (copies > 1 or workload == "stack4b") else s, i))
    # every copy gets its own zeros too, so no copy reads L2-resident ones
    zeros_list = [None if zeros_of.get((N, K) if workload == "stack4b" else i) is None
                  else zeros_of[(N, K) if workload == "stack4b" else i].clone() for (N, K, _, _, i) in mats]
    cache.clear()
    out = {}
    T = Timer(torch)
    for M in Ms:
        xs = {}
        ys = []
        for (N, K, p, s, i) in mats:
            if (K, i if workload != "stack4b" else 0) not in xs:
                xs[(K, i if workload != "stack4b" else 0)] = wl.activations(workload, M, K, i, device=dev)
            ys.append(torch.empty((M, N), dtype=torch.bfloat16, device=dev))

        if grouped:
            # One plan per copy of the workload (a layer, or the whole stack):
            # copies exist only to rotate inputs through L2, and must not
            # enlarge the group a launch balances its work over.
            n_per = len(mats) // copies
            plans = [w4.w4_grouped_plan([(xs[(K, i if workload != "stack4b" else 0)], p, s, ys[j])
                                         for j, (N, K, p, s, i) in enumerate(mats)
                                         if j % copies == c], group=group,
                                        zeros=[zeros_list[j] for j in range(len(mats)) if j % copies == c]
                                        if asym else None)
                     for c in range(copies)]
            assert all(len(pl.tensors) == (5 if asym else 4) * n_per for pl in plans)

            def run():
                for pl in plans:
                    w4.w4_gemm_grouped(pl)
        else:
            def run():
                for j, (N, K, p, s, i) in enumerate(mats):
                    x = xs[(K, i if workload != "stack4b" else 0)]
                    if path is None:
                        w4.w4_gemm(x, p, s, out=ys[j])
                    else:
                        w4.w4_gemm_ex(x, p, s, out=ys[j], path=path)

        g = capture(torch, run)
        nb = sum(affine_bytes(M, N, K, group, asym) for (N, K, _, _, _) in mats) / copies
        fl = sum(2 * M * N * K for (N, K, _, _, _) in mats) / copies
        t_hbm = nb / (pk["hbm_gbs"] * 1e9)
        t_tc = fl / (tensor_peak(pk) * 1e12)
        clocks = None
        if t_tc > t_hbm:
            # Tensor-bound: soak for half a second and time under the clock
            # sampler, to record the (power-capped) SM clock the fraction uses.
            with ClockSampler(dev.index) as clk:
                t_end = time.time() + 0.5
                while time.time() < t_end:
                    g.replay()
                torch.cuda.synchronize()
                t = T.time(g.replay, reps=reps) / copies
            clocks = clk.summary()
        else:
            t = T.time(g.replay, reps=reps) / copies
        out[f"M{M}"] = {"us": t * 1e6, "GB/s": nb / t / 1e9, "TFLOP/s": fl / t / 1e12,
                        "tok/s": M / t, "bound": "hbm" if t_hbm >= t_tc else "tensor",
                        "frac": max(t_hbm, t_tc) / t,
                        "frac_sustained_tc": fl / t / 1e12 / pk["bf16_tflops_sustained"]
                        if pk.get("bf16_tflops_sustained") else None,
                        "path": "grouped" if grouped else
                        (w4.w4_gemm_path_for(M, mats[0][0], mats[0][1]) if path is None else path)}
        if clocks is not None:
            out[f"M{M}"]["clocks"] = clocks
        if grouped:
            out[f"M{M}"]["launches_per_set"] = 1
            del plans
        del g, ys, xs
    assert w4.w4_last_device_status() == 0
    del mats
    torch.cuda.empty_cache()
    return out


def quant_set(torch, w4, wl, workload, pk, reps=10, scaled=False):
    """The quantiser alone over rotating copies; with ``scaled``, the
    channel-scaled variant (AWQ-style s, fp32 [K], read once per launch)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    N, K = wl.SHAPES[workload][0]
    W0 = wl.weight(workload, 0, device=dev)
    R, _ = n_copies(torch, quant_bytes(N, K))
    Ws = [W0.clone() for _ in range(R)]
    Ps = [torch.empty((N, K // 2), dtype=torch.uint8, device=dev) for _ in range(R)]
    Ss = [torch.empty((N, K // 128), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    if scaled:
        s = wl.workload_channel_scales(workload, device=dev)
        g = capture(torch, lambda: [w4.w4_quantize_rtn_scaled(Ws[r], s, packed=Ps[r], scales=Ss[r])
                                    for r in range(R)])
    else:
        g = capture(torch, lambda: [w4.w4_quantize_rtn(Ws[r], packed=Ps[r], scales=Ss[r]) for r in range(R)])
    t = Timer(torch).time(g.replay, reps=reps) / R
    b = quant_bytes(N, K) + (4 * K if scaled else 0)
    del Ws, Ps, Ss, g
    torch.cuda.empty_cache()
    return {"us": t * 1e6, "GB/s": b / t / 1e9, "frac": b / t / 1e9 / pk["hbm_gbs"], "shape": [N, K]}


def scale_act_set(torch, w4, wl, workload, M, pk, reps=20):
    """x' = x / s (w4_scale_activations) on M rows of the workload's first K,
    over rotating copies of x; bytes = x read + x' written + s read."""
    dev = torch.device("cuda", torch.cuda.current_device())
    K = wl.SHAPES[workload][0][1]
    b = 4 * M * K + 4 * K
    R, _ = n_copies(torch, b)
    x0 = wl.activations(workload, M, K, device=dev)
    s = wl.workload_channel_scales(workload, device=dev)
    xs = [x0.clone() for _ in range(R)]
    outs = [torch.empty_like(x0) for _ in range(R)]
    g = capture(torch, lambda: [w4.w4_scale_activations(xs[r], s, out=outs[r]) for r in range(R)])
    t = Timer(torch).time(g.replay, reps=reps) / R
    del xs, outs, g
    torch.cuda.empty_cache()
    return {"us": t * 1e6, "GB/s": b / t / 1e9, "frac": b / t / 1e9 / pk["hbm_gbs"], "shape": [M, K]}


def affine_bytes(M, N, K, group, asym):
    """Algorithmic bytes of one affine-format matmul: codes + scales (+ zeros) + x + y."""
    return N * K // 2 + N * (K // group) * (3 if asym else 2) + 2 * M * K + 2 * M * N


def affine_set(torch, w4, wl, workload, matrix, Ms, group, asym, pk, reps=10):
    """Quantiser (group, asym) and w4_gemm_affine on one matrix of a workload,
    over rotating copies of its inputs."""
    dev = torch.device("cuda", torch.cuda.current_device())
    N, K = wl.SHAPES[workload][matrix]
    W0 = wl.weight(workload, matrix, device=dev)
    qb = 2 * N * K + N * K // 2 + N * (K // group) * (3 if asym else 2)
    R, _ = n_copies(torch, qb)
    Ws = [W0.clone() for _ in range(R)]
    outs = [(torch.empty((N, K // 2), dtype=torch.uint8, device=dev),
             torch.empty((N, K // group), dtype=torch.bfloat16, device=dev),
             torch.empty((N, K // group), dtype=torch.int8, device=dev) if asym else None) for _ in range(R)]
    del W0

    def quant():
        for r in range(R):
            p, s, z = outs[r]
            if asym:
                w4.w4_quantize_rtn_asym(Ws[r], group, packed=p, scales=s, zeros=z)
            else:
                w4.w4_quantize_rtn(Ws[r], group, packed=p, scales=s)
    g = capture(torch, quant)
    t = Timer(torch).time(g.replay, reps=reps) / R
    res = {"format": f"g{group} {'asym' if asym else 'sym'}", "shape": [N, K],
           "quant": {"us": t * 1e6, "GB/s": qb / t / 1e9, "frac": qb / t / 1e9 / pk["hbm_gbs"]}}
    del Ws, g
    torch.cuda.empty_cache()
    for M in Ms:
        x = wl.activations(workload, M, K, matrix, device=dev)
        ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(R)]

        def mm():
            for r in range(R):
                p, s, z = outs[r]
                w4.w4_gemm_affine(x, p, s, z, group=group, out=ys[r])
        g = capture(torch, mm)
        t = Timer(torch).time(g.replay, reps=reps) / R
        b = affine_bytes(M, N, K, group, asym)
        fl = 2 * M * N * K
        t_hbm, t_tc = b / (pk["hbm_gbs"] * 1e9), fl / (tensor_peak(pk) * 1e12)
        res[f"M{M}"] = {"us": t * 1e6, "GB/s": b / t / 1e9, "TFLOP/s": fl / t / 1e12,
                        "bound": "hbm" if t_hbm >= t_tc else "tensor", "frac": max(t_hbm, t_tc) / t}
        del g, ys
    assert w4.w4_last_device_status() == 0
    del outs
    torch.cuda.empty_cache()
    return res


FP64_NOMINAL_TFLOPS = 1.25  # GB300 dense fp64, nominal (no measured figure in MEASURED_PEAKS.json)


def gptq_set(torch, w4, wl, workload, pk, T=4096, reps=3):
    """GPTQ of one matrix of a workload: the factor of its input's calibration
    statistic (once per input) and the per-matrix quantisation, both fp64."""
    dev = torch.device("cuda", torch.cuda.current_device())
    N, K = wl.SHAPES[workload][0]
    W = wl.weight(workload, 0, device=dev)
    H = wl.calibration_hessian(K, T, seed=wl.seed_for(workload, 0, 4), device=dev)
    U = torch.empty((K, K), dtype=torch.float64, device=dev)
    fws = torch.empty(w4.w4_gptq_factor_workspace_bytes(K), dtype=torch.uint8, device=dev)
    qws = torch.empty(w4.w4_gptq_workspace_bytes(N, K), dtype=torch.uint8, device=dev)
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((N, K // 128), dtype=torch.bfloat16, device=dev)
    w4.w4_gptq_factor(H, U=U, workspace=fws)
    w4.w4_gptq_quantize(W, U, packed=packed, scales=scales, workspace=qws)
    T_ = Timer(torch)
    t_f = T_.time(lambda: w4.w4_gptq_factor(H, U=U, workspace=fws), reps=reps)
    t_q = T_.time(lambda: w4.w4_gptq_quantize(W, U, packed=packed, scales=scales, workspace=qws), reps=reps)
    assert w4.w4_last_device_status() == 0
    f_f = 2.0 / 3.0 * K ** 3  # potrf K³/3 + trtri K³/3
    f_q = 2.0 * N * 128 * sum(K - i2 for i2 in range(128, K, 128)) + N * K * 128
    del W, H, U, fws, qws, packed, scales
    torch.cuda.empty_cache()
    return {"shape": [N, K], "calibration_rows": T,
            "factor": {"ms": t_f * 1e3, "GFLOP/s": f_f / t_f / 1e9, "bound": "fp64",
                       "frac": f_f / t_f / 1e12 / FP64_NOMINAL_TFLOPS, "peak": "nominal 1.25 TFLOP/s fp64"},
            "quantize": {"ms": t_q * 1e3, "GFLOP/s": f_q / t_q / 1e9, "bound": "fp64",
                         "frac": f_q / t_q / 1e12 / FP64_NOMINAL_TFLOPS, "peak": "nominal 1.25 TFLOP/s fp64"}}


_ORACLE_DATA = {}


_BLAS_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def _oracle_worker_init(W_bits, x_bits, K) -> None:
    """Pool initializer: keeps the inputs, sent once per worker."""
    _ORACLE_DATA.update(W=W_bits, x=x_bits, K=K)


def _oracle_task(task):
    """Oracle quantise + fp64 matmul of rows [r0, r1) of the worker's matrix,
    `reps` times; returns the seconds it took in this worker."""
    r0, r1, reps = task
    from oracle import w4_oracle as O

    W, x, K = _ORACLE_DATA["W"][r0:r1], _ORACLE_DATA["x"], _ORACLE_DATA["K"]
    t0 = time.perf_counter()
    for _ in range(reps):
        p, s = O.quantize_rtn(W)
        O.gemm_reference(x, p, s, K)
    return time.perf_counter() - t0


class OraclePool:
    """The CPU oracle, unchanged, run over row slices of one matrix by a pool
    of worker processes (spawned, never forked: the parent holds a CUDA
    context), one BLAS thread each."""

    def __init__(self, workers: int, W_bits, x_bits, K):
        import multiprocessing as mp

        self.workers = workers
        self.rows = W_bits.shape[0]
        # The workers inherit the environment at spawn time, before numpy
        # (needed to unpickle the inputs) starts its BLAS threads.
        saved = {v: os.environ.get(v) for v in _BLAS_THREAD_VARS}
        os.environ.update({v: "1" for v in _BLAS_THREAD_VARS})
        try:
            self.pool = mp.get_context("spawn").Pool(workers, initializer=_oracle_worker_init,
                                                     initargs=(W_bits, x_bits, K))
        finally:
            for v, old in saved.items():
                if old is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = old

    def close(self):
        self.pool.close()
        self.pool.join()

    def run(self, reps=1):
        """Wall seconds for `reps` passes of quantise + matmul over every row,
        the rows split evenly over the workers."""
        w = min(self.workers, self.rows)
        bounds = [self.rows * i // w for i in range(w + 1)]
        t0 = time.perf_counter()
        self.pool.map(_oracle_task, [(bounds[i], bounds[i + 1], reps) for i in range(w)], chunksize=1)
        return time.perf_counter() - t0


def _oracle_inputs(wl, workload, M, rows=None):
    N, K = wl.SHAPES[workload][0]
    W = wl.bits(wl.weight(workload))
    if rows is not None:
        W = W[:rows]
    return W, wl.bits(wl.activations(workload, M, K)), K


def cpu_oracle_baseline(wl, seconds_all=6.0, seconds_one=3.0):
    """The oracle on the host cores: all cores on the headline workload (the
    full 2560×9216 outlier matrix at M = 8, quantise + matmul), and one core
    on row samples of the ffn (M = 1) and outlier (M = 8) workloads."""
    workers = cores()
    out = {}
    W, x, K = _oracle_inputs(wl, HEADLINE, HEADLINE_M)
    pool = OraclePool(workers, W, x, K)
    try:
        pool.run(1)  # worker start-up and imports
        reps = max(1, int(seconds_all / max(pool.run(1), 1e-3)))
        t = pool.run(reps)
        N = W.shape[0]
        out["all_cores"] = {"value": reps * (quant_bytes(N, K) + gemm_bytes(HEADLINE_M, N, K)) / t / 1e9,
                            "cores": workers, "reps": reps, "seconds": t,
                            "sample": f"full {N}x{K} {HEADLINE} matrix per pass (M={HEADLINE_M})"}
    finally:
        pool.close()
    for workload, M in (("ffn", 1), (HEADLINE, HEADLINE_M)):
        W, x, K = _oracle_inputs(wl, workload, M, rows=128)
        one = OraclePool(1, W, x, K)
        try:
            one.run(1)
            reps = max(1, int(seconds_one / max(one.run(1), 1e-3)))
            t = one.run(reps)
        finally:
            one.close()
        N = W.shape[0]
        out[f"one_core_{workload}_M{M}"] = {
            "value": reps * (quant_bytes(N, K) + gemm_bytes(M, N, K)) / t / 1e9, "cores": 1,
            "reps": reps, "seconds": t, "sample": f"{N} of 2560 rows, quantise + matmul"}
    return out


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def config_block(extra=None):
    N, K = (2560, 9216)
    c = {"workload": f"{HEADLINE}: W {N}x{K} bf16 N(0,0.02^2) with 1% input channels x8, "
                     f"RTN sym INT4 g128, x {HEADLINE_M}x{K} bf16 N(0,1)",
         "M": HEADLINE_M, "N": N, "K": K, "group": 128,
         "step": "quantise + matmul: w4_quantize_rtn of one matrix copy, then w4_gemm (M=8) of "
                 "another copy; value = the step's algorithmic bytes (both kernels) / step time",
         "l2": "inputs rotate over copies totalling > 4x L2 (no L2 reuse between steps)"}
    if extra:
        c.update(extra)
    return c


def rank_barrier() -> None:
    """Barrier over all ranks when a process group is up (brackets the timed
    region, with a device synchronize on both sides)."""
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def max_over_ranks(t_local: float, device="cpu") -> float:
    """The job's step time: the largest per-rank time (all-reduce MAX, then a
    barrier).  With no process group, or one rank, the local time."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return t_local
    t = torch.tensor([t_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def job_value(bytes_per_rank_step: float, world: int, t_step: float) -> float:
    """Whole-job GB/s: every rank processes its own copy of the step's work
    (replicas, weak scaling), timed by the slowest rank."""
    return world * bytes_per_rank_step / t_step / 1e9


def run_gpu(args):
    import torch
    import gemm_rtn_sym_gb300 as w4
    from gemm_rtn_sym_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    w4.load()
    pk = peaks()
    res = headline(torch, w4, wl, args.steps, args.warmup, pk)
    t_step = max_over_ranks(res["ms_per_step"] / 1e3, device="cuda")
    N, K = wl.SHAPES[HEADLINE][0]
    bytes_step = quant_bytes(N, K) + gemm_bytes(HEADLINE_M, N, K)
    value = job_value(bytes_step, world, t_step)

    sub = {}
    if not args.no_sub and rank == 0:
        only = set(filter(None, args.only.split(",")))
        want = lambda k: not only or k in only
        if want("ffn"):
            sub["ffn_m1"] = gemm_set(torch, w4, wl, "ffn", [1], pk)["M1"]
        if want("outlier"):
            sub["outlier_m8"] = gemm_set(torch, w4, wl, "outlier", [8], pk)["M8"]
        if want("quant"):
            sub["quant_ffn"] = quant_set(torch, w4, wl, "ffn", pk)
        if want("gptq"):
            sub["gptq_ffn"] = gptq_set(torch, w4, wl, "ffn", pk)
        if want("affine"):
            for group, asym in ((128, True), (64, True), (32, True), (32, False)):
                key = f"affine_g{group}_{'asym' if asym else 'sym'}"
                sub[key + "_outlier"] = affine_set(torch, w4, wl, "outlier", 0, [1, 8], group, asym, pk)
                sub[key + "_gateup70b"] = affine_set(torch, w4, wl, "layer70b", 2, [208], group, asym, pk, reps=5)
        if want("awq"):
            sub["quant_scaled_outlier"] = quant_set(torch, w4, wl, "outlier", pk, scaled=True)
            sub["scale_act_m8"] = scale_act_set(torch, w4, wl, "outlier", 8, pk)
            sub["scale_act_m208"] = scale_act_set(torch, w4, wl, "layer70b", 208, pk)
        if want("layer27b"):
            sub["layer27b"] = gemm_set(torch, w4, wl, "layer27b", wl.ROWS["layer27b"], pk, reps=10)
        if want("layer70b"):
            sub["layer70b"] = gemm_set(torch, w4, wl, "layer70b", wl.ROWS["layer70b"], pk, reps=5)
        if want("layer27b_grouped"):
            sub["layer27b_grouped"] = gemm_set(torch, w4, wl, "layer27b", wl.ROWS["layer27b"], pk, reps=10,
                                               grouped=True)
        if want("stack4b") and not args.no_sweep:
            sub["stack4b"] = gemm_set(torch, w4, wl, "stack4b", wl.ROWS["stack4b"], pk, reps=3)
        if want("layer70b_grouped"):
            sub["layer70b_grouped"] = gemm_set(torch, w4, wl, "layer70b", wl.ROWS["layer70b"], pk, reps=5,
                                               grouped=True)
        if want("stack4b_grouped") and not args.no_sweep:
            sub["stack4b_grouped"] = gemm_set(torch, w4, wl, "stack4b", wl.ROWS["stack4b"], pk, reps=3, grouped=True)
        if want("affine_grouped"):
            for group, asym in ((128, True), (32, True)):
                key = f"layer27b_grouped_g{group}_{'asym' if asym else 'sym'}"
                sub[key] = gemm_set(torch, w4, wl, "layer27b", [1, 8, 32], pk, reps=10, grouped=True,
                                    fmt=(group, asym))

    if rank != 0:
        return
    if not args.no_sub:
        sub["hbm_read_probe"] = read_probe(torch)
    cpu = cpu_oracle_baseline(wl)
    allc = cpu["all_cores"]
    k = res["kernels"]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "dtype_detail": "bf16 activations x int4 weights (decoded to bf16), fp32 accumulate",
        "data": "synthetic (seeded; no model weights)",
        "config": config_block({"parallelism": f"replicas x{world}" if world > 1 else "single GPU"}),
        "quant_frac": round(k["quantize"]["frac"], 4), "gemm_m8_frac": round(k["gemm_m8"]["frac"], 4),
        "roofline": res["roofline"], "kernels": res["kernels"], "e2e": res["e2e"],
        "clocks": res["clocks"], "gpu_launches": res["gpu_launches"],
        "cpu_baseline": {"value": allc["value"], "unit": "GB/s", "cores": allc["cores"], "kind": "oracle",
                         "sample": f"{allc['sample']}, {allc['reps']} passes in {allc['seconds']:.1f} s, "
                                   f"oracle unchanged on a spawned process pool, one BLAS thread per worker",
                         "one_core": {kk[9:]: round(v["value"], 4) for kk, v in cpu.items()
                                      if kk.startswith("one_core_")}},
        "peaks": {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                  "bf16_tflops_sustained": pk.get("bf16_tflops_sustained"), "source": pk["source"],
                  "hbm_nominal_gbs": HBM_NOMINAL_GBS},
        "configs": compact_configs(sub, pk),
    }
    print("# detail " + json.dumps({"sub": sub, "cpu_baseline": cpu, "rotation": res["rotation"]}), flush=True)
    print(json.dumps(line, separators=(",", ":")), flush=True)


def read_probe(torch, gib=4, reps=5):
    """Read-only HBM streaming figure for context beside the copy-based peak:
    torch.sum over a 4 GiB fp32 tensor (a library reduction, not this path)."""
    a = torch.ones(gib * (1 << 28), dtype=torch.float32, device="cuda")
    a.sum()
    t = Timer(torch).time(lambda: a.sum(), reps=reps)
    b = a.numel() * 4
    del a
    torch.cuda.empty_cache()
    return {"GB/s": b / t / 1e9, "what": f"torch.sum over {gib} GiB fp32"}


def compact_configs(sub, pk):
    """The five workloads at a glance, short enough to stay in a log tail:
    [us per launch (a layer or the stack: per set of matrices), fraction of
    the roofline that bounds it]; a third entry "tc" marks a tensor-bound
    case, graded against the measured burst bf16 peak."""
    def entry(v):
        e = [round(v["us"], 1), round(v["frac"], 3)]
        if v.get("bound") == "tensor":
            e.append("tc")
        return e

    c = {"legend": "[us, frac of roofline]; HBM %.0f GB/s measured (x%.3f for the nominal %.0f), "
                   "tc = tensor-bound vs burst bf16 %.0f TFLOP/s" % (
                       pk["hbm_gbs"], pk["hbm_gbs"] / HBM_NOMINAL_GBS, HBM_NOMINAL_GBS, pk["bf16_tflops"])}
    for key, label in (("ffn_m1", "1_ffn"), ("outlier_m8", "2_outlier")):
        if key in sub:
            c[label] = entry(sub[key])
    for key, label in (("layer27b", "3_layer27b"), ("layer27b_grouped", "3_layer27b_grouped"),
                       ("layer70b", "4_layer70b"), ("layer70b_grouped", "4_layer70b_grouped"),
                       ("stack4b", "5_stack4b"), ("stack4b_grouped", "5_stack4b_grouped")):
        if key in sub:
            c[label] = {m: entry(v) for m, v in sub[key].items()}
    if "quant_ffn" in sub:
        c["quant_ffn"] = entry(sub["quant_ffn"])
    return c


def run_reference(args):
    """The CPU oracle as the reference arm: each step is one pass of quantise +
    matmul (M = 8) over the full headline matrix, its rows split over a
    spawned pool with one worker per host core."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from gemm_rtn_sym_gb300 import workloads as wl

    W, x, K = _oracle_inputs(wl, HEADLINE, HEADLINE_M)
    N = W.shape[0]
    workers = cores()
    pool = OraclePool(workers, W, x, K)
    try:
        for _ in range(max(1, args.warmup)):
            pool.run(1)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            pool.run(1)
        el = time.perf_counter() - t0
    finally:
        pool.close()
    b = quant_bytes(N, K) + gemm_bytes(HEADLINE_M, N, K)
    v = b * args.steps / el / 1e9
    sample = (f"each step: oracle quantise + fp64 matmul (M={HEADLINE_M}) of all {N} rows, "
              f"split over {workers} spawned worker processes (one BLAS thread each)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": config_block(),
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": workers, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
