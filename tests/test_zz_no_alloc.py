"""w4_gemm_grouped_noalloc: the grouped matmul through the library's static
plan buffer, for callers that cannot allocate device memory.  Collected last
(file name), so that a run stopping at its first failure has run every other
test first.  Results must equal the plan-based w4_gemm_grouped bit for bit
(same kernels, same schedule) on two successive calls with different
activations, and match the oracle; two calls with different problem sets,
queued back to back on one stream with no synchronisation between them,
must each give their own problems' results (the second call's plan must not
overwrite the first one's while its kernels still read it)."""
import pytest
import torch

import gemm_rtn_sym_gb300 as w4
from gemm_rtn_sym_gb300 import workloads as wl
from tests.helpers import check_gemm, quantize_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _problems(cuda_lib):
    shapes = [(2560, 512), (300, 1152), (1000, 4096), (64, 256)]
    Ms = [1, 13, 40, 208]
    Ws, probs = [], []
    for i, ((N, K), M) in enumerate(zip(shapes, Ms)):
        W = wl.random_bf16((N, K), 0.02, seed=500 + i, device=DEV)
        packed, scales = quantize_gpu(cuda_lib, W)
        x = wl.random_bf16((M, K), 1.0, seed=600 + i, device=DEV)
        Ws.append(W)
        probs.append((x, packed, scales, torch.empty((M, N), dtype=torch.bfloat16, device=DEV)))
    return Ws, probs


def test_noalloc_matches_plan_on_two_calls(cuda_lib):
    Ws, probs = _problems(cuda_lib)
    ref = [(x, p, s, torch.empty_like(y)) for (x, p, s, y) in probs]
    plan = w4.w4_grouped_plan(ref)
    for call in range(2):
        if call == 1:  # new activations in the same buffers
            for i, (x, _, _, _) in enumerate(probs):
                x.copy_(wl.random_bf16(tuple(x.shape), 1.0, seed=700 + i, device=DEV))
        w4.w4_gemm_grouped_noalloc(probs)
        w4.w4_gemm_grouped(plan)
        torch.cuda.synchronize()
        assert w4.w4_last_device_status() == 0
        for (x, _, _, y), (_, _, _, yr), W in zip(probs, ref, Ws):
            assert torch.equal(y.view(torch.int16), yr.view(torch.int16))
            check_gemm(W, x, y)


def test_noalloc_rejects_a_plan_larger_than_its_buffer(cuda_lib):
    W = wl.random_bf16((1, 128), 0.02, seed=1, device=DEV)
    packed, scales = quantize_gpu(cuda_lib, W)
    x = wl.random_bf16((1, 128), 1.0, seed=2, device=DEV)
    n = 6000  # 6000 problem records of 384 bytes exceed the 2 MB buffer
    ys = torch.empty((n, 1), dtype=torch.bfloat16, device=DEV)
    probs = [(x, packed, scales, ys[i:i + 1]) for i in range(n)]
    with pytest.raises(w4.W4Error) as e:
        w4.w4_gemm_grouped_noalloc(probs)
    assert e.value.status == w4.W4_ERR_UNSUPPORTED
    # a plan that fits still runs
    w4.w4_gemm_grouped_noalloc(probs[:8])
    torch.cuda.synchronize()
    check_gemm(W, x, ys[3:4])


def test_noalloc_two_problem_sets_back_to_back(cuda_lib):
    """Call A (small-M problems only) and call B (a tensor-core problem and a
    small-M problem of other shapes) share the static plan array: queued on one
    stream without a synchronisation, A's kernels must still see A's plan."""
    def make(shapes_ms, seed):
        Ws, probs = [], []
        for i, ((N, K), M) in enumerate(shapes_ms):
            W = wl.random_bf16((N, K), 0.02, seed=seed + i, device=DEV)
            packed, scales = quantize_gpu(cuda_lib, W)
            x = wl.random_bf16((M, K), 1.0, seed=seed + 50 + i, device=DEV)
            Ws.append(W)
            probs.append((x, packed, scales, torch.empty((M, N), dtype=torch.bfloat16, device=DEV)))
        return Ws, probs

    Wa, a = make([((4096, 2048), 1), ((640, 4608), 8), ((300, 1152), 5)], 900)
    Wb, b = make([((1000, 1024), 40), ((512, 3072), 16)], 950)
    torch.cuda.synchronize()
    w4.w4_gemm_grouped_noalloc(a)
    w4.w4_gemm_grouped_noalloc(b)
    torch.cuda.synchronize()
    assert w4.w4_last_device_status() == 0
    for W, (x, _, _, y) in zip(Wa + Wb, a + b):
        check_gemm(W, x, y)
