"""GPU parity of the grouped matmul (w4_gemm_grouped) against the CPU oracle:
every problem of a plan element by element within 4e-3·Σ|ŵx| + 1 bf16 ulp,
outputs guarded, runs deterministic, plans reusable and graph-capturable."""
import pytest
import torch

import gemm_rtn_sym_gb300 as w4
from gemm_rtn_sym_gb300 import workloads as wl
from tests.helpers import check_gemm, guarded, guards_intact, quantize_gpu, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make_problems(cuda_lib, shapes, Ms, seed=0):
    Ws, probs, bufs = [], [], []
    for i, ((N, K), M) in enumerate(zip(shapes, Ms)):
        W = wl.random_bf16((N, K), 0.02, seed=seed + 31 * i + N, device=DEV)
        packed, scales = quantize_gpu(cuda_lib, W)
        x = wl.random_bf16((M, K), 1.0, seed=seed + 17 * i + M, device=DEV)
        y, ybuf = guarded((M, N), torch.bfloat16, DEV)
        Ws.append(W)
        probs.append((x, packed, scales, y))
        bufs.append(ybuf)
    return Ws, probs, bufs


SHAPES = [(1, 128), (7, 256), (129, 1152), (200, 4096), (64, 384), (2560, 512), (96, 30720)]


@pytest.mark.parametrize("Ms,rows", [([1, 2, 3, 5, 8, 1, 4], 8), ([9, 1, 13, 16, 8, 12, 11], 16),
                                     ([1, 1, 2, 1, 2, 2, 1], 2), ([3, 1, 4, 2, 4, 1, 3], 4),
                                     ([1, 1, 1, 1, 1, 1, 1], 2)])
def test_grouped_small_problems(cuda_lib, Ms, rows):
    """Plans whose largest M selects each one-tile variant of the small-M
    kernel (2, 4 or 8 token rows staged) and the 16-row variant."""
    Ws, probs, bufs = make_problems(cuda_lib, SHAPES, Ms, seed=len(Ms) * Ms[0] + sum(Ms))
    plan = w4.w4_grouped_plan(probs)
    assert plan.plan.token_rows == rows
    w4.w4_gemm_grouped(plan)
    torch.cuda.synchronize()
    assert w4.w4_last_device_status() == 0
    for W, (x, _, _, y), b in zip(Ws, probs, bufs):
        assert guards_intact(b), "grouped matmul wrote outside an output"
        check_gemm(W, x, y)
    # deterministic, and the plan is reusable
    first = [p[3].clone() for p in probs]
    for _ in range(3):
        w4.w4_gemm_grouped(plan)
    torch.cuda.synchronize()
    for f, p in zip(first, probs):
        assert torch.equal(f.view(torch.int16), p[3].view(torch.int16))


def test_grouped_new_inputs_and_graph_replay(cuda_lib):
    Ws, probs, _ = make_problems(cuda_lib, SHAPES[:5], [1, 4, 8, 2, 3], seed=5)
    plan = w4.w4_grouped_plan(probs)
    g = torch.cuda.CUDAGraph()
    w4.w4_gemm_grouped(plan)  # warm-up outside capture
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        w4.w4_gemm_grouped(plan)
    for rep in range(2):
        for i, (x, _, _, _) in enumerate(probs):  # new activations in the same buffers
            x.copy_(wl.random_bf16(tuple(x.shape), 1.0, seed=1000 + 10 * rep + i, device=DEV))
        g.replay()
        torch.cuda.synchronize()
        for W, (x, _, _, y) in zip(Ws, probs):
            check_gemm(W, x, y)


def test_grouped_unaligned_scales(cuda_lib):
    """Scales at an address that is 2-byte but not 8-byte aligned are staged
    one element at a time (otherwise four groups of a row per 8-byte load):
    the outputs are bit-identical to those of the same problems with aligned
    scales."""
    shapes = [(200, 4096), (2560, 512), (96, 30720)]
    Ws, probs, _ = make_problems(cuda_lib, shapes, [1, 3, 2], seed=11)
    w4.w4_gemm_grouped(w4.w4_grouped_plan(probs))
    moved = []
    for x, p, s, y in probs:
        buf = torch.empty(s.numel() + 4, dtype=s.dtype, device=DEV)
        s2 = buf[1:1 + s.numel()].view(s.shape)
        s2.copy_(s)
        assert s2.data_ptr() % 8 == 2
        moved.append((x, p, s2, torch.empty_like(y)))
    w4.w4_gemm_grouped(w4.w4_grouped_plan(moved))
    torch.cuda.synchronize()
    assert w4.w4_last_device_status() == 0
    for W, (x, _, _, y), (_, _, _, y2) in zip(Ws, probs, moved):
        check_gemm(W, x, y)
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_grouped_three_ctas_per_sm_ragged_groups(cuda_lib):
    """A plan of many equal items (64 problems × 5 row blocks) runs three CTAs
    per SM, where the producer warp stages the scales; K = 128·(9..12) gives
    rows whose scales are loaded element by element (groups not a multiple of
    four) as well as in 8-byte loads. Every problem within the parity bound."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shapes = [(320, 128 * (9 + i % 4)) for i in range(64)]
    Ws, probs, bufs = make_problems(cuda_lib, shapes, [1 + i % 2 for i in range(64)], seed=21)
    plan = w4.w4_grouped_plan(probs)
    assert plan.plan.ctas > 2 * sms, plan.plan.ctas
    w4.w4_gemm_grouped(plan)
    torch.cuda.synchronize()
    assert w4.w4_last_device_status() == 0
    for W, (x, _, _, y), b in zip(Ws, probs, bufs):
        assert guards_intact(b), "grouped matmul wrote outside an output"
        check_gemm(W, x, y)


@pytest.mark.parametrize("Ms", [[17, 33, 64, 208, 100, 257, 19], [1, 40, 13, 208, 8, 24, 2],
                                [32, 28, 1, 5, 64, 25, 33]])
def test_grouped_tensor_and_mixed(cuda_lib, Ms):
    """Problems with M ≥ 25 take the tensor-core grouped kernel, the others the
    small-M kernel at the token width of the largest (24 rows in the second
    set); a plan mixing both kinds runs both kernels."""
    Ws, probs, bufs = make_problems(cuda_lib, SHAPES, Ms, seed=3 + Ms[1])
    plan = w4.w4_grouped_plan(probs)
    assert plan.plan.tc_items > 0
    w4.w4_gemm_grouped(plan)
    torch.cuda.synchronize()
    assert w4.w4_last_device_status() == 0
    for W, (x, _, _, y), b in zip(Ws, probs, bufs):
        assert guards_intact(b), "grouped matmul wrote outside an output"
        check_gemm(W, x, y)
    first = [p[3].clone() for p in probs]
    for _ in range(2):
        w4.w4_gemm_grouped(plan)
    torch.cuda.synchronize()
    for f, p in zip(first, probs):
        assert torch.equal(f.view(torch.int16), p[3].view(torch.int16))


def test_grouped_rejects(cuda_lib):
    _, probs, _ = make_problems(cuda_lib, [(64, 256), (64, 256)], [4, 4], seed=9)
    x, p, s, y = probs[0]
    with pytest.raises(w4.W4Error) as e:  # two problems writing the same output
        w4.w4_grouped_plan([(x, p, s, y), (probs[1][0], probs[1][1], probs[1][2], y)])
    assert e.value.status == w4.W4_ERR_INVALID_ARG
    x1, p1, s1, y1 = probs[1]
    with pytest.raises(w4.W4Error) as e:  # output overlapping another problem's input
        w4.w4_grouped_plan([(x, p, s, x1.view(-1)[:256].view(4, 64)), (x1, p1, s1, y1)])
    assert e.value.status == w4.W4_ERR_INVALID_ARG


@pytest.mark.slow
@pytest.mark.parametrize("M", [1, 2, 4, 5, 13, 24, 32])
def test_grouped_layer27b_sampled(cuda_lib, M):
    shapes = wl.SHAPES["layer27b"]
    Ws, probs = [], []
    for i, (N, K) in enumerate(shapes):
        W = wl.weight("layer27b", i, device=DEV)
        packed, scales = quantize_gpu(cuda_lib, W)
        x = wl.activations("layer27b", M, K, i, device=DEV)
        Ws.append(W)
        probs.append((x, packed, scales, torch.empty((M, N), dtype=torch.bfloat16, device=DEV)))
    plan = w4.w4_grouped_plan(probs)
    w4.w4_gemm_grouped(plan)
    torch.cuda.synchronize()
    assert w4.w4_last_device_status() == 0
    for i, (W, (x, _, _, y)) in enumerate(zip(Ws, probs)):
        rows = torch.from_numpy(sample_rows(W.shape[0], 64, seed=i)).to(DEV)
        check_gemm(W[rows].cpu(), x, y[:, rows])


@pytest.mark.slow
def test_grouped_stack_subset(cuda_lib):
    """Two matrices of each stack shape (8 problems, 4 shapes) in one plan."""
    shapes = wl.SHAPES["stack4b"]
    pick = [0, 1, 56, 57, 112, 113, 156, 157]
    Ws, probs = [], []
    for j, i in enumerate(pick):
        N, K = shapes[i]
        W = wl.weight("stack4b", i, device=DEV)
        packed, scales = quantize_gpu(cuda_lib, W)
        x = wl.activations("stack4b", 8, K, i, device=DEV)
        Ws.append(W)
        probs.append((x, packed, scales, torch.empty((8, N), dtype=torch.bfloat16, device=DEV)))
    plan = w4.w4_grouped_plan(probs)
    w4.w4_gemm_grouped(plan)
    torch.cuda.synchronize()
    for j, (W, (x, _, _, y)) in enumerate(zip(Ws, probs)):
        rows = torch.from_numpy(sample_rows(W.shape[0], 48, seed=j)).to(DEV)
        check_gemm(W[rows].cpu(), x, y[:, rows])


@pytest.mark.slow
def test_grouped_layer70b_m208_sampled(cuda_lib):
    shapes = wl.SHAPES["layer70b"]
    Ws, probs = [], []
    for i, (N, K) in enumerate(shapes):
        W = wl.weight("layer70b", i, device=DEV)
        packed, scales = quantize_gpu(cuda_lib, W)
        x = wl.activations("layer70b", 208, K, i, device=DEV)
        Ws.append(W)
        probs.append((x, packed, scales, torch.empty((208, N), dtype=torch.bfloat16, device=DEV)))
    plan = w4.w4_grouped_plan(probs)
    w4.w4_gemm_grouped(plan)
    torch.cuda.synchronize()
    assert w4.w4_last_device_status() == 0
    for i, (W, (x, _, _, y)) in enumerate(zip(Ws, probs)):
        rows = torch.from_numpy(sample_rows(W.shape[0], 32, seed=i)).to(DEV)
        check_gemm(W[rows].cpu(), x, y[:, rows])


@pytest.mark.slow
def test_grouped_tensor_repeat_is_bit_identical(cuda_lib):
    """The tensor-core grouped kernel's rings hand shared-memory slots back to
    TMA while other warps keep working: 40 back-to-back runs of the 70B-class
    layer at M = 208 must give bit-identical outputs (a slot released before
    its data was read shows up as a rare changed element), and the first run
    matches the oracle on sampled rows."""
    shapes = wl.SHAPES["layer70b"]
    Ws, probs = [], []
    for i, (N, K) in enumerate(shapes):
        W = wl.weight("layer70b", i, device=DEV)
        packed, scales = quantize_gpu(cuda_lib, W)
        x = wl.activations("layer70b", 208, K, i, device=DEV)
        Ws.append(W)
        probs.append((x, packed, scales, torch.empty((208, N), dtype=torch.bfloat16, device=DEV)))
    plan = w4.w4_grouped_plan(probs)
    w4.w4_gemm_grouped(plan)
    torch.cuda.synchronize()
    first = [p[3].clone() for p in probs]
    for i, (W, (x, _, _, _)) in enumerate(zip(Ws, probs)):
        rows = torch.from_numpy(sample_rows(W.shape[0], 8, seed=100 + i)).to(DEV)
        check_gemm(W[rows].cpu(), x, first[i][:, rows])
    changed = 0
    for _ in range(40):
        w4.w4_gemm_grouped(plan)
        torch.cuda.synchronize()
        for f, p in zip(first, probs):
            changed += int((f.view(torch.int16) != p[3].view(torch.int16)).sum())
    assert w4.w4_last_device_status() == 0
    assert changed == 0, f"{changed} output elements differed between runs"
