"""GPU parity of the affine formats (Qwen3.5-4B quantisation study, §1
group-quantisation equation with a free zero point z; §2 settings table on
smaller groups) against the CPU oracle: w4_quantize_rtn at groups 32/64 and
w4_quantize_rtn_asym at 32/64/128 must give the oracle's packed bytes, scale
bits and zeros exactly; w4_gemm_affine must stay within the parity bound on
both kernel paths."""
import numpy as np
import pytest
import torch

from gemm_rtn_sym_gb300 import W4_PATH_SMALL_M, W4_PATH_TENSOR
from gemm_rtn_sym_gb300 import workloads as wl
from oracle import w4_oracle as O
from tests.helpers import guarded, guards_intact
from tests.test_gpu_quantize import tie_and_range_matrix

pytestmark = pytest.mark.gpu
DEV = "cuda"


def quantize_gpu(w4, W, group, asym):
    N, K = W.shape
    packed, pbuf = guarded((N, K // 2), torch.uint8, W.device)
    scales, sbuf = guarded((N, K // group), torch.bfloat16, W.device)
    if asym:
        zeros, zbuf = guarded((N, K // group), torch.uint8, W.device)
        zeros = zeros.view(torch.int8)
        w4.w4_quantize_rtn_asym(W, group, packed=packed, scales=scales, zeros=zeros)
    else:
        zeros, zbuf = None, None
        w4.w4_quantize_rtn(W, group, packed=packed, scales=scales)
    torch.cuda.synchronize()
    assert guards_intact(pbuf) and guards_intact(sbuf), "quantiser wrote outside its outputs"
    if zbuf is not None:
        assert guards_intact(zbuf), "quantiser wrote outside the zeros"
    return packed, scales, zeros


def check(W, group, asym, packed, scales, zeros):
    Wb = wl.bits(W)
    if asym:
        p_ref, s_ref, z_ref = O.quantize_rtn_asym(Wb, group)
        zg = zeros.cpu().numpy()
        assert np.array_equal(zg, z_ref), f"zeros differ in {np.count_nonzero(zg != z_ref)} places"
    else:
        p_ref, s_ref = O.quantize_rtn(Wb, group)
    sg, pg = wl.bits(scales), packed.cpu().numpy()
    assert np.array_equal(sg, s_ref), f"scale bits differ in {np.count_nonzero(sg != s_ref)} places"
    assert np.array_equal(pg, p_ref), f"packed bytes differ in {np.count_nonzero(pg != p_ref)} places"


FORMATS = [(32, False), (64, False), (32, True), (64, True), (128, True)]


@pytest.mark.parametrize("group,asym", FORMATS)
@pytest.mark.parametrize("N,K", [(1, 128), (7, 256), (129, 1152), (300, 9216), (33, 2560)])
def test_quantize_small_shapes(cuda_lib, N, K, group, asym):
    W = wl.random_bf16((N, K), 0.02, seed=N * 1000 + K + group, device=DEV)
    check(W, group, asym, *quantize_gpu(cuda_lib, W, group, asym))


@pytest.mark.parametrize("group,asym", FORMATS)
def test_quantize_full_outlier(cuda_lib, group, asym):
    W = wl.weight("outlier", device=DEV)
    check(W, group, asym, *quantize_gpu(cuda_lib, W, group, asym))


@pytest.mark.parametrize("group,asym", FORMATS)
def test_quantize_every_quotient_and_tie(cuda_lib, group, asym):
    """Normal, tiny and subnormal groups, exact ties, signed mixes."""
    Wc = tie_and_range_matrix()
    check(Wc, group, asym, *quantize_gpu(cuda_lib, Wc.to(DEV), group, asym))


@pytest.mark.parametrize("group,asym", FORMATS)
def test_quantize_16_byte_aligned_input(cuda_lib, group, asym):
    W = wl.random_bf16((129, 1152), 0.02, seed=7 + group, device=DEV)
    N, K = W.shape
    flat = torch.empty(N * K + 64, dtype=torch.bfloat16, device=DEV)
    Wv = flat[8:8 + N * K].view(N, K)
    Wv.copy_(W)
    check(W, group, asym, *quantize_gpu(cuda_lib, Wv, group, asym))


def test_asym_special_groups(cuda_lib):
    K = 512
    W = torch.zeros((7, K), dtype=torch.float32)
    W[1, :128] = 0.25 + torch.arange(128) / 512      # all positive
    W[2, :128] = -(0.25 + torch.arange(128) / 512)   # all negative
    W[3, :128] = 0.75                                # constant
    W[4, 128:256] = torch.linspace(-1e-38, 3e-38, 128)
    W[5, 256:] = 3e-39
    Wb = W.to(torch.bfloat16)
    Wb.view(torch.int16)[6, :128] = -32737          # 0x801F: subnormal, clipped zero point
    Wb.view(torch.int16)[6, 130] = 1
    for group in (32, 64, 128):
        check(Wb, group, True, *quantize_gpu(cuda_lib, Wb.to(DEV), group, True))


@pytest.mark.parametrize("group,asym", FORMATS + [(128, False)])
@pytest.mark.parametrize("M", [1, 5, 8, 16, 17, 33, 208])
def test_gemm_affine_parity(cuda_lib, group, asym, M):
    N, K = 300, 1152
    W = wl.random_bf16((N, K), 0.02, seed=11 + group, device=DEV)
    x = wl.random_bf16((M, K), 1.0, seed=M, device=DEV)
    packed, scales, zeros = quantize_gpu(cuda_lib, W, group, asym)
    Wb = wl.bits(W)
    if asym:
        p_ref, s_ref, z_ref = O.quantize_rtn_asym(Wb, group)
    else:
        (p_ref, s_ref), z_ref = O.quantize_rtn(Wb, group), None
    y_ref, s_abs = O.gemm_reference(wl.bits(x), p_ref, s_ref, K, group, z_ref)
    for path in (W4_PATH_SMALL_M, W4_PATH_TENSOR):
        y, ybuf = guarded((M, N), torch.bfloat16, x.device)
        cuda_lib.w4_gemm_affine(x, packed, scales, zeros, group=group, out=y, path=path)
        torch.cuda.synchronize()
        assert guards_intact(ybuf), "matmul wrote outside y"
        assert cuda_lib.w4_last_device_status() == 0
        excess = O.parity_excess(wl.bits(y), y_ref, s_abs)
        assert float(excess.max()) <= 1.0, (path, float(excess.max()))


@pytest.mark.parametrize("group,asym", FORMATS)
@pytest.mark.parametrize("M", [1, 8, 208])
def test_gemm_affine_full_outlier_sampled(cuda_lib, group, asym, M):
    W = wl.weight("outlier", device=DEV)
    N, K = W.shape
    x = wl.activations("outlier", M, K, device=DEV)
    packed, scales, zeros = quantize_gpu(cuda_lib, W, group, asym)
    y = cuda_lib.w4_gemm_affine(x, packed, scales, zeros, group=group)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(8), np.arange(N - 8, N),
                                     np.random.default_rng(group + M).choice(N, 96, replace=False)]))
    Wb = wl.bits(W)[rows]
    if asym:
        p_ref, s_ref, z_ref = O.quantize_rtn_asym(Wb, group)
    else:
        (p_ref, s_ref), z_ref = O.quantize_rtn(Wb, group), None
    y_ref, s_abs = O.gemm_reference(wl.bits(x), p_ref, s_ref, K, group, z_ref)
    excess = O.parity_excess(wl.bits(y)[:, rows], y_ref, s_abs)
    assert float(excess.max()) <= 1.0


def test_affine_group128_symmetric_is_w4_gemm(cuda_lib):
    W = wl.random_bf16((256, 2048), 0.02, seed=3, device=DEV)
    packed, scales = cuda_lib.w4_quantize_rtn(W)
    for M in (1, 8, 40):
        x = wl.random_bf16((M, 2048), 1.0, seed=M + 1, device=DEV)
        a = cuda_lib.w4_gemm_ex(x, packed, scales)
        b = cuda_lib.w4_gemm_affine(x, packed, scales, None, group=128)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("group", [32, 64, 128])
def test_gemm_affine_repeat_is_bit_identical(cuda_lib, group):
    W = wl.random_bf16((512, 4096), 0.02, seed=5, device=DEV)
    packed, scales, zeros = quantize_gpu(cuda_lib, W, group, True)
    for M in (3, 13, 64):
        x = wl.random_bf16((M, 4096), 1.0, seed=M, device=DEV)
        ys = [cuda_lib.w4_gemm_affine(x, packed, scales, zeros, group=group) for _ in range(5)]
        torch.cuda.synchronize()
        assert all(torch.equal(ys[0].view(torch.int16), v.view(torch.int16)) for v in ys[1:])


@pytest.mark.parametrize("group", [32, 64])
def test_gemm_affine_unaligned_scales_and_zeros(cuda_lib, group):
    """Scales only 2-byte aligned and zeros at an odd address take the
    unpaired loads; the result must equal the one from aligned buffers."""
    W = wl.random_bf16((200, 1152), 0.02, seed=31, device=DEV)
    N, K = W.shape
    packed, scales, zeros = quantize_gpu(cuda_lib, W, group, True)
    sb = torch.empty(N * (K // group) + 1, dtype=torch.bfloat16, device=DEV)
    s_odd = sb[1:].view(N, K // group)
    s_odd.copy_(scales)
    zb = torch.empty(N * (K // group) + 1, dtype=torch.int8, device=DEV)
    z_odd = zb[1:].view(N, K // group)
    z_odd.copy_(zeros)
    assert s_odd.data_ptr() % 4 == 2 and z_odd.data_ptr() % 2 == 1
    for M in (8, 40):
        x = wl.random_bf16((M, K), 1.0, seed=M, device=DEV)
        for path in (W4_PATH_SMALL_M, W4_PATH_TENSOR):
            a = cuda_lib.w4_gemm_affine(x, packed, scales, zeros, group=group, path=path)
            b = cuda_lib.w4_gemm_affine(x, packed, s_odd, z_odd, group=group, path=path)
            torch.cuda.synchronize()
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (M, path)


GROUPED_SHAPES = [(300, 1152), (7, 256), (129, 2560), (64, 384), (1000, 512)]


@pytest.mark.parametrize("group,asym", FORMATS)
@pytest.mark.parametrize("Ms", [[1, 2, 1, 2, 1], [8, 3, 5, 1, 7], [16, 9, 13, 4, 2], [24, 32, 17, 1, 30],
                                [40, 208, 33, 8, 1]])
def test_grouped_affine_parity(cuda_lib, group, asym, Ms):
    """The grouped matmul over the affine formats (w4_grouped_plan_init_affine):
    every problem within the parity bound of the oracle's dequantised matmul
    with its zeros, on plans that select every small-M variant (2 to 24 token
    rows staged) and mix in the tensor-core kernel (M ≥ 25); repeat runs
    bit-identical."""
    probs, refs, zs = [], [], []
    for i, ((N, K), M) in enumerate(zip(GROUPED_SHAPES, Ms)):
        W = wl.random_bf16((N, K), 0.02, seed=40 + 7 * i + group, device=DEV)
        x = wl.random_bf16((M, K), 1.0, seed=90 + M + i, device=DEV)
        packed, scales, zeros = quantize_gpu(cuda_lib, W, group, asym)
        # one problem without zeros in an asymmetric plan: symmetric codes there
        if asym and i == 3:
            packed, scales, zeros = quantize_gpu(cuda_lib, W, group, False)
        y, ybuf = guarded((M, N), torch.bfloat16, DEV)
        probs.append((x, packed, scales, y))
        zs.append(zeros)
        Wb = wl.bits(W)
        if zeros is not None:
            p_ref, s_ref, z_ref = O.quantize_rtn_asym(Wb, group)
        else:
            (p_ref, s_ref), z_ref = O.quantize_rtn(Wb, group), None
        refs.append((O.gemm_reference(wl.bits(x), p_ref, s_ref, K, group, z_ref), ybuf))
    plan = cuda_lib.w4_grouped_plan(probs, group=group, zeros=zs if asym else None)
    assert plan.plan.format == group
    cuda_lib.w4_gemm_grouped(plan)
    torch.cuda.synchronize()
    assert cuda_lib.w4_last_device_status() == 0
    first = []
    for (x, _, _, y), ((y_ref, s_abs), ybuf) in zip(probs, refs):
        assert guards_intact(ybuf), "grouped matmul wrote outside an output"
        excess = O.parity_excess(wl.bits(y), y_ref, s_abs)
        assert float(excess.max()) <= 1.0, float(excess.max())
        first.append(y.clone())
    cuda_lib.w4_gemm_grouped(plan)
    torch.cuda.synchronize()
    for f, (_, _, _, y) in zip(first, probs):
        assert torch.equal(f.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("group", [32, 64, 128])
def test_grouped_affine_unaligned_scales_and_zeros(cuda_lib, group):
    """Scales at a 2-byte and zero points at a 1-byte aligned address are
    staged element by element instead of in 4- to 16-byte copies: outputs
    bit-identical to those of the same problems with aligned ones."""
    shapes = [(200, 4096), (96, 2560), (64, 1152)]
    probs, zs, moved, zs2 = [], [], [], []
    for i, (N, K) in enumerate(shapes):
        W = wl.random_bf16((N, K), 0.02, seed=70 + i + group, device=DEV)
        x = wl.random_bf16((1 + 3 * i, K), 1.0, seed=80 + i, device=DEV)
        packed, scales, zeros = quantize_gpu(cuda_lib, W, group, True)
        probs.append((x, packed, scales, torch.empty((x.shape[0], N), dtype=torch.bfloat16, device=DEV)))
        zs.append(zeros)
        sbuf = torch.empty(scales.numel() + 8, dtype=scales.dtype, device=DEV)
        s2 = sbuf[1:1 + scales.numel()].view(scales.shape)
        s2.copy_(scales)
        zbuf = torch.empty(zeros.numel() + 16, dtype=zeros.dtype, device=DEV)
        z2 = zbuf[1:1 + zeros.numel()].view(zeros.shape)
        z2.copy_(zeros)
        assert s2.data_ptr() % 4 == 2 and z2.data_ptr() % 2 == 1
        moved.append((x, packed, s2, torch.empty_like(probs[-1][3])))
        zs2.append(z2)
    cuda_lib.w4_gemm_grouped(cuda_lib.w4_grouped_plan(probs, group=group, zeros=zs))
    cuda_lib.w4_gemm_grouped(cuda_lib.w4_grouped_plan(moved, group=group, zeros=zs2))
    torch.cuda.synchronize()
    assert cuda_lib.w4_last_device_status() == 0
    for (_, _, _, y), (_, _, _, y2) in zip(probs, moved):
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_grouped_affine_group128_without_zeros_is_the_symmetric_plan(cuda_lib):
    W = wl.random_bf16((500, 2048), 0.02, seed=3, device=DEV)
    x = wl.random_bf16((5, 2048), 1.0, seed=4, device=DEV)
    packed, scales, _ = quantize_gpu(cuda_lib, W, 128, False)
    y0 = torch.empty((5, 500), dtype=torch.bfloat16, device=DEV)
    y1 = torch.empty_like(y0)
    p0 = cuda_lib.w4_grouped_plan([(x, packed, scales, y0)])
    p1 = cuda_lib.w4_grouped_plan([(x, packed, scales, y1)], group=128, zeros=[None])
    assert p0.plan.format == 0 and p1.plan.format == 0
    cuda_lib.w4_gemm_grouped(p0)
    cuda_lib.w4_gemm_grouped(p1)
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
