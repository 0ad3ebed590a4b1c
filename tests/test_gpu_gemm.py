"""GPU parity of w4_gemm against the CPU oracle, element by element:
|y_gpu − y_ref| ≤ 4e-3 · Σ_k|ŵ_k x_k| + 1 bf16 ulp, y_ref the fp64 dequantised
matmul the oracle computes from W itself (never from the GPU's packed output)."""
import numpy as np
import pytest
import torch

import gemm_rtn_sym_gb300 as w4
from gemm_rtn_sym_gb300 import workloads as wl
from tests.helpers import check_gemm, check_quantize, gemm_gpu, quantize_gpu, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"
PATHS = [pytest.param(w4.W4_PATH_SMALL_M, id="small"), pytest.param(w4.W4_PATH_TENSOR, id="tensor")]
PATH_VALUES = [w4.W4_PATH_SMALL_M, w4.W4_PATH_TENSOR]


def run(cuda_lib, W, M, path, seed=0, x=None):
    packed, scales = quantize_gpu(cuda_lib, W)
    if x is None:
        x = wl.random_bf16((M, W.shape[1]), 1.0, seed=seed, device=DEV)
    y = gemm_gpu(cuda_lib, x, packed, scales, path)
    return x, y, packed, scales


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("N,K", [(1, 128), (7, 256), (16, 384), (129, 1152), (200, 4096)])
@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 9, 13, 16, 17])
def test_small_and_ragged(cuda_lib, path, N, K, M):
    W = wl.random_bf16((N, K), 0.02, seed=7 * N + K, device=DEV)
    x, y, _, _ = run(cuda_lib, W, M, path, seed=M)
    check_gemm(W, x, y)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M", [32, 63, 64, 65, 208, 257])
def test_larger_m(cuda_lib, path, M):
    W = wl.random_bf16((136, 1280), 0.02, seed=M, device=DEV)
    x, y, _, _ = run(cuda_lib, W, M, path, seed=M + 1)
    check_gemm(W, x, y)


@pytest.mark.parametrize("path", PATHS)
def test_ffn_m1_full(cuda_lib, path):
    W = wl.weight("ffn", device=DEV)
    x = wl.activations("ffn", 1, W.shape[1], device=DEV)
    _, y, _, _ = run(cuda_lib, W, 1, path, x=x)
    check_gemm(W, x, y)


@pytest.mark.parametrize("path", PATHS)
def test_outlier_m8_full(cuda_lib, path):
    W = wl.weight("outlier", device=DEV)
    x = wl.activations("outlier", 8, W.shape[1], device=DEV)
    _, y, _, _ = run(cuda_lib, W, 8, path, x=x)
    check_gemm(W, x, y)


def test_auto_path_matches_explicit(cuda_lib):
    W = wl.random_bf16((96, 1024), 0.02, seed=5, device=DEV)
    for M in (1, 8, 16, 17, 40):
        packed, scales = quantize_gpu(cuda_lib, W)
        x = wl.random_bf16((M, 1024), 1.0, seed=M, device=DEV)
        y_auto = w4.w4_gemm(x, packed, scales)
        y_exp = w4.w4_gemm_ex(x, packed, scales, path=w4.w4_gemm_path_for(M, 96, 1024))
        torch.cuda.synchronize()
        assert torch.equal(y_auto.view(torch.int16), y_exp.view(torch.int16))
        check_gemm(W, x, y_auto)


def test_deterministic(cuda_lib):
    W = wl.random_bf16((512, 4096), 0.02, seed=3, device=DEV)
    packed, scales = quantize_gpu(cuda_lib, W)
    for M in (1, 8, 13, 64):
        x = wl.random_bf16((M, 4096), 1.0, seed=M, device=DEV)
        ys = [w4.w4_gemm(x, packed, scales) for _ in range(5)]
        torch.cuda.synchronize()
        for y in ys[1:]:
            assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))


@pytest.mark.parametrize("N,K", [(1280, 8192), (2000, 2560), (4160, 1152), (96, 30720), (10240, 384)])
@pytest.mark.parametrize("M", [1, 5, 13])
def test_split_shapes(cuda_lib, N, K, M):
    """Shapes whose split-K choice ranges from none to eight-CTA clusters,
    with ragged row blocks and groups per CTA."""
    W = wl.random_bf16((N, K), 0.02, seed=N + K, device=DEV)
    x, y, _, _ = run(cuda_lib, W, M, w4.W4_PATH_SMALL_M, seed=M)
    check_gemm(W, x, y)


def test_repeat_is_bit_identical_mid_m(cuda_lib):
    """Many repeats of a 16-token pass on a matrix whose row blocks are split
    over cluster CTAs: a stage released before its fragments were read would
    show up as an occasional difference."""
    W = wl.random_bf16((10240, 2048), 0.02, seed=11, device=DEV)
    packed, scales = quantize_gpu(cuda_lib, W)
    for M in (13, 16):
        x = wl.random_bf16((M, 2048), 1.0, seed=M, device=DEV)
        ref = w4.w4_gemm_ex(x, packed, scales, path=w4.W4_PATH_SMALL_M)
        ys = [w4.w4_gemm_ex(x, packed, scales, path=w4.W4_PATH_SMALL_M) for _ in range(40)]
        torch.cuda.synchronize()
        for y in ys:
            assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


@pytest.mark.slow
@pytest.mark.parametrize("N,K,M", [(57344, 8192, 208), (2560, 9216, 64), (10240, 2048, 33)])
def test_tensor_repeat_is_bit_identical(cuda_lib, N, K, M):
    """Many repeats of the tensor-core tile: more tiles than SMs (57344 rows
    at M = 208, three waves), split-K over a cluster (2560 rows), one token
    tile of 48 (M = 33).  A code slot handed back to TMA before its read
    completed would show up as an occasional difference; the first run is
    checked against the oracle on sampled rows."""
    W = wl.random_bf16((N, K), 0.02, seed=N + M, device=DEV)
    packed, scales = quantize_gpu(cuda_lib, W)
    x = wl.random_bf16((M, K), 1.0, seed=M, device=DEV)
    ref = w4.w4_gemm_ex(x, packed, scales, path=w4.W4_PATH_TENSOR)
    ys = [w4.w4_gemm_ex(x, packed, scales, path=w4.W4_PATH_TENSOR) for _ in range(30)]
    torch.cuda.synchronize()
    assert w4.w4_last_device_status() == 0
    rows = torch.from_numpy(sample_rows(N, 16, seed=N)).to(DEV)
    check_gemm(W[rows].cpu(), x, ref[:, rows])
    for y in ys:
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


def test_empty_and_degenerate(cuda_lib):
    packed = torch.empty((4, 0), dtype=torch.uint8, device=DEV)
    scales = torch.empty((4, 0), dtype=torch.bfloat16, device=DEV)
    x = torch.empty((3, 0), dtype=torch.bfloat16, device=DEV)
    y = torch.full((3, 4), 7.0, dtype=torch.bfloat16, device=DEV)
    w4.w4_gemm(x, packed, scales, out=y)  # K = 0: y = 0
    torch.cuda.synchronize()
    assert not y.float().any()
    W = wl.random_bf16((5, 256), 0.02, seed=1, device=DEV)
    packed, scales = quantize_gpu(cuda_lib, W)
    y0 = w4.w4_gemm(torch.empty((0, 256), dtype=torch.bfloat16, device=DEV), packed, scales)
    assert y0.shape == (0, 5)
    # all-zero weights and all-zero activations give exact zeros
    Wz = torch.zeros((17, 384), dtype=torch.bfloat16, device=DEV)
    pz, sz = quantize_gpu(cuda_lib, Wz)
    xz = wl.random_bf16((3, 384), 1.0, seed=2, device=DEV)
    assert not w4.w4_gemm(xz, pz, sz).float().any()
    x0 = torch.zeros((4, 256), dtype=torch.bfloat16, device=DEV)
    assert not w4.w4_gemm(x0, packed, scales).float().any()


def test_index_probe(cuda_lib):
    """One-hot activations read back single dequantised columns: any misplaced
    row, group or k shows up as a wrong value at a known place."""
    N, K = 48, 512
    W = wl.random_bf16((N, K), 0.02, seed=17, device=DEV)
    packed, scales = quantize_gpu(cuda_lib, W)
    p_ref, s_ref = check_quantize(W, packed, scales)
    from oracle import w4_oracle as O
    what = O.dequantize_fp64(p_ref, s_ref, K)
    ks = [0, 1, 2, 7, 8, 31, 32, 127, 128, 129, 300, 511]
    x = torch.zeros((len(ks), K), dtype=torch.bfloat16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    for path in PATH_VALUES:
        y = gemm_gpu(cuda_lib, x.to(DEV), packed, scales, path).float().cpu().numpy()
        for i, k in enumerate(ks):
            expect = what[:, k].astype(np.float32)
            got = y[i]
            assert np.allclose(got, expect, rtol=2 ** -8, atol=0), (path, k)


@pytest.mark.slow
@pytest.mark.parametrize("path", PATHS)
def test_layer27b_sampled(cuda_lib, path):
    for i, (N, K) in enumerate(wl.SHAPES["layer27b"]):
        W = wl.weight("layer27b", i, device=DEV)
        packed, scales = quantize_gpu(cuda_lib, W)
        rows = torch.from_numpy(sample_rows(N, 64, seed=i)).to(DEV)
        for M in wl.ROWS["layer27b"]:
            x = wl.activations("layer27b", M, K, i, device=DEV)
            y = gemm_gpu(cuda_lib, x, packed, scales, path)
            check_gemm(W[rows].cpu(), x, y[:, rows])
        del W, packed, scales


@pytest.mark.slow
@pytest.mark.parametrize("path", PATHS)
def test_layer70b_sampled(cuda_lib, path):
    for i, (N, K) in enumerate(wl.SHAPES["layer70b"]):
        W = wl.weight("layer70b", i, device=DEV)
        packed, scales = quantize_gpu(cuda_lib, W)
        rows = torch.from_numpy(sample_rows(N, 48, seed=i)).to(DEV)
        x = wl.activations("layer70b", 208, K, i, device=DEV)
        y = gemm_gpu(cuda_lib, x, packed, scales, path)
        check_gemm(W[rows].cpu(), x, y[:, rows])
        del W, packed, scales


@pytest.mark.slow
def test_stack4b_sampled(cuda_lib):
    seen = set()
    for i, (N, K) in enumerate(wl.SHAPES["stack4b"]):
        if (N, K) in seen:
            continue
        seen.add((N, K))
        W = wl.weight("stack4b", i, device=DEV)
        packed, scales = quantize_gpu(cuda_lib, W)
        rows = torch.from_numpy(sample_rows(N, 32, seed=i)).to(DEV)
        for M in wl.ROWS["stack4b"]:
            x = wl.activations("stack4b", M, K, i, device=DEV)
            path = w4.w4_gemm_path_for(M, N, K)
            y = gemm_gpu(cuda_lib, x, packed, scales, path)
            check_gemm(W[rows].cpu(), x, y[:, rows])
