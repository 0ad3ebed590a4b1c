"""GPU parity of the AWQ-style channel scaling (Qwen3.5-4B quantisation study,
§2 AWQ equation W'_ij = W_ij·s_j, x'_j = x_j/s_j) against the CPU oracle:
w4_quantize_rtn_scaled must give the oracle's packed bytes and scale bits for
W' = bf16(W·s) exactly, w4_scale_activations the oracle's x' bits exactly, and
the matmul of the two must stay within the usual parity bound."""
import numpy as np
import pytest
import torch

from gemm_rtn_sym_gb300 import W4_PATH_SMALL_M, W4_PATH_TENSOR, W4Error
from gemm_rtn_sym_gb300 import workloads as wl
from oracle import w4_oracle as O
from tests.helpers import guarded, guards_intact
from tests.test_gpu_quantize import tie_and_range_matrix
from tests.test_oracle_pins import double_rounding_cases

pytestmark = pytest.mark.gpu
DEV = "cuda"


def quantize_scaled_gpu(w4, W, s):
    N, K = W.shape
    packed, pbuf = guarded((N, K // 2), torch.uint8, W.device)
    scales, sbuf = guarded((N, K // 128), torch.bfloat16, W.device)
    w4.w4_quantize_rtn_scaled(W, s, packed=packed, scales=scales)
    torch.cuda.synchronize()
    assert guards_intact(pbuf) and guards_intact(sbuf), "quantiser wrote outside its outputs"
    return packed, scales


def check_scaled(W, s, packed, scales):
    p_ref, s_ref = O.quantize_rtn_scaled(wl.bits(W), s.cpu().numpy())
    sg, pg = wl.bits(scales), packed.cpu().numpy()
    assert np.array_equal(sg, s_ref), f"scale bits differ in {np.count_nonzero(sg != s_ref)} places"
    assert np.array_equal(pg, p_ref), f"packed bytes differ in {np.count_nonzero(pg != p_ref)} places"


def scale_activations_gpu(w4, x, s):
    out, obuf = guarded(tuple(x.shape), torch.bfloat16, x.device)
    w4.w4_scale_activations(x, s, out=out)
    torch.cuda.synchronize()
    assert guards_intact(obuf), "activation scaling wrote outside its output"
    return out


@pytest.mark.parametrize("N,K", [(1, 128), (7, 256), (16, 384), (129, 1152), (300, 9216), (33, 2560)])
def test_scaled_small_shapes(cuda_lib, N, K):
    W = wl.random_bf16((N, K), 0.02, seed=N * 1000 + K + 7, device=DEV)
    s = wl.channel_scales(K, seed=K + N, device=DEV)
    packed, scales = quantize_scaled_gpu(cuda_lib, W, s)
    check_scaled(W, s, packed, scales)


@pytest.mark.parametrize("workload", ["ffn", "outlier"])
def test_scaled_full_matrix(cuda_lib, workload):
    W = wl.weight(workload, device=DEV)
    s = wl.workload_channel_scales(workload, device=DEV)
    packed, scales = quantize_scaled_gpu(cuda_lib, W, s)
    check_scaled(W, s, packed, scales)


def test_unit_and_power_of_two_scales(cuda_lib):
    """s = 1 reproduces w4_quantize_rtn; s = 2^e per group keeps the codes and
    multiplies every group scale by 2^e."""
    W = wl.random_bf16((64, 1024), 0.02, seed=5, device=DEV)
    p0, d0 = cuda_lib.w4_quantize_rtn(W)
    p1, d1 = quantize_scaled_gpu(cuda_lib, W, torch.ones(1024, dtype=torch.float32, device=DEV))
    assert torch.equal(p0, p1) and torch.equal(d0.view(torch.int16), d1.view(torch.int16))
    e = torch.tensor([-4.0, -1.0, 0.0, 1.0, 2.0, 3.0, 6.0, -2.0])
    s = torch.exp2(e).repeat_interleave(128).to(DEV)
    p2, d2 = quantize_scaled_gpu(cuda_lib, W, s)
    assert torch.equal(p0, p2)
    assert torch.equal(d2.float().cpu(), d0.float().cpu() * torch.exp2(e)[None, :])


def test_rounds_through_fp32(cuda_lib):
    """Products that land on a bf16 tie only after rounding to fp32: the stated
    reading (fp32 product, then bf16) decides them."""
    cases = double_rounding_cases()
    K = ((len(cases) + 127) // 128) * 128
    wb = np.zeros((1, K), dtype=np.uint16)
    sv = np.ones(K, dtype=np.float32)
    wb[0, :len(cases)] = [w for w, _ in cases]
    sv[:len(cases)] = [sk for _, sk in cases]
    W = torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16).to(DEV)
    s = torch.from_numpy(sv).to(DEV)
    packed, scales = quantize_scaled_gpu(cuda_lib, W, s)
    check_scaled(W, s, packed, scales)


def test_scaled_every_quotient_and_tie(cuda_lib):
    """The tie/range matrix (normal, tiny and subnormal groups) under non-trivial
    channel scales: products reach fp32 subnormals and every code path."""
    Wc = tie_and_range_matrix()
    K = Wc.shape[1]
    for seed in (1, 2):
        s = wl.channel_scales(K, seed=seed, alpha=1.0, device=DEV)
        packed, scales = quantize_scaled_gpu(cuda_lib, Wc.to(DEV), s)
        check_scaled(Wc, s, packed, scales)


@pytest.mark.parametrize("offset_elems", [8, 16])
def test_scaled_input_alignment_variants(cuda_lib, offset_elems):
    W = wl.random_bf16((129, 1152), 0.02, seed=17, device=DEV)
    N, K = W.shape
    s = wl.channel_scales(K, seed=3, device=DEV)
    flat = torch.empty(N * K + 64, dtype=torch.bfloat16, device=DEV)
    Wv = flat[offset_elems:offset_elems + N * K].view(N, K)
    Wv.copy_(W)
    packed, scales = quantize_scaled_gpu(cuda_lib, Wv, s)
    check_scaled(W, s, packed, scales)


@pytest.mark.parametrize("M,K", [(1, 128), (1, 9216), (3, 384), (17, 2560), (208, 8192)])
def test_scale_activations_bit_exact(cuda_lib, M, K):
    x = wl.random_bf16((M, K), 1.0, seed=M * 10 + K, device=DEV)
    s = wl.channel_scales(K, seed=K, device=DEV)
    out = scale_activations_gpu(cuda_lib, x, s)
    ref = O.awq_scale_activations(wl.bits(x), s.cpu().numpy())
    got = wl.bits(out)
    assert np.array_equal(got, ref), f"x' bits differ in {np.count_nonzero(got != ref)} places"


def test_scale_activations_in_place_and_edges(cuda_lib):
    K = 1024
    x = wl.random_bf16((4, K), 1.0, seed=8, device=DEV)
    x.view(torch.int16)[0, :8] = torch.tensor([0, -32768, 1, -32767, 0x7F7F, 0x0080, 0x3F80, 0x4000],
                                               dtype=torch.int16)
    s = wl.channel_scales(K, seed=9, device=DEV)
    s[:8] = torch.tensor([3.0, 0.1, 0.5, 2.0, 0.75, 4.0, 1.0, 3.0])
    ref = O.awq_scale_activations(wl.bits(x), s.cpu().numpy())
    y = x.clone()
    cuda_lib.w4_scale_activations(y, s, out=y)
    torch.cuda.synchronize()
    assert np.array_equal(wl.bits(y), ref)


@pytest.mark.parametrize("M,path", [(1, W4_PATH_SMALL_M), (8, W4_PATH_SMALL_M), (33, W4_PATH_TENSOR)])
def test_scaled_matmul_parity(cuda_lib, M, path):
    """y = Ŵ'x' through the library's own kernels, against the oracle's fp64
    matmul of the oracle's W' codes and x'."""
    W = wl.weight("outlier", device=DEV)[:512].contiguous()
    N, K = W.shape
    s = wl.workload_channel_scales("outlier", device=DEV)
    x = wl.activations("outlier", M, K, device=DEV)
    packed, scales = quantize_scaled_gpu(cuda_lib, W, s)
    xs = scale_activations_gpu(cuda_lib, x, s)
    y = cuda_lib.w4_gemm_ex(xs, packed, scales, path=path)
    torch.cuda.synchronize()
    sn = s.cpu().numpy()
    p_ref, d_ref = O.quantize_rtn_scaled(wl.bits(W), sn)
    x_ref = O.awq_scale_activations(wl.bits(x), sn)
    y_ref, s_abs = O.gemm_reference(x_ref, p_ref, d_ref, K)
    excess = O.parity_excess(wl.bits(y), y_ref, s_abs)
    assert float(excess.max()) <= 1.0


def test_rejects(cuda_lib):
    W = wl.random_bf16((4, 256), 0.02, seed=1, device=DEV)
    s = torch.ones(256, dtype=torch.float32, device=DEV)
    with pytest.raises(ValueError):
        cuda_lib.w4_quantize_rtn_scaled(W, s[:128])
    with pytest.raises(TypeError):
        cuda_lib.w4_quantize_rtn_scaled(W, s.to(torch.bfloat16))
    buf = torch.ones(260, dtype=torch.float32, device=DEV)
    with pytest.raises(W4Error):
        cuda_lib.w4_quantize_rtn_scaled(W, buf[1:257])  # 4-byte aligned only
    x = wl.random_bf16((2, 256), 1.0, seed=2, device=DEV)
    with pytest.raises(W4Error):
        cuda_lib.w4_scale_activations(x, buf[2:258])   # 8-byte aligned only
