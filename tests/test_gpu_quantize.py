"""GPU parity of w4_quantize_rtn against the CPU oracle: packed bytes and scale
bits must be identical (bit-exact), outputs must not be written outside."""
import numpy as np
import pytest
import torch

from gemm_rtn_sym_gb300 import workloads as wl
from oracle import w4_oracle as O
from tests.helpers import check_quantize, quantize_gpu, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("N,K", [(1, 128), (7, 256), (16, 384), (129, 1152), (300, 9216), (33, 2560)])
def test_small_shapes(cuda_lib, N, K):
    W = wl.random_bf16((N, K), 0.02, seed=N * 1000 + K, device=DEV)
    packed, scales = quantize_gpu(cuda_lib, W)
    check_quantize(W, packed, scales)


@pytest.mark.parametrize("workload", ["ffn", "outlier"])
def test_ffn_matrix_full(cuda_lib, workload):
    W = wl.weight(workload, device=DEV)
    packed, scales = quantize_gpu(cuda_lib, W)
    check_quantize(W, packed, scales)


def tie_and_range_matrix():
    """Every group maximum a over all 128 mantissas at 20 exponents (normal and
    subnormal) with, for each a, four groups whose other 127 weights take every
    mantissa at the exponents of a, a/2, a/4 and a/8 (values above |a| clipped
    to a).  This walks every w/d quotient the rounding can meet, ties included."""
    exps = list(range(0, 3)) + list(range(100, 134, 2)) + [200]  # biased exponents
    rows = []
    for e in exps:
        for m in range(128):
            a = (e << 7) | m
            if a == 0:
                continue
            for de in range(4):
                ew = max(e - de, 0)
                w = (ew << 7) | np.arange(1, 128)
                w = np.where(w > a, a, w)
                sign = np.where(np.arange(127) % 2 == 0, 0, 0x8000)
                grp = np.concatenate([[a | (0x8000 if (m + de) % 2 else 0)], w | sign])
                rows.append(grp)
    M = np.array(rows, dtype=np.uint16)
    M = M[: (M.shape[0] // 8) * 8].reshape(-1, 8 * 128)  # 8 groups per row
    return torch.from_numpy(M.view(np.int16)).view(torch.bfloat16)


def test_every_quotient_and_tie(cuda_lib):
    Wc = tie_and_range_matrix()
    packed, scales = quantize_gpu(cuda_lib, Wc.to(DEV))
    check_quantize(Wc, packed, scales)


@pytest.mark.parametrize("offset_elems", [8, 16])
def test_input_alignment_variants(cuda_lib, offset_elems):
    """W at a 16-byte (not 32-byte) offset takes the 16-byte-load variant; both
    variants must give the oracle's bytes, on the tie/range matrix too."""
    for W in (wl.random_bf16((129, 1152), 0.02, seed=7, device=DEV), tie_and_range_matrix().to(DEV)):
        N, K = W.shape
        flat = torch.empty(N * K + 64, dtype=torch.bfloat16, device=DEV)
        Wv = flat[offset_elems:offset_elems + N * K].view(N, K)
        Wv.copy_(W)
        assert Wv.data_ptr() % 16 == 0
        packed, scales = quantize_gpu(cuda_lib, Wv)
        check_quantize(W.cpu(), packed, scales)


def test_special_groups(cuda_lib):
    W = torch.zeros((6, 256), dtype=torch.float32)
    W[1, :] = -0.375                       # all equal
    W[2, 17] = 3e-39                       # subnormal single element
    W[3, 0] = 1e-41                        # tiny: bf16(a/7) may be zero
    W[4, 128:] = torch.linspace(-1e-38, 1e-38, 128)
    W[5, ::2] = 0.5
    W[5, 1::2] = -0.5
    Wb = W.to(torch.bfloat16)
    Wb.view(torch.int16)[0, 5] = 0x0001    # smallest subnormal: d rounds to 0
    Wb.view(torch.int16)[0, 200] = -32768  # -0.0
    packed, scales = quantize_gpu(cuda_lib, Wb.to(DEV))
    check_quantize(Wb, packed, scales)
    assert wl.bits(scales)[0, 0] == 0 and not packed[0, :64].any()


def test_layout_round_trip(cuda_lib):
    W = wl.random_bf16((64, 512), 0.02, seed=99, device=DEV)
    packed, scales = quantize_gpu(cuda_lib, W)
    q = O.unpack_p1(packed.cpu().numpy(), 512)
    assert q.min() >= -7 and q.max() <= 7


@pytest.mark.slow
@pytest.mark.parametrize("workload", ["layer27b", "layer70b"])
def test_layer_matrices_sampled(cuda_lib, workload):
    for i, (N, K) in enumerate(wl.SHAPES[workload]):
        W = wl.weight(workload, i, device=DEV)
        packed, scales = quantize_gpu(cuda_lib, W)
        rows = sample_rows(N, 96, seed=i)
        check_quantize(W[torch.from_numpy(rows).to(DEV)].cpu(), packed[torch.from_numpy(rows).to(DEV)],
                       scales[torch.from_numpy(rows).to(DEV)])
        del W, packed, scales
        torch.cuda.empty_cache()


@pytest.mark.slow
def test_stack4b_distinct_shapes_sampled(cuda_lib):
    seen = set()
    for i, (N, K) in enumerate(wl.SHAPES["stack4b"]):
        if (N, K) in seen:
            continue
        seen.add((N, K))
        W = wl.weight("stack4b", i, device=DEV)
        packed, scales = quantize_gpu(cuda_lib, W)
        rows = torch.from_numpy(sample_rows(N, 64, seed=i)).to(DEV)
        check_quantize(W[rows].cpu(), packed[rows], scales[rows])
