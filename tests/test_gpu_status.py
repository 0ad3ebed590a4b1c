"""Bounded device waits: a wait that nothing completes gives up, records
W4_ERR_TIMEOUT in the status word and the kernel exits; the context stays
usable.  No GPU fault, trap or hang is involved."""
import pytest
import torch

import gemm_rtn_sym_gb300 as w4
from gemm_rtn_sym_gb300 import workloads as wl
from tests.helpers import check_gemm, quantize_gpu

pytestmark = pytest.mark.gpu


def test_wait_completes(cuda_lib):
    w4.w4_wait_probe(50_000_000, arrive=True)
    assert w4.w4_last_device_status() == w4.W4_OK


def test_wait_times_out_and_context_survives(cuda_lib):
    w4.w4_wait_probe(2_000_000, arrive=False)  # 2 ms, nothing arrives
    assert w4.w4_last_device_status() == w4.W4_ERR_TIMEOUT
    assert w4.w4_last_device_status() == w4.W4_OK  # reading clears it
    W = wl.random_bf16((64, 512), 0.02, seed=1, device="cuda")
    packed, scales = quantize_gpu(cuda_lib, W)
    x = wl.random_bf16((3, 512), 1.0, seed=2, device="cuda")
    y = w4.w4_gemm(x, packed, scales)
    torch.cuda.synchronize()
    check_gemm(W, x, y)
