"""GPU parity of GPTQ (Qwen3.5-4B quantisation study, §2 settings table: GPTQ
with the RTN storage, damping 0.01, original column order, 128-column blocks;
§2 H' = H + λI) against the CPU oracle.  Both sides run fp64, so codes and
scales must match exactly; H is a seeded synthetic calibration statistic given
to both as the same fp32 bits."""
import numpy as np
import pytest
import torch

from gemm_rtn_sym_gb300 import W4_ERR_INVALID_ARG, W4_ERR_NUMERIC, W4Error
from gemm_rtn_sym_gb300 import workloads as wl
from oracle import w4_oracle as O
from tests.helpers import guarded, guards_intact

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_gptq(w4, W, H, group=128):
    N, K = W.shape
    U = w4.w4_gptq_factor(H.to(DEV))
    packed, pbuf = guarded((N, K // 2), torch.uint8, W.device)
    scales, sbuf = guarded((N, K // group), torch.bfloat16, W.device)
    w4.w4_gptq_quantize(W, U, group, packed=packed, scales=scales)
    torch.cuda.synchronize()
    assert guards_intact(pbuf) and guards_intact(sbuf), "GPTQ wrote outside its outputs"
    assert w4.w4_last_device_status() == 0
    return packed, scales


def check(W, H, group, packed, scales, rows=None):
    Wb = wl.bits(W)
    if rows is not None:
        Wb = Wb[rows]
        packed, scales = packed[torch.as_tensor(rows, device=packed.device)], scales[torch.as_tensor(rows, device=packed.device)]
    p_ref, s_ref = O.gptq_quantize(Wb, H.cpu().double().numpy(), group)
    sg, pg = wl.bits(scales), packed.cpu().numpy()
    assert np.array_equal(sg, s_ref), f"scale bits differ in {np.count_nonzero(sg != s_ref)} places"
    assert np.array_equal(pg, p_ref), f"packed bytes differ in {np.count_nonzero(pg != p_ref)} places"


@pytest.mark.parametrize("group", [128, 64, 32])
@pytest.mark.parametrize("N,K", [(64, 256), (37, 1152), (130, 2048)])
def test_gptq_parity(cuda_lib, N, K, group):
    W = wl.random_bf16((N, K), 0.02, seed=N + K, device=DEV)
    H = wl.calibration_hessian(K, 2 * K, seed=K)
    check(W, H, group, *run_gptq(cuda_lib, W, H, group))


def test_gptq_outlier_rows_differ_from_rtn(cuda_lib):
    W = wl.weight("outlier", device=DEV, shape=(96, 2304))
    H = wl.calibration_hessian(2304, 4096, seed=5)
    packed, scales = run_gptq(cuda_lib, W, H)
    check(W, H, 128, packed, scales)
    p0, _ = cuda_lib.w4_quantize_rtn(W)
    assert (packed != p0).float().mean().item() > 0.05


def test_gptq_diagonal_h_is_rtn(cuda_lib):
    W = wl.random_bf16((200, 1024), 0.02, seed=9, device=DEV)
    H = torch.diag(torch.linspace(0.1, 10.0, 1024))
    packed, scales = run_gptq(cuda_lib, W, H)
    p0, s0 = cuda_lib.w4_quantize_rtn(W)
    assert torch.equal(packed, p0) and torch.equal(scales.view(torch.int16), s0.view(torch.int16))


def test_gptq_singular_h(cuda_lib):
    W = wl.random_bf16((40, 512), 0.02, seed=10, device=DEV)
    H = wl.calibration_hessian(512, 64, seed=11)  # rank 64 < 512: only the damping makes it definite
    check(W, H, 128, *run_gptq(cuda_lib, W, H))


def test_gptq_repeat_is_bit_identical(cuda_lib):
    W = wl.random_bf16((300, 1536), 0.02, seed=12, device=DEV)
    H = wl.calibration_hessian(1536, 2048, seed=13)
    a = run_gptq(cuda_lib, W, H)
    b = run_gptq(cuda_lib, W, H)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1].view(torch.int16), b[1].view(torch.int16))


def test_gptq_not_positive_definite_reports_numeric(cuda_lib):
    H = -torch.eye(256)
    cuda_lib.w4_gptq_factor(H.to(DEV))
    torch.cuda.synchronize()
    assert cuda_lib.w4_last_device_status() == W4_ERR_NUMERIC
    assert cuda_lib.w4_last_device_status() == 0  # reading clears it


def test_gptq_small_workspace_rejected(cuda_lib):
    W = wl.random_bf16((8, 256), 0.02, seed=1, device=DEV)
    U = cuda_lib.w4_gptq_factor(torch.eye(256, device=DEV))
    ws = torch.empty(1024, dtype=torch.uint8, device=DEV)
    with pytest.raises(W4Error) as e:
        cuda_lib.w4_gptq_quantize(W, U, workspace=ws)
    assert e.value.status == W4_ERR_INVALID_ARG


@pytest.mark.slow
def test_gptq_ffn_matrix_sampled_rows(cuda_lib):
    """The full 2560×9216 matrix on the GPU; the oracle checks 48 sampled rows
    (GPTQ treats rows independently given U)."""
    W = wl.weight("ffn", device=DEV)
    H = wl.calibration_hessian(9216, 2048, seed=17, device=DEV)
    packed, scales = run_gptq(cuda_lib, W, H)
    rows = np.unique(np.concatenate([[0, 1, 2559], np.random.default_rng(3).choice(2560, 45, replace=False)]))
    check(W, H, 128, packed, scales, rows=rows)
