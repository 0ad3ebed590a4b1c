"""Seeded synthetic inputs for the W4A16 matmul and the RTN quantiser.

This module only draws random tensors; it holds none of the quantiser's or the
matmul's arithmetic.  Tests, the CPU oracle's callers and the benchmark all take
their inputs from here, so that both sides of every comparison see the same
bf16 bits.

The shapes and value distributions follow the workloads the source pages run
the format on (Qwen3.5-4B whole-model quantisation study, §1 FFN example
2560×9216 and the 200-matrix / ~3.565B-weight scope table; 27B-class and
70B-class dense layers; speculative-verify row counts K+1):

* ``ffn``      — one 2560×9216 matrix, W ~ N(0, 0.02²), x ~ N(0, 1);
* ``outlier``  — the same matrix with 1 % of the input channels (92 of 9216,
  chosen by a seeded permutation) multiplied by 8;
* ``layer27b`` — q/k/v 7168×5120, o 5120×5120, gate/up 34816×5120,
  down 5120×17408, N(0, 0.02²);
* ``layer70b`` — q/k/v 10240×8192, o 8192×8192, gate/up 57344×8192,
  down 8192×28672, Student-t(ν=5)·0.02;
* ``stack4b``  — 56×(2560×9216) + 56×(9216×2560) + 44×(2560×4096) +
  44×(4096×2560) = 3,565,158,400 weights, N(0, 0.02²).

Channel scales for the AWQ-style scaled quantiser (§2 AWQ equation and the
paragraph after it: s_j ∝ (mean|x_j|)^α, α = k/19): :func:`channel_scales`
draws synthetic per-channel input magnitudes m_j (log-normal, with the same
1 % of channels ×8 as ``outlier``), raises them to α = 10/19 and divides by
their geometric mean.  No calibration activations exist here, and the search
over α is not part of the library; the scales are only inputs.

Seeds: 1000·workload_id + 10·matrix_index + {0: W, 1: x, 2: aux, 3: s}.
Each draw is fp32 from a seeded ``torch.Generator`` on the requested device,
then converted to bf16 with round-to-nearest-even.
"""
from __future__ import annotations

import torch

WORKLOAD_IDS = {"ffn": 1, "outlier": 2, "layer27b": 3, "layer70b": 4, "stack4b": 5}

SHAPES = {
    "ffn": [(2560, 9216)],
    "outlier": [(2560, 9216)],
    "layer27b": [(7168, 5120), (5120, 5120), (34816, 5120), (5120, 17408)],
    "layer70b": [(10240, 8192), (8192, 8192), (57344, 8192), (8192, 28672)],
    "stack4b": [(2560, 9216)] * 56 + [(9216, 2560)] * 56
    + [(2560, 4096)] * 44 + [(4096, 2560)] * 44,
}

ROWS = {
    "ffn": [1],
    "outlier": [8],
    "layer27b": [1, 5, 7, 13],
    "layer70b": [208],
    "stack4b": [1, 2, 4, 8, 16, 32, 64, 128],
}

W_STD = 0.02
OUTLIER_FRACTION = 0.01
OUTLIER_FACTOR = 8.0
STUDENT_NU = 5


def seed_for(workload: str, matrix_index: int, role: int) -> int:
    return 1000 * WORKLOAD_IDS[workload] + 10 * matrix_index + role


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def student_t_bf16(shape, nu: int, scale: float, seed: int, device="cpu") -> torch.Tensor:
    """z / sqrt(χ²_ν / ν) with χ²_ν the sum of ν squared seeded normals."""
    g = _gen(seed, device)
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(nu):
        chi2 += torch.randn(shape, generator=g, device=device, dtype=torch.float32).square()
    return (z / torch.sqrt(chi2 / nu) * scale).to(torch.bfloat16)


def outlier_channels(K: int, seed: int, device="cpu") -> torch.Tensor:
    """Indices of round(1 % · K) input channels, from a seeded permutation."""
    g = _gen(seed, device)
    n = int(round(OUTLIER_FRACTION * K))
    return torch.randperm(K, generator=g, device=device)[:n]


AWQ_ALPHA = 10 / 19
CHANNEL_LOG_STD = 0.5


def channel_scales(K: int, seed: int, alpha: float = AWQ_ALPHA, device="cpu") -> torch.Tensor:
    """fp32 [K] channel scales s_j = (m_j)^α / geomean(m^α), with synthetic
    magnitudes m_j = exp(N(0, 0.5²)) and 1 % of the channels ×8.  Drawn on the
    CPU (the same values for every device), then moved to ``device``."""
    g = _gen(seed, "cpu")
    m = torch.exp(torch.randn(K, generator=g, dtype=torch.float64) * CHANNEL_LOG_STD)
    m[outlier_channels(K, seed + 1)] *= OUTLIER_FACTOR
    p = m ** alpha
    s = p / torch.exp(torch.log(p).mean())
    return s.to(torch.float32).to(device)


def calibration_hessian(K: int, T: int, seed: int, device="cpu") -> torch.Tensor:
    """fp32 [K, K] H = Xᵀ X / T of synthetic calibration inputs X [T, K] for
    the GPTQ quantiser (the study calibrates on 128 × 1,024 tokens; none are
    available here): seeded N(0, 1) rows mixed across channels by
    (I + 0.3·G/√K) with G seeded N(0, 1), scaled per channel by log-normal
    magnitudes (σ = 0.5) with 1 % of the channels ×8, and symmetrised exactly."""
    g = _gen(seed, device)
    Z = torch.randn((T, K), generator=g, device=device, dtype=torch.float32)
    G = torch.randn((K, K), generator=g, device=device, dtype=torch.float32)
    m = torch.exp(torch.randn(K, generator=g, device=device, dtype=torch.float32) * CHANNEL_LOG_STD)
    m[outlier_channels(K, seed + 1, device)] *= OUTLIER_FACTOR
    X = (Z @ (torch.eye(K, device=device) + 0.3 * G / K ** 0.5)) * m
    H = X.T @ X / T
    return (H + H.T) / 2


def workload_channel_scales(workload: str, matrix_index: int = 0, device="cpu") -> torch.Tensor:
    """The channel scales of one matrix of a workload (K of that matrix)."""
    K = SHAPES[workload][matrix_index][1]
    return channel_scales(K, seed_for(workload, matrix_index, 3), device=device)


def weight(workload: str, matrix_index: int = 0, device="cpu", shape=None) -> torch.Tensor:
    """W bf16 [N, K] for one matrix of a workload (``shape`` overrides the size
    for reduced-size test cases, keeping the distribution)."""
    N, K = shape if shape is not None else SHAPES[workload][matrix_index]
    s = seed_for(workload, matrix_index, 0)
    if workload == "layer70b":
        return student_t_bf16((N, K), STUDENT_NU, W_STD, s, device)
    W = normal_bf16((N, K), W_STD, s, device)
    if workload == "outlier":
        cols = outlier_channels(K, seed_for(workload, matrix_index, 2), device)
        W[:, cols] = (W[:, cols].float() * OUTLIER_FACTOR).to(torch.bfloat16)  # exact: ×2³
    return W


def activations(workload: str, M: int, K: int, matrix_index: int = 0, device="cpu") -> torch.Tensor:
    """x bf16 [M, K] ~ N(0, 1)."""
    return normal_bf16((M, K), 1.0, seed_for(workload, matrix_index, 1), device)


def random_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """Generic seeded N(0, std²) bf16 tensor for edge-case tests."""
    return normal_bf16(shape, std, seed, device)


def bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a bf16 tensor, as a numpy array on the host."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")
