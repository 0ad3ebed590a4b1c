"""Pins for the oracle's GPTQ (Qwen3.5-4B quantisation study, §2 settings table:
GPTQ with the same storage as RTN, damping 0.01, original column order,
128-column blocks; §2 H' = H + λI, λ = 0.01·mean(diag H); the update rule of
the published GPTQ algorithm, Frantar et al. 2022).  None of these retypes the
oracle: the main pin is a second route to the same result (optimal-brain-
surgeon updates with an explicitly eliminated inverse, no Cholesky factor), the
others are properties the definition fixes."""
import numpy as np
import pytest

from oracle import w4_oracle as O
from gemm_rtn_sym_gb300 import workloads as wl


def correlated_h(K, T, seed):
    """Gram matrix of correlated synthetic inputs (channels mixed, a few
    channels larger), fp64."""
    rng = np.random.default_rng(seed)
    Z = rng.standard_normal((T, K))
    A = np.eye(K) + 0.3 * rng.standard_normal((K, K)) / np.sqrt(K)
    X = Z @ A * np.exp(0.5 * rng.standard_normal(K))
    return X.T @ X, X


def obs_route(W_bits, H, group=128, damp=0.01):
    """GPTQ as a sequence of optimal-brain-surgeon steps: round column c, move
    the later columns by −err·Hinv[c, c+1:] / Hinv[c, c], then eliminate c from
    the inverse (Hinv -= Hinv[:, c] Hinv[c, :] / Hinv[c, c]).  Scales as in the
    study's group rule, from the current weights at each group start."""
    W = O.bf16_bits_to_f32(W_bits).astype(np.float64)
    N, K = W.shape
    Hd = H + damp * np.mean(np.diag(H)) * np.eye(K)
    Hinv = np.linalg.inv(Hd)
    q = np.zeros((N, K), dtype=np.int8)
    s = np.zeros((N, K // group), dtype=np.uint16)
    for c in range(K):
        if c % group == 0:
            a = np.max(np.abs(W[:, c:c + group]), axis=1)
            s[:, c // group] = O.f32_to_bf16_bits_rne((a / 7.0).astype(np.float32))
            d = O.bf16_bits_to_f32(s[:, c // group]).astype(np.float64)
        with np.errstate(divide="ignore", invalid="ignore"):
            r = np.where(d == 0, 0.0, W[:, c] / np.where(d == 0, 1.0, d))
        qc = np.clip(np.rint(r), -8, 7)
        q[:, c] = qc
        err = (W[:, c] - d * qc) / Hinv[c, c]
        W[:, c:] -= np.outer(err, Hinv[c, c:])
        Hinv = Hinv - np.outer(Hinv[:, c], Hinv[c, :]) / Hinv[c, c]
    return O.pack_p1(q), s


@pytest.mark.parametrize("group", [128, 64, 32])
def test_gptq_matches_obs_route(group):
    W = wl.bits(wl.random_bf16((12, 384), 0.02, seed=5))
    H, _ = correlated_h(384, 1024, seed=6)
    p, s = O.gptq_quantize(W, H, group)
    p2, s2 = obs_route(W, H, group)
    assert np.array_equal(s, s2)
    assert np.array_equal(p, p2)
    assert np.mean(p != O.quantize_rtn(W, group)[0]) > 0.05  # the corrections do change codes


def test_gptq_diagonal_h_is_rtn():
    """With a diagonal H no error reaches another column: GPTQ is RTN."""
    W = wl.bits(wl.weight("outlier", shape=(16, 1024)))
    for seed in (1, 2):
        H = np.diag(np.random.default_rng(seed).uniform(0.1, 10, 1024))
        p, s = O.gptq_quantize(W, H)
        p0, s0 = O.quantize_rtn(W)
        assert np.array_equal(p, p0) and np.array_equal(s, s0)


@pytest.mark.parametrize("block", [32, 64, 256, 512])
def test_gptq_block_size_does_not_change_the_result(block):
    """The lazy block update only delays corrections: any block size gives the
    codes and scales of block 128."""
    W = wl.bits(wl.random_bf16((10, 512), 0.02, seed=7))
    H, _ = correlated_h(512, 1024, seed=8)
    p, s = O.gptq_quantize(W, H)
    p2, s2 = O.gptq_quantize(W, H, block=block)
    assert np.array_equal(s, s2) and np.array_equal(p, p2)


def test_gptq_scale_invariant_in_h():
    """Damping proportional to mean(diag H) makes the result independent of the
    scale of H."""
    W = wl.bits(wl.random_bf16((10, 256), 0.02, seed=9))
    H, _ = correlated_h(256, 512, seed=10)
    p, s = O.gptq_quantize(W, H)
    for c in (0.25, 3.7, 1e6):
        p2, s2 = O.gptq_quantize(W, H * c)
        assert np.array_equal(s, s2) and np.array_equal(p, p2)


def test_gptq_first_group_scale_is_rtn():
    """Nothing is corrected before column 0, so the first group's scale and
    first code are RTN's."""
    W = wl.bits(wl.random_bf16((20, 256), 0.02, seed=11))
    H, _ = correlated_h(256, 512, seed=12)
    p, s = O.gptq_quantize(W, H)
    p0, s0 = O.quantize_rtn(W)
    assert np.array_equal(s[:, 0], s0[:, 0])
    assert np.array_equal(O.unpack_p1(p, 256)[:, 0], O.unpack_p1(p0, 256)[:, 0])
    assert not np.array_equal(s[:, 1], s0[:, 1])  # later groups see corrected weights


def test_gptq_lowers_the_output_error():
    """The point of the corrections: ||(W − Ŵ) Xᵀ|| on the calibration inputs is
    well below RTN's."""
    W = wl.bits(wl.random_bf16((32, 512), 0.02, seed=13))
    H, X = correlated_h(512, 2048, seed=14)
    w = O.bf16_bits_to_f32(W).astype(np.float64)
    e = {}
    for name, (p, s) in {"gptq": O.gptq_quantize(W, H), "rtn": O.quantize_rtn(W)}.items():
        e[name] = np.sum(((w - O.dequantize_fp64(p, s, 512)) @ X.T) ** 2)
    assert e["gptq"] < 0.9 * e["rtn"]


def test_gptq_singular_h():
    """Fewer calibration rows than inputs: H is singular, H' is not."""
    W = wl.bits(wl.random_bf16((8, 256), 0.02, seed=15))
    rng = np.random.default_rng(16)
    X = rng.standard_normal((64, 256))
    p, s = O.gptq_quantize(W, X.T @ X)
    q = O.unpack_p1(p, 256)
    assert q.min() >= -8 and q.max() <= 7 and np.all(s > 0)


def test_gptq_rejects():
    W = wl.bits(wl.random_bf16((2, 256), 0.02, seed=3))
    H = np.eye(256)
    with pytest.raises(ValueError):
        O.gptq_quantize(W, H, group=96)
    with pytest.raises(ValueError):
        O.gptq_quantize(W, H, group=128, block=96)
