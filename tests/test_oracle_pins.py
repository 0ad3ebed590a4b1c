"""Pins for the CPU oracle: checks against values and facts the definition fixes,
never against the oracle's own formulas retyped.

Definition: Qwen3.5-4B quantisation study (parksieon.github.io), §1 group
quantisation equation with z = 0, §1 group-of-128 paragraph (72 groups per row
at 9216 inputs), §2 settings table (RTN minmax · symmetric, 4-bit weights /
BF16 inputs; smaller groups), §2 AWQ equation W'_ij = W_ij·s_j, x'_j = x_j/s_j,
W'x' = Wx, and the §1 equation with a free zero point z (asymmetric).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import w4_oracle as O
from gemm_rtn_sym_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rtn_hand_worked.txt")


# ---------------------------------------------------------------------------
# Exact rational arithmetic, independent of binary floating point.
# ---------------------------------------------------------------------------
def bf16_exact(bits: int) -> Fraction:
    bits = int(bits) & 0xFFFF
    sign = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    assert e != 0xFF, "no inf/nan here"
    if e == 0:
        return sign * Fraction(m, 1) * Fraction(1, 2 ** 133)
    v = Fraction(128 + m) * (Fraction(2) ** (e - 127 - 7))
    return sign * v


def round_half_even(v: Fraction) -> int:
    fl = v.numerator // v.denominator
    rem = v - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl + (fl & 1)


def bf16_rne_bits(v: Fraction) -> int:
    """Nearest bf16 (ties to even) to a non-negative rational, as bits."""
    assert v >= 0
    if v == 0:
        return 0
    e = v.numerator.bit_length() - v.denominator.bit_length()
    while Fraction(2) ** e > v:
        e -= 1
    while Fraction(2) ** (e + 1) <= v:
        e += 1
    e_eff = max(e, -126)
    m = round_half_even(v / (Fraction(2) ** (e_eff - 7)))
    if m == 0:
        return 0
    if m < 128:  # subnormal
        return m
    if m == 256:
        m, e_eff = 128, e_eff + 1
    return ((e_eff + 127) << 7) | (m - 128)


def f_to_bf16_bits(vals):
    """Exact float -> bf16 bit pattern (values given here are exactly bf16)."""
    a = np.asarray(vals, dtype=np.float32).view(np.uint32)
    assert np.all((a & 0xFFFF) == 0)
    return (a >> 16).astype(np.uint16)


def exact_rtn_group(w_bits):
    """Exact-rational RTN of one group: (d bits, q list)."""
    w = [bf16_exact(b) for b in w_bits]
    a = max(abs(v) for v in w)
    d_bits = bf16_rne_bits(a / 7)
    d = bf16_exact(d_bits)
    if d == 0:
        return d_bits, [0] * len(w)
    return d_bits, [min(7, max(-8, round_half_even(v / d))) for v in w]


def float_rne(v: Fraction, p: int, emin: int) -> Fraction:
    """Nearest binary float with p significant bits and minimum normal exponent
    emin to a rational (ties to even); no overflow."""
    if v == 0:
        return Fraction(0)
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (max(e, emin) - (p - 1))
    r = round_half_even(a / ulp) * ulp
    return r if v > 0 else -r


def fp32(v: Fraction) -> Fraction:
    return float_rne(v, 24, -126)


def exact_asym_group(w_bits):
    """Exact-rational asymmetric RTN of one group, each fp32 step rounded as
    the reading states: (d bits, z, q list)."""
    w = [bf16_exact(b) for b in w_bits]
    lo = min(min(w), Fraction(0))
    hi = max(max(w), Fraction(0))
    d_bits = bf16_rne_bits(fp32(fp32(hi - lo) / 15))
    d = bf16_exact(d_bits)
    if d == 0:
        return d_bits, 8, [8] * len(w)
    z = min(15, max(0, round_half_even(fp32(-lo / d))))
    return d_bits, z, [min(15, max(0, round_half_even(fp32(v / d)) + z)) for v in w]


def read_golden():
    rows = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = [p.strip() for p in line.split("|")]
            rows[parts[0]] = parts[1:]
    return rows


def one_group_matrix(values):
    w = np.zeros((1, 128), dtype=np.float32)
    w[0, : len(values)] = values
    return f_to_bf16_bits(w)


# ---------------------------------------------------------------------------
# P1: hand-worked groups (fixture under tests/golden/).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["A", "B"])
def test_hand_worked_groups(name):
    w_s, d_s, q_s, sum_s = read_golden()[name]
    w = [float(v) for v in w_s.split()]
    W = one_group_matrix(w)
    packed, s = O.quantize_rtn(W)
    assert O.bf16_bits_to_f32(s)[0, 0] == float(d_s)
    q = O.unpack_p1(packed, 128)[0]
    expect = [int(v) for v in q_s.split()]
    assert list(q[: len(expect)]) == expect
    assert not q[len(expect):].any()
    x_ones = f_to_bf16_bits(np.ones((1, 128), dtype=np.float32))
    y, _ = O.gemm_reference(x_ones, packed, s, 128)
    assert y[0, 0] == float(sum_s)


def test_hand_worked_packed_bytes():
    rows = read_golden()
    w = [float(v) for v in rows["A"][0].split()]
    packed, _ = O.quantize_rtn(one_group_matrix(w))
    expect = [int(b, 16) for b in rows["A_packed_first8"][0].split()]
    assert list(packed[0, :8]) == expect
    assert not packed[0, 8:].any()


def test_hand_worked_error_is_half_step():
    w = [float(v) for v in read_golden()["A"][0].split()]
    packed, s = O.quantize_rtn(one_group_matrix(w))
    what = O.dequantize_fp64(packed, s, 128)[0, : len(w)]
    assert np.max(np.abs(what - np.array(w))) == 0.0625 / 2


# ---------------------------------------------------------------------------
# P5: every positive finite bf16 group maximum, fp32-divide-then-bf16 scale vs
# the exactly rounded rational a / 7.
# ---------------------------------------------------------------------------
def test_scale_rounding_exhaustive():
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint16)  # all positive finite bf16
    W = np.zeros((bits.size, 128), dtype=np.uint16)
    W[:, 5] = bits
    W[:, 77] = bits ^ np.uint16(0x8000)  # the negative of the same value
    got = O.rtn_scales(W)[:, 0]
    exact = np.array([bf16_rne_bits(bf16_exact(int(b)) / 7) for b in bits], dtype=np.uint16)
    assert np.array_equal(got, exact)


# ---------------------------------------------------------------------------
# P4: brute force on small inputs with exact rational arithmetic.
# ---------------------------------------------------------------------------
def tie_heavy_rows(n_rows=4):
    """Rows whose groups hit many exact .5 quotients: d = 2^-4 and w on the
    half-step grid."""
    rng = np.random.default_rng(7)
    rows = []
    for r in range(n_rows):
        k = rng.integers(-14, 15, size=256).astype(np.float32)
        k[0] = 14 if r % 2 == 0 else -14
        k[128] = -14
        rows.append(k * np.float32(1 / 32))
    return f_to_bf16_bits(np.stack(rows))


@pytest.mark.parametrize("kind", ["normal", "ties", "outlier"])
def test_bruteforce_quantize_4x256(kind):
    if kind == "normal":
        W = wl.bits(wl.random_bf16((4, 256), 0.02, seed=11))
    elif kind == "ties":
        W = tie_heavy_rows()
    else:
        W = wl.bits(wl.random_bf16((4, 256), 0.02, seed=12)).copy()
        W[:, 3] = f_to_bf16_bits(O.bf16_bits_to_f32(W[:, 3]) * 8)
    packed, s = O.quantize_rtn(W)
    q = O.unpack_p1(packed, 256)
    for n in range(4):
        for g in range(2):
            d_bits, q_exact = exact_rtn_group(W[n, 128 * g: 128 * g + 128])
            assert s[n, g] == d_bits
            assert list(q[n, 128 * g: 128 * g + 128]) == q_exact


def test_bruteforce_matmul_3x4x256():
    W = wl.bits(wl.random_bf16((4, 256), 0.02, seed=21))
    x = wl.bits(wl.random_bf16((3, 256), 1.0, seed=22))
    packed, s = O.quantize_rtn(W)
    y, sabs = O.gemm_reference(x, packed, s, 256)
    assert y.shape == (3, 4)
    for n in range(4):
        qd = []
        for g in range(2):
            d_bits, qg = exact_rtn_group(W[n, 128 * g: 128 * g + 128])
            qd += [bf16_exact(d_bits) * qv for qv in qg]
        for m in range(3):
            xs = [bf16_exact(b) for b in x[m]]
            exact = sum(a * b for a, b in zip(qd, xs))
            exact_abs = sum(abs(a * b) for a, b in zip(qd, xs))
            assert abs(y[m, n] - float(exact)) <= 1e-12 * float(exact_abs)
            assert abs(sabs[m, n] - float(exact_abs)) <= 1e-12 * float(exact_abs)


# ---------------------------------------------------------------------------
# P2 / P6: invariants on workload-shaped matrices and special groups.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("workload", ["ffn", "outlier", "layer70b"])
def test_invariants(workload):
    K = 9216 if workload != "layer70b" else 8192
    W = wl.bits(wl.weight(workload, shape=(16, K)))
    packed, s = O.quantize_rtn(W)
    assert s.shape == (16, K // 128)
    if K == 9216:
        assert s.shape[1] == 72  # 72 groups per row at 9216 inputs
    assert packed.nbytes + s.nbytes == 0.515625 * 16 * K
    q = O.unpack_p1(packed, K)
    assert q.min() >= -7  # -8 is never produced with d = max|w|/7
    w = O.bf16_bits_to_f32(W).astype(np.float64).reshape(16, -1, 128)
    d = O.bf16_bits_to_f32(s).astype(np.float64)[:, :, None]
    what = q.astype(np.float64).reshape(16, -1, 128) * d
    assert np.all(np.abs(what - w) <= d / 2)
    # the group's largest-magnitude element maps to ±7 with its sign
    idx = np.argmax(np.abs(w), axis=2)
    wmax = np.take_along_axis(w, idx[:, :, None], 2)[:, :, 0]
    qmax = np.take_along_axis(q.reshape(16, -1, 128), idx[:, :, None], 2)[:, :, 0]
    assert np.all(qmax == 7 * np.sign(wmax))


def test_special_groups():
    W = np.zeros((4, 128), dtype=np.float32)
    W[1, :] = -0.375                 # all equal -> every q = -7
    W[2, 17] = 3e-39                 # single tiny (subnormal) element
    W[3, 0] = 1e-41                  # so tiny that bf16(a/7) is still > 0?
    Wb = O.f32_to_bf16_bits_rne(W)
    packed, s = O.quantize_rtn(Wb)
    q = O.unpack_p1(packed, 128)
    assert s[0, 0] == 0 and not q[0].any()          # all-zero group: d = +0
    assert np.all(q[1] == -7)
    assert q[2, 17] == 7 and np.count_nonzero(q[2]) == 1
    d_exact = bf16_rne_bits(bf16_exact(int(Wb[3, 0])) / 7)
    assert s[3, 0] == d_exact
    if d_exact == 0:
        assert not q[3].any()
    else:
        assert q[3, 0] == 7


def test_scale_underflow_to_zero():
    # smallest bf16 subnormal: a/7 rounds to 0 -> the group is treated as zero
    Wb = np.zeros((1, 128), dtype=np.uint16)
    Wb[0, 9] = 0x0001
    Wb[0, 10] = 0x8001
    packed, s = O.quantize_rtn(Wb)
    assert s[0, 0] == bf16_rne_bits(bf16_exact(1) / 7) == 0
    assert not packed.any()


# ---------------------------------------------------------------------------
# P3: the channel-scaling identity W'x' = Wx (§2 AWQ equation) for the fp64
# matmul step, and a brute-force loop for its orientation.
# ---------------------------------------------------------------------------
def test_channel_scaling_identity():
    rng = np.random.default_rng(3)
    W = rng.standard_normal((24, 384)) * 0.02
    x = rng.standard_normal((5, 384))
    s = np.exp2(rng.uniform(-2, 3, size=384))  # s_j in [0.25, 8], not powers of 2
    y = O.matmul_fp64(x, W)
    y2 = O.matmul_fp64(x / s, W * s)
    mag = np.abs(x) @ np.abs(W).T
    assert np.all(np.abs(y - y2) <= 1e-13 * mag)
    loop = np.array([[math.fsum(W[n, k] * x[m, k] for k in range(384)) for n in range(24)]
                     for m in range(5)])
    assert np.allclose(y, loop, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------------------
# P4: AWQ channel scaling applied before RTN (§2 AWQ equation), against exact
# rational arithmetic.  Reading: W' = bf16_rne(fp32(w·s_k)) and
# x' = bf16_rne(fp32(x / s_k)), both rounded twice (fp32, then bf16).
# ---------------------------------------------------------------------------
def fp32_then_bf16_bits(v: Fraction, negative: bool) -> int:
    return bf16_rne_bits(abs(float_rne(v, 24, -126))) | (0x8000 if negative else 0)


def exact_scaled_weight(w_bits: int, s: float) -> int:
    return fp32_then_bf16_bits(bf16_exact(w_bits) * Fraction(float(s)), bool(w_bits & 0x8000))


def exact_scaled_input(x_bits: int, s: float) -> int:
    return fp32_then_bf16_bits(bf16_exact(x_bits) / Fraction(float(s)), bool(x_bits & 0x8000))


def test_awq_unit_scale_is_plain_rtn():
    W = wl.bits(wl.random_bf16((5, 384), 0.02, seed=61))
    x = wl.bits(wl.random_bf16((3, 384), 1.0, seed=62))
    ones = np.ones(384, dtype=np.float32)
    p0, d0 = O.quantize_rtn(W)
    p1, d1 = O.quantize_rtn_scaled(W, ones)
    assert np.array_equal(p0, p1) and np.array_equal(d0, d1)
    assert np.array_equal(O.awq_scale_activations(x, ones), x)


@pytest.mark.parametrize("seed", [71, 72])
def test_awq_bruteforce_4x256(seed):
    rng = np.random.default_rng(seed)
    W = wl.bits(wl.random_bf16((4, 256), 0.02, seed=seed))
    x = wl.bits(wl.random_bf16((3, 256), 1.0, seed=seed + 100))
    s = np.exp2(rng.uniform(-3, 3, size=256)).astype(np.float32)
    assert np.mean(np.log2(s) == np.round(np.log2(s))) < 0.01  # not powers of two
    Wp = O.awq_scale_weights(W, s)
    packed, d = O.quantize_rtn_scaled(W, s)
    q = O.unpack_p1(packed, 256)
    for n in range(4):
        wp = [exact_scaled_weight(W[n, k], s[k]) for k in range(256)]
        assert list(Wp[n]) == wp
        for g in range(2):
            d_bits, q_exact = exact_rtn_group(wp[128 * g: 128 * g + 128])
            assert d[n, g] == d_bits
            assert list(q[n, 128 * g: 128 * g + 128]) == q_exact
    xp = O.awq_scale_activations(x, s)
    for m in range(3):
        assert list(xp[m]) == [exact_scaled_input(x[m, k], s[k]) for k in range(256)]


def double_rounding_cases():
    """(w bits, s) pairs whose exact product rounds to a bf16 tie in fp32, so
    that rounding once (exact -> bf16) and twice (exact -> fp32 -> bf16) give
    different bf16 results."""
    out = []
    for j in range(1, 128, 2):
        w = Fraction(128 + j, 128)
        for m in range(0, 128, 9):
            tie = Fraction(256 + 2 * m + 1, 256)  # halfway between two bf16 in [1, 2)
            s = float_rne(tie / w, 24, -126)
            p = w * s
            if p == tie or float_rne(p, 24, -126) != tie:
                continue
            if bf16_rne_bits(p) != bf16_rne_bits(tie):
                out.append((bf16_rne_bits(w), float(s)))
    return out


def test_awq_rounds_through_fp32():
    cases = double_rounding_cases()
    assert len(cases) >= 50
    W = np.array([[w for w, _ in cases]], dtype=np.uint16)
    s = np.array([s for _, s in cases], dtype=np.float32)
    Wp = O.awq_scale_weights(W, s)
    for k, (w, sk) in enumerate(cases):
        assert Wp[0, k] == exact_scaled_weight(w, sk)
        assert Wp[0, k] != bf16_rne_bits(bf16_exact(w) * Fraction(float(sk)))


def test_awq_power_of_two_group_scales():
    """s constant 2^e over each group: W' = W·2^e exactly, so the codes are the
    unscaled codes and every group scale is multiplied by 2^e exactly."""
    W = wl.bits(wl.random_bf16((6, 512), 0.02, seed=81))
    x = wl.bits(wl.random_bf16((2, 512), 1.0, seed=82))
    e = np.array([-3.0, 0.0, 2.0, 5.0])
    s = np.repeat(np.exp2(e), 128).astype(np.float32)
    p0, d0 = O.quantize_rtn(W)
    p1, d1 = O.quantize_rtn_scaled(W, s)
    assert np.array_equal(p0, p1)
    f0 = O.bf16_bits_to_f32(d0).astype(np.float64)
    f1 = O.bf16_bits_to_f32(d1).astype(np.float64)
    assert np.array_equal(f1, f0 * np.exp2(e)[None, :])
    xf = O.bf16_bits_to_f32(x).astype(np.float64)
    xs = O.bf16_bits_to_f32(O.awq_scale_activations(x, s)).astype(np.float64)
    assert np.array_equal(xs, xf / s[None, :])


def test_awq_rejects_bad_scales():
    W = wl.bits(wl.random_bf16((2, 256), 0.02, seed=91))
    for bad in (np.ones(128, np.float32), -np.ones(256, np.float32),
                np.full(256, np.inf, np.float32), np.zeros(256, np.float32)):
        with pytest.raises(ValueError):
            O.quantize_rtn_scaled(W, bad)


# ---------------------------------------------------------------------------
# P7: group sizes 32 / 64 and the asymmetric quantiser (§1 equation with a
# free zero point; §2 settings table on smaller groups).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["C", "D"])
def test_hand_worked_asym_groups(name):
    w_s, d_s, z_s, q_s, sum_s = read_golden()[name]
    w = [float(v) for v in w_s.split()]
    packed, s, zeros = O.quantize_rtn_asym(one_group_matrix(w))
    assert O.bf16_bits_to_f32(s)[0, 0] == float(d_s)
    assert int(zeros[0, 0]) == int(z_s) - 8
    c = O.unpack_p1(packed, 128)[0].astype(int)
    expect = [int(v) for v in q_s.split()]
    assert list(c[: len(expect)] + 8) == expect
    assert np.all(c[len(expect):] + 8 == int(z_s))
    x_ones = f_to_bf16_bits(np.ones((1, 128), dtype=np.float32))
    y, _ = O.gemm_reference(x_ones, packed, s, 128, 128, zeros)
    assert y[0, 0] == float(sum_s)


def asym_rows(kind, n_rows=4, K=256):
    if kind == "normal":
        return wl.bits(wl.random_bf16((n_rows, K), 0.02, seed=13))
    if kind == "ties":
        return tie_heavy_rows(n_rows)
    if kind == "skewed":  # one-signed groups, some with a single outlier
        W = np.abs(O.bf16_bits_to_f32(wl.bits(wl.random_bf16((n_rows, K), 0.02, seed=14))))
        W[1] = -W[1]
        W[2, 40] = 1.5
        W[3, 100:164] = 0.0
        return f_to_bf16_bits(W.astype(np.float32))
    raise ValueError(kind)


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("kind", ["normal", "ties", "skewed"])
def test_bruteforce_asym(kind, group):
    W = asym_rows(kind)
    packed, s, zeros = O.quantize_rtn_asym(W, group)
    c = O.unpack_p1(packed, W.shape[1]).astype(int)
    for n in range(W.shape[0]):
        for g in range(W.shape[1] // group):
            d_bits, z, q = exact_asym_group(W[n, group * g: group * g + group])
            assert s[n, g] == d_bits
            assert int(zeros[n, g]) == z - 8
            assert list(c[n, group * g: group * g + group] + 8) == q


@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("kind", ["normal", "ties", "outlier"])
def test_bruteforce_small_groups(kind, group):
    if kind == "outlier":
        W = wl.bits(wl.random_bf16((4, 256), 0.02, seed=12)).copy()
        W[:, 3] = f_to_bf16_bits(O.bf16_bits_to_f32(W[:, 3]) * 8)
    else:
        W = asym_rows(kind)
    packed, s = O.quantize_rtn(W, group)
    assert s.shape == (4, 256 // group)
    q = O.unpack_p1(packed, 256)
    for n in range(4):
        for g in range(256 // group):
            d_bits, q_exact = exact_rtn_group(W[n, group * g: group * g + group])
            assert s[n, g] == d_bits
            assert list(q[n, group * g: group * g + group]) == q_exact


@pytest.mark.parametrize("group", [32, 64, 128])
def test_asym_matmul_bruteforce(group):
    W = wl.bits(wl.random_bf16((3, 256), 0.02, seed=23))
    x = wl.bits(wl.random_bf16((2, 256), 1.0, seed=24))
    packed, s, zeros = O.quantize_rtn_asym(W, group)
    y, sabs = O.gemm_reference(x, packed, s, 256, group, zeros)
    for n in range(3):
        what = []
        for g in range(256 // group):
            d_bits, z, q = exact_asym_group(W[n, group * g: group * g + group])
            what += [bf16_exact(d_bits) * (qv - z) for qv in q]
        for m in range(2):
            xs = [bf16_exact(b) for b in x[m]]
            exact = sum(a * b for a, b in zip(what, xs))
            exact_abs = sum(abs(a * b) for a, b in zip(what, xs))
            assert abs(y[m, n] - float(exact)) <= 1e-12 * float(exact_abs)
            assert abs(sabs[m, n] - float(exact_abs)) <= 1e-12 * float(exact_abs)


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("workload", ["ffn", "outlier", "layer70b"])
def test_asym_invariants(workload, group):
    """Real zero is exact; the error is at most half a step (plus the clamp's
    margin from rounding d); d·z' is within half a step of lo."""
    N, K = wl.SHAPES[workload][0]
    W = wl.bits(wl.weight(workload, shape=(96, K)))
    packed, s, zeros = O.quantize_rtn_asym(W, group)
    w = O.bf16_bits_to_f32(W).astype(np.float64)
    what = O.dequantize_fp64(packed, s, K, group, zeros)
    d = np.repeat(O.bf16_bits_to_f32(s).astype(np.float64), group, axis=1)
    assert np.all(what[w == 0] == 0)
    assert np.all(np.abs(what - w) <= 0.5625 * d)
    lo = np.minimum(w.reshape(96, -1, group).min(axis=2), 0)
    dg = O.bf16_bits_to_f32(s).astype(np.float64)
    zq = zeros.astype(np.float64) + 8
    assert np.all(np.abs(-dg * zq - lo) <= 0.5 * dg + 1e-30)


def test_asym_special_groups():
    K = 512
    W = np.zeros((5, K), dtype=np.float32)
    W[1, :128] = 0.25 + np.arange(128) / 512        # all positive: z = 0
    W[2, :128] = -(0.25 + np.arange(128) / 512)     # all negative: z = 15
    W[3, :128] = 0.75                               # constant: q = 15
    W[4, :128] = -0.75                              # constant negative: q = 0
    Wb = np.concatenate([f_to_bf16_bits(W), np.zeros((1, K), dtype=np.uint16)])
    # Subnormal all-negative group: d = bf16(31·2^-133 / 15) = 2^-132 rounds
    # down so far that −lo/d = 15.5 rounds to 16, which the clip brings to 15.
    Wb[5, :128] = 0x801F
    packed, s, zeros = O.quantize_rtn_asym(Wb)
    c = O.unpack_p1(packed, K).astype(int)
    d_bits, z, q = exact_asym_group(Wb[5, :128])
    assert (d_bits, z) == (0x0002, 15) and s[5, 0] == 0x0002 and zeros[5, 0] == 7
    assert np.all(c[5, :128] == -8) and q == [0] * 128
    assert not s[0].any() and not zeros[0].any() and not packed[0].any()  # all-zero groups
    assert zeros[1, 0] == -8 and zeros[2, 0] == 7
    assert np.all(c[3, :128] == 7) and zeros[3, 0] == -8
    assert np.all(c[4, :128] == -8) and zeros[4, 0] == 7
    what = O.dequantize_fp64(packed, s, K, 128, zeros)
    d3 = float(O.bf16_bits_to_f32(s)[3, 0])
    assert what[3, 0] == 15 * d3 and abs(what[3, 0] - 0.75) <= d3 / 2


def test_group_size_rejects():
    W = wl.bits(wl.random_bf16((2, 256), 0.02, seed=3))
    for g in (16, 96, 256):
        with pytest.raises(ValueError):
            O.quantize_rtn(W, g)
        with pytest.raises(ValueError):
            O.quantize_rtn_asym(W, g)
    with pytest.raises(ValueError):
        O.quantize_rtn(wl.bits(wl.random_bf16((2, 96), 0.02, seed=3)), 32)


# ---------------------------------------------------------------------------
# Layout: the property the kernels use.  For word w of chunk j and slot i,
# ((word >> 4i) & 0x000F000F) ^ 0x43084308 is a bf16 pair (136 + q_k,
# 136 + q_{k+1}) with k = 32j + 8w + 2i.
# ---------------------------------------------------------------------------
def test_layout_pair_extraction():
    W = wl.bits(wl.random_bf16((8, 512), 0.02, seed=31))
    packed, s = O.quantize_rtn(W)
    q = O.unpack_p1(packed, 512).astype(np.int64)
    words = packed.view("<u4").reshape(8, 4, 4, 4)  # [n, g, chunk, word]
    for i in range(4):
        pair = ((words >> (4 * i)) & 0x000F000F) ^ 0x43084308
        lo = O.bf16_bits_to_f32((pair & 0xFFFF).astype(np.uint16)).astype(np.int64)
        hi = O.bf16_bits_to_f32((pair >> 16).astype(np.uint16)).astype(np.int64)
        for j in range(4):
            for wd in range(4):
                k = 32 * j + 8 * wd + 2 * i
                qg = q.reshape(8, 4, 128)
                assert np.array_equal(lo[:, :, j, wd] - 136, qg[:, :, k])
                assert np.array_equal(hi[:, :, j, wd] - 136, qg[:, :, k + 1])


def test_canonical_and_p1_hold_the_same_codes():
    W = wl.bits(wl.random_bf16((3, 256), 0.02, seed=41))
    packed, s = O.quantize_rtn(W)
    q = O.unpack_p1(packed, 256)
    canon = O.canonical_pack(q)
    lo = (canon & 0xF).astype(np.int16)
    hi = (canon >> 4).astype(np.int16)
    back = np.empty((3, 256), dtype=np.int16)
    back[:, 0::2], back[:, 1::2] = lo, hi
    back = np.where(back >= 8, back - 16, back)
    assert np.array_equal(back, q)
    # the byte multiset of each group block is not what matters; the codes are
    assert np.array_equal(np.sort(O.unpack_p1(O.pack_p1(q), 256), axis=1), np.sort(q, axis=1))


# ---------------------------------------------------------------------------
# bf16 rounding and ulp helpers against exact arithmetic.
# ---------------------------------------------------------------------------
def test_bf16_rne_against_exact():
    rng = np.random.default_rng(5)
    f = np.concatenate([
        rng.standard_normal(2000).astype(np.float32),
        (rng.standard_normal(500) * 1e-39).astype(np.float32),  # subnormals
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 - 2 ** -9, 2 ** -133 * 1.5], dtype=np.float32),
    ])
    got = O.f32_to_bf16_bits_rne(f)
    for v, b in zip(f, got):
        fr = Fraction(float(v))
        want = bf16_rne_bits(abs(fr)) | (0x8000 if fr < 0 else 0)
        if want & 0x7FFF == 0:
            want = 0x8000 if np.signbit(v) else 0
        assert int(b) == want


def test_bf16_ulp():
    assert O.bf16_ulp(np.array([1.0]))[0] == 2 ** -7
    assert O.bf16_ulp(np.array([-3.0]))[0] == 2 ** -6
    assert O.bf16_ulp(np.array([0.0]))[0] == 2 ** -133
    assert O.bf16_ulp(np.array([1e-39]))[0] == 2 ** -133


def test_parity_bound_accepts_exact_and_rejects_offset():
    W = wl.bits(wl.random_bf16((16, 256), 0.02, seed=51))
    x = wl.bits(wl.random_bf16((2, 256), 1.0, seed=52))
    packed, s = O.quantize_rtn(W)
    y, sabs = O.gemm_reference(x, packed, s, 256)
    yb = O.f32_to_bf16_bits_rne(y.astype(np.float32))
    assert O.parity_excess(yb, y, sabs).max() <= 1
    bad = O.f32_to_bf16_bits_rne((y + 0.05 * sabs).astype(np.float32))
    assert O.parity_excess(bad, y, sabs).max() > 1


# Hand-worked edges of the matmul tolerance |y − y_ref| ≤ 4e-3·Σ|ŵx| + ulp_bf16(y_ref):
# (y_ref, Σ|ŵx|, bf16 bits of y, inside the bound?).
#   y_ref = 1, Σ = 10: bound = 0.04 + 2⁻⁷ = 0.0478125; bf16 steps near 1 are 2⁻⁷ above and
#   2⁻⁸ below, so 1 ± 6/128 (0x3F86, 0x3F74) are inside and 1 ± 7/128 (0x3F87, 0x3F72) outside.
#   y_ref = 3, Σ = 0: ulp = 2^(1−7) = 2⁻⁶; 3 + 2⁻⁶ (0x4041) inside, 3 + 2⁻⁵ (0x4042) outside.
#   y_ref = 0, Σ = 0: ulp = 2⁻¹³³, the smallest bf16 subnormal (0x0001) inside, 2⁻¹³² (0x0002) outside.
BOUND_EDGES = [
    (1.0, 10.0, 0x3F80, True), (1.0, 10.0, 0x3F86, True), (1.0, 10.0, 0x3F87, False),
    (1.0, 10.0, 0x3F74, True), (1.0, 10.0, 0x3F72, False),
    (3.0, 0.0, 0x4041, True), (3.0, 0.0, 0x4042, False),
    (0.0, 0.0, 0x0001, True), (0.0, 0.0, 0x0002, False),
]


def test_parity_bound_edges():
    for y_ref, sabs, bits, inside in BOUND_EDGES:
        e = O.parity_excess(np.array([bits], dtype=np.uint16), np.array([y_ref]), np.array([sabs]))[0]
        assert (e <= 1) == inside, (y_ref, sabs, hex(bits), e)
