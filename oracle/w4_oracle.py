"""CPU oracle for symmetric INT4 group-128 RTN quantisation and the W4A16 matmul.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and bench.py's
CPU-baseline / reference leg may import this module. The product package
(``gemm_rtn_sym_gb300``) never imports it and shares no code with it: the CUDA
path is checked against this file, never built from it.

What it computes, and from which passage
-----------------------------------------
Source: "Qwen3.5-4B, 작게 저장하면 무엇이 달라질까?" (Qwen3.5-4B whole-model
quantisation study, parksieon.github.io).

* §1, group-quantisation equation: q = clip(round(w/d) + z, q_min, q_max),
  ŵ = d·(q − z).  The symmetric case has z = 0 (§1 symbol table: symmetric
  quantisation searches no free zero point).
* §1, paragraph under the FFN example: a group is 128 consecutive weights of one
  row along the input direction (72 groups per row at 9216 inputs); each weight
  keeps its own 4-bit code, only the restore scale d is shared (16 codes, §1
  symbol table).
* §2 settings table: RTN group 128, 4-bit weights / BF16 inputs, "minmax ·
  symmetric" range from the group's extremes, no clipping-ratio search, no
  calibration input.
* §2 AWQ equation: scaling input channel j of W by s_j and of x by 1/s_j keeps
  W'x' = Wx; the channel scale s_j is not the group scale d and is not limited
  to powers of two (§2, paragraph after the equation).  W' is then quantised
  like any other weight matrix.
* §1 FFN example y = W x (2560×9216) and §2 Δy = (Ŵ − W) x: the matmul reads the
  restored weights ŵ = d·q against BF16 inputs.

Where the page is silent this module takes these readings (the library takes the
same ones, independently):

* divisor and code range: d = max|w| / 7 and q ∈ [−8, 7];
* d is computed as an fp32 IEEE quotient max|w| / 7, rounded to bf16 with
  round-to-nearest-even, and w is divided by that STORED bf16 d (so that
  |ŵ − w| ≤ d/2 holds for the stored scale);
* round() is round-half-to-even, applied to the fp32 IEEE quotient w / d;
* an all-zero group, or one whose bf16 d rounds to zero, has d = +0 and q = 0;
* no flush-to-zero anywhere: subnormal weights and scales are legal;
* NaN / Inf weights are outside the contract (results unspecified);
* storage: packed u8 [N, K/2] whose 64-byte block per (row, group) uses the
  "P1" nibble order defined by :func:`p1_nibble_position`; scales bf16 [N, K/128];
* AWQ channel scaling (§2 AWQ equation): s is a caller-supplied fp32 vector
  of K finite positive scales; W' = bf16_rne(fp32(w·s_k)) is quantised by the
  same RTN, and x' = bf16_rne(fp32(x / s_k)); results where w·s_k overflows
  are unspecified, like Inf weights;
* group sizes 32 and 64 (§2 settings table: a smaller group follows the range
  more closely at the cost of more scales) use the same rules per group; the
  packed code layout stays per 128 inputs, scales are [N, K/group];
* asymmetric (§1 equation with z ≠ 0; z is the code of real zero, §1 symbol
  table): lo = min(0, min w), hi = max(0, max w), d = bf16_rne(fp32(fp32(hi −
  lo) / 15)), z = clip(round_half_even(fp32(−lo / d)), 0, 15),
  q = clip(round_half_even(fp32(w / d)) + z, 0, 15); where d = 0, z = 8 and
  q = z.  Stored: the nibble q − 8 in the same layout and an int8 zero z − 8
  per group, so ŵ = d·(stored code − stored zero);
* GPTQ (§2 settings table and H' equation; the update rule of the published
  GPTQ algorithm): fp64 throughout; λ = 0.01·mean(diag H); columns in their
  original order; blocks of 128 columns; each group's scale is taken at the
  group's first column from its current (corrected) weights, d =
  bf16_rne(fp32(max|w|/7)) with the quotient in fp64, and q =
  clip(round_half_even(w/d), −8, 7) in fp64; H is an input (the study's
  calibration statistic; there is no calibration data here);
* the matmul reference accumulates ŵ·x in fp64 (exact products), and the
  parity bound is |y_gpu − y_ref| ≤ 4e-3 · Σ_k |ŵ_k x_k| + ulp_bf16(y_ref).

Every function below is plain numpy; nothing is blocked, fused or reordered
beyond what the definitions state.
"""
from __future__ import annotations

import numpy as np

GROUP = 128
GROUPS = (32, 64, 128)
Q_MIN, Q_MAX = -8, 7
DIVISOR = 7.0
# Asymmetric (z != 0) codes are unsigned, 0..15; the stored nibble is q - 8.
QA_MIN, QA_MAX = 0, 15
DIVISOR_ASYM = 15.0
ZERO_OF_EMPTY = 8
TOL_REL = 4e-3

# P1 nibble order: inside each 32-bit word (8 consecutive k), nibble slot i
# holds k offset P1_SLOT_K[i].  Slots i and i+4 therefore hold the pair
# (2i, 2i+1).
P1_SLOT_K = (0, 2, 4, 6, 1, 3, 5, 7)


# ---------------------------------------------------------------------------
# bf16 <-> binary32, from the IEEE 754 definition of bfloat16 as the upper half
# of a binary32 word.
# ---------------------------------------------------------------------------
def bf16_bits_to_f32(bits) -> np.ndarray:
    """Exact widening: a bf16 pattern is the high 16 bits of a binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16_bits_rne(values) -> np.ndarray:
    """Round binary32 to bfloat16, round-to-nearest, ties to even.

    The 16 discarded bits are compared with half an ulp (0x8000); the kept
    part is incremented when above half, or exactly half with an odd kept LSB.
    NaN stays a quiet NaN.
    """
    f = np.ascontiguousarray(values, dtype=np.float32)
    u = f.view(np.uint32)
    kept = u >> np.uint32(16)
    rest = u & np.uint32(0xFFFF)
    round_up = (rest > 0x8000) | ((rest == 0x8000) & ((kept & np.uint32(1)) == 1))
    out = (kept + round_up.astype(np.uint32)).astype(np.uint32)
    nan = np.isnan(f)
    out = np.where(nan, (kept | np.uint32(0x0040)), out)
    return out.astype(np.uint16)


def bf16_ulp(y) -> np.ndarray:
    """One bf16 ulp at |y|: 2^(max(e, −126) − 7) with e = floor(log2|y|);
    2^−133 (the smallest bf16 subnormal) at y = 0."""
    y = np.abs(np.asarray(y, dtype=np.float64))
    out = np.full(y.shape, 2.0 ** -133)
    nz = y > 0
    e = np.floor(np.log2(y[nz]))
    out[nz] = np.exp2(np.maximum(e, -126.0) - 7.0)
    return out


# ---------------------------------------------------------------------------
# RTN quantiser (§1 equation with z = 0, §2 "minmax · symmetric", group 128).
# ---------------------------------------------------------------------------
def _groups(W_bits: np.ndarray, group: int) -> np.ndarray:
    W_bits = np.asarray(W_bits, dtype=np.uint16)
    if W_bits.ndim != 2:
        raise ValueError("W must be 2-D [N, K]")
    N, K = W_bits.shape
    if group not in GROUPS:
        raise ValueError("group must be 32, 64 or 128")
    if K % GROUP:
        raise ValueError("K must be a multiple of 128 (the packed block)")
    return bf16_bits_to_f32(W_bits).reshape(N, K // group, group)


def rtn_scales(W_bits: np.ndarray, group: int = GROUP) -> np.ndarray:
    """Per (row, group): a = max|w|; d = bf16_rne(fp32(a / 7)).  Returns the
    scale bit patterns, uint16 [N, K/128]."""
    w = _groups(W_bits, group)
    a = np.max(np.abs(w), axis=2)                       # exact
    d32 = (a / np.float32(DIVISOR)).astype(np.float32)  # IEEE fp32 quotient, RN
    return f32_to_bf16_bits_rne(d32)


def rtn_codes(W_bits: np.ndarray, scale_bits: np.ndarray, group: int = GROUP) -> np.ndarray:
    """q = clip(round_half_even(w / d), −8, 7), with w / d the fp32 IEEE
    quotient by the stored bf16 d; q = 0 where d = 0.  int8 [N, K]."""
    w = _groups(W_bits, group)
    d = bf16_bits_to_f32(scale_bits)[:, :, None]
    zero = d == 0
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (w / np.where(zero, np.float32(1), d)).astype(np.float32)
    q = np.clip(np.rint(r), Q_MIN, Q_MAX)
    q = np.where(zero, 0.0, q)
    return q.astype(np.int8).reshape(w.shape[0], -1)


def p1_nibble_position(k_local: int) -> tuple[int, int]:
    """Where code k_local (0..127) of a group lives inside the group's 64-byte
    block: returns (byte offset in the block, bit shift inside that byte).

    Chunk j = k_local // 32 is the 16-byte piece at byte 16j; inside it, the
    32-bit little-endian word w = (k_local % 32) // 8 holds 8 consecutive k;
    offset e = k_local % 8 sits in nibble slot i with P1_SLOT_K[i] = e, i.e.
    bits 4i..4i+3 of the word.
    """
    j, rem = divmod(k_local, 32)
    w, e = divmod(rem, 8)
    i = P1_SLOT_K.index(e)
    bit = 4 * i
    return 16 * j + 4 * w + bit // 8, bit % 8


def canonical_pack(q: np.ndarray) -> np.ndarray:
    """Plain nibble packing: byte [n, k/2] holds code(k) in bits 0-3 and
    code(k+1) in bits 4-7 (two's complement nibbles)."""
    c = (np.asarray(q, dtype=np.int16) & 0xF).astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def pack_p1(q: np.ndarray) -> np.ndarray:
    """Stored layout: packed u8 [N, K/2]; the 64-byte block of (n, g) starts
    at byte n·K/2 + 64g and places each code by :func:`p1_nibble_position`."""
    q = np.asarray(q, dtype=np.int8)
    N, K = q.shape
    G = K // GROUP
    c = (q.astype(np.int16) & 0xF).astype(np.uint8).reshape(N, G, GROUP)
    blocks = np.zeros((N, G, 64), dtype=np.uint8)
    for k_local in range(GROUP):
        byte, shift = p1_nibble_position(k_local)
        blocks[:, :, byte] |= (c[:, :, k_local] << shift).astype(np.uint8)
    return blocks.reshape(N, K // 2)


def unpack_p1(packed: np.ndarray, K: int) -> np.ndarray:
    """Inverse of :func:`pack_p1`: int8 codes [N, K], sign-extended."""
    packed = np.asarray(packed, dtype=np.uint8)
    N = packed.shape[0]
    G = K // GROUP
    blocks = packed.reshape(N, G, 64)
    c = np.zeros((N, G, GROUP), dtype=np.int16)
    for k_local in range(GROUP):
        byte, shift = p1_nibble_position(k_local)
        c[:, :, k_local] = (blocks[:, :, byte] >> shift) & 0xF
    c = np.where(c >= 8, c - 16, c)
    return c.reshape(N, K).astype(np.int8)


def quantize_rtn(W_bits: np.ndarray, group: int = GROUP):
    """RTN symmetric INT4: W bf16 bits [N, K] -> (packed u8 [N, K/2],
    scale bits uint16 [N, K/group]).  The packed layout does not depend on the
    group size."""
    s = rtn_scales(W_bits, group)
    q = rtn_codes(W_bits, s, group)
    return pack_p1(q), s


# ---------------------------------------------------------------------------
# Asymmetric RTN: the §1 equation with a free zero point z (the position of
# real zero on the code grid, §1 symbol table), q in 0..15.
# ---------------------------------------------------------------------------
def asym_params(W_bits: np.ndarray, group: int = GROUP):
    """Per (row, group): lo = min(0, min w), hi = max(0, max w) (so that real 0
    lies on the grid); d = bf16_rne(fp32(fp32(hi − lo) / 15));
    z = clip(round_half_even(fp32(−lo / d)), 0, 15), and z = 8 where d = 0.
    Returns (scale bits uint16 [N, K/group], z int8 [N, K/group])."""
    w = _groups(W_bits, group)
    lo = np.minimum(np.min(w, axis=2), np.float32(0)).astype(np.float32)
    hi = np.maximum(np.max(w, axis=2), np.float32(0)).astype(np.float32)
    span = (hi - lo).astype(np.float32)                        # fp32 IEEE, RN
    d32 = (span / np.float32(DIVISOR_ASYM)).astype(np.float32)  # fp32 IEEE quotient, RN
    d_bits = f32_to_bf16_bits_rne(d32)
    d = bf16_bits_to_f32(d_bits)
    zero = d == 0
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (-lo / np.where(zero, np.float32(1), d)).astype(np.float32)
    z = np.clip(np.rint(r), QA_MIN, QA_MAX)
    z = np.where(zero, ZERO_OF_EMPTY, z)
    return d_bits, z.astype(np.int8)


def asym_codes(W_bits: np.ndarray, scale_bits: np.ndarray, z: np.ndarray, group: int = GROUP) -> np.ndarray:
    """q = clip(round_half_even(fp32(w / d)) + z, 0, 15), with the stored bf16
    d; q = z where d = 0 (so ŵ = 0).  int16 [N, K]."""
    w = _groups(W_bits, group)
    d = bf16_bits_to_f32(scale_bits)[:, :, None]
    zz = np.asarray(z, dtype=np.int16)[:, :, None]
    zero = d == 0
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (w / np.where(zero, np.float32(1), d)).astype(np.float32)
    n = np.where(zero, 0.0, np.rint(r)).astype(np.int64)
    q = np.clip(n + zz, QA_MIN, QA_MAX)
    return q.astype(np.int16).reshape(w.shape[0], -1)


def quantize_rtn_asym(W_bits: np.ndarray, group: int = GROUP):
    """RTN asymmetric INT4 -> (packed u8 [N, K/2] holding q − 8 in the same
    nibble layout, scale bits uint16 [N, K/group], zeros int8 [N, K/group]
    holding z − 8).  Then ŵ = d·(q − z) = d·(stored code − stored zero), and
    the symmetric format is the case stored zero = 0."""
    d_bits, z = asym_params(W_bits, group)
    q = asym_codes(W_bits, d_bits, z, group)
    return pack_p1((q - 8).astype(np.int8)), d_bits, (z.astype(np.int16) - 8).astype(np.int8)


# ---------------------------------------------------------------------------
# AWQ-style channel scaling (§2 AWQ equation: W'_ij = W_ij·s_j, x'_j = x_j/s_j,
# so that W'x' = Wx).  The caller supplies s; how s is searched (the §2 grid of
# exponents over calibration statistics) is not part of this module.
# ---------------------------------------------------------------------------
def _channel_scales(s, K: int) -> np.ndarray:
    s = np.asarray(s, dtype=np.float32)
    if s.shape != (K,):
        raise ValueError("s must be a vector of K channel scales")
    if not np.all(np.isfinite(s)) or np.any(s <= 0):
        raise ValueError("channel scales must be finite and positive")
    return s


def awq_scale_weights(W_bits: np.ndarray, s) -> np.ndarray:
    """W'[n, k] = bf16_rne(fp32(w[n, k] · s[k])): the fp32 IEEE product of the
    bf16 weight and the fp32 scale of its input channel k, rounded to bf16 with
    ties to even.  uint16 [N, K]."""
    w = bf16_bits_to_f32(np.asarray(W_bits, dtype=np.uint16))
    s = _channel_scales(s, w.shape[1])
    return f32_to_bf16_bits_rne((w * s[None, :]).astype(np.float32))


def awq_scale_activations(x_bits: np.ndarray, s) -> np.ndarray:
    """x'[m, k] = bf16_rne(fp32(x[m, k] / s[k])), the fp32 IEEE quotient.
    uint16 [M, K]."""
    x = bf16_bits_to_f32(np.asarray(x_bits, dtype=np.uint16))
    s = _channel_scales(s, x.shape[1])
    return f32_to_bf16_bits_rne((x / s[None, :]).astype(np.float32))


def quantize_rtn_scaled(W_bits: np.ndarray, s, group: int = GROUP):
    """RTN of the channel-scaled weights: quantize_rtn(W') with W' from
    :func:`awq_scale_weights`.  Same storage as :func:`quantize_rtn`."""
    return quantize_rtn(awq_scale_weights(W_bits, s), group)


# ---------------------------------------------------------------------------
# GPTQ into the same storage (§2 settings table: GPTQ, same storage as RTN,
# damping 0.01, no reordering, 128-column blocks; §2 H' = H + λI with
# λ = 0.01·mean(diag H); §2 method table: quantise one column, then correct
# the remaining weights).  The update rule is the published GPTQ algorithm
# (Frantar et al., "GPTQ: Accurate Post-Training Quantization for Generative
# Pre-trained Transformers", 2022, Algorithm 1), restated in fp64.
# ---------------------------------------------------------------------------
GPTQ_DAMP = 0.01
GPTQ_BLOCK = 128


def gptq_damped(H, damp: float = GPTQ_DAMP) -> np.ndarray:
    """H' = H + λI with λ = damp·mean(diag H), fp64."""
    H = np.asarray(H, dtype=np.float64)
    K = H.shape[0]
    return H + damp * np.mean(np.diag(H)) * np.eye(K)


def gptq_inverse_factor(H, damp: float = GPTQ_DAMP) -> np.ndarray:
    """Upper-triangular U with Uᵀ U = (H')⁻¹ (library inverse and Cholesky)."""
    Hinv = np.linalg.inv(gptq_damped(H, damp))
    L = np.linalg.cholesky((Hinv + Hinv.T) / 2)  # lower: Hinv = L Lᵀ
    return L.T


def gptq_group_scale(w: np.ndarray) -> np.ndarray:
    """Scale bits of groups of real-valued weights (last axis): d =
    bf16_rne(fp32(max|w| / 7)), the quotient taken in fp64 then rounded to fp32
    (for bf16 weights this is the RTN scale exactly)."""
    a = np.max(np.abs(np.asarray(w, dtype=np.float64)), axis=-1)
    return f32_to_bf16_bits_rne((a / DIVISOR).astype(np.float32))


def gptq_round(w: np.ndarray, d: np.ndarray) -> np.ndarray:
    """q = clip(round_half_even(w / d), −8, 7) in fp64, q = 0 where d = 0."""
    zero = d == 0
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(zero, 0.0, w / np.where(zero, 1.0, d))
    return np.clip(np.rint(r), Q_MIN, Q_MAX)


def gptq_quantize(W_bits: np.ndarray, H, group: int = GROUP, block: int = GPTQ_BLOCK,
                  damp: float = GPTQ_DAMP):
    """GPTQ of W (bf16 bits [N, K]) with the calibration statistic H ([K, K],
    symmetric positive semi-definite) -> (packed u8 [N, K/2], scale bits
    [N, K/group]), the RTN storage.

    Columns are taken in their original order in blocks of ``block``.  At the
    first column of each group the group's scale comes from its current
    (already corrected) weights.  Column c is rounded with that scale; its
    error, divided by U[c, c], corrects the later columns of the block at once
    (row c of U) and the columns after the block when the block ends."""
    W = bf16_bits_to_f32(np.asarray(W_bits, dtype=np.uint16)).astype(np.float64)
    N, K = W.shape
    if group not in GROUPS or K % GROUP:
        raise ValueError("group must be 32, 64 or 128 and K a multiple of 128")
    if block % group and group % block:
        raise ValueError("block and group sizes must divide one another")
    U = gptq_inverse_factor(H, damp)
    q = np.zeros((N, K), dtype=np.int8)
    s = np.zeros((N, K // group), dtype=np.uint16)
    d = np.zeros(N)
    for i1 in range(0, K, block):
        i2 = min(i1 + block, K)
        W1 = W[:, i1:i2].copy()
        E1 = np.zeros_like(W1)
        for j in range(i2 - i1):
            c = i1 + j
            if c % group == 0:
                # Current weights of the group: inside the block they carry the
                # block's corrections so far; a group longer than the block
                # starts at a block start, where W is already current.
                cur = W1[:, j:j + group] if j + group <= i2 - i1 else W[:, c:c + group]
                s[:, c // group] = gptq_group_scale(cur)
                d = bf16_bits_to_f32(s[:, c // group]).astype(np.float64)
            qc = gptq_round(W1[:, j], d)
            q[:, c] = qc.astype(np.int8)
            err = (W1[:, j] - d * qc) / U[c, c]
            W1[:, j:] -= np.outer(err, U[c, c:i2])
            E1[:, j] = err
        W[:, i2:] -= E1 @ U[i1:i2, i2:]
    return pack_p1(q), s


# ---------------------------------------------------------------------------
# Matmul y = Ŵ x  (§1 FFN example; ŵ = d·q from the §1 equation).
# ---------------------------------------------------------------------------
def dequantize_fp64(packed: np.ndarray, scale_bits: np.ndarray, K: int, group: int = GROUP,
                    zeros: np.ndarray | None = None) -> np.ndarray:
    """ŵ = d·(c − z') in fp64, c the stored code and z' the stored zero (0 when
    ``zeros`` is None, the symmetric case).  Exact: d has 8 significant bits,
    c − z' at most 5."""
    c = unpack_p1(packed, K).astype(np.float64)
    d = bf16_bits_to_f32(scale_bits).astype(np.float64)
    N = c.shape[0]
    c = c.reshape(N, K // group, group)
    if zeros is not None:
        c = c - np.asarray(zeros, dtype=np.float64)[:, :, None]
    return (c * d[:, :, None]).reshape(N, K)


def matmul_fp64(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y[m, n] = Σ_k w[n, k] · x[m, k], fp64 (a library matmul as one step)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T


def gemm_reference(x_bits: np.ndarray, packed: np.ndarray, scale_bits: np.ndarray, K: int,
                   group: int = GROUP, zeros: np.ndarray | None = None):
    """Returns (y_ref, s_abs), both fp64 [M, N]: y_ref = Ŵ x and
    s_abs = Σ_k |ŵ_k x_k|, the magnitude the parity bound scales with."""
    x = bf16_bits_to_f32(np.asarray(x_bits, dtype=np.uint16)).astype(np.float64)
    w = dequantize_fp64(packed, scale_bits, K, group, zeros)
    return matmul_fp64(x, w), matmul_fp64(np.abs(x), np.abs(w))


def parity_bound(y_ref: np.ndarray, s_abs: np.ndarray) -> np.ndarray:
    """Allowed |y_gpu − y_ref| per element: 4e-3 · Σ|ŵx| + one bf16 ulp."""
    return TOL_REL * s_abs + bf16_ulp(y_ref)


def parity_excess(y_bits: np.ndarray, y_ref: np.ndarray, s_abs: np.ndarray) -> np.ndarray:
    """|y_gpu − y_ref| / bound per element (≤ 1 passes)."""
    y = bf16_bits_to_f32(np.asarray(y_bits, dtype=np.uint16)).astype(np.float64)
    return np.abs(y - y_ref) / parity_bound(y_ref, s_abs)
