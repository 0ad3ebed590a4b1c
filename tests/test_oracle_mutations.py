"""Planted mistakes: each mutant is a copy of the oracle with one plausible error
(a wrong rounding rule, a dropped rounding of the scale, a swapped nibble, a
transposed operand, a wrong divisor ...).  At least one pin must reject every
mutant, otherwise the pins would not be pinning the oracle down.  The mistakes
are planted on the CPU, in the oracle's source text; nothing here touches the
CUDA library.
"""
import os
import types

import pytest

import tests.test_oracle_gptq as gptq
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "w4_oracle.py")

MUTANTS = {
    "round_half_away": ("q = np.clip(np.rint(r), Q_MIN, Q_MAX)",
                        "q = np.clip(np.trunc(r + np.copysign(0.5, r)), Q_MIN, Q_MAX)"),
    "round_down_ties": ("q = np.clip(np.rint(r), Q_MIN, Q_MAX)",
                        "q = np.clip(np.ceil(r - 0.5), Q_MIN, Q_MAX)"),
    "divisor_8": ("DIVISOR = 7.0", "DIVISOR = 8.0"),
    "clip_symmetric_7": ("Q_MIN, Q_MAX = -8, 7", "Q_MIN, Q_MAX = -7, 6"),
    "scale_truncated": ("return f32_to_bf16_bits_rne(d32)",
                        "return (d32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)"),
    "divide_by_unrounded_scale": (
        "d = bf16_bits_to_f32(scale_bits)[:, :, None]\n    zero = d == 0",
        "d = (np.max(np.abs(w), axis=2) / np.float32(DIVISOR)).astype(np.float32)[:, :, None]\n    zero = d == 0"),
    "slot_order_swapped": ("P1_SLOT_K = (0, 2, 4, 6, 1, 3, 5, 7)", "P1_SLOT_K = (0, 1, 2, 3, 4, 5, 6, 7)"),
    "chunk_order_reversed": ("return 16 * j + 4 * w + bit // 8, bit % 8",
                             "return 16 * (3 - j) + 4 * w + bit // 8, bit % 8"),
    "no_sign_extension": ("c = np.where(c >= 8, c - 16, c)", "c = c"),
    "matmul_reversed_k": ("return np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T",
                          "return np.asarray(x, dtype=np.float64)[:, ::-1] @ np.asarray(w, dtype=np.float64).T"),
    "matmul_weights_transposed": ("return np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T",
                                  "return (np.asarray(w, dtype=np.float64) @ np.asarray(x, dtype=np.float64).T).T[:, ::-1]"),
    "scale_dropped_in_dequant": ("return (c * d[:, :, None]).reshape(N, K)",
                                 "return c.reshape(N, K)"),
    "abs_sum_signed": ("return matmul_fp64(x, w), matmul_fp64(np.abs(x), np.abs(w))",
                       "return matmul_fp64(x, w), np.abs(matmul_fp64(x, w))"),
    "ulp_off_by_one": ("out[nz] = np.exp2(np.maximum(e, -126.0) - 7.0)",
                       "out[nz] = np.exp2(np.maximum(e, -126.0) - 6.0)"),
    "bf16_round_half_up": ("round_up = (rest > 0x8000) | ((rest == 0x8000) & ((kept & np.uint32(1)) == 1))",
                           "round_up = rest >= 0x8000"),
    "awq_weights_divided": ("return f32_to_bf16_bits_rne((w * s[None, :]).astype(np.float32))",
                            "return f32_to_bf16_bits_rne((w / s[None, :]).astype(np.float32))"),
    "awq_channels_reversed": ("return f32_to_bf16_bits_rne((w * s[None, :]).astype(np.float32))",
                              "return f32_to_bf16_bits_rne((w * s[None, ::-1]).astype(np.float32))"),
    "awq_weights_truncated": ("return f32_to_bf16_bits_rne((w * s[None, :]).astype(np.float32))",
                              "return ((w * s[None, :]).astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)"),
    "awq_inputs_multiplied": ("return f32_to_bf16_bits_rne((x / s[None, :]).astype(np.float32))",
                              "return f32_to_bf16_bits_rne((x * s[None, :]).astype(np.float32))"),
    "awq_scale_ignored": ("return quantize_rtn(awq_scale_weights(W_bits, s), group)",
                          "return quantize_rtn(W_bits, group)"),
    "asym_divisor_16": ("DIVISOR_ASYM = 15.0", "DIVISOR_ASYM = 16.0"),
    "asym_range_without_zero": (
        "lo = np.minimum(np.min(w, axis=2), np.float32(0)).astype(np.float32)",
        "lo = np.min(w, axis=2).astype(np.float32)"),
    "asym_zero_added_before_rounding": (
        "n = np.where(zero, 0.0, np.rint(r)).astype(np.int64)\n    q = np.clip(n + zz, QA_MIN, QA_MAX)",
        "n = np.where(zero, 0.0, r).astype(np.float64)\n    q = np.clip(np.rint(n + zz), QA_MIN, QA_MAX).astype(np.int64)"),
    "asym_zero_point_unclipped": ("z = np.clip(np.rint(r), QA_MIN, QA_MAX)", "z = np.rint(r)"),
    "asym_zeros_ignored_in_dequant": ("c = c - np.asarray(zeros, dtype=np.float64)[:, :, None]", "c = c"),
    "asym_zero_sign_flipped": ("c = c - np.asarray(zeros, dtype=np.float64)[:, :, None]",
                               "c = c + np.asarray(zeros, dtype=np.float64)[:, :, None]"),
    "asym_empty_zero_0": ("ZERO_OF_EMPTY = 8", "ZERO_OF_EMPTY = 0"),
    "asym_codes_unshifted": ("return pack_p1((q - 8).astype(np.int8)), d_bits",
                             "return pack_p1(q.astype(np.int8)), d_bits"),
    "dequant_group_fixed_128": ("c = c.reshape(N, K // group, group)", "c = c.reshape(N, K // GROUP, GROUP)"),
    "gptq_lower_factor": ("    return L.T\n", "    return L\n"),
    "gptq_absolute_damping": ("return H + damp * np.mean(np.diag(H)) * np.eye(K)", "return H + damp * np.eye(K)"),
    "gptq_no_damping": ("return H + damp * np.mean(np.diag(H)) * np.eye(K)", "return H + 0.0 * np.eye(K)"),
    "gptq_error_unscaled": ("err = (W1[:, j] - d * qc) / U[c, c]", "err = (W1[:, j] - d * qc)"),
    "gptq_no_block_carry": ("W[:, i2:] -= E1 @ U[i1:i2, i2:]", "W[:, i2:] -= 0.0"),
    "gptq_column_not_row": ("W1[:, j:] -= np.outer(err, U[c, c:i2])", "W1[:, j:] -= np.outer(err, U[c:i2, c])"),
    "tolerance_10x_loose": ("TOL_REL = 4e-3", "TOL_REL = 4e-2"),
    "tolerance_ulp_dropped": ("    return TOL_REL * s_abs + bf16_ulp(y_ref)", "    return TOL_REL * s_abs + 0.0"),
    "tolerance_ulp_x4": ("    return TOL_REL * s_abs + bf16_ulp(y_ref)", "    return TOL_REL * s_abs + 4 * bf16_ulp(y_ref)"),
    "tolerance_signed_error": ("    return np.abs(y - y_ref) / parity_bound(y_ref, s_abs)",
                               "    return (y - y_ref) / parity_bound(y_ref, s_abs)"),
    "gptq_round_unclipped": ("    return np.clip(np.rint(r), Q_MIN, Q_MAX)\n\n\ndef gptq_quantize",
                             "    return np.rint(r)\n\n\ndef gptq_quantize"),
    "gptq_scale_divisor_8": ("    return f32_to_bf16_bits_rne((a / DIVISOR).astype(np.float32))",
                             "    return f32_to_bf16_bits_rne((a / 8.0).astype(np.float32))"),
    "gptq_scale_from_original": (
        "cur = W1[:, j:j + group] if j + group <= i2 - i1 else W[:, c:c + group]",
        "cur = bf16_bits_to_f32(np.asarray(W_bits, dtype=np.uint16))[:, c:c + group]"),
}

PIN_TESTS = [
    lambda: pins.test_hand_worked_groups("A"),
    lambda: pins.test_hand_worked_groups("B"),
    pins.test_hand_worked_packed_bytes,
    pins.test_hand_worked_error_is_half_step,
    pins.test_scale_rounding_exhaustive,
    lambda: pins.test_bruteforce_quantize_4x256("normal"),
    lambda: pins.test_bruteforce_quantize_4x256("ties"),
    lambda: pins.test_bruteforce_quantize_4x256("outlier"),
    pins.test_bruteforce_matmul_3x4x256,
    lambda: pins.test_invariants("ffn"),
    lambda: pins.test_invariants("outlier"),
    pins.test_special_groups,
    pins.test_channel_scaling_identity,
    pins.test_layout_pair_extraction,
    pins.test_bf16_rne_against_exact,
    pins.test_bf16_ulp,
    pins.test_parity_bound_accepts_exact_and_rejects_offset,
    pins.test_parity_bound_edges,
    pins.test_awq_unit_scale_is_plain_rtn,
    lambda: pins.test_awq_bruteforce_4x256(71),
    pins.test_awq_rounds_through_fp32,
    pins.test_awq_power_of_two_group_scales,
    lambda: pins.test_hand_worked_asym_groups("C"),
    lambda: pins.test_hand_worked_asym_groups("D"),
    lambda: pins.test_bruteforce_asym("ties", 32),
    lambda: pins.test_bruteforce_asym("skewed", 128),
    lambda: pins.test_bruteforce_small_groups("normal", 64),
    lambda: pins.test_asym_matmul_bruteforce(32),
    lambda: pins.test_asym_invariants("ffn", 64),
    pins.test_asym_special_groups,
    lambda: gptq.test_gptq_matches_obs_route(128),
    lambda: gptq.test_gptq_matches_obs_route(32),
    gptq.test_gptq_diagonal_h_is_rtn,
    lambda: gptq.test_gptq_block_size_does_not_change_the_result(32),
    gptq.test_gptq_scale_invariant_in_h,
    gptq.test_gptq_first_group_scale_is_rtn,
    gptq.test_gptq_singular_h,
]


def load_mutant(old: str, new: str) -> types.ModuleType:
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mod = types.ModuleType("w4_oracle_mutant")
    exec(compile(src.replace(old, new), "w4_oracle_mutant", "exec"), mod.__dict__)
    return mod


def test_every_pin_passes_on_the_oracle():
    """A pin that fails (or cannot be called) on the unmutated oracle would
    count every mutant as caught: each one must pass here first."""
    for t in PIN_TESTS:
        t()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_mutant_is_caught(name, monkeypatch):
    mutant = load_mutant(*MUTANTS[name])
    monkeypatch.setattr(pins, "O", mutant)
    monkeypatch.setattr(gptq, "O", mutant)
    caught = []
    for t in PIN_TESTS:
        try:
            t()
        except Exception as e:  # an assertion, or the mutant breaking outright
            caught.append(type(e).__name__)
    assert caught, f"no pin rejects the planted mistake {name!r}"
