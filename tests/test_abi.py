"""C-ABI library checks that need no GPU: every symbol include/w4.h declares is
exported, and argument errors are rejected on the host before any launch."""
import ctypes
import os
import re

import pytest

import gemm_rtn_sym_gb300 as w4
from gemm_rtn_sym_gb300 import build as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(w4.library_path()):
        b.build()
    return w4.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "w4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(w4_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("w4_quantize_rtn", "w4_gemm", "w4_packed_bytes", "w4_scales_bytes",
                     "w4_last_device_status", "w4_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in w4.h but not exported"
        assert name in w4._SIGNATURES, f"{name} has no binding"


def test_size_helpers(lib):
    assert lib.w4_packed_bytes(2560, 9216) == 2560 * 9216 // 2
    assert lib.w4_scales_bytes(2560, 9216, 128) == 2560 * 72 * 2
    assert lib.w4_scales_bytes(2560, 9216, 64) == 2560 * 144 * 2
    assert lib.w4_scales_bytes(2560, 9216, 32) == 2560 * 288 * 2
    assert lib.w4_scales_bytes(2560, 9216, 96) == 0
    assert lib.w4_zeros_bytes(2560, 9216, 128) == 2560 * 72
    assert lib.w4_zeros_bytes(2560, 9216, 32) == 2560 * 288
    assert lib.w4_zeros_bytes(2560, 9216, 16) == 0
    assert lib.w4_zeros_bytes(4, 100, 32) == 0
    assert lib.w4_packed_bytes(4, 100) == 0
    assert lib.w4_packed_bytes(-1, 128) == 0
    # packed + scales = 0.515625 bytes per weight
    assert lib.w4_packed_bytes(7, 384) + lib.w4_scales_bytes(7, 384, 128) == 0.515625 * 7 * 384


def test_path_choice(lib):
    assert lib.w4_gemm_path_for(1, 2560, 9216) == w4.W4_PATH_SMALL_M
    assert lib.w4_gemm_path_for(16, 2560, 9216) == w4.W4_PATH_SMALL_M
    assert lib.w4_gemm_path_for(24, 2560, 9216) == w4.W4_PATH_SMALL_M
    assert lib.w4_gemm_path_for(25, 2560, 9216) == w4.W4_PATH_TENSOR
    assert lib.w4_gemm_path_for(208, 8192, 8192) == w4.W4_PATH_TENSOR
    assert lib.w4_gemm_path_for(-1, 2560, 9216) == -w4.W4_ERR_INVALID_ARG
    assert lib.w4_gemm_path_for(1, 2560, 100) == -w4.W4_ERR_UNSUPPORTED


def test_status_strings(lib):
    for s in range(7):
        assert lib.w4_status_string(s).decode().startswith("W4_")
    assert b"unknown" in lib.w4_status_string(99)


A16 = 0x10000  # fake, never dereferenced: every case below fails its checks first


@pytest.mark.parametrize("args,expect", [
    ((A16, 4, 256, 96, A16, A16, None), w4.W4_ERR_UNSUPPORTED),        # group 96
    ((A16, 4, 256, 16, A16, A16, None), w4.W4_ERR_UNSUPPORTED),        # group 16
    ((A16, 4, 200, 128, A16, A16, None), w4.W4_ERR_UNSUPPORTED),       # K % 128
    ((A16, -4, 256, 128, A16, A16, None), w4.W4_ERR_INVALID_ARG),      # negative N
    ((None, 4, 256, 128, A16, A16, None), w4.W4_ERR_INVALID_ARG),      # null W
    ((A16 + 8, 4, 256, 128, A16 * 4, A16 * 8, None), w4.W4_ERR_MISALIGNED),
    ((A16, 4, 256, 128, A16 + 512, A16 * 8, None), w4.W4_ERR_INVALID_ARG),  # packed inside W
    ((A16, 1 << 40, 1 << 30, 128, A16 * 4, A16 * 8, None), w4.W4_ERR_INVALID_ARG),  # overflow
])
def test_quantize_rejects(lib, args, expect):
    assert lib.w4_quantize_rtn(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((A16, 4, 256, 128, None, A16 * 4, A16 * 8, None), w4.W4_ERR_INVALID_ARG),           # null s
    ((A16, 4, 256, 128, A16 * 12 + 4, A16 * 4, A16 * 8, None), w4.W4_ERR_MISALIGNED),    # s at 4 B
    ((A16, 4, 256, 128, A16 * 8, A16 * 4, A16 * 8, None), w4.W4_ERR_INVALID_ARG),        # s on scales
    ((A16, 4, 256, 128, A16 * 4 + 256, A16 * 4, A16 * 8, None), w4.W4_ERR_INVALID_ARG),  # s in packed
    ((A16, 4, 256, 64, A16 * 12, A16 * 4, A16 * 8, None), w4.W4_ERR_UNSUPPORTED),        # group 64
])
def test_quantize_scaled_rejects(lib, args, expect):
    assert lib.w4_quantize_rtn_scaled(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((A16, 2, 200, A16 * 4, A16 * 8, None), w4.W4_ERR_UNSUPPORTED),       # K % 128
    ((A16, -2, 256, A16 * 4, A16 * 8, None), w4.W4_ERR_INVALID_ARG),
    ((None, 2, 256, A16 * 4, A16 * 8, None), w4.W4_ERR_INVALID_ARG),
    ((A16, 2, 256, None, A16 * 8, None), w4.W4_ERR_INVALID_ARG),
    ((A16, 2, 256, A16 * 4 + 8, A16 * 8, None), w4.W4_ERR_MISALIGNED),
    ((A16, 2, 256, A16 * 4, A16 * 8 + 2, None), w4.W4_ERR_MISALIGNED),
    ((A16, 2, 256, A16 * 4, A16 + 16, None), w4.W4_ERR_INVALID_ARG),     # out overlaps x, not equal
    ((A16, 2, 256, A16 * 4, A16 * 4 + 512, None), w4.W4_ERR_INVALID_ARG),  # out overlaps s
])
def test_scale_activations_rejects(lib, args, expect):
    assert lib.w4_scale_activations(*args) == expect


def test_awq_empty_is_noop(lib):
    assert lib.w4_quantize_rtn_scaled(None, 0, 256, 128, None, None, None, None) == w4.W4_OK
    assert lib.w4_scale_activations(None, 0, 256, None, None, None) == w4.W4_OK
    assert lib.w4_scale_activations(None, 3, 0, None, None, None) == w4.W4_OK


@pytest.mark.parametrize("args,expect", [
    ((A16, 4, 256, 96, A16 * 4, A16 * 8, A16 * 12, None), w4.W4_ERR_UNSUPPORTED),      # group 96
    ((A16, 4, 256, 32, A16 * 4, A16 * 8, None, None), w4.W4_ERR_INVALID_ARG),          # null zeros
    ((A16, 4, 256, 32, A16 * 4, A16 * 8, A16 * 8 + 8, None), w4.W4_ERR_INVALID_ARG),   # zeros in scales
    ((A16, 4, 256, 32, A16 * 4, A16 * 8, A16 + 100, None), w4.W4_ERR_INVALID_ARG),     # zeros in W
    ((A16, 4, 256, 64, A16 * 4 + 8, A16 * 8, A16 * 12, None), w4.W4_ERR_MISALIGNED),   # packed at 8 B
])
def test_quantize_asym_rejects(lib, args, expect):
    assert lib.w4_quantize_rtn_asym(*args) == expect


def test_quantize_scaled_needs_group_128(lib):
    assert lib.w4_quantize_rtn_scaled(A16, 4, 256, 64, A16 * 12, A16 * 4, A16 * 8, None) == w4.W4_ERR_UNSUPPORTED


@pytest.mark.parametrize("args,expect", [
    ((A16, 1, 4, 256, 96, A16 * 2, A16 * 4, None, A16 * 8, None, 0), w4.W4_ERR_UNSUPPORTED),  # group 96
    ((A16, 1, 4, 200, 32, A16 * 2, A16 * 4, None, A16 * 8, None, 0), w4.W4_ERR_UNSUPPORTED),  # K % 128
    ((A16, 1, 4, 256, 32, A16 * 2, A16 * 4, None, A16 * 8, None, 5), w4.W4_ERR_INVALID_ARG),  # bad path
    ((A16, 1, 4, 256, 32, A16 * 2, A16 * 4, A16 * 8, A16 * 8, None, 0), w4.W4_ERR_INVALID_ARG),  # y on zeros
    ((A16, 1, 4, 256, 64, A16 * 2 + 4, A16 * 4, None, A16 * 8, None, 0), w4.W4_ERR_MISALIGNED),
])
def test_gemm_affine_rejects(lib, args, expect):
    assert lib.w4_gemm_affine(*args) == expect


def test_gptq_rejects_without_gpu(lib):
    # w4_gptq_quantize(W, N, K, group, U, packed, scales, workspace, bytes, stream)
    assert lib.w4_gptq_quantize(A16, 4, 256, 96, A16 * 8, A16 * 2, A16 * 3, A16 * 16, 4096, None) == \
        w4.W4_ERR_UNSUPPORTED
    assert lib.w4_gptq_quantize(A16, 4, 200, 128, A16 * 8, A16 * 2, A16 * 3, A16 * 16, 4096, None) == \
        w4.W4_ERR_UNSUPPORTED
    assert lib.w4_gptq_quantize(A16, 4, 256, 128, None, A16 * 2, A16 * 3, A16 * 16, 4096, None) == \
        w4.W4_ERR_INVALID_ARG
    assert lib.w4_gptq_quantize(A16, 4, 256, 128, A16 * 8 + 4, A16 * 2, A16 * 3, A16 * 16, 4096, None) == \
        w4.W4_ERR_MISALIGNED
    assert lib.w4_gptq_quantize(A16, 4, 256, 128, A16 * 8, A16 * 2, A16 * 3, A16 * 16 + 16, 4096, None) == \
        w4.W4_ERR_MISALIGNED
    assert lib.w4_gptq_quantize(A16, 4, 256, 128, A16 * 8, A16 * 8 + 64, A16 * 3, A16 * 16, 4096, None) == \
        w4.W4_ERR_INVALID_ARG  # packed inside U
    assert lib.w4_gptq_quantize(None, 0, 256, 128, None, None, None, None, 0, None) == w4.W4_OK
    # w4_gptq_factor(H, K, damp, U, workspace, bytes, stream)
    assert lib.w4_gptq_factor(A16, 200, 0.01, A16 * 8, A16 * 16, 4096, None) == w4.W4_ERR_UNSUPPORTED
    assert lib.w4_gptq_factor(A16, 256, -1.0, A16 * 8, A16 * 16, 4096, None) == w4.W4_ERR_INVALID_ARG
    assert lib.w4_gptq_factor(A16, 256, float("nan"), A16 * 8, A16 * 16, 4096, None) == w4.W4_ERR_INVALID_ARG
    assert lib.w4_gptq_factor(A16, 256, 0.01, A16 * 8 + 4, A16 * 16, 4096, None) == w4.W4_ERR_MISALIGNED
    assert lib.w4_gptq_factor(A16, 256, 0.01, A16 + 1024, A16 * 16, 4096, None) == w4.W4_ERR_INVALID_ARG  # U on H
    assert lib.w4_gptq_workspace_bytes(2560, 9216) == 2560 * 9216 * 8 + 2560 * 128 * 8
    assert lib.w4_gptq_workspace_bytes(4, 200) == 0


def test_quantize_empty_is_noop(lib):
    assert lib.w4_quantize_rtn(None, 0, 256, 128, None, None, None) == w4.W4_OK
    assert lib.w4_quantize_rtn(None, 4, 0, 128, None, None, None) == w4.W4_OK


@pytest.mark.parametrize("args,expect", [
    ((A16, 1, 4, 200, A16 * 2, A16 * 4, A16 * 8, None, 0), w4.W4_ERR_UNSUPPORTED),
    ((A16, -1, 4, 256, A16 * 2, A16 * 4, A16 * 8, None, 0), w4.W4_ERR_INVALID_ARG),
    ((A16, 1, 4, 256, A16 * 2, A16 * 4, A16 * 8, None, 3), w4.W4_ERR_INVALID_ARG),   # bad path
    ((A16, 1, 4, 256, A16 * 2, A16 * 4, A16 * 8, None, -1), w4.W4_ERR_INVALID_ARG),
    ((None, 1, 4, 256, A16 * 2, A16 * 4, A16 * 8, None, 0), w4.W4_ERR_INVALID_ARG),
    ((A16, 1, 4, 256, A16 * 2, A16 * 4, None, None, 0), w4.W4_ERR_INVALID_ARG),
    ((A16 + 4, 1, 4, 256, A16 * 2, A16 * 4, A16 * 8, None, 0), w4.W4_ERR_MISALIGNED),
    ((A16, 1, 4, 256, A16 * 2 + 1, A16 * 4, A16 * 8, None, 0), w4.W4_ERR_MISALIGNED),
    ((A16, 1, 4, 256, A16 * 2, A16 * 4, A16 * 8 + 1, None, 0), w4.W4_ERR_MISALIGNED),
    ((A16, 4, 4, 256, A16 * 2, A16 * 4, A16, None, 0), w4.W4_ERR_INVALID_ARG),       # y aliases x
    ((A16, 1, 4, 256, A16 * 2, A16 * 4, A16 * 2 + 2, None, 0), w4.W4_ERR_INVALID_ARG),  # y in packed
])
def test_gemm_rejects(lib, args, expect):
    assert lib.w4_gemm_ex(*args) == expect


def test_grouped_rejects_without_gpu(lib):
    probs = (w4._Problem * 2)()
    probs[0] = w4._Problem(A16, 1, 4, 256, A16 * 2, A16 * 4, A16 * 8)
    probs[1] = w4._Problem(A16, 4, 4, 200, A16 * 2, A16 * 4, A16 * 16)  # K % 128 != 0
    assert lib.w4_grouped_plan_bytes(1, probs) == 640  # 128 + 384 + 4·2 + 8, rounded to 128
    assert lib.w4_grouped_plan_bytes(2, probs) == 0
    assert lib.w4_grouped_plan_bytes(0, probs) == 0
    plan = w4._Plan()
    assert lib.w4_grouped_plan_init(plan, A16 * 32 + 64, 4096, 1, probs) == w4.W4_ERR_MISALIGNED
    assert lib.w4_grouped_plan_init(plan, A16 * 32, 4096, 2, probs) == w4.W4_ERR_UNSUPPORTED
    assert lib.w4_gemm_grouped(None, None) == w4.W4_ERR_INVALID_ARG


def test_gemm_empty_is_noop(lib):
    assert lib.w4_gemm(None, 0, 4, 256, None, None, None, None) == w4.W4_OK
    assert lib.w4_gemm(None, 3, 0, 256, None, None, None, None) == w4.W4_OK


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(w4, "_lib", None)
    monkeypatch.setattr(w4, "library_path", lambda: str(tmp_path / "libw4.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        w4.load()


@pytest.mark.parametrize("lang", ["c", "c++"])
def test_header_is_a_c_abi(lib, lang, tmp_path):
    """w4.h compiles as strict C99 and as C++17, and a program that takes the
    address of every declared entry point links against libw4.so with the
    unmangled names (the header's extern "C" guard)."""
    import shutil
    import subprocess

    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip(f"no {lang} compiler")
    names = declared_functions()
    src = tmp_path / ("abi.c" if lang == "c" else "abi.cpp")
    body = ",\n    ".join(f"(void (*)(void)){n}" for n in names)
    src.write_text(
        '#include "w4.h"\n'
        "#include <stdio.h>\n"
        f"void (*const entry_points[])(void) = {{\n    {body}\n}};\n"
        "int main(void) {\n"
        "    static w4_gemm_problem p;\n"
        "    static w4_grouped_plan plan;\n"
        "    (void)p; (void)plan;\n"
        "    printf(\"%d\\n\", (int)(sizeof entry_points / sizeof entry_points[0]));\n"
        "    return w4_status_string(W4_OK) == NULL;\n"
        "}\n")
    std = ["-std=c99", "-pedantic"] if lang == "c" else ["-std=c++17"]
    lib_dir = os.path.dirname(w4.library_path())
    cmd = [cc, *std, "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
           "-o", str(tmp_path / "abi"), "-L", lib_dir, "-lw4", "-Wl,--unresolved-symbols=ignore-in-shared-libs"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
