"""gemm_rtn_sym_gb300 — symmetric INT4 group-128 RTN quantiser and W4A16 matmul
for NVIDIA GB300 (sm_103a).

A thin ctypes binding over the C ABI in include/w4.h (libw4.so, built in-tree by
``gemm_rtn_sym_gb300.build``).  The functions here only check and marshal
arguments: torch tensors provide device memory and the current CUDA stream;
every step of the computation runs in the library's CUDA kernels.  There is no
CPU fallback: if libw4.so is missing or a CUDA device is absent, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "load", "library_path", "W4Error",
    "w4_quantize_rtn", "w4_gemm", "w4_gemm_ex", "w4_gemm_path_for",
    "w4_packed_bytes", "w4_scales_bytes", "w4_last_device_status", "w4_wait_probe",
    "w4_status_string", "W4_PATH_AUTO", "W4_PATH_SMALL_M", "W4_PATH_TENSOR", "GROUP",
]

GROUP = 128
W4_OK, W4_ERR_INVALID_ARG, W4_ERR_UNSUPPORTED, W4_ERR_MISALIGNED, W4_ERR_CUDA, W4_ERR_TIMEOUT = range(6)
W4_PATH_AUTO, W4_PATH_SMALL_M, W4_PATH_TENSOR = 0, 1, 2

_PKG = os.path.dirname(os.path.abspath(__file__))
_lib = None
_lock = threading.Lock()

_i64, _i32, _vp, _sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
_SIGNATURES = {
    "w4_packed_bytes": (_sz, [_i64, _i64]),
    "w4_scales_bytes": (_sz, [_i64, _i64, _i32]),
    "w4_quantize_rtn": (ctypes.c_int, [_vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "w4_gemm": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "w4_gemm_ex": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _i32]),
    "w4_gemm_path_for": (ctypes.c_int, [_i64, _i64, _i64]),
    "w4_last_device_status": (ctypes.c_int, [_vp]),
    "w4_wait_probe": (ctypes.c_int, [_i64, _i32, _vp]),
    "w4_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}


class W4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {w4_status_string(status)}")


def library_path() -> str:
    return os.path.join(_PKG, "libw4.so")


def load() -> ctypes.CDLL:
    """Load libw4.so (built by gemm_rtn_sym_gb300.build); raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with `python -m gemm_rtn_sym_gb300.build` "
                    "(there is no CPU fallback)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype, fn.argtypes = res, args
            _lib = lib
    return _lib


def w4_status_string(status: int) -> str:
    return load().w4_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != W4_OK:
        raise W4Error(status, where)


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _cuda_tensor(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor")


def w4_packed_bytes(N: int, K: int) -> int:
    return load().w4_packed_bytes(N, K)


def w4_scales_bytes(N: int, K: int, group: int = GROUP) -> int:
    return load().w4_scales_bytes(N, K, group)


def w4_gemm_path_for(M: int, N: int, K: int) -> int:
    r = load().w4_gemm_path_for(M, N, K)
    if r < 0:
        raise W4Error(-r, "w4_gemm_path_for")
    return r


def w4_quantize_rtn(W: torch.Tensor, group: int = GROUP, packed: torch.Tensor | None = None,
                    scales: torch.Tensor | None = None):
    """RTN symmetric INT4 of W (bf16 [N, K]) -> (packed u8 [N, K/2], scales bf16 [N, K/128])."""
    _cuda_tensor(W, "W", torch.bfloat16, 2)
    N, K = W.shape
    if group != GROUP or K % GROUP:
        raise W4Error(W4_ERR_UNSUPPORTED, "w4_quantize_rtn")
    if packed is None:
        packed = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
    if scales is None:
        scales = torch.empty((N, K // GROUP), dtype=torch.bfloat16, device=W.device)
    _cuda_tensor(packed, "packed", torch.uint8, 2)
    _cuda_tensor(scales, "scales", torch.bfloat16, 2)
    if tuple(packed.shape) != (N, K // 2) or tuple(scales.shape) != (N, K // GROUP):
        raise ValueError("packed / scales have the wrong shape")
    with torch.cuda.device(W.device):
        _check(load().w4_quantize_rtn(W.data_ptr(), N, K, group, packed.data_ptr(),
                                      scales.data_ptr(), _stream(W.device)), "w4_quantize_rtn")
    return packed, scales


def w4_gemm_ex(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
               out: torch.Tensor | None = None, path: int = W4_PATH_AUTO) -> torch.Tensor:
    """y = Ŵ x: x bf16 [M, K], packed u8 [N, K/2], scales bf16 [N, K/128] -> y bf16 [M, N]."""
    _cuda_tensor(x, "x", torch.bfloat16, 2)
    _cuda_tensor(packed, "packed", torch.uint8, 2)
    _cuda_tensor(scales, "scales", torch.bfloat16, 2)
    M, K = x.shape
    N = packed.shape[0]
    if tuple(packed.shape) != (N, K // 2) or tuple(scales.shape) != (N, K // GROUP) or K % GROUP:
        raise ValueError("x / packed / scales shapes disagree")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _cuda_tensor(out, "out", torch.bfloat16, 2)
    if tuple(out.shape) != (M, N):
        raise ValueError("out has the wrong shape")
    with torch.cuda.device(x.device):
        _check(load().w4_gemm_ex(x.data_ptr(), M, N, K, packed.data_ptr(), scales.data_ptr(),
                                 out.data_ptr(), _stream(x.device), path), "w4_gemm")
    return out


def w4_gemm(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
            out: torch.Tensor | None = None) -> torch.Tensor:
    return w4_gemm_ex(x, packed, scales, out, W4_PATH_AUTO)


def w4_last_device_status(device=None) -> int:
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        return load().w4_last_device_status(_stream(device))


def w4_wait_probe(limit_ns: int, arrive: bool, device=None) -> None:
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        _check(load().w4_wait_probe(int(limit_ns), int(bool(arrive)), _stream(device)), "w4_wait_probe")
