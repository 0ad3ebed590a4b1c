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
    "w4_quantize_rtn", "w4_quantize_rtn_scaled", "w4_scale_activations", "w4_quantize_rtn_asym",
    "w4_gemm", "w4_gemm_ex", "w4_gemm_affine", "w4_gemm_path_for", "w4_zeros_bytes", "GROUPS",
    "w4_gptq_factor", "w4_gptq_quantize", "w4_gptq_workspace_bytes", "w4_gptq_factor_workspace_bytes",
    "W4_ERR_NUMERIC",
    "w4_packed_bytes", "w4_scales_bytes", "w4_last_device_status", "w4_wait_probe",
    "w4_status_string", "W4_PATH_AUTO", "W4_PATH_SMALL_M", "W4_PATH_TENSOR", "GROUP",
    "GroupedPlan", "w4_grouped_plan", "w4_gemm_grouped", "w4_gemm_grouped_noalloc",
]

GROUP = 128
GROUPS = (32, 64, 128)
W4_OK, W4_ERR_INVALID_ARG, W4_ERR_UNSUPPORTED, W4_ERR_MISALIGNED, W4_ERR_CUDA, W4_ERR_TIMEOUT, W4_ERR_NUMERIC = range(7)
W4_PATH_AUTO, W4_PATH_SMALL_M, W4_PATH_TENSOR = 0, 1, 2

_PKG = os.path.dirname(os.path.abspath(__file__))
_lib = None
_lock = threading.Lock()

_i64, _i32, _vp, _sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t


class _Problem(ctypes.Structure):
    """w4_gemm_problem of include/w4.h."""
    _fields_ = [("x", _vp), ("M", _i64), ("N", _i64), ("K", _i64), ("packed", _vp), ("scales", _vp), ("y", _vp)]


class _Plan(ctypes.Structure):
    """w4_grouped_plan of include/w4.h."""
    _fields_ = [("device_plan", _vp), ("bytes", _sz), ("count", _i32), ("device", _i32), ("items", _i32),
                ("ctas", _i32), ("token_rows", _i32), ("tc_items", _i32), ("tc_ctas", _i32), ("tc_max_bm", _i32),
                ("tc_offset", _sz), ("format", _i32)]

_SIGNATURES = {
    "w4_packed_bytes": (_sz, [_i64, _i64]),
    "w4_scales_bytes": (_sz, [_i64, _i64, _i32]),
    "w4_quantize_rtn": (ctypes.c_int, [_vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "w4_quantize_rtn_scaled": (ctypes.c_int, [_vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp]),
    "w4_quantize_rtn_asym": (ctypes.c_int, [_vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp]),
    "w4_zeros_bytes": (_sz, [_i64, _i64, _i32]),
    "w4_gptq_factor_workspace_bytes": (_sz, [_i64]),
    "w4_gptq_factor": (ctypes.c_int, [_vp, _i64, ctypes.c_double, _vp, _vp, _sz, _vp]),
    "w4_gptq_workspace_bytes": (_sz, [_i64, _i64]),
    "w4_gptq_quantize": (ctypes.c_int, [_vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "w4_gemm_affine": (ctypes.c_int, [_vp, _i64, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _i32]),
    "w4_scale_activations": (ctypes.c_int, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "w4_gemm": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "w4_gemm_ex": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _i32]),
    "w4_gemm_path_for": (ctypes.c_int, [_i64, _i64, _i64]),
    "w4_last_device_status": (ctypes.c_int, [_vp]),
    "w4_wait_probe": (ctypes.c_int, [_i64, _i32, _vp]),
    "w4_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "w4_grouped_plan_bytes": (_sz, [_i32, ctypes.POINTER(_Problem)]),
    "w4_grouped_plan_init": (ctypes.c_int, [ctypes.POINTER(_Plan), _vp, _sz, _i32, ctypes.POINTER(_Problem)]),
    "w4_gemm_grouped": (ctypes.c_int, [ctypes.POINTER(_Plan), _vp]),
    "w4_gemm_grouped_noalloc": (ctypes.c_int, [_i32, ctypes.POINTER(_Problem), _vp]),
    "w4_grouped_plan_bytes_affine": (_sz, [_i32, ctypes.POINTER(_Problem), _i32, ctypes.POINTER(_vp)]),
    "w4_grouped_plan_init_affine": (ctypes.c_int, [ctypes.POINTER(_Plan), _vp, _sz, _i32, ctypes.POINTER(_Problem),
                                                   _i32, ctypes.POINTER(_vp)]),
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


def w4_zeros_bytes(N: int, K: int, group: int = GROUP) -> int:
    return load().w4_zeros_bytes(N, K, group)


def w4_gemm_path_for(M: int, N: int, K: int) -> int:
    r = load().w4_gemm_path_for(M, N, K)
    if r < 0:
        raise W4Error(-r, "w4_gemm_path_for")
    return r


def _quant_outputs(W, group, packed, scales, where):
    _cuda_tensor(W, "W", torch.bfloat16, 2)
    N, K = W.shape
    if group not in GROUPS or K % GROUP:
        raise W4Error(W4_ERR_UNSUPPORTED, where)
    if packed is None:
        packed = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
    if scales is None:
        scales = torch.empty((N, K // group), dtype=torch.bfloat16, device=W.device)
    _cuda_tensor(packed, "packed", torch.uint8, 2)
    _cuda_tensor(scales, "scales", torch.bfloat16, 2)
    if tuple(packed.shape) != (N, K // 2) or tuple(scales.shape) != (N, K // group):
        raise ValueError("packed / scales have the wrong shape")
    return N, K, packed, scales


def w4_quantize_rtn(W: torch.Tensor, group: int = GROUP, packed: torch.Tensor | None = None,
                    scales: torch.Tensor | None = None):
    """RTN symmetric INT4 of W (bf16 [N, K]) -> (packed u8 [N, K/2], scales bf16 [N, K/group])."""
    N, K, packed, scales = _quant_outputs(W, group, packed, scales, "w4_quantize_rtn")
    with torch.cuda.device(W.device):
        _check(load().w4_quantize_rtn(W.data_ptr(), N, K, group, packed.data_ptr(),
                                      scales.data_ptr(), _stream(W.device)), "w4_quantize_rtn")
    return packed, scales


def w4_quantize_rtn_asym(W: torch.Tensor, group: int = GROUP, packed: torch.Tensor | None = None,
                         scales: torch.Tensor | None = None, zeros: torch.Tensor | None = None):
    """RTN asymmetric INT4 of W -> (packed u8 [N, K/2], scales bf16 [N, K/group],
    zeros int8 [N, K/group])."""
    N, K, packed, scales = _quant_outputs(W, group, packed, scales, "w4_quantize_rtn_asym")
    if zeros is None:
        zeros = torch.empty((N, K // group), dtype=torch.int8, device=W.device)
    _cuda_tensor(zeros, "zeros", torch.int8, 2)
    if tuple(zeros.shape) != (N, K // group):
        raise ValueError("zeros has the wrong shape")
    with torch.cuda.device(W.device):
        _check(load().w4_quantize_rtn_asym(W.data_ptr(), N, K, group, packed.data_ptr(), scales.data_ptr(),
                                           zeros.data_ptr(), _stream(W.device)), "w4_quantize_rtn_asym")
    return packed, scales, zeros


def _channel_scales(s: torch.Tensor, K: int) -> None:
    _cuda_tensor(s, "s", torch.float32, 1)
    if s.shape[0] != K:
        raise ValueError("s must hold one scale per input channel (K)")


def w4_quantize_rtn_scaled(W: torch.Tensor, s: torch.Tensor, group: int = GROUP,
                           packed: torch.Tensor | None = None, scales: torch.Tensor | None = None):
    """RTN of the channel-scaled weights W' = bf16(W · s) (s fp32 [K], finite, > 0)
    -> (packed u8 [N, K/2], scales bf16 [N, K/128])."""
    _cuda_tensor(W, "W", torch.bfloat16, 2)
    N, K = W.shape
    _channel_scales(s, K)
    if group != GROUP or K % GROUP:
        raise W4Error(W4_ERR_UNSUPPORTED, "w4_quantize_rtn_scaled")
    if packed is None:
        packed = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
    if scales is None:
        scales = torch.empty((N, K // GROUP), dtype=torch.bfloat16, device=W.device)
    _cuda_tensor(packed, "packed", torch.uint8, 2)
    _cuda_tensor(scales, "scales", torch.bfloat16, 2)
    if tuple(packed.shape) != (N, K // 2) or tuple(scales.shape) != (N, K // GROUP):
        raise ValueError("packed / scales have the wrong shape")
    with torch.cuda.device(W.device):
        _check(load().w4_quantize_rtn_scaled(W.data_ptr(), N, K, group, s.data_ptr(), packed.data_ptr(),
                                             scales.data_ptr(), _stream(W.device)), "w4_quantize_rtn_scaled")
    return packed, scales


def w4_scale_activations(x: torch.Tensor, s: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """x' = bf16(x / s): x bf16 [M, K], s fp32 [K] -> bf16 [M, K]; out may be x (in place)."""
    _cuda_tensor(x, "x", torch.bfloat16, 2)
    M, K = x.shape
    _channel_scales(s, K)
    if out is None:
        out = torch.empty_like(x)
    _cuda_tensor(out, "out", torch.bfloat16, 2)
    if tuple(out.shape) != (M, K):
        raise ValueError("out has the wrong shape")
    with torch.cuda.device(x.device):
        _check(load().w4_scale_activations(x.data_ptr(), M, K, s.data_ptr(), out.data_ptr(),
                                           _stream(x.device)), "w4_scale_activations")
    return out


def w4_gptq_factor(H: torch.Tensor, damp: float = 0.01, U: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None) -> torch.Tensor:
    """U (fp64 [K, K], upper triangle) with Uᵀ U = (H + λI)⁻¹, λ = damp·mean(diag H)."""
    _cuda_tensor(H, "H", torch.float32, 2)
    K = H.shape[0]
    if tuple(H.shape) != (K, K):
        raise ValueError("H must be square")
    if U is None:
        U = torch.empty((K, K), dtype=torch.float64, device=H.device)
    _cuda_tensor(U, "U", torch.float64, 2)
    if tuple(U.shape) != (K, K):
        raise ValueError("U must be [K, K]")
    with torch.cuda.device(H.device):
        need = load().w4_gptq_factor_workspace_bytes(K)
        if need == 0:
            raise W4Error(W4_ERR_UNSUPPORTED, "w4_gptq_factor_workspace_bytes")
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=H.device)
        _cuda_tensor(workspace, "workspace", torch.uint8, 1)
        _check(load().w4_gptq_factor(H.data_ptr(), K, float(damp), U.data_ptr(), workspace.data_ptr(),
                                     workspace.numel(), _stream(H.device)), "w4_gptq_factor")
    return U


def w4_gptq_quantize(W: torch.Tensor, U: torch.Tensor, group: int = GROUP, packed: torch.Tensor | None = None,
                     scales: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """GPTQ of W (bf16 [N, K]) given U from w4_gptq_factor -> (packed u8 [N, K/2],
    scales bf16 [N, K/group]), the RTN storage."""
    N, K, packed, scales = _quant_outputs(W, group, packed, scales, "w4_gptq_quantize")
    _cuda_tensor(U, "U", torch.float64, 2)
    if tuple(U.shape) != (K, K):
        raise ValueError("U must be [K, K]")
    with torch.cuda.device(W.device):
        need = load().w4_gptq_workspace_bytes(N, K)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=W.device)
        _cuda_tensor(workspace, "workspace", torch.uint8, 1)
        _check(load().w4_gptq_quantize(W.data_ptr(), N, K, group, U.data_ptr(), packed.data_ptr(),
                                       scales.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                       _stream(W.device)), "w4_gptq_quantize")
    return packed, scales


def w4_gptq_workspace_bytes(N: int, K: int) -> int:
    return load().w4_gptq_workspace_bytes(N, K)


def w4_gptq_factor_workspace_bytes(K: int) -> int:
    return load().w4_gptq_factor_workspace_bytes(K)


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


def w4_gemm_affine(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor | None = None,
                   group: int = GROUP, out: torch.Tensor | None = None, path: int = W4_PATH_AUTO) -> torch.Tensor:
    """y = Ŵ x with ŵ = d·(code − zero) per group of ``group`` (zeros int8 [N, K/group] or None)."""
    _cuda_tensor(x, "x", torch.bfloat16, 2)
    _cuda_tensor(packed, "packed", torch.uint8, 2)
    _cuda_tensor(scales, "scales", torch.bfloat16, 2)
    M, K = x.shape
    N = packed.shape[0]
    if group not in GROUPS:
        raise W4Error(W4_ERR_UNSUPPORTED, "w4_gemm_affine")
    if tuple(packed.shape) != (N, K // 2) or K % GROUP or tuple(scales.shape) != (N, K // group):
        raise ValueError("x / packed / scales shapes disagree")
    if zeros is not None:
        _cuda_tensor(zeros, "zeros", torch.int8, 2)
        if tuple(zeros.shape) != (N, K // group):
            raise ValueError("zeros has the wrong shape")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _cuda_tensor(out, "out", torch.bfloat16, 2)
    if tuple(out.shape) != (M, N):
        raise ValueError("out has the wrong shape")
    with torch.cuda.device(x.device):
        _check(load().w4_gemm_affine(x.data_ptr(), M, N, K, group, packed.data_ptr(), scales.data_ptr(),
                                     zeros.data_ptr() if zeros is not None else None, out.data_ptr(),
                                     _stream(x.device), path), "w4_gemm_affine")
    return out


class GroupedPlan:
    """A built grouped-matmul plan: the device memory holding it (a torch
    tensor) and the C descriptor.  Keeps the problems' tensors referenced, since
    the plan records their addresses."""

    def __init__(self, memory: torch.Tensor, plan: _Plan, tensors: list):
        self.memory = memory
        self.plan = plan
        self.tensors = tensors

    @property
    def items(self) -> int:
        return self.plan.items + self.plan.tc_items


def w4_grouped_plan(problems, group: int = GROUP, zeros=None) -> GroupedPlan:
    """Plan for many matmuls y_i = Ŵ_i x_i run by one w4_gemm_grouped call.
    problems: sequence of (x, packed, scales, y) CUDA tensors with the shapes
    of w4_gemm, all on one device.  For the affine formats of w4_gemm_affine:
    group (32, 64 or 128; scales [N, K/group]) and zeros, None or one entry
    per problem (an int8 [N, K/group] tensor, or None for symmetric codes)."""
    problems = list(problems)
    arr, n, device = _problem_array(problems, group)
    tensors = [t for p in problems for t in p]
    affine = group != GROUP or zeros is not None
    zarr = None
    if zeros is not None:
        zeros = list(zeros)
        if len(zeros) != n:
            raise ValueError("zeros needs one entry per problem")
        zarr = (_vp * n)()
        for i, (z, (x, packed, _, _)) in enumerate(zip(zeros, problems)):
            if z is None:
                continue
            _cuda_tensor(z, "zeros", torch.int8, 2)
            if tuple(z.shape) != (packed.shape[0], x.shape[1] // group) or z.device != device:
                raise ValueError(f"problem {i}: zeros must be int8 [N, K/group] on the problems' device")
            zarr[i] = z.data_ptr()
            tensors.append(z)
    with torch.cuda.device(device):
        if affine:
            nbytes = load().w4_grouped_plan_bytes_affine(n, arr, int(group), zarr)
        else:
            nbytes = load().w4_grouped_plan_bytes(n, arr)
        size = max(nbytes, 128)
        memory = torch.empty(size + 128, dtype=torch.uint8, device=device)
        off = (-memory.data_ptr()) % 128
        plan = _Plan()
        if affine:
            status = load().w4_grouped_plan_init_affine(ctypes.byref(plan), memory.data_ptr() + off, nbytes, n, arr,
                                                        int(group), zarr)
        else:
            status = load().w4_grouped_plan_init(ctypes.byref(plan), memory.data_ptr() + off, nbytes, n, arr)
        if status == W4_OK and nbytes == 0:
            status = W4_ERR_INVALID_ARG
        _check(status, "w4_grouped_plan_init")
    return GroupedPlan(memory, plan, tensors)


def _problem_array(problems, group: int = GROUP):
    """The w4_gemm_problem array of (x, packed, scales, y) tuples, after the
    shape, dtype and device checks (scales [N, K/group]); returns (array,
    count, device)."""
    problems = list(problems)
    if not problems:
        raise ValueError("no problems")
    arr = (_Problem * len(problems))()
    device = problems[0][0].device
    for i, (x, packed, scales, y) in enumerate(problems):
        _cuda_tensor(x, "x", torch.bfloat16, 2)
        _cuda_tensor(packed, "packed", torch.uint8, 2)
        _cuda_tensor(scales, "scales", torch.bfloat16, 2)
        _cuda_tensor(y, "y", torch.bfloat16, 2)
        M, K = x.shape
        N = packed.shape[0]
        if tuple(packed.shape) != (N, K // 2) or tuple(scales.shape) != (N, K // group) or tuple(y.shape) != (M, N):
            raise ValueError(f"problem {i}: x / packed / scales / y shapes disagree")
        if x.device != device or packed.device != device or scales.device != device or y.device != device:
            raise ValueError("all tensors of a grouped call must be on one device")
        arr[i] = _Problem(x.data_ptr(), M, N, K, packed.data_ptr(), scales.data_ptr(), y.data_ptr())
    return arr, len(problems), device


def w4_gemm_grouped_noalloc(problems) -> None:
    """Every problem (x, packed, scales, y) through the library's static plan
    buffer (no caller memory, no allocation; see w4.h for its race rules)."""
    arr, n, device = _problem_array(problems)
    with torch.cuda.device(device):
        _check(load().w4_gemm_grouped_noalloc(n, arr, _stream(device)), "w4_gemm_grouped_noalloc")


def w4_gemm_grouped(plan: GroupedPlan) -> None:
    """Runs every problem of the plan on the current stream of its device."""
    device = torch.device("cuda", plan.plan.device)
    with torch.cuda.device(device):
        _check(load().w4_gemm_grouped(ctypes.byref(plan.plan), _stream(device)), "w4_gemm_grouped")


def w4_last_device_status(device=None) -> int:
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        return load().w4_last_device_status(_stream(device))


def w4_wait_probe(limit_ns: int, arrive: bool, device=None) -> None:
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        _check(load().w4_wait_probe(int(limit_ns), int(bool(arrive)), _stream(device)), "w4_wait_probe")
