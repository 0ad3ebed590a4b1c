"""Shared helpers for the parity tests (host side only)."""
import numpy as np
import torch

from gemm_rtn_sym_gb300 import workloads as wl
from oracle import w4_oracle as O

GUARD = 256  # elements of guard band around every output buffer
SENTINEL_U8 = 0xA5
SENTINEL_BF16 = 0x7FA5  # a NaN pattern no kernel writes


def guarded(shape, dtype, device):
    """An output tensor embedded in a larger buffer whose margins hold a sentinel.
    Returns (view, buffer)."""
    n = int(np.prod(shape)) if len(shape) else 1
    buf = torch.empty(n + 2 * GUARD, dtype=dtype, device=device)
    if dtype == torch.uint8:
        buf.fill_(SENTINEL_U8)
    else:
        buf.view(torch.int16).fill_(SENTINEL_BF16)
    return buf[GUARD:GUARD + n].view(shape), buf


def guards_intact(buf) -> bool:
    head, tail = buf[:GUARD], buf[-GUARD:]
    if buf.dtype == torch.uint8:
        return bool((head == SENTINEL_U8).all() and (tail == SENTINEL_U8).all())
    h = head.view(torch.int16)
    t = tail.view(torch.int16)
    return bool((h == SENTINEL_BF16).all() and (t == SENTINEL_BF16).all())


def sample_rows(N: int, count: int, seed: int) -> np.ndarray:
    """Sorted distinct rows: the first and last 8 plus random ones."""
    rng = np.random.default_rng(seed)
    edge = set(range(min(8, N))) | set(range(max(0, N - 8), N))
    rest = rng.choice(N, size=min(N, count), replace=False)
    return np.array(sorted(edge | set(int(r) for r in rest)))


def quantize_gpu(w4, W):
    N, K = W.shape
    packed, pbuf = guarded((N, K // 2), torch.uint8, W.device)
    scales, sbuf = guarded((N, K // 128), torch.bfloat16, W.device)
    w4.w4_quantize_rtn(W, packed=packed, scales=scales)
    torch.cuda.synchronize()
    assert guards_intact(pbuf) and guards_intact(sbuf), "quantiser wrote outside its outputs"
    return packed, scales


def gemm_gpu(w4, x, packed, scales, path):
    M = x.shape[0]
    N = packed.shape[0]
    y, ybuf = guarded((M, N), torch.bfloat16, x.device)
    w4.w4_gemm_ex(x, packed, scales, out=y, path=path)
    torch.cuda.synchronize()
    assert guards_intact(ybuf), "matmul wrote outside y"
    assert w4.w4_last_device_status() == 0
    return y


def check_quantize(W, packed, scales, rows=None):
    Wb = wl.bits(W)
    pg = packed.cpu().numpy()
    sg = wl.bits(scales)
    if rows is not None:
        Wb, pg, sg = Wb[rows], pg[rows], sg[rows]
    p_ref, s_ref = O.quantize_rtn(Wb)
    assert np.array_equal(sg, s_ref), f"scale bits differ in {np.count_nonzero(sg != s_ref)} places"
    assert np.array_equal(pg, p_ref), f"packed bytes differ in {np.count_nonzero(pg != p_ref)} places"
    return p_ref, s_ref


def check_gemm(W, x, y, rows=None):
    """Oracle quantises W's (sampled) rows itself and compares y element by element."""
    Wb = wl.bits(W)
    yb = wl.bits(y)
    if rows is not None:
        Wb, yb = Wb[rows], yb[:, rows]
    K = Wb.shape[1]
    p_ref, s_ref = O.quantize_rtn(Wb)
    y_ref, s_abs = O.gemm_reference(wl.bits(x), p_ref, s_ref, K)
    excess = O.parity_excess(yb, y_ref, s_abs)
    worst = float(excess.max()) if excess.size else 0.0
    assert worst <= 1.0, f"max |err| / bound = {worst:.4g} at {np.unravel_index(np.argmax(excess), excess.shape)}"
    return worst
