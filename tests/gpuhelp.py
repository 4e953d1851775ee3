"""Helpers of the GPU parity tests: run the library through the C ABI on
device tensors, and run the oracle on host copies of the same inputs."""
import numpy as np
import torch

import oracle
from q8_quantized_gemv_gb300 import lk

DEV = "cuda"
TOL = 1e-5  # relative to sum_k |W x| per row


def to_dev(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if t.dtype == torch.uint16:
        t = t.view(torch.int16)
    return t.to(DEV)


def host(t):
    return t.detach().cpu().numpy()


def bits(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint64)


def act_buffers(M, K, mode):
    xq = torch.zeros((M, K), dtype=torch.int8, device=DEV)
    xl = torch.zeros((M, K), dtype=torch.int8, device=DEV) if mode == lk.LK_TWOPASS else None
    xs = torch.zeros((M, K // 32), dtype=torch.float32, device=DEV)
    return xq, xl, xs


def gpu_quantize(x_dev, mode):
    M, K = x_dev.shape
    xq, xl, xs = act_buffers(M, K, mode)
    lk.lk_quantize_act(x_dev, mode, xq, xl, xs)
    return xq, xl, xs


def gpu_gemv(wq_d, ws_d, mode, acts, M, amax=False):
    """acts: dict with x (Dequant) or xq/xl/xs.  Returns (y, parts, n_parts)."""
    N = wq_d.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    parts = None
    if amax:
        parts = torch.zeros((M * lk.lk_argmax_parts_max(N),), dtype=torch.int64, device=DEV)
    n = lk.lk_gemv_q8(wq_d, ws_d, mode, y, M=M, argmax_parts=parts, **acts)
    return y, parts, n


def oracle_acts(x_np, mode):
    if mode == oracle.DEQUANT:
        return dict(x=x_np)
    hi, lo, s = oracle.quantize(x_np, mode)
    return dict(hi=hi, lo=lo, s=s)


def dev_acts(x_np, mode):
    """Device activations for `mode`, quantized by the ORACLE (so GEMV parity
    is checked on identical inputs independently of the GPU quantizer)."""
    if mode == oracle.DEQUANT:
        return dict(x=to_dev(x_np))
    hi, lo, s = oracle.quantize(x_np, mode)
    d = dict(xq=to_dev(hi), xs=to_dev(s))
    if mode == oracle.TWOPASS:
        d["xl"] = to_dev(lo)
    return d


def assert_gemv_close(y_gpu, y_or, wq, ws, x_np, mode, rows=None, exact_quantized=True):
    """Quantized modes follow the oracle's order step for step: bit-exact.
    Dequant: within TOL * sum|W x| per row."""
    if mode != oracle.DEQUANT and exact_quantized:
        bad = np.nonzero(bits(y_gpu) != bits(y_or))
        assert bad[0].size == 0, f"{bad[0].size} mismatches, first at {tuple(b[0] for b in bad)}: " \
                                 f"gpu {y_gpu[tuple(b[0] for b in bad)]} oracle {y_or[tuple(b[0] for b in bad)]}"
    mag = oracle.absdot(wq, ws, x_np, rows=rows)
    err = np.abs(y_gpu.astype(np.float64) - y_or.astype(np.float64))
    assert np.all(err <= TOL * mag + 1e-30), float((err / np.maximum(mag, 1e-30)).max())


def ring_takes(N, K, mode, M):
    """Whether the bulk-copy ring kernel (the fused prologue's kernel) takes
    this shape, whatever kernel lk_gemv_q8 would pick for it."""
    prev = lk.lk_get_option("gemv_path")
    lk.lk_set_option("gemv_path", 2)
    try:
        return lk.lk_gemv_kernel_for(N, K, mode, M, 0) == 2
    finally:
        lk.lk_set_option("gemv_path", prev)
