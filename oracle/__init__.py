"""Plain CPU oracle of the Q8_0 decode-projection path.

TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the
benchmark's CPU-baseline leg call it; the library (``q8_quantized_gemv_gb300``)
never imports it, and it imports nothing from the library.  The arithmetic
lives in ``oracle.c`` and, for the GGUF block formats other than Q8_0,
``formats.c`` (plain C built with ``-ffp-contract=off``, one thread by
default; its GEMV row loops can be spread over host threads without changing
any bit); this module builds them and wraps them for numpy arrays.

Sources, by page:
  * "kernels.rs" (logicaffeine_compile codegen_cuda lane kernel library):
    the numerics modes, the activation quantizer, the quantized block step and
    its four-partial order, RMSNorm and its reduction tree (with the residual
    add), the gated projection pair (SwiGLU), the balanced split, and the
    decoder library of block formats (lk_sub, lk_sub_dot, lk_row_dot).
  * the QWEN38_EXTRA_KERNELS constant: "SPLIT-K FOR THE NARROW PROJECTIONS",
    the fused add + norm + quantize kernels and the SwiGLU + requantize one.
  * model-as-a-kernel "megakernel.cu": the argmax's first index of equal maxima.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

DEQUANT, INT8ACT, TWOPASS = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "formats.c")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, -O2 -ffp-contract=off)."""
    stale = (not os.path.exists(_LIB)) or any(os.path.getmtime(_LIB) < os.path.getmtime(f) for f in _SRCS)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-o", tmp] + _SRCS + ["-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i32, i64, f32 = ctypes.c_int, ctypes.c_long, ctypes.c_float
    lib.oracle_half_to_float.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_float.restype = f32
    lib.oracle_quantize_row.argtypes = [P, i32, i32, P, P, P]
    lib.oracle_norm_threads.argtypes = [i32]
    lib.oracle_norm_threads.restype = i32
    lib.oracle_sumsq_f32.argtypes = [P, i32]
    lib.oracle_sumsq_f32.restype = f32
    lib.oracle_sumsq_f64.argtypes = [P, i32]
    lib.oracle_sumsq_f64.restype = ctypes.c_double
    lib.oracle_rmsnorm_row.argtypes = [P, P, i32, f32, i32, P]
    lib.oracle_block_dots.argtypes = [P, i32, i32, P, P, P, P]
    lib.oracle_gemv_rows.argtypes = [P, P, i32, i32, P, P, P, P, i64, i64, P]
    lib.oracle_splitk_bound.argtypes = [i32, i32, i32]
    lib.oracle_splitk_bound.restype = i32
    lib.oracle_gemv_splitk_rows.argtypes = [P, P, i32, i32, P, P, P, P, i32, i64, i64, P, P, P]
    lib.oracle_absdot_rows.argtypes = [P, P, i32, P, i64, i64, P]
    lib.oracle_add_rmsnorm_row.argtypes = [P, P, P, i32, f32, i32, P, P]
    lib.oracle_add_rmsnorm_row.restype = i32
    lib.oracle_swiglu.argtypes = [P, P, i64, P]
    lib.oracle_set_threads.argtypes = [i32]
    lib.oracle_set_threads.restype = i32
    lib.oracle_get_threads.argtypes = []
    lib.oracle_get_threads.restype = i32
    lib.oracle_argmax.argtypes = [P, i64]
    lib.oracle_format_row_bytes.argtypes = [i32, i32]
    lib.oracle_format_row_bytes.restype = i64
    lib.oracle_sub_decode.argtypes = [i32, P, i32, P, P, P]
    lib.oracle_dequant_row.argtypes = [i32, P, i32, P]
    lib.oracle_gemv_blk_rows.argtypes = [i32, P, i64, i32, i32, P, P, P, P, i64, i64, P]
    lib.oracle_absdot_blk_rows.argtypes = [i32, P, i64, i32, P, i64, i64, P]
    lib.oracle_argmax.restype = i64
    _lib = lib
    return lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> int:
    """Host threads of the GEMV row loops (1, the default, is the plain
    single-threaded oracle; any count gives the same bits).  Returns the
    count in effect."""
    return _load().oracle_set_threads(int(n))


def get_threads() -> int:
    """Host threads the GEMV row loops use now."""
    return _load().oracle_get_threads()


def half_to_float(h) -> np.ndarray:
    """f16 bit patterns (uint16) -> f32 values, from the binary16 definition."""
    lib = _load()
    h = np.asarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    flat = out.reshape(-1)
    for i, v in enumerate(h.reshape(-1)):
        flat[i] = lib.oracle_half_to_float(int(v))
    return out


def quantize(v, mode: int):
    """Per-32-group activation quantizer.  v: [M, K] f32.  Returns (hi, lo, s):
    int8 [M, K], int8 [M, K] (zeros unless TwoPass), f32 [M, K/32]."""
    lib = _load()
    v = _c(np.atleast_2d(v), np.float32)
    M, K = v.shape
    assert K % 32 == 0 and mode in (INT8ACT, TWOPASS)
    hi = np.zeros((M, K), np.int8)
    lo = np.zeros((M, K), np.int8)
    s = np.zeros((M, K // 32), np.float32)
    for t in range(M):
        lib.oracle_quantize_row(_p(v[t]), K, mode, _p(hi[t]), _p(lo[t]), _p(s[t]))
    return hi, lo, s


def norm_threads(K: int) -> int:
    return _load().oracle_norm_threads(K)


def sumsq(v, mode: int) -> float:
    """The canonical-order sum of squares of one row (f32 unless Dequant)."""
    lib = _load()
    v = _c(v, np.float32)
    if mode == DEQUANT:
        return lib.oracle_sumsq_f64(_p(v), v.size)
    return np.float32(lib.oracle_sumsq_f32(_p(v), v.size))


def rmsnorm(x, g, mode: int, eps: float = 1e-6) -> np.ndarray:
    """Row-wise RMSNorm times gain g.  x: [M, K] f32 -> [M, K] f32."""
    lib = _load()
    x = _c(np.atleast_2d(x), np.float32)
    g = _c(g, np.float32)
    M, K = x.shape
    y = np.zeros((M, K), np.float32)
    for t in range(M):
        lib.oracle_rmsnorm_row(_p(x[t]), _p(g), K, eps, mode, _p(y[t]))
    return y


def add_rmsnorm(x, r, g, mode: int, eps: float = 1e-6):
    """Residual add, then RMSNorm: s = x + r (f32), y = RMSNorm(s) * g.
    x, r: [M, K] f32.  Returns (s, y)."""
    lib = _load()
    x = _c(np.atleast_2d(x), np.float32)
    r = _c(np.atleast_2d(r), np.float32)
    g = _c(g, np.float32)
    M, K = x.shape
    assert r.shape == (M, K)
    s = np.zeros((M, K), np.float32)
    y = np.zeros((M, K), np.float32)
    for t in range(M):
        assert lib.oracle_add_rmsnorm_row(_p(x[t]), _p(r[t]), _p(g), K, eps, mode, _p(s[t]), _p(y[t])) == 0
    return s, y


def swiglu(g, u) -> np.ndarray:
    """h = silu(g) * u = g / (1 + e^-g) * u, elementwise (f64, one rounding)."""
    lib = _load()
    g = _c(g, np.float32)
    u = _c(u, np.float32)
    assert g.shape == u.shape
    h = np.zeros(g.shape, np.float32)
    lib.oracle_swiglu(_p(g), _p(u), g.size, _p(h))
    return h


def glu(wg, wsg, wu, wsu, mode: int, x=None, hi=None, lo=None, s=None):
    """The gated projection pair of a decoder's MLP: g = Wg x and u = Wu x by
    gemv(), then h = swiglu(g, u), and h quantized by quantize() for the
    quantized modes.  Returns (g, u, h, (hq, hl, hs) or None)."""
    acts = dict(x=x, hi=hi, lo=lo, s=s)
    g = gemv(wg, wsg, mode, **acts)
    u = gemv(wu, wsu, mode, **acts)
    h = swiglu(g, u)
    return g, u, h, (quantize(h, mode) if mode != DEQUANT else None)


def block_dots(wq, hi, lo=None):
    """Exact int32 block dots of every (row, block) for one activation row."""
    lib = _load()
    wq = _c(wq, np.int8)
    N, K = wq.shape
    hi = _c(hi, np.int8)
    lo = None if lo is None else _c(lo, np.int8)
    d = np.zeros((N, K // 32), np.int32)
    e = np.zeros((N, K // 32), np.int32)
    lib.oracle_block_dots(_p(wq), N, K, _p(hi), _p(lo), _p(d), _p(e))
    return d, (e if lo is not None else None)


def _rows(rows, N):
    if rows is None:
        return 0, N
    r0, r1 = rows
    assert 0 <= r0 <= r1 <= N
    return r0, r1


def gemv(wq, ws, mode: int, x=None, hi=None, lo=None, s=None, rows=None) -> np.ndarray:
    """GEMV rows [r0, r1) for every activation row.  wq int8 [N, K], ws uint16
    (f16 bits) [N, K/32]; Dequant reads x [M, K] f32, the quantized modes read
    hi/lo [M, K] int8 and s [M, K/32] f32.  Returns y [M, r1-r0] f32."""
    lib = _load()
    wq = _c(wq, np.int8)
    ws = _c(ws, np.uint16)
    N, K = wq.shape
    r0, r1 = _rows(rows, N)
    acts = [_c(np.atleast_2d(a), dt) if a is not None else None
            for a, dt in ((x, np.float32), (hi, np.int8), (lo, np.int8), (s, np.float32))]
    M = next(a.shape[0] for a in acts if a is not None)
    y = np.zeros((M, r1 - r0), np.float32)
    for t in range(M):
        xt, ht, lt, st = (None if a is None else a[t] for a in acts)
        lib.oracle_gemv_rows(_p(wq), _p(ws), K, mode, _p(xt), _p(ht), _p(lt), _p(st), r0, r1,
                             _p(y[t]))
    return y


def splitk_bound(nb: int, S: int, c: int) -> int:
    return _load().oracle_splitk_bound(nb, S, c)


def gemv_splitk(wq, ws, mode: int, S: int, x=None, hi=None, lo=None, s=None, rows=None):
    """Split-K GEMV rows [r0, r1): returns (y [M, n] f32, chunks [S, M, n]) with
    chunks f32 for the quantized modes and f64 for Dequant."""
    lib = _load()
    wq = _c(wq, np.int8)
    ws = _c(ws, np.uint16)
    N, K = wq.shape
    r0, r1 = _rows(rows, N)
    n = r1 - r0
    acts = [_c(np.atleast_2d(a), dt) if a is not None else None
            for a, dt in ((x, np.float32), (hi, np.int8), (lo, np.int8), (s, np.float32))]
    M = next(a.shape[0] for a in acts if a is not None)
    y = np.zeros((M, n), np.float32)
    chunks = np.zeros((S, M, n), np.float64 if mode == DEQUANT else np.float32)
    for t in range(M):
        xt, ht, lt, st = (None if a is None else a[t] for a in acts)
        cf = np.zeros((S, n), np.float32)
        cd = np.zeros((S, n), np.float64)
        lib.oracle_gemv_splitk_rows(_p(wq), _p(ws), K, mode, _p(xt), _p(ht), _p(lt), _p(st), S,
                                    r0, r1, _p(y[t]), _p(cf), _p(cd))
        chunks[:, t, :] = cd if mode == DEQUANT else cf
    return y, chunks


def absdot(wq, ws, x, rows=None) -> np.ndarray:
    """sum_k |W[o,k] x[t,k]| in f64: [M, r1-r0], the scale of the tolerance."""
    lib = _load()
    wq = _c(wq, np.int8)
    ws = _c(ws, np.uint16)
    N, K = wq.shape
    r0, r1 = _rows(rows, N)
    x = _c(np.atleast_2d(x), np.float32)
    out = np.zeros((x.shape[0], r1 - r0), np.float64)
    for t in range(x.shape[0]):
        lib.oracle_absdot_rows(_p(wq), _p(ws), K, _p(x[t]), r0, r1, _p(out[t]))
    return out


def argmax(v) -> int:
    """First index of the maximum of a 1-D f32 array (linear scan, strict >)."""
    v = _c(v, np.float32).reshape(-1)
    assert v.size >= 1
    return int(_load().oracle_argmax(_p(v), v.size))


# ---- the GGUF block formats other than Q8_0 (formats.c) --------------------------

FORMATS = {"q4_0": 2, "q4_1": 3, "q5_0": 6, "q5_1": 7, "q2_k": 10, "q3_k": 11, "q4_k": 12, "q5_k": 13,
           "q6_k": 14, "iq4_nl": 20, "iq4_xs": 23, "mxfp4": 39}


def format_row_bytes(F: int, K: int) -> int:
    """Bytes of a row of K values in format F (0: K not a whole number of blocks)."""
    return int(_load().oracle_format_row_bytes(F, K))


def sub_decode(F: int, row, sb: int):
    """Sub-block sb of a row (uint8 bytes): (levels int8[32], d f32[2], c f32[2])."""
    row = _c(row, np.uint8)
    v = np.zeros(32, np.int8)
    d = np.zeros(2, np.float32)
    c = np.zeros(2, np.float32)
    assert _load().oracle_sub_decode(F, _p(row), sb, _p(v), _p(d), _p(c)) == 0
    return v, d, c


def dequant(F: int, w, K: int) -> np.ndarray:
    """w uint8 [N, row_bytes] -> the dequantized weights f32 [N, K]."""
    w = _c(np.atleast_2d(w), np.uint8)
    out = np.zeros((w.shape[0], K), np.float32)
    for o in range(w.shape[0]):
        assert _load().oracle_dequant_row(F, _p(w[o]), K, _p(out[o])) == 0
    return out


def gemv_blk(F: int, w, K: int, mode: int, x=None, hi=None, lo=None, s=None, rows=None) -> np.ndarray:
    """Block-format GEMV rows [r0, r1) for every activation row: w uint8
    [N, row_bytes]; activations as gemv.  Returns y [M, r1 - r0] f32."""
    lib = _load()
    w = _c(np.atleast_2d(w), np.uint8)
    N, rb = w.shape
    assert rb == format_row_bytes(F, K)
    r0, r1 = _rows(rows, N)
    acts = [_c(np.atleast_2d(a), dt) if a is not None else None
            for a, dt in ((x, np.float32), (hi, np.int8), (lo, np.int8), (s, np.float32))]
    M = next(a.shape[0] for a in acts if a is not None)
    y = np.zeros((M, r1 - r0), np.float32)
    for t in range(M):
        xt, ht, lt, st = (None if a is None else a[t] for a in acts)
        assert lib.oracle_gemv_blk_rows(F, _p(w), rb, K, mode, _p(xt), _p(ht), _p(lt), _p(st), r0, r1,
                                        _p(y[t])) == 0
    return y


def absdot_blk(F: int, w, K: int, x, rows=None) -> np.ndarray:
    """sum_k |w_k x_k| in f64 per row (w dequantized), [M, r1 - r0]."""
    lib = _load()
    w = _c(np.atleast_2d(w), np.uint8)
    N, rb = w.shape
    r0, r1 = _rows(rows, N)
    x = _c(np.atleast_2d(x), np.float32)
    out = np.zeros((x.shape[0], r1 - r0), np.float64)
    for t in range(x.shape[0]):
        assert lib.oracle_absdot_blk_rows(F, _p(w), rb, K, _p(x[t]), r0, r1, _p(out[t])) == 0
    return out
