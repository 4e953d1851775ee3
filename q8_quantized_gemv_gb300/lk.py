"""Thin ctypes binding of liblk.so (the C ABI declared in include/lk.h).

Each ``lk_*`` function here has the name and argument order of the C entry
point; it only checks and marshals torch tensors (dtype, device, contiguity,
sizes) into pointers and the current CUDA stream.  All arithmetic runs in the
library's sm_103a kernels.  If liblk.so is missing the first call raises: there
is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblk.so")

LK_DEQUANT, LK_INT8ACT, LK_TWOPASS = 0, 1, 2
MODES = {"dequant": LK_DEQUANT, "int8act": LK_INT8ACT, "twopass": LK_TWOPASS}
LK_MAX_M = 8
LK_MAX_BATCH = 64
LK_MAX_SPLITK = 64
LK_TRACE_REC = 8  # entries of one launch record of option "trace" 3
LK_TRACE_MAX_RECORDS = 4096 // LK_TRACE_REC  # records the timeline keeps before wrapping

STATUS = {0: "LK_OK", -1: "LK_ERR_ARG", -2: "LK_ERR_ALIGN", -3: "LK_ERR_SHAPE",
          -4: "LK_ERR_WORKSPACE", -5: "LK_ERR_CUDA", -6: "LK_ERR_DEVICE_TIMEOUT"}


class LkChainOp(ctypes.Structure):
    """One step of lk_gemv_chain (the C struct lk_chain_op)."""
    _fields_ = [("wq", ctypes.c_void_p), ("ws", ctypes.c_void_p), ("N", ctypes.c_int), ("K", ctypes.c_int),
                ("x", ctypes.c_void_p), ("gain", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("argmax_parts", ctypes.c_void_p), ("argmax_idx", ctypes.c_void_p), ("wait", ctypes.c_int),
                ("reserved", ctypes.c_int)]


class LkGemvTarget(ctypes.Structure):
    """One matrix of lk_gemv_q8_group (the C struct lk_gemv_target)."""
    _fields_ = [("wq", ctypes.c_void_p), ("ws", ctypes.c_void_p), ("N", ctypes.c_int), ("reserved", ctypes.c_int),
                ("y", ctypes.c_void_p)]


CFG_FIELDS = ("pdl", "prefill", "path", "grid_ctas", "ring_tk", "mma_min_m", "mma_tk", "mma_warps", "mma_depth",
              "mma_i8", "mma_group", "mma_act16")
PATHS = {"auto": 0, "direct": 1, "ring": 2, "mma": 3}


class LkLaunchCfg(ctypes.Structure):
    """Per-call launch settings (the C struct lk_launch_cfg; see include/lk.h)."""
    _fields_ = [(f, ctypes.c_int) for f in CFG_FIELDS]


def launch_cfg(**kw) -> LkLaunchCfg:
    """lk_launch_cfg from keyword fields (every other field 0, the default):
    pdl, prefill, path (0..3 or "auto"/"direct"/"ring"/"mma"), grid_ctas,
    ring_tk, mma_min_m, mma_tk, mma_warps, mma_depth, mma_i8, mma_group,
    mma_act16."""
    bad = set(kw) - set(CFG_FIELDS)
    if bad:
        raise TypeError(f"launch_cfg: unknown fields {sorted(bad)}")
    if isinstance(kw.get("path"), str):
        kw["path"] = PATHS[kw["path"]]
    return LkLaunchCfg(*[int(kw.get(f, 0)) for f in CFG_FIELDS])


def _cfg(cfg):
    return None if cfg is None else ctypes.byref(cfg)


class LkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({_load().lk_status_string(status).decode()})")


_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built: run q8_quantized_gemv_gb300.build.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, L, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_long, ctypes.c_float, ctypes.c_size_t
    sig = {
        "lk_status_string": ([I], ctypes.c_char_p),
        "lk_version": ([], I),
        "lk_rmsnorm_quant": ([P, P, I, I, F, I, P, P, P, P, P, P], I),
        "lk_quantize_act": ([P, I, I, I, P, P, P, P, P], I),
        "lk_gemv_q8": ([P, P, I, I, I, P, P, P, P, I, P, P, P, P, P], I),
        "lk_splitk_workspace_bytes": ([I, I, I, I], S),
        "lk_gemv_q8_splitk": ([P, P, I, I, I, P, P, P, P, I, I, P, S, P, P], I),
        "lk_splitk_combine": ([I, P, I, I, I, P, P, P], I),
        "lk_splitk_chunks_for": ([I, I, I, I], I),
        "lk_format_row_bytes": ([I, I], S),
        "lk_gemv_blk": ([I, P, I, I, I, P, P, P, P, I, P, P, P], I),
        "lk_dequant_blk": ([I, P, I, I, P, P], I),
        "lk_argmax_parts_max": ([I], I),
        "lk_argmax_scratch_entries": ([I], I),
        "lk_argmax": ([P, P, I, I, I, P, P, P], I),
        "lk_q8_block_dots": ([P, I, I, P, P, P, P, P], I),
        "lk_set_option": ([ctypes.c_char_p, L], I),
        "lk_get_option": ([ctypes.c_char_p], L),
        "lk_device_error": ([I, ctypes.POINTER(I)], I),
        "lk_selftest_wait_timeout": ([ctypes.c_uint, P], I),
        "lk_gemv_kernel_for": ([I, I, I, I, I, P], I),
        "lk_rmsnorm_quant_gemv_q8": ([P, P, I, I, I, P, P, F, I, P, P, P, P, P], I),
        "lk_chain_sync_bytes": ([], S),
        "lk_trace_read": ([P, I], I),
        "lk_argmax_noalloc": ([P, I, I, P, P], I),
        "lk_gemv_chain": ([P, P, I, I, I, F, P, P, P], I),
        "lk_gemv_q8_group": ([P, I, I, I, P, P, P, P, I, P, P], I),
        "lk_add_rmsnorm_quant": ([P, P, P, I, I, F, I, P, P, P, P, P, P, P], I),
        "lk_swiglu_quant": ([P, P, I, I, L, I, P, P, P, P, P, P], I),
        "lk_gemv_q8_glu": ([P, P, P, P, I, I, I, P, P, P, P, I, P, P, P, P, P, P, P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def exported_symbols():
    return ["lk_status_string", "lk_version", "lk_rmsnorm_quant", "lk_quantize_act", "lk_gemv_q8",
            "lk_splitk_workspace_bytes", "lk_gemv_q8_splitk", "lk_splitk_combine",
            "lk_argmax_parts_max", "lk_argmax_scratch_entries", "lk_argmax", "lk_q8_block_dots",
            "lk_set_option", "lk_get_option", "lk_device_error", "lk_selftest_wait_timeout", "lk_gemv_kernel_for",
            "lk_rmsnorm_quant_gemv_q8", "lk_chain_sync_bytes", "lk_gemv_chain", "lk_trace_read",
            "lk_argmax_noalloc", "lk_gemv_q8_group", "lk_add_rmsnorm_quant", "lk_swiglu_quant",
            "lk_gemv_q8_glu", "lk_splitk_chunks_for", "lk_format_row_bytes", "lk_gemv_blk", "lk_dequant_blk"]


def _ok(st, where):
    if st != 0:
        raise LkError(st, where)


def _mode(mode):
    return MODES[mode] if isinstance(mode, str) else int(mode)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


_I8 = torch.int8
_F32 = torch.float32
_WS = (torch.int16, torch.float16)


def lk_status_string(status: int) -> str:
    return _load().lk_status_string(status).decode()


def lk_version() -> int:
    return _load().lk_version()


def lk_rmsnorm_quant(x, gain, mode, eps=1e-6, xn=None, xq=None, xl=None, xs=None, stream=None, cfg=None):
    M, K = x.shape
    _ok(_load().lk_rmsnorm_quant(_ptr(x, _F32, "x"), _ptr(gain, _F32, "gain"), M, K, eps, _mode(mode),
                                 _ptr(xn, _F32, "xn"), _ptr(xq, _I8, "xq"), _ptr(xl, _I8, "xl"),
                                 _ptr(xs, _F32, "xs"), _cfg(cfg), _stream(stream)), "lk_rmsnorm_quant")


def lk_add_rmsnorm_quant(x, r, gain, mode, eps=1e-6, s=None, xn=None, xq=None, xl=None, xs=None, stream=None,
                         cfg=None):
    """s = x + r (optional output), then lk_rmsnorm_quant of the sum."""
    M, K = x.shape
    if tuple(r.shape) != (M, K):
        raise ValueError("r must have the shape of x")
    _ok(_load().lk_add_rmsnorm_quant(_ptr(x, _F32, "x"), _ptr(r, _F32, "r"), _ptr(gain, _F32, "gain"), M, K, eps,
                                     _mode(mode), _ptr(s, _F32, "s"), _ptr(xn, _F32, "xn"), _ptr(xq, _I8, "xq"),
                                     _ptr(xl, _I8, "xl"), _ptr(xs, _F32, "xs"), _cfg(cfg), _stream(stream)),
        "lk_add_rmsnorm_quant")


def _pitched_rows(t, name):
    """Pointer and row pitch (elements) of a 2-D f32 CUDA tensor whose rows
    are contiguous (a column slice of a wider row-major tensor is fine)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != _F32 or t.dim() != 2:
        raise TypeError(f"{name} must be a 2-D float32 CUDA tensor")
    if t.stride(1) != 1:
        raise ValueError(f"{name} rows must be contiguous")
    return ctypes.c_void_p(t.data_ptr()), t.stride(0)


def lk_swiglu_quant(gate, up, mode, h=None, hq=None, hl=None, hs=None, stream=None, cfg=None):
    """h = silu(gate) * up, quantized for the next GEMV.  gate and up are
    [M, F] f32 with contiguous rows and the same row pitch (e.g. the two
    halves gu[:, :F], gu[:, F:] of a fused gate/up output)."""
    M, F = gate.shape
    if tuple(up.shape) != (M, F):
        raise ValueError("up must have the shape of gate")
    pg, ldg = _pitched_rows(gate, "gate")
    pu, ldu = _pitched_rows(up, "up")
    if ldg != ldu:
        raise ValueError("gate and up must have the same row pitch")
    _ok(_load().lk_swiglu_quant(pg, pu, M, F, ldg, _mode(mode), _ptr(h, _F32, "h"), _ptr(hq, _I8, "hq"),
                                _ptr(hl, _I8, "hl"), _ptr(hs, _F32, "hs"), _cfg(cfg), _stream(stream)),
        "lk_swiglu_quant")


def lk_quantize_act(x, mode, xq, xl, xs, stream=None, cfg=None):
    M, K = x.shape
    _ok(_load().lk_quantize_act(_ptr(x, _F32, "x"), M, K, _mode(mode), _ptr(xq, _I8, "xq"),
                                _ptr(xl, _I8, "xl"), _ptr(xs, _F32, "xs"), _cfg(cfg), _stream(stream)),
        "lk_quantize_act")


def lk_gemv_q8(wq, ws, mode, y, x=None, xq=None, xl=None, xs=None, argmax_parts=None, M=None,
               stream=None, cfg=None) -> int:
    """y[M, N] = W x.  Returns the number of argmax partial keys written per
    activation row (0 when argmax_parts is None).  cfg: launch_cfg(...) or
    None (the defaults)."""
    N, K = wq.shape
    if M is None:
        M = (x if x is not None else xq).shape[0]
    n = ctypes.c_int(0)
    args = [_ptr(wq, _I8, "wq"), _ptr(ws, _WS, "ws"), N, K, _mode(mode), _ptr(x, _F32, "x"), _ptr(xq, _I8, "xq"),
            _ptr(xl, _I8, "xl"), _ptr(xs, _F32, "xs"), M, _ptr(y, _F32, "y"),
            _ptr(argmax_parts, torch.int64, "argmax_parts"), ctypes.byref(n) if argmax_parts is not None else None]
    _ok(_load().lk_gemv_q8(*args, _cfg(cfg), _stream(stream)), "lk_gemv_q8")
    return n.value


def lk_gemv_q8_group(mats, mode, x=None, xq=None, xl=None, xs=None, M=None, stream=None, cfg=None):
    """mats: [(wq, ws, y), ...] sharing K and the activation: y = W x for
    each, with the bits of one lk_gemv_q8 call per matrix; one launch where
    the tensor-core kernel (2..8 rows) or, for two or more matrices, the
    chain kernel's ring arrangement (one row) takes the shapes."""
    K = mats[0][0].shape[1]
    if M is None:
        M = (x if x is not None else xq).shape[0]
    arr = (LkGemvTarget * len(mats))(*[LkGemvTarget(_ptr(wq, _I8, "wq"), _ptr(ws, _WS, "ws"), wq.shape[0], 0,
                                                    _ptr(y, _F32, "y")) for wq, ws, y in mats])
    for wq, _, _ in mats:
        if wq.shape[1] != K:
            raise ValueError("lk_gemv_q8_group: matrices of one group share K")
    args = [ctypes.cast(arr, ctypes.c_void_p), len(mats), K, _mode(mode), _ptr(x, _F32, "x"), _ptr(xq, _I8, "xq"),
            _ptr(xl, _I8, "xl"), _ptr(xs, _F32, "xs"), M]
    _ok(_load().lk_gemv_q8_group(*args, _cfg(cfg), _stream(stream)), "lk_gemv_q8_group")


def lk_gemv_q8_glu(wg, wsg, wu, wsu, mode, gu, x=None, xq=None, xl=None, xs=None, h=None, hq=None, hl=None,
                   hs=None, cnt=None, M=None, stream=None, cfg=None):
    """g = Wg x, u = Wu x into gu [2, M, F]; h = silu(g) * u (optional f32
    [M, F]) and its quantized words hq/hl/hs for the next GEMV.  cnt: int32
    [F/32] zeroed counters (enables the one-launch kernel at M = 1)."""
    F, K = wg.shape
    if tuple(wu.shape) != (F, K):
        raise ValueError("the gate and up matrices must have the same shape")
    if M is None:
        M = (x if x is not None else xq).shape[0]
    if tuple(gu.shape) != (2, M, F):
        raise ValueError("gu must be [2, M, F]")
    args = [_ptr(wg, _I8, "wg"), _ptr(wsg, _WS, "wsg"), _ptr(wu, _I8, "wu"), _ptr(wsu, _WS, "wsu"), F, K,
            _mode(mode), _ptr(x, _F32, "x"), _ptr(xq, _I8, "xq"), _ptr(xl, _I8, "xl"), _ptr(xs, _F32, "xs"), M,
            _ptr(gu, _F32, "gu"), _ptr(h, _F32, "h"), _ptr(hq, _I8, "hq"), _ptr(hl, _I8, "hl"), _ptr(hs, _F32, "hs"),
            _ptr(cnt, torch.int32, "cnt")]
    _ok(_load().lk_gemv_q8_glu(*args, _cfg(cfg), _stream(stream)), "lk_gemv_q8_glu")


def lk_gemv_kernel_for(N, K, mode, M, S=0, cfg=None) -> int:
    """1 direct kernel, 2 bulk-copy ring kernel, 3 tensor-core kernel, 0 none
    (see include/lk.h)."""
    return _load().lk_gemv_kernel_for(N, K, _mode(mode), M, S, _cfg(cfg))


def lk_rmsnorm_quant_gemv_q8(wq, ws, mode, x, y, gain=None, eps=1e-6, argmax_parts=None,
                             stream=None, cfg=None) -> int:
    """RMSNorm (gain given) or quantize only (gain None) -> GEMV in one launch.
    Returns the number of argmax partial keys per activation row."""
    N, K = wq.shape
    M = x.shape[0]
    n = ctypes.c_int(0)
    _ok(_load().lk_rmsnorm_quant_gemv_q8(_ptr(wq, _I8, "wq"), _ptr(ws, _WS, "ws"), N, K, _mode(mode),
                                         _ptr(x, _F32, "x"), _ptr(gain, _F32, "gain"), eps, M,
                                         _ptr(y, _F32, "y"),
                                         _ptr(argmax_parts, torch.int64, "argmax_parts"),
                                         ctypes.byref(n) if argmax_parts is not None else None,
                                         _cfg(cfg), _stream(stream)), "lk_rmsnorm_quant_gemv_q8")
    return n.value


def lk_splitk_workspace_bytes(mode, S, M, N) -> int:
    return _load().lk_splitk_workspace_bytes(_mode(mode), S, M, N)


def lk_gemv_q8_splitk(wq, ws, mode, S, part, x=None, xq=None, xl=None, xs=None, M=None, stream=None, cfg=None):
    N, K = wq.shape
    if M is None:
        M = (x if x is not None else xq).shape[0]
    _ok(_load().lk_gemv_q8_splitk(_ptr(wq, _I8, "wq"), _ptr(ws, _WS, "ws"), N, K, _mode(mode),
                                  _ptr(x, _F32, "x"), _ptr(xq, _I8, "xq"), _ptr(xl, _I8, "xl"),
                                  _ptr(xs, _F32, "xs"), M, S, _ptr(part, None, "part"),
                                  part.numel() * part.element_size(), _cfg(cfg), _stream(stream)),
        "lk_gemv_q8_splitk")


def lk_splitk_combine(mode, part, S, M, N, y, stream=None, cfg=None):
    _ok(_load().lk_splitk_combine(_mode(mode), _ptr(part, None, "part"), S, M, N, _ptr(y, _F32, "y"),
                                  _cfg(cfg), _stream(stream)), "lk_splitk_combine")


def lk_splitk_chunks_for(N, K, mode, M) -> int:
    """The split-K chunk count the library favours for this shape (1: the
    plain GEMV; see include/lk.h)."""
    return _load().lk_splitk_chunks_for(N, K, _mode(mode), M)


def lk_argmax_parts_max(N) -> int:
    return _load().lk_argmax_parts_max(N)


def lk_argmax_scratch_entries(N) -> int:
    return _load().lk_argmax_scratch_entries(N)


def lk_argmax(idx, M, N, logits=None, parts=None, n_parts=0, scratch=None, stream=None):
    _ok(_load().lk_argmax(_ptr(logits, _F32, "logits"), _ptr(parts, torch.int64, "parts"), n_parts, M,
                          N, _ptr(idx, torch.int32, "idx"), _ptr(scratch, torch.int64, "scratch"),
                          _stream(stream)), "lk_argmax")


def lk_q8_block_dots(wq, xq, d, xl=None, e=None, stream=None):
    N, K = wq.shape
    _ok(_load().lk_q8_block_dots(_ptr(wq, _I8, "wq"), N, K, _ptr(xq, _I8, "xq"), _ptr(xl, _I8, "xl"),
                                 _ptr(d, torch.int32, "d"), _ptr(e, torch.int32, "e"), _stream(stream)),
        "lk_q8_block_dots")


def lk_set_option(name: str, value: int):
    _ok(_load().lk_set_option(name.encode(), int(value)), f"lk_set_option({name})")


def lk_get_option(name: str) -> int:
    return _load().lk_get_option(name.encode())


def lk_device_error(reset: bool = True) -> int:
    code = ctypes.c_int(0)
    st = _load().lk_device_error(1 if reset else 0, ctypes.byref(code))
    if st not in (0, -6):
        raise LkError(st, "lk_device_error")
    return code.value


def lk_selftest_wait_timeout(limit_us: int, stream=None):
    _ok(_load().lk_selftest_wait_timeout(int(limit_us), _stream(stream)), "lk_selftest_wait_timeout")


def lk_chain_sync_bytes() -> int:
    return _load().lk_chain_sync_bytes()


def chain_op(wq, ws, x, y, gain=None, argmax_parts=None, argmax_idx=None, wait=False) -> LkChainOp:
    """Marshal one lk_chain_op from device tensors (they must outlive the chain)."""
    N, K = wq.shape
    return LkChainOp(_ptr(wq, _I8, "wq"), _ptr(ws, _WS, "ws"), N, K, _ptr(x, _F32, "x"),
                     _ptr(gain, _F32, "gain"), _ptr(y, _F32, "y"),
                     _ptr(argmax_parts, torch.int64, "argmax_parts"), _ptr(argmax_idx, torch.int32, "argmax_idx"),
                     1 if wait else 0, 0)


class Chain:
    """A host array of lk_chain_op, its device copy and a zeroed sync buffer."""

    def __init__(self, ops, device):
        self.n = len(ops)
        self.host = (LkChainOp * self.n)(*ops)
        raw = bytes(self.host)
        self.dev = torch.frombuffer(bytearray(raw), dtype=torch.uint8).to(device)
        self.sync = torch.zeros((lk_chain_sync_bytes() // 4,), dtype=torch.int32, device=device)


def lk_gemv_chain(chain: "Chain", mode, M, eps=1e-6, stream=None, cfg=None):
    _ok(_load().lk_gemv_chain(ctypes.cast(chain.host, ctypes.c_void_p), _ptr(chain.dev, None, "ops_dev"),
                              chain.n, _mode(mode), M, eps, _ptr(chain.sync, None, "sync"), _cfg(cfg),
                              _stream(stream)), "lk_gemv_chain")


def lk_trace_read(n: int):
    """Block 0's timestamps of the last traced launch (ns), as a list."""
    buf = (ctypes.c_uint64 * n)()
    _ok(_load().lk_trace_read(ctypes.cast(buf, ctypes.c_void_p), n), "lk_trace_read")
    return list(buf)


def lk_argmax_noalloc(logits, idx, stream=None):
    """Argmax of logits [M, N] into idx [M] with no caller scratch (see lk.h)."""
    M, N = logits.shape
    _ok(_load().lk_argmax_noalloc(_ptr(logits, _F32, "logits"), M, N, _ptr(idx, torch.int32, "idx"),
                                  _stream(stream)), "lk_argmax_noalloc")


# ---- the GGUF block formats other than Q8_0 ------------------------------------------

FORMATS = {"q4_0": 2, "q4_1": 3, "q5_0": 6, "q5_1": 7, "q2_k": 10, "q3_k": 11, "q4_k": 12, "q5_k": 13,
           "q6_k": 14, "iq4_nl": 20, "iq4_xs": 23, "mxfp4": 39}


def _fmt(fmt):
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def lk_format_row_bytes(fmt, K) -> int:
    return int(_load().lk_format_row_bytes(_fmt(fmt), K))


def lk_gemv_blk(fmt, w, K, mode, y, x=None, xq=None, xl=None, xs=None, M=None, stream=None, cfg=None):
    """y[M, N] = W x for a block-format matrix w (uint8 [N, row_bytes])."""
    N = w.shape[0]
    if M is None:
        M = (x if x is not None else xq).shape[0]
    if w.shape[1] != lk_format_row_bytes(fmt, K):
        raise ValueError("w rows must be lk_format_row_bytes(fmt, K) bytes")
    _ok(_load().lk_gemv_blk(_fmt(fmt), _ptr(w, torch.uint8, "w"), N, K, _mode(mode), _ptr(x, _F32, "x"),
                            _ptr(xq, _I8, "xq"), _ptr(xl, _I8, "xl"), _ptr(xs, _F32, "xs"), M, _ptr(y, _F32, "y"),
                            _cfg(cfg), _stream(stream)), "lk_gemv_blk")


def lk_dequant_blk(fmt, w, K, out, stream=None):
    """The decoded weights f32 [N, K] of a block-format matrix (test hook)."""
    _ok(_load().lk_dequant_blk(_fmt(fmt), _ptr(w, torch.uint8, "w"), w.shape[0], K, _ptr(out, _F32, "out"),
                               _stream(stream)), "lk_dequant_blk")
