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


# ---- whole decode tokens ------------------------------------------------------------

def run_token_capture(st):
    """One token of a DecodeStack through its per-launch path, recording after
    every GEMV launch (synchronized) host copies of what it wrote: a list with
    one dict per layer (q, k, v, o, gu, h) and the final logits and argmax."""
    layers, final = [], {}

    def hook(name, launch):
        r = launch()
        torch.cuda.synchronize()
        if name in ("qkv", "q"):
            layers.append({})
        if name == "qkv":
            for n in ("q", "k", "v"):
                layers[-1][n] = host(st.out[n]).copy()
        elif name in ("q", "k", "v", "o", "gu"):
            layers[-1][name] = host(st.out[name]).copy()
        elif name == "down":
            layers[-1]["h"] = host(st.h).copy()
        elif name == "lm":
            final["logits"] = host(st.logits).copy()
        return r

    idx = st.run_token(hook=hook)
    torch.cuda.synchronize()
    final["idx"] = host(idx).copy()
    assert len(layers) == st.L and all(len(r) == 6 for r in layers)
    return layers, final


def _host_w(pair):
    return host(pair[0]), host(pair[1]).view(np.uint16)


def check_token(st, layers, final):
    """Every GEMV of a captured token against the oracle on that GEMV's own
    input (the GPU's previous outputs, copied back): RMSNorm -> quantize ->
    GEMV in the oracle, then bit-exact (Int8Act, TwoPass) or within
    TOL * sum|W x| per row (Dequant).  Bit-exact steps chained from the same
    first input make the GPU token the oracle's own token.  The argmax must be
    the oracle's first index of the maximum of the GPU's logits (and, for the
    quantized modes, the logits are the oracle's bit for bit)."""
    m = st.mode
    eps = st.eps

    def step(wpair, x, gain, y_gpu, what):
        a = oracle.rmsnorm(x, host(gain), m, eps) if gain is not None else x
        wq, ws = wpair
        y_or = oracle.gemv(wq, ws, m, **oracle_acts(a, m))
        try:
            assert_gemv_close(y_gpu, y_or, wq, ws, a, m)
        except AssertionError as e:
            raise AssertionError(f"{what}: {e}") from None

    x = host(st.x_buf)
    for l, w in enumerate(st.layers):
        rec = layers[l]
        for n in ("q", "k", "v"):
            step(_host_w(w[n]), x, w["g_attn"], rec[n], f"layer {l} {n}")
        step(_host_w(w["o"]), host(w["o_in"]), None, rec["o"], f"layer {l} o")
        step(_host_w(w["gu"]), rec["o"], w["g_mlp"], rec["gu"], f"layer {l} gate/up")
        step(_host_w(w["down"]), host(w["d_in"]), None, rec["h"], f"layer {l} down")
        x = rec["h"]
    step(_host_w(st.lm), x, st.g_final, final["logits"], "lm-head")
    assert final["idx"].tolist() == [oracle.argmax(final["logits"][t]) for t in range(st.B)]
