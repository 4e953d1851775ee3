"""Helpers of the GPU parity tests: run the library through the C ABI on
device tensors, and run the oracle on host copies of the same inputs."""
import os

import numpy as np
import torch

import oracle
from q8_quantized_gemv_gb300 import lk

DEV = "cuda"
TOL = 1e-5  # relative to sum_k |W x| per row

# the oracle's GEMV rows over every host core: the same bits as one thread
# (tests/test_oracle.py), much less wall time at the full sizes
oracle.set_threads(os.cpu_count() or 1)


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


def gpu_gemv(wq_d, ws_d, mode, acts, M, amax=False, cfg=None):
    """acts: dict with x (Dequant) or xq/xl/xs; cfg: lk.launch_cfg(...) or
    None.  Returns (y, parts, n_parts)."""
    N = wq_d.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    parts = None
    if amax:
        parts = torch.zeros((M * lk.lk_argmax_parts_max(N),), dtype=torch.int64, device=DEV)
    n = lk.lk_gemv_q8(wq_d, ws_d, mode, y, M=M, argmax_parts=parts, cfg=cfg, **acts)
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
    return lk.lk_gemv_kernel_for(N, K, mode, M, 0, cfg=lk.launch_cfg(path=2)) == 2


# ---- whole decode tokens ------------------------------------------------------------

def run_token_capture(st):
    """One token of a DecodeStack through its per-launch path, recording after
    every GEMV launch (synchronized) host copies of what it wrote: a list with
    one dict per layer and the final logits and argmax.  Per layer: q, k, v,
    o; glu=False: gu (the fused gate/up output) and h (the down output);
    glu=True: h_in (the residual stream entering the layer, from layer 1 on),
    h_mid (after the attention residual add), gate, up, hglu (SwiGLU f32) and
    its quantized words hq/hl/hs, and down (the down output)."""
    layers, final = [], {}

    def acts_ffn():
        a = st.acts[st.F]
        return {k: host(a[k]).copy() for k in ("xq", "xl", "xs") if k in a}

    def hook(name, launch):
        r = launch()
        torch.cuda.synchronize()
        if name in ("qkv", "q"):
            layers.append({})
            if st.glu and len(layers) > 1:
                layers[-1]["h_in"] = host(st.hbuf[1]).copy()
        if name == "qkv":
            for n in ("q", "k", "v"):
                layers[-1][n] = host(st.out[n]).copy()
        elif name in ("q", "k", "v", "o") or (name == "gu" and not st.glu):
            layers[-1][name] = host(st.out[name]).copy()
        elif name == "gu":
            gu = host(st.gu_buf).copy()
            layers[-1].update(gate=gu[0], up=gu[1], hglu=host(st.hglu).copy(), h_mid=host(st.hbuf[0]).copy())
            if st.mode != 0:
                layers[-1]["hact"] = acts_ffn()
        elif name == "down":
            layers[-1]["down" if st.glu else "h"] = host(st.out["down"] if st.glu else st.h).copy()
        elif name == "lm":
            final["logits"] = host(st.logits).copy()
            if st.glu:
                final["h"] = host(st.hbuf[1]).copy()
        return r

    idx = st.run_token(hook=hook)
    torch.cuda.synchronize()
    final["idx"] = host(idx).copy()
    assert len(layers) == st.L
    return layers, final


def check_swiglu(h_gpu, g, u):
    """h within 2^-20 |g u| of the oracle's f64 SwiGLU of the same f32 g, u
    (the GPU's f32 form with expf differs by a few ulp)."""
    h_or = oracle.swiglu(g, u)
    tol = 2.0 ** -20 * np.abs(g.astype(np.float64) * u) + 1e-38
    err = np.abs(h_gpu.astype(np.float64) - h_or)
    assert np.all(err <= tol), float((err - tol).max())


def _host_w(pair):
    return host(pair[0]), host(pair[1]).view(np.uint16)


def check_token(st, layers, final):
    """Every GEMV of a captured token against the oracle on that GEMV's own
    input (the GPU's previous outputs, copied back): RMSNorm -> quantize ->
    GEMV in the oracle, then bit-exact (Int8Act, TwoPass) or within
    TOL * sum|W x| per row (Dequant).  Bit-exact steps chained from the same
    first input make the GPU token the oracle's own token.  The argmax must be
    the oracle's first index of the maximum of the GPU's logits (and, for the
    quantized modes, the logits are the oracle's bit for bit).  A projection
    the stack runs as split-K (st.splitk) is the oracle's split-K value with
    the same chunk count."""
    m = st.mode
    eps = st.eps

    def chunks(what):
        name = what.split()[-1]
        name = "qkv" if name in ("q", "k", "v") else "gu" if name == "gate/up" else name
        return st.splitk.get(name, 1)

    def step(wpair, x, gain, y_gpu, what):
        a = oracle.rmsnorm(x, host(gain), m, eps) if gain is not None else x
        wq, ws = wpair
        S = chunks(what)
        if S > 1:
            y_or = oracle.gemv_splitk(wq, ws, m, S, **oracle_acts(a, m))[0]
        else:
            y_or = oracle.gemv(wq, ws, m, **oracle_acts(a, m))
        try:
            assert_gemv_close(y_gpu, y_or, wq, ws, a, m)
        except AssertionError as e:
            raise AssertionError(f"{what}: {e}") from None

    if st.glu:
        return _check_token_glu(st, layers, final, step)
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


def _check_token_glu(st, layers, final, step):
    """check_token for the pre-norm decoder dataflow: the residual adds and
    norms bit for bit (every mode), each GEMV on its own input as in
    check_token, the SwiGLU within check_swiglu's bound, its quantized words
    the oracle quantizer's of the GPU's f32 value, and the down projection on
    those words."""
    m, eps = st.mode, st.eps

    def add_norm(x, r, gain, s_gpu, what):
        s, y = oracle.add_rmsnorm(x, r, host(gain), m, eps)
        assert np.array_equal(bits(s), bits(s_gpu)), f"{what}: residual stream"
        return y

    x_buf = host(st.x_buf)
    h_cur = x_buf
    for l, w in enumerate(st.layers):
        rec = layers[l]
        if l == 0:
            a = oracle.rmsnorm(x_buf, host(w["g_attn"]), m, eps)
        else:
            a = add_norm(layers[l - 1]["down"], h_cur, w["g_attn"], rec["h_in"], f"layer {l} attention norm")
            h_cur = rec["h_in"]
        for n in ("q", "k", "v"):
            step(_host_w(w[n]), a, None, rec[n], f"layer {l} {n}")
        step(_host_w(w["o"]), host(w["o_in"]), None, rec["o"], f"layer {l} o")
        a = add_norm(rec["o"], h_cur, w["g_mlp"], rec["h_mid"], f"layer {l} MLP norm")
        h_cur = rec["h_mid"]
        step(_host_w(w["gate"]), a, None, rec["gate"], f"layer {l} gate")
        step(_host_w(w["up"]), a, None, rec["up"], f"layer {l} up")
        check_swiglu(rec["hglu"], rec["gate"], rec["up"])
        if m != oracle.DEQUANT:
            hi, lo, sc = oracle.quantize(rec["hglu"], m)
            q = rec["hact"]
            assert np.array_equal(q["xq"], hi) and np.array_equal(bits(q["xs"]), bits(sc)), f"layer {l} h words"
            if m == oracle.TWOPASS:
                assert np.array_equal(q["xl"], lo), f"layer {l} h low words"
        step(_host_w(w["down"]), rec["hglu"], None, rec["down"], f"layer {l} down")
    a = add_norm(layers[-1]["down"], h_cur, st.g_final, final["h"], "final norm")
    step(_host_w(st.lm), a, None, final["logits"], "lm-head")
    assert final["idx"].tolist() == [oracle.argmax(final["logits"][t]) for t in range(st.B)]
