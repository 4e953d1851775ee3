"""Pins of the CPU oracle to facts fixed outside itself: hand-worked values
(tests/golden), closed forms, exact rational brute force on tiny inputs,
invariants, and library routines for the special cases that reduce to one.
No GPU."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from casebuild import (MODES, block_case, f16_bits, lo_case, order_records,
                       quantizer_records)
from q8_quantized_gemv_gb300 import synth

DQ, I8, TP = oracle.DEQUANT, oracle.INT8ACT, oracle.TWOPASS
U32 = 2.0 ** -24
# Int8Act: groups with max|v| below 127 * 2^-126 (a/127 not a normal float)
# are quantized as the all-zero group (the reading for tiny groups)
INT8ACT_MIN_MAX = 127.0 * 2.0 ** -126


# ---- f16 scales -----------------------------------------------------------

def test_half_to_float_every_pattern_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_float(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ---- quantizer ----------------------------------------------------------

@pytest.mark.parametrize("rec", quantizer_records(), ids=lambda r: f"{r['name']}-{r['mode']}")
def test_quantizer_hand_worked(rec):
    hi, lo, s = oracle.quantize(rec["x"], rec["mode"])
    assert s.view(np.uint32)[0, 0] == rec["s_bits"]
    n = rec["n"]
    assert hi[0, :n].tolist() == rec["hi"]
    assert not hi[0, n:].any()
    if rec["lo"] is not None:
        assert lo[0, :n].tolist() == rec["lo"]
        assert not lo[0, n:].any()


def _groups(seed, n=400):
    r = np.random.default_rng(seed)
    g = r.standard_normal((n, 32)).astype(np.float32)
    g *= (2.0 ** r.integers(-20, 20, size=(n, 1))).astype(np.float32)
    g[r.random((n, 32)) < 0.01] *= 20
    g[::17, 5] = 0.0          # zeros inside groups
    g[::29, :] = 0.0          # all-zero groups
    g[::31, :] = np.float32(0.5)  # all equal
    # groups whose largest magnitude is tiny: subnormal, and straddling the
    # Int8Act threshold 127 * 2^-126 below which a group is quantized as zero
    g[3::37, :] = (g[3::37, :] * np.float32(2.0 ** -140)).astype(np.float32)
    g[7::41, :] = (g[7::41, :] / np.abs(g[7::41, :]).max(axis=1, keepdims=True)
                   * np.float32(INT8ACT_MIN_MAX) * np.float32(1.5)).astype(np.float32)
    g[11::43, :] = (g[11::43, :] / np.abs(g[11::43, :]).max(axis=1, keepdims=True)
                    * np.float32(INT8ACT_MIN_MAX) * np.float32(0.75)).astype(np.float32)
    return g.reshape(1, -1)


@pytest.mark.parametrize("mode", [I8, TP])
def test_quantizer_invariants(mode):
    v = _groups(7)
    hi, lo, s = oracle.quantize(v, mode)
    K = v.shape[1]
    vg = v.reshape(-1, 32).astype(np.float64)
    a = np.abs(v.reshape(-1, 32)).max(axis=1)
    # the scale: max|v|/127 as one IEEE f32 division (numpy), with the per-mode floor
    if mode == I8:
        want = np.where(a >= INT8ACT_MIN_MAX, a / np.float32(127.0), np.float32(1.0)).astype(np.float32)
        assert (a < INT8ACT_MIN_MAX).sum() > (a == 0).sum()  # tiny groups are present
    else:
        want = (np.maximum(a, np.float32(1e-30)) / np.float32(127.0)).astype(np.float32)
    assert np.array_equal(s[0].view(np.uint32), want.view(np.uint32))
    h = hi.reshape(-1, 32).astype(np.float64)
    sc = s.reshape(-1, 1).astype(np.float64)
    assert h.min() >= -127 and h.max() <= 127
    if mode == I8:
        assert np.all(np.abs(vg - h * sc) <= sc * (0.5 + 1e-5))
    else:
        l = lo.reshape(-1, 32).astype(np.float64)
        resid = np.abs(vg - h * sc - l * sc / 128.0)
        assert np.all(resid <= sc / 256.0 * (1 + 1e-4) + 1e-45)
        # the low word is never the bound itself: |lo| <= 64 + 1
        assert np.abs(l).max() <= 65
    # sign symmetry: q(-v) = -q(v), same scale
    hi2, lo2, s2 = oracle.quantize(-v, mode)
    assert np.array_equal(hi2, -hi) and np.array_equal(s2, s)
    if mode == TP:
        assert np.array_equal(lo2, -lo)
    # power-of-two scaling: words unchanged, scale scaled (nonzero, in-range groups)
    keep = (a > 1e-20) & (a < 1e20)
    for k in (-3, 5):
        hi3, lo3, s3 = oracle.quantize(v * np.float32(2.0 ** k), mode)
        kk = np.repeat(keep, 32)
        assert np.array_equal(hi3[0, kk], hi[0, kk])
        assert np.array_equal(s3[0, keep], s[0, keep] * np.float32(2.0 ** k))
        if mode == TP:
            assert np.array_equal(lo3[0, kk], lo[0, kk])


def test_quantizer_rounding_matches_rint():
    # every value of a group with max 127 has s = 1, so hi = rint(v) (ties to even)
    r = np.random.default_rng(3)
    v = np.round(r.uniform(-126, 126, size=(1, 32 * 64)) * 4) / 4  # many exact .5 / .25
    v = v.astype(np.float32)
    v[0, ::32] = 127.0
    hi, _, s = oracle.quantize(v, I8)
    assert np.all(s == 1.0)
    assert np.array_equal(hi[0].astype(np.float32), np.rint(v[0]))


# ---- block dots ------------------------------------------------------------

def test_block_dots_brute_force():
    wq, _ = synth.q8_matrix(5, 320, 11)
    x = synth.activation(1, 320, 12, outliers=True)
    hi, lo, _ = oracle.quantize(x, TP)
    d, e = oracle.block_dots(wq, hi[0], lo[0])
    W = wq.astype(np.int64).reshape(5, 10, 32)
    assert np.array_equal(d, np.einsum("obk,bk->ob", W, hi[0].astype(np.int64).reshape(10, 32)))
    assert np.array_equal(e, np.einsum("obk,bk->ob", W, lo[0].astype(np.int64).reshape(10, 32)))


# ---- GEMV: hand-worked orders ---------------------------------------------

@pytest.mark.parametrize("name", ["gemv_sum4", "gemv_chain"])
@pytest.mark.parametrize("mode", ["dequant", "int8act", "twopass"])
def test_gemv_order_examples(name, mode):
    rec = order_records()[name]
    wq, ws, x = block_case(int(rec["K"]), rec["blocks"])
    m = MODES[mode]
    if m == DQ:
        y = oracle.gemv(wq, ws, m, x=x)
    else:
        hi, lo, s = oracle.quantize(x, m)
        assert np.all(s == 1.0) and not lo.any()
        y = oracle.gemv(wq, ws, m, hi=hi, lo=lo, s=s)
    assert y[0, 0] == np.float32(rec[f"y_{mode}"])


@pytest.mark.parametrize("mode", ["dequant", "int8act", "twopass"])
def test_gemv_low_word_weight(mode):
    rec = order_records()["gemv_lo"]
    wq, ws, x = lo_case(rec)
    m = MODES[mode]
    if m == DQ:
        y = oracle.gemv(wq, ws, m, x=x)
    else:
        hi, lo, s = oracle.quantize(x, m)
        y = oracle.gemv(wq, ws, m, hi=hi, lo=lo, s=s)
    assert y[0, 0] == np.float32(rec[f"y_{mode}"])


@pytest.mark.parametrize("mode", ["dequant", "int8act", "twopass"])
def test_splitk_combine_example(mode):
    rec = order_records()["splitk_combine"]
    K, S = int(rec["K"]), int(rec["S"])
    wq, ws, x = block_case(K, rec["blocks"])
    m = MODES[mode]
    kw = dict(x=x) if m == DQ else dict(zip(("hi", "lo", "s"), oracle.quantize(x, m)))
    y_plain = oracle.gemv(wq, ws, m, **kw)
    y_split, chunks = oracle.gemv_splitk(wq, ws, m, S, **kw)
    assert y_plain[0, 0] == np.float32(rec[f"y_plain_{mode}"])
    assert y_split[0, 0] == np.float32(rec[f"y_split_{mode}"])
    assert [oracle.splitk_bound(K // 32, S, c) for c in range(S + 1)] == [0, 4, 8, 12]


def test_splitk_bounds():
    # balanced floor split over four-block groups; the last chunk ends at nb
    assert [oracle.splitk_bound(160, 8, c) for c in range(9)] == list(range(0, 161, 20))
    assert [oracle.splitk_bound(800, 8, c) for c in range(9)] == list(range(0, 801, 100))
    assert [oracle.splitk_bound(10, 4, c) for c in range(5)] == [0, 0, 4, 4, 10]
    assert [oracle.splitk_bound(7, 2, c) for c in range(3)] == [0, 0, 7]
    assert [oracle.splitk_bound(128, 1, c) for c in range(2)] == [0, 128]


# ---- GEMV: exact rational brute force on tiny inputs -----------------------

def _frac(v):
    return Fraction(float(v))


@pytest.mark.parametrize("mode", [I8, TP])
@pytest.mark.parametrize("K", [32, 96, 512, 1056])
def test_gemv_quantized_within_error_bound(mode, K):
    N = 4
    wq, ws = synth.q8_matrix(N, K, 100 + K)
    x = synth.activation(1, K, 200 + K, outliers=True)
    hi, lo, s = oracle.quantize(x, mode)
    y = oracle.gemv(wq, ws, mode, hi=hi, lo=lo, s=s)
    wsf = f16_bits_to_f64(ws)
    nb = K // 32
    d, e = oracle.block_dots(wq, hi[0], lo[0] if mode == TP else None)
    for o in range(N):
        exact = Fraction(0)
        mag = Fraction(0)
        for b in range(nb):
            t = _frac(wsf[o, b]) * _frac(s[0, b]) * (Fraction(int(d[o, b])) +
                                                    (Fraction(int(e[o, b]), 128) if mode == TP else 0))
            exact += t
            mag += abs(t)
        steps = nb // 4 + 8
        err = abs(_frac(y[0, o]) - exact)
        assert err <= Fraction(steps) * Fraction(U32) * mag * Fraction(11, 10), (o, float(err), float(mag))


def f16_bits_to_f64(ws):
    return ws.view(np.float16).astype(np.float64)


@pytest.mark.parametrize("K", [32, 160, 1024])
def test_gemv_dequant_within_f64_bound(K):
    N = 3
    wq, ws = synth.q8_matrix(N, K, 300 + K)
    x = synth.activation(1, K, 400 + K, outliers=True)
    y = oracle.gemv(wq, ws, DQ, x=x)
    W = wq.astype(np.float64) * np.repeat(f16_bits_to_f64(ws), 32, axis=1)
    for o in range(N):
        exact = sum((_frac(W[o, k]) * _frac(x[0, k]) for k in range(K)), Fraction(0))
        # f64 sum (K roundings of 2^-53) then one f32 rounding
        mag = sum(abs(W[o, k] * float(x[0, k])) for k in range(K))
        bound = abs(float(exact)) * U32 + K * 2.0 ** -53 * mag * 1.1 + 1e-300
        assert abs(float(y[0, o]) - float(exact)) <= bound


def test_gemv_special_cases():
    K, N = 256, 6
    wq, ws = synth.q8_matrix(N, K, 5)
    # one-hot activation in Dequant gives column k of W exactly
    x = np.zeros((1, K), np.float32)
    x[0, 77] = 1.0
    y = oracle.gemv(wq, ws, DQ, x=x)
    col = wq[:, 77].astype(np.float32) * ws[:, 77 // 32].view(np.float16).astype(np.float32)
    assert np.array_equal(y[0], col)
    # identity weights with unit scales give back the dequantized activation
    eye = np.eye(K, dtype=np.int8)
    ones = f16_bits(np.ones((K, K // 32), np.float32))
    xa = synth.activation(1, K, 6)
    for m in (I8, TP):
        hi, lo, s = oracle.quantize(xa, m)
        y = oracle.gemv(eye, ones, m, hi=hi, lo=lo, s=s)
        deq = hi[0].astype(np.float64) * np.repeat(s[0], 32)
        if m == TP:
            deq = deq + lo[0].astype(np.float64) * np.repeat(s[0], 32) / 128
        assert np.allclose(y[0], deq, rtol=2 ** -22, atol=0)
    # equal rows give bitwise equal outputs; batch column t equals the 1-row result
    wq2 = np.repeat(wq[:1], 4, axis=0)
    ws2 = np.repeat(ws[:1], 4, axis=0)
    xb = synth.activation(3, K, 8)
    for m in (I8, TP):
        hi, lo, s = oracle.quantize(xb, m)
        yb = oracle.gemv(wq2, ws2, m, hi=hi, lo=lo, s=s)
        assert np.all(yb == yb[:, :1])
        for t in range(3):
            y1 = oracle.gemv(wq2, ws2, m, hi=hi[t:t + 1], lo=lo[t:t + 1], s=s[t:t + 1])
            assert np.array_equal(y1[0].view(np.uint32), yb[t].view(np.uint32))


def test_splitk_s1_is_plain_and_chunks_sum():
    K, N = 1024, 5
    wq, ws = synth.q8_matrix(N, K, 21)
    x = synth.activation(1, K, 22, outliers=True)
    for m in (I8, TP):
        hi, lo, s = oracle.quantize(x, m)
        y = oracle.gemv(wq, ws, m, hi=hi, lo=lo, s=s)
        y1, _ = oracle.gemv_splitk(wq, ws, m, 1, hi=hi, lo=lo, s=s)
        assert np.array_equal(y1, y)
        for S in (2, 3, 8):
            yS, ch = oracle.gemv_splitk(wq, ws, m, S, hi=hi, lo=lo, s=s)
            acc = np.zeros_like(yS)
            for c in range(S):
                acc = (acc + ch[c]).astype(np.float32)
            assert np.array_equal(acc, yS)
            assert np.allclose(yS, y, rtol=1e-5, atol=1e-3)
    y = oracle.gemv(wq, ws, DQ, x=x)
    for S in (1, 4):
        yS, ch = oracle.gemv_splitk(wq, ws, DQ, S, x=x)
        assert ch.dtype == np.float64
        assert np.allclose(yS, y, rtol=1e-6, atol=0)


def test_absdot_one_hot():
    K, N = 64, 3
    wq, ws = synth.q8_matrix(N, K, 31)
    x = np.zeros((1, K), np.float32)
    x[0, 40] = -2.0
    a = oracle.absdot(wq, ws, x)
    want = np.abs(wq[:, 40].astype(np.float64) * ws[:, 1].view(np.float16).astype(np.float64) * 2.0)
    assert np.array_equal(a[0], want)


# ---- RMSNorm ------------------------------------------------------------------

@pytest.mark.parametrize("name", ["sumsq_tree_k32", "sumsq_tree_k1024", "sumsq_tree_k2048"])
def test_sumsq_tree_order(name):
    rec = order_records()[name]
    K = int(rec["K"])
    v = np.zeros(K, np.float32)
    for item in rec["nonzero"].split():
        i, val = item.split(":")
        v[int(i)] = float(val)
    assert oracle.sumsq(v, I8) == np.float32(rec["sumsq_f32"])
    # in f64 the same inputs sum exactly
    assert oracle.sumsq(v, DQ) == float(np.sum(v.astype(np.float64) ** 2))


def test_norm_threads():
    assert [oracle.norm_threads(k) for k in (32, 33, 1000, 1024, 4096, 25600)] == \
        [32, 64, 1000 + 24, 1024, 1024, 1024]


@pytest.mark.parametrize("K", [32, 96, 4096])
def test_rmsnorm_constant_row_closed_form(K):
    # constant c = 2^-10: every square is 2^-20 exactly, so any order sums to
    # K * 2^-20 exactly and y = c / sqrt(2^-20 + eps) * g (eps comparable to
    # the mean, so a dropped or misplaced eps fails)
    c = np.float32(2.0 ** -10)
    v = np.full((1, K), c, np.float32)
    g = synth.norm_gain(K, 9)
    y = oracle.rmsnorm(v, g, I8)
    den = np.sqrt(np.float32(2.0 ** -20) + np.float32(1e-6), dtype=np.float32)
    assert np.array_equal(y[0], (c / den * g).astype(np.float32))
    yd = oracle.rmsnorm(v, g, DQ)
    dend = np.sqrt(2.0 ** -20 + float(np.float32(1e-6)))
    assert np.array_equal(yd[0], (float(c) / dend * g.astype(np.float64)).astype(np.float32))


@pytest.mark.parametrize("mode", [DQ, I8])
@pytest.mark.parametrize("K", [64, 1056, 5120])
def test_rmsnorm_brute_force(mode, K):
    x = synth.activation(2, K, 40 + K, outliers=True)
    g = synth.norm_gain(K, 41)
    y = oracle.rmsnorm(x, g, mode)
    for t in range(2):
        xt = x[t].astype(np.float64)
        exact = xt / np.sqrt(np.sum(xt * xt) / K + float(np.float32(1e-6))) * g.astype(np.float64)
        rel = np.abs(y[t] - exact) / np.maximum(np.abs(exact), 1e-30)
        # f32: a sum of K squares (<= ~log2 depth + K/1024 chain), a divide, a
        # sqrt, a divide and a multiply; f64: one final rounding to f32
        tol = (2 + K / 1024 + 16) * U32 if mode == I8 else 1.01 * U32 / 2 * 2
        assert rel.max() <= tol, rel.max()


# ---- argmax -----------------------------------------------------------------

def test_argmax_first_of_equal_maxima():
    r = np.random.default_rng(5)
    for n in (1, 2, 7, 2048, 2049, 151936):
        v = r.standard_normal(n).astype(np.float32)
        assert oracle.argmax(v) == int(np.argmax(v))
        if n > 10:
            idx = sorted(r.choice(n, 3, replace=False))
            v[idx] = v.max() + 1
            assert oracle.argmax(v) == idx[0] == int(np.argmax(v))
    v = np.array([-1.0, -0.0, 0.0, -0.0], np.float32)
    assert oracle.argmax(v) == 1
    assert oracle.argmax(np.zeros(100, np.float32)) == 0
    assert oracle.argmax(np.full(5, -np.inf, np.float32)) == 0


# ---- residual add + RMSNorm ------------------------------------------------

@pytest.mark.parametrize("mode", [DQ, I8])
def test_add_rmsnorm_sum_is_the_f32_sum(mode):
    r = np.random.default_rng(21)
    x = r.standard_normal((2, 1024)).astype(np.float32)
    res = (r.standard_normal((2, 1024)) * 3).astype(np.float32)
    g = synth.norm_gain(1024, 22)
    s, y = oracle.add_rmsnorm(x, res, g, mode)
    assert np.array_equal(s.view(np.uint32), (x + res).view(np.uint32))  # numpy's IEEE f32 add
    # the norm sees the sum: within a few ulp of the long-double definition
    v = s.astype(np.longdouble)
    den = np.sqrt((v * v).sum(axis=1, keepdims=True) / 1024 + np.longdouble(np.float32(1e-6)))
    want = v / den * g.astype(np.longdouble)
    assert np.all(np.abs(y - want) <= 4 * np.spacing(np.abs(want).astype(np.float32)))


@pytest.mark.parametrize("mode", [DQ, I8])
@pytest.mark.parametrize("K", [32, 1024, 4096])
def test_add_rmsnorm_constant_sum_closed_form(mode, K):
    # x + r = c exactly in every element (x = c - r with few significant bits):
    # y_i = g_i c / sqrt(c^2 + eps), which a norm of x alone (or of r) misses
    r = np.random.default_rng(K)
    res = r.integers(-64, 64, size=(1, K)).astype(np.float32) / np.float32(8)
    c = np.float32(0.375)
    x = (c - res).astype(np.float32)
    assert np.all(x + res == c)
    g = synth.norm_gain(K, 23)
    s, y = oracle.add_rmsnorm(x, res, g, mode)
    assert np.all(s == c)
    eps = np.float32(1e-6)
    want = g.astype(np.float64) * float(c) / np.sqrt(float(c) ** 2 + float(eps))
    assert np.allclose(y[0], want, rtol=4 * U32, atol=0)


# ---- SwiGLU ---------------------------------------------------------------------

def test_swiglu_closed_forms():
    u = np.array([1.0, -2.0, 0.5, 3.0, 96.0, -0.25], np.float32)
    # silu(0) = 0; for g tiny the slope is 1/2: h = g u / 2 exactly
    assert not oracle.swiglu(np.zeros_like(u), u).any()
    t = np.float32(2.0 ** -30)
    assert np.array_equal(oracle.swiglu(np.full_like(u, t), u), (t * u / 2).astype(np.float32))
    # sigma(50) = 1 - 2e-22: h = 50 u (representable) exactly; sigma(-50) ~ 2e-22
    assert np.array_equal(oracle.swiglu(np.full_like(u, 50.0), u), (50 * u).astype(np.float32))
    h = oracle.swiglu(np.full_like(u, -50.0), u)
    assert np.allclose(h, -50.0 * np.exp(-50.0) * u.astype(np.float64), rtol=1e-6)
    # far beyond the f64 range of e^-g: a signed zero for g -> -inf, g u for g -> +inf
    assert not oracle.swiglu(np.full_like(u, -1000.0), u).any()
    assert np.array_equal(oracle.swiglu(np.full_like(u, 1000.0), u), (1000 * u).astype(np.float32))


def test_swiglu_identities():
    r = np.random.default_rng(31)
    g = (r.standard_normal(4096) * 4).astype(np.float32)
    u = r.standard_normal(4096).astype(np.float32)
    h = oracle.swiglu(g, u).astype(np.float64)
    # silu(g) - silu(-g) = g (sigma(g) + sigma(-g) = 1): catches e^g for e^-g,
    # a dropped sign, or the gate and up operands exchanged
    d = h - oracle.swiglu(-g, u).astype(np.float64)
    gu = g.astype(np.float64) * u
    assert np.all(np.abs(d - gu) <= 2 * np.spacing(np.abs(gu).astype(np.float32)) + 1e-38)
    # linear in u: doubling u doubles h exactly
    assert np.array_equal(oracle.swiglu(g, 2 * u), 2 * oracle.swiglu(g, u))
    # |silu(g)| <= |g| and silu(g) >= min over g (about -0.2785)
    s1 = oracle.swiglu(g, np.ones_like(g)).astype(np.float64)
    assert np.all(np.abs(s1) <= np.abs(g) + 1e-30) and s1.min() > -0.2785


def test_glu_composition():
    # gate and up are two GEMVs of one activation; h their SwiGLU, then quantized
    wg, wsg = synth.q8_matrix(64, 256, 41)
    wu, wsu = synth.q8_matrix(64, 256, 42)
    x = synth.activation(2, 256, 43, outliers=True)
    for mode in (DQ, I8, TP):
        if mode == DQ:
            acts = dict(x=x)
        else:
            hi, lo, s = oracle.quantize(x, mode)
            acts = dict(hi=hi, lo=lo, s=s)
        g, u, h, q = oracle.glu(wg, wsg, wu, wsu, mode, **acts)
        assert np.array_equal(g, oracle.gemv(wg, wsg, mode, **acts))
        assert np.array_equal(u, oracle.gemv(wu, wsu, mode, **acts))
        assert np.array_equal(h, oracle.swiglu(g, u))
        if mode == DQ:
            assert q is None
        else:
            for a, b in zip(q, oracle.quantize(h, mode)):
                assert np.array_equal(a, b)


def test_threads_give_the_same_bits():
    """The all-cores oracle (rows spread over host threads) is bit-identical
    to the single-threaded one, in every mode and in split-K."""
    wq, ws = synth.q8_matrix(301, 512, 51)
    x = synth.activation(2, 512, 52, outliers=True)
    outs = {}
    prev = oracle.get_threads()
    for n in (1, 4):
        assert oracle.set_threads(n) == n
        try:
            r = []
            for mode in (DQ, I8, TP):
                a = dict(x=x) if mode == DQ else dict(zip(("hi", "lo", "s"), oracle.quantize(x, mode)))
                r.append(oracle.gemv(wq, ws, mode, **a))
                r.extend(oracle.gemv_splitk(wq, ws, mode, 3, **a))
            r.append(oracle.absdot(wq, ws, x))
        finally:
            oracle.set_threads(prev)
        outs[n] = r
    for a, b in zip(outs[1], outs[4]):
        assert a.dtype == b.dtype and np.array_equal(a.view(np.uint8), b.view(np.uint8))
