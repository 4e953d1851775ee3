"""The fused neighbouring steps of a decoder layer against the oracle:
residual add -> RMSNorm -> quantize (lk_add_rmsnorm_quant) bit for bit, and
SwiGLU -> quantize (lk_swiglu_quant): the f32 gated value within a few ulp
of the oracle's f64 definition (the GPU evaluates it in f32 with expf, the
pages' form), and its quantized words and scales exactly the oracle's
quantizer applied to that f32 value (the integer decision taken on the same
float on both sides)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpuhelp import DEV, act_buffers, assert_gemv_close, bits, check_swiglu, host, to_dev  # noqa: E402
from q8_quantized_gemv_gb300 import build, lk, synth  # noqa: E402

pytestmark = pytest.mark.gpu

DQ, I8, TP = 0, 1, 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield


# K: the 256-thread split kernel (multiples of 1024 up to 8192), the vt-thread
# split kernel (K < 1024, or K = 1024 u with u <= 8 handled above), the
# one-block-per-row kernel (longer rows), and ragged group counts
@pytest.mark.parametrize("K", [32, 96, 1024, 4096, 5120, 12288, 25600])
@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("mode", [DQ, I8, TP])
def test_add_rmsnorm_quant_bitexact(mode, M, K):
    x = synth.activation(M, K, synth.SEED_BASE + 500 + K, outliers=True)
    r = (3 * synth.activation(M, K, synth.SEED_BASE + 501 + K)).astype(np.float32)
    g = synth.norm_gain(K, synth.SEED_BASE + 502)
    s_or, y_or = oracle.add_rmsnorm(x, r, g, mode)
    s = torch.full((M, K), float("nan"), dtype=torch.float32, device=DEV)
    xn = torch.full((M, K), float("nan"), dtype=torch.float32, device=DEV)
    xq, xl, xs = act_buffers(M, K, mode)
    lk.lk_add_rmsnorm_quant(to_dev(x), to_dev(r), to_dev(g), mode, 1e-6, s=s, xn=xn,
                            xq=xq if mode else None, xl=xl, xs=xs if mode else None)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(s)), bits(s_or))
    assert np.array_equal(bits(host(xn)), bits(y_or))
    if mode:
        hi, lo, sc = oracle.quantize(y_or, mode)
        assert np.array_equal(host(xq), hi) and np.array_equal(bits(host(xs)), bits(sc))
        if mode == TP:
            assert np.array_equal(host(xl), lo)
    # without the optional outputs the quantized words are the same
    if mode:
        xq2, xl2, xs2 = act_buffers(M, K, mode)
        lk.lk_add_rmsnorm_quant(to_dev(x), to_dev(r), to_dev(g), mode, 1e-6, xq=xq2, xl=xl2, xs=xs2)
        torch.cuda.synchronize()
        assert torch.equal(xq2, xq) and torch.equal(xs2.view(torch.int32), xs.view(torch.int32))


def test_add_rmsnorm_matches_norm_of_the_sum():
    """The fused step is lk_rmsnorm_quant of x + r, bit for bit."""
    M, K = 2, 4096
    x = to_dev(synth.activation(M, K, 7, outliers=True))
    r = to_dev(synth.activation(M, K, 8))
    g = to_dev(synth.norm_gain(K, 9))
    for mode in (I8, TP):
        a = act_buffers(M, K, mode)
        b = act_buffers(M, K, mode)
        lk.lk_add_rmsnorm_quant(x, r, g, mode, 1e-6, xq=a[0], xl=a[1], xs=a[2])
        lk.lk_rmsnorm_quant(x + r, g, mode, 1e-6, None, b[0], b[1], b[2])
        torch.cuda.synchronize()
        for u, v in zip(a, b):
            if u is not None:
                assert torch.equal(u.view(torch.int8) if u.dtype == torch.int8 else u.view(torch.int32),
                                   v.view(torch.int8) if v.dtype == torch.int8 else v.view(torch.int32))


def _swiglu_inputs(M, F, seed):
    r = np.random.default_rng(seed)
    g = (r.standard_normal((M, F)) * 3).astype(np.float32)
    u = r.standard_normal((M, F)).astype(np.float32)
    # planted: silu's zero, saturation both ways, the f32 expf overflow (g < -88.7)
    special = np.array([0.0, -0.0, 50.0, -50.0, 100.0, -100.0, 1e-30, -1e-30], np.float32)
    g[0, :special.size] = special
    return g, u


@pytest.mark.parametrize("F", [32, 1536, 12288])
@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("mode", [DQ, I8, TP])
def test_swiglu_quant(mode, M, F):
    g, u = _swiglu_inputs(M, F, synth.SEED_BASE + 600 + F)
    # the two halves of one fused gate/up output [M][2F]
    gu = torch.from_numpy(np.concatenate([g, u], axis=1)).to(DEV)
    h = torch.full((M, F), float("nan"), dtype=torch.float32, device=DEV)
    hq, hl, hs = act_buffers(M, F, mode)
    lk.lk_swiglu_quant(gu[:, :F], gu[:, F:], mode, h=h, hq=hq if mode else None, hl=hl, hs=hs if mode else None)
    torch.cuda.synchronize()
    hh = host(h)
    check_swiglu(hh, g, u)
    if mode:
        hi, lo, sc = oracle.quantize(hh, mode)
        assert np.array_equal(host(hq), hi) and np.array_equal(bits(host(hs)), bits(sc))
        if mode == TP:
            assert np.array_equal(host(hl), lo)
        # separate gate and up rows (pitch F) and no f32 output: the same words
        hq2, hl2, hs2 = act_buffers(M, F, mode)
        lk.lk_swiglu_quant(to_dev(g), to_dev(u), mode, hq=hq2, hl=hl2, hs=hs2)
        torch.cuda.synchronize()
        assert torch.equal(hq2, hq) and torch.equal(hs2.view(torch.int32), hs.view(torch.int32))
        if mode == TP:
            assert torch.equal(hl2, hl)


def _glu_case(F, K, M, mode, seed):
    wg, wsg = synth.q8_matrix(F, K, seed)
    wu, wsu = synth.q8_matrix(F, K, seed + 1)
    x = synth.activation(M, K, seed + 2, outliers=True)
    if mode == DQ:
        acts_or, acts = dict(x=x), dict(x=to_dev(x))
    else:
        hi, lo, s = oracle.quantize(x, mode)
        acts_or = dict(hi=hi, lo=lo, s=s)
        acts = dict(xq=to_dev(hi), xs=to_dev(s), xl=to_dev(lo) if mode == TP else None)
    return (wg, wsg, wu, wsu), acts_or, acts, x


# F: one group, a group count that leaves blocks with partial groups, the
# decoder's 12288; K: the ring kernel (K % 256 == 0) and the direct kernel
@pytest.mark.parametrize("F,K", [(32, 256), (96, 512), (1056, 1024), (12288, 4096), (224, 1056)])
@pytest.mark.parametrize("M", [1, 3])
@pytest.mark.parametrize("mode", [DQ, I8, TP])
@pytest.mark.parametrize("with_cnt", [True, False])
def test_gemv_q8_glu(mode, M, F, K, with_cnt):
    (wg, wsg, wu, wsu), acts_or, acts, x = _glu_case(F, K, M, mode, synth.SEED_BASE + 700 + F + K)
    g_or, u_or, _, _ = oracle.glu(wg, wsg, wu, wsu, mode, **acts_or)
    d = [to_dev(a) for a in (wg, wsg, wu, wsu)]
    cnt = torch.zeros((F // 32,), dtype=torch.int32, device=DEV) if with_cnt else None
    for call in range(2):  # twice: the counters are left ready for the next call
        gu = torch.full((2, M, F), float("nan"), dtype=torch.float32, device=DEV)
        h = torch.full((M, F), float("nan"), dtype=torch.float32, device=DEV)
        hq, hl, hs = act_buffers(M, F, mode)
        lk.lk_gemv_q8_glu(*d, mode, gu, h=h, hq=hq if mode else None, hl=hl, hs=hs if mode else None, cnt=cnt,
                          **acts)
        torch.cuda.synchronize()
        assert lk.lk_device_error(reset=True) == 0
        guh = host(gu)
        # the GEMV part: each matrix exactly lk_gemv_q8's value (bit-exact
        # in the quantized modes, the tolerance under Dequant)
        assert_gemv_close(guh[0], g_or, wg, wsg, x, mode)
        assert_gemv_close(guh[1], u_or, wu, wsu, x, mode)
        # the SwiGLU of the GPU's gate/up values, then its quantizer
        hh = host(h)
        check_swiglu(hh, guh[0], guh[1])
        if mode:
            hi, lo, sc = oracle.quantize(hh, mode)
            assert np.array_equal(host(hq), hi) and np.array_equal(bits(host(hs)), bits(sc))
            if mode == TP:
                assert np.array_equal(host(hl), lo)
        if with_cnt:
            assert not host(cnt).any()


def test_gemv_q8_glu_equals_its_two_launch_form():
    """The one-launch gated pair (ring kernel, M = 1) gives the bits of the
    grouped GEMVs followed by lk_swiglu_quant."""
    F, K = 12288, 4096
    for mode in (I8, TP):
        (wg, wsg, wu, wsu), _, acts, _ = _glu_case(F, K, 1, mode, 77)
        d = [to_dev(a) for a in (wg, wsg, wu, wsu)]
        outs = []
        for cnt in (torch.zeros((F // 32,), dtype=torch.int32, device=DEV), None):
            gu = torch.empty((2, 1, F), dtype=torch.float32, device=DEV)
            h = torch.empty((1, F), dtype=torch.float32, device=DEV)
            hq, hl, hs = act_buffers(1, F, mode)
            lk.lk_gemv_q8_glu(*d, mode, gu, h=h, hq=hq, hl=hl, hs=hs, cnt=cnt, **acts)
            torch.cuda.synchronize()
            outs.append([host(t).copy() for t in (gu, h, hq, hs) + ((hl,) if mode == TP else ())])
        for a, b in zip(*outs):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
