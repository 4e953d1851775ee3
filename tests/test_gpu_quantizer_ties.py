"""The activation quantizer and the RMSNorm on the GPU against the oracle, bit
for bit, on inputs built to sit on or next to rounding boundaries: group
values whose quotient v/s is a half-integer exactly or offset from one by
2^-24 .. 2^-10 (around the width the device's reciprocal shortcut hands over
to the IEEE division), low-word residuals near ties, scales across the
exponent range, and long random rows for the norm's quotient."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpuhelp import DEV, act_buffers, bits, host, to_dev  # noqa: E402
from q8_quantized_gemv_gb300 import build, lk, synth  # noqa: E402

pytestmark = pytest.mark.gpu

I8, TP = 1, 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield


def near_tie_groups(n_groups, seed):
    """Groups of 32: value 0 is the group maximum 127 s0; the others are
    (k + 1/2 + d) s0 for integers k and offsets d around the hand-over width."""
    r = np.random.default_rng(seed)
    s0 = (2.0 ** r.integers(-40, 40, size=(n_groups, 1))) * r.uniform(1.0, 2.0, size=(n_groups, 1))
    k = r.integers(-127, 127, size=(n_groups, 32)).astype(np.float64)
    offs = np.array([0.0, 2.0 ** -24, -2.0 ** -24, 2.0 ** -16, -2.0 ** -16, 2.0 ** -13, -2.0 ** -13,
                     2.0 ** -12, -2.0 ** -12, 2.0 ** -11, -2.0 ** -11, 2.0 ** -10, 0.25, -0.25])
    d = offs[r.integers(0, offs.size, size=(n_groups, 32))]
    v = ((k + 0.5 + d) * s0).astype(np.float32)
    v[:, 0] = (127.0 * s0[:, 0]).astype(np.float32)
    # low-word ties: v = (h + l/128 + 1/256) s with the residual's quotient at a half-integer
    lw = r.integers(0, n_groups, size=n_groups // 4)
    h = r.integers(-120, 120, size=(lw.size, 31)).astype(np.float64)
    l = r.integers(-60, 60, size=(lw.size, 31)).astype(np.float64)
    v[lw, 1:] = ((h + (l + 0.5) / 128.0) * s0[lw]).astype(np.float32)
    return v.reshape(1, -1)


@pytest.mark.parametrize("mode", [I8, TP])
def test_quantizer_near_rounding_boundaries(mode):
    x = near_tie_groups(1 << 15, 11 + mode)  # 2^20 values
    # the oracle quantizes row by row; four rows of 2^18 values
    x = x.reshape(4, -1)
    M, K = x.shape
    hi, lo, s = oracle.quantize(x, mode)
    xq, xl, xs = act_buffers(M, K, mode)
    lk.lk_quantize_act(to_dev(x), mode, xq, xl, xs)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(xs)), bits(s))
    bad = np.nonzero(host(xq) != hi)
    assert bad[0].size == 0, (bad[0].size, x[bad][:4], host(xq)[bad][:4], hi[bad][:4])
    if mode == TP:
        assert np.array_equal(host(xl), lo)


@pytest.mark.parametrize("mode", [0, I8, TP])
@pytest.mark.parametrize("K", [4096, 25600])
def test_norm_quotients_long_rows(mode, K):
    """64 rows at scales from 2^-30 to 2^30: the norm's quotient v / den and
    its product with the gain, then the quantizer, bit for bit."""
    M = 64
    x = synth.activation(M, K, 900 + K, outliers=True)
    x *= (2.0 ** np.linspace(-30, 30, M)).astype(np.float32)[:, None]
    x = x.astype(np.float32)
    g = synth.norm_gain(K, 901)
    yn = oracle.rmsnorm(x, g, mode)
    xn = torch.empty((M, K), dtype=torch.float32, device=DEV)
    if mode == 0:
        lk.lk_rmsnorm_quant(to_dev(x), to_dev(g), mode, 1e-6, xn)
    else:
        xq, xl, xs = act_buffers(M, K, mode)
        lk.lk_rmsnorm_quant(to_dev(x), to_dev(g), mode, 1e-6, xn, xq, xl, xs)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(xn)), bits(yn))
    if mode:
        hi, lo, s = oracle.quantize(yn, mode)
        assert np.array_equal(host(xq), hi) and np.array_equal(bits(host(xs)), bits(s))
        if mode == TP:
            assert np.array_equal(host(xl), lo)
