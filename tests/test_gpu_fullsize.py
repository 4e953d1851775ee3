"""Parity at the full workload sizes, in the launch configuration the
benchmark uses (the library's automatic kernel choice): the RMSNorm ->
quantize launch over the whole activation, and every output row of the GEMV
against the oracle (all 151936 rows of the lm-head included).  The argmax
must be the oracle's first-index argmax of the GPU's logits, which are
themselves checked row by row."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpuhelp import (DEV, act_buffers, assert_gemv_close, bits, host,  # noqa: E402
                     oracle_acts, to_dev)
from q8_quantized_gemv_gb300 import build, lk, synth  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

DQ, I8, TP = 0, 1, 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield
    torch.cuda.empty_cache()


def weights(N, K, seed):
    if N * K <= (1 << 27):
        wq, ws = synth.q8_matrix(N, K, seed)
        return to_dev(wq), to_dev(ws)
    return synth.q8_matrix_torch(N, K, seed, DEV)


def norm_quant(x_np, g_np, mode):
    """GPU prologue, checked bit-exact against the oracle; returns the device
    activations and the oracle's normed f32 rows."""
    M, K = x_np.shape
    yn = oracle.rmsnorm(x_np, g_np, mode)
    xn = torch.empty((M, K), dtype=torch.float32, device=DEV)
    acts = {}
    if mode == DQ:
        lk.lk_rmsnorm_quant(to_dev(x_np), to_dev(g_np), mode, 1e-6, xn)
        acts["x"] = xn
    else:
        xq, xl, xs = act_buffers(M, K, mode)
        lk.lk_rmsnorm_quant(to_dev(x_np), to_dev(g_np), mode, 1e-6, xn, xq, xl, xs)
        hi, lo, s = oracle.quantize(yn, mode)
        assert np.array_equal(host(xq), hi) and np.array_equal(bits(host(xs)), bits(s))
        if mode == TP:
            assert np.array_equal(host(xl), lo)
        acts.update(xq=xq, xs=xs)
        if mode == TP:
            acts["xl"] = xl
    assert np.array_equal(bits(host(xn)), bits(yn))
    return acts, yn


def check_all_rows(y_dev, wq_d, ws_d, mode, yn):
    """Every output row of y against the oracle (bit-exact in the quantized
    modes, within the tolerance under Dequant)."""
    wq = host(wq_d)
    ws = host(ws_d).view(np.uint16)
    y_or = oracle.gemv(wq, ws, mode, **oracle_acts(yn, mode))
    assert_gemv_close(host(y_dev), y_or, wq, ws, yn, mode)


@pytest.mark.parametrize("mode", [DQ, I8, TP])
@pytest.mark.parametrize("N", [4096, 24576])
def test_fused_norm_quant_gemv_hidden4096(mode, N):
    K = 4096
    x = synth.activation(1, K, synth.SEED_BASE + 1, outliers=True)
    g = synth.norm_gain(K, synth.SEED_BASE + 11)
    wq_d, ws_d = weights(N, K, synth.SEED_BASE + 100 + N)
    acts, yn = norm_quant(x, g, mode)
    y = torch.empty((1, N), dtype=torch.float32, device=DEV)
    lk.lk_gemv_q8(wq_d, ws_d, mode, y, M=1, **acts)
    check_all_rows(y, wq_d, ws_d, mode, yn)
    y2 = torch.empty_like(y)
    lk.lk_gemv_q8(wq_d, ws_d, mode, y2, M=1, **acts)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))


@pytest.mark.parametrize("mode", [DQ, TP])
@pytest.mark.parametrize("K", [5120, 25600])
def test_splitk_narrow_projections(mode, K):
    N = 5120
    x = synth.activation(1, K, synth.SEED_BASE + 2, outliers=True)
    wq_d, ws_d = weights(N, K, synth.SEED_BASE + 200 + K)
    if mode == DQ:
        acts, xa = {"x": to_dev(x)}, x
    else:
        hi, lo, s = oracle.quantize(x, mode)
        acts, xa = {"xq": to_dev(hi), "xl": to_dev(lo), "xs": to_dev(s)}, x
    wq = host(wq_d)
    ws = host(ws_d).view(np.uint16)
    for S in (1, 2, 4, 8):
        y_or, ch_or = oracle.gemv_splitk(wq, ws, mode, S, **oracle_acts(xa, mode))
        dt = torch.float64 if mode == DQ else torch.float32
        part = torch.empty((S, 1, N), dtype=dt, device=DEV)
        lk.lk_gemv_q8_splitk(wq_d, ws_d, mode, S, part, M=1, **acts)
        y = torch.empty((1, N), dtype=torch.float32, device=DEV)
        lk.lk_splitk_combine(mode, part, S, 1, N, y)
        p = host(part)
        if mode == DQ:
            mag = oracle.absdot(wq, ws, xa)
            assert np.all(np.abs(p - ch_or) <= 1e-5 * mag[None] + 1e-30)
        else:
            assert np.array_equal(bits(p), bits(ch_or))
        assert_gemv_close(host(y), y_or, wq, ws, xa, mode)
        y2 = torch.empty_like(y)
        part2 = torch.empty_like(part)
        lk.lk_gemv_q8_splitk(wq_d, ws_d, mode, S, part2, M=1, **acts)
        lk.lk_splitk_combine(mode, part2, S, 1, N, y2)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), y2.view(torch.int32))


@pytest.mark.parametrize("mode", [DQ, I8, TP])
def test_lm_head_argmax_planted_ties(mode):
    N, K = 151936, 4096
    x = synth.activation(1, K, synth.SEED_BASE + 3)
    g = synth.norm_gain(K, synth.SEED_BASE + 13)
    wq_d, ws_d = weights(N, K, synth.SEED_BASE + 300)
    acts, yn = norm_quant(x, g, mode)
    # the dominant row: 127 * sign of the normed activation, scale 1.0
    dom = torch.from_numpy((127 * np.sign(yn[0])).astype(np.int8)).to(DEV)
    planted = [5, 2047, 2048, N - 1]
    for i in planted:
        wq_d[i] = dom
        ws_d[i] = torch.tensor(np.float16(1.0).view(np.int16), device=DEV)
    y = torch.empty((1, N), dtype=torch.float32, device=DEV)
    parts = torch.zeros((lk.lk_argmax_parts_max(N),), dtype=torch.int64, device=DEV)
    n = lk.lk_gemv_q8(wq_d, ws_d, mode, y, M=1, argmax_parts=parts, **acts)
    idx = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    lk.lk_argmax(idx, 1, N, parts=parts, n_parts=n)
    torch.cuda.synchronize()
    check_all_rows(y, wq_d, ws_d, mode, yn)
    logits = host(y)[0]
    assert int(host(idx)[0]) == 5 == oracle.argmax(logits)
    assert len(set(bits(logits[planted]).tolist())) == 1
    # all-zero weights: every logit is 0, the first index wins
    wz = torch.zeros_like(wq_d)
    lk.lk_gemv_q8(wz, ws_d, mode, y, M=1, argmax_parts=parts, **acts)
    lk.lk_argmax(idx, 1, N, parts=parts, n_parts=n)
    torch.cuda.synchronize()
    assert int(host(idx)[0]) == 0 and not host(y).any()


@pytest.mark.parametrize("mode", [I8, TP])
@pytest.mark.parametrize("name,N,K", [("q", 4096, 4096), ("kv", 1024, 4096), ("gate_up", 24576, 4096),
                                      ("down", 4096, 12288), ("lm_head", 151936, 4096)])
def test_batch8_sequence_projections(mode, name, N, K):
    """The 36-layer sequence's projections at batch 8, in the kernel the
    library picks for 8 rows (the tensor-core kernel where it applies), with
    the lm-head's argmax epilogue for all 8 rows."""
    M = 8
    x = synth.activation(M, K, synth.SEED_BASE + 40 + K, outliers=True)
    g = synth.norm_gain(K, synth.SEED_BASE + 41)
    wq_d, ws_d = weights(N, K, synth.SEED_BASE + 400 + N + K)
    acts, yn = norm_quant(x, g, mode)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    parts = torch.zeros((M * lk.lk_argmax_parts_max(N),), dtype=torch.int64, device=DEV)
    n = lk.lk_gemv_q8(wq_d, ws_d, mode, y, M=M, argmax_parts=parts, **acts)
    idx = torch.full((M,), -1, dtype=torch.int32, device=DEV)
    lk.lk_argmax(idx, M, N, parts=parts, n_parts=n)
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) == 0
    check_all_rows(y, wq_d, ws_d, mode, yn)
    logits = host(y)
    assert host(idx).tolist() == [oracle.argmax(logits[t]) for t in range(M)]
    y2 = torch.empty_like(y)
    lk.lk_gemv_q8(wq_d, ws_d, mode, y2, M=M, **acts)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))
