"""Parity of the CUDA path (called through the C ABI) with the CPU oracle on
seeded inputs: several tiles, ragged tails in N and K, every mode, batch
1..8, split-K, argmax, plus the hand-worked fixtures.  Integer and byte
results and the quantized-mode GEMV are compared bit for bit; Dequant within
1e-5 of sum|W x| per row."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from casebuild import (MODES, block_case, lo_case, order_records,  # noqa: E402
                       quantizer_records)
from gpuhelp import (DEV, act_buffers, assert_gemv_close, bits, dev_acts,  # noqa: E402
                     gpu_gemv, gpu_quantize, host, oracle_acts, ring_takes, to_dev)
from q8_quantized_gemv_gb300 import build, lk, synth  # noqa: E402

pytestmark = pytest.mark.gpu

DQ, I8, TP = 0, 1, 2
PATHS = {"direct": 1, "ring": 2, "mma": 3}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    lk._load()
    yield


@pytest.fixture(params=sorted(PATHS))
def path(request):
    return request.param


def cfgp(path):
    """Launch settings forcing the GEMV kernel of `path`."""
    return lk.launch_cfg(path=PATHS[path])


def need(path, K, N=64, mode=1, M=1, S=0):
    """Skip the ring-path case when the ring kernel does not take the shape
    (K % 256 != 0, or the activation does not fit in shared memory), and the
    tensor-core case outside its domain (quantized modes, 2..8 rows, no
    split-K)."""
    if path == "ring" and lk.lk_gemv_kernel_for(N, K, mode, M, S, cfg=cfgp(path)) != 2:
        pytest.skip("shape not taken by the ring kernel")
    if path == "mma" and (S > 0 or lk.lk_gemv_kernel_for(N, K, mode, M, 0, cfg=cfgp(path)) != 3):
        pytest.skip("shape not taken by the tensor-core kernel")


def sync_check():
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) == 0


# ---- quantizer and norm --------------------------------------------------------

@pytest.mark.parametrize("rec", quantizer_records(), ids=lambda r: f"{r['name']}-{r['mode']}")
def test_quantizer_hand_worked_on_gpu(rec):
    xq, xl, xs = gpu_quantize(to_dev(rec["x"]), rec["mode"])
    n = rec["n"]
    assert bits(host(xs))[0, 0] == rec["s_bits"]
    assert host(xq)[0, :n].tolist() == rec["hi"]
    if rec["lo"] is not None:
        assert host(xl)[0, :n].tolist() == rec["lo"]


@pytest.mark.parametrize("mode", [I8, TP])
@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (8, 4096), (2, 25600)])
def test_quantize_act_bitexact(mode, M, K):
    x = synth.activation(M, K, 1000 + K + M, outliers=True)
    x[0, :32] = 0.0                         # an all-zero group
    x[-1, 64:96] = np.float32(1e-38) if K >= 96 else x[-1, 64:96]  # subnormal-range scale
    hi, lo, s = oracle.quantize(x, mode)
    xq, xl, xs = gpu_quantize(to_dev(x), mode)
    sync_check()
    assert np.array_equal(host(xq), hi)
    assert np.array_equal(bits(host(xs)), bits(s))
    if mode == TP:
        assert np.array_equal(host(xl), lo)


@pytest.mark.parametrize("mode", [DQ, I8, TP])
@pytest.mark.parametrize("M,K", [(1, 32), (2, 544), (1, 1024), (3, 1056), (8, 4096), (1, 5120),
                                 (2, 12288), (1, 25600)])
def test_rmsnorm_quant_bitexact(mode, M, K):
    x = synth.activation(M, K, 2000 + K, outliers=True)
    g = synth.norm_gain(K, 2001)
    yn = oracle.rmsnorm(x, g, mode)
    xn = torch.full((M, K), float("nan"), dtype=torch.float32, device=DEV)
    xq = xl = xs = None
    if mode != DQ:
        xq, xl, xs = act_buffers(M, K, mode)
    lk.lk_rmsnorm_quant(to_dev(x), to_dev(g), mode, 1e-6, xn, xq, xl, xs)
    sync_check()
    assert np.array_equal(bits(host(xn)), bits(yn))
    if mode != DQ:
        hi, lo, s = oracle.quantize(yn, mode)
        assert np.array_equal(host(xq), hi)
        assert np.array_equal(bits(host(xs)), bits(s))
        if mode == TP:
            assert np.array_equal(host(xl), lo)


@pytest.mark.parametrize("name", ["sumsq_tree_k32", "sumsq_tree_k1024", "sumsq_tree_k2048"])
def test_rmsnorm_tree_fixture_on_gpu(name):
    rec = order_records()[name]
    K = int(rec["K"])
    v = np.zeros((1, K), np.float32)
    for item in rec["nonzero"].split():
        i, val = item.split(":")
        v[0, int(i)] = float(val)
    g = np.ones(K, np.float32)
    xn = torch.zeros((1, K), dtype=torch.float32, device=DEV)
    xq, _, xs = act_buffers(1, K, I8)
    lk.lk_rmsnorm_quant(to_dev(v), to_dev(g), I8, 1e-6, xn, xq, None, xs)
    sync_check()
    # y_0 = 4096 / sqrt(sumsq/K + eps) with the fixture's sum of squares
    ss = np.float32(rec["sumsq_f32"])
    den = np.sqrt(ss / np.float32(K) + np.float32(1e-6), dtype=np.float32)
    assert host(xn)[0, 0] == np.float32(np.float32(4096.0) / den)
    assert np.array_equal(bits(host(xn)), bits(oracle.rmsnorm(v, g, I8)))


# ---- block dots -------------------------------------------------------------------

@pytest.mark.parametrize("N,K", [(37, 544), (5, 32), (64, 4096)])
def test_block_dots_exact(N, K):
    wq, _ = synth.q8_matrix(N, K, 3000 + K)
    x = synth.activation(1, K, 3001, outliers=True)
    hi, lo, _ = oracle.quantize(x, TP)
    d0, e0 = oracle.block_dots(wq, hi[0], lo[0])
    d = torch.zeros((N, K // 32), dtype=torch.int32, device=DEV)
    e = torch.zeros_like(d)
    lk.lk_q8_block_dots(to_dev(wq), to_dev(hi[0]), d, xl=to_dev(lo[0]), e=e)
    sync_check()
    assert np.array_equal(host(d), d0) and np.array_equal(host(e), e0)


# ---- GEMV --------------------------------------------------------------------------

SHAPES = [(33, 32), (37, 544), (100, 4096), (1024, 1024), (257, 1056), (33, 256), (300, 1280),
          (1000, 512)]


@pytest.mark.parametrize("mode", [DQ, I8, TP])
@pytest.mark.parametrize("M", [1, 2, 5, 8])
@pytest.mark.parametrize("N,K", SHAPES)
def test_gemv_parity(path, mode, M, N, K):
    need(path, K, N, mode, M)
    wq, ws = synth.q8_matrix(N, K, 4000 + N + K)
    x = synth.activation(M, K, 4001 + M, outliers=True)
    y_or = oracle.gemv(wq, ws, mode, **oracle_acts(x, mode))
    wq_d, ws_d = to_dev(wq), to_dev(ws)
    y, _, _ = gpu_gemv(wq_d, ws_d, mode, dev_acts(x, mode), M, cfg=cfgp(path))
    sync_check()
    assert_gemv_close(host(y), y_or, wq, ws, x, mode)
    # run to run: the same bytes
    y2, _, _ = gpu_gemv(wq_d, ws_d, mode, dev_acts(x, mode), M, cfg=cfgp(path))
    sync_check()
    assert np.array_equal(bits(host(y2)), bits(host(y)))


@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("K", [8192, 12288, 25600])
def test_dequant_long_rows_same_sign(path, M, K):
    """Dequant where every product w*x is positive (no cancellation to hide
    rounding): the longest whole-row stages (K = 8192, 64 segments summed in
    f32 per lane) and sliced rows stay within 1e-5 of sum|W x|."""
    need(path, K, 64, DQ, M)
    rng = np.random.default_rng(4200 + K + M)
    wq = rng.integers(1, 128, size=(64, K), dtype=np.int16).astype(np.int8)
    _, ws = synth.q8_matrix(64, K, 4201 + K)
    x = np.abs(synth.activation(M, K, 4202 + K + M, outliers=True)).astype(np.float32)
    y_or = oracle.gemv(wq, ws, DQ, x=x)
    y, _, _ = gpu_gemv(to_dev(wq), to_dev(ws), DQ, dev_acts(x, DQ), M, cfg=cfgp(path))
    sync_check()
    assert_gemv_close(host(y), y_or, wq, ws, x, DQ)


@pytest.mark.parametrize("mode", [DQ, I8, TP])
def test_gemv_batch_invariance(path, mode):
    N, K, M = 300, 2048, 8
    wq, ws = synth.q8_matrix(N, K, 4100)
    x = synth.activation(M, K, 4101, outliers=True)
    need(path, K, N, mode, M)
    wq_d, ws_d = to_dev(wq), to_dev(ws)
    yb, _, _ = gpu_gemv(wq_d, ws_d, mode, dev_acts(x, mode), M, cfg=cfgp(path))
    one = None if path == "mma" else cfgp(path)  # mma: single rows through the default (batch-1) kernel
    for t in range(M):
        y1, _, _ = gpu_gemv(wq_d, ws_d, mode, dev_acts(x[t:t + 1], mode), 1, cfg=one)
        assert np.array_equal(bits(host(y1))[0], bits(host(yb))[t])
    sync_check()


@pytest.mark.parametrize("name", ["gemv_sum4", "gemv_chain"])
@pytest.mark.parametrize("mode", ["dequant", "int8act", "twopass"])
def test_gemv_order_fixture_on_gpu(path, name, mode):
    rec = order_records()[name]
    K = int(rec["K"])
    pad = -(-K // 256) * 256 if path != "direct" else None  # zero-weight blocks up to K % 256 == 0
    wq, ws, x = block_case(K, rec["blocks"], pad_to=pad)
    m = MODES[mode]
    x, M = fixture_rows(path, m, x)
    y, _, _ = gpu_gemv(to_dev(wq), to_dev(ws), m, dev_acts(x, m), M, cfg=cfgp(path))
    sync_check()
    assert host(y)[:, 0].tolist() == [np.float32(rec[f"y_{mode}"])] * M


def fixture_rows(path, mode, x):
    """The tensor-core kernel takes 2..8 rows of quantized activations: the
    one-row fixtures run there as two equal rows."""
    if path == "mma":
        if mode == DQ:
            pytest.skip("Dequant is not a tensor-core mode")
        return np.repeat(x, 2, axis=0), 2
    return x, 1


@pytest.mark.parametrize("mode", ["dequant", "int8act", "twopass"])
def test_gemv_low_word_fixture_on_gpu(path, mode):
    rec = order_records()["gemv_lo"]
    wq, ws, x = lo_case(rec, pad_to=256 if path != "direct" else None)
    m = MODES[mode]
    x, M = fixture_rows(path, m, x)
    y, _, _ = gpu_gemv(to_dev(wq), to_dev(ws), m, dev_acts(x, m), M, cfg=cfgp(path))
    sync_check()
    assert host(y)[:, 0].tolist() == [np.float32(rec[f"y_{mode}"])] * M


def test_gemv_k_zero_and_empty():
    wq = torch.zeros((5, 0), dtype=torch.int8, device=DEV)
    ws = torch.zeros((5, 0), dtype=torch.int16, device=DEV)
    xq = torch.zeros((1, 0), dtype=torch.int8, device=DEV)
    xs = torch.zeros((1, 0), dtype=torch.float32, device=DEV)
    y = torch.full((1, 5), 7.0, device=DEV)
    lk.lk_gemv_q8(wq, ws, I8, y, xq=xq, xs=xs, M=1)
    sync_check()
    assert np.all(host(y) == 0.0)


# ---- split-K -----------------------------------------------------------------------

@pytest.mark.parametrize("mode", [DQ, I8, TP])
@pytest.mark.parametrize("S", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("N,K,M", [(37, 544, 1), (64, 5120, 2), (40, 1024, 8), (300, 2304, 3)])
def test_splitk_parity(path, mode, S, N, K, M):
    need(path, K, N, mode, M, S)
    wq, ws = synth.q8_matrix(N, K, 5000 + K)
    x = synth.activation(M, K, 5001, outliers=True)
    y_or, ch_or = oracle.gemv_splitk(wq, ws, mode, S, **oracle_acts(x, mode))
    wq_d, ws_d = to_dev(wq), to_dev(ws)
    dt = torch.float64 if mode == DQ else torch.float32
    part = torch.full((S, M, N), float("nan"), dtype=dt, device=DEV)
    acts = dev_acts(x, mode)
    lk.lk_gemv_q8_splitk(wq_d, ws_d, mode, S, part, M=M, cfg=cfgp(path), **acts)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    lk.lk_splitk_combine(mode, part, S, M, N, y)
    sync_check()
    if mode == DQ:
        mag = oracle.absdot(wq, ws, x)
        assert np.all(np.abs(host(part) - ch_or) <= 1e-5 * mag[None] + 1e-30)
    else:
        assert np.array_equal(bits(host(part)), bits(ch_or))
    assert_gemv_close(host(y), y_or, wq, ws, x, mode)
    if S == 1 and mode != DQ:
        y1, _, _ = gpu_gemv(wq_d, ws_d, mode, acts, M, cfg=cfgp(path))
        assert np.array_equal(host(y1), host(y))
    # run to run
    part2 = torch.zeros_like(part)
    lk.lk_gemv_q8_splitk(wq_d, ws_d, mode, S, part2, M=M, cfg=cfgp(path), **acts)
    y2 = torch.zeros_like(y)
    lk.lk_splitk_combine(mode, part2, S, M, N, y2)
    sync_check()
    assert torch.equal(part2.view(torch.int64 if mode == DQ else torch.int32),
                       part.view(torch.int64 if mode == DQ else torch.int32))
    assert torch.equal(y2.view(torch.int32), y.view(torch.int32))


@pytest.mark.parametrize("mode", ["dequant", "int8act", "twopass"])
def test_splitk_combine_fixture_on_gpu(path, mode):
    rec = order_records()["splitk_combine"]
    K, S = int(rec["K"]), int(rec["S"])
    need(path, K, 1, MODES[mode], 1, S)
    wq, ws, x = block_case(K, rec["blocks"])
    m = MODES[mode]
    part = torch.zeros((S, 1, 1), dtype=torch.float64 if m == DQ else torch.float32, device=DEV)
    lk.lk_gemv_q8_splitk(to_dev(wq), to_dev(ws), m, S, part, M=1, cfg=cfgp(path), **dev_acts(x, m))
    y = torch.zeros((1, 1), device=DEV)
    lk.lk_splitk_combine(m, part, S, 1, 1, y)
    yp, _, _ = gpu_gemv(to_dev(wq), to_dev(ws), m, dev_acts(x, m), 1, cfg=cfgp(path))
    sync_check()
    assert host(y)[0, 0] == np.float32(rec[f"y_split_{mode}"])
    assert host(yp)[0, 0] == np.float32(rec[f"y_plain_{mode}"])


# ---- argmax -------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 5, 2048, 2049, 151936])
@pytest.mark.parametrize("M", [1, 3])
def test_argmax_logits(N, M):
    r = np.random.default_rng(N + M)
    lg = r.standard_normal((M, N)).astype(np.float32)
    if N > 10:
        for t in range(M):
            idx = sorted(r.choice(N, 3, replace=False))
            lg[t, idx] = lg[t].max() + 1
    if N == 5:
        lg[0] = [-1.0, -0.0, 0.0, -0.0, -3.0]  # -0 == +0: first wins
    idx = torch.full((M,), -1, dtype=torch.int32, device=DEV)
    scratch = torch.zeros((M * lk.lk_argmax_scratch_entries(N),), dtype=torch.int64, device=DEV)
    lk.lk_argmax(idx, M, N, logits=to_dev(lg), scratch=scratch)
    sync_check()
    assert host(idx).tolist() == [oracle.argmax(lg[t]) for t in range(M)]


@pytest.mark.parametrize("mode", [DQ, I8, TP])
def test_gemv_argmax_epilogue_planted_ties(path, mode):
    N, K, M = 5000, 256, 2
    need(path, K, N, mode, M)
    wq, ws = synth.q8_matrix(N, K, 6000)
    x = synth.activation(M, K, 6001)
    # one dominant row (levels 127*sign of activation row 0, scale 1.0) copied
    # to rows on both sides of block boundaries; the first copy must win
    dom = (127 * np.sign(x[0])).astype(np.int8)
    planted = [31, 32, 2047, 4999]
    for i in planted:
        wq[i] = dom
        ws[i] = np.float16(1.0).view(np.uint16)
    y_or = oracle.gemv(wq, ws, mode, **oracle_acts(x, mode))
    y, parts, n = gpu_gemv(to_dev(wq), to_dev(ws), mode, dev_acts(x, mode), M, amax=True, cfg=cfgp(path))
    idx = torch.full((M,), -1, dtype=torch.int32, device=DEV)
    lk.lk_argmax(idx, M, N, parts=parts, n_parts=n)
    sync_check()
    want = [oracle.argmax(y_or[t]) for t in range(M)]
    assert want[0] == 31
    assert host(idx).tolist() == want
    assert_gemv_close(host(y), y_or, wq, ws, x, mode)


# ---- failure path: a bounded device wait gives up without hanging the GPU ------------

def test_bounded_wait_reports_timeout_and_context_survives():
    lk.lk_device_error(reset=True)
    lk.lk_selftest_wait_timeout(2000)  # 2 ms on an mbarrier nothing completes
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) != 0
    assert lk.lk_device_error(reset=True) == 0
    # the context is still usable: a GEMV on each path matches the oracle
    N, K = 64, 512
    wq, ws = synth.q8_matrix(N, K, 7000)
    x = synth.activation(1, K, 7001)
    y_or = oracle.gemv(wq, ws, I8, **oracle_acts(x, I8))
    for p in (1, 2):
        y, _, _ = gpu_gemv(to_dev(wq), to_dev(ws), I8, dev_acts(x, I8), 1, cfg=lk.launch_cfg(path=p))
        sync_check()
        assert np.array_equal(bits(host(y)), bits(y_or))


# ---- fused RMSNorm -> quantize -> GEMV (one launch) -----------------------------------

@pytest.mark.parametrize("pdl", [0, 1])
@pytest.mark.parametrize("mode", [DQ, I8, TP])
@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("N,K,norm", [(300, 1280, True), (1000, 4096, True), (77, 256, False),
                                      (64, 12288, False), (5, 2048, True)])
def test_fused_norm_quant_gemv(pdl, mode, M, N, K, norm):
    if not ring_takes(N, K, mode, M):
        pytest.skip("activation area does not fit the ring kernel")
    cfg = lk.launch_cfg(pdl=pdl)
    wq, ws = synth.q8_matrix(N, K, 8000 + N + K)
    x = synth.activation(M, K, 8001 + M, outliers=True)
    g = synth.norm_gain(K, 8002) if norm else None
    xa = oracle.rmsnorm(x, g, mode) if norm else x
    y_or = oracle.gemv(wq, ws, mode, **oracle_acts(xa, mode))
    wq_d, ws_d = to_dev(wq), to_dev(ws)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    parts = torch.zeros((M * lk.lk_argmax_parts_max(N),), dtype=torch.int64, device=DEV)
    n = lk.lk_rmsnorm_quant_gemv_q8(wq_d, ws_d, mode, to_dev(x), y, gain=to_dev(g) if norm else None,
                                    argmax_parts=parts, cfg=cfg)
    idx = torch.full((M,), -1, dtype=torch.int32, device=DEV)
    lk.lk_argmax(idx, M, N, parts=parts, n_parts=n)
    sync_check()
    assert_gemv_close(host(y), y_or, wq, ws, xa, mode)
    assert host(idx).tolist() == [oracle.argmax(y_or[t]) for t in range(M)]
    # the same bits as the unfused launches (for 2..8 rows: the tensor-core kernel)
    if mode != DQ:
        y2 = torch.zeros_like(y)
        xq, xl, xs = act_buffers(M, K, mode)
        if norm:
            lk.lk_rmsnorm_quant(to_dev(x), to_dev(g), mode, 1e-6, None, xq, xl, xs, cfg=cfg)
        else:
            lk.lk_quantize_act(to_dev(x), mode, xq, xl, xs, cfg=cfg)
        lk.lk_gemv_q8(wq_d, ws_d, mode, y2, xq=xq, xl=xl, xs=xs, M=M, cfg=cfg)
        sync_check()
        assert torch.equal(y.view(torch.int32), y2.view(torch.int32))


def test_fused_pdl_chain_in_a_graph():
    """A chain of fused launches where each reads the previous one's output,
    captured in one CUDA graph with programmatic dependent launches, gives the
    same bits as the same chain launched plainly."""
    K = N = 1024
    L = 6
    mats = [synth.q8_matrix(N, K, 8100 + l) for l in range(L)]
    gains = [synth.norm_gain(K, 8200 + l) for l in range(L)]
    x0 = synth.activation(1, K, 8300)
    dm = [(to_dev(w), to_dev(s)) for w, s in mats]
    dg = [to_dev(g) for g in gains]
    bufs = [torch.zeros((1, N), dtype=torch.float32, device=DEV) for _ in range(L + 1)]
    bufs[0].copy_(to_dev(x0))

    def chain(cfg=None):
        for l in range(L):
            lk.lk_rmsnorm_quant_gemv_q8(dm[l][0], dm[l][1], I8, bufs[l], bufs[l + 1], gain=dg[l], cfg=cfg)

    chain()
    torch.cuda.synchronize()
    ref = host(bufs[L]).copy()
    # oracle of the whole chain
    v = x0
    for l in range(L):
        a = oracle.rmsnorm(v, gains[l], I8)
        v = oracle.gemv(mats[l][0], mats[l][1], I8, **oracle_acts(a, I8))
    assert np.array_equal(bits(ref), bits(v))
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        chain(lk.launch_cfg(pdl=1))
    for _ in range(3):
        for b in bufs[1:]:
            b.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(host(bufs[L])), bits(ref))
    sync_check()
