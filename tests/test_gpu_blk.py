"""The GGUF block formats other than Q8_0 on the GPU against the oracle: every
format's decoder bit for bit (the decode hook against the oracle's dequantized
weights), and the block-format GEMV bit for bit under Int8Act and TwoPass and
within 1e-5 * sum|w x| per row under Dequant, at 1, 3 and 8 activation rows,
over shapes with a ragged row count and several blocks per lane."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpuhelp import DEV, bits, host, to_dev  # noqa: E402
from q8_quantized_gemv_gb300 import build, lk, synth  # noqa: E402

pytestmark = pytest.mark.gpu

FMTS = sorted(synth.BLK_LAYOUT)
SHAPES = [(37, 256), (300, 2048), (64, 4096)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield


def takes(fmt, K):
    rb = lk.lk_format_row_bytes(fmt, K)
    return rb > 0 and rb % 16 == 0 and K % 256 == 0


@pytest.mark.parametrize("fmt", FMTS)
def test_decoders_bit_for_bit(fmt):
    N, K = 50, 4096
    w = synth.blk_matrix(fmt, N, K, 300 + oracle.FORMATS[fmt])
    out = torch.full((N, K), float("nan"), dtype=torch.float32, device=DEV)
    lk.lk_dequant_blk(fmt, to_dev(w), K, out)
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) == 0
    want = oracle.dequant(oracle.FORMATS[fmt], w, K)
    assert np.array_equal(bits(host(out)), bits(want))


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_blk_matches_oracle(fmt, N, K, M, mode):
    if not takes(fmt, K):
        pytest.skip("row not a multiple of 16 bytes at this K")
    F = oracle.FORMATS[fmt]
    w = synth.blk_matrix(fmt, N, K, 400 + F + N + K)
    x = synth.activation(M, K, 401 + M, outliers=True)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    if mode == 0:
        y_or = oracle.gemv_blk(F, w, K, 0, x=x)
        lk.lk_gemv_blk(fmt, to_dev(w), K, 0, y, x=to_dev(x), M=M)
    else:
        hi, lo, s = oracle.quantize(x, mode)
        y_or = oracle.gemv_blk(F, w, K, mode, hi=hi, lo=lo, s=s)
        lk.lk_gemv_blk(fmt, to_dev(w), K, mode, y, xq=to_dev(hi), xs=to_dev(s),
                       xl=to_dev(lo) if mode == 2 else None, M=M)
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) == 0
    yg = host(y)
    if mode == 0:
        mag = oracle.absdot_blk(F, w, K, x)
        err = np.abs(yg.astype(np.float64) - y_or.astype(np.float64))
        assert np.all(err <= 1e-5 * mag + 1e-30), float((err / np.maximum(mag, 1e-30)).max())
    else:
        bad = np.nonzero(bits(yg) != bits(y_or))
        assert bad[0].size == 0, (bad[0].size, yg[bad][:4], y_or[bad][:4])


def test_gemv_blk_run_to_run_and_pdl_graph():
    """The same bits on every run, and as programmatic dependent launches in
    a captured graph."""
    fmt, N, K, M = "q4_k", 1000, 4096, 2
    w = to_dev(synth.blk_matrix(fmt, N, K, 500))
    x = synth.activation(M, K, 501)
    hi, lo, s = oracle.quantize(x, 1)
    acts = dict(xq=to_dev(hi), xs=to_dev(s))
    y1 = torch.empty((M, N), dtype=torch.float32, device=DEV)
    lk.lk_gemv_blk(fmt, w, K, 1, y1, M=M, **acts)
    torch.cuda.synchronize()
    outs = [torch.empty_like(y1) for _ in range(4)]
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for o in outs:
            lk.lk_gemv_blk(fmt, w, K, 1, o, M=M, cfg=lk.launch_cfg(pdl=1), **acts)
    for _ in range(3):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for o in outs:
            assert torch.equal(o.view(torch.int32), y1.view(torch.int32))


def test_gemv_blk_argument_checks():
    w = torch.zeros((4, lk.lk_format_row_bytes("q4_0", 256)), dtype=torch.uint8, device=DEV)
    xq = torch.zeros((1, 256), dtype=torch.int8, device=DEV)
    xs = torch.zeros((1, 8), dtype=torch.float32, device=DEV)
    y = torch.zeros((1, 4), dtype=torch.float32, device=DEV)
    lib = lk._load()
    P = lambda t: None if t is None else __import__("ctypes").c_void_p(t.data_ptr())  # noqa: E731
    assert lib.lk_gemv_blk(5, P(w), 4, 256, 1, None, P(xq), None, P(xs), 1, P(y), None, None) == -1
    assert lib.lk_gemv_blk(2, P(w), 4, 288, 1, None, P(xq), None, P(xs), 1, P(y), None, None) == -3
    assert lib.lk_gemv_blk(39, P(w), 4, 256, 1, None, P(xq), None, P(xs), 1, P(y), None, None) == -3  # 136 B rows
    assert lib.lk_gemv_blk(2, P(w), 4, 256, 1, None, P(xq), None, P(xs), 9, P(y), None, None) == -3
    assert lib.lk_gemv_blk(2, P(w), 4, 256, 2, None, P(xq), None, P(xs), 1, P(y), None, None) == -1
    assert lk.lk_format_row_bytes("q6_k", 4096) == 16 * 210 and lk.lk_format_row_bytes("q4_k", 100) == 0


@pytest.mark.parametrize("fmt,mode,M", [("q4_0", 1, 1), ("q4_k", 1, 1), ("q6_k", 2, 1), ("iq4_xs", 1, 8),
                                        ("q5_1", 2, 8), ("mxfp4", 1, 3)])
def test_gemv_blk_full_size_all_rows(fmt, mode, M):
    """The gate/up-sized GEMV the bench times (24576 x 4096, the launch
    `bench.py --workload gemv --format f` makes): every output bit for bit
    the oracle's."""
    N, K = 24576, 4096
    F = oracle.FORMATS[fmt]
    w = synth.blk_matrix(fmt, N, K, 600 + F)
    x = synth.activation(M, K, 601 + M, outliers=True)
    hi, lo, s = oracle.quantize(x, mode)
    y_or = oracle.gemv_blk(F, w, K, mode, hi=hi, lo=lo, s=s)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    lk.lk_gemv_blk(fmt, to_dev(w), K, mode, y, xq=to_dev(hi), xs=to_dev(s),
                   xl=to_dev(lo) if mode == 2 else None, M=M, cfg=lk.launch_cfg(pdl=1))
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) == 0
    assert np.array_equal(bits(host(y)), bits(y_or))


@pytest.mark.parametrize("fmt", ["q4_k", "q4_0", "iq4_nl"])
@pytest.mark.parametrize("mode,M", [(1, 1), (2, 3), (0, 1)])
def test_blk_decode_stack_token(fmt, mode, M):
    """A small block-format decode stack (3 layers, hidden 1024): every GEMV
    of one token against the oracle on the GPU's own activation (bit for bit
    under Int8Act / TwoPass, within 1e-5 * sum|w x| under Dequant), and the
    argmax the oracle's first maximum of the GPU's logits."""
    from q8_quantized_gemv_gb300.decode import BlkDecodeStack
    st = BlkDecodeStack(fmt, layers=3, hidden=1024, q_dim=1024, kv_dim=256, ffn=1024, vocab=4096, batch=M,
                        mode=mode, device=DEV, pdl=True)
    F = oracle.FORMATS[fmt]
    seen = []

    def hook(name, launch):
        r = launch()
        torch.cuda.synchronize()
        seen.append(name)
        return r

    # record each GEMV's activation and output as it runs
    checks = []
    orig = st._gemv

    def gemv(w, K, y, a):
        orig(w, K, y, a)
        torch.cuda.synchronize()
        checks.append((host(w), K, {k: host(v) for k, v in a.items() if v is not None}, host(y).copy()))

    st._gemv = gemv
    idx = st.run_token(hook=hook)
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) == 0
    assert len(checks) == 3 * 4 + 1 and st.launches_per_token() == 3 * (8 if mode else 6) + 3
    for w, K, a, y in checks:
        if mode == 0:
            y_or = oracle.gemv_blk(F, w, K, 0, x=a["x"])
            mag = oracle.absdot_blk(F, w, K, a["x"])
            err = np.abs(y.astype(np.float64) - y_or.astype(np.float64))
            assert np.all(err <= 1e-5 * mag + 1e-30)
        else:
            y_or = oracle.gemv_blk(F, w, K, mode, hi=a["xq"], lo=a.get("xl"), s=a["xs"])
            assert np.array_equal(bits(y), bits(y_or))
    logits = host(st.logits)
    for t in range(M):
        assert int(host(idx)[t]) == oracle.argmax(logits[t])
