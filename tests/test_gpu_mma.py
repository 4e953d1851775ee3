"""The tensor-core GEMV (2..8 activation rows, Int8Act and TwoPassInt8)
against the CPU oracle, bit for bit: every row count, ragged N (a partial
last 16-row tile) and ragged K (a partial last stage slice), and every stage
layout the options allow (bytes of K per stage, warps, stages per warp), so
that each ring arrangement and tail path is exercised; plus the argmax
epilogue, the shapes it declines, and the grouped call (several matrices
sharing one activation in one launch)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpuhelp import DEV, bits, dev_acts, gpu_gemv, host, oracle_acts, to_dev  # noqa: E402
from q8_quantized_gemv_gb300 import build, lk, synth  # noqa: E402

pytestmark = pytest.mark.gpu

I8, TP = 1, 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield


def mma(**kw):
    """Launch settings forcing the tensor-core kernel (and the given fields)."""
    return lk.launch_cfg(path=kw.pop("path", 3), **kw)


def run_case(N, K, M, mode, seed, amax=False, cfg=None):
    cfg = cfg if cfg is not None else mma()
    assert lk.lk_gemv_kernel_for(N, K, mode, M, 0, cfg=cfg) == 3
    wq, ws = synth.q8_matrix(N, K, seed)
    x = synth.activation(M, K, seed + 1, outliers=True)
    y_or = oracle.gemv(wq, ws, mode, **oracle_acts(x, mode))
    y, parts, n = gpu_gemv(to_dev(wq), to_dev(ws), mode, dev_acts(x, mode), M, amax=amax, cfg=cfg)
    idx = None
    if amax:
        idx = torch.full((M,), -1, dtype=torch.int32, device=DEV)
        lk.lk_argmax(idx, M, N, parts=parts, n_parts=n)
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) == 0
    yg = host(y)
    bad = np.nonzero(bits(yg) != bits(y_or))
    assert bad[0].size == 0, f"{bad[0].size} mismatches, first (row, col) {bad[0][0]}, {bad[1][0]}: " \
                             f"{yg[bad[0][0], bad[1][0]]} vs {y_or[bad[0][0], bad[1][0]]}"
    if amax:
        assert host(idx).tolist() == [oracle.argmax(y_or[t]) for t in range(M)]
    return y


@pytest.mark.parametrize("path", ["f16", "f16-act16", "f16-g4", "f16-g4-act16", "i8"])
@pytest.mark.parametrize("mode", [I8, TP])
@pytest.mark.parametrize("M", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("N,K", [(16, 256), (1000, 1280), (333, 4096), (2500, 2304)])
def test_mma_rows_and_tails(path, mode, M, N, K):
    """f16: the dots as f16 MMAs on converted levels, activations held as int8
    (or f16: act16); g4: four warps per 16-row tile (one partial each,
    combined through shared memory); i8: the dots as int8 MMAs."""
    cfg = mma(mma_i8=1 if path == "i8" else 2, mma_group=4 if "g4" in path else 1,
              mma_act16=1 if "act16" in path else 2)
    run_case(N, K, M, mode, 7000 + N + K + M, cfg=cfg)


@pytest.mark.parametrize("i8", [1, 2])
@pytest.mark.parametrize("group", [1, 4])
@pytest.mark.parametrize("act16", [1, 2])
@pytest.mark.parametrize("mode", [I8, TP])
@pytest.mark.parametrize("tk,warps,depth", [(256, 0, 0), (512, 0, 0), (1024, 0, 0), (2048, 0, 0),
                                            (1024, 1, 2), (1024, 3, 1), (512, 16, 1), (256, 4, 4),
                                            (1024, 2, 3)])
def test_mma_stage_layouts(i8, group, act16, mode, tk, warps, depth):
    if group == 4 and (warps % 4 or (depth and depth < 2)):
        pytest.skip("four-warp tiles take warps in fours and two or more stages per group")
    if i8 == 1 and (group == 4 or act16 == 1):
        pytest.skip("the int8 path is one warp per tile on int8 activation rows")
    cfg = mma(mma_i8=i8, mma_group=group, mma_act16=act16, mma_tk=tk, mma_warps=warps, mma_depth=depth)
    run_case(777, 3328, 8, mode, 7100 + tk + warps, cfg=cfg)


@pytest.mark.parametrize("M", [2, 8])
@pytest.mark.parametrize("N,K", [(1024, 4096), (300, 12288), (4096, 4096)])
def test_mma_auto_layout_few_tiles(N, K, M):
    """The automatic choice for Int8Act launches with few tiles per SM (four
    warps per tile, 1 KB or 2 KB slices): bit for bit the oracle."""
    assert lk.lk_gemv_kernel_for(N, K, I8, M, 0) == 3
    run_case(N, K, M, I8, 7250 + N + M, cfg=lk.launch_cfg())


@pytest.mark.parametrize("group", [1, 4])
@pytest.mark.parametrize("ctas", [1, 7, 152])
def test_mma_grid_sizes(ctas, group):
    run_case(4100, 1024, 5, I8, 7200 + ctas, cfg=mma(mma_group=group, grid_ctas=ctas))


@pytest.mark.parametrize("group", [1, 4])
@pytest.mark.parametrize("i8", [1, 2])
@pytest.mark.parametrize("mode", [I8, TP])
def test_mma_argmax_with_ties(mode, group, i8):
    cfg = mma(mma_group=group, mma_i8=i8)
    N, K, M = 3001, 512, 8
    wq, ws = synth.q8_matrix(N, K, 7300)
    x = synth.activation(M, K, 7301)
    dom = (127 * np.sign(x[3])).astype(np.int8)
    for i in (15, 16, 2999):   # tile boundary, then the ragged last tile
        wq[i] = dom
        ws[i] = np.float16(1.0).view(np.uint16)
    y_or = oracle.gemv(wq, ws, mode, **oracle_acts(x, mode))
    y, parts, n = gpu_gemv(to_dev(wq), to_dev(ws), mode, dev_acts(x, mode), M, amax=True, cfg=cfg)
    idx = torch.full((M,), -1, dtype=torch.int32, device=DEV)
    lk.lk_argmax(idx, M, N, parts=parts, n_parts=n)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(y)), bits(y_or))
    want = [oracle.argmax(y_or[t]) for t in range(M)]
    assert want[3] == 15
    assert host(idx).tolist() == want


def test_mma_matches_batch1_kernel_bits():
    """Each of the 8 rows through the batch-1 kernel gives the same bits."""
    N, K, M = 600, 4096, 8
    wq, ws = synth.q8_matrix(N, K, 7400)
    x = synth.activation(M, K, 7401, outliers=True)
    wq_d, ws_d = to_dev(wq), to_dev(ws)
    for mode in (I8, TP):
        yb, _, _ = gpu_gemv(wq_d, ws_d, mode, dev_acts(x, mode), M, cfg=mma())
        for t in range(M):
            y1, _, _ = gpu_gemv(wq_d, ws_d, mode, dev_acts(x[t:t + 1], mode), 1)
            assert np.array_equal(bits(host(y1))[0], bits(host(yb))[t])


def test_mma_declines():
    assert lk.lk_gemv_kernel_for(4096, 4096, 1, 8, 0) == 3
    assert lk.lk_gemv_kernel_for(4096, 4096, 0, 8, 0) != 3   # Dequant
    assert lk.lk_gemv_kernel_for(4096, 4096, 1, 1, 0) != 3   # one row
    assert lk.lk_gemv_kernel_for(4096, 4128, 1, 8, 0) != 3   # K % 256 != 0
    assert lk.lk_gemv_kernel_for(4096, 4096, 1, 8, 2) == 3   # split-K too (each block: its chunk)
    # TwoPass activations of 8 rows x 12288 (209 KB) leave room for one warp's
    # two 512-byte stages: still taken
    assert lk.lk_gemv_kernel_for(4096, 12288, 2, 8, 0) == 3
    # ... but not with 4 KB stages forced
    assert lk.lk_gemv_kernel_for(4096, 12288, 2, 8, 0, cfg=lk.launch_cfg(mma_tk=4096)) != 3
    assert lk.lk_gemv_kernel_for(4096, 4096, 1, 8, 0, cfg=lk.launch_cfg(mma_min_m=9)) != 3


@pytest.mark.parametrize("group", [1, 4])
@pytest.mark.parametrize("mode", [I8, TP])
@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("Ns", [(4096, 1024, 1024), (100, 37, 1000, 16), (5,)])
def test_group_matches_single_calls_and_oracle(mode, M, Ns, group):
    """lk_gemv_q8_group over matrices with ragged N: each output has the bits
    of its own lk_gemv_q8 call and of the oracle (one launch for 2..8 rows,
    one launch per matrix for a single row)."""
    cfg = lk.launch_cfg(mma_group=group)
    K = 1280
    mats = [synth.q8_matrix(N, K, 7500 + i + N) for i, N in enumerate(Ns)]
    x = synth.activation(M, K, 7600 + M, outliers=True)
    acts = dev_acts(x, mode)
    dm = [(to_dev(w), to_dev(s), torch.full((M, w.shape[0]), float("nan"), device=DEV)) for w, s in mats]
    lk.lk_gemv_q8_group(dm, mode, M=M, cfg=cfg, **acts)
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) == 0
    for (w, s), (wd, sd, y) in zip(mats, dm):
        y_or = oracle.gemv(w, s, mode, **oracle_acts(x, mode))
        assert np.array_equal(bits(host(y)), bits(y_or))
        y1, _, _ = gpu_gemv(wd, sd, mode, acts, M, cfg=cfg)
        assert np.array_equal(bits(host(y1)), bits(host(y)))


# ---- more than 8 activation rows -------------------------------------------------------

@pytest.mark.parametrize("path", ["f16", "f16-g4", "i8"])
@pytest.mark.parametrize("mode", [I8, TP])
@pytest.mark.parametrize("M", [9, 16, 33, 64])
@pytest.mark.parametrize("N,K", [(16, 256), (1000, 1280), (2500, 4096)])
def test_mma_batches_past_eight_rows(path, mode, M, N, K):
    """Groups of 8 activation rows side by side on the SMs: every value bit for
    bit the oracle's (the 8-row arithmetic), the argmax of every row, with
    ragged row groups (9, 33) and ragged tiles."""
    cfg = mma(mma_i8=1 if path == "i8" else 2, mma_group=4 if "g4" in path else 1)
    run_case(N, K, M, mode, 9100 + N + K + M, amax=True, cfg=cfg)


@pytest.mark.parametrize("mode", [I8, TP])
def test_batch_past_eight_matches_groups_of_eight(mode):
    """M = 24 in one launch equals three launches of 8 rows, bit for bit, and
    the grouped call (q, k, v) at 24 rows equals per-matrix calls."""
    N, K, M = 2048, 4096, 24
    wq, ws = synth.q8_matrix(N, K, 91)
    x = synth.activation(M, K, 92, outliers=True)
    acts = dev_acts(x, mode)
    wq_d, ws_d = to_dev(wq), to_dev(ws)
    y, _, _ = gpu_gemv(wq_d, ws_d, mode, acts, M)
    parts = []
    for r in range(0, M, 8):
        sub = {k: (v[r:r + 8].contiguous() if v is not None else None) for k, v in acts.items()}
        yy, _, _ = gpu_gemv(wq_d, ws_d, mode, sub, 8)
        parts.append(yy)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), torch.cat(parts).view(torch.int32))
    mats = [(wq_d, ws_d, torch.empty((M, N), dtype=torch.float32, device=DEV)),
            (wq_d[:1024], ws_d[:1024], torch.empty((M, 1024), dtype=torch.float32, device=DEV))]
    lk.lk_gemv_q8_group(mats, mode, M=M, **acts)
    torch.cuda.synchronize()
    assert torch.equal(mats[0][2].view(torch.int32), y.view(torch.int32))
    assert torch.equal(mats[1][2].view(torch.int32), y[:, :1024].contiguous().view(torch.int32))


def test_past_eight_rows_needs_the_tensor_core_path():
    """Past 8 rows only the tensor-core kernel runs (split-K included):
    Dequant and K % 256 != 0 are shape errors, not silent fallbacks."""
    assert lk.lk_gemv_kernel_for(4096, 4096, I8, 64, 0) == 3
    assert lk.lk_gemv_kernel_for(4096, 4096, I8, 65, 0) == 0
    assert lk.lk_gemv_kernel_for(4096, 4096, 0, 16, 0) == 0
    assert lk.lk_gemv_kernel_for(4096, 1056, I8, 16, 0) == 0
    assert lk.lk_gemv_kernel_for(4096, 4096, I8, 16, 2) == 3
    wq, ws = to_dev(np.zeros((64, 1056), np.int8)), to_dev(np.zeros((64, 33), np.uint16))
    x = to_dev(np.zeros((16, 1056), np.float32))
    y = torch.empty((16, 64), dtype=torch.float32, device=DEV)
    with pytest.raises(lk.LkError):
        lk.lk_gemv_q8(wq, ws, 0, y, x=x, M=16)


# ---- split-K on the tensor-core kernel -------------------------------------------------

@pytest.mark.parametrize("layout", ["f16", "f16-g4", "i8"])
@pytest.mark.parametrize("mode", [I8, TP])
@pytest.mark.parametrize("M", [2, 8, 33, 64])
@pytest.mark.parametrize("S", [2, 3, 8])
@pytest.mark.parametrize("N,K", [(1000, 1280), (300, 12288), (2500, 4096)])
def test_mma_splitk_matches_oracle(layout, mode, M, S, N, K):
    """lk_gemv_q8_splitk on the tensor-core kernel (each block holds only its
    chunk's columns of the activation rows): every chunk's partials bit for
    bit the oracle's chunks, including chunks that start 4 blocks past a
    16-byte scale boundary (S = 3), and the ascending combine bit for bit the
    oracle's split-K value; run to run identical."""
    cfg = mma(mma_i8=1 if layout == "i8" else 2, mma_group=4 if "g4" in layout else 1)
    if lk.lk_gemv_kernel_for(N, K, mode, M, S, cfg=cfg) != 3:
        pytest.skip("layout does not fit")
    wq, ws = synth.q8_matrix(N, K, 9300 + N + K)
    x = synth.activation(M, K, 9301 + M, outliers=True)
    y_or, ch_or = oracle.gemv_splitk(wq, ws, mode, S, **oracle_acts(x, mode))
    wq_d, ws_d, acts = to_dev(wq), to_dev(ws), dev_acts(x, mode)
    outs = []
    for _ in range(2):
        part = torch.full((S, M, N), float("nan"), dtype=torch.float32, device=DEV)
        lk.lk_gemv_q8_splitk(wq_d, ws_d, mode, S, part, M=M, cfg=cfg, **acts)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        lk.lk_splitk_combine(mode, part, S, M, N, y)
        torch.cuda.synchronize()
        assert lk.lk_device_error(reset=True) == 0
        assert np.array_equal(bits(host(part)), bits(ch_or))
        assert np.array_equal(bits(host(y)), bits(y_or))
        outs.append(host(y).copy())
    assert np.array_equal(bits(outs[0]), bits(outs[1]))


def test_mma_splitk_declines_empty_chunks():
    """A chunk with no block (S > K / 128) is not the tensor-core kernel's:
    up to 8 rows the other kernels take it (with its zero partials), past 8
    rows it is a shape error."""
    assert lk.lk_gemv_kernel_for(64, 256, I8, 8, 4) in (1, 2)
    assert lk.lk_gemv_kernel_for(64, 256, I8, 16, 4) == 0
    assert lk.lk_gemv_kernel_for(64, 1024, I8, 16, 8) == 3
    wq, ws = to_dev(np.zeros((64, 256), np.int8)), to_dev(np.zeros((64, 8), np.uint16))
    xq, xs = to_dev(np.zeros((16, 256), np.int8)), to_dev(np.zeros((16, 8), np.float32))
    part = torch.empty((4, 16, 64), dtype=torch.float32, device=DEV)
    with pytest.raises(lk.LkError):
        lk.lk_gemv_q8_splitk(wq, ws, I8, 4, part, xq=xq, xs=xs, M=16)
