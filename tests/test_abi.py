"""The C-ABI library builds for sm_103a, loads, exports every entry point that
include/lk.h declares, and rejects bad arguments on the host before any
launch.  No GPU: only host-side validation paths are called (the pointers
below are never dereferenced)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

torch = pytest.importorskip("torch")

from q8_quantized_gemv_gb300 import build, lk  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    build.build()
    return lk._load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "lk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lk_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(lk.exported_symbols()) == names


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lk.lk_status_string(code) != "unknown status"
    assert lk.lk_version() >= 100


FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


def P(v):
    return ctypes.c_void_p(v)


def test_gemv_argument_checks(lib):
    g = lib.lk_gemv_q8
    ok_ptrs = dict(wq=P(FAKE), ws=P(FAKE), x=P(FAKE), xq=P(FAKE), xl=P(FAKE), xs=P(FAKE), y=P(FAKE))

    def call(N=64, K=64, mode=1, M=1, cfg=None, **kw):
        a = dict(ok_ptrs, **kw)
        return g(a["wq"], a["ws"], N, K, mode, a["x"], a["xq"], a["xl"], a["xs"], M, a["y"], None, None,
                 lk._cfg(cfg), None)

    assert call(K=48) == -3             # K % 32
    assert call(M=9) == -3              # M > LK_MAX_M
    assert call(N=-1) == -3
    assert call(mode=3) == -1
    assert call(wq=None) == -1
    assert call(mode=2, xl=None) == -1  # TwoPass needs the low words
    assert call(mode=0, x=None) == -1   # Dequant needs f32 x
    assert call(wq=P(FAKE + 8)) == -2   # 16-byte rows
    assert call(xq=P(FAKE + 4)) == -2
    assert call(xs=P(FAKE + 2)) == -2
    assert call(mode=0, x=P(FAKE + 4)) == -2
    assert call(N=0) == 0 and call(M=0) == 0  # empty problems launch nothing
    # argmax parts need the host count pointer
    a = ok_ptrs
    assert g(a["wq"], a["ws"], 64, 64, 1, None, a["xq"], None, a["xs"], 1, a["y"], P(FAKE), None,
             None, None) == -1
    # launch settings out of range, checked before anything else
    for bad in (dict(pdl=2), dict(pdl=-1), dict(prefill=-1), dict(prefill=17), dict(path=4), dict(grid_ctas=-1),
                dict(ring_tk=512), dict(ring_tk=9216), dict(mma_min_m=66), dict(mma_tk=100), dict(mma_tk=8448),
                dict(mma_warps=17), dict(mma_depth=9), dict(mma_i8=3), dict(mma_group=2), dict(mma_act16=3)):
        assert call(cfg=lk.launch_cfg(**bad)) == -1, bad
    for good in (dict(pdl=1), dict(prefill=16), dict(path=3), dict(ring_tk=8192), dict(mma_min_m=65),
                 dict(mma_tk=8192), dict(mma_group=4), dict(mma_i8=2), dict(mma_act16=2)):
        assert call(N=0, cfg=lk.launch_cfg(**good)) == 0, good
    # argmax keys are sized by lk_argmax_parts_max: no more blocks than that
    big = lk.launch_cfg(grid_ctas=lk.lk_argmax_parts_max(64) + 1)
    assert g(a["wq"], a["ws"], 64, 64, 1, None, a["xq"], None, a["xs"], 1, a["y"], P(FAKE),
             ctypes.byref(ctypes.c_int(0)), lk._cfg(big), None) == -1


def test_splitk_and_combine_checks(lib):
    f = lib.lk_gemv_q8_splitk
    args = [P(FAKE), P(FAKE), 64, 256, 1, None, P(FAKE), None, P(FAKE), 1]
    need = lk.lk_splitk_workspace_bytes(1, 4, 1, 64)
    assert need == 4 * 64 * 4
    assert lk.lk_splitk_workspace_bytes(0, 4, 2, 64) == 4 * 2 * 64 * 8
    assert f(*args, 0, P(FAKE), need, None, None) == -3
    assert f(*args, 65, P(FAKE), need, None, None) == -3
    assert f(*args, 4, P(FAKE), need - 1, None, None) == -4
    assert f(*args, 4, None, need, None, None) == -1
    assert f(*args, 4, P(FAKE), need, lk._cfg(lk.launch_cfg(pdl=3)), None) == -1
    c = lib.lk_splitk_combine
    assert c(1, P(FAKE), 0, 1, 64, P(FAKE), None, None) == -3
    assert c(1, P(FAKE), 2, 65, 64, P(FAKE), None, None) == -3  # M <= LK_MAX_BATCH
    assert c(0, P(FAKE + 4), 2, 1, 64, P(FAKE), None, None) == -2  # f64 partials
    assert c(1, P(FAKE), 2, 0, 64, P(FAKE), None, None) == 0
    assert c(1, P(FAKE), 2, 1, 64, P(FAKE), lk._cfg(lk.launch_cfg(pdl=5)), None) == -1


def test_norm_quant_argmax_checks(lib):
    r = lib.lk_rmsnorm_quant
    assert r(P(FAKE), P(FAKE), 1, 33, 1e-6, 1, None, P(FAKE), None, P(FAKE), None, None) == -3
    assert r(P(FAKE), P(FAKE), 1, 64, 1e-6, 0, None, None, None, None, None, None) == -1  # Dequant needs xn
    assert r(P(FAKE), P(FAKE), 1, 64, 1e-6, 2, None, P(FAKE), None, P(FAKE), None, None) == -1
    assert r(P(FAKE), P(FAKE), 1, 64, 1e-6, 1, None, P(FAKE), None, P(FAKE), lk._cfg(lk.launch_cfg(pdl=2)),
             None) == -1
    q = lib.lk_quantize_act
    assert q(P(FAKE), 1, 64, 0, P(FAKE), None, P(FAKE), None, None) == -1  # nothing to quantize
    assert q(P(FAKE), 65, 64, 1, P(FAKE), None, P(FAKE), None, None) == -3  # M <= LK_MAX_BATCH
    assert q(P(FAKE), 1, 64, 1, P(FAKE), None, P(FAKE), lk._cfg(lk.launch_cfg(prefill=-1)), None) == -1
    a = lib.lk_argmax
    assert a(P(FAKE), None, 0, 1, 0, P(FAKE), P(FAKE), None) == -3  # N >= 1
    assert a(P(FAKE), None, 0, 1, 10, P(FAKE), None, None) == -1    # logits form needs scratch
    assert a(None, P(FAKE), 0, 1, 10, P(FAKE), None, None) == -3    # parts form needs n_parts
    assert [lk.lk_argmax_scratch_entries(n) for n in (1, 2048, 2049, 151936, 10 ** 8)] == [1, 1, 2, 64, 64]
    assert lk.lk_argmax_parts_max(151936) >= (151936 + 31) // 32


def test_kernel_choice_without_gpu(lib):
    # invalid shapes and settings answer 0 before any device query
    assert lk.lk_gemv_kernel_for(64, 48, 1, 1, 0) == 0
    assert lk.lk_gemv_kernel_for(64, 64, 1, 9, 0) == 0      # past 8 rows: the tensor-core path only
    assert lk.lk_gemv_kernel_for(4096, 4096, 1, 65, 0) == 0  # past LK_MAX_BATCH
    assert lk.lk_gemv_kernel_for(64, 4096, 1, 1, 0, cfg=lk.launch_cfg(path=5)) == 0
    assert lk.lk_gemv_kernel_for(64, 4096, 1, 1, 0, cfg=lk.launch_cfg(path="direct")) == 1


def test_launch_cfg_fields():
    c = lk.launch_cfg(pdl=1, path="mma", mma_group=4)
    assert (c.pdl, c.prefill, c.path, c.mma_group, c.grid_ctas) == (1, 0, 3, 4, 0)
    assert ctypes.sizeof(lk.LkLaunchCfg) == 4 * len(lk.CFG_FIELDS)
    with pytest.raises(TypeError):
        lk.launch_cfg(gemv_path=1)


def test_options(lib):
    """Two diagnostic options remain; every launch setting is per call."""
    assert lk.lk_get_option("trace") == 0 and lk.lk_get_option("wait_us") == 0
    lk.lk_set_option("wait_us", 2000)
    assert lk.lk_get_option("wait_us") == 2000
    lk.lk_set_option("wait_us", 0)
    for name, bad in (("trace", 4), ("trace", -1), ("wait_us", -1), ("wait_us", 60000001)):
        with pytest.raises(lk.LkError):
            lk.lk_set_option(name, bad)
    for gone in ("gemv_path", "pdl", "mma_i8", "ring_prefill", "grid_ctas", "no_such_option"):
        with pytest.raises(lk.LkError):
            lk.lk_set_option(gone, 0)
        assert lk.lk_get_option(gone) == -1


def test_group_argument_checks(lib):
    g = lib.lk_gemv_q8_group

    def targets(*specs):
        arr = (lk.LkGemvTarget * max(1, len(specs)))(*[lk.LkGemvTarget(w, s, n, 0, y) for w, s, n, y in specs])
        return ctypes.cast(arr, ctypes.c_void_p)

    good = (FAKE, FAKE, 64, FAKE)

    def call(ts, n, K=256, mode=1, M=8, xq=P(FAKE), xl=P(FAKE), xs=P(FAKE)):
        return g(ts, n, K, mode, None, xq, xl, xs, M, None, None)

    assert call(None, 1) == -1                            # no targets
    assert call(targets(good), 0) == -1                   # n out of range
    assert call(targets(*[good] * 5), 5) == -1
    assert call(targets(good, (FAKE, FAKE, 64, None)), 2) == -1     # null y
    assert call(targets(good, (FAKE + 8, FAKE, 64, FAKE)), 2) == -2  # misaligned levels
    assert call(targets(good, (FAKE, FAKE, 0, FAKE)), 2) == -3       # an empty matrix
    assert call(targets(good), 1, K=48) == -3             # K % 32
    assert call(targets(good), 1, M=9) == -3
    assert call(targets(good), 1, mode=2, xl=None) == -1  # TwoPass needs the low words


def test_add_rmsnorm_quant_checks(lib):
    f = lib.lk_add_rmsnorm_quant
    n = 4 * 256  # M x K floats

    def call(x=FAKE, r=FAKE + 16 * n, g=FAKE + 32 * n, M=4, K=256, mode=1, s=FAKE + 48 * n, xn=None,
             xq=FAKE + 64 * n, xl=None, xs=FAKE + 80 * n):
        return f(P(x), P(r) if r else None, P(g) if g else None, M, K, 1e-6, mode, P(s) if s else None,
                 P(xn) if xn else None, P(xq) if xq else None, P(xl) if xl else None, P(xs) if xs else None, None,
                 None)

    assert call(K=48) == -3
    assert call(M=65) == -3
    assert call(mode=3) == -1
    assert call(r=None) == -1 and call(g=None) == -1
    assert call(xq=None) == -1                  # the quantized output is required
    assert call(mode=2) == -1                   # TwoPass needs the low words
    assert call(mode=0) == -1                   # Dequant needs the normed rows
    assert call(x=FAKE + 2) == -2
    assert call(s=FAKE + 2) == -2
    # the new residual stream may not overlap either operand
    assert call(s=FAKE) == -1
    assert call(s=FAKE + 4 * n - 4) == -1       # last element of x
    assert call(s=FAKE + 16 * n + 8) == -1      # inside r
    assert call(M=0) == 0 and call(K=0) == 0


def test_swiglu_quant_checks(lib):
    f = lib.lk_swiglu_quant

    def call(gate=FAKE, up=FAKE + 4096, M=2, F=1024, ld=2048, mode=1, h=None, hq=FAKE + 65536, hl=None,
             hs=FAKE + 131072):
        return f(P(gate) if gate else None, P(up) if up else None, M, F, ld, mode, P(h) if h else None,
                 P(hq) if hq else None, P(hl) if hl else None, P(hs) if hs else None, None, None)

    assert call(F=48) == -3                     # F % 32
    assert call(ld=512) == -3                   # pitch below the row length
    assert call(M=65) == -3
    assert call(mode=5) == -1
    assert call(gate=None) == -1
    assert call(mode=0) == -1                   # Dequant needs h
    assert call(mode=2) == -1                   # TwoPass needs the low words
    assert call(hq=None) == -1
    assert call(hs=FAKE + 2) == -2
    assert call(M=0) == 0 and call(F=0) == 0
