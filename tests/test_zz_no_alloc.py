"""The allocation-free argmax entry point (lk_argmax_noalloc), called
through the C ABI, against the existing lk_argmax with a caller scratch
buffer, on two calls in a row.  It is for callers that cannot allocate
device memory where they call it (for example inside CUDA-graph capture);
its partial keys live in a fixed device array inside the library.  This file
is collected last; it must pass alone in a fresh process and after the
other tests."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from q8_quantized_gemv_gb300 import build, lk
    build.build()
    return lk


def call_noalloc(lk, logits, idx):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    M, N = logits.shape
    return lk._load().lk_argmax_noalloc(ctypes.c_void_p(logits.data_ptr()), M, N,
                                        ctypes.c_void_p(idx.data_ptr()), stream)


def call_scratch(lk, logits, idx):
    M, N = logits.shape
    scratch = torch.zeros((M * lk.lk_argmax_scratch_entries(N),), dtype=torch.int64, device="cuda")
    lk.lk_argmax(idx, M, N, logits=logits, scratch=scratch)


@pytest.mark.parametrize("M,N", [(1, 151936), (8, 5000), (3, 1), (2, 2049)])
def test_noalloc_argmax_matches_scratch_version_twice(lib, M, N):
    lk = lib
    r = np.random.default_rng(M * 100003 + N)
    for call in range(2):  # two calls in a row share (and overwrite) the fixed array
        lg = r.standard_normal((M, N)).astype(np.float32)
        if N > 10:
            for t in range(M):
                lg[t, r.choice(N, 3, replace=False)] = lg[t].max() + 1.0  # planted ties
        logits = torch.from_numpy(lg).cuda()
        want = torch.full((M,), -1, dtype=torch.int32, device="cuda")
        got = torch.full((M,), -2, dtype=torch.int32, device="cuda")
        call_scratch(lk, logits, want)
        assert call_noalloc(lk, logits, got) == 0, f"call {call}"
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"call {call}: {got.tolist()} != {want.tolist()}"
        assert got.tolist() == [int(np.argmax(lg[t])) for t in range(M)]


def test_noalloc_argmax_rejects_bad_sizes(lib):
    lk = lib
    logits = torch.zeros((9, 10), device="cuda")
    idx = torch.zeros((9,), dtype=torch.int32, device="cuda")
    assert call_noalloc(lk, logits, idx) == -3  # M above LK_MAX_M
