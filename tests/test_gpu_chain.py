"""The GEMV chain (a whole token's projections in one cooperative launch)
against the per-launch path and the CPU oracle, on a small synthetic decoder
(3 layers, hidden 1024) under every mode and batch 1 / 3; run-to-run
identity; and the bounded grid barrier's failure path."""
import pytest

torch = pytest.importorskip("torch")

from gpuhelp import check_token, run_token_capture  # noqa: E402
from q8_quantized_gemv_gb300 import build, lk  # noqa: E402
from q8_quantized_gemv_gb300.decode import DecodeStack  # noqa: E402

pytestmark = pytest.mark.gpu

SMALL = dict(layers=3, hidden=1024, q_dim=1024, kv_dim=256, ffn=1536, vocab=3000)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield
    lk.lk_set_option("wait_us", 0)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("batch", [1, 3])
def test_chain_matches_launches_and_oracle(mode, batch, fused):
    """The chain against the per-launch sequence, with separate norm/quantize
    launches (fused False) or the GEMVs' own prologue (True); the per-launch
    token's every GEMV against the oracle on its own input (bit for bit in
    the quantized modes, within 1e-5 * sum|W x| per row under Dequant)."""
    a = DecodeStack(**SMALL, batch=batch, mode=mode, chain=True)
    # (split-K off: the chain runs every GEMV unsplit)
    b = DecodeStack(**SMALL, batch=batch, mode=mode, chain=False, fused=fused, glu=False, splitk=False)
    assert a.chain is not None and b.chain is None
    ia = a.run_token().clone()
    layers, final = run_token_capture(b)
    ib = b.idx.clone()
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) == 0
    check_token(b, layers, final)
    # the chain is the same arithmetic as the per-launch fused path: same bits
    for name in ("q", "k", "v", "o", "gu"):
        assert torch.equal(a.out[name].view(torch.int32), b.out[name].view(torch.int32)), name
    assert torch.equal(a.h.view(torch.int32), b.h.view(torch.int32))
    assert torch.equal(a.logits.view(torch.int32), b.logits.view(torch.int32))
    assert torch.equal(ia, ib)
    # run to run
    for _ in range(2):
        a.run_token()
        torch.cuda.synchronize()
        assert torch.equal(a.logits.view(torch.int32), b.logits.view(torch.int32))


def test_chain_in_cuda_graph():
    a = DecodeStack(**SMALL, batch=1, mode=1, chain=True)
    a.run_token()
    torch.cuda.synchronize()
    ref = a.logits.clone()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        a.run_token()
    for _ in range(3):
        a.logits.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(a.logits.view(torch.int32), ref.view(torch.int32))


def test_chain_barrier_timeout_is_reported_and_recoverable():
    a = DecodeStack(**SMALL, batch=1, mode=1, chain=True)
    a.run_token()
    torch.cuda.synchronize()
    ref = a.logits.clone()
    lk.lk_device_error(reset=True)
    # a sync counter that can never reach "last arrival": every barrier wait
    # runs out (2 ms), the blocks drain their copies and exit
    lk.lk_set_option("wait_us", 2000)
    a.chain.sync[0] = 0x40000000
    a.run_token()
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) != 0
    # zeroed again, the chain runs normally in the same context
    a.chain.sync.zero_()
    lk.lk_set_option("wait_us", 0)
    a.logits.zero_()
    a.run_token()
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) == 0
    assert torch.equal(a.logits.view(torch.int32), ref.view(torch.int32))


@pytest.mark.parametrize("prefill", [0, 1, 12])
@pytest.mark.parametrize("fused", [False, True])
def test_pdl_graph_replays_identical(fused, prefill):
    """A captured token with programmatic dependent launches, replayed many
    times, gives the bits of the plain launches every time, with any number
    of warps filling before the dependency wait: every kernel's reads of what
    the kernel before it wrote come after that kernel is complete (the
    dependent starts early and must not read such data through a cache that
    can hold lines from before)."""
    every = ("q", "k", "v", "qkv", "o", "gu", "down", "lm")
    a = DecodeStack(**SMALL, batch=1, mode=1, chain=False, fused=fused, pdl=False,
                    prefill={n: prefill for n in every} if prefill else None)
    a.run_token()
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in list(a.out.items()) + [("h", a.h), ("logits", a.logits)]}
    a.pdl = True
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        a.run_token()
    for r in range(60):
        a.logits.zero_()
        a.h.zero_()
        g.replay()
        torch.cuda.synchronize()
        got = {k: v for k, v in list(a.out.items()) + [("h", a.h), ("logits", a.logits)]}
        for k in ref:
            assert torch.equal(got[k].view(torch.int32), ref[k].view(torch.int32)), (r, k)
    assert lk.lk_device_error(reset=True) == 0


@pytest.mark.parametrize("fused_qkv", [False, True])
@pytest.mark.parametrize("fused", [False, True])
def test_grouped_qkv_pdl_graph_matches_plain(fused, fused_qkv):
    """The per-launch sequence with q, k, v in one launch -- one GEMV over the
    fused q|k|v matrix, or one grouped launch over three matrices -- after one
    norm launch or with the fused prologue: captured with programmatic
    dependent launches in a graph, it gives the same bits as launched plainly,
    and the oracle's token."""
    a = DecodeStack(**SMALL, batch=1, mode=1, chain=False, fused=fused, fused_qkv=fused_qkv)
    assert (a.qkv is not None) == (fused and not fused_qkv) and a.qkv_one == fused_qkv
    layers, final = run_token_capture(a)
    check_token(a, layers, final)
    ref = a.logits.clone()
    a.pdl = True
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        a.run_token()
    for _ in range(3):
        a.logits.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(a.logits.view(torch.int32), ref.view(torch.int32))
    assert lk.lk_device_error(reset=True) == 0
