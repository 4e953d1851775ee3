"""Parity of whole decode tokens at the benchmark's size: the synthetic
36-layer, hidden-4096 decoder (q 4096x4096, k and v 1024x4096, o 4096x4096,
gate/up 2 x 12288x4096, down 4096x12288, lm-head 151936x4096 with the
argmax) at batch 1 and 8, in the decoder dataflow (residual adds, norms,
SwiGLU) and in the projections-alone one.  Every output of every layer --
q, k, v, o, gate and up, the SwiGLU and its quantized words, down, the
residual stream -- and the logits and argmax are compared with the oracle,
each step on its own input: bit for bit under Int8Act and TwoPass (the norms
and residual adds in every mode), within 1e-5 * sum|W x| per row under
Dequant, the SwiGLU within a few ulp.  The same token replayed the way the
benchmark times it (one CUDA graph, programmatic dependent launches) must
give the same bits as the plain launches."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gpuhelp import check_token, host, run_token_capture  # noqa: E402
from q8_quantized_gemv_gb300 import build, lk  # noqa: E402
from q8_quantized_gemv_gb300.decode import DecodeStack  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield
    torch.cuda.empty_cache()


def _final_bits(st):
    bufs = dict(st.out, logits=st.logits)
    if st.glu:
        bufs.update(h0=st.hbuf[0], h1=st.hbuf[1], gu=st.gu_buf, hglu=st.hglu)
    else:
        bufs["h"] = st.h
    outs = {n: host(t).view(np.uint32).copy() for n, t in bufs.items()}
    outs["idx"] = host(st.idx).copy()
    return outs


@pytest.mark.parametrize("mode,batch,glu", [(1, 1, True), (2, 1, True), (0, 1, True), (1, 8, True), (2, 8, True),
                                            (1, 1, False), (2, 8, False)],
                         ids=["int8act-b1", "twopass-b1", "dequant-b1", "int8act-b8", "twopass-b8",
                              "int8act-b1-projections", "twopass-b8-projections"])
def test_full_decode_token_matches_oracle(mode, batch, glu):
    st = DecodeStack(batch=batch, mode=mode, glu=glu)  # the benchmark's 36-layer configuration
    try:
        layers, final = run_token_capture(st)
        assert lk.lk_device_error(reset=True) == 0
        check_token(st, layers, final)
        plain = _final_bits(st)
        # the benchmark's form: one graph per token, every launch a
        # programmatic dependent of the one before
        st.pdl = True
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            st.run_token()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            st.run_token()
        for _ in range(3):
            st.logits.zero_()
            st.h.zero_()
            g.replay()
            torch.cuda.synchronize()
            got = _final_bits(st)
            for k in plain:
                assert np.array_equal(got[k], plain[k]), k
        assert lk.lk_device_error(reset=True) == 0
    finally:
        del st
        torch.cuda.empty_cache()
