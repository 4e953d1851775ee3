"""The launch-timeline trace (option "trace" 3): every norm, quantize and GEMV
launch of a token writes one record, in launch order, with consistent
timestamps; and the records do not change the results."""
import pytest

torch = pytest.importorskip("torch")

from q8_quantized_gemv_gb300 import build, lk  # noqa: E402
from q8_quantized_gemv_gb300.decode import DecodeStack  # noqa: E402

pytestmark = pytest.mark.gpu

SMALL = dict(layers=2, hidden=1024, q_dim=1024, kv_dim=256, ffn=1536, vocab=3000)
KINDS = {1: "ring", 2: "chain", 3: "tensor-core", 4: "norm", 5: "quantize", 6: "split-K combine"}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield
    lk.lk_set_option("trace", 0)


@pytest.mark.parametrize("batch", [1, 8])
def test_timeline_records(batch):
    st = DecodeStack(**SMALL, batch=batch, mode=1, glu=False)
    st.run_token()
    torch.cuda.synchronize()
    ref = st.logits.clone()
    lk.lk_set_option("trace", 3)
    try:
        st.run_token()
        torch.cuda.synchronize()
    finally:
        lk.lk_set_option("trace", 0)
    assert torch.equal(st.logits.view(torch.int32), ref.view(torch.int32))
    raw = lk.lk_trace_read(4096)
    # one record per traced launch (all but the argmax reduce), in launch order
    n = st.launches_per_token() - 1
    R = lk.LK_TRACE_REC
    used = [raw[i * R:(i + 1) * R] for i in range(n)]
    gemv = 1 if batch == 1 else 3
    assert (batch == 1) == (not st.splitk)  # split-K: 2 or more rows

    def g(name):  # one GEMV (over the fused q|k|v matrix for "qkv"), and its combine if split
        return [gemv] + ([6] if name in st.splitk else [])

    layer = [4] + g("qkv") + [5] + g("o") + [4] + g("gu") + [5] + g("down")
    want = layer * SMALL["layers"] + [4, gemv]
    assert [r[5] for r in used] == want
    assert [r[6] for r in used if r[5] == 4] == [SMALL["hidden"]] * (2 * SMALL["layers"] + 1)
    for r in used:
        assert r[5] in KINDS
        assert r[0] <= r[1] <= r[3]                  # start, past the wait, last block's end
        assert r[0] <= r[4] <= r[3]                  # block 0's end
        if r[5] in (1, 2, 3):
            assert r[1] <= r[2] <= r[4]              # activation ready before block 0 ends
    starts = [r[0] for r in used]
    ends = [r[3] for r in used]
    # launch order: each launch ends no earlier than its predecessor starts
    assert all(ends[i] >= starts[i - 1] for i in range(1, len(used)))


def test_timeline_records_glu_token():
    """The decoder dataflow at batch 1: first norm, then per layer q/k/v,
    quantize, o, add+norm, the gate/up pair with its SwiGLU epilogue (one ring
    launch), down, add+norm; then the lm-head."""
    st = DecodeStack(**SMALL, batch=1, mode=1, glu=True)
    assert st.glu and st.glu_launches() == 1
    st.run_token()
    torch.cuda.synchronize()
    ref = st.logits.clone()
    lk.lk_set_option("trace", 3)
    try:
        st.run_token()
        torch.cuda.synchronize()
    finally:
        lk.lk_set_option("trace", 0)
    assert torch.equal(st.logits.view(torch.int32), ref.view(torch.int32))
    raw = lk.lk_trace_read(4096)
    n = st.launches_per_token() - 1
    kinds = [raw[i * lk.LK_TRACE_REC + 5] for i in range(n)]
    assert kinds == [4] + [1, 5, 1, 4, 1, 1, 4] * SMALL["layers"] + [1]
