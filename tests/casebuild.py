"""Builders for the hand-worked fixtures in tests/golden (inputs only; the
expected values are the fixtures' own)."""
import numpy as np

from conftest import read_golden

MODES = {"dequant": 0, "int8act": 1, "twopass": 2}


def f16_bits(v):
    return np.array(v, dtype=np.float16).view(np.uint16)


def parse_scale(tok):
    if tok.startswith("2^"):
        return float(2 ** int(tok[2:]))
    return float(tok)


def block_case(K, blocks, pad_to=None):
    """Inputs of an order example: every block's activation group is
    [127,127,127,127,4,1,0,...] (s = 1 and hi = the values); a block listed
    as b:scale:d gets weight levels giving dot d and that f16 scale; other
    blocks have zero weights and scale 1.  pad_to appends zero-weight blocks
    up to that K (each adds an exact zero step, so the results do not change)."""
    K = max(K, pad_to or 0)
    nb = K // 32
    x = np.zeros((1, K), np.float32)
    wq = np.zeros((1, K), np.int8)
    sc = np.ones(nb, np.float32)
    for b in range(nb):
        x[0, 32 * b: 32 * b + 6] = [127, 127, 127, 127, 4, 1]
    for item in blocks.split():
        b, s, d = item.split(":")
        b, d = int(b), int(d)
        sc[b] = parse_scale(s)
        if d == 512:
            wq[0, 32 * b: 32 * b + 5] = 1
        elif d == -512:
            wq[0, 32 * b: 32 * b + 5] = -1
        elif d == 1:
            wq[0, 32 * b + 5] = 1
        else:
            raise ValueError(d)
    return wq, f16_bits(sc).reshape(1, nb), x


def lo_case(rec, pad_to=None):
    K = max(int(rec["K"]), pad_to or 0)
    x = np.zeros((1, K), np.float32)
    act = [float(v) for v in rec["act"].split()]
    x[0, : len(act)] = act
    wq = np.zeros((1, K), np.int8)
    w = [int(v) for v in rec["w"].split()]
    wq[0, : len(w)] = w
    ws = f16_bits(np.full(K // 32, parse_scale(rec["scale"]), np.float32)).reshape(1, K // 32)
    return wq, ws, x


def quantizer_records():
    out = []
    for rec in read_golden("quantizer_examples.txt"):
        vals = [float(v) for v in rec["values"].split()]
        x = np.zeros((1, 32), np.float32)
        x[0, : len(vals)] = vals
        hi = [int(v) for v in rec["hi"].split()]
        lo = [int(v) for v in rec["lo"].split()] if "lo" in rec else None
        out.append(dict(name=rec["name"], mode=MODES[rec["mode"]], x=x, n=len(vals),
                        s_bits=int(rec["s_bits"], 16), hi=hi, lo=lo))
    return out


def order_records():
    return {rec["name"]: rec for rec in read_golden("order_examples.txt")}
