"""Pins of the block-format oracle (oracle/formats.c) against things other
than itself: every format's decoder against an encoder written here from the
format's byte layout (random fields in, the same fields out), the Dequant GEMV
against an f64 brute force over the decoded weights, and the quantized modes
against hand-worked closed forms and a lane-order fixture (a value only the
pages' order -- sub-block sb in lane sb mod 32, then the shuffle-down tree --
gives)."""
import struct

import numpy as np
import pytest

import oracle

F = oracle.FORMATS
IQ4 = [-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113]
E2M1x2 = [0, 1, 2, 3, 4, 6, 8, 12, 0, -1, -2, -3, -4, -6, -8, -12]


def f16(x):
    return np.float16(x)


def h16(x):
    return struct.pack("<e", float(np.float16(x)))


def f32(x):
    return np.float32(x)


def pack_nibbles(lo16, hi16):
    """16 bytes: byte i = lo16[i] | hi16[i] << 4."""
    return bytes(int(a) | (int(b) << 4) for a, b in zip(lo16, hi16))


# ---- encoders: fields -> bytes, and the decode every format promises ----------------

def enc_32(fmt, r, tame=False):
    """One 32-value block: (bytes, levels[32], d[2], c[2]); tame: MXFP4
    exponents near 1 (sums stay finite)."""
    d = f16(r.uniform(0.01, 2.0) * r.choice([-1, 1]))
    c = [f32(0), f32(0)]
    if fmt in ("q4_0", "q4_1"):
        u = r.integers(0, 16, 32)
        payload = pack_nibbles(u[:16], u[16:])
        if fmt == "q4_0":
            return h16(d) + payload, u - 8, [f32(d)] * 2, c
        m = f16(r.uniform(-1, 1))
        return h16(d) + h16(m) + payload, u, [f32(d)] * 2, [f32(m)] * 2
    if fmt in ("q5_0", "q5_1"):
        u = r.integers(0, 32, 32)
        qh = sum(int(u[i] >> 4) << i for i in range(32))
        payload = struct.pack("<I", qh) + pack_nibbles(u[:16] & 15, u[16:] & 15)
        if fmt == "q5_0":
            return h16(d) + payload, u - 16, [f32(d)] * 2, c
        m = f16(r.uniform(-1, 1))
        return h16(d) + h16(m) + payload, u, [f32(d)] * 2, [f32(m)] * 2
    if fmt == "iq4_nl":
        n = r.integers(0, 16, 32)
        return h16(d) + pack_nibbles(n[:16], n[16:]), np.array([IQ4[i] for i in n]), [f32(d)] * 2, c
    if fmt == "mxfp4":
        e = int(r.integers(118, 139) if tame else r.integers(0, 256))
        n = r.integers(0, 16, 32)
        scale = f32(2.0 ** (e - 128))
        return bytes([e]) + pack_nibbles(n[:16], n[16:]), np.array([E2M1x2[i] for i in n]), [scale] * 2, c
    raise ValueError(fmt)


def enc_256(fmt, r):
    """One 256-value super-block: (bytes, levels[8][32], d[8][2], c[8][2])."""
    D = f16(r.uniform(0.001, 0.1))
    DM = f16(r.uniform(0.001, 0.1))
    lv = np.zeros((8, 32), np.int64)
    d = [[f32(0)] * 2 for _ in range(8)]
    c = [[f32(0)] * 2 for _ in range(8)]
    if fmt in ("q4_k", "q5_k"):
        sc = r.integers(0, 64, 8)
        mn = r.integers(0, 64, 8)
        s12 = bytearray(12)
        for j in range(4):
            s12[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
            s12[j + 4] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
            s12[8 + j] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
        top = 32 if fmt == "q5_k" else 16
        u = r.integers(0, top, (8, 32))
        qs = bytearray(128)
        qh = bytearray(32)
        for j in range(8):
            for l in range(32):
                qs[(j >> 1) * 32 + l] |= (int(u[j, l]) & 15) << (4 * (j & 1))
                if fmt == "q5_k":
                    qh[l] |= (int(u[j, l]) >> 4) << j
            lv[j] = u[j]
            d[j] = [f32(f32(D) * f32(sc[j]))] * 2
            c[j] = [f32(-(f32(DM) * f32(mn[j])))] * 2
        body = h16(D) + h16(DM) + bytes(s12) + (bytes(qh) if fmt == "q5_k" else b"") + bytes(qs)
        return body, lv, d, c
    if fmt == "q2_k":
        scm = r.integers(0, 256, 16)
        u = r.integers(0, 4, (8, 32))
        qs = bytearray(64)
        for j in range(8):
            half, k = j >> 2, j & 3
            for l in range(32):
                qs[half * 32 + l] |= int(u[j, l]) << (2 * k)
            lv[j] = u[j]
            for h in range(2):
                s = int(scm[half * 8 + k * 2 + h])
                d[j][h] = f32(f32(D) * f32(s & 15))
                c[j][h] = f32(-(f32(DM) * f32(s >> 4)))
        return bytes(int(v) for v in scm) + bytes(qs) + h16(D) + h16(DM), lv, d, c
    if fmt == "q3_k":
        s6 = r.integers(0, 64, 16)
        u = r.integers(-4, 4, (8, 32))
        hmask = bytearray(32)
        qs = bytearray(64)
        for j in range(8):
            half, k = j >> 2, j & 3
            for l in range(32):
                low2 = int(u[j, l]) & 3
                hbit = 1 if u[j, l] >= 0 else 0   # the mask bit set: +0, clear: -4
                qs[half * 32 + l] |= low2 << (2 * k)
                hmask[l] |= hbit << (half * 4 + k)
            lv[j] = u[j]
            for h in range(2):
                d[j][h] = f32(f32(D) * f32(int(s6[half * 8 + k * 2 + h]) - 32))
        s12 = bytearray(12)
        for i in range(16):
            if i < 8:
                s12[i] |= int(s6[i]) & 15
            else:
                s12[i - 8] |= (int(s6[i]) & 15) << 4
            s12[8 + (i & 3)] |= (int(s6[i]) >> 4) << (2 * (i >> 2))
        return bytes(hmask) + bytes(qs) + bytes(s12) + h16(D), lv, d, c
    if fmt == "q6_k":
        sc = r.integers(-128, 128, 16)
        u = r.integers(0, 64, (8, 32))
        ql = bytearray(128)
        qh = bytearray(64)
        for j in range(8):
            half, k = j >> 2, j & 3
            for l in range(32):
                lo4, hi2 = int(u[j, l]) & 15, int(u[j, l]) >> 4
                ql[half * 64 + (k & 1) * 32 + l] |= lo4 << (4 * (k >> 1))
                qh[half * 32 + l] |= hi2 << (2 * k)
            lv[j] = u[j] - 32
            d[j] = [f32(f32(D) * f32(sc[half * 8 + 2 * k])), f32(f32(D) * f32(sc[half * 8 + 2 * k + 1]))]
        return bytes(ql) + bytes(qh) + bytes(int(v) & 255 for v in sc) + h16(D), lv, d, c
    if fmt == "iq4_xs":
        ls = r.integers(0, 64, 8)
        n = r.integers(0, 16, (8, 32))
        sh = sum((int(ls[j]) >> 4) << (2 * j) for j in range(8))
        sl = bytearray(4)
        for j in range(8):
            sl[j >> 1] |= (int(ls[j]) & 15) << (4 * (j & 1))
        qs = b"".join(pack_nibbles(n[j, :16], n[j, 16:]) for j in range(8))
        for j in range(8):
            lv[j] = [IQ4[i] for i in n[j]]
            d[j] = [f32(f32(D) * f32(int(ls[j]) - 32))] * 2
        return h16(D) + struct.pack("<H", sh) + bytes(sl) + qs, lv, d, c
    raise ValueError(fmt)


def encode_row(fmt, K, r, tame=False):
    """A row of K values: (bytes as uint8 array, levels[K/32][32], d[K/32][2], c[K/32][2])."""
    parts, levels, ds, cs = [], [], [], []
    big = fmt.endswith("_k") or fmt == "iq4_xs"
    for _ in range(K // (256 if big else 32)):
        if big:
            b, lv, d, c = enc_256(fmt, r)
            levels += list(lv)
            ds += d
            cs += c
        else:
            b, lv, d, c = enc_32(fmt, r, tame)
            levels.append(lv)
            ds.append(d)
            cs.append(c)
        parts.append(b)
    raw = np.frombuffer(b"".join(parts), np.uint8)
    return raw, np.array(levels), np.array(ds, np.float32), np.array(cs, np.float32)


@pytest.mark.parametrize("fmt", sorted(F))
def test_decoder_returns_the_encoded_fields(fmt):
    r = np.random.default_rng(F[fmt])
    K = 512
    raw, levels, ds, cs = encode_row(fmt, K, r)
    assert raw.size == oracle.format_row_bytes(F[fmt], K)
    for sb in range(K // 32):
        v, d, c = oracle.sub_decode(F[fmt], raw, sb)
        assert np.array_equal(v.astype(np.int64), levels[sb]), (fmt, sb)
        assert np.array_equal(d.view(np.uint32), ds[sb].view(np.uint32)), (fmt, sb, d, ds[sb])
        assert np.array_equal(c.view(np.uint32), cs[sb].view(np.uint32)), (fmt, sb, c, cs[sb])
    # the dequantized row: RN(RN(d v) + c) per value
    w = oracle.dequant(F[fmt], raw[None], K)[0]
    want = np.array([f32(f32(ds[i // 32][(i % 32) // 16] * f32(levels[i // 32][i % 32]))
                         + ds.dtype.type(cs[i // 32][(i % 32) // 16])) for i in range(K)], np.float32)
    assert np.array_equal(w.view(np.uint32), want.view(np.uint32))


def test_row_bytes():
    assert oracle.format_row_bytes(F["q4_0"], 4096) == 128 * 18
    assert oracle.format_row_bytes(F["q6_k"], 4096) == 16 * 210
    assert oracle.format_row_bytes(F["q4_k"], 4000) == 0      # not whole super-blocks
    assert oracle.format_row_bytes(F["mxfp4"], 64) == 34
    assert oracle.format_row_bytes(99, 256) == 0


@pytest.mark.parametrize("fmt", sorted(F))
def test_dequant_gemv_is_the_f64_sum_of_the_decoded_weights(fmt):
    r = np.random.default_rng(100 + F[fmt])
    K, N = 1024, 5
    rows = [encode_row(fmt, K, r, tame=True)[0] for _ in range(N)]
    w = np.stack(rows)
    x = r.standard_normal((2, K)).astype(np.float32)
    y = oracle.gemv_blk(F[fmt], w, K, oracle.DEQUANT, x=x)
    wd = oracle.dequant(F[fmt], w, K).astype(np.float64)
    exact = x.astype(np.float64) @ wd.T
    mag = np.abs(x.astype(np.float64)) @ np.abs(wd).T
    assert np.all(np.abs(y - exact) <= 1e-7 * mag + 1e-30)
    assert np.allclose(oracle.absdot_blk(F[fmt], w, K, x), mag, rtol=1e-12)


def _q40_row(K, terms):
    """A Q4_0 row whose sub-block sb has scale d_sb and level 1 at value 0
    (levels 0 elsewhere): terms {sb: d_sb}."""
    blocks = []
    for sb in range(K // 32):
        u = np.full(32, 8)
        if sb in terms:
            u[0] = 9
        blocks.append(h16(terms.get(sb, 0.0)) + pack_nibbles(u[:16], u[16:]))
    return np.frombuffer(b"".join(blocks), np.uint8)


def test_quantized_term_closed_forms():
    """K = 32: y = s * part with part = d0 dh0 + c0 sh0 + d1 dh1 + c1 sh1, by
    hand; TwoPass adds 2^-7 of the low words' term."""
    u = np.full(32, 8)
    u[0], u[17] = 11, 3                      # levels 3 (value 0) and -5 (value 17)
    raw = np.frombuffer(h16(0.5) + pack_nibbles(u[:16], u[16:]), np.uint8)[None]
    hi = np.zeros((1, 32), np.int8)
    hi[0, 0], hi[0, 17], hi[0, 5] = 7, 2, 100
    s = np.array([[0.25]], np.float32)
    y = oracle.gemv_blk(F["q4_0"], raw, 32, oracle.INT8ACT, hi=hi, s=s)
    # dh0 = 3*7 + 0*100 = 21, dh1 = -5*2 = -10, c = 0: part = 0.5*21 + 0.5*(-10) = 5.5
    assert y[0, 0] == np.float32(0.25 * 5.5)
    lo = np.zeros((1, 32), np.int8)
    lo[0, 0] = 64
    y2 = oracle.gemv_blk(F["q4_0"], raw, 32, oracle.TWOPASS, hi=hi, lo=lo, s=s)
    # low term: 0.5 * 3 * 64 = 96, times 2^-7 = 0.75: part 6.25
    assert y2[0, 0] == np.float32(0.25 * 6.25)
    # the offset: Q4_1 with m = -1, levels 2 everywhere, hi = 1 on the first half
    u = np.full(32, 2)
    raw1 = np.frombuffer(h16(0.5) + h16(-1.0) + pack_nibbles(u[:16], u[16:]), np.uint8)[None]
    h1 = np.zeros((1, 32), np.int8)
    h1[0, :16] = 1
    y3 = oracle.gemv_blk(F["q4_1"], raw1, 32, oracle.INT8ACT, hi=h1, s=np.ones((1, 1), np.float32))
    # d0 dh0 + c0 sh0 = 0.5 * 32 + (-1) * 16 = 0
    assert y3[0, 0] == np.float32(0.0)


def test_lane_order_fixture():
    """Terms 2^-24 at sub-blocks 0 and 16 (lanes 0 and 16) and 1.0 at
    sub-block 1 (lane 1): the shuffle-down tree adds lane 16 into lane 0
    first (2^-23), then lane 1, giving 1 + 2^-23; summing the sub-blocks in
    ascending order would give 1.0 (1 + 2^-24 ties to even, twice)."""
    K = 1024
    raw = _q40_row(K, {0: 2.0 ** -10, 16: 2.0 ** -10, 1: 1.0})[None]
    hi = np.zeros((1, K), np.int8)
    hi[0, ::32] = 1                          # value 0 of every sub-block
    s = np.ones((1, K // 32), np.float32)
    s[0, 0] = s[0, 16] = 2.0 ** -14
    y = oracle.gemv_blk(F["q4_0"], raw, K, oracle.INT8ACT, hi=hi, s=s)
    assert y[0, 0] == np.float32(1 + 2.0 ** -23)


@pytest.mark.parametrize("fmt", sorted(F))
def test_quantized_gemv_within_f32_rounding_of_the_exact_sum(fmt):
    """Int8Act: y within (nb + 40) * 2^-24 * sum|terms| of the exact sum of
    s * (d * level + c) * word over the row (catches a dropped term, a wrong
    sign or index)."""
    r = np.random.default_rng(200 + F[fmt])
    K, N = 1024, 3
    w = np.stack([encode_row(fmt, K, r, tame=True)[0] for _ in range(N)])
    x = r.standard_normal((1, K)).astype(np.float32)
    hi, lo, s = oracle.quantize(x, oracle.INT8ACT)
    y = oracle.gemv_blk(F[fmt], w, K, oracle.INT8ACT, hi=hi, s=s)
    for o in range(N):
        ex = 0.0
        mag = 0.0
        for sb in range(K // 32):
            v, d, c = oracle.sub_decode(F[fmt], w[o], sb)
            for i in range(32):
                t = float(s[0, sb]) * (float(d[i // 16]) * int(v[i]) + float(c[i // 16])) * int(hi[0, 32 * sb + i])
                ex += t
                mag += abs(t)
        assert abs(float(y[0, o]) - ex) <= (K // 32 + 40) * 2.0 ** -24 * mag + 1e-30, (fmt, o)
