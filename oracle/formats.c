/*
 * Block-format oracle: the GGUF block formats other than Q8_0 that the
 * "kernels.rs" decoder library (lk_sub, lk_row_dot, lk_sub_dot) runs
 * through the same projection path.  TEST INFRASTRUCTURE ONLY, like
 * oracle.c (built into the same liboracle.so with -ffp-contract=off): every
 * product and sum below is rounded on its own, in IEEE single or double
 * precision as stated.  Shares no code or table with the CUDA path.
 *
 * Formats (the ggml type numbers the pages use as F), bytes per block:
 *   2 Q4_0    32 values, 18 B: f16 d, 16 B of 4-bit levels (level - 8)
 *   3 Q4_1    32 values, 20 B: f16 d, f16 m, 16 B of 4-bit levels (c = m)
 *   6 Q5_0    32 values, 22 B: f16 d, 32 high bits, 16 B of low nibbles (level - 16)
 *   7 Q5_1    32 values, 24 B: f16 d, f16 m, 32 high bits, 16 B low nibbles (c = m)
 *  20 IQ4_NL  32 values, 18 B: f16 d, 16 B of indices into 16 non-linear levels
 *  39 MXFP4   32 values, 17 B: an E8M0 exponent byte, 16 B of E2M1 codes
 *  10 Q2_K   256 values, 84 B: 16 scale|min bytes, 64 B of 2-bit levels, f16 d, f16 dmin
 *  11 Q3_K   256 values, 110 B: 32 B high-bit mask, 64 B of 2-bit levels,
 *            12 B of sixteen 6-bit scales, f16 d
 *  12 Q4_K   256 values, 144 B: f16 d, f16 dmin, 12 B of eight 6-bit scales
 *            and mins, 128 B of 4-bit levels
 *  13 Q5_K   256 values, 176 B: as Q4_K plus 32 B of fifth bits before the levels
 *  14 Q6_K   256 values, 210 B: 128 B low nibbles, 64 B of 2-bit highs, 16
 *            signed 8-bit scales, f16 d
 *  23 IQ4_XS 256 values, 136 B: f16 d, 16-bit high scale bits, 4 B of low
 *            scale nibbles, 128 B of indices into the IQ4_NL levels
 * Every format is read as 32-value sub-blocks: int8 levels v[0..31] and, per
 * half (values 0..15, 16..31), a scale d[h] and an offset c[h]; the weight
 * is RN(RN(d[h] v[i]) + c[h]) in f32 ("as the CPU dequantizer rounds it").
 * The byte layouts are the formats' own (an interface: a decoder must read
 * exactly these bits); the code below is written from them.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

float oracle_half_to_float(uint16_t h); /* oracle.c */

/* Values and bytes of one block of format F (0, 0 for an unknown F). */
static int fmt_block(int F, int* values)
{
    switch (F) {
        case 2: *values = 32; return 18;
        case 3: *values = 32; return 20;
        case 6: *values = 32; return 22;
        case 7: *values = 32; return 24;
        case 20: *values = 32; return 18;
        case 39: *values = 32; return 17;
        case 10: *values = 256; return 84;
        case 11: *values = 256; return 110;
        case 12: *values = 256; return 144;
        case 13: *values = 256; return 176;
        case 14: *values = 256; return 210;
        case 23: *values = 256; return 136;
        default: *values = 0; return 0;
    }
}

/* Bytes of a row of K values in format F, 0 if K is not a whole number of blocks. */
long oracle_format_row_bytes(int F, int K)
{
    int qk;
    int b = fmt_block(F, &qk);
    if (!b || K <= 0 || K % qk) return 0;
    return (long)(K / qk) * b;
}

static float f16_at(const uint8_t* p) { return oracle_half_to_float((uint16_t)(p[0] | (p[1] << 8))); }
static uint32_t u32_at(const uint8_t* p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

/* The non-linear 4-bit levels of IQ4_NL / IQ4_XS, and MXFP4's E2M1 values
 * doubled (so they are integers; the E8M0 scale is halved to match). */
static const int8_t iq4_levels[16] = {-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113};
static const int8_t e2m1_twice[16] = {0, 1, 2, 3, 4, 6, 8, 12, 0, -1, -2, -3, -4, -6, -8, -12};

/* Scale and min j (0..7) of a Q4_K / Q5_K super-block from its 12 packed
 * bytes: j < 4 in the low 6 bits of bytes j and j + 4; j >= 4 a low nibble
 * from byte j + 4 and the top two bits of byte j - 4 (scale) or j (min). */
static void kquant_scale_min(const uint8_t* q, int j, int* sc, int* m)
{
    if (j < 4) {
        *sc = q[j] & 63;
        *m = q[j + 4] & 63;
    } else {
        *sc = (q[j + 4] & 15) | ((q[j - 4] >> 6) << 4);
        *m = (q[j + 4] >> 4) | ((q[j] >> 6) << 4);
    }
}

/* Q3_K's scale i (0..15): a low nibble (bytes 0..7, low then high nibbles)
 * and two high bits (bytes 8..11, two bits per group of four scales), minus 32. */
static int q3k_scale(const uint8_t* s, int i)
{
    int lo4 = i < 8 ? (s[i] & 15) : (s[i - 8] >> 4);
    int hi2 = (s[8 + (i & 3)] >> (2 * (i >> 2))) & 3;
    return (lo4 | (hi2 << 4)) - 32;
}

/* Sub-block sb (32 values) of a row of format F: levels, and per half the
 * scale and offset.  [lane] decoder library lk_sub.  Returns 0, or -1 for
 * an unknown format. */
int oracle_sub_decode(int F, const uint8_t* row, int sb, int8_t* v, float* d, float* c)
{
    c[0] = c[1] = 0.f;
    if (F == 2 || F == 3 || F == 20) {
        const uint8_t* b = row + (long)sb * (F == 3 ? 20 : 18);
        const uint8_t* qs = b + (F == 3 ? 4 : 2);
        d[0] = d[1] = f16_at(b);
        if (F == 3) c[0] = c[1] = f16_at(b + 2);
        for (int i = 0; i < 16; ++i) {
            int lo = qs[i] & 15, hi = qs[i] >> 4;
            if (F == 20) {
                v[i] = iq4_levels[lo];
                v[i + 16] = iq4_levels[hi];
            } else {
                v[i] = (int8_t)(lo - (F == 2 ? 8 : 0));
                v[i + 16] = (int8_t)(hi - (F == 2 ? 8 : 0));
            }
        }
        return 0;
    }
    if (F == 6 || F == 7) {
        const uint8_t* b = row + (long)sb * (F == 7 ? 24 : 22);
        const uint8_t* hb = b + (F == 7 ? 4 : 2);
        uint32_t qh = u32_at(hb);
        const uint8_t* qs = hb + 4;
        d[0] = d[1] = f16_at(b);
        if (F == 7) c[0] = c[1] = f16_at(b + 2);
        int off = F == 6 ? 16 : 0;
        for (int i = 0; i < 16; ++i) {
            v[i] = (int8_t)(((qs[i] & 15) | (((qh >> i) & 1) << 4)) - off);
            v[i + 16] = (int8_t)(((qs[i] >> 4) | (((qh >> (i + 16)) & 1) << 4)) - off);
        }
        return 0;
    }
    if (F == 39) {
        const uint8_t* b = row + (long)sb * 17;
        /* E8M0 exponent e: 2^(e - 127); halved for the doubled E2M1 values */
        d[0] = d[1] = ldexpf(1.0f, (int)b[0] - 128);
        for (int i = 0; i < 16; ++i) {
            v[i] = e2m1_twice[b[1 + i] & 15];
            v[i + 16] = e2m1_twice[b[1 + i] >> 4];
        }
        return 0;
    }
    const uint8_t* sup;
    int j = sb & 7;
    if (F == 12 || F == 13) {
        sup = row + (long)(sb >> 3) * (F == 12 ? 144 : 176);
        int sc, m;
        kquant_scale_min(sup + 4, j, &sc, &m);
        float dd = f16_at(sup) * (float)sc, cc = -(f16_at(sup + 2) * (float)m);
        d[0] = d[1] = dd;
        c[0] = c[1] = cc;
        /* levels: 32-byte groups, each holding sub-blocks 2g (low nibbles)
         * and 2g + 1 (high nibbles); Q5_K's fifth bit j of byte l of the
         * 32-byte high-bit area */
        const uint8_t* ql = sup + (F == 12 ? 16 : 48) + (j >> 1) * 32;
        for (int l = 0; l < 32; ++l) {
            int lv = (j & 1) ? (ql[l] >> 4) : (ql[l] & 15);
            if (F == 13 && (sup[16 + l] >> j) & 1) lv += 16;
            v[l] = (int8_t)lv;
        }
        return 0;
    }
    if (F == 10) {
        sup = row + (long)(sb >> 3) * 84;
        int half = j >> 2, k = j & 3;
        const uint8_t* q = sup + 16 + half * 32;
        float D = f16_at(sup + 80), DM = f16_at(sup + 82);
        for (int l = 0; l < 32; ++l) v[l] = (int8_t)((q[l] >> (2 * k)) & 3);
        for (int h = 0; h < 2; ++h) {
            int s = sup[half * 8 + k * 2 + h];
            d[h] = D * (float)(s & 15);
            c[h] = -(DM * (float)(s >> 4));
        }
        return 0;
    }
    if (F == 11) {
        sup = row + (long)(sb >> 3) * 110;
        int half = j >> 2, k = j & 3;
        const uint8_t* q = sup + 32 + half * 32;
        int bit = half * 4 + k;
        float D = f16_at(sup + 108);
        for (int l = 0; l < 32; ++l)
            v[l] = (int8_t)(((q[l] >> (2 * k)) & 3) - (((sup[l] >> bit) & 1) ? 0 : 4));
        for (int h = 0; h < 2; ++h) d[h] = D * (float)q3k_scale(sup + 96, half * 8 + k * 2 + h);
        return 0;
    }
    if (F == 14) {
        sup = row + (long)(sb >> 3) * 210;
        int half = j >> 2, k = j & 3;
        const uint8_t* ql = sup + half * 64;
        const uint8_t* qh = sup + 128 + half * 32;
        const int8_t* sc = (const int8_t*)(sup + 192 + half * 8);
        float D = f16_at(sup + 208);
        for (int l = 0; l < 32; ++l) {
            int lo = (k & 1) ? ql[l + 32] : ql[l];
            lo = (k & 2) ? (lo >> 4) : (lo & 15);
            v[l] = (int8_t)((lo | (((qh[l] >> (2 * k)) & 3) << 4)) - 32);
        }
        d[0] = D * (float)sc[2 * k];
        d[1] = D * (float)sc[2 * k + 1];
        return 0;
    }
    if (F == 23) {
        sup = row + (long)(sb >> 3) * 136;
        int sh = sup[2] | (sup[3] << 8);
        int ls = ((sup[4 + (j >> 1)] >> (4 * (j & 1))) & 15) | (((sh >> (2 * j)) & 3) << 4);
        d[0] = d[1] = f16_at(sup) * (float)(ls - 32);
        const uint8_t* qs = sup + 8 + 16 * j;
        for (int i = 0; i < 16; ++i) {
            v[i] = iq4_levels[qs[i] & 15];
            v[i + 16] = iq4_levels[qs[i] >> 4];
        }
        return 0;
    }
    return -1;
}

/* The dequantized row: out[k] = RN(RN(d v) + c) (the CPU dequantizer's
 * rounding).  Returns 0, or -1 for an unknown format or K. */
int oracle_dequant_row(int F, const uint8_t* row, int K, float* out)
{
    if (!oracle_format_row_bytes(F, K)) return -1;
    int8_t v[32];
    float d[2], c[2];
    for (int sb = 0; sb < K / 32; ++sb) {
        if (oracle_sub_decode(F, row, sb, v, d, c)) return -1;
        for (int i = 0; i < 32; ++i) out[32 * sb + i] = d[i >> 4] * (float)v[i] + c[i >> 4];
    }
    return 0;
}

static float tree32f(float* s)
{
    for (int w = 16; w >= 1; w /= 2)
        for (int l = 0; l < w; ++l) s[l] = s[l] + s[l + w];
    return s[0];
}
static double tree32d(double* s)
{
    for (int w = 16; w >= 1; w /= 2)
        for (int l = 0; l < w; ++l) s[l] = s[l] + s[l + w];
    return s[0];
}

/* One half-sub-block pair's term before the activation scale ([lane]
 * lk_sub_dot): with the exact integer dots dh0, dh1 (levels . activation
 * words over values 0..15, 16..31) and the word sums sh0, sh1,
 *   part = ((d0 dh0 + c0 sh0) + d1 dh1) + c1 sh1,
 * each product and sum rounded to f32 (the expression as printed, taken
 * without contraction). */
static float sub_term(const int8_t* v, const float* d, const float* c, const int8_t* a)
{
    int32_t dh[2] = {0, 0}, sh[2] = {0, 0};
    for (int i = 0; i < 32; ++i) {
        dh[i >> 4] += (int32_t)v[i] * (int32_t)a[i];
        sh[i >> 4] += (int32_t)a[i];
    }
    float p = d[0] * (float)dh[0];
    p = p + c[0] * (float)sh[0];
    p = p + d[1] * (float)dh[1];
    p = p + c[1] * (float)sh[1];
    return p;
}

/* Rows r0..r1 of the block-format GEMV ([lane] lk_row_dot).  Sub-block sb of
 * a row goes to lane sb mod 32; a lane adds its sub-blocks' terms in
 * ascending sb, and the 32 lanes' sums meet in the shuffle-down tree of
 * lk_warp_sum.  Int8Act / TwoPass: a lane's f32 sum gets s[sb] * part (f32
 * product, then f32 sum), TwoPass's part adds 2^-7 times the low words' term.
 * Dequant: each weight as oracle_dequant_row rounds it, times x in f64 (exact),
 * added to the lane's f64 sum in value order; the tree in f64, then one
 * rounding to f32.  rb = bytes per row (oracle_format_row_bytes). */
int oracle_gemv_blk_rows(int F, const uint8_t* w, long rb, int K, int mode, const float* x, const int8_t* hi,
                         const int8_t* lo, const float* s, long r0, long r1, float* y)
{
    if (!oracle_format_row_bytes(F, K)) return -1;
    int nb = K / 32;
    for (long o = r0; o < r1; ++o) {
        const uint8_t* row = w + o * rb;
        int8_t v[32];
        float d[2], c[2];
        if (mode == 0) {
            double lane[32];
            for (int l = 0; l < 32; ++l) lane[l] = 0.0;
            for (int sb = 0; sb < nb; ++sb) {
                oracle_sub_decode(F, row, sb, v, d, c);
                for (int i = 0; i < 32; ++i) {
                    float wv = d[i >> 4] * (float)v[i] + c[i >> 4];
                    lane[sb & 31] += (double)wv * (double)x[32 * sb + i];
                }
            }
            y[o - r0] = (float)tree32d(lane);
        } else {
            float lane[32];
            for (int l = 0; l < 32; ++l) lane[l] = 0.f;
            for (int sb = 0; sb < nb; ++sb) {
                oracle_sub_decode(F, row, sb, v, d, c);
                float part = sub_term(v, d, c, hi + 32 * sb);
                if (mode == 2) part = part + 0.0078125f * sub_term(v, d, c, lo + 32 * sb);
                lane[sb & 31] = lane[sb & 31] + s[sb] * part;
            }
            y[o - r0] = tree32f(lane);
        }
    }
    return 0;
}

/* sum_k |w_k x_k| in f64 over rows r0..r1, w as oracle_dequant_row rounds it
 * (the scale of the Dequant tolerance). */
int oracle_absdot_blk_rows(int F, const uint8_t* w, long rb, int K, const float* x, long r0, long r1, double* out)
{
    if (!oracle_format_row_bytes(F, K)) return -1;
    int8_t v[32];
    float d[2], c[2];
    for (long o = r0; o < r1; ++o) {
        double acc = 0.0;
        for (int sb = 0; sb < K / 32; ++sb) {
            oracle_sub_decode(F, w + o * rb, sb, v, d, c);
            for (int i = 0; i < 32; ++i)
                acc += fabs((double)(d[i >> 4] * (float)v[i] + c[i >> 4]) * (double)x[32 * sb + i]);
        }
        out[o - r0] = acc;
    }
    return 0;
}
