/*
 * Q8_0 GEMV oracle: a plain, slow, single-threaded CPU restatement of what the
 * decode-projection path computes.  TEST INFRASTRUCTURE ONLY: the test suite,
 * the package smoke check and the CPU-baseline leg of the benchmark load it;
 * the library never does.  It shares no code, header or table with the CUDA
 * path.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -fPIC -shared oracle.c -lm
 * (-ffp-contract=off: every fused multiply-add below is written out with
 * fmaf/fma; every other product and sum is rounded on its own, in IEEE
 * single or double precision as stated.)  The GEMV row loops may run on
 * several host threads (oracle_set_threads; 1 by default): each output row
 * is computed by one thread exactly as written, so any thread count gives
 * the same bits.
 *
 * Sources (three web pages on the subject):
 *   [lane]   "kernels.rs" of logicaffeine_compile::codegen_cuda::lane: the
 *            module doc on the numerics modes (Q8MatKind), the PRELUDE
 *            helpers (lk_two_scale / lk_two_words, lk_quant_lane, lk_q8_term,
 *            lk_q8_sum4, lk_q8_rows_dot), RMSNORM (lk_rmsnorm_row,
 *            lk_warps_sum), norm_threads, GEMM_BLK's balanced k-split.
 *   [extra]  the QWEN38_EXTRA_KERNELS constant: "SPLIT-K FOR THE NARROW
 *            PROJECTIONS" (gk_gemv_hl_sk, gk_sk_combine).
 *   [mak]    model-as-a-kernel "megakernel.cu": amax_key, ph_argmax_part,
 *            ph_argmax_fin (first index of equal maxima).
 *
 * Every function below states the passage it follows.  Where the pages leave
 * a step open the reading taken is stated beside it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Host threads of the GEMV row loops (1 = the plain single-threaded oracle). */
static int or_threads = 1;
int oracle_set_threads(int n)
{
#ifdef _OPENMP
    or_threads = n < 1 ? 1 : n;
#else
    (void)n;
    or_threads = 1;
#endif
    return or_threads;
}
int oracle_get_threads(void) { return or_threads; }

#define OR_DEQUANT 0
#define OR_INT8ACT 1
#define OR_TWOPASS 2

/* IEEE binary16 -> binary32, from the format's definition: sign, 5-bit
 * exponent biased by 15, 10-bit fraction; exponent 0 is subnormal
 * (fraction * 2^-24), exponent 31 is inf/NaN.  The Q8_0 block scale is an f16
 * ([lane] module doc: a Q8_0 matrix reaches the device as two arrays, the int8
 * levels and one f16 scale for every 32 weights).  The value is exact in f32. */
float oracle_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    float v;
    if (e == 0)
        v = ldexpf((float)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* Round to nearest, ties to even (the pages' __float2int_rn).  The distance
 * to the floor is taken in f64, where it is exact for any f32 input.  Values
 * outside the int range saturate and NaN gives 0, as the GPU's conversion
 * does; the quantizer below never produces either (its quotients stay within
 * about +-128), so this only keeps the function defined everywhere. */
static int round_half_even(float v)
{
    if (v != v) return 0;
    if (v >= 2147483648.0f) return 2147483647;
    if (v < -2147483648.0f) return -2147483647 - 1;
    double fl = floor((double)v);
    double diff = (double)v - fl;
    long n = (long)fl;
    if (diff > 0.5) return (int)(n + 1);
    if (diff < 0.5) return (int)n;
    return (int)((n % 2 == 0) ? n : n + 1);
}

static int clamp8(int v) { return v > 127 ? 127 : (v < -128 ? -128 : v); }

/* ---- activation quantizer ------------------------------------------------
 * [lane] module doc and PRELUDE (lk_quant_lane, lk_two_scale, lk_two_words):
 * a group of 32 values shares one scale from its largest magnitude a.
 *   Int8Act:  s = a/127 (1 for an all-zero group);  hi = rn(v/s)
 *   TwoPass:  s = max(a, 1e-30)/127;   hi = clamp(rn(v/s));
 *             r = fma(-hi, s, v);      lo = clamp(rn(r / (s * 2^-7)))
 * The quotient form is the definition (the reciprocal variant lk_two_words_r is
 * a kernel shortcut and is not used).  Dequant keeps f32 and quantizes nothing.
 *
 * Reading for Int8Act groups whose largest magnitude is tiny: the pages give
 * the scale 1 only to a = 0, but for 0 < a < 127 * 2^-126 the scale a/127 is
 * subnormal or zero, loses bits, and v/s then leaves [-127, 127] (even inf or
 * NaN), so hi would not fit its int8.  Such a group is treated as the all-zero
 * group (s = 1, every hi = 0): then |v - hi*s| = |v| < 2^-119 <= s/2 still
 * holds, and for every a >= 127 * 2^-126 the scale is a normal float and
 * |v/s| <= 127 (1 + 2^-24), so rn(v/s) is within [-127, 127] without a clamp.
 * TwoPass needs no such rule: its scale is at least 1e-30/127, a normal float.
 * v has K values, K a multiple of 32; hi/lo have K entries, s has K/32. */
#define OR_INT8ACT_MIN_MAX 0x1.fcp-120f /* 127 * 2^-126 */
void oracle_quantize_row(const float* v, int K, int mode, int8_t* hi, int8_t* lo, float* s)
{
    for (int g = 0; g < K / 32; ++g) {
        const float* vg = v + 32 * g;
        float a = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float m = fabsf(vg[i]);
            if (m > a) a = m;
        }
        float sc;
        if (mode == OR_INT8ACT)
            sc = a >= OR_INT8ACT_MIN_MAX ? a / 127.0f : 1.0f;
        else
            sc = (a > 1e-30f ? a : 1e-30f) / 127.0f;
        s[g] = sc;
        for (int i = 0; i < 32; ++i) {
            int h = round_half_even(vg[i] / sc);
            if (mode == OR_INT8ACT) {
                hi[32 * g + i] = (int8_t)h;
            } else {
                h = clamp8(h);
                float r = fmaf(-(float)h, sc, vg[i]);
                int l = clamp8(round_half_even(r / (sc * 0.0078125f)));
                hi[32 * g + i] = (int8_t)h;
                lo[32 * g + i] = (int8_t)l;
            }
        }
    }
}

/* ---- RMSNorm ---------------------------------------------------------------
 * [lane] module doc: the norm divides each value by the square root of the
 * mean square plus 1e-6, then multiplies by the gain; RMSNORM
 * (lk_rmsnorm_row): y_i = v_i / sqrt(sum(v^2)/K + eps) * g_i, the sum in the
 * accumulator of the mode (f64 under Dequant, f32 otherwise: lk_acc).
 *
 * The f32 sum of squares is not associative, so its order is part of the
 * definition.  The pages' block is norm_threads(K) = min(roundup32(K), 1024)
 * threads; thread t adds the squares of values t, t+vt, t+2vt, ... in that
 * order, each as one fused multiply-add (the reading of `acc += v*v` under
 * nvcc's default contraction); each warp of 32 threads then sums its lanes by
 * the shuffle-down tree of distances 16, 8, 4, 2, 1 (lane l adds lane l+d),
 * and the warps' totals, padded with zeros to 32, are summed by the same tree
 * (lk_warp_sum, lk_warps_sum).  In f64 the squares are exact and the same
 * order is kept.
 */
static float tree32_f(float* s)
{
    for (int d = 16; d >= 1; d /= 2)
        for (int l = 0; l < d; ++l) s[l] = s[l] + s[l + d];
    return s[0];
}
static double tree32_d(double* s)
{
    for (int d = 16; d >= 1; d /= 2)
        for (int l = 0; l < d; ++l) s[l] = s[l] + s[l + d];
    return s[0];
}

int oracle_norm_threads(int K)
{
    int r = ((K + 31) / 32) * 32;
    return r < 1024 ? r : 1024;
}

/* The canonical sum of squares of one row (exported so the tests can pin the
 * order on a case where a different order gives a different float). */
float oracle_sumsq_f32(const float* v, int K)
{
    int vt = oracle_norm_threads(K), vw = vt / 32;
    float warp_tot[32];
    for (int w = 0; w < 32; ++w) warp_tot[w] = 0.0f;
    for (int w = 0; w < vw; ++w) {
        float lane[32];
        for (int l = 0; l < 32; ++l) {
            int t = 32 * w + l;
            float acc = 0.0f;
            for (int i = t; i < K; i += vt) acc = fmaf(v[i], v[i], acc);
            lane[l] = acc;
        }
        warp_tot[w] = tree32_f(lane);
    }
    return tree32_f(warp_tot);
}

double oracle_sumsq_f64(const float* v, int K)
{
    int vt = oracle_norm_threads(K), vw = vt / 32;
    double warp_tot[32];
    for (int w = 0; w < 32; ++w) warp_tot[w] = 0.0;
    for (int w = 0; w < vw; ++w) {
        double lane[32];
        for (int l = 0; l < 32; ++l) {
            int t = 32 * w + l;
            double acc = 0.0;
            for (int i = t; i < K; i += vt) acc = fma((double)v[i], (double)v[i], acc);
            lane[l] = acc;
        }
        warp_tot[w] = tree32_d(lane);
    }
    return tree32_d(warp_tot);
}

/* y[K] = RMSNorm(v[K]) * g under the accumulator of `mode`. */
void oracle_rmsnorm_row(const float* v, const float* g, int K, float eps, int mode, float* y)
{
    if (K <= 0) return;
    if (mode == OR_DEQUANT) {
        double den = sqrt(oracle_sumsq_f64(v, K) / (double)K + (double)eps);
        for (int i = 0; i < K; ++i) y[i] = (float)((double)v[i] / den * (double)g[i]);
    } else {
        float den = sqrtf(oracle_sumsq_f32(v, K) / (float)K + eps);
        for (int i = 0; i < K; ++i) y[i] = v[i] / den * g[i];
    }
}

/* ---- residual add + RMSNorm ------------------------------------------------
 * [lane] RMSNORM lk_rmsnorm_row with ADD (and SUM): the residual r is added to
 * the row first, v_i = x_i + r_i as one f32 addition, the sum v is the
 * residual stream the next block reads (written to s when s != NULL), and v is
 * what the norm sees; [extra] gk_add_rmsnorm_q8_hl is the same step (x += y,
 * then the norm and the quantizer).  The norm is oracle_rmsnorm_row's, on v.
 * Returns 0, or -1 if the scratch row cannot be allocated. */
int oracle_add_rmsnorm_row(const float* x, const float* r, const float* g, int K, float eps, int mode,
                           float* s, float* y)
{
    if (K <= 0) return 0;
    float* v = (float*)malloc(sizeof(float) * (size_t)K);
    if (!v) return -1;
    for (int i = 0; i < K; ++i) {
        v[i] = x[i] + r[i];
        if (s) s[i] = v[i];
    }
    oracle_rmsnorm_row(v, g, K, eps, mode, y);
    free(v);
    return 0;
}

/* ---- SwiGLU ------------------------------------------------------------------
 * [lane] GLU (lk_gemv_glu with ACT -1, lk_swiglu) and [extra] gk_silu_had_q8:
 * the gated activation of a gate value g and an up value u is
 *   h = silu(g) * u = g / (1 + e^-g) * u.
 * The pages evaluate it in f32 with the GPU's expf; the oracle takes the
 * definition in f64 from the f32 inputs and rounds h to f32 once (for
 * g < -709 the f64 e^-g overflows and h is a signed zero, as the f32 form
 * gives below g = -88.7).  h feeds the activation quantizer of the down
 * projection (oracle_quantize_row). */
void oracle_swiglu(const float* g, const float* u, long n, float* h)
{
    for (long i = 0; i < n; ++i) {
        double gv = (double)g[i];
        h[i] = (float)(gv / (1.0 + exp(-gv)) * (double)u[i]);
    }
}

/* ---- block dots ------------------------------------------------------------
 * [lane] lk_q8_block_dot: the int8 dot of one 32-value block, exact in int32.
 * d[o*nb+b] = sum_k wq[o][32b+k] * hi[32b+k]; e likewise with lo (TwoPass). */
void oracle_block_dots(const int8_t* wq, int N, int K, const int8_t* hi, const int8_t* lo,
                       int32_t* d, int32_t* e)
{
    int nb = K / 32;
    for (int o = 0; o < N; ++o)
        for (int b = 0; b < nb; ++b) {
            int32_t dd = 0, ee = 0;
            for (int k = 0; k < 32; ++k) {
                int w = wq[(long)o * K + 32 * b + k];
                dd += w * hi[32 * b + k];
                if (lo) ee += w * lo[32 * b + k];
            }
            d[(long)o * nb + b] = dd;
            if (e) e[(long)o * nb + b] = ee;
        }
}

/* ---- one quantized block step ---------------------------------------------
 * [lane] lk_q8_term / lk_q8_acc, each operation rounded as written there:
 *   Int8Act:  p = fma(w*s, d, p)                    (w*s one f32 product)
 *   TwoPass:  p = fma(w, fma(s, d, (s*2^-7)*e), p)  ((s*2^-7)*e one product)
 * w is the block's f16 weight scale, s the activation group's scale. */
static float q8_step(int mode, float p, float w, float s, int32_t d, int32_t e)
{
    if (mode == OR_INT8ACT) {
        float t = w * s;
        return fmaf(t, (float)d, p);
    }
    float le = (s * 0.0078125f) * (float)e;
    float u = fmaf(s, (float)d, le);
    return fmaf(w, u, p);
}

static int32_t block_dot(const int8_t* w, const int8_t* a)
{
    int32_t r = 0;
    for (int k = 0; k < 32; ++k) r += (int32_t)w[k] * (int32_t)a[k];
    return r;
}

/* The quantized value of row o over blocks [b0, b1): [lane] lk_q8_rows_dot —
 * block b's step goes into partial b mod 4 (global block index), a partial's
 * blocks in ascending order; the four partials sum as (p0+p2)+(p1+p3)
 * (lk_q8_sum4). */
static float q8_row_range(const int8_t* wq, const uint16_t* ws, int K, int mode, long o,
                          const int8_t* hi, const int8_t* lo, const float* s, int b0, int b1)
{
    int nb = K / 32;
    float p[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int b = b0; b < b1; ++b) {
        const int8_t* wr = wq + o * K + 32 * b;
        int32_t d = block_dot(wr, hi + 32 * b);
        int32_t e = mode == OR_TWOPASS ? block_dot(wr, lo + 32 * b) : 0;
        float w = oracle_half_to_float(ws[o * nb + b]);
        p[b % 4] = q8_step(mode, p[b % 4], w, s[b], d, e);
    }
    return (p[0] + p[2]) + (p[1] + p[3]);
}

/* Dequant value of row o over columns [k0, k1): the plain definition, W = f16
 * scale * level (exact in f32), each product (double)W*(double)x exact in f64,
 * summed in ascending k in f64 ([lane] module doc: Dequant's dot is an f64
 * sum).  Returned unrounded. */
static double deq_row_range(const int8_t* wq, const uint16_t* ws, int K, long o, const float* x,
                            int k0, int k1)
{
    int nb = K / 32;
    double acc = 0.0;
    for (int k = k0; k < k1; ++k) {
        float w = oracle_half_to_float(ws[o * nb + k / 32]) * (float)wq[o * K + k];
        acc += (double)w * (double)x[k];
    }
    return acc;
}

/* y[i] = row r0+i of the GEMV for one activation row, i < r1-r0.
 * Dequant reads x (f32); the quantized modes read hi, lo (TwoPass), s. */
void oracle_gemv_rows(const int8_t* wq, const uint16_t* ws, int K, int mode, const float* x,
                      const int8_t* hi, const int8_t* lo, const float* s, long r0, long r1,
                      float* y)
{
#pragma omp parallel for schedule(static) num_threads(or_threads) if (or_threads > 1)
    for (long o = r0; o < r1; ++o) {
        if (mode == OR_DEQUANT)
            y[o - r0] = (float)deq_row_range(wq, ws, K, o, x, 0, K);
        else
            y[o - r0] = q8_row_range(wq, ws, K, mode, o, hi, lo, s, 0, K / 32);
    }
}

/* ---- split-K -----------------------------------------------------------------
 * [extra] "SPLIT-K FOR THE NARROW PROJECTIONS": K is cut into S chunks, each
 * chunk's value is computed on its own, and a separate combine adds the
 * chunks in ascending order from zero (gk_sk_combine), never atomically.
 * Reading of the cut: [lane] GEMM_BLK's balanced split over groups of four
 * blocks (128 values): chunk c starts at block 4*floor(c*G/S), G = nb/4
 * (floor), and the last chunk ends at nb, taking any blocks past 4G.
 * (Not [extra]'s ceil over 512-value units, which leaves chunks empty for
 * K=5120, S=8.)  A chunk's quantized value is the row rule above restricted
 * to its blocks, partial index still the global b mod 4; a Dequant chunk is
 * its f64 sum, the chunks added in f64 and rounded to f32 once. */
int oracle_splitk_bound(int nb, int S, int c)
{
    if (c >= S) return nb;
    int G = nb / 4;
    return 4 * (int)(((long)c * G) / S);
}

/* y[i] for rows r0.., and the chunk values (f32 for quantized modes into
 * chunk_f [S][r1-r0], f64 for Dequant into chunk_d) if those are non-NULL. */
void oracle_gemv_splitk_rows(const int8_t* wq, const uint16_t* ws, int K, int mode, const float* x,
                             const int8_t* hi, const int8_t* lo, const float* s, int S, long r0,
                             long r1, float* y, float* chunk_f, double* chunk_d)
{
    int nb = K / 32;
    long n = r1 - r0;
#pragma omp parallel for schedule(static) num_threads(or_threads) if (or_threads > 1)
    for (long o = r0; o < r1; ++o) {
        if (mode == OR_DEQUANT) {
            double acc = 0.0;
            for (int c = 0; c < S; ++c) {
                int b0 = oracle_splitk_bound(nb, S, c), b1 = oracle_splitk_bound(nb, S, c + 1);
                double v = deq_row_range(wq, ws, K, o, x, 32 * b0, 32 * b1);
                if (chunk_d) chunk_d[(long)c * n + (o - r0)] = v;
                acc = acc + v;
            }
            y[o - r0] = (float)acc;
        } else {
            float acc = 0.0f;
            for (int c = 0; c < S; ++c) {
                int b0 = oracle_splitk_bound(nb, S, c), b1 = oracle_splitk_bound(nb, S, c + 1);
                float v = q8_row_range(wq, ws, K, mode, o, hi, lo, s, b0, b1);
                if (chunk_f) chunk_f[(long)c * n + (o - r0)] = v;
                acc = acc + v;
            }
            y[o - r0] = acc;
        }
    }
}

/* sum_k |W[o][k] * x[k]| in f64 for rows r0..r1: the scale of the tolerance
 * (x is the f32 activation that enters the mode, after the norm). */
void oracle_absdot_rows(const int8_t* wq, const uint16_t* ws, int K, const float* x, long r0,
                        long r1, double* out)
{
    int nb = K / 32;
#pragma omp parallel for schedule(static) num_threads(or_threads) if (or_threads > 1)
    for (long o = r0; o < r1; ++o) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k) {
            float w = oracle_half_to_float(ws[o * nb + k / 32]) * (float)wq[o * K + k];
            acc += fabs((double)w * (double)x[k]);
        }
        out[o - r0] = acc;
    }
}

/* ---- argmax ------------------------------------------------------------------
 * [lane] module doc: of equal maxima the arg-max returns the first; [mak]
 * ph_argmax_part: lowest index on ties.  A linear scan with a strict `>` over
 * the logits as stored in f32 (so -0 == +0).  n >= 1.  NaN is unspecified. */
long oracle_argmax(const float* v, long n)
{
    long best = 0;
    for (long i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}
