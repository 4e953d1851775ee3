// Device helpers shared by the library's kernels (sm_103a).
//
// Every float operation whose rounding is part of the result is written with
// an explicit IEEE intrinsic (__fdiv_rn, __fmul_rn, __fmaf_rn, ...) so that no
// compiler contraction or fast-math flag can change it.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace lk {

constexpr unsigned FULL = 0xffffffffu;

// ---- order-free warp reductions (exact: max) ---------------------------------
__device__ __forceinline__ float warp_max_xor(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(FULL, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// ---- launch timeline records (option "trace" 3) ---------------------------------
// Record `slot` holds TREC entries: [0] block 0 start, [1] block 0 past the
// dependency wait, [2] block 0's activation ready, [3] the last block's end,
// [4] block 0's end, [5] kernel kind, [6] rows (or K), [7] block 0's first
// weight stages issued (GEMV kernels).
constexpr int TREC = 8;
enum : int { TR_START = 0, TR_WAITED = 1, TR_ACT = 2, TR_END_MAX = 3, TR_END0 = 4, TR_KIND = 5, TR_ROWS = 6,
             TR_ISSUED = 7 };
enum : int { TK_RING = 1, TK_CHAIN = 2, TK_MMA = 3, TK_NORM = 4, TK_QUANT = 5, TK_COMBINE = 6 };
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Small kernels' records without a block barrier: thread 0 of every block.
__device__ __forceinline__ void trec_stamp(unsigned long long* tr, int slot, int i) {
  if (tr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) tr[slot * TREC + i] = globaltimer_ns();
}
__device__ __forceinline__ void trec_end(unsigned long long* tr, int slot, int kind, long rows) {
  if (!tr || threadIdx.x != 0) return;
  const unsigned long long now = globaltimer_ns();
  atomicMax(tr + slot * TREC + TR_END_MAX, now);
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    tr[slot * TREC + TR_END0] = now;
    tr[slot * TREC + TR_KIND] = (unsigned long long)kind;
    tr[slot * TREC + TR_ROWS] = (unsigned long long)rows;
  }
}

// ---- the canonical sum tree ("kernels.rs" lk_warp_sum) -------------------------
// Lane l adds lane l+d for d = 16, 8, 4, 2, 1; lane 0 ends with the total.
template <typename A>
__device__ __forceinline__ A warp_tree_sum(A v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = v + __shfl_down_sync(FULL, v, o);
  return v;
}

// ---- the activation quantizer ("kernels.rs" PRELUDE: lk_quant_lane,
// lk_two_scale, lk_two_words) ------------------------------------------------
// A warp quantizes NG 32-value groups at once, one value of each per lane;
// the groups' steps are written phase by phase, so their independent chains
// (the IEEE divisions above all) interleave.  Per group, a = max|v|:
//   Int8Act (Q 1): s = a/127; a group with a < 127 * 2^-126 (a/127 not a
//                  normal float, the all-zero group included) gets s = 1 and
//                  hi = 0; otherwise |v/s| <= 127 (1 + 2^-24) and
//                  hi = rn(v/s) needs no clamp.
//   TwoPass (Q 2): s = max(a, 1e-30)/127; hi = clamp(rn(v/s)) and
//                  lo = clamp(rn(fma(-hi, s, v) / (s/128))).
// rn rounds to nearest even; every division is the IEEE one.
constexpr float kInt8ActMinMax = 0x1.fcp-120f;  // 127 * 2^-126

// max|v| over the warp in one instruction: for non-negative floats the IEEE
// order is the order of their bit patterns, so the integer max of the bits
// of |v| is the bits of max|v| (exact; NaN inputs are unspecified).
__device__ __forceinline__ float warp_absmax(float v) {
  return __uint_as_float(__reduce_max_sync(FULL, __float_as_uint(fabsf(v))));
}

// ---- IEEE quotients of the quantizer without the division sequence --------
// a / 127 for finite a >= 0, correctly rounded: Markstein's correction step
// (P. Markstein, IBM J. Res. Develop. 34(1), 1990) from r = RN(1/127):
// q0 = RN(a r), rem = fma(-q0, 127, a), q = fma(rem, r, q0).  Checked equal to
// the IEEE quotient for every finite non-negative binary32 on the host
// (tests/csrc/div127_check.c), with the same IEEE binary32 operations.
__device__ __forceinline__ float div127(float a) {
  const float r = 0x1.020408p-7f;
  const float q0 = __fmul_rn(a, r);
  return __fmaf_rn(__fmaf_rn(-q0, 127.0f, a), r, q0);
}

// rn(v / s) as an integer, |v / s| < 129, with rs an approximate 1/s (the
// hardware reciprocal, relative error below 2^-22): qa = RN(v rs) is within
// 129 (2^-22 + 2^-24) < 2^-14 of v / s, and RN(v / s) within 2^-18 of it, so
// unless qa lies within 2^-12 of a half-integer both round to the same
// integer; near one (a tie or close: about 1 value in 2000) the IEEE
// quotient decides.
__device__ __forceinline__ float approx_rcp(float s) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}
__device__ __forceinline__ int rn_quot(float v, float s, float rs) {
  const float qa = __fmul_rn(v, rs);
  const float m = fabsf(qa);
  if (fabsf(__fsub_rn(__fsub_rn(m, floorf(m)), 0.5f)) < 0x1p-12f) return __float2int_rn(__fdiv_rn(v, s));
  return __float2int_rn(qa);
}

template <int Q>
__device__ __forceinline__ float act_scale(float a) {
  if constexpr (Q == 1) return a >= kInt8ActMinMax ? div127(a) : 1.0f;
  return div127(fmaxf(a, 1e-30f));
}

__device__ __forceinline__ int sat_i8(int v) { return min(max(v, -128), 127); }

// Groups G_k = g + k * step (k < NG) of one activation row: lane `lane`
// holds v[k], element 32 G_k + lane of the row; groups with ok[k] false are
// computed but not stored.  hi, lo (TwoPass only) and xs point at the row.
template <int Q, int NG>
__device__ __forceinline__ void quant_groups(const float (&v)[NG], const bool (&ok)[NG], int8_t* __restrict__ hi,
                                             int8_t* __restrict__ lo, float* __restrict__ xs, long g, long step,
                                             int lane) {
  float s[NG], rs[NG];
  int h[NG], l[NG];
#pragma unroll
  for (int k = 0; k < NG; ++k) {
    s[k] = act_scale<Q>(warp_absmax(v[k]));
    rs[k] = approx_rcp(s[k]);
  }
  // |v / s| <= 127 (1 + 2^-24): rn_quot applies (a tiny group: |v| / 1 rounds to 0)
#pragma unroll
  for (int k = 0; k < NG; ++k) h[k] = rn_quot(v[k], s[k], rs[k]);
  if constexpr (Q == 2) {
#pragma unroll
    for (int k = 0; k < NG; ++k) {
      h[k] = sat_i8(h[k]);
      // the low word's quotient res / (s/128) = 128 res / s, |.| <= 65: s/128
      // is exact (s is a normal float at least 1e-30/127), so is 128 res
      const float res = __fmaf_rn(-(float)h[k], s[k], v[k]);
      l[k] = sat_i8(rn_quot(__fmul_rn(res, 128.0f), s[k], rs[k]));
    }
  }
#pragma unroll
  for (int k = 0; k < NG; ++k) {
    if (!ok[k]) continue;
    const long e = 32 * (g + k * step) + lane;
    hi[e] = (int8_t)h[k];
    if constexpr (Q == 2) lo[e] = (int8_t)l[k];
    if (lane == 0) xs[g + k * step] = s[k];
  }
}

// One group: lane `lane` holds v, element 32 g + lane.
template <int Q>
__device__ __forceinline__ void quant_lane(float v, int8_t* __restrict__ hi, int8_t* __restrict__ lo,
                                           float* __restrict__ xs, long g, int lane) {
  const float vv[1] = {v};
  const bool ok[1] = {true};
  quant_groups<Q, 1>(vv, ok, hi, lo, xs, g, 0, lane);
}

// ---- SwiGLU ("kernels.rs" lk_gemv_glu with ACT -1): h = g / (1 + e^-g) * u,
// each operation rounded to f32 as written (expf is the CUDA library's).
__device__ __forceinline__ float swiglu(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// ---- RMSNorm arithmetic ("kernels.rs" lk_rmsnorm_row: accumulator f64 under
// Dequant (Q 0), f32 otherwise; y = v / sqrt(sum/K + eps) * g)
template <int Q>
struct acc_of { typedef float t; };
template <>
struct acc_of<0> { typedef double t; };

__device__ __forceinline__ float fma_acc(float v, float acc) { return __fmaf_rn(v, v, acc); }
__device__ __forceinline__ double fma_acc(double v, double acc) { return __fma_rn(v, v, acc); }
__device__ __forceinline__ float norm_div_add(float sum, int K, float eps) {
  return __fsqrt_rn(__fadd_rn(__fdiv_rn(sum, (float)K), eps));
}
__device__ __forceinline__ double norm_div_add(double sum, int K, float eps) {
  return __dsqrt_rn(__dadd_rn(__ddiv_rn(sum, (double)K), (double)eps));
}
__device__ __forceinline__ float norm_scale(float v, float den, float g) {
  return __fmul_rn(__fdiv_rn(v, den), g);
}

// RN(v / d) for finite v and a normal d > 0, given yd = RN(1/d) (__frcp_rn,
// once per row): Markstein's correction q = fma(fma(-q0, d, v), yd, q0) with
// q0 = RN(v yd), accepted only where it is provably the correctly rounded
// quotient: for 2^-60 <= |q| < 2^64 with q not a power of two (its two
// neighbours one ulp away), the residual rem = fma(-q, d, v) is exact
// (q within an ulp of v/d), and |rem| < ulp(q)/2 * d (a power of two times d:
// exact) means |v/d - q| < ulp(q)/2 strictly, so q = RN(v/d) and no tie.
// Anything else (zero, a tie or near one, tiny or huge quotients) takes the
// IEEE division.  The same bits as __fdiv_rn(v, d) in every case.
__device__ __forceinline__ float div_row(float v, float d, float yd) {
  const float q0 = __fmul_rn(v, yd);
  const float q = __fmaf_rn(__fmaf_rn(-q0, d, v), yd, q0);
  const unsigned b = __float_as_uint(q), e = b & 0x7F800000u;
  if (e >= (67u << 23) && e < (191u << 23) && (b & 0x007FFFFFu) != 0u) {
    const float rem = __fmaf_rn(-q, d, v);
    const float half = __uint_as_float(e - (24u << 23));  // ulp(q) / 2 = 2^(E - 127 - 24)
    if (fabsf(rem) < __fmul_rn(half, d)) return q;
  }
  return __fdiv_rn(v, d);
}
__device__ __forceinline__ float norm_scale_r(float v, float den, float yd, float g) {
  return __fmul_rn(div_row(v, den, yd), g);
}
__device__ __forceinline__ float norm_scale(float v, double den, float g) {
  return __double2float_rn(__dmul_rn(__ddiv_rn((double)v, den), (double)g));
}

// ---- argmax key ("megakernel.cu" amax_key) --------------------------------------
// Order-preserving image of the f32 value (after -0 -> +0) in the high word,
// 0xFFFFFFFF - index in the low word: the largest key is the largest value,
// then the lowest index.
__device__ __forceinline__ unsigned long long amax_key(float v, unsigned idx) {
  if (v == 0.0f) v = 0.0f;
  unsigned u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

// ---- the quantized block step ("kernels.rs" lk_q8_term / lk_q8_acc) --------------
template <int Q>
__device__ __forceinline__ float q8_step(float p, float w, float s, int d, int e) {
  if (Q == 1) return __fmaf_rn(__fmul_rn(w, s), (float)d, p);
  const float u = __fmaf_rn(s, (float)d, __fmul_rn(__fmul_rn(s, 0.0078125f), (float)e));
  return __fmaf_rn(w, u, p);
}

// Byte k of w (a signed int8) as an f32, exactly: (b + 128) in the low
// mantissa bits of 2^23 gives the float 2^23 + b + 128; subtracting
// 2^23 + 128 leaves b.  One byte permute and one add instead of an
// integer-to-float conversion (a quarter-rate instruction).  u = w ^ 0x80808080.
__device__ __forceinline__ float i8_as_f32(unsigned u, int k) {
  const unsigned bits = __byte_perm(u, 0x4B000000u, 0x7440u | (unsigned)k);
  return __fadd_rn(__uint_as_float(bits), -8388736.0f);
}

// The float 2^23 + 128 + b for byte k of u = w ^ 0x80808080 (i8_as_f32
// before its subtraction).
__device__ __forceinline__ float i8_bits_f32(unsigned u, int k) {
  return __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440u | (unsigned)k));
}

// Packed pairs of f32 (sm_100 and later: one instruction for both halves,
// each rounded to nearest like its scalar form).
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 f2_pack(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(f32x2 v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

__device__ __forceinline__ int dot16(int4 w, int4 x) {
  int d = __dp4a(w.x, x.x, 0);
  d = __dp4a(w.y, x.y, d);
  d = __dp4a(w.z, x.z, d);
  d = __dp4a(w.w, x.w, d);
  return d;
}

// Streaming 16-byte load of weights: read-only path, no L1 allocation.
__device__ __forceinline__ int4 ld_stream16(const void* p) {
  int4 r;
  asm("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Split-K chunk bound: the balanced split over four-block groups
// ("kernels.rs" GEMM_BLK), the last chunk ending at nb.
__host__ __device__ __forceinline__ int splitk_bound(int nb, int S, int c) {
  if (c >= S) return nb;
  const int G = nb >> 2;
  return 4 * (int)(((long long)c * G) / S);
}

}  // namespace lk
