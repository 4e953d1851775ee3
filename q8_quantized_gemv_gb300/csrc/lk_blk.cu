// GEMV on the GGUF block formats other than Q8_0 ("kernels.rs" decoder
// library: lk_sub, lk_sub_dot, lk_row_dot), sm_103a.
//
// Every format is read as 32-value sub-blocks: 32 int8 levels and, per half
// (values 0..15, 16..31), a scale d and an offset c, the weight being
// RN(RN(d level) + c).  The quantized modes' row value is fixed by the pages'
// arrangement, so this kernel keeps it: sub-block sb of a row belongs to lane
// sb mod 32, a lane adds s[sb] * part in ascending sb (f32 product, f32 sum)
// with part = ((d0 dh0 + c0 sh0) + d1 dh1) + c1 sh1 -- dh the exact int8
// dots of the levels with the activation words over each half, sh the
// words' sums (TwoPass adds 2^-7 times the low words' part) -- and the lanes
// meet in the shuffle-down tree (lane l adds lane l + d, d = 16 .. 1).
// Dequant (f32 activations) is held to the tolerance instead: each lane
// sums its sub-blocks' products in f32 with a compensation term and the
// lanes' totals are added in f64.
//
// Data movement: a warp owns whole rows.  Its next row's bytes are copied
// into one of the warp's two shared-memory buffers by 16-byte asynchronous
// copies (cp.async) while it computes the current one; the lanes then decode
// their sub-blocks from shared memory.  The activation rows are copied into
// shared memory once per block, 16 bytes of padding after every 32 values so
// that 32 lanes reading 32 consecutive sub-blocks hit every bank once.  The
// levels are built directly as packed int8 x 4 words (per-byte subtraction
// and bit spreading), so the dots are dp4a.
#include <cuda_fp16.h>

#include "lk_device.cuh"
#include "lk_host.h"

namespace lkblk {

using namespace lk;

constexpr int BW = 8;  // warps per block at most

// Values of one block and bytes of one block, by format number (0: unknown).
__host__ __device__ constexpr int blk_values(int F) {
  return (F == 10 || F == 11 || F == 12 || F == 13 || F == 14 || F == 23) ? 256
         : (F == 2 || F == 3 || F == 6 || F == 7 || F == 20 || F == 39) ? 32 : 0;
}
__host__ __device__ constexpr int blk_bytes(int F) {
  return F == 2 ? 18 : F == 3 ? 20 : F == 6 ? 22 : F == 7 ? 24 : F == 20 ? 18 : F == 39 ? 17
       : F == 10 ? 84 : F == 11 ? 110 : F == 12 ? 144 : F == 13 ? 176 : F == 14 ? 210 : F == 23 ? 136 : 0;
}

// Shared-memory byte helpers (the staged row: 16-byte aligned, arbitrary
// byte offsets inside it).
__device__ __forceinline__ unsigned u8(const unsigned char* p) { return *p; }
// (every f16 field of these layouts sits at an even offset of a 16-byte
// aligned row: blocks of 18, 20, 22, 24 bytes, super-blocks of 84, 110,
// 136, 144, 176, 210 bytes with even field offsets)
__device__ __forceinline__ float half_at(const unsigned char* p) { return __half2float(*(const __half*)p); }
// Four bytes from any offset: the two aligned words around them.
__device__ __forceinline__ unsigned w32(const unsigned char* p) {
  const uintptr_t a = (uintptr_t)p;
  const unsigned* q = (const unsigned*)(a & ~(uintptr_t)3);
  const unsigned sh = 8u * (unsigned)(a & 3);
  return sh ? __funnelshift_r(q[0], q[1], sh) : q[0];
}
// NW consecutive 4-byte words from any offset: the NW + 1 aligned words
// around them, funnel-shifted by the offset's byte position (the same for
// every word; no per-word branch).
template <int NW>
__device__ __forceinline__ void words_at(const unsigned char* p, unsigned (&out)[NW]) {
  const uintptr_t a = (uintptr_t)p;
  const unsigned* q = (const unsigned*)(a & ~(uintptr_t)3);
  const unsigned sh = 8u * (unsigned)(a & 3);
  unsigned v[NW + 1];
#pragma unroll
  for (int i = 0; i <= NW; ++i) v[i] = q[i];
#pragma unroll
  for (int i = 0; i < NW; ++i) out[i] = __funnelshift_r(v[i], v[i + 1], sh);
}

// The same, shifted right by e more bits (0 <= e <= 7): bit field e.. of
// every byte in one funnel shift (the bits that enter from the next word
// at bit 32 - e and above, past the top byte's field when it is at most
// 8 - e bits wide).
template <int NW>
__device__ __forceinline__ void words_at_sh(const unsigned char* p, unsigned e, unsigned (&out)[NW]) {
  const uintptr_t a = (uintptr_t)p;
  const unsigned* q = (const unsigned*)(a & ~(uintptr_t)3);
  const unsigned sh = 8u * (unsigned)(a & 3) + e;
  unsigned v[NW + 1];
#pragma unroll
  for (int i = 0; i <= NW; ++i) v[i] = q[i];
#pragma unroll
  for (int i = 0; i < NW; ++i) out[i] = __funnelshift_r(v[i], v[i + 1], sh);
}

// Formats whose level words sit at 4-byte-aligned offsets of a staged row
// (16-byte aligned): blocks of 20 or 24 bytes with 4- or 8-byte headers,
// super-blocks of 84, 136, 144 or 176 bytes.  Their words are read as they
// are; the others (17-, 18-, 22-, 110- and 210-byte blocks) go through w32.
template <int F>
__device__ __forceinline__ unsigned word_at(const unsigned char* p) {
  if constexpr (F == 3 || F == 7 || F == 10 || F == 12 || F == 13 || F == 23) return *(const unsigned*)p;
  return w32(p);
}

// Bits 0..3 of b spread to bit 0 of bytes 0..3.
__device__ __forceinline__ unsigned spread4(unsigned b) { return ((b & 15u) * 0x00204081u) & 0x01010101u; }

// The 16-entry int8 level tables (IQ4_NL / IQ4_XS: sixteen non-linear
// levels; MXFP4: the E2M1 values doubled), four entries to a word, held in
// registers.
struct Lut16 {
  unsigned t0, t1, t2, t3;
};
__host__ __device__ constexpr unsigned pack4(int a, int b, int c, int d) {
  return (unsigned)(a & 255) | ((unsigned)(b & 255) << 8) | ((unsigned)(c & 255) << 16) | ((unsigned)(d & 255) << 24);
}
template <int F>
__device__ __forceinline__ Lut16 level_lut() {
  if constexpr (F == 39)
    return Lut16{pack4(0, 1, 2, 3), pack4(4, 6, 8, 12), pack4(0, -1, -2, -3), pack4(-4, -6, -8, -12)};
  return Lut16{pack4(-127, -104, -83, -65), pack4(-49, -35, -22, -10), pack4(1, 13, 25, 38),
               pack4(53, 69, 89, 113)};
}

// prmt.b32 in its generic mode: byte i of the result is byte (c_i & 7) of
// {b:a} (a the low four), or, where bit 3 of selector nibble c_i is set,
// that byte's bit 7 copied to all eight bits.  Only the selector's low 16
// bits count.
__device__ __forceinline__ unsigned prmt(unsigned a, unsigned b, unsigned c) {
  unsigned r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// The table applied to the low and the high nibbles of a word: bytes of
// `lo` = table[low nibbles], `hi` = table[high nibbles].  The word's eight
// nibbles, in order low0 high0 low1 high1 ..., serve as byte selectors as
// they stand: a nibble n < 8 picks entry n from the low eight; n ^ 8 picks
// entry n from the high eight when n >= 8 (the other pick, in sign mode, is
// discarded).  Bit 3 of each nibble, replicated over its byte (the msb of
// each byte of q << 4 for the low nibbles, of q for the high ones), chooses
// between the two; one last permute puts the lows and the highs in order.
template <int F>
__device__ __forceinline__ void table_word(unsigned q, unsigned& lo, unsigned& hi) {
  const Lut16 T = level_lut<F>();
  const unsigned qx = q ^ 0x88888888u;
  const unsigned q4 = q << 4;
  const unsigned a0 = prmt(T.t0, T.t1, q), a1 = prmt(T.t2, T.t3, qx);                // low0 high0 low1 high1
  const unsigned b0 = prmt(T.t0, T.t1, q >> 16), b1 = prmt(T.t2, T.t3, qx >> 16);    // low2 high2 low3 high3
  const unsigned ma = prmt(q4, q, 0xD9C8u), mb = prmt(q4, q, 0xFBEAu);
  const unsigned wa = (a0 & ~ma) | (a1 & ma), wb = (b0 & ~mb) | (b1 & mb);
  lo = prmt(wa, wb, 0x6420u);
  hi = prmt(wa, wb, 0x7531u);
}

// The table formats' levels for the integer dots, as two words per four
// values whose entries are all 0..127: P holds the entries of nibbles n < 8,
// N those of n >= 8, each 0 where the other applies (the pick in sign mode
// of a byte whose bit 7 is clear).  IQ4 (lower half negative, upper
// positive): P = -T[n], N = T[n], level = N - P; MXFP4 (upper half the
// negated lower): P = T[n], N = -T[n], level = P - N.  No choice between the
// halves is formed: each half has its own dot.
template <int F>
__host__ __device__ constexpr bool is_table() { return F == 20 || F == 23 || F == 39; }
template <int F>
__device__ __forceinline__ void table_word_pn(unsigned q, unsigned& pl, unsigned& ph, unsigned& nl, unsigned& nh) {
  constexpr bool mx = F == 39;
  constexpr unsigned p0 = mx ? pack4(0, 1, 2, 3) : pack4(127, 104, 83, 65);
  constexpr unsigned p1 = mx ? pack4(4, 6, 8, 12) : pack4(49, 35, 22, 10);
  constexpr unsigned n0 = mx ? pack4(0, 1, 2, 3) : pack4(1, 13, 25, 38);
  constexpr unsigned n1 = mx ? pack4(4, 6, 8, 12) : pack4(53, 69, 89, 113);
  const unsigned qx = q ^ 0x88888888u;
  const unsigned pa = prmt(p0, p1, q), pb = prmt(p0, p1, q >> 16);    // low0 high0 low1 high1, low2 ...
  const unsigned na = prmt(n0, n1, qx), nb = prmt(n0, n1, qx >> 16);
  pl = prmt(pa, pb, 0x6420u);
  ph = prmt(pa, pb, 0x7531u);
  nl = prmt(na, nb, 0x6420u);
  nh = prmt(na, nb, 0x7531u);
}

// The constant some formats subtract from every stored level (Q4_0 8,
// Q5_0 16, Q3_K 4, Q6_K 32).  decode leaves it in the level bytes; the
// integer dots take it out once per half (dot(n - o, h) = dot(n, h) -
// o sum(h), exact), Dequant in the bias of its float conversion.
template <int F>
__host__ __device__ constexpr int level_offset() {
  return F == 2 ? 8 : F == 6 ? 16 : F == 11 ? 4 : F == 14 ? 32 : 0;
}

// Sub-block sb of a staged row in format F: w[0..7] the 32 stored levels
// plus level_offset<F>() four to a word (value 4i + k in byte k of w[i]),
// d/c per half.
// PN (the table formats only): w the P words and wn the N words of
// table_word_pn instead of the levels.
template <int F, bool PN>
__device__ __forceinline__ void decode_impl(const unsigned char* row, int sb, unsigned (&w)[8],
                                            float (&d)[2], float (&c)[2], unsigned (&wn)[8]) {
  c[0] = c[1] = 0.f;
  if constexpr (F == 2 || F == 3 || F == 20) {
    const unsigned char* b = row + sb * blk_bytes(F);
    const unsigned char* qs = b + (F == 3 ? 4 : 2);
    d[0] = d[1] = half_at(b);
    if (F == 3) c[0] = c[1] = half_at(b + 2);
    unsigned qw[4];
    if constexpr (F == 3) {
#pragma unroll
      for (int i = 0; i < 4; ++i) qw[i] = word_at<F>(qs + 4 * i);
    } else {
      words_at<4>(qs, qw);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const unsigned q = qw[i];
      if constexpr (F == 20) {
        if constexpr (PN) table_word_pn<F>(q, w[i], w[4 + i], wn[i], wn[4 + i]);
        else table_word<F>(q, w[i], w[4 + i]);
      } else {
        w[i] = q & 0x0F0F0F0Fu;
        w[4 + i] = (q >> 4) & 0x0F0F0F0Fu;
      }
    }
  } else if constexpr (F == 6 || F == 7) {
    const unsigned char* b = row + sb * blk_bytes(F);
    const unsigned char* hb = b + (F == 7 ? 4 : 2);
    unsigned hw[5];  // the high-bit word, then the four level words
    if constexpr (F == 7) {
#pragma unroll
      for (int i = 0; i < 5; ++i) hw[i] = word_at<F>(hb + 4 * i);
    } else {
      words_at<5>(hb, hw);
    }
    const unsigned qh = hw[0];
    d[0] = d[1] = half_at(b);
    if (F == 7) c[0] = c[1] = half_at(b + 2);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const unsigned q = hw[1 + i];
      w[i] = (q & 0x0F0F0F0Fu) + (spread4(qh >> (4 * i)) << 4);  // disjoint bits: shift-adds
      w[4 + i] = ((q >> 4) & 0x0F0F0F0Fu) + (spread4(qh >> (16 + 4 * i)) << 4);
    }
  } else if constexpr (F == 39) {
    const unsigned char* b = row + sb * 17;
    const unsigned e = u8(b);
    // E8M0 exponent e is 2^(e - 127); halved for the doubled E2M1 values:
    // 2^(e - 128), subnormal below e = 2
    d[0] = d[1] = __uint_as_float(e < 2u ? (0x00200000u << e) : ((e - 1u) << 23));
    unsigned qw[4];
    words_at<4>(b + 1, qw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (PN) table_word_pn<F>(qw[i], w[i], w[4 + i], wn[i], wn[4 + i]);
      else table_word<F>(qw[i], w[i], w[4 + i]);
    }
  } else if constexpr (F == 12 || F == 13) {
    const unsigned char* sup = row + (sb >> 3) * blk_bytes(F);
    const int j = sb & 7;
    // the super-block's 16-byte head (d, dmin, twelve packed 6-bit scales
    // and mins) in one read: the super-blocks sit 16-byte aligned in the row
    const uint4 hd = *(const uint4*)sup;
    // byte 4 + i of the head (scales area byte i, 0 <= i < 12)
    auto sm = [&](int i) {
      const int b = 4 + i;
      const unsigned wv = b < 8 ? hd.y : b < 12 ? hd.z : hd.w;
      return (int)((wv >> (8 * (b & 3))) & 0xFFu);
    };
    int sc, m;
    if (j < 4) {
      sc = sm(j) & 63;
      m = sm(j + 4) & 63;
    } else {
      sc = (sm(j + 4) & 15) | ((sm(j - 4) >> 6) << 4);
      m = (sm(j + 4) >> 4) | ((sm(j) >> 6) << 4);
    }
    d[0] = d[1] = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu))), (float)sc);
    c[0] = c[1] = -__fmul_rn(__half2float(__ushort_as_half((unsigned short)(hd.x >> 16))), (float)m);
    const unsigned char* ql = sup + (F == 12 ? 16 : 48) + (j >> 1) * 32;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const unsigned q = word_at<F>(ql + 4 * i);
      w[i] = (j & 1) ? ((q >> 4) & 0x0F0F0F0Fu) : (q & 0x0F0F0F0Fu);
      if (F == 13) w[i] |= ((word_at<F>(sup + 16 + 4 * i) >> j) & 0x01010101u) << 4;
    }
  } else if constexpr (F == 10) {
    const unsigned char* sup = row + (sb >> 3) * 84;
    const int j = sb & 7, half = j >> 2, k = j & 3;
    const unsigned char* q = sup + 16 + half * 32;
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = (word_at<F>(q + 4 * i) >> (2 * k)) & 0x03030303u;
    const float D = half_at(sup + 80), DM = half_at(sup + 82);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int s = sup[half * 8 + k * 2 + h];
      d[h] = __fmul_rn(D, (float)(s & 15));
      c[h] = -__fmul_rn(DM, (float)(s >> 4));
    }
  } else if constexpr (F == 11) {
    const unsigned char* sup = row + (sb >> 3) * 110;
    const int j = sb & 7, half = j >> 2, k = j & 3, bit = half * 4 + k;
    const unsigned char* q = sup + 32 + half * 32;
    unsigned qw[8], mw[8];
    words_at_sh<8>(q, 2u * k, qw);
    words_at_sh<8>(sup, (unsigned)bit, mw);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const unsigned low2 = qw[i] & 0x03030303u;
      const unsigned mb = mw[i] & 0x01010101u;  // set: +0, clear: -4
      w[i] = low2 + (mb << 2);                    // disjoint bits: one shift-add
    }
    const unsigned char* s12 = sup + 96;
    const float D = half_at(sup + 108);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = half * 8 + k * 2 + h;
      const int lo4 = i < 8 ? (s12[i] & 15) : (s12[i - 8] >> 4);
      const int hi2 = (s12[8 + (i & 3)] >> (2 * (i >> 2))) & 3;
      d[h] = __fmul_rn(D, (float)((lo4 | (hi2 << 4)) - 32));
    }
  } else if constexpr (F == 14) {
    const unsigned char* sup = row + (sb >> 3) * 210;
    const int j = sb & 7, half = j >> 2, k = j & 3;
    const unsigned char* ql = sup + half * 64 + (k & 1) * 32;
    const unsigned char* qh = sup + 128 + half * 32;
    unsigned lw[8], hw[8];
    words_at_sh<8>(ql, 4u * (k >> 1), lw);
    words_at_sh<8>(qh, 2u * k, hw);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const unsigned lo = lw[i] & 0x0F0F0F0Fu;
      const unsigned hi = hw[i] & 0x03030303u;
      w[i] = lo + (hi << 4);  // disjoint bits: one shift-add
    }
    const float D = half_at(sup + 208);
    d[0] = __fmul_rn(D, (float)(signed char)sup[192 + half * 8 + 2 * k]);
    d[1] = __fmul_rn(D, (float)(signed char)sup[192 + half * 8 + 2 * k + 1]);
  } else if constexpr (F == 23) {
    const unsigned char* sup = row + (sb >> 3) * 136;
    const int j = sb & 7;
    const int sh = sup[2] | (sup[3] << 8);
    const int ls = ((sup[4 + (j >> 1)] >> (4 * (j & 1))) & 15) | (((sh >> (2 * j)) & 3) << 4);
    d[0] = d[1] = __fmul_rn(half_at(sup), (float)(ls - 32));
    const unsigned char* qs = sup + 8 + 16 * j;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (PN) table_word_pn<F>(word_at<F>(qs + 4 * i), w[i], w[4 + i], wn[i], wn[4 + i]);
      else table_word<F>(word_at<F>(qs + 4 * i), w[i], w[4 + i]);
    }
  }
}
template <int F>
__device__ __forceinline__ void decode(const unsigned char* row, int sb, unsigned (&w)[8], float (&d)[2],
                                       float (&c)[2]) {
  decode_impl<F, false>(row, sb, w, d, c, w);
}


// f32 part of one sub-block for one activation row: ((d0 dh0 + c0 sh0) +
// d1 dh1) + c1 sh1, each product and sum rounded; sh: the activation
// halves' sums (exact integers, formed once when the rows are staged).
// A sub-block's term from its halves' exact integer dots dh0, dh1 and
// activation sums sh0, sh1: ((d0 dh0 + c0 sh0) + d1 dh1) + c1 sh1, each
// product and sum rounded to f32.
__device__ __forceinline__ float sub_combine(const float (&d)[2], const float (&c)[2], int dh0, int dh1, int sh0,
                                             int sh1) {
  float p = __fmul_rn(d[0], (float)dh0);
  p = __fadd_rn(p, __fmul_rn(c[0], (float)sh0));
  p = __fadd_rn(p, __fmul_rn(d[1], (float)dh1));
  return __fadd_rn(p, __fmul_rn(c[1], (float)sh1));
}

template <int O>
__device__ __forceinline__ float sub_part(const unsigned (&w)[8], const float (&d)[2], const float (&c)[2],
                                          const unsigned (&h)[8], int2 sh) {
  int dh0 = 0, dh1 = 0;
  const int sh0 = sh.x, sh1 = sh.y;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    dh0 = __dp4a((int)w[i], (int)h[i], dh0);
    dh1 = __dp4a((int)w[4 + i], (int)h[4 + i], dh1);
  }
  if (O) {
    dh0 -= O * sh0;
    dh1 -= O * sh1;
  }
  return sub_combine(d, c, dh0, dh1, sh0, sh1);
}

// The table formats' term from their P and N words (table_word_pn): each
// half's exact integer dot is the difference of two dots.
template <int F>
__device__ __forceinline__ float sub_part_pn(const unsigned (&wp)[8], const unsigned (&wn)[8], const float (&d)[2],
                                             const float (&c)[2], const unsigned (&h)[8], int2 sh) {
  int p0 = 0, p1 = 0, n0 = 0, n1 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    p0 = __dp4a((int)wp[i], (int)h[i], p0);
    p1 = __dp4a((int)wp[4 + i], (int)h[4 + i], p1);
    n0 = __dp4a((int)wn[i], (int)h[i], n0);
    n1 = __dp4a((int)wn[4 + i], (int)h[4 + i], n1);
  }
  const int dh0 = F == 39 ? p0 - n0 : n0 - p0, dh1 = F == 39 ? p1 - n1 : n1 - p1;
  return sub_combine(d, c, dh0, dh1, sh.x, sh.y);
}


__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((unsigned)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct BlkArgs {
  const unsigned char* w;  // N rows of rb bytes (16-byte aligned, rb % 16 == 0)
  long rb;
  int N, K, M, mode;
  const float* x;          // Dequant [M][K]
  const int8_t* xq;        // [M][K]
  const int8_t* xl;        // [M][K] (TwoPass)
  const float* xs;         // [M][K/32]
  float* y;                // [M][N]
  float* dq;               // dequant hook: [N][K] (or NULL)
  int pdl;
  unsigned act_stride;     // bytes per activation row in shared memory
  unsigned act_bytes;      // the activation area
  unsigned rb_pad;         // one row buffer (rb rounded up to 16, plus 16)
};

// Padded shared-memory index of value k of an activation row: 16 bytes of
// padding after every 32 values (of `bytes` bytes each).
__device__ __forceinline__ unsigned pad_index(unsigned k, unsigned bytes) {
  return (k >> 5) * (32u * bytes + 16u) + (k & 31u) * bytes;
}

// The activation rows into shared memory (all threads; after the dependency
// wait): words (and low words) with the padding, scales dense; or f32 values.
template <int Q, int MM>
__device__ __forceinline__ void stage_act(const BlkArgs& a, unsigned char* act) {
  const int K = a.K;
  if constexpr (Q == 0) {
    for (int t = 0; t < a.M; ++t)
      for (int i = threadIdx.x; i < K / 4; i += blockDim.x) {
        const float4 v = __ldcg((const float4*)(a.x + (long)t * K) + i);
        *(float4*)(act + (size_t)t * a.act_stride + pad_index(4u * i, 4u)) = v;
      }
  } else {
    const unsigned nb = (unsigned)K / 32u;
    // the byte sum of a 16-value half, exact
    auto sum16 = [](uint4 v) {
      int r = __dp4a((int)v.x, 0x01010101, 0);
      r = __dp4a((int)v.y, 0x01010101, r);
      r = __dp4a((int)v.z, 0x01010101, r);
      return __dp4a((int)v.w, 0x01010101, r);
    };
    for (int t = 0; t < a.M; ++t) {
      unsigned char* base = act + (size_t)t * a.act_stride;
      float* s = (float*)(base + nb * 48u * (Q == 2 ? 2u : 1u));
      int* sums = (int*)(s + nb);  // [2 nb] halves of the words, then [2 nb] of the low words
      for (int i = threadIdx.x; i < K / 16; i += blockDim.x) {
        const uint4 hv = __ldcg((const uint4*)(a.xq + (long)t * K) + i);
        *(uint4*)(base + pad_index(16u * i, 1u)) = hv;
        sums[i] = sum16(hv);
        if (Q == 2) {
          const uint4 lv = __ldcg((const uint4*)(a.xl + (long)t * K) + i);
          *(uint4*)(base + pad_index(16u * i, 1u) + nb * 48u) = lv;
          sums[2 * nb + i] = sum16(lv);
        }
      }
      for (int i = threadIdx.x; i < (int)nb; i += blockDim.x) s[i] = __ldcg(a.xs + (long)t * nb + i);
    }
  }
}

template <int F, int Q, int MM>
__global__ void __launch_bounds__(BW * 32) gemv_blk_kernel(const BlkArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned char* act = smem;
  unsigned char* bufs = smem + a.act_bytes + (size_t)warp * 2 * a.rb_pad;
  const int K = a.K, nb = K >> 5;
  const long stride = (long)gridDim.x * nw;
  long row = (long)blockIdx.x * nw + warp;
  if (a.pdl && threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" :::);
  // the first row's bytes (weights: no dependence on the previous kernel)
  auto fetch = [&](long r, unsigned char* dst) {
    if (r < a.N) {
      const unsigned char* src = a.w + r * a.rb;
      for (long o = 16 * lane; o < a.rb; o += 512) cp_async16(dst + o, src + o);
    }
    cp_commit();
  };
  fetch(row, bufs);
  if (a.pdl) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (a.dq == nullptr) stage_act<Q, MM>(a, act);
  __syncthreads();
  int cur = 0;
  for (; row < a.N; row += stride) {
    fetch(row + stride, bufs + (cur ^ 1) * a.rb_pad);
    cp_wait<1>();
    __syncwarp();
    const unsigned char* rbuf = bufs + cur * a.rb_pad;
    if (a.dq) {
      // the decode hook: every value as the CPU dequantizer rounds it
      for (int sb = lane; sb < nb; sb += 32) {
        unsigned w[8];
        float d[2], c[2];
        decode<F>(rbuf, sb, w, d, c);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float v = (float)((int)(signed char)(w[i >> 2] >> (8 * (i & 3))) - level_offset<F>());
          a.dq[row * (long)K + 32 * sb + i] = __fadd_rn(__fmul_rn(d[i >> 4], v), c[i >> 4]);
        }
      }
    } else if constexpr (Q == 0) {
      float s1[MM], s2[MM];  // a lane's sum and its compensation, per activation row
#pragma unroll
      for (int t = 0; t < MM; ++t) s1[t] = s2[t] = 0.f;
      for (int sb = lane; sb < nb; sb += 32) {
        unsigned w[8];
        float d[2], c[2];
        decode<F>(rbuf, sb, w, d, c);
        // the weights RN(RN(d level) + c) as packed pairs (values 4q + k and
        // 4q + k + 2 of word q): the level bytes placed in the mantissa of
        // 2^23 + 128 + b and the bias subtracted (exact), then the scale and
        // the offset, each rounded as the scalar form
        f32x2 wv[16];
        constexpr float B = -8388736.0f - (float)level_offset<F>();  // -(2^23 + 128 + offset), exact
        const f32x2 bias = f2_pack(B, B);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const unsigned u = w[q] ^ 0x80808080u;
          const f32x2 dd = f2_pack(d[q >> 2], d[q >> 2]), cc = f2_pack(c[q >> 2], c[q >> 2]);
          wv[2 * q] = f2_add(f2_mul(dd, f2_add(f2_pack(i8_bits_f32(u, 0), i8_bits_f32(u, 2)), bias)), cc);
          wv[2 * q + 1] = f2_add(f2_mul(dd, f2_add(f2_pack(i8_bits_f32(u, 1), i8_bits_f32(u, 3)), bias)), cc);
        }
#pragma unroll
        for (int t = 0; t < MM; ++t) {
          if (t >= a.M) break;
          const float* xr = (const float*)(act + (size_t)t * a.act_stride + pad_index(32u * sb, 4u));
          // two interleaved chains of products (the tolerance, not the
          // pages' order, binds Dequant), joined at the sub-block's end
          f32x2 acc2 = f2_pack(0.f, 0.f);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 xv = *(const float4*)(xr + 4 * q);
            acc2 = f2_fma(wv[2 * q], f2_pack(xv.x, xv.z), acc2);
            acc2 = f2_fma(wv[2 * q + 1], f2_pack(xv.y, xv.w), acc2);
          }
          float a0, a1;
          f2_unpack(acc2, a0, a1);
          const float acc = __fadd_rn(a0, a1);
          // s1 + s2 += acc (Kahan-Babuska: the rounding error kept in s2)
          const float sum = __fadd_rn(s1[t], acc);
          const float bp = __fsub_rn(sum, s1[t]);
          s2[t] = __fadd_rn(s2[t], __fadd_rn(__fsub_rn(s1[t], __fsub_rn(sum, bp)), __fsub_rn(acc, bp)));
          s1[t] = sum;
        }
      }
#pragma unroll
      for (int t = 0; t < MM; ++t) {
        if (t >= a.M) break;
        double v = (double)s1[t] + (double)s2[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
        if (lane == 0) a.y[(long)t * a.N + row] = (float)v;
      }
    } else {
      float acc[MM];
#pragma unroll
      for (int t = 0; t < MM; ++t) acc[t] = 0.f;
      const unsigned nbu = (unsigned)nb;
#pragma unroll 2
      for (int sb = lane; sb < nb; sb += 32) {
        unsigned w[8], wn[8];
        float d[2], c[2];
        decode_impl<F, is_table<F>()>(rbuf, sb, w, d, c, wn);
#pragma unroll
        for (int t = 0; t < MM; ++t) {
          if (t >= a.M) break;
          const unsigned char* base = act + (size_t)t * a.act_stride;
          const unsigned char* hp = base + pad_index(32u * sb, 1u);
          unsigned h[8];
          *(uint4*)&h[0] = *(const uint4*)hp;
          *(uint4*)&h[4] = *(const uint4*)(hp + 16);
          const float* srow = (const float*)(base + nbu * 48u * (Q == 2 ? 2u : 1u));
          const int2* sums = (const int2*)(srow + nbu);
          float part = is_table<F>() ? sub_part_pn<F>(w, wn, d, c, h, sums[sb])
                                     : sub_part<level_offset<F>()>(w, d, c, h, sums[sb]);
          if constexpr (Q == 2) {
            const unsigned char* lp = hp + nbu * 48u;
            unsigned l[8];
            *(uint4*)&l[0] = *(const uint4*)lp;
            *(uint4*)&l[4] = *(const uint4*)(lp + 16);
            const float lpart = is_table<F>() ? sub_part_pn<F>(w, wn, d, c, l, sums[nbu + sb])
                                              : sub_part<level_offset<F>()>(w, d, c, l, sums[nbu + sb]);
            part = __fadd_rn(part, __fmul_rn(0.0078125f, lpart));
          }
          const float s = srow[sb];
          acc[t] = __fadd_rn(acc[t], __fmul_rn(s, part));
        }
      }
#pragma unroll
      for (int t = 0; t < MM; ++t) {
        if (t >= a.M) break;
        float v = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, o));
        if (lane == 0) a.y[(long)t * a.N + row] = v;
      }
    }
    __syncwarp();
    cur ^= 1;
  }
  cp_wait<0>();
}

typedef void (*blk_fn)(const BlkArgs);

template <int F>
blk_fn pick_q(int mode, int M) {
  if (mode == 0) return M <= 1 ? gemv_blk_kernel<F, 0, 1> : M <= 4 ? gemv_blk_kernel<F, 0, 4> : gemv_blk_kernel<F, 0, 8>;
  if (mode == 1) return M <= 1 ? gemv_blk_kernel<F, 1, 1> : M <= 4 ? gemv_blk_kernel<F, 1, 4> : gemv_blk_kernel<F, 1, 8>;
  return M <= 1 ? gemv_blk_kernel<F, 2, 1> : M <= 4 ? gemv_blk_kernel<F, 2, 4> : gemv_blk_kernel<F, 2, 8>;
}

blk_fn pick(int F, int mode, int M) {
  switch (F) {
    case 2: return pick_q<2>(mode, M);
    case 3: return pick_q<3>(mode, M);
    case 6: return pick_q<6>(mode, M);
    case 7: return pick_q<7>(mode, M);
    case 10: return pick_q<10>(mode, M);
    case 11: return pick_q<11>(mode, M);
    case 12: return pick_q<12>(mode, M);
    case 13: return pick_q<13>(mode, M);
    case 14: return pick_q<14>(mode, M);
    case 20: return pick_q<20>(mode, M);
    case 23: return pick_q<23>(mode, M);
    case 39: return pick_q<39>(mode, M);
    default: return nullptr;
  }
}

// Row bytes of format F at K values (0: unknown format or not whole blocks).
long row_bytes(int F, int K) {
  const int v = blk_values(F);
  if (!v || K <= 0 || K % v) return 0;
  return (long)(K / v) * blk_bytes(F);
}

lk_status launch(int F, const unsigned char* w, int N, int K, int mode, const float* x, const int8_t* xq,
                 const int8_t* xl, const float* xs, int M, float* y, float* dq, const lk_launch_cfg* cfg,
                 cudaStream_t stream) {
  const lkh::DeviceInfo* dev = lkh::device_info(nullptr);
  if (!dev) return LK_ERR_CUDA;
  BlkArgs a;
  a.w = w;
  a.rb = row_bytes(F, K);
  a.N = N;
  a.K = K;
  a.M = M;
  a.mode = mode;
  a.x = x;
  a.xq = xq;
  a.xl = xl;
  a.xs = xs;
  a.y = y;
  a.dq = dq;
  a.pdl = lkh::cfg_pdl(cfg);
  const unsigned nb = (unsigned)K / 32u;
  a.act_stride = dq ? 0u
                    : mode == 0 ? nb * (32u * 4u + 16u)
                                : ((nb * 48u * (mode == 2 ? 2u : 1u) + nb * 4u + nb * 8u * (mode == 2 ? 2u : 1u) +
                                    15u) & ~15u);
  a.act_bytes = a.act_stride * (unsigned)(dq ? 0 : M);
  // 16 bytes of slack after a row: a word read at the row's last bytes may
  // load the aligned word after them
  a.rb_pad = (unsigned)((a.rb + 15) & ~15L) + 16u;
  // (less a small margin)
  long room = (long)dev->smem_optin - 256L - (long)a.act_bytes;
  int nw = room > 0 ? (int)(room / (2L * a.rb_pad)) : 0;
  if (nw > BW) nw = BW;
  if (nw < 1) return LK_ERR_SHAPE;
  const unsigned total = a.act_bytes + (unsigned)nw * 2u * a.rb_pad;
  blk_fn f = pick(F, dq ? 1 : mode, dq ? 1 : M);
  if (!f) return LK_ERR_ARG;
  // the dynamic cap: the device's opt-in maximum less the kernel's static
  // shared memory (the two together may not exceed it)
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, f) != cudaSuccess) return LK_ERR_CUDA;
  if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           dev->smem_optin - (int)fa.sharedSizeBytes) != cudaSuccess)
    return LK_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, nw * 32, total) != cudaSuccess || per_sm < 1)
    return LK_ERR_SHAPE;
  long blocks = ((long)N + nw - 1) / nw;
  const long cap = (long)dev->sm_count * per_sm;
  if (cfg && cfg->grid_ctas > 0) blocks = cfg->grid_ctas < blocks ? cfg->grid_ctas : blocks;
  else if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)blocks);
  lc.blockDim = dim3(nw * 32);
  lc.dynamicSmemBytes = total;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = a.pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&lc, f, a) != cudaSuccess) return LK_ERR_CUDA;
  return lkh::launch_status();
}

}  // namespace lkblk

using lkh::aligned;

extern "C" {

size_t lk_format_row_bytes(int format, int K) { return (size_t)lkblk::row_bytes(format, K); }

lk_status lk_gemv_blk(int format, const uint8_t* w, int N, int K, lk_mode mode, const float* x, const int8_t* xq,
                      const int8_t* xl, const float* xs, int M, float* y, const lk_launch_cfg* cfg,
                      cudaStream_t stream) {
  if (mode < LK_DEQUANT || mode > LK_TWOPASS || lkh::check_launch_cfg(cfg)) return LK_ERR_ARG;
  if (lkblk::blk_values(format) == 0) return LK_ERR_ARG;
  const long rb = lkblk::row_bytes(format, K);
  if (N < 0 || M < 0 || M > LK_MAX_M || K < 0 || (K > 0 && (rb == 0 || K % 256 || rb % 16))) return LK_ERR_SHAPE;
  if (N == 0 || M == 0 || K == 0) {
    if (K == 0 && N > 0 && M > 0 && y) cudaMemsetAsync(y, 0, sizeof(float) * (size_t)M * (size_t)N, stream);
    return K == 0 && N > 0 && M > 0 && !y ? LK_ERR_ARG : LK_OK;
  }
  if (!w || !y) return LK_ERR_ARG;
  if (mode == LK_DEQUANT ? !x : (!xq || !xs || (mode == LK_TWOPASS && !xl))) return LK_ERR_ARG;
  if (!aligned(w, 16) || !aligned(y, 4)) return LK_ERR_ALIGN;
  if (mode == LK_DEQUANT ? !aligned(x, 16)
                         : (!aligned(xq, 16) || !aligned(xs, 4) || (mode == LK_TWOPASS && !aligned(xl, 16))))
    return LK_ERR_ALIGN;
  return lkblk::launch(format, w, N, K, mode, x, xq, xl, xs, M, y, nullptr, cfg, stream);
}

lk_status lk_dequant_blk(int format, const uint8_t* w, int N, int K, float* out, cudaStream_t stream) {
  if (lkblk::blk_values(format) == 0) return LK_ERR_ARG;
  const long rb = lkblk::row_bytes(format, K);
  if (N < 0 || K < 0 || (K > 0 && (rb == 0 || K % 256 || rb % 16))) return LK_ERR_SHAPE;
  if (N == 0 || K == 0) return LK_OK;
  if (!w || !out) return LK_ERR_ARG;
  if (!aligned(w, 16) || !aligned(out, 4)) return LK_ERR_ALIGN;
  return lkblk::launch(format, w, N, K, LK_INT8ACT, nullptr, nullptr, nullptr, nullptr, 1, nullptr, out, nullptr,
                       stream);
}

}  // extern "C"
