// Small-batch Q8_0 GEMV on the tensor cores (Int8Act and TwoPassInt8, 2..8
// activation rows), sm_103a.
//
// At batch 8 every weight byte meets 8 activation rows: the block dots form a
// dense int8 contraction [N x K] x [K x 8].  This kernel runs it as
// mma.sync m16n8k16 with f16 operands and f32 accumulators: the int8 levels
// (weights and activation hi/lo words) are exact in f16, every product is an
// integer of magnitude <= 2^14, and one 32-block's dot (two k16 MMAs) stays
// below 2^20, so the accumulator holds the exact int32 dot d (and e).  The
// combine is then the same per-block f32 chain as every other path
// ("kernels.rs" lk_q8_term / lk_q8_acc, partial b mod 4 in ascending block
// order, (p0 + p2) + (p1 + p3)): the result has the same bits as the M = 1
// kernels and the oracle.
//
// Fragments.  A warp owns a tile of 16 weight rows; its 32 lanes are 8
// groups g of 4 lanes t.  Inside a 32-block the k order of both operands is
// permuted the same way so that lane (g, t) reads 8 contiguous bytes:
// physical bytes 8t..8t+3 are the first MMA's k slots {2t, 2t+1, 2t+8,
// 2t+9}, bytes 8t+4..8t+7 the second MMA's.  The A fragment (weights) is rows
// g and g+8, the B fragment (activations) is activation row g, and the
// accumulator gives rows g, g+8 x activation rows 2t, 2t+1.  Activation rows
// >= M read as zeros.  The int8 -> f16 step is exact: (0x6400 | (b ^ 0x80))
// is the f16 1024 + b + 128, minus 1152.
//
// More than 8 activation rows (up to LK_MAX_BATCH): the rows form groups of
// 8 (blockIdx.y), each group with its own share of the SMs (gridDim.x blocks
// per group) running the 8-row arithmetic above over every tile.  All groups
// run at once, so a tile is read from HBM once and from L2 by the other
// groups at about the same time; each (row, activation) value is computed
// exactly as at 8 rows.
//
// Data movement is the ring kernel's: weights stream through per-warp ring
// slots by 1-D bulk copies (TMA) completing on mbarriers, every wait bounded.
// A stage is one tile's slice of tk bytes of K: 16 copies of a weight row
// slice into rows padded to tk + 32 bytes (rows g and g + 4 then fall in
// different banks, so the warp's 8-byte reads take the minimum two
// wavefronts) and 16 copies of the matching scale slices.  The activation
// rows (int8 words, scales) are copied once per block into shared memory, row
// stride K + 32 bytes for the same reason.  Tiles are dealt to warps across
// the grid first (tile i -> block i mod grid, then warp), so small matrices
// still spread over every SM.
//
// Split-K (lk_gemv_q8_splitk, S chunks): blockIdx.z is the chunk.  A block
// holds only its chunk's columns of the activation rows (so long rows leave
// room for more stages) and runs every tile over the chunk's blocks
// [4 floor(c G / S), 4 floor((c + 1) G / S)) (G = K / 128, the last chunk
// ending at K / 32): partial index = global block index mod 4 (chunks start
// on a multiple of 4 blocks), and the chunk's (p0 + p2) + (p1 + p3) goes to
// part[c][t][o].  The blocks of a row group are split evenly over the
// chunks, so the tiles x chunks work units still spread over every SM.
#include "lk_ring_kernel.cuh"

namespace lkmma {

using namespace lk;
using namespace lkring;

constexpr int TR = 16;          // weight rows per tile (the MMA's M)
constexpr int TN = 8;           // activation rows per tile (the MMA's N)
constexpr int MW = 16;          // warps per block at most
constexpr int MST = 32;         // ring stages per block at most
// barriers (one per stage + the activation's), abort flag, argmax keys [8][MW]
constexpr unsigned MTAIL = 8 * (MST + 1) + 16 + 8 * TN * MW;

constexpr int MG = LK_MAX_GROUP;  // matrices of one grouped launch at most

struct MmaArgs {
  lkh::GemvProblem p;      // activations, K, M, mode, argmax keys (one matrix only)
  int nmat;                // matrices sharing the activation (1..MG)
  const int8_t* wq[MG];
  const unsigned char* ws[MG];  // f16 scales, as bytes
  long N[MG];
  float* y[MG];
  long tile0[MG + 1];      // first tile of matrix m; tile0[nmat] = all tiles
  int nw;                  // warps per block
  int depth;               // ring stages per warp
  int gx;                  // blocks per activation-row group (gridDim.x)
  long ntiles;             // sum over the matrices of ceil(N / 16)
  unsigned tk;             // bytes of K per stage (multiple of 256)
  unsigned rs;             // stage row stride (tk + 32)
  unsigned srs;            // stage scale row stride (tk / 16 + 16)
  unsigned s_off;          // scale area inside a stage (16 * rs)
  unsigned stage_bytes;
  unsigned ar;             // activation row stride, bytes (K + 32)
  unsigned xsr;            // activation scale row stride, floats (K / 32 + 4)
  unsigned a_lo, a_xs;     // offsets of the low words and the scales in the activation area
  unsigned ring_off;
  unsigned long long wait_ns;
  unsigned long long pol_w;
  int pdl;
  int* err;
  unsigned long long* trace;  // option "trace" 3: the launch timeline, else NULL
  int tslot;
  int prefill;             // warps that fill their stages before the dependency wait
  int S;                   // split-K chunks (gridDim.z), 1: the plain GEMV
  long part_stride;        // split-K: elements of one chunk's partials (M * N)
};

// This block's split-K chunk: its first 32-block and its length in bytes of
// K (the whole row when S == 1).
struct Chunk {
  int k_lo, kc;
};
__device__ __forceinline__ Chunk chunk_of(const MmaArgs& ra) {
  const int nb = ra.p.K >> 5;
  if (ra.S <= 1) return Chunk{0, ra.p.K};
  const int b_lo = splitk_bound(nb, ra.S, blockIdx.z), b_hi = splitk_bound(nb, ra.S, blockIdx.z + 1);
  return Chunk{32 * b_lo, 32 * (b_hi - b_lo)};
}

// int8 x 4 (b0 lowest) -> two f16x2: (b0, b1) and (b2, b3), exact.
__device__ __forceinline__ void i8x4_to_h2(unsigned w, unsigned& lo, unsigned& hi) {
  const unsigned u = w ^ 0x80808080u;
  const unsigned a = __byte_perm(u, 0x64646464u, 0x4140);
  const unsigned b = __byte_perm(u, 0x64646464u, 0x4342);
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

struct Frag8 {   // one 8-byte run of levels as the two MMAs' f16 pairs
  unsigned m0lo, m0hi, m1lo, m1hi;
};
__device__ __forceinline__ Frag8 frag8(uint2 v) {
  Frag8 f;
  i8x4_to_h2(v.x, f.m0lo, f.m0hi);
  i8x4_to_h2(v.y, f.m1lo, f.m1hi);
  return f;
}

// d += A(16x16, rows g/g+8) * B(16x8, column g), f32 accumulate
__device__ __forceinline__ void mma16816(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                         unsigned b0, unsigned b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d += A(16x32 int8, rows g/g+8) * B(32x8 int8, column g), exact int32
// (m16n8k32: a0/a2 row g, a1/a3 row g+8, each 4 consecutive k; b0/b1 4 k each)
__device__ __forceinline__ void imma16832(int (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                          unsigned b0, unsigned b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The block's exact dot on the int8 tensor path: lane (g, t)'s 8 bytes of
// each operand are the k slots {4t..4t+3} (first word) and {4t+16..4t+19}
// (second word) of one m16n8k32, the same permutation for A and B.  The
// int32 result (|d| < 2^20) becomes an f32 by the magic-number add: its bits
// added to those of 1.5 * 2^23, minus 1.5 * 2^23, exactly.
__device__ __forceinline__ void block_dot_i8(float (&d)[4], uint2 w0, uint2 w8, uint2 x) {
  int di[4] = {0, 0, 0, 0};
  imma16832(di, w0.x, w8.x, w0.y, w8.y, x.x, x.y);
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] = __fadd_rn(__int_as_float(di[e] + 0x4B400000), -12582912.0f);
}

// The block's exact dot for rows (g, g+8) x activation rows (2t, 2t+1).
__device__ __forceinline__ void block_dot(float (&d)[4], const Frag8& wg, const Frag8& wg8, const Frag8& x) {
  d[0] = d[1] = d[2] = d[3] = 0.f;
  mma16816(d, wg.m0lo, wg8.m0lo, wg.m0hi, wg8.m0hi, x.m0lo, x.m0hi);
  mma16816(d, wg.m1lo, wg8.m1lo, wg.m1hi, wg8.m1hi, x.m1lo, x.m1hi);
}

// The B fragment of activation row g for the 32-block at level offset k:
// read as f16 (A16) or as int8 and converted; zeros for rows >= M.
template <bool A16>
__device__ __forceinline__ Frag8 act_frag(const unsigned char* X, int k, bool ok) {
  if (A16) {
    const uint4 v = ok ? *(const uint4*)(X + 2 * k) : make_uint4(0u, 0u, 0u, 0u);
    return Frag8{v.x, v.y, v.z, v.w};
  }
  return frag8(ok ? *(const uint2*)(X + k) : make_uint2(0u, 0u));
}


struct Tiles {
  long base, stride, ntiles;
  int nsl;
};

// A position in a warp's stage sequence (tile, slice), advanced without
// divisions: slice c of tile base + stride * r.
struct Cursor {
  long tile;
  int c;
  __device__ __forceinline__ void next(const Tiles& tl) {
    if (++c == tl.nsl) {
      c = 0;
      tile += tl.stride;
    }
  }
};

// The matrix a tile belongs to, with constant indices into the launch
// arguments (no local-memory copy of the arrays).
struct Mat {
  const int8_t* wq;
  const unsigned char* ws;
  long N;
  float* y;
  long row0;  // the tile's first row in its matrix
};
__device__ __forceinline__ Mat mat_of(const MmaArgs& ra, long tile) {
  Mat m{ra.wq[0], ra.ws[0], ra.N[0], ra.y[0], tile * TR};
#pragma unroll
  for (int i = 1; i < MG; ++i)
    if (i < ra.nmat && tile >= ra.tile0[i]) m = Mat{ra.wq[i], ra.ws[i], ra.N[i], ra.y[i], (tile - ra.tile0[i]) * TR};
  return m;
}

// Bytes between a stage's scale row start (a 16-byte boundary) and the
// scale of level offset k0 (a multiple of 128): 0 or 8.
__device__ __forceinline__ unsigned scale_shift(int k0) { return (unsigned)((k0 >> 5) & 7) * 2u; }

// Slice c of tile `tile` (of the chunk ch) into the stage buffer st,
// completing on `full`.
__device__ __forceinline__ void issue(const MmaArgs& ra, const Chunk& ch, long tile, int c, unsigned char* st,
                                      unsigned full, unsigned long long pol, int lane) {
  const int K = ra.p.K;
  const Mat m = mat_of(ra, tile);
  const int rows = m.N - m.row0 < TR ? (int)(m.N - m.row0) : TR;
  const int kl = c * (int)ra.tk;
  const int len = ch.kc - kl < (int)ra.tk ? ch.kc - kl : (int)ra.tk;
  const int k0 = ch.k_lo + kl;
  // a row's scales from the 16-byte boundary at or before them (a chunk may
  // start 4 blocks = 8 bytes past one): scale_shift(k0) bytes of lead
  const unsigned sh = scale_shift(k0);
  const unsigned slen = ((unsigned)len / 16u + sh + 15u) & ~15u;
  if (lane == 0) mbar_arrive_expect_tx(full, (unsigned)rows * ((unsigned)len + slen));
  __syncwarp();
  const int r = lane & 15;
  if (r < rows) {
    const long row = m.row0 + r;
    if (lane < 16)
      bulk(st + r * ra.rs, m.wq + row * K + k0, (unsigned)len, full, pol);
    else
      bulk(st + ra.s_off + r * ra.srs, m.ws + (row * (K >> 5) + (k0 >> 5)) * 2 - sh, slen, full, pol);
  }
  __syncwarp();
}

// The activation rows into shared memory (all threads call it, after the
// dependency wait): f16 rows converted by every thread (A16), or the int8
// rows by warp 0's bulk copies completing on act_bar (bounded wait).
// Returns false when that wait gave up.
template <int Q, bool A16>
__device__ __forceinline__ bool load_rows(const MmaArgs& ra, const Chunk& ch, int M, int row0, unsigned char* act,
                                          unsigned act_bar, volatile int* abort_flag) {
  const lkh::GemvProblem& a = ra.p;
  const int KG = a.K, nbg = KG >> 5;  // the rows' length in global memory
  const int K = ch.kc, nb = K >> 5;   // the chunk's columns, held from offset 0
  // this block's group of activation rows: rows row0 .. row0 + M - 1, from
  // the chunk's first column
  const int8_t* gxq = a.xq + (long)row0 * KG + ch.k_lo;
  const int8_t* gxl = Q == 2 ? a.xl + (long)row0 * KG + ch.k_lo : nullptr;
  const float* gxs = a.xs + (long)row0 * nbg + (ch.k_lo >> 5);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // the activation rows: int8 words (and low words) and scales, row-padded
  if (A16) {
    // every thread converts 16-byte runs of the int8 rows into f16 rows
    const int runs = K >> 4, nrun = M * runs * (Q == 2 ? 2 : 1);
    constexpr int U = 4;  // loads in flight per thread
    for (int i0 = threadIdx.x; i0 < nrun; i0 += U * blockDim.x) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i < nrun) {
          const int lo = Q == 2 && i >= M * runs;
          const int j = lo ? i - M * runs : i;
          const int row = j / runs, off = (j - row * runs) << 4;
          v[u] = ld_cg16((lo ? gxl : gxq) + (long)row * KG + off);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i < nrun) {
          const int lo = Q == 2 && i >= M * runs;
          const int j = lo ? i - M * runs : i;
          const int row = j / runs, off = (j - row * runs) << 4;
          uint4 h0, h1;
          i8x4_to_h2(v[u].x, h0.x, h0.y);
          i8x4_to_h2(v[u].y, h0.z, h0.w);
          i8x4_to_h2(v[u].z, h1.x, h1.y);
          i8x4_to_h2(v[u].w, h1.z, h1.w);
          uint4* dst = (uint4*)(act + (lo ? ra.a_lo : 0u) + (size_t)row * ra.ar + 2 * off);
          dst[0] = h0;
          dst[1] = h1;
        }
      }
    }
    for (int i = threadIdx.x; i < M * nb; i += blockDim.x) {
      const int row = i / nb, b = i - row * nb;
      ((float*)(act + ra.a_xs))[(size_t)row * ra.xsr + b] = __ldcg(gxs + (long)row * nbg + b);
    }
    __syncthreads();
  } else if (warp == 0) {
    // int8 rows as they are, by bulk copies: with few warps (long K, few
    // tiles) plain loads of up to 200 KB take several round trips, while
    // the copies' wait behind the weight stages issued before them is short
    const unsigned long long pol_a = evict_last_policy();
    if (lane == 0)
      mbar_arrive_expect_tx(act_bar, (unsigned)M * ((unsigned)K * (Q == 2 ? 2u : 1u) + (unsigned)nb * 4u));
    __syncwarp();
    if (lane < M) bulk(act + (size_t)lane * ra.ar, gxq + (long)lane * KG, (unsigned)K, act_bar, pol_a);
    if (Q == 2 && lane >= 8 && lane < 8 + M)
      bulk(act + ra.a_lo + (size_t)(lane - 8) * ra.ar, gxl + (long)(lane - 8) * KG, (unsigned)K, act_bar, pol_a);
    if (lane >= 16 && lane < 16 + M)
      bulk(act + ra.a_xs + (size_t)(lane - 16) * ra.xsr * 4, gxs + (long)(lane - 16) * nbg, (unsigned)nb * 4u,
           act_bar, pol_a);
    __syncwarp();
  }
  bool ok = true;
  if (!A16) {
    ok = __all_sync(FULL, mbar_wait(act_bar, 0, ra.wait_ns, abort_flag));
    if (!ok && lane == 0) raise_error(ra.err, ERR_WAIT_ACT, abort_flag);
  }

  return ok;
}

// A16: the activation rows are held in shared memory already converted to
// f16 (row stride 2K + 64 bytes: a quarter-warp's 16-byte reads of rows g,
// g+1 then cover 128 distinct bytes), so the B fragment is one 16-byte read
// per 32-block instead of a read and 10 conversion instructions per warp.
// Else the int8 words are held (stride K + 32) and converted per use.
// I8: the dots on the int8 tensor path (mma m16n8k32 s8, no level
// conversions; activation rows held as int8), else on the f16 path.
template <int Q, bool A16, bool I8 = false>
__global__ void __launch_bounds__(MW * 32, 1) gemv_mma_kernel(const MmaArgs ra) {
  extern __shared__ __align__(128) unsigned char smem[];
  const lkh::GemvProblem& a = ra.p;
  const int nw = ra.nw, D = ra.depth, NS = nw * D;
  const int row0 = TN * (int)blockIdx.y;                  // this block's group of activation rows
  const int M = a.M - row0 < TN ? a.M - row0 : TN;
  const Chunk ch = chunk_of(ra);
  const int K = ch.kc;                                    // the chunk's bytes of K
  const long ystep = ra.S > 1 ? (long)blockIdx.z * ra.part_stride : 0;  // this chunk's partials
  unsigned char* act = smem;
  unsigned char* ring = smem + ra.ring_off;
  unsigned long long* bars = (unsigned long long*)(ring + (size_t)NS * ra.stage_bytes);
  volatile int* abort_flag = (volatile int*)(bars + MST + 1);
  unsigned long long* keys = (unsigned long long*)(bars + MST + 3);  // [TN][MW]
  const unsigned full0 = smem_u32(bars);
  const unsigned act_bar = smem_u32(bars + MST);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;

  Tiles tl;
  tl.base = blockIdx.x + (long)ra.gx * warp;
  tl.stride = (long)ra.gx * nw;
  tl.ntiles = ra.ntiles;
  tl.nsl = (K + (int)ra.tk - 1) / (int)ra.tk;
  const long my_tiles = tl.base < tl.ntiles ? (tl.ntiles - 1 - tl.base) / tl.stride + 1 : 0;
  const long T = my_tiles * tl.nsl;
  const unsigned long long pol_w = ra.pol_w ? evict_first_policy() : 0ull;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(full0 + 8 * s, 1);
    mbar_init(act_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (ra.pdl && threadIdx.x == 0) griddep_launch();
  tstamp(ra.trace, ra.tslot, TR_START);

  // weights do not depend on the previous kernel: start streaming at once
  long issued = 0;
  Cursor ic{tl.base, 0};
  // (warps >= prefill fill their stages once the activation is loaded)
  const bool early = warp < ra.prefill;
  for (; early && issued < T && issued < D; ++issued, ic.next(tl))
    issue(ra, ch, ic.tile, ic.c, ring + (size_t)(warp * D + issued) * ra.stage_bytes,
          full0 + 8 * (warp * D + (int)issued), pol_w, lane);

  if (ra.pdl) griddep_wait();
  tstamp(ra.trace, ra.tslot, TR_WAITED);
  bool ok = load_rows<Q, A16>(ra, ch, M, row0, act, act_bar, abort_flag);
  tstamp(ra.trace, ra.tslot, TR_ACT);
  for (; !early && issued < T && issued < D; ++issued, ic.next(tl))
    issue(ra, ch, ic.tile, ic.c, ring + (size_t)(warp * D + issued) * ra.stage_bytes,
          full0 + 8 * (warp * D + (int)issued), pol_w, lane);
  // activation row g's words and the scales of activation rows 2t, 2t+1
  const bool gx_ok = g < M;
  const unsigned char* XH = act + (size_t)g * ra.ar + (A16 ? 16 : 8) * t;
  const unsigned char* XL = act + ra.a_lo + (size_t)g * ra.ar + (A16 ? 16 : 8) * t;
  const float* XS0 = (const float*)(act + ra.a_xs) + (size_t)(2 * t) * ra.xsr;
  const float* XS1 = XS0 + ra.xsr;
  const bool s0_ok = 2 * t < M, s1_ok = 2 * t + 1 < M;

  float p[4][4];  // [partial q][element: (g,2t) (g,2t+1) (g+8,2t) (g+8,2t+1)]
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int e = 0; e < 4; ++e) p[q][e] = 0.f;
  unsigned long long best0 = 0, best1 = 0;

  long n = 0;
  Cursor cc{tl.base, 0};
  int cs = 0;          // slot of stage n within the warp's D
  unsigned cph = 0;    // its phase parity
  for (; ok && n < T; ++n) {
    const int slot = warp * D + cs;
    if (!__all_sync(FULL, mbar_wait(full0 + 8 * slot, cph, ra.wait_ns, abort_flag))) {
      if (lane == 0) raise_error(ra.err, ERR_WAIT_FULL, abort_flag);
      ok = false;
      break;
    }
    unsigned char* st = ring + (size_t)slot * ra.stage_bytes;
    const int c = cc.c;
    const int k0 = c * (int)ra.tk;
    const int len = K - k0 < (int)ra.tk ? K - k0 : (int)ra.tk;
    const unsigned char* W0 = st + g * ra.rs + 8 * t;
    const unsigned char* W8 = W0 + 8 * ra.rs;
    const unsigned char* S0 = st + ra.s_off + g * ra.srs + scale_shift(ch.k_lo + k0);
    const unsigned char* S8 = S0 + 8 * ra.srs;
    const int b0 = k0 >> 5;
    const int ngrp = len >> 7;  // groups of 4 blocks (partials 0..3)
#pragma unroll 2
    for (int gi = 0; gi < ngrp; ++gi) {
      // scales of the group's 4 blocks: weight rows g, g+8; activation rows 2t, 2t+1
      const uint2 sw0 = *(const uint2*)(S0 + 8 * gi);
      const uint2 sw8 = *(const uint2*)(S8 + 8 * gi);
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 sx0 = s0_ok ? *(const float4*)(XS0 + b0 + 4 * gi) : z4;
      const float4 sx1 = s1_ok ? *(const float4*)(XS1 + b0 + 4 * gi) : z4;
      const float wa[4] = {__half2float(__ushort_as_half((unsigned short)(sw0.x & 0xffff))),
                           __half2float(__ushort_as_half((unsigned short)(sw0.x >> 16))),
                           __half2float(__ushort_as_half((unsigned short)(sw0.y & 0xffff))),
                           __half2float(__ushort_as_half((unsigned short)(sw0.y >> 16)))};
      const float wb[4] = {__half2float(__ushort_as_half((unsigned short)(sw8.x & 0xffff))),
                           __half2float(__ushort_as_half((unsigned short)(sw8.x >> 16))),
                           __half2float(__ushort_as_half((unsigned short)(sw8.y & 0xffff))),
                           __half2float(__ushort_as_half((unsigned short)(sw8.y >> 16)))};
      const float xa[4] = {sx0.x, sx0.y, sx0.z, sx0.w};
      const float xb[4] = {sx1.x, sx1.y, sx1.z, sx1.w};
      // int8 path: the group's four blocks' MMAs first, back to back, so
      // their latencies overlap; the combines below then read them in order
      int di[4][4], fi[4][4];
      if constexpr (I8) {
        const uint2 z = make_uint2(0u, 0u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int bb = 4 * gi + q;
          const uint2 rw0 = *(const uint2*)(W0 + 32 * bb), rw8 = *(const uint2*)(W8 + 32 * bb);
          const uint2 xh = gx_ok ? *(const uint2*)(XH + k0 + 32 * bb) : z;
#pragma unroll
          for (int e = 0; e < 4; ++e) di[q][e] = fi[q][e] = 0;
          imma16832(di[q], rw0.x, rw8.x, rw0.y, rw8.y, xh.x, xh.y);
          if (Q == 2) {
            const uint2 xl = gx_ok ? *(const uint2*)(XL + k0 + 32 * bb) : z;
            imma16832(fi[q], rw0.x, rw8.x, rw0.y, rw8.y, xl.x, xl.y);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int bb = 4 * gi + q;  // block within the slice; b0 % 4 == 0, so partial q
        float d[4], f[4];
        if constexpr (I8) {
          // exact int32 (|d| < 2^20) -> f32 by the magic-number add, as block_dot_i8
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            d[e] = __fadd_rn(__int_as_float(di[q][e] + 0x4B400000), -12582912.0f);
            f[e] = __fadd_rn(__int_as_float(fi[q][e] + 0x4B400000), -12582912.0f);
          }
        } else {
          const uint2 rw0 = *(const uint2*)(W0 + 32 * bb), rw8 = *(const uint2*)(W8 + 32 * bb);
          const Frag8 fw0 = frag8(rw0), fw8 = frag8(rw8);
          block_dot(d, fw0, fw8, act_frag<A16>(XH, k0 + 32 * bb, gx_ok));
          if (Q == 2) block_dot(f, fw0, fw8, act_frag<A16>(XL, k0 + 32 * bb, gx_ok));
        }
        const float ws_[4] = {wa[q], wa[q], wb[q], wb[q]};
        const float xs_[4] = {xa[q], xb[q], xa[q], xb[q]};
        if constexpr (Q == 1) {
#pragma unroll
          for (int e = 0; e < 4; ++e) p[q][e] = __fmaf_rn(__fmul_rn(ws_[e], xs_[e]), d[e], p[q][e]);
        } else {
          // q8_step<2> with the dots already in f32 (exact integers)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float u = __fmaf_rn(xs_[e], d[e], __fmul_rn(__fmul_rn(xs_[e], 0.0078125f), f[e]));
            p[q][e] = __fmaf_rn(ws_[e], u, p[q][e]);
          }
        }
      }
    }
    // the slot is free: refill it with this warp's stage n + D (generic-proxy
    // reads ordered before the bulk copy's async-proxy writes)
    __syncwarp();
    if (issued < T) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(ra, ch, ic.tile, ic.c, st, full0 + 8 * slot, pol_w, lane);
      ic.next(tl);
      ++issued;
    }
    if (c == tl.nsl - 1) {
      // the tile is done: (p0 + p2) + (p1 + p3) per element ("kernels.rs" lk_q8_sum4)
      const Mat mt = mat_of(ra, cc.tile);
      const long r0 = mt.row0 + g, r8 = r0 + 8;
      const int t0 = 2 * t, t1 = 2 * t + 1;
      float yv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        yv[e] = __fadd_rn(__fadd_rn(p[0][e], p[2][e]), __fadd_rn(p[1][e], p[3][e]));
#pragma unroll
        for (int q = 0; q < 4; ++q) p[q][e] = 0.f;
      }
      if (r0 < mt.N) {
        if (t0 < M) {
          mt.y[ystep + (long)(row0 + t0) * mt.N + r0] = yv[0];
          const unsigned long long k = amax_key(yv[0], (unsigned)r0);
          best0 = k > best0 ? k : best0;
        }
        if (t1 < M) {
          mt.y[ystep + (long)(row0 + t1) * mt.N + r0] = yv[1];
          const unsigned long long k = amax_key(yv[1], (unsigned)r0);
          best1 = k > best1 ? k : best1;
        }
      }
      if (r8 < mt.N) {
        if (t0 < M) {
          mt.y[ystep + (long)(row0 + t0) * mt.N + r8] = yv[2];
          const unsigned long long k = amax_key(yv[2], (unsigned)r8);
          best0 = k > best0 ? k : best0;
        }
        if (t1 < M) {
          mt.y[ystep + (long)(row0 + t1) * mt.N + r8] = yv[3];
          const unsigned long long k = amax_key(yv[3], (unsigned)r8);
          best1 = k > best1 ? k : best1;
        }
      }
    }
    cc.next(tl);
    if (++cs == D) {
      cs = 0;
      cph ^= 1u;
    }
  }
  // drain: stages issued but not consumed (only after an abort) must land
  // before the block may end; they occupy the slots from cs on, in order
  if (lane == 0) {
    for (long m = n; m < issued; ++m) {
      drain_wait(full0 + 8 * (unsigned)(warp * D + cs), cph, ra.wait_ns, ra.err);
      if (++cs == D) {
        cs = 0;
        cph ^= 1u;
      }
    }
    if (!A16 && warp == 0) drain_wait(act_bar, 0, ra.wait_ns, ra.err);
  }
  __syncwarp();
  if (a.amax) {
    // per activation row: max over the lanes holding it (same t), then the block
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      const unsigned long long v0 = __shfl_xor_sync(FULL, best0, o);
      const unsigned long long v1 = __shfl_xor_sync(FULL, best1, o);
      best0 = v0 > best0 ? v0 : best0;
      best1 = v1 > best1 ? v1 : best1;
    }
    if (g == 0) {
      keys[(2 * t) * MW + warp] = best0;
      keys[(2 * t + 1) * MW + warp] = best1;
    }
    __syncthreads();
    if (threadIdx.x < M) {
      unsigned long long m = 0;
      for (int w = 0; w < nw; ++w) m = keys[threadIdx.x * MW + w] > m ? keys[threadIdx.x * MW + w] : m;
      a.amax[(long)(row0 + threadIdx.x) * gridDim.x + blockIdx.x] = m;
    }
  }
  tend(ra.trace, ra.tslot, ra.ntiles * TR, 3);
}

// ---- four warps per tile --------------------------------------------------------------
//
// Where a launch has few tiles per SM (down 4096 x 12288 at 8 rows: 1.7), one
// warp per tile leaves most warps idle and serializes a tile's 32-blocks on
// one warp.  Here a group of four warps shares each 16-row tile: warp q of
// the group computes the blocks b = q mod 4 of every stage, i.e. exactly
// partial q of the combine ("kernels.rs" lk_q8_rows_dot), and at the end of
// the tile the group's leader (q = 0) adds (p0 + p2) + (p1 + p3) from the
// other three warps' partials in shared memory: the same operations in the
// same order, so the same bits.  A group's stages are filled by its leader
// and released by all four warps (an "empty" mbarrier of 4 arrivals); the
// partials go through a per-group buffer guarded by two mbarriers (written,
// read).  Every wait is bounded.
constexpr int G4 = 4;                          // warps per group
constexpr int MGRP = MW / G4;                  // groups per block at most
constexpr unsigned G4_CBUF = MGRP * 3 * 4 * 32 * 4;  // partials of warps 1..3, [grp][q-1][elem][lane]
constexpr unsigned MTAIL4 = MTAIL + 8 * MST + 8 * 2 * MGRP + G4_CBUF;

template <int Q, bool A16>
__global__ void __launch_bounds__(MW * 32, 1) gemv_mma_g4_kernel(const MmaArgs ra) {
  extern __shared__ __align__(128) unsigned char smem[];
  const lkh::GemvProblem& a = ra.p;
  const int nw = ra.nw, NG = nw / G4, D = ra.depth, NS = NG * D;
  const int row0 = TN * (int)blockIdx.y;                  // this block's group of activation rows
  const int M = a.M - row0 < TN ? a.M - row0 : TN;
  const Chunk ch = chunk_of(ra);
  const int K = ch.kc;                                    // the chunk's bytes of K
  const long ystep = ra.S > 1 ? (long)blockIdx.z * ra.part_stride : 0;  // this chunk's partials
  unsigned char* act = smem;
  unsigned char* ring = smem + ra.ring_off;
  unsigned long long* bars = (unsigned long long*)(ring + (size_t)NS * ra.stage_bytes);
  volatile int* abort_flag = (volatile int*)(bars + MST + 1);
  unsigned long long* keys = (unsigned long long*)(bars + MST + 3);  // [TN][MW]
  unsigned long long* ebars = keys + TN * MW;                          // empty, [MST]
  unsigned long long* cbars = ebars + MST;                             // written [MGRP], read [MGRP]
  float* cbuf = (float*)(cbars + 2 * MGRP);
  const unsigned full0 = smem_u32(bars), empty0 = smem_u32(ebars), act_bar = smem_u32(bars + MST);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = warp / G4, q = warp % G4;
  const bool leader = q == 0;
  const int g = lane >> 2, t = lane & 3;
  const unsigned cw_bar = smem_u32(cbars + grp), cr_bar = smem_u32(cbars + MGRP + grp);

  Tiles tl;
  tl.base = blockIdx.x + (long)ra.gx * grp;
  tl.stride = (long)ra.gx * NG;
  tl.ntiles = ra.ntiles;
  tl.nsl = (K + (int)ra.tk - 1) / (int)ra.tk;
  const long my_tiles = tl.base < tl.ntiles ? (tl.ntiles - 1 - tl.base) / tl.stride + 1 : 0;
  const long T = my_tiles * tl.nsl;
  const unsigned long long pol_w = ra.pol_w ? evict_first_policy() : 0ull;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, G4);
    }
    mbar_init(act_bar, 1);
    for (int gi = 0; gi < NG; ++gi) {
      mbar_init(smem_u32(cbars + gi), 32 * (G4 - 1));  // every lane of warps 1..3 has written
      mbar_init(smem_u32(cbars + MGRP + gi), 32);       // every lane of the leader has read
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (ra.pdl && threadIdx.x == 0) griddep_launch();
  tstamp(ra.trace, ra.tslot, TR_START);

  long issued = 0;
  Cursor ic{tl.base, 0};
  const bool early = grp < ra.prefill;  // groups that fill before the dependency wait
  if (leader)
    for (; early && issued < T && issued < D; ++issued, ic.next(tl))
      issue(ra, ch, ic.tile, ic.c, ring + (size_t)(grp * D + issued) * ra.stage_bytes,
            full0 + 8 * (grp * D + (int)issued), pol_w, lane);
  if (ra.pdl) griddep_wait();
  tstamp(ra.trace, ra.tslot, TR_WAITED);
  bool ok = load_rows<Q, A16>(ra, ch, M, row0, act, act_bar, abort_flag);
  tstamp(ra.trace, ra.tslot, TR_ACT);
  if (leader)
    for (; !early && issued < T && issued < D; ++issued, ic.next(tl))
      issue(ra, ch, ic.tile, ic.c, ring + (size_t)(grp * D + issued) * ra.stage_bytes,
            full0 + 8 * (grp * D + (int)issued), pol_w, lane);

  const bool gx_ok = g < M;
  const unsigned char* XH = act + (size_t)g * ra.ar + (A16 ? 16 : 8) * t;
  const unsigned char* XL = act + ra.a_lo + (size_t)g * ra.ar + (A16 ? 16 : 8) * t;
  const float* XS0 = (const float*)(act + ra.a_xs) + (size_t)(2 * t) * ra.xsr;
  const float* XS1 = XS0 + ra.xsr;
  const bool s0_ok = 2 * t < M, s1_ok = 2 * t + 1 < M;

  float p[4] = {0.f, 0.f, 0.f, 0.f};  // this warp's partial q: (g,2t) (g,2t+1) (g+8,2t) (g+8,2t+1)
  unsigned long long best0 = 0, best1 = 0;
  long n = 0;
  Cursor cc{tl.base, 0};
  int cs = 0;
  unsigned cph = 0, jt = 0;  // phase parity of the current slot round; tiles finished
  for (; ok && n < T; ++n) {
    const int slot = grp * D + cs;
    if (!__all_sync(FULL, mbar_wait(full0 + 8 * slot, cph, ra.wait_ns, abort_flag))) {
      if (lane == 0) raise_error(ra.err, ERR_WAIT_FULL, abort_flag);
      ok = false;
      break;
    }
    unsigned char* st = ring + (size_t)slot * ra.stage_bytes;
    const int c = cc.c;
    const int k0 = c * (int)ra.tk;
    const int len = K - k0 < (int)ra.tk ? K - k0 : (int)ra.tk;
    const unsigned char* W0 = st + g * ra.rs + 8 * t;
    const unsigned char* W8 = W0 + 8 * ra.rs;
    const unsigned char* S0 = st + ra.s_off + g * ra.srs + scale_shift(ch.k_lo + k0);
    const unsigned char* S8 = S0 + 8 * ra.srs;
    const int b0 = k0 >> 5, nblk = len >> 5;
#pragma unroll 4
    for (int bb = q; bb < nblk; bb += G4) {  // b0 % 4 == 0: block b0 + bb is in partial q
      const float wa = __half2float(*(const __half*)(S0 + 2 * bb));
      const float wb = __half2float(*(const __half*)(S8 + 2 * bb));
      const float xa = s0_ok ? XS0[b0 + bb] : 0.f;
      const float xb = s1_ok ? XS1[b0 + bb] : 0.f;
      const Frag8 fw0 = frag8(*(const uint2*)(W0 + 32 * bb));
      const Frag8 fw8 = frag8(*(const uint2*)(W8 + 32 * bb));
      float d[4];
      block_dot(d, fw0, fw8, act_frag<A16>(XH, k0 + 32 * bb, gx_ok));
      const float ws_[4] = {wa, wa, wb, wb};
      const float xs_[4] = {xa, xb, xa, xb};
      if constexpr (Q == 1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) p[e] = __fmaf_rn(__fmul_rn(ws_[e], xs_[e]), d[e], p[e]);
      } else {
        float f[4];
        block_dot(f, fw0, fw8, act_frag<A16>(XL, k0 + 32 * bb, gx_ok));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float u = __fmaf_rn(xs_[e], d[e], __fmul_rn(__fmul_rn(xs_[e], 0.0078125f), f[e]));
          p[e] = __fmaf_rn(ws_[e], u, p[e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * slot);  // this warp is done with the stage
    if (c == tl.nsl - 1) {
      // the tile is done: (p0 + p2) + (p1 + p3) across the group ("kernels.rs" lk_q8_sum4)
      float* buf = cbuf + (size_t)grp * 3 * 4 * 32;
      if (!leader) {
        // the leader has read the previous tile's partials before these are written
        if (jt > 0 && !__all_sync(FULL, mbar_wait(cr_bar, (jt - 1) & 1u, ra.wait_ns, abort_flag))) {
          if (lane == 0) raise_error(ra.err, ERR_WAIT_FULL, abort_flag);
          ok = false;
          break;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) buf[((q - 1) * 4 + e) * 32 + lane] = p[e];
        mbar_arrive(cw_bar);
      } else {
        if (!__all_sync(FULL, mbar_wait(cw_bar, jt & 1u, ra.wait_ns, abort_flag))) {
          if (lane == 0) raise_error(ra.err, ERR_WAIT_FULL, abort_flag);
          ok = false;
          break;
        }
        float yv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p1 = buf[(0 * 4 + e) * 32 + lane], p2 = buf[(1 * 4 + e) * 32 + lane],
                      p3 = buf[(2 * 4 + e) * 32 + lane];
          yv[e] = __fadd_rn(__fadd_rn(p[e], p2), __fadd_rn(p1, p3));
        }
        mbar_arrive(cr_bar);
        const Mat mt = mat_of(ra, cc.tile);
        const long r0 = mt.row0 + g, r8 = r0 + 8;
        const int t0 = 2 * t, t1 = 2 * t + 1;
        if (r0 < mt.N) {
          if (t0 < M) {
            mt.y[ystep + (long)(row0 + t0) * mt.N + r0] = yv[0];
            const unsigned long long k = amax_key(yv[0], (unsigned)r0);
            best0 = k > best0 ? k : best0;
          }
          if (t1 < M) {
            mt.y[ystep + (long)(row0 + t1) * mt.N + r0] = yv[1];
            const unsigned long long k = amax_key(yv[1], (unsigned)r0);
            best1 = k > best1 ? k : best1;
          }
        }
        if (r8 < mt.N) {
          if (t0 < M) {
            mt.y[ystep + (long)(row0 + t0) * mt.N + r8] = yv[2];
            const unsigned long long k = amax_key(yv[2], (unsigned)r8);
            best0 = k > best0 ? k : best0;
          }
          if (t1 < M) {
            mt.y[ystep + (long)(row0 + t1) * mt.N + r8] = yv[3];
            const unsigned long long k = amax_key(yv[3], (unsigned)r8);
            best1 = k > best1 ? k : best1;
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) p[e] = 0.f;
      ++jt;
    }
    // the leader refills the slot once all four warps are done with it
    if (leader && issued < T) {
      if (!__all_sync(FULL, mbar_wait(empty0 + 8 * slot, cph, ra.wait_ns, abort_flag))) {
        if (lane == 0) raise_error(ra.err, ERR_WAIT_EMPTY, abort_flag);
        ok = false;
        break;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(ra, ch, ic.tile, ic.c, st, full0 + 8 * slot, pol_w, lane);
      ic.next(tl);
      ++issued;
    }
    cc.next(tl);
    if (++cs == D) {
      cs = 0;
      cph ^= 1u;
    }
  }
  // drain: the leader's stages issued but not consumed (only after an abort)
  // must land before the block may end; they occupy the slots from cs on
  if (leader && lane == 0) {
    for (long m = n; m < issued; ++m) {
      drain_wait(full0 + 8 * (unsigned)(grp * D + cs), cph, ra.wait_ns, ra.err);
      if (++cs == D) {
        cs = 0;
        cph ^= 1u;
      }
    }
  }
  if (!A16 && warp == 0 && lane == 0) drain_wait(act_bar, 0, ra.wait_ns, ra.err);
  __syncwarp();
  if (a.amax) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      const unsigned long long v0 = __shfl_xor_sync(FULL, best0, o);
      const unsigned long long v1 = __shfl_xor_sync(FULL, best1, o);
      best0 = v0 > best0 ? v0 : best0;
      best1 = v1 > best1 ? v1 : best1;
    }
    if (g == 0) {
      keys[(2 * t) * MW + warp] = best0;
      keys[(2 * t + 1) * MW + warp] = best1;
    }
    __syncthreads();
    if (threadIdx.x < M) {
      unsigned long long m = 0;
      for (int w = 0; w < nw; ++w) m = keys[threadIdx.x * MW + w] > m ? keys[threadIdx.x * MW + w] : m;
      a.amax[(long)(row0 + threadIdx.x) * gridDim.x + blockIdx.x] = m;
    }
  }
  tend(ra.trace, ra.tslot, ra.ntiles * TR, 3);
}

struct MmaLayout {
  unsigned tk, rs, srs, s_off, stage_bytes, ar, xsr, a_lo, a_xs, ring_off, total;
  int nw, depth;  // g4: warps (4 per group) and stages per group
  bool a16, g4, i8;
};

unsigned round_up(unsigned v, unsigned a) { return (v + a - 1) / a * a; }

// Bytes of K a block holds: the whole row, or the longest split-K chunk.
unsigned chunk_k(const lkh::GemvProblem& p) {
  if (!p.split || p.S <= 1) return (unsigned)p.K;
  const int nb = p.K / 32;
  int m = 0;
  for (int c = 0; c < p.S; ++c) {
    const int w = splitk_bound(nb, p.S, c + 1) - splitk_bound(nb, p.S, c);
    m = w > m ? w : m;
  }
  return 32u * (unsigned)m;
}

// Stage layout.  A warp computes its tiles alone, one 32-block after the
// other, so two regimes (measured, 8 rows):
//  * many tiles per SM (gate/up 24576 x 4096: 10 per SM): warps beat stages
//    per warp.  512-byte slices, one stage per warp, as many warps as fit
//    (16): 29.5-30.8 us; two stages per warp (fewer warps) 44-48 us;
//    256-byte slices 48 us (too few bytes in flight).
//  * few tiles per SM (down 4096 x 12288: 1.7 per SM, so ~2 warps per SM
//    have work): bytes in flight per working warp decide.  1024-byte slices,
//    two stages per warp: 35.3 us; 512 x 1: 56.4 us; 256 x 1: 94.9 us.
// Below 4 tiles per SM the second regime's layout is tried first.
MmaLayout mma_layout_for(const lkh::GemvProblem& p, long ntiles, int sms, int smem_optin, bool a16) {
  MmaLayout L{};
  const unsigned K = chunk_k(p), nb = K / 32u, M = (unsigned)(p.M < TN ? p.M : TN);  // a block's rows
  L.a16 = a16;
  L.ar = a16 ? 2u * K + 64u : K + 32u;
  L.xsr = nb + 4u;
  L.a_lo = round_up(M * L.ar, 128u);
  L.a_xs = p.mode == LK_TWOPASS ? round_up(L.a_lo + M * L.ar, 128u) : L.a_lo;
  L.ring_off = round_up(L.a_xs + M * L.xsr * 4u, 128u);
  const bool few = ntiles < 4L * sms;
  // split-K launches (many work units of a short chunk each) take 1 KB
  // slices, one stage per warp first: measured at 8 rows, S = 4 (q|k|v
  // 6144 x 4096 11.4 -> 9.4 us, gate/up 26.4 -> 25.0, down 4096 x 12288
  // 21.1 -> 16.4 against 512-byte slices)
  const bool split = p.split && p.S > 1;
  const unsigned cand_tk[5] = {1024u, 512u, 512u, 256u, 1024u};
  const int cand_d[5] = {2, 2, 1, 1, 1};
  const int order[2][4] = {{0, 1, 2, 3}, {4, 2, 3, 3}};
  for (int j = split ? 0 : (few ? 0 : 2); j < 4; ++j) {
    const int i = order[split ? 1 : 0][j];
    unsigned tk = p.cfg.mma_tk > 0 ? (unsigned)p.cfg.mma_tk : cand_tk[i];
    if (tk > round_up(K, 256u)) tk = round_up(K, 256u);
    L.tk = tk;
    L.rs = tk + 32u;
    L.srs = tk / 16u + 16u;
    L.s_off = TR * L.rs;
    L.stage_bytes = round_up(L.s_off + TR * L.srs, 128u);
    const long room = (long)smem_optin - (long)L.ring_off - (long)MTAIL;
    int fit = room > 0 ? (int)(room / L.stage_bytes) : 0;
    if (fit > MST) fit = MST;
    int depth = p.cfg.mma_depth > 0 ? (int)p.cfg.mma_depth : cand_d[i];
    int w = p.cfg.mma_warps > 0 ? (int)p.cfg.mma_warps : fit / depth;
    if (w > MW) w = MW;
    if (w * depth > fit) w = fit / depth;
    L.nw = w;
    L.depth = depth;
    L.total = L.ring_off + (unsigned)(w * depth) * L.stage_bytes + MTAIL;
    if (w >= 2 || p.cfg.mma_tk > 0) break;
  }
  return L;
}

// Four warps per tile: 512-byte slices (256 when they do not fit), groups of
// four warps with at least three stages each (the group consumes a stage four
// times faster than one warp), as many groups as fit, up to four.
MmaLayout mma_layout_g4(const lkh::GemvProblem& p, int smem_optin, bool a16, unsigned tk_pref = 0) {
  MmaLayout L{};
  const unsigned K = chunk_k(p), nb = K / 32u, M = (unsigned)(p.M < TN ? p.M : TN);  // a block's rows
  L.a16 = a16;
  L.g4 = true;
  L.ar = a16 ? 2u * K + 64u : K + 32u;
  L.xsr = nb + 4u;
  L.a_lo = round_up(M * L.ar, 128u);
  L.a_xs = p.mode == LK_TWOPASS ? round_up(L.a_lo + M * L.ar, 128u) : L.a_lo;
  L.ring_off = round_up(L.a_xs + M * L.xsr * 4u, 128u);
  const unsigned cand_tk[2] = {tk_pref ? tk_pref : 512u, tk_pref ? tk_pref : 256u};
  for (int i = 0; i < 2; ++i) {
    unsigned tk = p.cfg.mma_tk > 0 ? (unsigned)p.cfg.mma_tk : cand_tk[i];
    if (tk > round_up(K, 256u)) tk = round_up(K, 256u);
    L.tk = tk;
    L.rs = tk + 32u;
    L.srs = tk / 16u + 16u;
    L.s_off = TR * L.rs;
    L.stage_bytes = round_up(L.s_off + TR * L.srs, 128u);
    const long room = (long)smem_optin - (long)L.ring_off - (long)MTAIL4;
    int fit = room > 0 ? (int)(room / L.stage_bytes) : 0;
    if (fit > MST) fit = MST;
    int ng = p.cfg.mma_warps > 0 ? (int)p.cfg.mma_warps / G4 : fit / 3;
    if (ng > MGRP) ng = MGRP;
    int depth = p.cfg.mma_depth > 0 ? (int)p.cfg.mma_depth : (ng > 0 ? fit / ng : 0);
    if (ng * depth > fit) ng = depth > 0 ? fit / depth : 0;
    L.nw = G4 * ng;
    L.depth = depth;
    L.total = L.ring_off + (unsigned)(ng * depth) * L.stage_bytes + MTAIL4;
    if (ng >= 1 || p.cfg.mma_tk > 0) break;
  }
  return L;
}

bool mma_layout_ok(const MmaLayout& L);

// The int8 tensor path (lk_launch_cfg.mma_i8: 0 auto, 1 always, 2 never).  An
// int8 MMA is a single instruction per 32-block with no level conversions,
// but on this GPU a long-latency one: it won where the tiles are many (8
// rows, Int8Act: gate/up 28.9 against 29.7 us, lm-head 127.9 against
// 133.2 us) and lost where a warp's chain of blocks is the critical path
// (4096x4096: 17.0 against 13.5 us; 4096x12288: 46.3 against 35.4 us; and
// TwoPass, two per block, everywhere).
bool use_i8(const lkh::GemvProblem& p, long ntiles, int sms) {
  if (p.cfg.mma_i8 == 2) return false;
  if (p.cfg.mma_i8 == 1) return true;
  return p.mode == LK_INT8ACT && ntiles >= 8L * sms;
}

// f16-held activations where they cost no warps (Int8Act at K = 4096: 16
// warps either way; TwoPass would drop from 16 to 10: measured 54.9 us
// against 36.9 us held as int8); lk_launch_cfg.mma_act16 1 forces them (if
// they fit at all), 2 forbids them.
MmaLayout mma_layout(const lkh::GemvProblem& p, long ntiles, int sms, int smem_optin) {
  if (use_i8(p, ntiles, sms)) {
    MmaLayout L = mma_layout_for(p, ntiles, sms, smem_optin, false);
    L.i8 = true;
    return L;
  }
  // Int8Act launches with few tiles per SM (the narrow projections at 8
  // rows: q, k, v, o, down): four warps per tile with 1 KB slices (2 KB for
  // rows longer than 8192), where such a layout fits.  Measured at 8 rows
  // against one warp per tile: down 4096x12288 35.4 -> 27.5 us, 4096x4096
  // 13.4 -> 10.7 us, 1024x4096 10.6 -> 5.9 us.  (TwoPass keeps one warp per
  // tile: its doubled activation area leaves four-warp groups too few
  // stages, down 64.2 -> 130.1 us.)
  if (p.cfg.mma_group == 0 && p.mode == LK_INT8ACT && ntiles < 4L * sms) {
    const MmaLayout G = mma_layout_g4(p, smem_optin, false, chunk_k(p) > 8192 ? 2048u : 1024u);
    if (mma_layout_ok(G)) return G;
  }
  if (p.cfg.mma_group == 4) {
    const MmaLayout G8 = mma_layout_g4(p, smem_optin, false);
    if (p.cfg.mma_act16 == 2) return G8;
    const MmaLayout G16 = mma_layout_g4(p, smem_optin, true);
    if (!mma_layout_ok(G16)) return G8;
    if (p.cfg.mma_act16 == 1) return G16;
    return G16.nw >= G8.nw ? G16 : G8;
  }
  const MmaLayout L8 = mma_layout_for(p, ntiles, sms, smem_optin, false);
  if (p.cfg.mma_act16 == 2) return L8;
  const MmaLayout L16 = mma_layout_for(p, ntiles, sms, smem_optin, true);
  if (!mma_layout_ok(L16)) return L8;
  if (p.cfg.mma_act16 == 1) return L16;
  return L16.nw >= L8.nw ? L16 : L8;
}

bool mma_layout_ok(const MmaLayout& L) {
  return L.g4 ? (L.nw >= G4 && L.depth >= 2) : (L.nw >= 1 && L.depth >= 1 && L.nw * L.depth >= 2);
}
// (a single-stage ring per warp still overlaps: the warps' copies are in
// flight while other warps compute)

typedef void (*mma_fn)(const MmaArgs);

}  // namespace lkmma

namespace lkh {

using namespace lkmma;

// Activation-row groups of a launch of M rows, and the blocks (SMs) each
// group gets: every group runs at once, one block per SM.
int mma_groups(int M) { return (M + TN - 1) / TN; }
int mma_group_blocks(int M, int sms) {
  const int g = sms / mma_groups(M);
  return g > 0 ? g : 1;
}

// Split-K chunks of a launch (1 for the plain GEMV).
int mma_chunks(const GemvProblem& p) { return p.split && p.S > 1 ? p.S : 1; }

bool mma_supports(const GemvProblem& p) {
  if (p.mode != LK_INT8ACT && p.mode != LK_TWOPASS) return false;
  if (p.fuse || p.F > 0) return false;
  // split-K: every chunk holds at least one group of four blocks (an empty
  // chunk would have no tile to write its zero partials)
  if (p.split && (p.S < 1 || p.K / 128 < p.S || p.amax)) return false;
  const int min_m = p.cfg.mma_min_m > 0 ? p.cfg.mma_min_m : 2;
  if (p.M < min_m || p.M > LK_MAX_BATCH) return false;
  if (p.K < 256 || p.K % 256 || p.N < 1) return false;
  if (!aligned(p.ws, 16) || !aligned(p.xq, 16) || !aligned(p.xs, 16) || (p.mode == LK_TWOPASS && !aligned(p.xl, 16)))
    return false;
  // each group's rows start 16-byte aligned (K % 256 == 0) and its scales too
  const DeviceInfo* d = device_info(nullptr);
  if (!d) return false;
  return mma_layout_ok(mma_layout(p, (p.N + TR - 1) / TR * mma_chunks(p), mma_group_blocks(p.M, d->sm_count),
                                  d->smem_optin));
}

// One launch over the matrices (wq[m], ws[m], N[m]) -> y[m], all reading
// the activation of p.  Argmax keys (p.amax) only for a single matrix.
lk_status mma_launch(const GemvProblem& p, int nmat, const int8_t* const* wq, const __half* const* ws,
                     const long* N, float* const* y, cudaStream_t stream, int* n_parts) {
  const DeviceInfo* d = device_info(nullptr);
  if (!d) return LK_ERR_CUDA;
  if (nmat < 1 || nmat > MG || (nmat > 1 && p.amax)) return LK_ERR_ARG;
  long all_tiles = 0;
  for (int m = 0; m < nmat; ++m) all_tiles += (N[m] + TR - 1) / TR;
  const int ngrp = mma_groups(p.M), gsms = mma_group_blocks(p.M, d->sm_count), S = mma_chunks(p);
  if (S > 1 && nmat > 1) return LK_ERR_ARG;
  const MmaLayout L = mma_layout(p, all_tiles * S, gsms, d->smem_optin);
  if (!mma_layout_ok(L)) return LK_ERR_SHAPE;
  mma_fn f = L.i8 ? (p.mode == LK_TWOPASS ? gemv_mma_kernel<2, false, true> : gemv_mma_kernel<1, false, true>)
           : L.g4 ? (p.mode == LK_TWOPASS ? (L.a16 ? gemv_mma_g4_kernel<2, true> : gemv_mma_g4_kernel<2, false>)
                                          : (L.a16 ? gemv_mma_g4_kernel<1, true> : gemv_mma_g4_kernel<1, false>))
                  : (p.mode == LK_TWOPASS ? (L.a16 ? gemv_mma_kernel<2, true> : gemv_mma_kernel<2, false>)
                                          : (L.a16 ? gemv_mma_kernel<1, true> : gemv_mma_kernel<1, false>));
  // (the cap is the device's maximum: see ring_gemv)
  if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, d->smem_optin) != cudaSuccess)
    return LK_ERR_CUDA;
  MmaArgs ra;
  ra.p = p;
  ra.nmat = nmat;
  long tiles = 0;
  for (int m = 0; m < MG; ++m) {
    const bool in = m < nmat;
    ra.wq[m] = in ? wq[m] : wq[0];
    ra.ws[m] = (const unsigned char*)(in ? ws[m] : ws[0]);
    ra.N[m] = in ? N[m] : 0;
    ra.y[m] = in ? y[m] : y[0];
    ra.tile0[m] = tiles;
    if (in) tiles += (N[m] + TR - 1) / TR;
  }
  ra.tile0[MG] = tiles;
  for (int m = nmat; m <= MG; ++m) ra.tile0[m] = tiles;
  ra.ntiles = tiles;
  if (tiles < 1) return LK_ERR_SHAPE;
  ra.nw = L.nw;
  ra.depth = L.depth;
  // a row group's blocks, split evenly over the chunks
  long gx = p.cfg.grid_ctas > 0 ? p.cfg.grid_ctas : (gsms / S > 0 ? gsms / S : 1);
  if (gx > ra.ntiles) gx = ra.ntiles;
  ra.gx = (int)gx;
  ra.S = S;
  ra.part_stride = (long)p.M * N[0];
  ra.tk = L.tk;
  ra.rs = L.rs;
  ra.srs = L.srs;
  ra.s_off = L.s_off;
  ra.stage_bytes = L.stage_bytes;
  ra.ar = L.ar;
  ra.xsr = L.xsr;
  ra.a_lo = L.a_lo;
  ra.a_xs = L.a_xs;
  ra.ring_off = L.ring_off;
  ra.wait_ns = opt_wait_us > 0 ? (unsigned long long)opt_wait_us * 1000ull : 2000000000ull;
  ra.pol_w = 1ull;  // L2 evict-first on the weight copies
  ra.pdl = p.cfg.pdl;
  ra.err = error_word_ptr();
  if (!ra.err) return LK_ERR_CUDA;
  ra.trace = opt_trace == 3 ? trace_ptr() : nullptr;
  ra.tslot = opt_trace == 3 ? trace_next_slot() : -1;
  ra.prefill = L.g4 ? prefill_warps(L.nw / G4, p.cfg.prefill) : prefill_warps(L.nw, p.cfg.prefill);  // groups, or warps
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)gx, (unsigned)ngrp, (unsigned)S);
  cfg.blockDim = dim3(L.nw * 32);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ra.pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, f, ra) != cudaSuccess) return LK_ERR_CUDA;
  if (n_parts) *n_parts = (int)gx;
  return launch_status();
}

lk_status mma_gemv(const GemvProblem& p, cudaStream_t stream, int* n_parts) {
  const int8_t* wq[1] = {p.wq};
  const __half* ws[1] = {p.ws};
  const long N[1] = {p.N};
  float* y[1] = {p.y};
  return mma_launch(p, 1, wq, ws, N, y, stream, n_parts);
}

}  // namespace lkh
