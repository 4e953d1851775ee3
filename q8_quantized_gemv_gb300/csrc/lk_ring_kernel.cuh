// Device side of the bulk-copy ring GEMV: layout constants, the launch
// arguments, PTX wrappers, the fused activation prologue and the kernel
// template.  Included by the per-mode translation units lk_ring_q*.cu, which
// instantiate the kernels, and by lk_ring.cu (host side).
#pragma once
#include "lk_device.cuh"
#include "lk_host.h"

namespace lkring {


using namespace lk;

constexpr int MAXW = 12;               // warps per block at most (168 registers a thread)
constexpr int THREADS_MAX = MAXW * 32;
constexpr int QR = 4;                  // rows per stage (one warp's quad)
constexpr int TKMAX = 8192;            // bytes of K per stage
constexpr int MAX_STAGES = 32;
// barriers (one per stage + the activation's), abort flag, argmax keys
// [M][MAXW], norm partial sums [M][32] and norm denominators [M] (8 B each)
constexpr unsigned TAIL =
    8 * (MAX_STAGES + 1) + 16 + 8 * LK_MAX_M * MAXW + 8 * LK_MAX_M * 32 + 8 * LK_MAX_M;

constexpr int LK_TRACE_MAX = 4096;  // timestamps kept by the "trace" option

enum : int { ERR_WAIT_FULL = 1, ERR_WAIT_EMPTY = 2, ERR_DRAIN = 4, ERR_SELFTEST = 8, ERR_WAIT_ACT = 16 };

struct RingArgs {
  lkh::GemvProblem p;
  int nwc;                 // warps of the block; each streams and computes its own quads
  int depth;               // ring stages owned by each warp
  int gx;                  // blocks along the rows
  unsigned tk;             // bytes of K per stage (<= TKMAX)
  unsigned srow;           // bytes per row of a stage's scale area
  unsigned stage_bytes;
  unsigned s_off;          // scale area inside a stage
  unsigned act_len;        // bytes of K in the activation area (the widest chunk)
  unsigned ring_off;       // ring start (after the activation area)
  unsigned long long wait_ns;
  unsigned long long pol_w;  // nonzero: L2 evict-first hint on the weight copies
  int pdl;                 // launched as a programmatic dependent of the previous kernel
  int* err;                // the device error word
  unsigned long long* trace;  // block 0's timestamps (option "trace"), or NULL
  int tslot;               // trace 3: this launch's record in the timeline, else -1
  int prefill;             // warps that fill their stages before the dependency wait
};

typedef void (*ring_fn)(const RingArgs);
template <int Q>
ring_fn ring_pick(int M, bool split, bool fuse, bool glu);

// ---- PTX wrappers -------------------------------------------------------------------------
__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return (unsigned)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned bar, unsigned bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(unsigned bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned long long gtimer_() { return gtimer(); }
// Bounded wait for the phase of parity `parity` to complete.  Returns false if
// the limit ran out or another thread raised the abort flag.
__device__ __forceinline__ bool mbar_wait(unsigned bar, unsigned parity, unsigned long long limit_ns,
                                          volatile int* abort_flag) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  for (unsigned n = 1;; ++n) {
    if (mbar_try(bar, parity)) return true;
    if ((n & 63u) == 0) {
      if (*abort_flag) return false;
      if (gtimer() - t0 > limit_ns) return false;
    }
  }
}
__device__ __forceinline__ unsigned long long evict_first_policy() {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ unsigned long long evict_last_policy() {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// 1-D bulk copy global -> this block's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, unsigned bar,
                                         unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_g2s_nohint(void* dst, const void* src, unsigned bytes, unsigned bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void raise_error(int* err, int code, volatile int* abort_flag) {
  atomicOr(err, code);
  *abort_flag = 1;
}

template <int Q>
struct part_t { typedef float t; };
template <>
struct part_t<0> { typedef double t; };

// Bytes of the activation area for `len` bytes of K (M rows).
template <int Q, int M>
__host__ __device__ constexpr unsigned act_area(unsigned len) {
  return Q == 0 ? M * len * 4u : M * len * (Q == 2 ? 2u : 1u) + M * len / 8u;
}

__device__ __forceinline__ void bulk(void* dst, const void* src, unsigned bytes, unsigned bar,
                                     unsigned long long policy) {
  if (policy) bulk_g2s(dst, src, bytes, bar, policy);
  else bulk_g2s_nohint(dst, src, bytes, bar);
}

// Trace records.  Options "trace" 1/2: block 0's stamps of the last launch
// from index 0.  Option 3 (launch timeline): each launch owns record `slot`
// of TREC entries: [0] block 0 start, [1] block 0 past the dependency wait,
// [2] block 0's activation ready, [3] the last block's end (max over blocks),
// [4] block 0's end, [5] kernel kind, [6] rows.
__device__ __forceinline__ void tstamp(unsigned long long* tr, int slot, int i) {
  if (tr && blockIdx.x == 0 && threadIdx.x == 0) tr[(slot < 0 ? 0 : slot * TREC) + i] = gtimer_();
}
// every block: the latest end (call after the block's last work, all threads)
__device__ __forceinline__ void tend(unsigned long long* tr, int slot, long rows, int kind) {
  if (!tr || slot < 0) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long now = gtimer_();
    atomicMax(tr + slot * TREC + TR_END_MAX, now);
    if (blockIdx.x == 0) {
      tr[slot * TREC + TR_END0] = now;
      tr[slot * TREC + TR_KIND] = (unsigned long long)kind;
      tr[slot * TREC + TR_ROWS] = (unsigned long long)rows;
    }
  }
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// The activation area computed in the block from the raw f32 rows: RMSNorm
// (when a gain is given) and the quantizer of mode Q, bit for bit what
// lk_rmsnorm_quant / lk_quantize_act compute.  The norm's sum of squares
// follows the block of vt = min(K, 1024) threads of "kernels.rs"
// lk_rmsnorm_row: its vt/32 warps are played by the block's nwc warps in turn
// (warp w plays w, w + nwc, ...), virtual warp v's lane l adding the squares
// of values 32v + l + vt*u in ascending u.  The same warp then normalizes and
// quantizes exactly the 32-groups v + (vt/32)*u it loaded, so each row is
// read from global memory once, all of a warp's loads in flight together.
constexpr int PRO_SLOTS = 32;  // groups per warp per batch held in registers by the prologue

// f32 loads that the compiler keeps where they are written: the prologue
// issues all of a lane's loads before using any, so a row costs one round
// trip to L2 instead of one per 32-group.  ld_keep (read-only path) is for
// data no kernel writes (the norm gains); ld_keep_cg (L2 only) for the raw
// activation, which the previous kernel writes: under a programmatic
// dependent launch this kernel starts while that kernel still runs, and the
// read-only path is only valid for data that stays unchanged over the
// reading kernel's whole lifetime (measured: ld.global.nc here gave stale
// values in a few replays in a hundred of a captured token).
__device__ __forceinline__ float ld_keep(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_keep_cg(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void compiler_fence() { asm volatile("" ::: "memory"); }

// The activation of four groups g, g + step, g + 2 step, g + 3 step of row t
// (those with ok set) into the area: f32 values under Dequant, else their
// quantized words and scales.
template <int Q, int M>
__device__ __forceinline__ void store_act4(unsigned char* act, unsigned L, int t, int g, int step, int lane,
                                           const float (&v)[4], const bool (&ok)[4]) {
  if constexpr (Q == 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (ok[k]) ((float*)act)[(size_t)t * L + 32 * (g + k * step) + lane] = v[k];
  } else {
    int8_t* XQ = (int8_t*)act + (size_t)t * L;
    int8_t* XL = (int8_t*)act + (size_t)M * L + (size_t)t * L;
    float* XS = (float*)(act + (size_t)M * L * (Q == 2 ? 2 : 1)) + (size_t)t * (L >> 5);
    quant_groups<Q, 4>(v, ok, XQ, XL, XS, g, step, lane);
  }
}

// dbg (option "trace" 1, block 0): [0] entry, [1] warp 0's squares summed,
// [2] denominators ready, [3] warp 0's groups stored, [4] exit.
__device__ __forceinline__ void pstamp(unsigned long long* dbg, int i) {
  if (dbg && blockIdx.x == 0 && threadIdx.x == 0) dbg[i] = gtimer();
}

// wait_first: the caller has not yet waited for the previous kernel
// (programmatic dependent launch); the first batch's gains, which do not
// depend on it, are requested before the wait, the values after it.
template <int Q, int M>
__device__ void fused_prologue(const lkh::GemvProblem& a, int nwc, int k_lo, unsigned L, unsigned char* act,
                               void* red_raw, void* den_raw, unsigned long long* dbg = nullptr,
                               bool wait_first = false) {
  typedef typename acc_of<Q>::t A;
  constexpr int QB = PRO_SLOTS;  // groups a warp quantizes per batch
  constexpr int KU_MAX = 8;      // values per virtual thread kept in registers (K <= 8192)
  A* red = (A*)red_raw;
  A* den = (A*)den_raw;
  const int lane = threadIdx.x & 31, cw = threadIdx.x >> 5;
  const int K = a.K;
  const bool norm = a.gain != nullptr;
  const int vt = K < 1024 ? K : 1024, nvw_all = vt >> 5;
  const int KU = (K + vt - 1) / vt;
  const int ng = (int)(L >> 5);
  pstamp(dbg, 0);
  // One round trip per row where the layouts agree (K = 1024 u, u <= 4, the
  // whole row, at least 11 warps): virtual warp w's values 32w + l + 1024u
  // are element l of the 32-groups w + 32u, so the values a warp loads for
  // the sum of squares are whole groups of the quantizer too -- loaded once,
  // kept in registers through the sum, the norm and the quantizer.
  if (norm && K % 1024 == 0 && KU <= 4 && k_lo == 0 && (int)L == K && nwc >= 11) {
    for (int t = 0; t < M; ++t) {
      const float* xr = a.xraw + (long)t * K;
      float xv[3][4], gv[3][4];
#pragma unroll
      for (int j = 0; j < 3; ++j)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int w = cw + j * nwc;
          gv[j][u] = (w < 32 && u < KU) ? ld_keep(a.gain + 32 * w + lane + 1024 * u) : 1.f;
        }
      if (t == 0 && wait_first) griddep_wait();
#pragma unroll
      for (int j = 0; j < 3; ++j)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int w = cw + j * nwc;
          xv[j][u] = (w < 32 && u < KU) ? ld_keep_cg(xr + 32 * w + lane + 1024 * u) : 0.f;
        }
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int w = cw + j * nwc;
        if (w >= 32) break;  // warp-uniform
        A acc = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (u < KU) acc = fma_acc((A)xv[j][u], acc);
        acc = warp_tree_sum(acc);
        if (lane == 0) red[t * 32 + w] = acc;
      }
      pstamp(dbg, 1);
      __syncthreads();
      if (cw == 0) {
        A v = red[t * 32 + lane];
        v = warp_tree_sum(v);
        if (lane == 0) den[t] = norm_div_add(v, K, a.eps);
      }
      __syncthreads();
      pstamp(dbg, 2);
      const A dn = den[t];
      const float rdn = sizeof(A) == 4 ? __frcp_rn((float)dn) : 0.f;  // for div_row (f32 norms)
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int w = cw + j * nwc;
        if (w >= 32) break;
        float v[4];
        bool ok[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          ok[u] = u < KU;
          if constexpr (sizeof(A) == 4) v[u] = norm_scale_r(xv[j][u], (float)dn, rdn, gv[j][u]);
          else v[u] = norm_scale(xv[j][u], dn, gv[j][u]);
        }
        store_act4<Q, M>(act, L, t, w, 32, lane, v, ok);  // groups w + 32 u
      }
      pstamp(dbg, 3);
    }
    __syncthreads();
    pstamp(dbg, 4);
    return;
  }
  for (int t = 0; t < M; ++t) {
    const float* xr = a.xraw + (long)t * K;
    // (1) the first batch of this warp's groups g = cw + nwc*b: its values and
    // gains are requested before anything else, so their round trip overlaps
    // the sum of squares below
    float qx[QB], qg[QB];
    auto load_gains = [&](int g0) {
#pragma unroll
      for (int b = 0; b < QB; ++b) {
        const int g = g0 + b * nwc, i = 32 * g + lane;
        const bool in = g < ng && k_lo + i < K;
        qg[b] = (norm && in) ? ld_keep(a.gain + k_lo + i) : 1.f;
      }
    };
    auto load_values = [&](int g0) {
#pragma unroll
      for (int b = 0; b < QB; ++b) {
        const int g = g0 + b * nwc, i = 32 * g + lane;
        const bool in = g < ng && k_lo + i < K;
        qx[b] = in ? ld_keep_cg(xr + k_lo + i) : 0.f;
      }
    };
    auto load_batch = [&](int g0) {
      load_gains(g0);
      load_values(g0);
    };
    load_gains(cw);
    if (t == 0 && wait_first) griddep_wait();
    load_values(cw);
    // (2) the norm's sum of squares: virtual warp w (played by warp w mod
    // nwc), lane l adds the squares of values 32w + l + vt*u in ascending u;
    // the next virtual warp's values are requested before this one's sum
    if (norm) {
      if (KU <= KU_MAX && K % vt == 0) {
        float cur[KU_MAX], nxt[KU_MAX];
#pragma unroll
        for (int u = 0; u < KU_MAX; ++u)
          if (u < KU && cw < nvw_all) cur[u] = ld_keep_cg(xr + 32 * cw + lane + vt * u);
        for (int w = cw; w < nvw_all; w += nwc) {
          const int wn = w + nwc;
#pragma unroll
          for (int u = 0; u < KU_MAX; ++u)
            if (u < KU && wn < nvw_all) nxt[u] = ld_keep_cg(xr + 32 * wn + lane + vt * u);
          A acc = 0;
#pragma unroll
          for (int u = 0; u < KU_MAX; ++u)
            if (u < KU) acc = fma_acc((A)cur[u], acc);
          acc = warp_tree_sum(acc);
          if (lane == 0) red[t * 32 + w] = acc;
#pragma unroll
          for (int u = 0; u < KU_MAX; ++u) cur[u] = nxt[u];
        }
      } else {
        for (int w = cw; w < nvw_all; w += nwc) {
          A acc = 0;
#pragma unroll 8
          for (int i = 32 * w + lane; i < K; i += vt) acc = fma_acc((A)__ldcg(xr + i), acc);
          acc = warp_tree_sum(acc);
          if (lane == 0) red[t * 32 + w] = acc;
        }
      }
      pstamp(dbg, 1);
      __syncthreads();
      if (cw == 0) {
        A v = lane < nvw_all ? red[t * 32 + lane] : (A)0;
        v = warp_tree_sum(v);
        if (lane == 0) den[t] = norm_div_add(v, K, a.eps);
      }
      __syncthreads();
      pstamp(dbg, 2);
    }
    const A dn = norm ? den[t] : (A)1;
    const float rdn = sizeof(A) == 4 ? __frcp_rn((float)dn) : 0.f;  // for div_row (f32 norms)
    // (3) normalize and quantize, batch by batch, four groups at a time in
    // lockstep (their division chains interleave)
    for (int g0 = cw; g0 < ng; g0 += QB * nwc) {
      if (g0 != cw) load_batch(g0);
      compiler_fence();
#pragma unroll
      for (int b0 = 0; b0 < QB; b0 += 4) {
        if (g0 + b0 * nwc >= ng) break;  // warp-uniform: the chunk is empty
        float v[4];
        bool ok[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int g = g0 + (b0 + k) * nwc;
          ok[k] = g < ng;
          v[k] = qx[b0 + k];
          // past the row's end (a chunk narrower than the area) the area keeps zeros
          if (norm && k_lo + 32 * g + lane < K) {
            if constexpr (sizeof(A) == 4) v[k] = norm_scale_r(v[k], (float)dn, rdn, qg[b0 + k]);
            else v[k] = norm_scale(v[k], dn, qg[b0 + k]);
          }
        }
        store_act4<Q, M>(act, L, t, g0 + b0 * nwc, nwc, lane, v, ok);
      }
    }
    pstamp(dbg, 3);
  }
  __syncthreads();
  pstamp(dbg, 4);
}

// ---- one GEMV's stage stream, shared by the ring and the chain kernels -------------

// Where a block's stages come from: rows [r0, r1) of a matrix, K chunk
// [k_lo, k_hi), cut into quads (4 rows) x slices (tk bytes of K).
struct Geom {
  const int8_t* wq;
  const unsigned char* ws;  // f16 scales, as bytes
  // The gated pair (F > 0): N = 2F logical rows interleaving the gate matrix
  // (wq, ws) and the up matrix (wq2, ws2) in 32-row tiles -- logical row L is
  // row 32 (L >> 6) + (L & 31) of the up matrix if bit 5 of L is set, else of
  // the gate matrix -- so a group of 32 outputs' gate and up rows are 64
  // neighbouring logical rows.  Quads are aligned to 4 rows, so a quad's rows
  // are consecutive rows of one matrix.
  const int8_t* wq2;
  const unsigned char* ws2;
  long F;
  long N;
  int K, nb;
  long r0, r1;
  int k_lo, k_hi, tk, nsl;
  bool whole;               // a stage is a whole quad: one copy of its levels, one per row of scales
  unsigned s_off, srow;     // scale area inside a stage, bytes per row there
};

__device__ __forceinline__ Geom make_geom(const int8_t* wq, const void* ws, long N, int K, long r0, long r1,
                                          int k_lo, int k_hi, int tk) {
  Geom g;
  g.wq = wq;
  g.ws = (const unsigned char*)ws;
  g.wq2 = nullptr;
  g.ws2 = nullptr;
  g.F = 0;
  g.N = N;
  g.K = K;
  g.nb = K >> 5;
  g.r0 = r0;
  g.r1 = r1;
  g.k_lo = k_lo;
  g.k_hi = k_hi;
  g.tk = tk;
  g.nsl = (k_hi - k_lo + tk - 1) / tk;
  g.whole = (k_lo == 0 && k_hi == K && tk >= K);
  g.s_off = (unsigned)(QR * tk);
  // 16 bytes of padding per row: the four rows' scales of a stage start in
  // different banks (a step's scale loads, one per row, need one wavefront)
  g.srow = (unsigned)tk / 16u + 16u;
  return g;
}

// Where logical row `row` lives: its matrix's levels and scales, and its row
// there (the row itself unless the geometry is a gated pair).
__device__ __forceinline__ void row_src(const Geom& g, long row, const int8_t*& wq, const unsigned char*& ws,
                                        long& prow) {
  if (g.F > 0) {
    const bool up = (row >> 5) & 1;
    wq = up ? g.wq2 : g.wq;
    ws = up ? g.ws2 : g.ws;
    prow = ((row >> 6) << 5) | (row & 31);
  } else {
    wq = g.wq;
    ws = g.ws;
    prow = row;
  }
}

// Stages of warp `warp` of `nwc`: its quads are warp, warp + nwc, ...
__device__ __forceinline__ long geom_stages(const Geom& g, int warp, int nwc) {
  const long nq = (g.r1 - g.r0 + QR - 1) / QR;
  return warp < nq ? ((nq - 1 - warp) / nwc + 1) * g.nsl : 0;
}

// Issue this warp's stage n (quad warp + nwc*(n / nsl), slice n % nsl) into
// the stage buffer `st`, completing on `full`.  All lanes call it.
__device__ __forceinline__ void issue_stage(const Geom& g, int warp, int nwc, long n, unsigned char* st,
                                            unsigned full, unsigned long long pol, int lane) {
  const long qi = warp + (long)nwc * (n / g.nsl);
  const int c = (int)(n % g.nsl);
  const long row0 = g.r0 + QR * qi;
  const int rows = g.r1 - row0 < QR ? (int)(g.r1 - row0) : QR;
  const int k0 = g.k_lo + c * g.tk;
  const int len = (g.k_hi - k0 < g.tk) ? g.k_hi - k0 : g.tk;
  const int8_t* wq;
  const unsigned char* ws;
  long prow0;
  row_src(g, row0, wq, ws, prow0);  // the quad's rows are prow0.. of one matrix
  if (g.whole) {
    if (lane == 0) {
      mbar_arrive_expect_tx(full, (unsigned)rows * (unsigned)g.K * 17u / 16u);
      bulk(st, wq + prow0 * g.K, rows * g.K, full, pol);
    }
    __syncwarp();
    if (lane < rows) bulk(st + g.s_off + lane * g.srow, ws + (prow0 + lane) * g.nb * 2, g.nb * 2, full, pol);
  } else {
    const int b0 = k0 >> 5, b1 = b0 + (len >> 5);
    const unsigned sh = (unsigned)(b0 & 7) * 2u;               // scales' offset in the first 16 B
    const unsigned slen = ((b1 - b0) * 2u + sh + 15u) & ~15u;  // 16-byte superset of a row's scales
    if (lane == 0) mbar_arrive_expect_tx(full, (unsigned)rows * (len + slen));
    __syncwarp();
    if (lane < rows) {
      const long row = prow0 + lane;
      bulk(st + lane * g.tk, wq + row * g.K + k0, len, full, pol);
      bulk(st + g.s_off + lane * g.srow, ws + ((row * g.nb + b0) * 2 - sh), slen, full, pol);
    }
  }
  __syncwarp();
}

// 16-byte load from L2 (not L1): for data an earlier kernel wrote.
__device__ __forceinline__ uint4 ld_cg16(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// The activation area of M rows over [k_lo, k_lo + L) (L a multiple of 128,
// k_lo of 128) loaded by every thread of the block with 16-byte L2 loads:
// int8 words (and low words) and f32 scales, or f32 values under Dequant, in
// the layout Act describes.  Plain loads rather than a bulk copy: a bulk copy
// issued after the block's weight stages completes only after them (the
// copy engine serves a block's copies in order), which held the activation
// back by the whole ring fill, several microseconds.
template <int Q, int M, int U = (M >= 4 ? 8 : 4)>  // U: loads in flight per thread
__device__ __forceinline__ void load_act(unsigned char* act, unsigned L, const lkh::GemvProblem& a, int k_lo) {
  const int K = a.K, nb = K >> 5, b_lo = k_lo >> 5;
  // 16-byte run i: its source and its place in the area
  auto run = [&](int i, const void*& src, unsigned char*& dst) {
    if constexpr (Q == 0) {
      const int per = (int)L / 4;
      const int t = i / per, c = i - t * per;
      src = a.x + (long)t * K + k_lo + 4 * c;
      dst = act + ((size_t)t * L + 4 * c) * 4;
    } else {
      const int per = (int)L / 16, pers = (int)L / 128, nw = M * per * (Q == 2 ? 2 : 1);
      if (i < nw) {
        const int lo = Q == 2 && i >= M * per;
        const int j = lo ? i - M * per : i;
        const int t = j / per, c = j - t * per;
        src = (lo ? a.xl : a.xq) + (long)t * K + k_lo + 16 * c;
        dst = act + (lo ? (size_t)M * L : 0) + (size_t)t * L + 16 * c;
      } else {
        const int j = i - nw, t = j / pers, c = j - t * pers;
        src = a.xs + (long)t * nb + b_lo + 4 * c;
        dst = act + (size_t)M * L * (Q == 2 ? 2 : 1) + (size_t)t * (L / 8) + 16 * c;
      }
    }
  };
  const int nrun = Q == 0 ? M * (int)L / 4 : M * (int)L / 16 * (Q == 2 ? 2 : 1) + M * (int)L / 128;
  for (int i0 = threadIdx.x; i0 < nrun; i0 += U * blockDim.x) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * blockDim.x;
      const void* src;
      unsigned char* dst;
      if (i < nrun) {
        run(i, src, dst);
        v[u] = ld_cg16(src);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * blockDim.x;
      const void* src;
      unsigned char* dst;
      if (i < nrun) {
        run(i, src, dst);
        *(uint4*)dst = v[u];
      }
    }
  }
  __syncthreads();
}

// The activation area of M rows over `L` bytes of K: int8 words (and low
// words) and f32 scales, or f32 values under Dequant.
struct Act {
  const unsigned char* base;
  unsigned L;
};

// Accumulate this warp's stage n (in `st`) into the partials p: 8 lanes per
// row, lane j reading bytes 16j..16j+15 of each 128-byte segment, lanes 2q and
// 2q+1 meeting by one xor-shuffle for block q's exact dot, lane 2q chaining
// partial q = b mod 4 in ascending block order ("kernels.rs" lk_q8_rows_dot,
// lk_q8_term).
template <int Q, int M>
__device__ __forceinline__ void compute_stage(typename part_t<Q>::t (&p)[M], const Geom& g, long n,
                                              const unsigned char* st, const Act& act, int lane) {
  const int rr = lane >> 3, j = lane & 7, q = j >> 1;
  const int c = (int)(n % g.nsl);
  const int k0 = g.k_lo + c * g.tk;
  const int len = (g.k_hi - k0 < g.tk) ? g.k_hi - k0 : g.tk;
  const int b0 = k0 >> 5;
  const unsigned sh = g.whole ? 0u : (unsigned)(b0 & 7) * 2u;
  const unsigned wrow = g.whole ? (unsigned)g.K : (unsigned)g.tk;
  const unsigned char* Wr = st + rr * wrow + 16 * j;
  const unsigned char* Sr = st + g.s_off + rr * g.srow + sh + 2 * q;
  const unsigned L = act.L;
  const unsigned char* XQ = act.base;
  const unsigned char* XL = act.base + (size_t)M * L;
  const float* XS = (const float*)(act.base + (size_t)M * L * (Q == 2 ? 2 : 1));
  const float* XF = (const float*)act.base;
  const int ka = k0 - g.k_lo;  // offset of this slice in the activation area
  const int nseg = len >> 7;
  if constexpr (Q == 0) {
    // Dequant: lane l takes values 4l..4l+3 of every 128-value segment, of
    // all four rows, so each f32 activation word is read from shared memory
    // once per warp (not once per row): its 4-value sums, scaled by the
    // block's weight scale, accumulate per lane and row in f32 over the
    // stage; at the stage's end each row's 32 lane sums are added by a
    // butterfly and lane 8r adds row r's total to its f64 partial (the
    // other lanes keep 0; finish_quad's reduction then only moves it).  The
    // order differs from a plain ascending sum; Dequant is held to the
    // tolerance (a stage of at most 64 segments adds at most ~75 f32
    // roundings of its sum of magnitudes, under 5e-6 of it).
    // The arithmetic runs on packed f32 pairs (values k and k+2 of the four
    // in the two halves): one instruction for two conversions, products or
    // sums.
    const unsigned char* W0 = st + 4 * lane;
    const unsigned char* S0 = st + g.s_off + sh + 2 * (lane >> 3);
    const f32x2 neg = f2_pack(-8388736.0f, -8388736.0f);  // 2^23 + 128, as in i8_as_f32
    f32x2 acc[M][QR];
#pragma unroll
    for (int t = 0; t < M; ++t)
#pragma unroll
      for (int r = 0; r < QR; ++r) acc[t][r] = f2_pack(0.f, 0.f);
#pragma unroll(M >= 4 ? 1 : 4)
    for (int seg = 0; seg < nseg; ++seg) {
      f32x2 w01[QR], w23[QR], ws2[QR];
#pragma unroll
      for (int r = 0; r < QR; ++r) {
        const unsigned u = *(const unsigned*)(W0 + r * wrow + 128 * seg) ^ 0x80808080u;
        const float wsr = __half2float(*(const __half*)(S0 + r * g.srow + 8 * seg));
        w01[r] = f2_add(f2_pack(i8_bits_f32(u, 0), i8_bits_f32(u, 1)), neg);
        w23[r] = f2_add(f2_pack(i8_bits_f32(u, 2), i8_bits_f32(u, 3)), neg);
        ws2[r] = f2_pack(wsr, wsr);
      }
#pragma unroll
      for (int t = 0; t < M; ++t) {
        const float4 xx = *(const float4*)(XF + (size_t)t * L + ka + 128 * seg + 4 * lane);
        const f32x2 x01 = f2_pack(xx.x, xx.y), x23 = f2_pack(xx.z, xx.w);
#pragma unroll
        for (int r = 0; r < QR; ++r) acc[t][r] = f2_fma(ws2[r], f2_fma(w23[r], x23, f2_mul(w01[r], x01)), acc[t][r]);
      }
    }
#pragma unroll
    for (int t = 0; t < M; ++t) {
#pragma unroll
      for (int r = 0; r < QR; ++r) {
        float a0, a1;
        f2_unpack(acc[t][r], a0, a1);
        float v = __fadd_rn(a0, a1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(FULL, v, o));
        if (lane == 8 * r) p[t] = __dadd_rn((double)p[t], (double)v);
      }
    }
    return;
  }
#pragma unroll 8
  for (int seg = 0; seg < nseg; ++seg) {
    const int4 w = *(const int4*)(Wr + 128 * seg);
    const float wsc = __half2float(*(const __half*)(Sr + 8 * seg));
    const int xo = ka + 128 * seg + 16 * j;
    const int bi = (ka >> 5) + 4 * seg + q;
#pragma unroll
    for (int t = 0; t < M; ++t) {
      const int4 hv = *(const int4*)(XQ + (size_t)t * L + xo);
      int d = dot16(w, hv);
      d += __shfl_xor_sync(FULL, d, 1);
      int e = 0;
      if constexpr (Q == 2) {
        const int4 lv = *(const int4*)(XL + (size_t)t * L + xo);
        e = dot16(w, lv);
        e += __shfl_xor_sync(FULL, e, 1);
      }
      const float s = XS[(size_t)t * (L / 32) + bi];
      p[t] = q8_step<Q>((float)p[t], wsc, s, d, e);
    }
  }
}

// The last slice of a quad: (p0 + p2) + (p1 + p3) within each row's 8 lanes
// ("kernels.rs" lk_q8_sum4), stored as y (and an argmax key) or as split-K
// partial `chunk`; p is reset.
template <int Q, int M, bool SPLIT>
__device__ __forceinline__ void finish_quad(typename part_t<Q>::t (&p)[M], const Geom& g, int warp, int nwc, long n,
                                            const lkh::GemvProblem& a, int chunk, float* y,
                                            unsigned long long (&best)[M], int lane) {
  typedef typename part_t<Q>::t P;
  const int rr = lane >> 3, j = lane & 7;
  const long qi = warp + (long)nwc * (n / g.nsl);
  const long row0 = g.r0 + QR * qi;
  const int rows = g.r1 - row0 < QR ? (int)(g.r1 - row0) : QR;
#pragma unroll
  for (int t = 0; t < M; ++t) {
    P v = p[t];
    v = v + __shfl_down_sync(FULL, v, 4);
    v = v + __shfl_down_sync(FULL, v, 2);
    p[t] = (P)0;
    if (j == 0 && rr < rows) {
      const long o = row0 + rr;
      if (SPLIT) {
        const long idx = ((long)chunk * M + t) * g.N + o;
        if constexpr (Q == 0) a.part64[idx] = (double)v;
        else a.y[idx] = (float)v;
      } else if (g.F > 0) {
        // the gated pair: gate values [M][F], then up values [M][F]
        const long prow = ((o >> 6) << 5) | (o & 31);
        y[(((o >> 5) & 1) * M + t) * g.F + prow] = Q == 0 ? __double2float_rn((double)v) : (float)v;
      } else {
        const float yv = Q == 0 ? __double2float_rn((double)v) : (float)v;
        y[(long)t * g.N + o] = yv;
        const unsigned long long kk = amax_key(yv, (unsigned)o);
        best[t] = kk > best[t] ? kk : best[t];
      }
    }
  }
}

// Bounded wait on `bar` that ignores the abort flag (used to drain copies).
__device__ __forceinline__ void drain_wait(unsigned bar, unsigned parity, unsigned long long limit_ns, int* err) {
  const unsigned long long t0 = gtimer();
  while (!mbar_try(bar, parity)) {
    if (gtimer() - t0 > limit_ns) {
      atomicOr(err, ERR_DRAIN);
      break;
    }
  }
}

// The SwiGLU epilogue of a gated pair ("kernels.rs" lk_gemv_glu with a
// quantized output): output group j (32 outputs) needs the 64 logical rows
// [64 j, 64 j + 64), its 32 gate and 32 up values.  A block whose rows hold
// the whole group finishes it; a group split between two blocks is finished
// by the one that completes its count: each adds the rows it wrote to
// glu_cnt[j] after a fence, and the one whose add reaches 64 reads the other's
// values back through L2 and resets the count for the next launch.  A warp
// per group: lane l computes h = swiglu(gate, up) of output 32 j + l for every
// activation row and quantizes the 32 values as one group.
template <int Q, int M>
__device__ __forceinline__ void glu_epilogue(const lkh::GemvProblem& a, const Geom& g, int nwc, int warp, int lane) {
  __threadfence();  // this block's gate/up values before any of its counts
  __syncthreads();
  if (g.r1 <= g.r0) return;
  const long F = a.F;
  const long j0 = g.r0 >> 6, j1 = (g.r1 - 1) >> 6;
  for (long j = j0 + warp; j <= j1; j += nwc) {
    const long lo = g.r0 > 64 * j ? g.r0 : 64 * j, hi = g.r1 < 64 * j + 64 ? g.r1 : 64 * j + 64;
    const int c = (int)(hi - lo);
    if (c < 64) {
      int old = 0;
      if (lane == 0) old = atomicAdd(a.glu_cnt + j, c);
      old = __shfl_sync(FULL, old, 0);
      if (old + c != 64) continue;  // the other block finishes the group
      if (lane == 0) a.glu_cnt[j] = 0;
      __threadfence();  // the other block's values after its count
    }
#pragma unroll
    for (int t = 0; t < M; ++t) {
      const long i = (long)t * F + 32 * j + lane;
      const float hv = swiglu(__ldcg(a.y + i), __ldcg(a.y + (long)M * F + i));
      if (a.h) a.h[i] = hv;
      if constexpr (Q > 0)
        quant_lane<Q>(hv, a.hq + (long)t * F, Q == 2 ? a.hl + (long)t * F : nullptr, a.hs + (long)t * (F >> 5), j,
                      lane);
    }
  }
}

template <int Q, int M, bool SPLIT, bool FUSE, bool GLU = false>
__global__ void __launch_bounds__(THREADS_MAX, 1) gemv_ring_kernel(const RingArgs ra) {
  typedef typename part_t<Q>::t P;
  extern __shared__ __align__(128) unsigned char smem[];
  const lkh::GemvProblem& a = ra.p;
  const int nwc = ra.nwc, D = ra.depth, NS = nwc * D;
  unsigned char* act = smem;
  unsigned char* ring = smem + ra.ring_off;
  unsigned long long* bars = (unsigned long long*)(ring + (size_t)NS * ra.stage_bytes);
  volatile int* abort_flag = (volatile int*)(bars + MAX_STAGES + 1);
  unsigned long long* keys = (unsigned long long*)(bars + MAX_STAGES + 3);  // [M][MAXW]
  double* nred = (double*)(keys + LK_MAX_M * MAXW);                        // [M][32]
  double* nden = nred + LK_MAX_M * 32;                                     // [M]
  const unsigned full0 = smem_u32(bars);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.K, nb = K >> 5;
  const long N = a.N;
  int b_lo = 0, b_hi = nb;
  if (SPLIT) {
    b_lo = splitk_bound(nb, a.S, blockIdx.y);
    b_hi = splitk_bound(nb, a.S, blockIdx.y + 1);
  }
  const int k_lo = 32 * b_lo;
  // a gated pair's rows are split in whole quads (a quad never straddles
  // the 32-row tiles of its matrices)
  const long q_lo = GLU ? 4 * ((long)blockIdx.x * (N >> 2) / ra.gx) : (long)blockIdx.x * N / ra.gx;
  const long q_hi = GLU ? 4 * ((long)(blockIdx.x + 1) * (N >> 2) / ra.gx) : (long)(blockIdx.x + 1) * N / ra.gx;
  Geom g = make_geom(a.wq, a.ws, N, K, q_lo, q_hi, k_lo, 32 * b_hi, (int)ra.tk);
  if (GLU) {
    g.wq2 = a.wq2;
    g.ws2 = (const unsigned char*)a.ws2;
    g.F = a.F;
  }
  const unsigned L = ra.act_len;
  const long T = geom_stages(g, warp, nwc);
  const unsigned long long pol_w = ra.pol_w ? evict_first_policy() : 0ull;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(full0 + 8 * s, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (ra.pdl && threadIdx.x == 0) griddep_launch();

  // Weights do not depend on the previous kernel: start streaming at once.
  tstamp(ra.trace, ra.tslot, TR_START);
  // (warps >= prefill issue their first stages only once the activation is
  // ready: a full ring's requests ahead of the dependency wait slow the
  // activation's own loads)
  long issued = 0;
  const bool early = warp < ra.prefill;
  for (; early && issued < T && issued < D; ++issued)
    issue_stage(g, warp, nwc, issued, ring + (size_t)(warp * D + issued % D) * ra.stage_bytes,
                full0 + 8 * (warp * D + (int)(issued % D)), pol_w, lane);
  tstamp(ra.trace, ra.tslot, TR_ISSUED);

  // from the dependency wait on: reads of activations, writes of outputs (the
  // fused prologue waits itself, after requesting the norm gains)
  if (ra.pdl && !FUSE) griddep_wait();
  tstamp(ra.trace, ra.tslot, TR_WAITED);
  bool ok = true;
  if (FUSE) {
    fused_prologue<Q, M>(a, nwc, k_lo, L, act, nred, nden, ra.trace && ra.tslot < 0 ? ra.trace + 32 : nullptr,
                         ra.pdl != 0);
  } else if (L > 0) {
    load_act<Q, M>(act, L, a, k_lo);
  }
  for (; !early && issued < T && issued < D; ++issued)
    issue_stage(g, warp, nwc, issued, ring + (size_t)(warp * D + issued % D) * ra.stage_bytes,
                full0 + 8 * (warp * D + (int)(issued % D)), pol_w, lane);

  const Act ac{act, L};
  tstamp(ra.trace, ra.tslot, TR_ACT);
  unsigned long long best[M];
  P p[M];
#pragma unroll
  for (int t = 0; t < M; ++t) {
    best[t] = 0;
    p[t] = (P)0;
  }
  long n = 0;
  for (; ok && n < T; ++n) {
    const int slot = warp * D + (int)(n % D);
    if (!__all_sync(FULL, mbar_wait(full0 + 8 * slot, (unsigned)(n / D) & 1u, ra.wait_ns, abort_flag))) {
      if (lane == 0) raise_error(ra.err, ERR_WAIT_FULL, abort_flag);
      ok = false;
      break;
    }
    unsigned char* st = ring + (size_t)slot * ra.stage_bytes;
    compute_stage<Q, M>(p, g, n, st, ac, lane);
    // The slot is free again: refill it with this warp's stage n + D.  The
    // generic-proxy reads above must be ordered before the bulk copy's
    // async-proxy writes into the same bytes.
    __syncwarp();
    if (issued < T) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue_stage(g, warp, nwc, issued, st, full0 + 8 * slot, pol_w, lane);
      ++issued;
    }
    if ((int)(n % g.nsl) == g.nsl - 1) finish_quad<Q, M, SPLIT>(p, g, warp, nwc, n, a, blockIdx.y, a.y, best, lane);
  }
  if (ra.trace && ra.tslot < 0 && blockIdx.x == 0 && lane == 0) ra.trace[3 + warp] = gtimer();
  // Drain: stages this warp issued but did not consume (only after an
  // abort) must land before the block may end.
  if (lane == 0) {
    for (long m = n; m < issued; ++m)
      drain_wait(full0 + 8 * (unsigned)(warp * D + m % D), (unsigned)(m / D) & 1u, ra.wait_ns, ra.err);
  }
  __syncwarp();
  if constexpr (GLU) {
    __syncthreads();
    if (!*abort_flag) glu_epilogue<Q, M>(a, g, nwc, warp, lane);
  }
  if (!SPLIT && !GLU && a.amax) {
#pragma unroll
    for (int t = 0; t < M; ++t) {
      const unsigned long long wmax = warp_max_u64(best[t]);
      if (lane == 0) keys[t * MAXW + warp] = wmax;
    }
    __syncthreads();
    if (threadIdx.x < M) {
      unsigned long long m = 0;
      for (int w = 0; w < nwc; ++w) m = keys[threadIdx.x * MAXW + w] > m ? keys[threadIdx.x * MAXW + w] : m;
      a.amax[(long)threadIdx.x * gridDim.x + blockIdx.x] = m;
    }
  }
  tend(ra.trace, ra.tslot, N, 1);
}

// Explicit instantiation of every (M, SPLIT, FUSE) kernel of mode Q.
#define LK_RING_PICK(Q)                                                             \
  template <>                                                                       \
  ring_fn ring_pick<Q>(int M, bool split, bool fuse, bool glu) {                    \
    if (glu) return gemv_ring_kernel<Q, 1, false, false, true>;                     \
    if (split) {                                                                    \
      switch (M) {                                                                  \
        case 1: return gemv_ring_kernel<Q, 1, true, false>;                         \
        case 2: return gemv_ring_kernel<Q, 2, true, false>;                         \
        case 3: return gemv_ring_kernel<Q, 3, true, false>;                         \
        case 4: return gemv_ring_kernel<Q, 4, true, false>;                         \
        case 5: return gemv_ring_kernel<Q, 5, true, false>;                         \
        case 6: return gemv_ring_kernel<Q, 6, true, false>;                         \
        case 7: return gemv_ring_kernel<Q, 7, true, false>;                         \
        default: return gemv_ring_kernel<Q, 8, true, false>;                        \
      }                                                                             \
    }                                                                               \
    if (fuse) {                                                                     \
      switch (M) {                                                                  \
        case 1: return gemv_ring_kernel<Q, 1, false, true>;                         \
        case 2: return gemv_ring_kernel<Q, 2, false, true>;                         \
        case 3: return gemv_ring_kernel<Q, 3, false, true>;                         \
        case 4: return gemv_ring_kernel<Q, 4, false, true>;                         \
        case 5: return gemv_ring_kernel<Q, 5, false, true>;                         \
        case 6: return gemv_ring_kernel<Q, 6, false, true>;                         \
        case 7: return gemv_ring_kernel<Q, 7, false, true>;                         \
        default: return gemv_ring_kernel<Q, 8, false, true>;                        \
      }                                                                             \
    }                                                                               \
    switch (M) {                                                                    \
      case 1: return gemv_ring_kernel<Q, 1, false, false>;                          \
      case 2: return gemv_ring_kernel<Q, 2, false, false>;                          \
      case 3: return gemv_ring_kernel<Q, 3, false, false>;                          \
      case 4: return gemv_ring_kernel<Q, 4, false, false>;                          \
      case 5: return gemv_ring_kernel<Q, 5, false, false>;                          \
      case 6: return gemv_ring_kernel<Q, 6, false, false>;                          \
      case 7: return gemv_ring_kernel<Q, 7, false, false>;                          \
      default: return gemv_ring_kernel<Q, 8, false, false>;                         \
    }                                                                               \
  }

}  // namespace lkring
