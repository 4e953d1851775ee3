// The Q8_0 GEMV entry points: plain GEMV (with the optional argmax
// epilogue), the split-K partial GEMV and the split-K combine.
//
// Direct-load kernel (any K % 32 == 0).  A warp owns 4 consecutive rows;
// lane = 8*r + j serves row r, and within each 128-byte segment of the row
// (four 32-blocks) lane j reads bytes 16j..16j+15, so the 8 lanes of a row
// read one contiguous 128-byte line and lanes 2q, 2q+1 hold block q of the
// segment.  The pair's two 16-value dots meet by one xor-shuffle, which
// makes the block's int32 dot exact on both lanes.  Block b = 4*seg + q is
// always in partial q = b mod 4 ("kernels.rs" lk_q8_rows_dot), so lane 2q
// carries that partial's fused chain over the row's segments in ascending
// order with no per-block shuffles; at the end (p0 + p2) + (p1 + p3)
// (lk_q8_sum4) takes two shuffle-downs inside the 8 lanes.  U segments'
// weights are loaded before any is used, so each lane keeps U 16-byte loads
// in flight.
#include "lk_device.cuh"
#include "lk_host.h"

using namespace lk;
using namespace lkh;

namespace {

constexpr int kWarps = 8;          // warps per block
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerBlock = kWarps * kRowsPerWarp;
constexpr int kU = 8;              // segments in flight per lane

template <int Q>
struct part_t { typedef float t; };
template <>
struct part_t<0> { typedef double t; };

template <int Q, int M, bool SPLIT>
__global__ void __launch_bounds__(256) gemv_direct_kernel(GemvProblem a) {
  typedef typename part_t<Q>::t P;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rr = lane >> 3, j = lane & 7, q = j >> 1, hf = j & 1;
  const long o = ((long)blockIdx.x * kWarps + warp) * kRowsPerWarp + rr;
  const bool row_ok = o < a.N;
  const int K = a.K, nb = K >> 5;
  int b_lo = 0, b_hi = nb;
  if (SPLIT) {
    b_lo = splitk_bound(nb, a.S, blockIdx.y);
    b_hi = splitk_bound(nb, a.S, blockIdx.y + 1);
  }
  const int sg_lo = b_lo >> 2, sg_hi = (b_hi + 3) >> 2;
  const long orow = row_ok ? o : 0;
  const int8_t* __restrict__ wrow = a.wq + orow * K + 16 * hf;
  const __half* __restrict__ srow = a.ws + orow * nb;
  const int4 zero = make_int4(0, 0, 0, 0);

  P p[M];
#pragma unroll
  for (int t = 0; t < M; ++t) p[t] = (P)0;

  for (int sg0 = sg_lo; sg0 < sg_hi; sg0 += kU) {
    int4 wv[kU];
    float wsv[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int b = 4 * (sg0 + u) + q;
      const bool ok = row_ok && b < b_hi;
      wv[u] = ok ? ld_stream16(wrow + 32L * b) : zero;
      wsv[u] = ok ? __half2float(srow[b]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (sg0 + u >= sg_hi) break;  // warp-uniform
      const int b = 4 * (sg0 + u) + q;
      const bool bok = b < b_hi;
      const long off = 32L * b + 16 * hf;
#pragma unroll
      for (int t = 0; t < M; ++t) {
        if constexpr (Q == 0) {
          const float4* xv = (const float4*)(a.x + (long)t * K + off);
          float4 xx[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) xx[c] = bok ? __ldg(xv + c) : make_float4(0.f, 0.f, 0.f, 0.f);
          const int wi[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
          float h = 0.f;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float xe[4] = {xx[c].x, xx[c].y, xx[c].z, xx[c].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) h = __fmaf_rn(i8_as_f32((unsigned)wi[c] ^ 0x80808080u, k), xe[k], h);
          }
          const float blk = __fadd_rn(h, __shfl_xor_sync(FULL, h, 1));
          if (bok) p[t] = __fma_rn((double)wsv[u], (double)blk, (double)p[t]);
        } else {
          const int4 hv = bok ? __ldg((const int4*)(a.xq + (long)t * K + off)) : zero;
          int d = dot16(wv[u], hv);
          d += __shfl_xor_sync(FULL, d, 1);
          int e = 0;
          if constexpr (Q == 2) {
            const int4 lv = bok ? __ldg((const int4*)(a.xl + (long)t * K + off)) : zero;
            e = dot16(wv[u], lv);
            e += __shfl_xor_sync(FULL, e, 1);
          }
          const float s = bok ? __ldg(a.xs + (long)t * nb + b) : 0.f;
          if (bok) p[t] = q8_step<Q>((float)p[t], wsv[u], s, d, e);
        }
      }
    }
  }

  // (p0 + p2) + (p1 + p3) within the row's 8 lanes; lane 8r holds the row.
  unsigned long long best[M];
#pragma unroll
  for (int t = 0; t < M; ++t) {
    P v = p[t];
    v = v + __shfl_down_sync(FULL, v, 4);
    v = v + __shfl_down_sync(FULL, v, 2);
    best[t] = 0;
    if (j == 0 && row_ok) {
      if (SPLIT) {
        const long idx = ((long)blockIdx.y * M + t) * a.N + o;
        if constexpr (Q == 0) a.part64[idx] = (double)v;
        else a.y[idx] = (float)v;
      } else {
        const float yv = Q == 0 ? __double2float_rn((double)v) : (float)v;
        a.y[(long)t * a.N + o] = yv;
        best[t] = amax_key(yv, (unsigned)o);
      }
    }
  }
  if (!SPLIT && a.amax) {
    __shared__ unsigned long long sh[M][kWarps];
#pragma unroll
    for (int t = 0; t < M; ++t) {
      const unsigned long long w = warp_max_u64(best[t]);
      if (lane == 0) sh[t][warp] = w;
    }
    __syncthreads();
    if (threadIdx.x < M) {
      unsigned long long m = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) m = sh[threadIdx.x][w] > m ? sh[threadIdx.x][w] : m;
      a.amax[(long)threadIdx.x * gridDim.x + blockIdx.x] = m;
    }
  }
}

typedef void (*kernel_fn)(GemvProblem);

template <int Q, bool SPLIT>
kernel_fn pick_m(int M) {
  switch (M) {
    case 1: return gemv_direct_kernel<Q, 1, SPLIT>;
    case 2: return gemv_direct_kernel<Q, 2, SPLIT>;
    case 3: return gemv_direct_kernel<Q, 3, SPLIT>;
    case 4: return gemv_direct_kernel<Q, 4, SPLIT>;
    case 5: return gemv_direct_kernel<Q, 5, SPLIT>;
    case 6: return gemv_direct_kernel<Q, 6, SPLIT>;
    case 7: return gemv_direct_kernel<Q, 7, SPLIT>;
    default: return gemv_direct_kernel<Q, 8, SPLIT>;
  }
}

kernel_fn pick(int mode, int M, bool split) {
  if (split) {
    if (mode == 0) return pick_m<0, true>(M);
    if (mode == 1) return pick_m<1, true>(M);
    return pick_m<2, true>(M);
  }
  if (mode == 0) return pick_m<0, false>(M);
  if (mode == 1) return pick_m<1, false>(M);
  return pick_m<2, false>(M);
}

lk_status direct_gemv(const GemvProblem& p, cudaStream_t stream, int* n_parts) {
  const long blocks = (p.N + kRowsPerBlock - 1) / kRowsPerBlock;
  if (blocks > 0x7fffffffL) return LK_ERR_SHAPE;
  kernel_fn f = pick(p.mode, p.M, false);
  f<<<(unsigned)blocks, kWarps * 32, 0, stream>>>(p);
  if (n_parts) *n_parts = (int)blocks;
  return launch_status();
}

lk_status check_common(const int8_t* wq, const uint16_t* ws, int N, int K, lk_mode mode,
                       const float* x, const int8_t* xq, const int8_t* xl, const float* xs, int M) {
  if (mode < LK_DEQUANT || mode > LK_TWOPASS) return LK_ERR_ARG;
  if (N < 0 || K < 0 || K % 32 || M < 0 || M > LK_MAX_BATCH) return LK_ERR_SHAPE;
  if (K == 0) return LK_OK;  // nothing is read: every output is 0
  if (!wq || !ws) return LK_ERR_ARG;
  if (mode == LK_DEQUANT ? !x : (!xq || !xs || (mode == LK_TWOPASS && !xl))) return LK_ERR_ARG;
  if (!aligned(wq, 16) || !aligned(ws, 2)) return LK_ERR_ALIGN;
  if (mode == LK_DEQUANT ? !aligned(x, 16)
                         : (!aligned(xq, 16) || !aligned(xs, 4) || (mode == LK_TWOPASS && !aligned(xl, 16))))
    return LK_ERR_ALIGN;
  return LK_OK;
}

GemvProblem make_problem(const int8_t* wq, const uint16_t* ws, int N, int K, lk_mode mode,
                         const float* x, const int8_t* xq, const int8_t* xl, const float* xs, int M) {
  GemvProblem p;
  p.wq = wq;
  p.ws = (const __half*)ws;
  p.N = N;
  p.K = K;
  p.mode = mode;
  p.x = x;
  p.xq = xq;
  p.xl = xl;
  p.xs = xs;
  p.M = M;
  p.S = 1;
  p.split = false;
  p.y = nullptr;
  p.part64 = nullptr;
  p.amax = nullptr;
  p.fuse = false;
  p.xraw = nullptr;
  p.gain = nullptr;
  p.eps = 0.f;
  p.F = 0;
  p.wq2 = nullptr;
  p.ws2 = nullptr;
  p.glu_cnt = nullptr;
  p.h = nullptr;
  p.hq = nullptr;
  p.hl = nullptr;
  p.hs = nullptr;
  apply_cfg(p, nullptr);
  return p;
}

// One output of the combine: y = (((0 + c0) + c1) + ...) in ascending
// chunk order, the partials read through L2 (an earlier kernel wrote them).
template <bool F64>
__device__ __forceinline__ void combine_one(const void* __restrict__ part, int S, long MN, float* __restrict__ y,
                                            long i) {
  if (F64) {
    const double* pp = (const double*)part;
    double acc = 0.0;
    for (int c = 0; c < S; ++c) acc = __dadd_rn(acc, __ldcg(pp + (long)c * MN + i));
    y[i] = __double2float_rn(acc);
  } else {
    const float* pp = (const float*)part;
    float acc = 0.f;
    for (int c = 0; c < S; ++c) acc = __fadd_rn(acc, __ldcg(pp + (long)c * MN + i));
    y[i] = acc;
  }
}

// Combine: y = (((0 + c0) + c1) + ...) in ascending chunk order.  As a
// programmatic dependent it lets its own dependent launch at once and reads
// the partials only after the split-K launch before it has completed.
template <bool F64>
__global__ void __launch_bounds__(256) splitk_combine_kernel(const void* __restrict__ part, int S, long MN,
                                                             float* __restrict__ y, unsigned long long* tr,
                                                             int slot) {
  asm volatile("griddepcontrol.launch_dependents;" :::);
  trec_stamp(tr, slot, TR_START);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  trec_stamp(tr, slot, TR_WAITED);
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < MN) {
    combine_one<F64>(part, S, MN, y, i);
  }
  trec_end(tr, slot, TK_COMBINE, MN);
}

}  // namespace

extern "C" {

lk_status lk_gemv_q8(const int8_t* wq, const uint16_t* ws, int N, int K, lk_mode mode, const float* x,
                     const int8_t* xq, const int8_t* xl, const float* xs, int M, float* y,
                     uint64_t* argmax_parts, int* n_parts_out, const lk_launch_cfg* cfg, cudaStream_t stream) {
  lk_status st = check_common(wq, ws, N, K, mode, x, xq, xl, xs, M);
  if (st) return st;
  st = check_launch_cfg(cfg);
  if (st) return st;
  if (argmax_parts && !n_parts_out) return LK_ERR_ARG;
  if (N == 0 || M == 0) {
    if (n_parts_out) *n_parts_out = 0;
    return LK_OK;
  }
  if (!y) return LK_ERR_ARG;
  if (!aligned(y, 4) || (argmax_parts && !aligned(argmax_parts, 8))) return LK_ERR_ALIGN;
  // the argmax keys are sized by lk_argmax_parts_max: no more blocks than that
  if (argmax_parts && cfg && cfg->grid_ctas > lk_argmax_parts_max(N)) return LK_ERR_ARG;
  GemvProblem p = make_problem(wq, ws, N, K, mode, x, xq, xl, xs, M);
  apply_cfg(p, cfg);
  p.y = y;
  p.amax = (unsigned long long*)argmax_parts;
  int n_parts = 0;
  const int path = p.cfg.path;
  if ((path == 0 || path == 3) && mma_supports(p)) {
    st = mma_gemv(p, stream, &n_parts);
  } else if (path == 3 || M > LK_MAX_M) {
    return LK_ERR_SHAPE;  // past 8 rows: the tensor-core kernel only
  } else if (path != 1 && ring_supports(p)) {
    st = ring_gemv(p, stream, &n_parts);
  } else {
    if (path == 2) return LK_ERR_SHAPE;
    st = direct_gemv(p, stream, &n_parts);
  }
  if (n_parts_out) *n_parts_out = n_parts;
  return st;
}

lk_status lk_gemv_q8_group(const lk_gemv_target* targets, int n, int K, lk_mode mode, const float* x,
                           const int8_t* xq, const int8_t* xl, const float* xs, int M, const lk_launch_cfg* cfg,
                           cudaStream_t stream) {
  if (!targets || n < 1 || n > LK_MAX_GROUP) return LK_ERR_ARG;
  {
    const lk_status st = check_launch_cfg(cfg);
    if (st) return st;
  }
  for (int i = 0; i < n; ++i) {
    const lk_gemv_target& t = targets[i];
    if (!t.wq || !t.ws || !t.y) return LK_ERR_ARG;
    lk_status st = check_common(t.wq, t.ws, t.N, K, mode, x, xq, xl, xs, M);
    if (st) return st;
    if (t.N < 1) return LK_ERR_SHAPE;
    if (!aligned(t.y, 4)) return LK_ERR_ALIGN;
  }
  if (M == 0 || K == 0) {
    for (int i = 0; i < n; ++i) {
      lk_status st = lk_gemv_q8(targets[i].wq, targets[i].ws, targets[i].N, K, mode, x, xq, xl, xs, M,
                                targets[i].y, nullptr, nullptr, cfg, stream);
      if (st) return st;
    }
    return LK_OK;
  }
  GemvProblem p = make_problem(targets[0].wq, targets[0].ws, targets[0].N, K, mode, x, xq, xl, xs, M);
  apply_cfg(p, cfg);
  const int path = p.cfg.path;
  bool one = (path == 0 || path == 3);
  for (int i = 0; i < n && one; ++i) {
    GemvProblem q = p;
    q.wq = targets[i].wq;
    q.ws = (const __half*)targets[i].ws;
    q.N = targets[i].N;
    one = mma_supports(q);
  }
  if (one) {
    const int8_t* wq[LK_MAX_GROUP];
    const __half* ws[LK_MAX_GROUP];
    long N[LK_MAX_GROUP];
    float* y[LK_MAX_GROUP];
    for (int i = 0; i < n; ++i) {
      wq[i] = targets[i].wq;
      ws[i] = (const __half*)targets[i].ws;
      N[i] = targets[i].N;
      y[i] = targets[i].y;
    }
    return mma_launch(p, n, wq, ws, N, y, stream, nullptr);
  }
  // one chain launch (the ring kernel's arrangement) where it takes the shape
  if (n > 1 && (path == 0 || path == 2)) {
    const lk_status st = chain_group(p, targets, n, stream);
    if (st != LK_ERR_SHAPE) return st;
  }
  for (int i = 0; i < n; ++i) {
    lk_status st = lk_gemv_q8(targets[i].wq, targets[i].ws, targets[i].N, K, mode, x, xq, xl, xs, M, targets[i].y,
                              nullptr, nullptr, cfg, stream);
    if (st) return st;
  }
  return LK_OK;
}

int lk_gemv_kernel_for(int N, int K, lk_mode mode, int M, int S, const lk_launch_cfg* cfg) {
  if (mode < LK_DEQUANT || mode > LK_TWOPASS || N < 1 || K < 32 || K % 32 || M < 1 || M > LK_MAX_BATCH || S < 0 ||
      S > LK_MAX_SPLITK || check_launch_cfg(cfg))
    return 0;
  // 16-byte aligned stand-in pointers: only the shape decides
  const void* a16 = (const void*)(uintptr_t)256;
  GemvProblem p = make_problem((const int8_t*)a16, (const uint16_t*)a16, N, K, mode, (const float*)a16,
                               (const int8_t*)a16, (const int8_t*)a16, (const float*)a16, M);
  p.split = S > 0;
  p.S = S > 0 ? S : 1;
  apply_cfg(p, cfg);
  const int path = p.cfg.path;
  if ((path == 0 || path == 3) && mma_supports(p)) return 3;
  if (M > LK_MAX_M || path == 3) return 0;
  if (path == 1) return 1;
  return ring_supports(p) ? 2 : (path == 2 ? 0 : 1);
}

lk_status lk_rmsnorm_quant_gemv_q8(const int8_t* wq, const uint16_t* ws, int N, int K, lk_mode mode,
                                   const float* x, const float* gain, float eps, int M, float* y,
                                   uint64_t* argmax_parts, int* n_parts_out, const lk_launch_cfg* cfg,
                                   cudaStream_t stream) {
  if (mode < LK_DEQUANT || mode > LK_TWOPASS || check_launch_cfg(cfg)) return LK_ERR_ARG;
  if (cfg && cfg->path != 0 && cfg->path != 2) return LK_ERR_SHAPE;
  if (N < 0 || K < 0 || K % 32 || M < 0 || M > LK_MAX_M) return LK_ERR_SHAPE;
  if (argmax_parts && !n_parts_out) return LK_ERR_ARG;
  if (N == 0 || M == 0) {
    if (n_parts_out) *n_parts_out = 0;
    return LK_OK;
  }
  if (!wq || !ws || !x || !y) return LK_ERR_ARG;
  if (!aligned(wq, 16) || !aligned(ws, 2) || !aligned(x, 4) || (gain && !aligned(gain, 4)) || !aligned(y, 4) ||
      (argmax_parts && !aligned(argmax_parts, 8)))
    return LK_ERR_ALIGN;
  if (argmax_parts && cfg && cfg->grid_ctas > lk_argmax_parts_max(N)) return LK_ERR_ARG;
  GemvProblem p = make_problem(wq, ws, N, K, mode, nullptr, nullptr, nullptr, nullptr, M);
  apply_cfg(p, cfg);
  p.fuse = true;
  p.xraw = x;
  p.gain = gain;
  p.eps = eps;
  p.y = y;
  p.amax = (unsigned long long*)argmax_parts;
  if (!ring_supports(p)) return LK_ERR_SHAPE;
  int n_parts = 0;
  lk_status st = ring_gemv(p, stream, &n_parts);
  if (n_parts_out) *n_parts_out = n_parts;
  return st;
}

lk_status lk_gemv_q8_glu(const int8_t* wg, const uint16_t* wsg, const int8_t* wu, const uint16_t* wsu, int F, int K,
                         lk_mode mode, const float* x, const int8_t* xq, const int8_t* xl, const float* xs, int M,
                         float* gu, float* h, int8_t* hq, int8_t* hl, float* hs, int* cnt, const lk_launch_cfg* cfg,
                         cudaStream_t stream) {
  lk_status st = check_common(wg, wsg, F, K, mode, x, xq, xl, xs, M);
  if (st) return st;
  st = check_launch_cfg(cfg);
  if (st) return st;
  st = check_common(wu, wsu, F, K, mode, x, xq, xl, xs, M);
  if (st) return st;
  if (F % 32) return LK_ERR_SHAPE;
  if (F == 0 || M == 0) return LK_OK;
  if (!gu) return LK_ERR_ARG;
  if (!aligned(gu, 4) || (h && !aligned(h, 4))) return LK_ERR_ALIGN;
  if (mode == LK_DEQUANT) {
    if (!h) return LK_ERR_ARG;
  } else {
    st = check_act_out(mode, hq, hl, hs);
    if (st) return st;
  }
  if (K > 0 && (!cfg || cfg->path == 0)) {
    GemvProblem p = make_problem(wg, wsg, 2 * F, K, mode, x, xq, xl, xs, M);
    apply_cfg(p, cfg);
    p.y = gu;
    p.F = F;
    p.wq2 = wu;
    p.ws2 = (const __half*)wsu;
    p.glu_cnt = cnt;
    p.h = h;
    p.hq = mode == LK_DEQUANT ? nullptr : hq;
    p.hl = mode == LK_TWOPASS ? hl : nullptr;
    p.hs = mode == LK_DEQUANT ? nullptr : hs;
    if (cnt && aligned(cnt, 4) && ring_supports(p)) return ring_gemv(p, stream, nullptr);
  }
  // two launches: both GEMVs (one grouped launch where the kernels allow),
  // then the SwiGLU -> quantize step over their outputs
  const lk_gemv_target t[2] = {{wg, wsg, F, 0, gu}, {wu, wsu, F, 0, gu + (long)M * F}};
  st = lk_gemv_q8_group(t, 2, K, mode, x, xq, xl, xs, M, cfg, stream);
  if (st) return st;
  return lk_swiglu_quant(gu, gu + (long)M * F, M, F, F, mode, h, hq, hl, hs, cfg, stream);
}

// Measured on GB300 (bench.py gemv workload, combine included, us; S = 1,
// 2, 4, 8, 12, 16, 24) for q|k|v 6144 x 4096, o 4096 x 4096, gate/up
// 24576 x 4096 and down 4096 x 12288:
//  * up to 8 rows, S = 8 is best or within 3 % everywhere: down 27.6 ->
//    17.6 (Int8Act, 8 rows), 64.2 -> 21.4 (TwoPass), q|k|v 14.0 -> 12.7,
//    gate/up 36.2 -> 31.3 (TwoPass); S = 12 .. 24 lose again;
//  * 16 rows: S = 8 (down 53.1 -> 26.7, q|k|v 23.7 -> 17.1), except where
//    the tiles x chunks per block pass ~100 (gate/up: S = 4, 50.9 -> 46.9);
//  * 64 rows (8 row groups of 19 SMs): the combine's reads grow with the
//    rows and a K = 4096 activation chunk frees little shared memory:
//    gate/up and o best at S = 1, q|k|v at 2, down at 2 (Int8Act, 139.6 ->
//    87.7) to 8 (TwoPass, 406.6 -> 110.9).
// With 1 KB slices for split launches (the tensor-core layout's first choice
// there), S = 4 then beat S = 8 at 8 rows: q|k|v 11.0 -> 9.4 us, gate/up
// 26.3 -> 25.0, down 16.9 -> 16.4 (Int8Act); TwoPass down 19.6 -> 18.7.
// Rule: S = 4 for one and two row groups; halved while the work units
// (tiles x S) pass 100 per block of a row group; past 16 rows also at most
// the activation bytes a block holds over 24 KB (a power of two).
int lk_splitk_chunks_for(int N, int K, lk_mode mode, int M) {
  if ((mode != LK_INT8ACT && mode != LK_TWOPASS) || M < 2 || M > LK_MAX_BATCH || N < 1 || K < 256 || K % 256)
    return 1;
  const DeviceInfo* d = device_info(nullptr);
  if (!d) return 1;
  const long tiles = ((long)N + 15) / 16;
  const int groups = (M + LK_MAX_M - 1) / LK_MAX_M;
  const long blocks = d->sm_count / groups > 0 ? d->sm_count / groups : 1;
  int S = 4;
  while (S > 1 && (tiles * S > 100 * blocks || K / 128 < S)) S >>= 1;
  if (M > 2 * LK_MAX_M) {
    const long act = (long)LK_MAX_M * K * (mode == LK_TWOPASS ? 2 : 1);
    while (S > 1 && act / S < 24 * 1024) S >>= 1;
  }
  return S > 1 && lk_gemv_kernel_for(N, K, mode, M, S, nullptr) == 3 ? S : 1;
}

size_t lk_splitk_workspace_bytes(lk_mode mode, int S, int M, int N) {
  if (S < 1 || M < 0 || N < 0) return 0;
  return (size_t)S * (size_t)M * (size_t)N * (mode == LK_DEQUANT ? 8 : 4);
}

lk_status lk_gemv_q8_splitk(const int8_t* wq, const uint16_t* ws, int N, int K, lk_mode mode,
                            const float* x, const int8_t* xq, const int8_t* xl, const float* xs, int M,
                            int S, void* part, size_t part_bytes, const lk_launch_cfg* cfg,
                            cudaStream_t stream) {
  lk_status st = check_common(wq, ws, N, K, mode, x, xq, xl, xs, M);
  if (st) return st;
  st = check_launch_cfg(cfg);
  if (st) return st;
  if (S < 1 || S > LK_MAX_SPLITK) return LK_ERR_SHAPE;
  if (N == 0 || M == 0) return LK_OK;
  if (!part) return LK_ERR_ARG;
  if (!aligned(part, mode == LK_DEQUANT ? 8 : 4)) return LK_ERR_ALIGN;
  if (part_bytes < lk_splitk_workspace_bytes(mode, S, M, N)) return LK_ERR_WORKSPACE;
  GemvProblem p = make_problem(wq, ws, N, K, mode, x, xq, xl, xs, M);
  apply_cfg(p, cfg);
  p.S = S;
  p.split = true;
  if (mode == LK_DEQUANT) p.part64 = (double*)part;
  else p.y = (float*)part;
  const int path = p.cfg.path;
  // 2.. LK_MAX_BATCH rows: the tensor-core kernel (past 8 rows the only one)
  if ((path == 0 || path == 3) && mma_supports(p)) return mma_gemv(p, stream, nullptr);
  if (path == 3 || M > LK_MAX_M) return LK_ERR_SHAPE;
  if (path != 1 && ring_supports(p)) return ring_gemv(p, stream, nullptr);
  if (path == 2) return LK_ERR_SHAPE;
  const long blocks = (p.N + kRowsPerBlock - 1) / kRowsPerBlock;
  kernel_fn f = pick(p.mode, p.M, true);
  f<<<dim3((unsigned)blocks, S), kWarps * 32, 0, stream>>>(p);
  return launch_status();
}

lk_status lk_splitk_combine(lk_mode mode, const void* part, int S, int M, int N, float* y,
                            const lk_launch_cfg* cfg, cudaStream_t stream) {
  if (mode < LK_DEQUANT || mode > LK_TWOPASS || check_launch_cfg(cfg)) return LK_ERR_ARG;
  if (S < 1 || S > LK_MAX_SPLITK || M < 0 || M > LK_MAX_BATCH || N < 0) return LK_ERR_SHAPE;
  if (N == 0 || M == 0) return LK_OK;
  if (!part || !y) return LK_ERR_ARG;
  if (!aligned(part, mode == LK_DEQUANT ? 8 : 4) || !aligned(y, 4)) return LK_ERR_ALIGN;
  const long MN = (long)M * N;
  const long blocks = (MN + 255) / 256;
  if (mode == LK_DEQUANT)
    launch_pdl(splitk_combine_kernel<true>, dim3((unsigned)blocks), dim3(256), stream, cfg_pdl(cfg), part, S, MN, y,
               tr_ptr(), tr_slot());
  else
    launch_pdl(splitk_combine_kernel<false>, dim3((unsigned)blocks), dim3(256), stream, cfg_pdl(cfg), part, S, MN, y,
               tr_ptr(), tr_slot());
  return launch_status();
}

}  // extern "C"
