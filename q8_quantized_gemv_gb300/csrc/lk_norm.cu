// RMSNorm -> activation quantizer, with an optional residual add in front
// ("kernels.rs" RMSNORM lk_rmsnorm_row with ADD / SUM; QWEN38_EXTRA_KERNELS
// gk_add_rmsnorm_q8_hl), and the SwiGLU -> quantizer step between a decoder's
// gate/up and down projections ("kernels.rs" GLU lk_gemv_glu, ACT -1;
// QWEN38_EXTRA_KERNELS gk_silu_had_q8).
//
// The norm's sum of squares follows the block of min(roundup32(K), 1024)
// threads of lk_rmsnorm_row: thread t accumulates the squares of values
// t, t + 1024, ... as fused multiply-adds, then a shuffle-down tree per warp
// and over the warps' totals.  Three kernels play that order: one block of
// that many threads per row (any K), K / vt blocks of vt threads per row
// (K a multiple of vt, at most 8 per thread), and K / 1024 blocks of 256
// threads playing the 1024 (K a multiple of 1024) -- every block of a row
// forms the same sum, then normalizes and quantizes only its own values.
#include "lk_device.cuh"
#include "lk_host.h"

using namespace lk;
using namespace lkh;

namespace {

struct NormArgs {
  const float* x;   // [M][K] rows
  const float* r;   // ADD: [M][K] residual added to x before the norm
  float* s;         // ADD, optional: [M][K] the sums x + r (the residual stream)
  const float* g;   // [K] gain
  int K;
  float eps;
  float* xn;        // optional (required under Dequant): [M][K] normed rows
  int8_t* xq;       // quantized modes: [M][K] high words
  int8_t* xl;       // TwoPass: [M][K] low words
  float* xs;        // quantized modes: [M][K/32] scales
  unsigned long long* tr;
  int slot;
};

// The residual sum x + r, stored with an L2 evict-last hint: it is the next
// residual add's r, read back after a GEMV or two whose weights (hundreds of
// MB) stream through L2 meanwhile.
__device__ __forceinline__ void store_keep(float* p, float v) {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}

// Value i of the row the norm sees: x, or x + r rounded once to f32.  Both
// reads go through L2: under a programmatic dependent launch the previous
// kernel may have written them.
template <bool ADD>
__device__ __forceinline__ float row_value(const NormArgs& a, long i) {
  const float v = __ldcg(a.x + i);
  return ADD ? __fadd_rn(v, __ldcg(a.r + i)) : v;
}

// Normalize value v (element i of the [M][K] layout) and store what the mode
// asks for; with ADD also the sum itself.
// The row's divisor and, for an f32 norm, its correctly rounded reciprocal
// (the quotients then take div_row's checked shortcut).
template <typename A>
struct Den {
  A d;
  float r;
};
template <typename A>
__device__ __forceinline__ Den<A> make_den(A d) {
  if constexpr (sizeof(A) == 4) return Den<A>{d, __frcp_rn(d)};
  return Den<A>{d, 0.f};
}

template <int Q, bool ADD, typename A>
__device__ __forceinline__ void finish_value(const NormArgs& a, long i, float v, Den<A> den, float gv, int lane) {
  if (ADD && a.s) store_keep(a.s + i, v);
  float yv;
  if constexpr (sizeof(A) == 4) yv = norm_scale_r(v, den.d, den.r, gv);
  else yv = norm_scale(v, den.d, gv);
  if (a.xn) a.xn[i] = yv;
  if constexpr (Q > 0) quant_lane<Q>(yv, a.xq, a.xl, a.xs, i >> 5, lane);
}

// One block of vt = min(roundup32(K), 1024) threads per row.
template <int Q, bool ADD>
__global__ void __launch_bounds__(1024) rmsnorm_row_kernel(const NormArgs a) {
  typedef typename acc_of<Q>::t A;
  __shared__ A red[32];
  __shared__ A total;
  // a programmatic dependent (a GEMV launched with lk_launch_cfg.pdl) may start its
  // weight stream now; it reads these outputs only after this grid completes.
  // Launched as a dependent itself (pdl), this grid reads its inputs and
  // writes its outputs only after the previous kernel has completed.
  asm volatile("griddepcontrol.launch_dependents;" :::);
  trec_stamp(a.tr, a.slot, TR_START);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  trec_stamp(a.tr, a.slot, TR_WAITED);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.K, vt = blockDim.x, nw = vt >> 5;
  const long base = (long)blockIdx.x * K;
  A acc = 0;
  for (int i = threadIdx.x; i < K; i += vt) acc = fma_acc((A)row_value<ADD>(a, base + i), acc);
  acc = warp_tree_sum(acc);
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  if (warp == 0) {
    A v = lane < nw ? red[lane] : (A)0;
    v = warp_tree_sum(v);
    if (lane == 0) total = v;
  }
  __syncthreads();
  const Den<A> den = make_den<A>(norm_div_add(total, K, a.eps));
  // warp w holds the 32-groups starting at 32w, 32w + vt, ... (vt % 32 == 0)
  for (int b = warp * 32; b < K; b += vt)
    finish_value<Q, ADD>(a, base + b + lane, row_value<ADD>(a, base + b + lane), den, __ldg(a.g + b + lane), lane);
  trec_end(a.tr, a.slot, TK_NORM, K);
}

// K / vt blocks of vt threads per row (K a multiple of vt, K / vt <= 8):
// thread t of every block loads the row's values t + vt*u once and forms the
// sum in rmsnorm_row_kernel's order; block y finishes the values t + vt*y.
template <int Q, bool ADD>
__global__ void __launch_bounds__(1024) rmsnorm_split_kernel(const NormArgs a) {
  typedef typename acc_of<Q>::t A;
  constexpr int KU_MAX = 8;
  __shared__ A red[32];
  __shared__ A total;
  asm volatile("griddepcontrol.launch_dependents;" :::);  // as in rmsnorm_row_kernel
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.K, vt = blockDim.x, nw = vt >> 5, KU = K / vt, u_mine = blockIdx.y;
  const long base = (long)blockIdx.x * K;
  const float gv = __ldg(a.g + threadIdx.x + vt * u_mine);  // independent of the previous kernel
  trec_stamp(a.tr, a.slot, TR_START);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  trec_stamp(a.tr, a.slot, TR_WAITED);
  float v[KU_MAX];
#pragma unroll
  for (int u = 0; u < KU_MAX; ++u) v[u] = u < KU ? row_value<ADD>(a, base + threadIdx.x + vt * u) : 0.f;
  A acc = 0;
#pragma unroll
  for (int u = 0; u < KU_MAX; ++u)
    if (u < KU) acc = fma_acc((A)v[u], acc);
  acc = warp_tree_sum(acc);
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  if (warp == 0) {
    A t = lane < nw ? red[lane] : (A)0;
    t = warp_tree_sum(t);
    if (lane == 0) total = t;
  }
  __syncthreads();
  const Den<A> den = make_den<A>(norm_div_add(total, K, a.eps));
  float mine = v[0];
#pragma unroll
  for (int u = 1; u < KU_MAX; ++u)
    if (u == u_mine) mine = v[u];
  finish_value<Q, ADD>(a, base + threadIdx.x + (long)vt * u_mine, mine, den, gv, lane);
  trec_end(a.tr, a.slot, TK_NORM, K);
}

// K / 1024 blocks of 256 threads per row (K a multiple of 1024, at most
// 8192): warp w plays the norm's warps w, w + 8, w + 16, w + 24, so a block
// needs few registers and can share an SM with a GEMV block of the
// neighbouring launches (a 1024-thread block cannot).  Under Dequant the
// f64 division per value (GB300's FP64 pipe is narrow) is spread further:
// JS = 4 blocks per 1024 values, each finishing one virtual warp per real
// warp (blockIdx.y = 4 u + j).
template <int Q, bool ADD>
__global__ void __launch_bounds__(256) rmsnorm_split256_kernel(const NormArgs a) {
  typedef typename acc_of<Q>::t A;
  constexpr int KU_MAX = 8, VT = 1024, NJ = 4;  // virtual warps per real warp
  constexpr int JS = Q == 0 ? 4 : 1;            // blocks per 1024 values
  __shared__ A red[32];
  __shared__ A total;
  asm volatile("griddepcontrol.launch_dependents;" :::);  // as in rmsnorm_row_kernel
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.K, KU = K / VT, u_mine = blockIdx.y / JS, j_mine = blockIdx.y % JS;
  const long base = (long)blockIdx.x * K;
  float gv[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) gv[j] = __ldg(a.g + 32 * (warp + 8 * j) + lane + VT * u_mine);
  trec_stamp(a.tr, a.slot, TR_START);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  trec_stamp(a.tr, a.slot, TR_WAITED);
  float v[NJ][KU_MAX];
#pragma unroll
  for (int j = 0; j < NJ; ++j)
#pragma unroll
    for (int u = 0; u < KU_MAX; ++u)
      v[j][u] = u < KU ? row_value<ADD>(a, base + 32 * (warp + 8 * j) + lane + VT * u) : 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    A acc = 0;
#pragma unroll
    for (int u = 0; u < KU_MAX; ++u)
      if (u < KU) acc = fma_acc((A)v[j][u], acc);
    acc = warp_tree_sum(acc);
    if (lane == 0) red[warp + 8 * j] = acc;
  }
  __syncthreads();
  if (warp == 0) {
    A t = red[lane];
    t = warp_tree_sum(t);
    if (lane == 0) total = t;
  }
  __syncthreads();
  const Den<A> den = make_den<A>(norm_div_add(total, K, a.eps));
  // this block's values: groups g0 + 8 j of the [M][K] layout, normalized,
  // then quantized four groups at a time (their chains interleave)
  const long i0 = base + (long)VT * u_mine + 32 * warp + lane;
  float yv[NJ];
  bool ok[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    if (JS > 1 && j % JS != j_mine) continue;
    float mine = v[j][0];
#pragma unroll
    for (int u = 1; u < KU_MAX; ++u)
      if (u == u_mine) mine = v[j][u];
    const long i = i0 + 256 * j;
    if (ADD && a.s) store_keep(a.s + i, mine);
    if constexpr (sizeof(A) == 4) yv[j] = norm_scale_r(mine, den.d, den.r, gv[j]);
    else yv[j] = norm_scale(mine, den.d, gv[j]);
    if (a.xn) a.xn[i] = yv[j];
    ok[j] = true;
  }
  if constexpr (Q > 0) quant_groups<Q, NJ>(yv, ok, a.xq, a.xl, a.xs, i0 >> 5, 8, lane);
  trec_end(a.tr, a.slot, TK_NORM, K);
}

template <int Q, bool ADD>
void launch_norm(const NormArgs& a, int M, int pdl, cudaStream_t stream) {
  const int K = a.K, vt = K < 1024 ? K : 1024;  // K % 32 == 0: roundup32(K) == K
  if (K % 1024 == 0 && K / 1024 <= 8)
    launch_pdl(rmsnorm_split256_kernel<Q, ADD>, dim3(M, K / 1024 * (Q == 0 ? 4 : 1)), dim3(256), stream, pdl, a);
  else if (K % vt == 0 && K / vt <= 8)
    launch_pdl(rmsnorm_split_kernel<Q, ADD>, dim3(M, K / vt), dim3(vt), stream, pdl, a);
  else
    launch_pdl(rmsnorm_row_kernel<Q, ADD>, dim3(M), dim3(vt), stream, pdl, a);
}

template <bool ADD>
lk_status norm_entry(const NormArgs& a, int M, lk_mode mode, int pdl, cudaStream_t stream) {
  if (mode == LK_DEQUANT) {
    if (!a.xn) return LK_ERR_ARG;
    launch_norm<0, ADD>(a, M, pdl, stream);
  } else {
    const lk_status st = check_act_out(mode, a.xq, a.xl, a.xs);
    if (st) return st;
    if (mode == LK_INT8ACT) launch_norm<1, ADD>(a, M, pdl, stream);
    else launch_norm<2, ADD>(a, M, pdl, stream);
  }
  return launch_status();
}

NormArgs norm_args(const float* x, const float* r, float* s, const float* g, int K, float eps, lk_mode mode,
                   float* xn, int8_t* xq, int8_t* xl, float* xs) {
  NormArgs a;
  a.x = x;
  a.r = r;
  a.s = s;
  a.g = g;
  a.K = K;
  a.eps = eps;
  a.xn = xn;
  a.xq = mode == LK_DEQUANT ? nullptr : xq;
  a.xl = mode == LK_TWOPASS ? xl : nullptr;
  a.xs = mode == LK_DEQUANT ? nullptr : xs;
  a.tr = tr_ptr();
  a.slot = tr_slot();
  return a;
}

// [p, p + n) and [q, q + n) floats overlap.
bool overlap(const float* p, const float* q, long n) { return p < q + n && q < p + n; }

// SwiGLU of one 32-group per warp: lane l takes value 32 j + l of row t,
// h = (g / (1 + expf(-g))) * u with each operation rounded as written
// ("kernels.rs" lk_gemv_glu, ACT -1), stored as f32 and/or quantized.
template <int Q>
__global__ void __launch_bounds__(256) swiglu_quant_kernel(const float* __restrict__ gate, const float* __restrict__ up,
                                                           long ld, int F, long groups, float* __restrict__ h,
                                                           int8_t* __restrict__ hq, int8_t* __restrict__ hl,
                                                           float* __restrict__ hs, unsigned long long* tr, int slot) {
  asm volatile("griddepcontrol.launch_dependents;" :::);  // as in rmsnorm_row_kernel
  trec_stamp(tr, slot, TR_START);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  trec_stamp(tr, slot, TR_WAITED);
  const long G = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (G < groups) {  // whole warps
    const int lane = threadIdx.x & 31, per = F >> 5;
    const long t = G / per, j = G - t * per;
    const long i = t * ld + 32 * j + lane;
    const float gv = __ldcg(gate + i), uv = __ldcg(up + i);
    const float hv = swiglu(gv, uv);
    const long o = t * F + 32 * j + lane;
    if (h) h[o] = hv;
    if constexpr (Q > 0) quant_lane<Q>(hv, hq + t * F, hl ? hl + t * F : nullptr, hs + t * per, j, lane);
  }
  trec_end(tr, slot, TK_QUANT, groups * 32);
}

}  // namespace

extern "C" {

lk_status lk_rmsnorm_quant(const float* x, const float* gain, int M, int K, float eps, lk_mode mode, float* xn,
                           int8_t* xq, int8_t* xl, float* xs, const lk_launch_cfg* cfg, cudaStream_t stream) {
  if (mode < LK_DEQUANT || mode > LK_TWOPASS || check_launch_cfg(cfg)) return LK_ERR_ARG;
  if (M < 0 || M > LK_MAX_BATCH || K < 0 || K % 32) return LK_ERR_SHAPE;
  if (M == 0 || K == 0) return LK_OK;
  if (!x || !gain) return LK_ERR_ARG;
  if (!aligned(x, 4) || !aligned(gain, 4) || (xn && !aligned(xn, 4))) return LK_ERR_ALIGN;
  return norm_entry<false>(norm_args(x, nullptr, nullptr, gain, K, eps, mode, xn, xq, xl, xs), M, mode,
                           cfg_pdl(cfg), stream);
}

lk_status lk_add_rmsnorm_quant(const float* x, const float* r, const float* gain, int M, int K, float eps,
                               lk_mode mode, float* s, float* xn, int8_t* xq, int8_t* xl, float* xs,
                               const lk_launch_cfg* cfg, cudaStream_t stream) {
  if (mode < LK_DEQUANT || mode > LK_TWOPASS || check_launch_cfg(cfg)) return LK_ERR_ARG;
  if (M < 0 || M > LK_MAX_BATCH || K < 0 || K % 32) return LK_ERR_SHAPE;
  if (M == 0 || K == 0) return LK_OK;
  if (!x || !r || !gain) return LK_ERR_ARG;
  if (!aligned(x, 4) || !aligned(r, 4) || !aligned(gain, 4) || (xn && !aligned(xn, 4)) || (s && !aligned(s, 4)))
    return LK_ERR_ALIGN;
  const long n = (long)M * K;
  if (s && (overlap(s, x, n) || overlap(s, r, n))) return LK_ERR_ARG;
  return norm_entry<true>(norm_args(x, r, s, gain, K, eps, mode, xn, xq, xl, xs), M, mode, cfg_pdl(cfg), stream);
}

lk_status lk_swiglu_quant(const float* gate, const float* up, int M, int F, long ld, lk_mode mode, float* h,
                          int8_t* hq, int8_t* hl, float* hs, const lk_launch_cfg* cfg, cudaStream_t stream) {
  if (mode < LK_DEQUANT || mode > LK_TWOPASS || check_launch_cfg(cfg)) return LK_ERR_ARG;
  if (M < 0 || M > LK_MAX_BATCH || F < 0 || F % 32 || ld < F) return LK_ERR_SHAPE;
  if (M == 0 || F == 0) return LK_OK;
  if (!gate || !up) return LK_ERR_ARG;
  if (!aligned(gate, 4) || !aligned(up, 4) || (h && !aligned(h, 4))) return LK_ERR_ALIGN;
  if (mode == LK_DEQUANT && !h) return LK_ERR_ARG;
  if (mode != LK_DEQUANT) {
    const lk_status st = check_act_out(mode, hq, hl, hs);
    if (st) return st;
  }
  const long groups = (long)M * (F / 32);
  const int per_block = 8;
  const dim3 grid((unsigned)((groups + per_block - 1) / per_block)), block(32 * per_block);
  const int pdl = cfg_pdl(cfg);
  if (mode == LK_DEQUANT)
    launch_pdl(swiglu_quant_kernel<0>, grid, block, stream, pdl, gate, up, ld, F, groups, h, (int8_t*)nullptr,
               (int8_t*)nullptr, (float*)nullptr, tr_ptr(), tr_slot());
  else if (mode == LK_INT8ACT)
    launch_pdl(swiglu_quant_kernel<1>, grid, block, stream, pdl, gate, up, ld, F, groups, h, hq, (int8_t*)nullptr, hs,
               tr_ptr(), tr_slot());
  else
    launch_pdl(swiglu_quant_kernel<2>, grid, block, stream, pdl, gate, up, ld, F, groups, h, hq, hl, hs, tr_ptr(),
               tr_slot());
  return launch_status();
}

}  // extern "C"
