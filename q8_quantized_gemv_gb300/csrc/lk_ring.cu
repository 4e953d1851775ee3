// Bulk-copy ring GEMV for sm_103a, and the device-side error word that every
// bounded wait sets when it gives up.
//
// One block per SM, persistent over a contiguous, balanced range of rows
// [r0, r1) (and one split-K chunk).  Warp 8 is the producer: it streams the
// rows' weights tile by tile (32 rows) and slice by slice (up to 1 KB of K)
// into a ring of shared-memory stages with 1-D bulk copies (TMA,
// cp.async.bulk ... mbarrier::complete_tx::bytes), one copy per row for the
// int8 levels and one for the row's f16 scales, plus the slice of the
// activation (words and scales) that every row of the tile shares.  Each
// stage has a "full" mbarrier (the producer's expect-tx arrival plus the
// copies' byte count) and an "empty" mbarrier (one arrival per consumer
// warp).  Warps 0..7 consume: warp w owns rows 4w..4w+3 of the tile with the
// same lane arrangement and the same per-block arithmetic as the direct
// kernel (8 lanes per row, lane j reading bytes 16j..16j+15 of each 128-byte
// segment, partial q = b mod 4 chained in ascending block order, then
// (p0 + p2) + (p1 + p3)), so both kernels give the same bits.
//
// Every wait on an mbarrier is bounded by a wall-clock limit (%globaltimer).
// A wait that runs out sets the error word and an abort flag in shared
// memory; every thread then leaves its loop, and the producer, before it
// exits, waits (again bounded) for the copies it issued so that no copy is
// still in flight into the block's shared memory when the block ends.
#include "lk_device.cuh"
#include "lk_host.h"

__device__ int lk_error_word;

namespace {

using namespace lk;

constexpr int NWC = 8;                 // consumer warps
constexpr int TR = 4 * NWC;            // rows per tile
constexpr int TK = 1024;               // bytes of K per stage slice (max)
constexpr int SROW = TK / 16 + 16;     // a row's slice of scales plus 16-byte alignment slack
constexpr int THREADS = (NWC + 1) * 32;
constexpr int MAX_STAGES = 8;

enum : int { ERR_WAIT_FULL = 1, ERR_WAIT_EMPTY = 2, ERR_DRAIN = 4, ERR_SELFTEST = 8 };

struct RingArgs {
  lkh::GemvProblem p;
  int stages;
  int gx;                  // blocks along the rows
  unsigned stage_bytes;
  unsigned s_off, x_off;   // scale and activation regions inside a stage
  unsigned long long wait_ns;
};

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
// Bounded wait for the phase of parity `parity` to complete.  Returns false if
// the limit ran out or another thread raised the abort flag.
__device__ __forceinline__ bool mbar_wait(unsigned bar, unsigned parity, unsigned long long limit_ns,
                                          volatile int* abort_flag) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  for (;;) {
    if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (gtimer() - t0 > limit_ns) return false;
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

__device__ __forceinline__ void raise_error(int code, volatile int* abort_flag) {
  atomicOr(&lk_error_word, code);
  *abort_flag = 1;
}

template <int Q>
struct part_t { typedef float t; };
template <>
struct part_t<0> { typedef double t; };

// Bytes of one stage's activation slice of `len` bytes of K.
template <int Q, int M>
__host__ __device__ constexpr unsigned act_bytes(unsigned len) {
  return Q == 0 ? M * len * 4u : M * len * (Q == 2 ? 2u : 1u) + M * len / 8u;
}

template <int Q, int M, bool SPLIT>
__global__ void __launch_bounds__(THREADS, 1) gemv_ring_kernel(const RingArgs ra) {
  typedef typename part_t<Q>::t P;
  extern __shared__ __align__(128) unsigned char smem[];
  const lkh::GemvProblem& a = ra.p;
  const int NS = ra.stages;
  unsigned char* ring = smem;
  unsigned long long* bars = (unsigned long long*)(smem + (size_t)NS * ra.stage_bytes);
  volatile int* abort_flag = (volatile int*)(bars + 2 * MAX_STAGES);
  unsigned long long* keys = (unsigned long long*)(bars + 2 * MAX_STAGES + 1);  // [M][NWC]
  const unsigned full0 = smem_u32(bars), empty0 = smem_u32(bars + MAX_STAGES);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.K, nb = K >> 5;
  const long N = a.N;
  const long r0 = (long)blockIdx.x * N / ra.gx, r1 = (long)(blockIdx.x + 1) * N / ra.gx;
  int b_lo = 0, b_hi = nb;
  if (SPLIT) {
    b_lo = splitk_bound(nb, a.S, blockIdx.y);
    b_hi = splitk_bound(nb, a.S, blockIdx.y + 1);
  }
  const int k_lo = 32 * b_lo, k_hi = 32 * b_hi;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, NWC);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == NWC) {
    // ------------------------------------------------------------------ producer
    const unsigned long long pol_w = evict_first_policy(), pol_a = evict_last_policy();
    int it = 0;
    bool ok = true;
    for (long t0 = r0; ok && t0 < r1; t0 += TR) {
      const int rows = (int)(r1 - t0 < TR ? r1 - t0 : TR);
      for (int k0 = k_lo; k0 < k_hi; k0 += TK) {
        const int len = (k_hi - k0 < TK) ? k_hi - k0 : TK;
        const int slot = it % NS;
        const unsigned ph = (unsigned)(it / NS) & 1u;
        // every lane waits; the outcome is made warp-uniform before anyone acts on it
        if (!__all_sync(FULL, mbar_wait(empty0 + 8 * slot, ph ^ 1u, ra.wait_ns, abort_flag))) {
          if (lane == 0) raise_error(ERR_WAIT_EMPTY, abort_flag);
          ok = false;
          break;
        }
        const int b0 = k0 >> 5, b1 = b0 + (len >> 5);
        const unsigned sh = (unsigned)(b0 & 7) * 2u;               // scales' offset in the first 16 B
        const unsigned slen = ((b1 - b0) * 2u + sh + 15u) & ~15u;  // 16-byte superset of the scales
        const unsigned full = full0 + 8 * slot;
        if (lane == 0) mbar_arrive_expect_tx(full, (unsigned)rows * (len + slen) + act_bytes<Q, M>(len));
        __syncwarp();
        unsigned char* st = ring + (size_t)slot * ra.stage_bytes;
        if (lane < rows) {
          const long row = t0 + lane;
          bulk_g2s(st + lane * TK, a.wq + row * K + k0, len, full, pol_w);
          bulk_g2s(st + ra.s_off + lane * SROW,
                   (const unsigned char*)a.ws + ((row * nb + b0) * 2 - sh), slen, full, pol_w);
        }
        unsigned char* X = st + ra.x_off;
        if (Q == 0) {
          if (lane < M) bulk_g2s(X + lane * TK * 4, a.x + (long)lane * K + k0, len * 4, full, pol_a);
        } else {
          if (lane < M) bulk_g2s(X + lane * TK, a.xq + (long)lane * K + k0, len, full, pol_a);
          if (Q == 2 && lane >= 8 && lane < 8 + M)
            bulk_g2s(X + M * TK + (lane - 8) * TK, a.xl + (long)(lane - 8) * K + k0, len, full, pol_a);
          if (lane >= 16 && lane < 16 + M) {
            const int t = lane - 16;
            bulk_g2s(X + M * TK * (Q == 2 ? 2 : 1) + t * (TK / 8), a.xs + (long)t * nb + b0, len / 8, full,
                     pol_a);
          }
        }
        ++it;
      }
    }
    // Drain: the copies of the last (up to NS) issued stages must have landed
    // before this warp may let the block end.
    if (lane == 0) {
      const int first = it > NS ? it - NS : 0;
      for (int i = first; i < it; ++i) {
        if (!mbar_wait(full0 + 8 * (i % NS), (unsigned)(i / NS) & 1u, ra.wait_ns, abort_flag)) {
          // on abort the flag is set: wait once more, bounded, ignoring it
          const unsigned long long t0 = gtimer();
          while (!mbar_try(full0 + 8 * (i % NS), (unsigned)(i / NS) & 1u)) {
            if (gtimer() - t0 > ra.wait_ns) {
              atomicOr(&lk_error_word, ERR_DRAIN);
              break;
            }
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ consumers
    const int rr = lane >> 3, j = lane & 7, q = j >> 1, hf = j & 1;
    const int lrow = warp * 4 + rr;
    P p[M];
    unsigned long long best[M];
#pragma unroll
    for (int t = 0; t < M; ++t) {
      p[t] = (P)0;
      best[t] = 0;
    }
    int it = 0;
    bool ok = true;
    for (long t0 = r0; ok && t0 < r1; t0 += TR) {
      const int rows = (int)(r1 - t0 < TR ? r1 - t0 : TR);
      const bool row_ok = lrow < rows;
      for (int k0 = k_lo; k0 < k_hi; k0 += TK) {
        const int len = (k_hi - k0 < TK) ? k_hi - k0 : TK;
        const int slot = it % NS;
        const unsigned ph = (unsigned)(it / NS) & 1u;
        if (!__all_sync(FULL, mbar_wait(full0 + 8 * slot, ph, ra.wait_ns, abort_flag))) {
          if (lane == 0) raise_error(ERR_WAIT_FULL, abort_flag);
          ok = false;
          break;
        }
        const unsigned char* st = ring + (size_t)slot * ra.stage_bytes;
        const int b0 = k0 >> 5;
        const unsigned sh = (unsigned)(b0 & 7) * 2u;
        const unsigned char* Wr = st + lrow * TK + 16 * j;
        const unsigned char* Sr = st + ra.s_off + lrow * SROW + sh + 2 * q;
        const unsigned char* X = st + ra.x_off;
        const int nseg = len >> 7;
        for (int seg = 0; seg < nseg; ++seg) {
          const int4 w = *(const int4*)(Wr + 128 * seg);
          const float wsc = __half2float(*(const __half*)(Sr + 8 * seg));
#pragma unroll
          for (int t = 0; t < M; ++t) {
            if constexpr (Q == 0) {
              const float4* xv = (const float4*)(X + (size_t)t * TK * 4 + (128 * seg + 16 * j) * 4);
              const int wi[4] = {w.x, w.y, w.z, w.w};
              float h = 0.f;
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const float4 xx = xv[c];
                const float xe[4] = {xx.x, xx.y, xx.z, xx.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) h = __fmaf_rn((float)(int8_t)(wi[c] >> (8 * k)), xe[k], h);
              }
              const float blk = __fadd_rn(h, __shfl_xor_sync(FULL, h, 1));
              p[t] = __fma_rn((double)wsc, (double)blk, (double)p[t]);
            } else {
              const int4 hv = *(const int4*)(X + t * TK + 128 * seg + 16 * j);
              int d = dot16(w, hv);
              d += __shfl_xor_sync(FULL, d, 1);
              int e = 0;
              if constexpr (Q == 2) {
                const int4 lv = *(const int4*)(X + M * TK + t * TK + 128 * seg + 16 * j);
                e = dot16(w, lv);
                e += __shfl_xor_sync(FULL, e, 1);
              }
              const float s = *(const float*)(X + M * TK * (Q == 2 ? 2 : 1) + t * (TK / 8) + 4 * (4 * seg + q));
              p[t] = q8_step<Q>((float)p[t], wsc, s, d, e);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);
        ++it;
      }
      if (!ok) break;
      // tile done: (p0 + p2) + (p1 + p3) within each row's 8 lanes
#pragma unroll
      for (int t = 0; t < M; ++t) {
        P v = p[t];
        v = v + __shfl_down_sync(FULL, v, 4);
        v = v + __shfl_down_sync(FULL, v, 2);
        p[t] = (P)0;
        if (j == 0 && row_ok) {
          const long o = t0 + lrow;
          if (SPLIT) {
            const long idx = ((long)blockIdx.y * M + t) * N + o;
            if constexpr (Q == 0) a.part64[idx] = (double)v;
            else a.y[idx] = (float)v;
          } else {
            const float yv = Q == 0 ? __double2float_rn((double)v) : (float)v;
            a.y[(long)t * N + o] = yv;
            const unsigned long long k = amax_key(yv, (unsigned)o);
            best[t] = k > best[t] ? k : best[t];
          }
        }
      }
    }
    if (!SPLIT && a.amax) {
#pragma unroll
      for (int t = 0; t < M; ++t) {
        const unsigned long long wmax = warp_max_u64(best[t]);
        if (lane == 0) keys[t * NWC + warp] = wmax;
      }
    }
  }
  if (!SPLIT && a.amax) {
    __syncthreads();
    if (threadIdx.x < M) {
      unsigned long long m = 0;
      for (int w = 0; w < NWC; ++w) m = keys[threadIdx.x * NWC + w] > m ? keys[threadIdx.x * NWC + w] : m;
      a.amax[(long)threadIdx.x * gridDim.x + blockIdx.x] = m;
    }
  }
}

// A wait on an mbarrier that nothing completes: the bounded wait must give
// up after `limit_ns`, raise the error word and return.
__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (!mbar_wait(smem_u32(&bar), 0, limit_ns, &abort_flag)) {
    if (threadIdx.x == 0) atomicOr(&lk_error_word, ERR_SELFTEST);
  }
}

typedef void (*ring_fn)(const RingArgs);

template <int Q, bool SPLIT>
ring_fn pick_m(int M) {
  switch (M) {
    case 1: return gemv_ring_kernel<Q, 1, SPLIT>;
    case 2: return gemv_ring_kernel<Q, 2, SPLIT>;
    case 3: return gemv_ring_kernel<Q, 3, SPLIT>;
    case 4: return gemv_ring_kernel<Q, 4, SPLIT>;
    case 5: return gemv_ring_kernel<Q, 5, SPLIT>;
    case 6: return gemv_ring_kernel<Q, 6, SPLIT>;
    case 7: return gemv_ring_kernel<Q, 7, SPLIT>;
    default: return gemv_ring_kernel<Q, 8, SPLIT>;
  }
}

ring_fn pick(int mode, int M, bool split) {
  if (split) return mode == 0 ? pick_m<0, true>(M) : mode == 1 ? pick_m<1, true>(M) : pick_m<2, true>(M);
  return mode == 0 ? pick_m<0, false>(M) : mode == 1 ? pick_m<1, false>(M) : pick_m<2, false>(M);
}

unsigned act_bytes_rt(int mode, int M, unsigned len) {
  return mode == 0 ? M * len * 4u : M * len * (mode == 2 ? 2u : 1u) + M * len / 8u;
}

struct Layout {
  unsigned stage_bytes, s_off, x_off, total;
  int stages;
};

Layout layout(int mode, int M, int smem_optin) {
  Layout L;
  L.s_off = TR * TK;
  L.x_off = L.s_off + TR * SROW;
  L.stage_bytes = (L.x_off + act_bytes_rt(mode, M, TK) + 127u) & ~127u;
  const unsigned tail = 8 * 2 * MAX_STAGES + 16 + 8 * LK_MAX_M * NWC;
  int ns = (int)((smem_optin - tail) / L.stage_bytes);
  if (ns > MAX_STAGES) ns = MAX_STAGES;
  if (lkh::opt_ring_stages > 0 && lkh::opt_ring_stages < ns) ns = (int)lkh::opt_ring_stages;
  L.stages = ns;
  L.total = ns * L.stage_bytes + tail;
  return L;
}

}  // namespace

namespace lkh {

bool ring_supports(const GemvProblem& p) {
  if (p.K < 256 || p.K % 256 || p.N < 1 || p.M < 1 || p.M > LK_MAX_M) return false;
  if (!aligned(p.ws, 16)) return false;
  if (p.mode == 0 ? !aligned(p.x, 16)
                  : (!aligned(p.xq, 16) || !aligned(p.xs, 16) || (p.mode == 2 && !aligned(p.xl, 16))))
    return false;
  const DeviceInfo* d = device_info(nullptr);
  if (!d) return false;
  return layout(p.mode, p.M, d->smem_optin).stages >= 2;
}

int ring_max_ctas(long) {
  const DeviceInfo* d = device_info(nullptr);
  long g = d ? d->sm_count : 1024;
  if (opt_grid_ctas > g) g = opt_grid_ctas;
  return (int)g;
}

lk_status ring_gemv(const GemvProblem& p, cudaStream_t stream, int* n_parts) {
  const DeviceInfo* d = device_info(nullptr);
  if (!d) return LK_ERR_CUDA;
  const Layout L = layout(p.mode, p.M, d->smem_optin);
  if (L.stages < 2) return LK_ERR_SHAPE;
  ring_fn f = pick(p.mode, p.M, p.split);
  // opt in to the large dynamic shared memory once per (kernel, device)
  // (cheap and idempotent: set on every launch rather than cached per device)
  if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total) != cudaSuccess)
    return LK_ERR_CUDA;
  RingArgs ra;
  ra.p = p;
  ra.stages = L.stages;
  ra.stage_bytes = L.stage_bytes;
  ra.s_off = L.s_off;
  ra.x_off = L.x_off;
  ra.wait_ns = opt_wait_us > 0 ? (unsigned long long)opt_wait_us * 1000ull : 2000000000ull;
  int S = p.S > 1 ? p.S : 1;
  int g = opt_grid_ctas > 0 ? (int)opt_grid_ctas : d->sm_count;
  int gx = (g + S - 1) / S;
  if (gx < 1) gx = 1;
  ra.gx = gx;
  f<<<dim3(gx, S), THREADS, L.total, stream>>>(ra);
  if (n_parts) *n_parts = gx;
  return launch_status();
}

}  // namespace lkh

extern "C" lk_status lk_device_error(int reset, int* code) {
  if (cudaDeviceSynchronize() != cudaSuccess) return LK_ERR_CUDA;
  int w = 0;
  if (cudaMemcpyFromSymbol(&w, lk_error_word, sizeof(int)) != cudaSuccess) return LK_ERR_CUDA;
  if (code) *code = w;
  if (reset && w) {
    const int z = 0;
    if (cudaMemcpyToSymbol(lk_error_word, &z, sizeof(int)) != cudaSuccess) return LK_ERR_CUDA;
  }
  return w ? LK_ERR_DEVICE_TIMEOUT : LK_OK;
}

extern "C" lk_status lk_selftest_wait_timeout(unsigned limit_us, cudaStream_t stream) {
  if (limit_us == 0 || limit_us > 10000000u) return LK_ERR_ARG;
  wait_selftest_kernel<<<1, 32, 0, stream>>>((unsigned long long)limit_us * 1000ull);
  return lkh::launch_status();
}
