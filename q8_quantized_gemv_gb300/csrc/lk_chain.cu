// GEMV chain: a sequence of fused RMSNorm/quantize -> Q8_0 GEMV steps (for
// example one decode token's projections) in ONE cooperative launch.
//
// One block per SM runs every step over its balanced row range, with the
// ring kernel's arrangement (each warp streams and computes its own quads).
// The warps' weight streams run across step boundaries: when a warp frees a
// stage it refills it with its next stage, which may belong to a later step,
// so while the blocks meet at a grid-wide barrier (a step whose input is an
// earlier step's output), the next step's first stages are already in flight.
// This is the GB300 form of the whole-model kernel of model-as-a-kernel
// "megakernel.cu" (phases separated by a grid barrier, the next GEMV's weights
// prefetched during it), restricted to the projection path.
//
// The grid barrier is a counter and a generation word in the caller's sync
// buffer; every wait on it is bounded by a wall-clock limit, after which the
// block raises the error word and an abort flag, drains its copies and exits.
#include "lk_ring_kernel.cuh"

namespace lkring {
namespace {

constexpr int ERR_BARRIER = 32;

struct ChainArgs {
  const lk_chain_op* ops;  // device copy
  int n_ops;
  int nwc, depth;
  unsigned stage_bytes, ring_off;
  float eps;
  unsigned* sync;           // [0] arrivals, [32] generation (separate 128-byte lines)
  unsigned long long wait_ns;
  unsigned long long pol_w;
  int* err;
  unsigned long long* trace;  // block 0's timestamps (option "trace"), or NULL
  int trace_all;              // also every block's and block 0's warps' step ends (trace 2)
  int pdl;                    // launched as a programmatic dependent (a chain without barriers)
  int tslot;                  // trace 3: this launch's record in the timeline, else -1
  int prefill;                // warps that fill their stages before the dependency wait
  // A group of GEMVs over one given activation (lk_gemv_q8_group): the ops
  // are held here (n_inl of them) and the activation rows are copied once
  // instead of computed by a prologue.
  int n_inl;
  lk_chain_op inl[LK_MAX_GROUP];
  const float* gx;            // Dequant: f32 rows [M][K]
  const int8_t* gxq;          // quantized: words, low words, scales
  const int8_t* gxl;
  const float* gxs;
};

// Step i of the chain: from the launch arguments (a group) or the ops array.
__device__ __forceinline__ lk_chain_op chain_op_at(const ChainArgs& ca, int i) {
  if (ca.n_inl) {
    lk_chain_op o = ca.inl[0];
#pragma unroll
    for (int k = 1; k < LK_MAX_GROUP; ++k)
      if (i == k) o = ca.inl[k];
    return o;
  }
  return ca.ops[i];
}

__device__ __forceinline__ void stamp(unsigned long long* trace, int i) {
  if (trace && blockIdx.x == 0 && threadIdx.x == 0 && i < LK_TRACE_MAX) trace[i] = gtimer();
}
// step stamps only in the per-launch modes (trace 1, 2)
#define CHAIN_STAMP(i) \
  if (ca.tslot < 0) stamp(ca.trace, (i))

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void st_relaxed_gpu(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_add_release_gpu(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// All blocks of the grid meet here (bounded).  Writes before it are visible
// to every block after it: the block's threads meet at a CTA barrier, thread
// 0 arrives with an acquire-release add on the counter (its release covers
// the block's writes ordered before it; the last arrival's acquire sees every
// earlier arrival's), the last arrival resets the counter and releases the
// next generation, and the others acquire it.  `gen` is the generation this
// block last saw (read once at kernel start), so an arrival costs one round
// trip.  No full fence is used, so the block's weight copies still in flight
// do not delay it.  Returns false after a timeout or an abort.
__device__ bool grid_sync(unsigned* sync, unsigned& gen, unsigned nblocks, unsigned long long limit_ns, int* err,
                          volatile int* abort_flag) {
  __syncthreads();
  if (threadIdx.x == 0 && !*abort_flag) {
    const unsigned prev = atom_add_acq_rel_gpu(sync, 1u);
    if (prev == nblocks - 1) {
      st_relaxed_gpu(sync, 0u);
      red_add_release_gpu(sync + 32, 1u);
    } else {
      const unsigned long long t0 = gtimer();
      unsigned spins = 0;
      while (ld_acquire_gpu(sync + 32) == gen) {
        if ((++spins & 63u) == 0 && gtimer() - t0 > limit_ns) {
          atomicOr(err, ERR_BARRIER);
          *abort_flag = 1;
          break;
        }
      }
    }
  }
  ++gen;  // every thread keeps the count; only thread 0's is used
  return __syncthreads_or(*abort_flag) == 0;  // the same answer in every thread
}

__device__ __forceinline__ int chain_tk(int K) { return K <= TKMAX ? K : 4096; }

__device__ __forceinline__ int quads_of(const Geom& g) { return (int)((g.r1 - g.r0 + QR - 1) / QR); }

__device__ __forceinline__ Geom op_geom(const lk_chain_op& o) {
  const long N = o.N;
  return make_geom(o.wq, o.ws, N, o.K, (long)blockIdx.x * N / gridDim.x, (long)(blockIdx.x + 1) * N / gridDim.x, 0,
                   o.K, chain_tk(o.K));
}

template <int Q, int M>
__global__ void __launch_bounds__(THREADS_MAX, 1) gemv_chain_kernel(const ChainArgs ca) {
  typedef typename part_t<Q>::t P;
  extern __shared__ __align__(128) unsigned char smem[];
  const int nwc = ca.nwc, D = ca.depth, NS = nwc * D;
  unsigned char* act = smem;
  unsigned char* ring = smem + ca.ring_off;
  unsigned long long* bars = (unsigned long long*)(ring + (size_t)NS * ca.stage_bytes);
  volatile int* abort_flag = (volatile int*)(bars + MAX_STAGES + 1);
  unsigned long long* keys = (unsigned long long*)(bars + MAX_STAGES + 3);  // [M][MAXW]
  double* nred = (double*)(keys + LK_MAX_M * MAXW);                        // [M][32]
  double* nden = nred + LK_MAX_M * 32;                                     // [M]
  const unsigned full0 = smem_u32(bars);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long pol_w = ca.pol_w ? evict_first_policy() : 0ull;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(full0 + 8 * s, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (ca.pdl && threadIdx.x == 0) griddep_launch();

  // The issue cursor walks this warp's stages of every step in order.  A
  // step's quads are dealt to the warps starting where the step before
  // stopped (rotation), so that steps of a few quads each (q, k, v of a
  // layer) spread over all warps instead of piling onto the first ones.
  int iop = 0, irot = 0;
  Geom gi = op_geom(chain_op_at(ca, 0));
  long in = 0, Ti = geom_stages(gi, warp, nwc), issued = 0;
  int ilw = warp;  // this warp's place in the step's deal
  auto issue_next = [&]() {
    while (in >= Ti) {
      if (++iop >= ca.n_ops) return;
      irot = (irot + quads_of(gi)) % nwc;
      gi = op_geom(chain_op_at(ca, iop));
      ilw = (warp - irot + nwc) % nwc;
      Ti = geom_stages(gi, ilw, nwc);
      in = 0;
    }
    const int slot = warp * D + (int)(issued % D);
    issue_stage(gi, ilw, nwc, in, ring + (size_t)slot * ca.stage_bytes, full0 + 8 * slot, pol_w, lane);
    ++in;
    ++issued;
  };
  CHAIN_STAMP(0);
  tstamp(ca.tslot >= 0 ? ca.trace : nullptr, ca.tslot, TR_START);
  // The barrier generation at launch.  No block can complete a barrier of
  // this launch before every block has read it (completion needs every
  // block's arrival, and a block arrives only after this read).
  unsigned gen = threadIdx.x == 0 && ca.sync ? ld_acquire_gpu(ca.sync + 32) : 0u;
  // (warps >= prefill fill their stages after the first step's activation)
  const bool early = warp < ca.prefill;
  for (int d = 0; early && d < D && iop < ca.n_ops; ++d) issue_next();

  // weights above do not depend on the previous kernel; activations do (the
  // first step's prologue waits itself, after requesting its norm gains)
  bool waited = ca.pdl == 0;
  tstamp(ca.tslot >= 0 ? ca.trace : nullptr, ca.tslot, TR_WAITED);
  long consumed = 0;
  int crot = 0;  // the consume side's deal rotation (as irot)
  bool ok = true;
  for (int op = 0; ok && op < ca.n_ops; ++op) {
    const lk_chain_op o = chain_op_at(ca, op);
    if (o.wait && !grid_sync(ca.sync, gen, gridDim.x, ca.wait_ns, ca.err, abort_flag)) {
      ok = false;
      break;
    }
    // the activation area is rewritten below: every warp is done with the last
    // step (a group keeps one activation: its warps run on through the steps)
    if (!ca.n_inl) __syncthreads();
    CHAIN_STAMP(1 + 3 * op);
    // a step that reads the same rows with the same gain as the one before it
    // (q, k and v of a layer) reuses the activation area as it is
    const lk_chain_op prev = chain_op_at(ca, op > 0 ? op - 1 : 0);
    const bool same = op > 0 && !o.wait && o.x == prev.x && o.gain == prev.gain && o.K == prev.K;
    if (ca.n_inl) {
      // a group: one load of the given activation rows, used by every step
      if (op == 0) {
        tstamp(ca.tslot >= 0 ? ca.trace : nullptr, ca.tslot, TR_ISSUED);
        if (!waited) griddep_wait();
        waited = true;
        tstamp(ca.tslot >= 0 ? ca.trace : nullptr, ca.tslot, TR_WAITED);
        lkh::GemvProblem pa;
        pa.K = o.K;
        pa.x = ca.gx;
        pa.xq = ca.gxq;
        pa.xl = ca.gxl;
        pa.xs = ca.gxs;
        load_act<Q, M, 2>(act, (unsigned)o.K, pa, 0);
      }
    } else if (!same) {
      lkh::GemvProblem pr;
      pr.K = o.K;
      pr.xraw = o.x;
      pr.gain = o.gain;
      pr.eps = ca.eps;
      fused_prologue<Q, M>(pr, nwc, 0, (unsigned)o.K, act, nred, nden, nullptr, !waited);
      waited = true;
    }
    CHAIN_STAMP(2 + 3 * op);
    if (op == 0) {
      tstamp(ca.tslot >= 0 ? ca.trace : nullptr, ca.tslot, TR_ACT);
      for (int d = 0; !early && d < D && iop < ca.n_ops; ++d) issue_next();
    }
    const Geom g = op_geom(o);
    const int lw = (warp - crot + nwc) % nwc;  // as the issue cursor dealt this step
    crot = (crot + quads_of(g)) % nwc;
    const long T = geom_stages(g, lw, nwc);
    const Act ac{act, (unsigned)o.K};
    unsigned long long best[M];
    P p[M];
#pragma unroll
    for (int t = 0; t < M; ++t) {
      best[t] = 0;
      p[t] = (P)0;
    }
    for (long n = 0; n < T; ++n) {
      const int slot = warp * D + (int)(consumed % D);
      if (!__all_sync(FULL, mbar_wait(full0 + 8 * slot, (unsigned)(consumed / D) & 1u, ca.wait_ns, abort_flag))) {
        if (lane == 0) raise_error(ca.err, ERR_WAIT_FULL, abort_flag);
        ok = false;
        break;
      }
      unsigned char* st = ring + (size_t)slot * ca.stage_bytes;
      // trace 2: block 0's warps' first stage of each step: data there, computed
      const bool tr2 = ca.trace && ca.trace_all && ca.tslot < 0 && n == 0 && blockIdx.x == 0 && lane == 0 &&
                       2048 + 2 * ((long)op * nwc + warp) + 1 < LK_TRACE_MAX;
      if (tr2) ca.trace[2048 + 2 * ((long)op * nwc + warp)] = gtimer();
      compute_stage<Q, M>(p, g, n, st, ac, lane);
      if (tr2) ca.trace[2048 + 2 * ((long)op * nwc + warp) + 1] = gtimer();
      __syncwarp();
      ++consumed;
      if (iop < ca.n_ops) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue_next();
      }
      if ((int)(n % g.nsl) == g.nsl - 1) {
        lkh::GemvProblem dummy;
        finish_quad<Q, M, false>(p, g, lw, nwc, n, dummy, 0, o.y, best, lane);
      }
    }
    if (ca.trace && ca.trace_all && ca.tslot < 0 && lane == 0 && blockIdx.x == 0) {
      const long i = 1024 + (long)ca.n_ops * gridDim.x + (long)op * nwc + warp;
      if (i < LK_TRACE_MAX) ca.trace[i] = gtimer();
    }
    if (!ca.n_inl) ok = __syncthreads_and(ok) != 0;  // every warp agrees before the next barrier
    CHAIN_STAMP(3 + 3 * op);
    if (ca.trace && ca.trace_all && ca.tslot < 0 && threadIdx.x == 0) {
      const long i = 1024 + (long)op * gridDim.x + blockIdx.x;
      if (i < LK_TRACE_MAX) ca.trace[i] = gtimer();
    }
    if (!ok) break;
    if (o.argmax_parts) {
#pragma unroll
      for (int t = 0; t < M; ++t) {
        const unsigned long long wmax = warp_max_u64(best[t]);
        if (lane == 0) keys[t * MAXW + warp] = wmax;
      }
      __syncthreads();
      if (threadIdx.x < M) {
        unsigned long long m = 0;
        for (int w = 0; w < nwc; ++w) m = keys[threadIdx.x * MAXW + w] > m ? keys[threadIdx.x * MAXW + w] : m;
        o.argmax_parts[(long)threadIdx.x * gridDim.x + blockIdx.x] = m;
      }
      if (o.argmax_idx) {
        ok = grid_sync(ca.sync, gen, gridDim.x, ca.wait_ns, ca.err, abort_flag);
        if (!ok) break;
        if (blockIdx.x == 0 && warp < M) {
          unsigned long long m = 0;
          for (int i = lane; i < (int)gridDim.x; i += 32) {
            const unsigned long long k = o.argmax_parts[(long)warp * gridDim.x + i];
            m = k > m ? k : m;
          }
          m = warp_max_u64(m);
          if (lane == 0) o.argmax_idx[warp] = (int)(0xFFFFFFFFu - (unsigned)(m & 0xFFFFFFFFull));
        }
      }
    }
  }
  // Drain: stages issued but not consumed (after an abort) must land before
  // the block may end.
  if (lane == 0)
    for (long m = consumed; m < issued; ++m)
      drain_wait(full0 + 8 * (unsigned)(warp * D + m % D), (unsigned)(m / D) & 1u, ca.wait_ns, ca.err);
  __syncwarp();
  tend(ca.tslot >= 0 ? ca.trace : nullptr, ca.tslot, ca.n_ops, 2);
}

typedef void (*chain_fn)(const ChainArgs);

template <int Q>
chain_fn pick_m(int M) {
  switch (M) {
    case 1: return gemv_chain_kernel<Q, 1>;
    case 2: return gemv_chain_kernel<Q, 2>;
    case 3: return gemv_chain_kernel<Q, 3>;
    case 4: return gemv_chain_kernel<Q, 4>;
    case 5: return gemv_chain_kernel<Q, 5>;
    case 6: return gemv_chain_kernel<Q, 6>;
    case 7: return gemv_chain_kernel<Q, 7>;
    default: return gemv_chain_kernel<Q, 8>;
  }
}

unsigned act_area_rt(int mode, int M, unsigned len) {
  return mode == 0 ? M * len * 4u : M * len * (mode == 2 ? 2u : 1u) + M * len / 8u;
}

unsigned stage_bytes_for(int K) {
  const unsigned tk = K <= TKMAX ? (unsigned)K : 4096u;
  const unsigned srow = tk / 16u + 16u;  // as make_geom (padded rows)
  return (QR * tk + QR * srow + 127u) & ~127u;
}

}  // namespace
}  // namespace lkring

using namespace lkring;

extern "C" size_t lk_chain_sync_bytes(void) { return 256; }

// Launch the chain kernel over `ops` (host copies; ops_dev their device copy,
// or NULL with the ops carried in the launch arguments: a group).
static lk_status chain_launch(const lk_chain_op* ops, const lk_chain_op* ops_dev, int n_ops, lk_mode mode, int M,
                              float eps, uint32_t* sync, const lkh::GemvProblem* given, const lk_launch_cfg& lc,
                              cudaStream_t stream) {
  unsigned act_cap = 0, sb = 0;
  for (int i = 0; i < n_ops; ++i) {
    const unsigned a = act_area_rt(mode, M, (unsigned)ops[i].K), s = stage_bytes_for(ops[i].K);
    act_cap = a > act_cap ? a : act_cap;
    sb = s > sb ? s : sb;
  }
  const lkh::DeviceInfo* d = lkh::device_info(nullptr);
  if (!d) return LK_ERR_CUDA;
  const unsigned ring_off = (act_cap + 127u) & ~127u;
  const long room = (long)d->smem_optin - (long)ring_off - (long)TAIL;
  int fit = room > 0 ? (int)(room / sb) : 0;
  if (fit > MAX_STAGES) fit = MAX_STAGES;
  const int w = fit < MAXW ? fit : MAXW;
  const int depth = w > 0 ? fit / w : 0;
  if (w < 1 || w * depth < 4) return LK_ERR_SHAPE;
  const unsigned total = ring_off + (unsigned)(w * depth) * sb + TAIL;
  chain_fn f = mode == 0 ? pick_m<0>(M) : mode == 1 ? pick_m<1>(M) : pick_m<2>(M);
  // (the cap is the device's maximum: see ring_gemv)
  if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, d->smem_optin) != cudaSuccess)
    return LK_ERR_CUDA;
  // Without a grid barrier (no step waits, no in-kernel argmax reduce) the
  // chain is an ordinary launch: a grouped GEMV, which may be a programmatic
  // dependent of the previous kernel.  With one it is a cooperative launch.
  bool barrier = false;
  for (int i = 0; i < n_ops; ++i) barrier = barrier || ops[i].wait || ops[i].argmax_idx;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, w * 32, total) != cudaSuccess || per_sm < 1)
    return LK_ERR_SHAPE;
  ChainArgs ca;
  ca.ops = ops_dev;
  ca.n_ops = n_ops;
  ca.nwc = w;
  ca.depth = depth;
  ca.stage_bytes = sb;
  ca.ring_off = ring_off;
  ca.eps = eps;
  ca.sync = sync;
  ca.wait_ns = lkh::opt_wait_us > 0 ? (unsigned long long)lkh::opt_wait_us * 1000ull : 2000000000ull;
  ca.pol_w = 1ull;  // L2 evict-first on the weight copies
  ca.err = lkh::error_word_ptr();
  if (!ca.err) return LK_ERR_CUDA;
  ca.trace = lkh::opt_trace ? lkh::trace_ptr() : nullptr;
  ca.trace_all = lkh::opt_trace == 2;
  ca.tslot = lkh::opt_trace == 3 ? lkh::trace_next_slot() : -1;
  ca.pdl = !barrier && lc.pdl ? 1 : 0;
  ca.prefill = lkh::prefill_warps(w, lc.prefill);
  ca.n_inl = 0;
  ca.gx = nullptr;
  ca.gxq = ca.gxl = nullptr;
  ca.gxs = nullptr;
  for (int i = 0; i < LK_MAX_GROUP; ++i) ca.inl[i] = ops[i < n_ops ? i : 0];
  if (given) {
    ca.n_inl = n_ops;
    ca.gx = given->x;
    ca.gxq = given->xq;
    ca.gxl = given->xl;
    ca.gxs = given->xs;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(d->sm_count);
  cfg.blockDim = dim3(w * 32);
  cfg.dynamicSmemBytes = total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (barrier) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (barrier || ca.pdl) ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, f, ca) != cudaSuccess) return LK_ERR_CUDA;
  return lkh::launch_status();
}

extern "C" lk_status lk_gemv_chain(const lk_chain_op* ops, const lk_chain_op* ops_dev, int n_ops, lk_mode mode,
                                   int M, float eps, uint32_t* sync, const lk_launch_cfg* cfg, cudaStream_t stream) {
  using lkh::aligned;
  if (mode < LK_DEQUANT || mode > LK_TWOPASS || lkh::check_launch_cfg(cfg)) return LK_ERR_ARG;
  if (M < 1 || M > LK_MAX_M || n_ops < 0) return LK_ERR_SHAPE;
  if (n_ops == 0) return LK_OK;
  if (!ops || !ops_dev || !sync) return LK_ERR_ARG;
  if (!aligned(ops_dev, 8) || !aligned(sync, 8)) return LK_ERR_ALIGN;
  for (int i = 0; i < n_ops; ++i) {
    const lk_chain_op& o = ops[i];
    if (o.N < 1 || o.K < 256 || o.K % 256) return LK_ERR_SHAPE;
    if (!o.wq || !o.ws || !o.x || !o.y || (o.argmax_idx && !o.argmax_parts)) return LK_ERR_ARG;
    if (!aligned(o.wq, 16) || !aligned(o.ws, 16) || !aligned(o.x, 4) || (o.gain && !aligned(o.gain, 4)) ||
        !aligned(o.y, 4) || (o.argmax_parts && !aligned(o.argmax_parts, 8)) ||
        (o.argmax_idx && !aligned(o.argmax_idx, 4)))
      return LK_ERR_ALIGN;
  }
  return chain_launch(ops, ops_dev, n_ops, mode, M, eps, sync, nullptr, cfg ? *cfg : lk_launch_cfg{}, stream);
}

// A group of GEMVs over one given activation (p: K, mode, M and the
// activation) on the chain kernel, in one launch without barriers.
// LK_ERR_SHAPE when the chain kernel does not take the shape.
lk_status lkh::chain_group(const GemvProblem& p, const lk_gemv_target* t, int n, cudaStream_t stream) {
  if (n < 1 || n > LK_MAX_GROUP || p.K < 256 || p.K % 256 || p.M < 1 || p.M > LK_MAX_M) return LK_ERR_SHAPE;
  if (p.mode == LK_DEQUANT ? !aligned(p.x, 16)
                           : (!aligned(p.xq, 16) || !aligned(p.xs, 16) || (p.mode == LK_TWOPASS && !aligned(p.xl, 16))))
    return LK_ERR_SHAPE;
  lk_chain_op ops[LK_MAX_GROUP];
  for (int i = 0; i < n; ++i) {
    if (!aligned(t[i].wq, 16) || !aligned(t[i].ws, 16)) return LK_ERR_SHAPE;
    ops[i] = lk_chain_op{t[i].wq, t[i].ws, t[i].N, p.K, nullptr, nullptr, t[i].y, nullptr, nullptr, 0, 0};
  }
  return chain_launch(ops, nullptr, n, (lk_mode)p.mode, p.M, 0.f, nullptr, &p, p.cfg, stream);
}
