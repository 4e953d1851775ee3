// Bulk-copy ring GEMV for sm_103a (host side: layout and launch), and the
// device-side error word that every bounded wait sets when it gives up.
//
// One block per SM, persistent over a contiguous, balanced range of rows
// (and one split-K chunk).  The block loads the activation slice it needs
// (words and scales of all M rows) into shared memory once.  Every warp then
// streams its own "quads" (4 consecutive rows; warp w takes quads w, w + W,
// ...) through its own ring stages with 1-D bulk copies (TMA:
// cp.async.bulk ... mbarrier::complete_tx::bytes, L2 evict-first), refilling
// a stage as soon as it has consumed it: a stage is a whole quad for rows up
// to 8 KB, else a 4 KB slice of it; each warp owns one stage where they fit
// (12 warps).  The consumer arithmetic is the direct kernel's (lk_gemv.cu),
// with the same bits.
//
// Every wait on an mbarrier is bounded by a wall-clock limit (%globaltimer).
// A wait that runs out sets the error word and an abort flag in shared
// memory; every thread then leaves its loops, and each warp waits (again
// bounded) for the copies it issued, so that no copy is still in flight into
// the block's shared memory when the block ends.
#include "lk_ring_kernel.cuh"

static_assert(lkring::TREC == LK_TRACE_REC, "trace record size of the public header");

__device__ int lk_error_word;
// Block 0's timestamps (%globaltimer, ns) of the last traced launch.
__device__ unsigned long long lk_trace_buf[lkring::LK_TRACE_MAX];

namespace lkring {
// A wait on an mbarrier that nothing completes: the bounded wait must give
// up after `limit_ns`, raise the error word and return.
__global__ void wait_selftest_kernel(unsigned long long limit_ns, int* err) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (!mbar_wait(smem_u32(&bar), 0, limit_ns, &abort_flag)) {
    if (threadIdx.x == 0) atomicOr(err, ERR_SELFTEST);
  }
}


namespace {
ring_fn pick(int mode, int M, bool split, bool fuse, bool glu) {
  if (split) fuse = false;  // the fused prologue is for whole rows only
  return mode == 0 ? ring_pick<0>(M, split, fuse, glu) : mode == 1 ? ring_pick<1>(M, split, fuse, glu)
                                                                  : ring_pick<2>(M, split, fuse, glu);
}

}  // namespace
}  // namespace lkring

// Device address of the error word on the current device, looked up once
// per device.
int* lkh::error_word_ptr() {
  static std::atomic<int*> cache[kMaxDevices];
  return device_symbol(cache, (const void*)&lk_error_word);
}

static std::atomic<int> trace_seq{0};
void lkh::trace_reset() { trace_seq.store(0); }
int lkh::trace_next_slot() { return trace_seq.fetch_add(1) % (lkring::LK_TRACE_MAX / lkring::TREC); }

unsigned long long* lkh::trace_ptr() {
  static std::atomic<unsigned long long*> cache[kMaxDevices];
  return device_symbol(cache, (const void*)lk_trace_buf);
}

namespace lkring {
namespace {

unsigned act_area_rt(int mode, int M, unsigned len) {
  return mode == 0 ? M * len * 4u : M * len * (mode == 2 ? 2u : 1u) + M * len / 8u;
}

struct Layout {
  unsigned tk, srow, stage_bytes, s_off, act_len, ring_off, total;
  int nwc, depth;
};

// The widest chunk of K any block of this launch works on.
int max_chunk_blocks(int nb, int S) {
  if (S <= 1) return nb;
  int m = 0;
  for (int c = 0; c < S; ++c) {
    int w = lk::splitk_bound(nb, S, c + 1) - lk::splitk_bound(nb, S, c);
    m = w > m ? w : m;
  }
  return m;
}

// Blocks of a ring launch along the rows (per split-K chunk).
int ring_gx(const lkh::GemvProblem& p, int sm_count) {
  const int S = p.split && p.S > 1 ? p.S : 1;
  const int g = p.cfg.grid_ctas > 0 ? p.cfg.grid_ctas : sm_count;
  const int gx = (g + S - 1) / S;
  return gx < 1 ? 1 : gx;
}

Layout layout(const lkh::GemvProblem& p, int smem_optin, int /*sm_count*/) {
  Layout L;
  const int nb = p.K / 32;
  const int S = p.split ? (p.S > 1 ? p.S : 1) : 1;
  L.act_len = 32u * (unsigned)max_chunk_blocks(nb, S);
  // whole quads (one copy of the levels, one per row of scales) up to TKMAX;
  // rows up to twice that in two equal slices (a multiple of 1 KB), longer
  // ones in 4 KB slices.  Measured (sequence, down 4096 x 12288, batch 1):
  // 4 KB slices 1790 us per token, 6 KB 1747, 2 KB 1770, 3 KB 1936, 8 KB
  // 1844: with 6.7 quads a block, two slices a quad take one round trip
  // fewer per busy warp than three.
  const bool halves = p.K > TKMAX && p.K <= 2 * TKMAX && (p.K / 2) % 1024 == 0;
  L.tk = p.K <= TKMAX ? (unsigned)p.K : halves ? (unsigned)(p.K / 2) : 4096u;
  if (p.cfg.ring_tk > 0 && p.cfg.ring_tk < p.K) L.tk = (unsigned)p.cfg.ring_tk;
  L.srow = L.tk / 16u + 16u;  // as make_geom (padded rows)
  L.s_off = QR * L.tk;
  L.stage_bytes = (L.s_off + QR * L.srow + 127u) & ~127u;
  L.ring_off = (act_area_rt(p.mode, p.M, L.act_len) + 127u) & ~127u;
  const long room = (long)smem_optin - (long)L.ring_off - (long)TAIL;
  int fit = room > 0 ? (int)(room / L.stage_bytes) : 0;
  if (fit > MAX_STAGES) fit = MAX_STAGES;
  // warps x stages per warp: as many stages in flight as fit, one warp per
  // stage up to MAXW warps (each warp streams its own quads).  Measured: for
  // rows in slices with few quads per block (down 4096 x 12288, 6.7 quads of
  // 3 slices), 6 warps of 2 stages lost to 12 of 1 (in the sequence: body
  // 10.2 against 9.7 us, 1815 against 1789 us per token)
  const int w = fit < MAXW ? fit : MAXW;
  L.nwc = w;
  L.depth = w > 0 ? fit / w : 0;
  L.total = L.ring_off + L.nwc * L.depth * L.stage_bytes + TAIL;
  return L;
}

bool layout_ok(const Layout& L) { return L.nwc > 0 && L.nwc * L.depth >= 4; }

}  // namespace
}  // namespace lkring

namespace lkh {

using namespace lkring;

bool ring_supports(const GemvProblem& p) {
  if (p.K < 256 || p.K % 256 || p.N < 1 || p.M < 1 || p.M > LK_MAX_M) return false;
  // the gated pair's epilogue kernel: one activation row, whole rows
  if (p.F > 0 && (p.M != 1 || p.split || p.fuse || p.N != 2 * p.F || p.F % 32 || !aligned(p.ws2, 16))) return false;
  if (!aligned(p.ws, 16)) return false;
  if (!p.fuse && (p.mode == 0 ? !aligned(p.x, 16)
                              : (!aligned(p.xq, 16) || !aligned(p.xs, 16) || (p.mode == 2 && !aligned(p.xl, 16)))))
    return false;
  const DeviceInfo* d = device_info(nullptr);
  if (!d) return false;
  return layout_ok(layout(p, d->smem_optin, d->sm_count));
}

int ring_max_ctas(long) {
  // one block per SM by default; lk_launch_cfg.grid_ctas up to four per SM
  // where the launch writes argmax keys
  const DeviceInfo* d = device_info(nullptr);
  return d ? 4 * d->sm_count : 4096;
}

lk_status ring_gemv(const GemvProblem& p, cudaStream_t stream, int* n_parts) {
  const DeviceInfo* d = device_info(nullptr);
  if (!d) return LK_ERR_CUDA;
  const Layout L = layout(p, d->smem_optin, d->sm_count);
  if (!layout_ok(L)) return LK_ERR_SHAPE;
  ring_fn f = pick(p.mode, p.M, p.split, p.fuse, p.F > 0);
  // The cap is the device's opt-in maximum, never this launch's size: one
  // instantiation serves launches of different sizes, and a cap lowered by a
  // later launch would make an earlier one (e.g. a node of a captured graph,
  // relaunched on its own by a profiler) exceed it.
  if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, d->smem_optin) != cudaSuccess)
    return LK_ERR_CUDA;
  RingArgs ra;
  ra.p = p;
  ra.nwc = L.nwc;
  ra.depth = L.depth;
  ra.tk = L.tk;
  ra.srow = L.srow;
  ra.stage_bytes = L.stage_bytes;
  ra.s_off = L.s_off;
  ra.act_len = L.act_len;
  ra.ring_off = L.ring_off;
  ra.wait_ns = opt_wait_us > 0 ? (unsigned long long)opt_wait_us * 1000ull : 2000000000ull;
  ra.pol_w = 1ull;  // L2 evict-first on the weight copies
  ra.pdl = p.cfg.pdl;
  ra.err = lkh::error_word_ptr();
  if (!ra.err) return LK_ERR_CUDA;
  ra.trace = opt_trace ? lkh::trace_ptr() : nullptr;
  ra.tslot = opt_trace == 3 ? lkh::trace_next_slot() : -1;
  ra.prefill = lkh::prefill_warps(L.nwc, p.cfg.prefill);
  const int S = p.split && p.S > 1 ? p.S : 1;
  const int gx = ring_gx(p, d->sm_count);
  ra.gx = gx;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx, S);
  cfg.blockDim = dim3(L.nwc * 32);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ra.pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, f, ra) != cudaSuccess) return LK_ERR_CUDA;
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
  int* err = lkh::error_word_ptr();
  if (!err) return LK_ERR_CUDA;
  lkring::wait_selftest_kernel<<<1, 32, 0, stream>>>((unsigned long long)limit_us * 1000ull, err);
  return lkh::launch_status();
}

extern "C" lk_status lk_trace_read(uint64_t* host_out, int n) {
  if (!host_out || n < 0 || n > lkring::LK_TRACE_MAX) return LK_ERR_ARG;
  if (n == 0) return LK_OK;
  if (cudaDeviceSynchronize() != cudaSuccess) return LK_ERR_CUDA;
  if (cudaMemcpyFromSymbol(host_out, lk_trace_buf, (size_t)n * 8) != cudaSuccess) return LK_ERR_CUDA;
  return LK_OK;
}
