// The small entry points of the C ABI: status names, options, device
// attributes, RMSNorm + quantize, the standalone quantizer, the argmax
// reductions and the block-dot test hook.
#include <string.h>

#include <mutex>

#include "lk_device.cuh"
#include "lk_host.h"

using namespace lk;

namespace lkh {

long opt_wait_us = 0;
long opt_trace = 0;

// Per-device attributes, queried once per device under a lock (concurrent
// first calls are safe).
static DeviceInfo g_info[kMaxDevices];
static std::atomic<int> g_info_ok[kMaxDevices];
static std::mutex g_info_lock;

const DeviceInfo* device_info(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (dev_out) *dev_out = dev;
  if (!g_info_ok[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> hold(g_info_lock);
    if (!g_info_ok[dev].load(std::memory_order_relaxed)) {
      DeviceInfo d;
      if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
        return nullptr;
      g_info[dev] = d;
      g_info_ok[dev].store(1, std::memory_order_release);
    }
  }
  return &g_info[dev];
}

lk_status check_launch_cfg(const lk_launch_cfg* cfg) {
  if (!cfg) return LK_OK;
  const lk_launch_cfg& c = *cfg;
  if (c.pdl < 0 || c.pdl > 1 || c.prefill < 0 || c.prefill > 16 || c.path < 0 || c.path > 3) return LK_ERR_ARG;
  if (c.grid_ctas < 0 || c.grid_ctas > (1 << 20)) return LK_ERR_ARG;
  if (c.ring_tk < 0 || c.ring_tk > 8192 || c.ring_tk % 1024) return LK_ERR_ARG;
  if (c.mma_min_m < 0 || c.mma_min_m > LK_MAX_BATCH + 1) return LK_ERR_ARG;
  if (c.mma_tk < 0 || c.mma_tk > 8192 || c.mma_tk % 256) return LK_ERR_ARG;
  if (c.mma_warps < 0 || c.mma_warps > 16 || c.mma_depth < 0 || c.mma_depth > 8) return LK_ERR_ARG;
  if (c.mma_i8 < 0 || c.mma_i8 > 2 || c.mma_act16 < 0 || c.mma_act16 > 2) return LK_ERR_ARG;
  if (c.mma_group != 0 && c.mma_group != 1 && c.mma_group != 4) return LK_ERR_ARG;
  return LK_OK;
}

}  // namespace lkh

using namespace lkh;

template <int Q>
__global__ void quantize_kernel(const float* __restrict__ x, long groups, int8_t* __restrict__ xq,
                                int8_t* __restrict__ xl, float* __restrict__ xs, unsigned long long* tr, int slot) {
  asm volatile("griddepcontrol.launch_dependents;" :::);  // as in rmsnorm_quant_kernel
  trec_stamp(tr, slot, TR_START);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  trec_stamp(tr, slot, TR_WAITED);
  const long g = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (g < groups) {  // whole warps
    const int lane = threadIdx.x & 31;
    const long i = g * 32 + lane;
    quant_lane<Q>(__ldcg(x + i), xq, xl, xs, g, lane);
  }
  trec_end(tr, slot, TK_QUANT, groups * 32);
}


extern "C" {

const char* lk_status_string(lk_status s) {
  switch (s) {
    case LK_OK: return "ok";
    case LK_ERR_ARG: return "invalid argument";
    case LK_ERR_ALIGN: return "misaligned pointer";
    case LK_ERR_SHAPE: return "unsupported shape";
    case LK_ERR_WORKSPACE: return "workspace too small";
    case LK_ERR_CUDA: return "CUDA runtime error";
    case LK_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int lk_version(void) { return 100; }

lk_status lk_set_option(const char* name, long value) {
  if (!name) return LK_ERR_ARG;
  if (!strcmp(name, "trace")) {
    if (value < 0 || value > 3) return LK_ERR_ARG;
    opt_trace = value;
    trace_reset();
  } else if (!strcmp(name, "wait_us")) {
    if (value < 0 || value > 60000000L) return LK_ERR_ARG;
    opt_wait_us = value;
  } else {
    return LK_ERR_ARG;
  }
  return LK_OK;
}

long lk_get_option(const char* name) {
  if (!name) return -1;
  if (!strcmp(name, "trace")) return opt_trace;
  if (!strcmp(name, "wait_us")) return opt_wait_us;
  return -1;
}

lk_status lk_quantize_act(const float* x, int M, int K, lk_mode mode, int8_t* xq, int8_t* xl,
                          float* xs, const lk_launch_cfg* cfg, cudaStream_t stream) {
  if (mode != LK_INT8ACT && mode != LK_TWOPASS) return LK_ERR_ARG;
  if (check_launch_cfg(cfg)) return LK_ERR_ARG;
  if (M < 0 || M > LK_MAX_BATCH || K < 0 || K % 32) return LK_ERR_SHAPE;
  if (M == 0 || K == 0) return LK_OK;
  if (!x) return LK_ERR_ARG;
  if (!aligned(x, 4)) return LK_ERR_ALIGN;
  lk_status st = check_act_out(mode, xq, xl, xs);
  if (st) return st;
  const long groups = (long)M * (K / 32);
  const int per_block = 8;
  const long blocks = (groups + per_block - 1) / per_block;
  if (mode == LK_INT8ACT)
    launch_pdl(quantize_kernel<1>, dim3((unsigned)blocks), dim3(32 * per_block), stream, cfg_pdl(cfg), x, groups,
               xq, (int8_t*)nullptr, xs, tr_ptr(), tr_slot());
  else
    launch_pdl(quantize_kernel<2>, dim3((unsigned)blocks), dim3(32 * per_block), stream, cfg_pdl(cfg), x, groups,
               xq, xl, xs, tr_ptr(), tr_slot());
  return launch_status();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Argmax.  Keys are exact, so the max over any partition is the same: the
// block-partial + final-reduce split changes nothing in the result.
__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v,
                                                            unsigned long long* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max_u64(v);
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  v = lane < nw ? sh[lane] : 0ull;
  return warp_max_u64(v);
}

// Final reduce: row t's n keys -> first index of the maximum.
__global__ void __launch_bounds__(256) argmax_reduce_kernel(const unsigned long long* __restrict__ parts,
                                                            int n, int* __restrict__ idx) {
  __shared__ unsigned long long sh[32];
  const long t = blockIdx.x;
  unsigned long long best = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const unsigned long long k = parts[t * n + i];
    best = k > best ? k : best;
  }
  best = block_max_u64(best, sh);
  if (threadIdx.x == 0) idx[t] = (int)(0xFFFFFFFFu - (unsigned)(best & 0xFFFFFFFFull));
}

// Partial keys of logits: block b of row t scans its slice ("kernels.rs"
// argmax_blocks spreads the row over at most 64 blocks).
__global__ void __launch_bounds__(256) argmax_logits_kernel(const float* __restrict__ logits, long N,
                                                            unsigned long long* __restrict__ out) {
  __shared__ unsigned long long sh[32];
  const long t = blockIdx.y;
  const long per = (N + gridDim.x - 1) / gridDim.x;
  const long i0 = (long)blockIdx.x * per, i1 = i0 + per < N ? i0 + per : N;
  unsigned long long best = 0;
  for (long i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const unsigned long long k = amax_key(__ldcg(logits + t * N + i), (unsigned)i);
    best = k > best ? k : best;
  }
  best = block_max_u64(best, sh);
  if (threadIdx.x == 0) out[t * gridDim.x + blockIdx.x] = best;
}

// Exact block dots, lanes arranged as in the GEMV: 8 lanes per row, lane j
// holding bytes 16j..16j+15 of a 128-byte segment (4 blocks); lanes 2q, 2q+1
// hold block q and meet with one xor-shuffle.
__global__ void __launch_bounds__(256) block_dots_kernel(const int8_t* __restrict__ wq, long N, int K,
                                                         const int8_t* __restrict__ xq,
                                                         const int8_t* __restrict__ xl,
                                                         int* __restrict__ d, int* __restrict__ e) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rr = lane >> 3, j = lane & 7, q = j >> 1, hf = j & 1;
  const long o = ((long)blockIdx.x * 8 + warp) * 4 + rr;
  const bool row_ok = o < N;
  const int nb = K >> 5, nsg = (nb + 3) >> 2;
  const int4 zero = make_int4(0, 0, 0, 0);
  for (int sg = 0; sg < nsg; ++sg) {
    const int b = 4 * sg + q;
    const bool ok = row_ok && b < nb;
    const long off = 32L * b + 16 * hf;
    const int4 w = ok ? *(const int4*)(wq + o * K + off) : zero;
    const int4 h = ok ? *(const int4*)(xq + off) : zero;
    int dd = dot16(w, h);
    dd += __shfl_xor_sync(FULL, dd, 1);
    int ee = 0;
    if (xl) {
      const int4 l = ok ? *(const int4*)(xl + off) : zero;
      ee = dot16(w, l);
      ee += __shfl_xor_sync(FULL, ee, 1);
    }
    if (ok && hf == 0) {
      d[o * nb + b] = dd;
      if (xl && e) e[o * nb + b] = ee;
    }
  }
}

extern "C" {

int lk_argmax_parts_max(int N) {
  if (N <= 0) return 0;
  const long a = lkh::ring_max_ctas(N);
  const long b = ((long)N + 31) / 32;
  return (int)(a > b ? a : b);
}

int lk_argmax_scratch_entries(int N) {
  if (N <= 0) return 0;
  long n = ((long)N + 2047) / 2048;
  return (int)(n < 1 ? 1 : (n > 64 ? 64 : n));
}

lk_status lk_argmax(const float* logits, const uint64_t* parts, int n_parts, int M, int N,
                    int32_t* idx, uint64_t* scratch, cudaStream_t stream) {
  if (M < 0 || M > LK_MAX_BATCH) return LK_ERR_SHAPE;
  if (M == 0) return LK_OK;
  if (N < 1) return LK_ERR_SHAPE;
  if (!idx) return LK_ERR_ARG;
  if (!aligned(idx, 4)) return LK_ERR_ALIGN;
  if (parts) {
    if (n_parts < 1) return LK_ERR_SHAPE;
    if (!aligned(parts, 8)) return LK_ERR_ALIGN;
    carveout_max_shared(argmax_reduce_kernel);
    argmax_reduce_kernel<<<M, 256, 0, stream>>>((const unsigned long long*)parts, n_parts, idx);
    return launch_status();
  }
  if (!logits || !scratch) return LK_ERR_ARG;
  if (!aligned(logits, 4) || !aligned(scratch, 8)) return LK_ERR_ALIGN;
  const int nblk = lk_argmax_scratch_entries(N);
  argmax_logits_kernel<<<dim3(nblk, M), 256, 0, stream>>>(logits, N, (unsigned long long*)scratch);
  lk_status st = launch_status();
  if (st) return st;
  argmax_reduce_kernel<<<M, 256, 0, stream>>>((const unsigned long long*)scratch, nblk, idx);
  return launch_status();
}

lk_status lk_q8_block_dots(const int8_t* wq, int N, int K, const int8_t* xq, const int8_t* xl,
                           int32_t* d, int32_t* e, cudaStream_t stream) {
  if (N < 0 || K < 0 || K % 32) return LK_ERR_SHAPE;
  if (N == 0 || K == 0) return LK_OK;
  if (!wq || !xq || !d) return LK_ERR_ARG;
  if (!aligned(wq, 16) || !aligned(xq, 16) || (xl && !aligned(xl, 16)) || !aligned(d, 4) ||
      (e && !aligned(e, 4)))
    return LK_ERR_ALIGN;
  const long blocks = ((long)N + 31) / 32;
  block_dots_kernel<<<(unsigned)blocks, 256, 0, stream>>>(wq, N, K, xq, (xl && e) ? xl : nullptr, d, e);
  return launch_status();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free argmax of logits.  The per-block partial keys live in a
// file-scope device array instead of a caller buffer: LK_MAX_M rows x 64
// blocks (the most lk_argmax_scratch_entries ever returns) = 512 keys, 4 KB.
// Every GPU that loads the library holds it until the process exits.
static __device__ __align__(256) unsigned long long lk_noalloc_argmax_scratch[LK_MAX_M * 64];

// The array's device address on the current device, looked up the first
// time the entry point runs on that device (cudaGetSymbolAddress with the
// device current) and kept per device; concurrent first calls are safe.
static unsigned long long* noalloc_scratch_ptr() {
  static std::atomic<unsigned long long*> cache[kMaxDevices];
  return device_symbol(cache, (const void*)lk_noalloc_argmax_scratch);
}

extern "C" lk_status lk_argmax_noalloc(const float* logits, int M, int N, int32_t* idx, cudaStream_t stream) {
  if (M < 0 || M > LK_MAX_M) return LK_ERR_SHAPE;
  if (M == 0) return LK_OK;
  if (N < 1) return LK_ERR_SHAPE;
  if (!logits || !idx) return LK_ERR_ARG;
  if (!aligned(logits, 4) || !aligned(idx, 4)) return LK_ERR_ALIGN;
  const int nblk = lk_argmax_scratch_entries(N);
  if ((long)M * nblk > LK_MAX_M * 64) return LK_ERR_WORKSPACE;
  unsigned long long* scratch = noalloc_scratch_ptr();
  if (!scratch) return LK_ERR_CUDA;
  argmax_logits_kernel<<<dim3(nblk, M), 256, 0, stream>>>(logits, N, scratch);
  lk_status st = launch_status();
  if (st) return st;
  argmax_reduce_kernel<<<M, 256, 0, stream>>>(scratch, nblk, idx);
  return launch_status();
}
