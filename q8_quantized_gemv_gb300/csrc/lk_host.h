// Host-side helpers shared by the library's translation units (not part of
// the public ABI).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "lk.h"

namespace lkh {

// Per-device attributes, queried once per device and cached.
struct DeviceInfo {
  int sm_count;
  int smem_optin;     // max dynamic shared memory per block (opt-in)
  int smem_per_sm;
  int l2_bytes;
};
const DeviceInfo* device_info(int* dev_out);

// Process-wide options (lk_set_option).
extern long opt_gemv_path;    // 0 auto, 1 direct, 2 ring, 3 tensor-core (small batch)
extern long opt_ring_stages;  // 0 default
extern long opt_grid_ctas;    // 0 default
extern long opt_ring_warps;   // 0 auto, else warps per block of the ring kernel (1..16)
extern long opt_ring_kb;      // 0: no cap, else shared memory per ring block in KB
extern long opt_ring_cps;     // ring blocks per SM in the grid (default 1)
extern long opt_pdl;          // 1: fused ring launches are programmatic dependents
extern long opt_l2_prefetch_kb;  // chain: KB of later steps each block requests into L2 ahead
extern long opt_trace;        // 1: kernels write block 0 timestamps to the trace buffer
extern long opt_ring_hint;    // 1: L2 evict-first hint on the weight copies (default)
extern long opt_wait_us;      // bound of every device-side wait, microseconds (0 = 2 s)
extern long opt_mma_min_m;    // fewest activation rows taking the tensor-core kernel (0 = 2)
extern long opt_mma_tk;       // its bytes of K per stage (0 auto, else a multiple of 256)
extern long opt_mma_warps;    // its warps per block (0 auto)
extern long opt_mma_depth;    // its ring stages per warp (0 = 1)
extern long opt_mma_i8;       // its dots on the int8 tensor path: 0 auto (Int8Act), 1 always, 2 never
extern long opt_mma_group;    // its tiles per warp: 0 auto, 1 one warp per tile, 4 four warps per tile
extern long opt_mma_act16;    // its activations held as f16: 0 auto, 1 force, 2 never
extern long opt_group_prefill; // the same for a grouped launch over one given activation (0: as ring_prefill)
extern long opt_ring_tk;       // ring kernel: bytes of K per stage for rows longer than that (0: auto)
extern long opt_ring_prefill; // warps that issue their first weight stages before the dependency wait (0: half)
extern long opt_l2_ahead_kb;  // ring/tensor-core kernels: KB per block of later stages requested into L2 at start

inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// Device address of a file-scope __device__ variable on the current device,
// looked up (cudaGetSymbolAddress, with that device current) the first time
// and kept per device.  `symbol` is the variable's host-side stand-in, which
// is not a device address.  Threads that race on a first lookup each store
// the same address (atomics, no data race).  The cached address belongs to
// the device's current context: it is stale after cudaDeviceReset().
constexpr int kMaxDevices = 64;
template <typename T>
inline T* device_symbol(std::atomic<T*> (&cache)[kMaxDevices], const void* symbol) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  T* p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    void* q = nullptr;
    if (cudaGetSymbolAddress(&q, symbol) != cudaSuccess || !q) return nullptr;
    p = (T*)q;
    cache[dev].store(p, std::memory_order_release);
  }
  return p;
}

inline lk_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? LK_OK : LK_ERR_CUDA;
}

// Everything one GEMV launch needs (plain, split-K partial, argmax epilogue).
struct GemvProblem {
  const int8_t* wq;
  const __half* ws;
  long N;
  int K;
  int mode;
  const float* x;
  const int8_t* xq;
  const int8_t* xl;
  const float* xs;
  int M;
  int S;                         // split-K chunks (1 for the plain GEMV)
  bool split;                    // write split-K partials instead of y
  float* y;                      // plain: y [M][N]; split quantized: part f32 [S][M][N]
  double* part64;                // split Dequant: part f64 [S][M][N]
  unsigned long long* amax;      // plain only: [M][n_parts]
  bool fuse;                     // activation computed in the kernel from xraw
  const float* xraw;             // fused: raw f32 rows [M][K]
  const float* gain;             // fused: RMSNorm gain [K], or NULL for quantize only
  float eps;
};

// Warps of a block of nw that fill their ring stages before the dependency
// wait (the others after the activation is loaded): option "ring_prefill",
// 0 = half of them (measured best: a full ring of requests ahead of the
// wait slowed the activation loads and the wait itself).
inline int prefill_warps(int nw) {
  const int p = opt_ring_prefill > 0 ? (int)opt_ring_prefill : (nw + 1) / 2;
  return p < nw ? p : nw;
}

// Device address of the error word that bounded device waits set (lk_ring.cu).
int* error_word_ptr();
// Device address of the trace buffer (option "trace").
unsigned long long* trace_ptr();
// Option "trace" 3: the next launch's record index in the timeline (wraps),
// and its reset (setting the option resets it).
int trace_next_slot();
void trace_reset();

// Bulk-copy ring kernel (lk_ring.cu).  Returns LK_ERR_SHAPE when the problem
// is outside what the ring kernel takes (the caller then uses the direct
// kernel), otherwise the launch status; *n_parts receives the blocks launched.
lk_status ring_gemv(const GemvProblem& p, cudaStream_t stream, int* n_parts);
bool ring_supports(const GemvProblem& p);

// Several GEMVs over one given activation on the chain kernel (lk_chain.cu):
// one launch; LK_ERR_SHAPE when the chain kernel does not take the shape.
lk_status chain_group(const GemvProblem& p, const lk_gemv_target* t, int n, cudaStream_t stream);

// Tensor-core kernel for 2..8 activation rows (lk_mma.cu), same contract.
lk_status mma_gemv(const GemvProblem& p, cudaStream_t stream, int* n_parts);
// The same over nmat matrices sharing p's activation, in one launch.
lk_status mma_launch(const GemvProblem& p, int nmat, const int8_t* const* wq, const __half* const* ws,
                     const long* N, float* const* y, cudaStream_t stream, int* n_parts);
bool mma_supports(const GemvProblem& p);
int ring_max_ctas(long N);

}  // namespace lkh
