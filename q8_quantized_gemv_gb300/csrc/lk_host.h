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

// The two process-wide diagnostic options (lk_set_option).  Neither
// changes which kernel runs, how it is launched or any result.
extern long opt_trace;        // 1..3: kernels write timestamps to the trace buffer
extern long opt_wait_us;      // bound of every device-side wait, microseconds (0 = 2 s)

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

// Checks of a caller's launch settings: LK_ERR_ARG, else LK_OK.
lk_status check_launch_cfg(const lk_launch_cfg* cfg);
// The pdl flag of cfg (NULL: 0).
inline int cfg_pdl(const lk_launch_cfg* cfg) { return cfg && cfg->pdl ? 1 : 0; }

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
  // The gated pair (lk_gemv_q8_glu; F > 0): wq/ws are the gate matrix,
  // wq2/ws2 the up matrix, F rows each, N = 2F; y receives the gate values
  // [M][F] followed by the up values [M][F]; the epilogue writes the SwiGLU
  // h (optional f32 [M][F]) and its quantized words hq/hl/hs, completing each
  // 32-output group once through the counters glu_cnt [F/32].
  long F;
  const int8_t* wq2;
  const __half* ws2;
  int* glu_cnt;
  float* h;
  int8_t* hq;
  int8_t* hl;
  float* hs;
  // the caller's per-call launch settings (all zero: the defaults)
  lk_launch_cfg cfg;
};

// GemvProblem's launch settings from cfg (NULL: the defaults).
inline void apply_cfg(GemvProblem& p, const lk_launch_cfg* cfg) {
  p.cfg = cfg ? *cfg : lk_launch_cfg{};
}

// Warps of a block of nw that fill their ring stages before the dependency
// wait (the others after the activation is loaded): `want`, 0 = half of
// them (measured best: a full ring of requests ahead of the wait slowed the
// activation loads and the wait itself).
inline int prefill_warps(int nw, int want = 0) {
  const int p = want > 0 ? want : (nw + 1) / 2;
  return p < nw ? p : nw;
}

// Option "trace" 3: the timeline buffer and this launch's record, else NULL / 0.
unsigned long long* trace_ptr();
int trace_next_slot();
inline unsigned long long* tr_ptr() { return opt_trace == 3 ? trace_ptr() : nullptr; }
inline int tr_slot() { return opt_trace == 3 ? trace_next_slot() : 0; }

// The small kernels run with the shared-memory carveout of the GEMV kernels
// (the largest), so that an SM need not be reconfigured between a norm or
// quantize launch and the GEMV that depends on it.
template <typename F>
inline void carveout_max_shared(F f) {
  cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
}

// Launch as a programmatic dependent of the previous kernel when pdl is set
// (lk_launch_cfg.pdl; the kernels wait for it before their first read of
// data that kernel writes and before their first write).
template <typename... KA, typename... A>
inline void launch_pdl(void (*f)(KA...), dim3 grid, dim3 block, cudaStream_t stream, int pdl, A... args) {
  carveout_max_shared(f);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaLaunchKernelEx(&cfg, f, ((KA)args)...);
}

// Output buffers of an activation quantizer: present for the mode, aligned.
inline lk_status check_act_out(lk_mode mode, const int8_t* xq, const int8_t* xl, const float* xs) {
  if (!xq || !xs || (mode == LK_TWOPASS && !xl)) return LK_ERR_ARG;
  if (!aligned(xs, 4)) return LK_ERR_ALIGN;
  return LK_OK;
}

// Device address of the error word that bounded device waits set (lk_ring.cu).
int* error_word_ptr();
// Option "trace" 3: resets the record index of the timeline (setting the
// option does it).
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
