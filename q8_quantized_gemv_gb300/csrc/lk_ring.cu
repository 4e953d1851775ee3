// Bulk-copy ring GEMV (placeholder until the ring kernel lands) and the
// device-side error word that bounded waits set.
#include "lk_device.cuh"
#include "lk_host.h"

__device__ int lk_error_word;

namespace lkh {

bool ring_supports(const GemvProblem&) { return false; }

int ring_max_ctas(long) { return 0; }

lk_status ring_gemv(const GemvProblem&, cudaStream_t, int*) { return LK_ERR_SHAPE; }

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
