// Ring GEMV kernels of numerics mode 2 (TwoPassInt8), compiled in a
// translation unit of their own so the three modes build in parallel.
#include "lk_ring_kernel.cuh"

namespace lkring {
LK_RING_PICK(2)
}  // namespace lkring
