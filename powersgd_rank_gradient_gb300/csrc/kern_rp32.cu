// Kernels of the PowerSGD step for padded rank 32.
#include "psgd_launch_rp.cuh"

namespace psgd {
PSGD_INSTANTIATE(32)
}  // namespace psgd
