// Kernels of the PowerSGD step for padded rank 16.
#include "psgd_launch_rp.cuh"

namespace psgd {
PSGD_INSTANTIATE(16)
}  // namespace psgd
