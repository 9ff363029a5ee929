// Kernels of the PowerSGD step for padded rank 1.
#include "psgd_launch_rp.cuh"

namespace psgd {
PSGD_INSTANTIATE(1)
}  // namespace psgd
