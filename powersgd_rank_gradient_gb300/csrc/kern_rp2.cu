// Kernels of the PowerSGD step for padded rank 2.
#include "psgd_launch_rp.cuh"

namespace psgd {
PSGD_INSTANTIATE(2)
}  // namespace psgd
