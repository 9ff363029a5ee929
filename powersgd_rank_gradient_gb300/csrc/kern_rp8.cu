// Kernels of the PowerSGD step for padded rank 8.
#include "psgd_launch_rp.cuh"

namespace psgd {
PSGD_INSTANTIATE(8)
}  // namespace psgd
