// Kernels of the PowerSGD step for padded rank 4.
#include "psgd_launch_rp.cuh"

namespace psgd {
PSGD_INSTANTIATE(4)
}  // namespace psgd
