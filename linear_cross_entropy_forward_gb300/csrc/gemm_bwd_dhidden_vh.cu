// Instantiation: dhidden += dlogits x weight chunk; dlogits K-major, weight [V,H] MN-major.
#include "flce_gemm.cuh"

namespace flce {
FLCE_DEFINE_LAUNCHER(launch_bwd_dhidden_vh, EPI_ACCUM, false, true, TN_DHIDDEN)
}  // namespace flce
