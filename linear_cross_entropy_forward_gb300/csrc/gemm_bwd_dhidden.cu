// Instantiation: dhidden += dlogits x weight chunk; dlogits K-major, weight [H,V] K-major.
#include "flce_gemm.cuh"

namespace flce {
FLCE_DEFINE_LAUNCHER(launch_bwd_dhidden, EPI_ACCUM, false, false, TN_DHIDDEN)
}  // namespace flce
