// Instantiation: backward recompute -> dlogits chunk; hidden K-major, weight [V,H] K-major.
#include "flce_gemm.cuh"

namespace flce {
FLCE_DEFINE_LAUNCHER(launch_bwd_dlogits_vh, EPI_DLOGITS, false, false, TN_DLOGITS)
}  // namespace flce
