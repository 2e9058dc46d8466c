// Instantiation: backward recompute -> dlogits chunk; hidden K-major, weight [H,V] MN-major.
#include "flce_gemm.cuh"

namespace flce {
FLCE_DEFINE_LAUNCHER(launch_bwd_dlogits, EPI_DLOGITS, false, true, TN_DLOGITS)
}  // namespace flce
