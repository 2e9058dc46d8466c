// Instantiation: dweight tiles from two MN-major operands (hidden^T x dlogits for [H,V], dlogits^T x hidden for [V,H]).
#include "flce_gemm.cuh"

namespace flce {
FLCE_DEFINE_LAUNCHER(launch_bwd_dweight, EPI_STORE_BF16, true, true, TN_DWEIGHT)
}  // namespace flce
