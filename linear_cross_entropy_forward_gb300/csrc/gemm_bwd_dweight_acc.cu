// Instantiation: dweight tiles from two MN-major operands, accumulated in fp32 over
// token chunks (flce_forward_backward with more than one chunk).
#include "flce_gemm.cuh"

namespace flce {
FLCE_DEFINE_LAUNCHER(launch_bwd_dweight_acc, EPI_ACCUM, true, true, TN_DWEIGHT)
}  // namespace flce
