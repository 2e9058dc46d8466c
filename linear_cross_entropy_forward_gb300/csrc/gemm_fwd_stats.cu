// Instantiation: forward logits tiles -> online-softmax partials; hidden K-major, weight [H,V] MN-major.
#include "flce_gemm.cuh"

namespace flce {
FLCE_DEFINE_LAUNCHER(launch_fwd_stats, EPI_FWD_STATS, false, true, TN_FWD)
}  // namespace flce
