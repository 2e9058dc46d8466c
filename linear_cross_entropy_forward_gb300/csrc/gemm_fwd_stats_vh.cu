// Instantiation: forward logits tiles -> online-softmax partials; hidden K-major, weight [V,H] K-major.
#include "flce_gemm.cuh"

namespace flce {
FLCE_DEFINE_LAUNCHER(launch_fwd_stats_vh, EPI_FWD_STATS, false, false, TN_FWD)
}  // namespace flce
