// Instantiation: forward logits tiles -> online-softmax partials; hidden K-major, weight [H,V] MN-major.
#include "flce_gemm.cuh"

namespace flce {
FLCE_DEFINE_LAUNCHER(launch_fwd_stats, EPI_FWD_STATS, false, true, TN_FWD)

int pair_capacity() {
  static std::atomic<int> cap[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int c = cap[dev].load();
  if (c <= 0) {
    if (pair_max_clusters<EPI_FWD_STATS, false, true, TN_FWD>(&c) != cudaSuccess) return 0;
    cap[dev].store(c);
  }
  return c;
}
}  // namespace flce
