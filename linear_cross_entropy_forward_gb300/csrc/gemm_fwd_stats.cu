// Instantiation: forward logits tiles -> online-softmax partials; hidden K-major, weight [H,V] MN-major.
#include "flce_gemm.cuh"

namespace flce {
FLCE_DEFINE_LAUNCHER(launch_fwd_stats, EPI_FWD_STATS, false, true, TN_FWD)

int cluster_capacity(int csize) {
  static std::atomic<int> cap[64][2];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int k = csize == 4 ? 1 : 0;
  int c = cap[dev][k].load();
  if (c <= 0) {
    if (pair_max_clusters<EPI_FWD_STATS, false, true, TN_FWD>(csize, &c) != cudaSuccess) return 0;
    cap[dev][k].store(c);
  }
  return c;
}
}  // namespace flce
