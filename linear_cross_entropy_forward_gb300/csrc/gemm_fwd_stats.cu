// Instantiation: forward logits tiles -> online-softmax partials (A = hidden K-major, B = weight MN-major).
#include <atomic>

#include "flce_gemm.cuh"

namespace flce {

cudaError_t launch_fwd_stats(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmShape& sh,
                           const EpiArgs& ea, cudaStream_t stream) {
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int mc = max_clusters[dev].load();
  if (mc <= 0) {
    e = pair_max_clusters<EPI_FWD_STATS, false, true, TN_FWD>(&mc);
    if (e != cudaSuccess) return e;
    if (mc <= 0) return cudaErrorInvalidConfiguration;
    max_clusters[dev].store(mc);
  }
  return launch_gemm_pair<EPI_FWD_STATS, false, true, TN_FWD>(tmA, tmB, sh, ea, mc, stream);
}

}  // namespace flce
