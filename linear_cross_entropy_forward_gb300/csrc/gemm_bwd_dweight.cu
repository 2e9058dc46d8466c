// Instantiation: dweight chunk = hidden^T @ dlogits (A = hidden MN-major, B = dlogits MN-major).
#include <atomic>

#include "flce_gemm.cuh"

namespace flce {

cudaError_t launch_bwd_dweight(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmShape& sh,
                           const EpiArgs& ea, cudaStream_t stream) {
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int mc = max_clusters[dev].load();
  if (mc <= 0) {
    e = pair_max_clusters<EPI_STORE_BF16, true, true, TN_DWEIGHT>(&mc);
    if (e != cudaSuccess) return e;
    if (mc <= 0) return cudaErrorInvalidConfiguration;
    max_clusters[dev].store(mc);
  }
  return launch_gemm_pair<EPI_STORE_BF16, true, true, TN_DWEIGHT>(tmA, tmB, sh, ea, mc, stream);
}

}  // namespace flce
