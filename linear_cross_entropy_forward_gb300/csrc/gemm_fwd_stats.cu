// Instantiation: forward logits tiles -> online-softmax partials (A = hidden K-major, B = weight MN-major).
#include "flce_gemm.cuh"

namespace flce {

cudaError_t launch_fwd_stats(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmShape& sh,
                           const EpiArgs& ea, int num_sms, cudaStream_t stream) {
  return launch_gemm<EPI_FWD_STATS, false, true>(tmA, tmB, sh, ea, num_sms, stream);
}

}  // namespace flce
