// Instantiation: dhidden += dlogits @ weight_chunk^T (A = dlogits K-major, B = weight K-major).
#include "flce_gemm.cuh"

namespace flce {

cudaError_t launch_bwd_dhidden(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmShape& sh,
                           const EpiArgs& ea, int num_sms, cudaStream_t stream) {
  return launch_gemm<EPI_ACCUM, false, false>(tmA, tmB, sh, ea, num_sms, stream);
}

}  // namespace flce
