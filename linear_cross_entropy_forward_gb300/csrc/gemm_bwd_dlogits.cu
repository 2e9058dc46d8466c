// Instantiation: backward recompute -> dlogits chunk (A = hidden K-major, B = weight MN-major).
#include "flce_gemm.cuh"

namespace flce {

cudaError_t launch_bwd_dlogits(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmShape& sh,
                           const EpiArgs& ea, int num_sms, cudaStream_t stream) {
  return launch_gemm<EPI_DLOGITS, false, true>(tmA, tmB, sh, ea, num_sms, stream);
}

}  // namespace flce
