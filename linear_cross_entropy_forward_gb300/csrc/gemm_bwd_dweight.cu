// Instantiation: dweight chunk = hidden^T @ dlogits (A = hidden MN-major, B = dlogits MN-major).
#include "flce_gemm.cuh"

namespace flce {

cudaError_t launch_bwd_dweight(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmShape& sh,
                           const EpiArgs& ea, int num_sms, cudaStream_t stream) {
  return launch_gemm<EPI_STORE_BF16, true, true>(tmA, tmB, sh, ea, num_sms, stream);
}

}  // namespace flce
