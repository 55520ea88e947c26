// Tensor-core (tcgen05 / TMEM / TMA) path of the lightning indexer.
#include "common.cuh"

namespace csa {

bool index_tc_supported(const csa_params& p, csa_dtype q_dtype, const csa_rows& keys, int Q) {
  (void)p; (void)q_dtype; (void)keys; (void)Q;
  return false;
}

cudaError_t launch_index_tc(const csa_params&, const void*, csa_dtype, const float*, const float*,
                            const csa_rows&, int64_t, int, int64_t, float*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace csa
