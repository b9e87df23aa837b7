// Backward main kernel with fused dropout and a block mask (causal or not):
// the SPARSE + DROP variants of fa_bwd_kernel.cuh (see fa_bwd_sparse.cu and
// fa_bwd_dropout.cu for the two features).
#include "fa_bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_main_dropout_sparse(const BwdLaunch& a, cudaStream_t stream) {
  const bool causal = a.causal != 0;
  if (a.d == 64)
    return causal ? launch_bwd_main_t<64, true, true, true>(a, stream)
                  : launch_bwd_main_t<64, false, true, true>(a, stream);
  return causal ? launch_bwd_main_t<128, true, true, true>(a, stream)
                : launch_bwd_main_t<128, false, true, true>(a, stream);
}

}  // namespace fa
