// Backward main kernel with fused dropout and a block mask (causal or not):
// the SPARSE + DROP variants of fa_bwd_kernel.cuh (see fa_bwd_sparse.cu and
// fa_bwd_dropout.cu for the two features).
#include "fa_bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_main_dropout_sparse(const BwdLaunch& a, const BwdGrid& g, int grid,
                                           cudaStream_t stream) {
  return launch_bwd_main_variant<kModeSparse, true>(a, g, grid, stream);
}

}  // namespace fa
