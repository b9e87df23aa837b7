// Block-sparse backward main kernel (causal or not): the SPARSE variants of
// fa_bwd_kernel.cuh. For each key tile the kernel visits only the query tiles
// whose mask row keeps it (and, if causal, that are not above the diagonal),
// so work and IO fall with the sparsity (condensed paper sample_paper.md,
// section 4: block-sparse FlashAttention, IO proportional to the sparsity).
#include "fa_bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_main_sparse(const BwdLaunch& a, const BwdGrid& g, int grid,
                                   cudaStream_t stream) {
  return launch_bwd_main_variant<kModeSparse, false>(a, g, grid, stream);
}

}  // namespace fa
