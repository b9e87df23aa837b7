// Block-sparse backward main kernel (causal or not): the SPARSE variants of
// fa_bwd_kernel.cuh. For each key tile the kernel visits only the query tiles
// whose mask row keeps it (and, if causal, that are not above the diagonal),
// so work and IO fall with the sparsity (condensed paper sample_paper.md,
// section 4: block-sparse FlashAttention, IO proportional to the sparsity).
#include "fa_bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_main_sparse(const BwdLaunch& a, cudaStream_t stream) {
  const bool causal = a.causal != 0;
  if (a.d == 64)
    return causal ? launch_bwd_main_t<64, true, true, false>(a, stream)
                  : launch_bwd_main_t<64, false, true, false>(a, stream);
  return causal ? launch_bwd_main_t<128, true, true, false>(a, stream)
                : launch_bwd_main_t<128, false, true, false>(a, stream);
}

}  // namespace fa
