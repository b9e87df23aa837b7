// Block-sparse forward: the SPARSE variants of the fused forward kernel
// (fa_fwd_kernel.cuh), with and without dropout. Each Q tile visits only the
// K/V tiles its block-mask row keeps, so work and IO fall with the sparsity
// (FlashAttention abstract, block-sparse FlashAttention; aggregator page, IO
// complexity proportional to the sparsity).
#include "fa_fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_sparse(const FwdLaunch& a, const FwdGrid& g, int grid, cudaStream_t stream) {
  return a.drop.enabled ? launch_fwd_variant<true, kModeSparse>(a, g, grid, stream)
                        : launch_fwd_variant<false, kModeSparse>(a, g, grid, stream);
}

}  // namespace fa
