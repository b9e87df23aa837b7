// Backward main kernel with fused dropout (dense, causal, key-padded): the
// DROP variants of fa_bwd_kernel.cuh. The keep decisions are regenerated from
// the element indices with the forward pass's counter-based generator
// (fa_philox.cuh), so the backward pass reads no mask. The preprocess and dQ
// conversion stages are those of the pass without dropout: D = rowsum(dO * O)
// still equals rowsum(P * dP) when O is formed from the dropped P.
#include "fa_bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_main_dropout(const BwdLaunch& a, const BwdGrid& g, int grid,
                                    cudaStream_t stream) {
  return launch_bwd_main_variant<kModePlain, true>(a, g, grid, stream);
}

}  // namespace fa
