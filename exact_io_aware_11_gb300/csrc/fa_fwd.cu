// Forward pass without dropout (dense, causal, key-padded and block-sparse):
// instantiates the fused forward kernel of fa_fwd_kernel.cuh. The dropout
// variants are compiled in fa_fwd_dropout.cu.
#include "fa_fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream) {
  if (a.drop.enabled) return launch_fwd_dropout(a, stream);
  const bool causal = a.causal != 0;
  if (a.d == 64)
    return causal ? launch_fwd_t<64, true, false>(a, stream) : launch_fwd_t<64, false, false>(a, stream);
  return causal ? launch_fwd_t<128, true, false>(a, stream) : launch_fwd_t<128, false, false>(a, stream);
}

}  // namespace fa
