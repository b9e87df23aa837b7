// Forward with the last wave of work items split over every SM: the SPLIT
// variants of the fused forward kernel (fa_fwd_kernel.cuh), with and without
// dropout, each followed by the merge kernel that combines the parts of the
// cut items (the online-softmax rescaling of the condensed paper's section 3,
// applied across the parts).
#include "fa_fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_split(const FwdLaunch& a, const FwdGrid& g, int grid, cudaStream_t stream) {
  return a.drop.enabled ? launch_fwd_variant<true, kModeSplit>(a, g, grid, stream)
                        : launch_fwd_variant<false, kModeSplit>(a, g, grid, stream);
}

}  // namespace fa
