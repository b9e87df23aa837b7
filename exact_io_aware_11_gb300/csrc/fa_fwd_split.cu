// Forward with the last wave of work items split over every SM: the SPLIT
// variants of the fused forward kernel (fa_fwd_kernel.cuh), with and without
// dropout, which run the tail of a split plan after the plain kernel has run
// its whole rounds, each followed by the merge kernel that combines the parts
// of the cut items (the online-softmax rescaling of the condensed paper's
// section 3, applied across the parts).
#include "fa_fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_split(const FwdLaunch& a, const FwdGrid& g, int grid, const MergeTable& m,
                             cudaStream_t stream) {
  const bool causal = a.causal != 0, drop = a.drop.enabled != 0;
  if (a.d == 64) {
    if (drop)
      return causal ? launch_fwd_tail<64, true, true>(a, g, grid, m, stream)
                    : launch_fwd_tail<64, false, true>(a, g, grid, m, stream);
    return causal ? launch_fwd_tail<64, true, false>(a, g, grid, m, stream)
                  : launch_fwd_tail<64, false, false>(a, g, grid, m, stream);
  }
  if (drop)
    return causal ? launch_fwd_tail<128, true, true>(a, g, grid, m, stream)
                  : launch_fwd_tail<128, false, true>(a, g, grid, m, stream);
  return causal ? launch_fwd_tail<128, true, false>(a, g, grid, m, stream)
                : launch_fwd_tail<128, false, false>(a, g, grid, m, stream);
}

}  // namespace fa
