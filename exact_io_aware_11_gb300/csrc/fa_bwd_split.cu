// Backward main kernel with the last wave of key-tile items split over every
// SM: the SPLIT variants of fa_bwd_kernel.cuh, with and without dropout, which
// run the tail of a split plan after the plain kernel has run its whole
// rounds, each followed by the merge kernel that sums the parts' dK and dV.
#include "fa_bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_main_split(const BwdLaunch& a, const BwdGrid& g, int grid,
                                  const MergeTable& m, cudaStream_t stream) {
  const bool causal = a.causal != 0, drop = a.drop.enabled != 0;
  if (a.d == 64) {
    if (drop)
      return causal ? launch_bwd_tail<64, true, true>(a, g, grid, m, stream)
                    : launch_bwd_tail<64, false, true>(a, g, grid, m, stream);
    return causal ? launch_bwd_tail<64, true, false>(a, g, grid, m, stream)
                  : launch_bwd_tail<64, false, false>(a, g, grid, m, stream);
  }
  if (drop)
    return causal ? launch_bwd_tail<128, true, true>(a, g, grid, m, stream)
                  : launch_bwd_tail<128, false, true>(a, g, grid, m, stream);
  return causal ? launch_bwd_tail<128, true, false>(a, g, grid, m, stream)
                : launch_bwd_tail<128, false, false>(a, g, grid, m, stream);
}

}  // namespace fa
