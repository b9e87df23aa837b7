// Backward main kernel with the last wave of key-tile items split over every
// SM: the SPLIT variants of fa_bwd_kernel.cuh, with and without dropout, each
// followed by the merge kernel that sums the parts' dK and dV.
#include "fa_bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_main_split(const BwdLaunch& a, const BwdGrid& g, int grid,
                                  cudaStream_t stream) {
  return a.drop.enabled ? launch_bwd_main_variant<kModeSplit, true>(a, g, grid, stream)
                        : launch_bwd_main_variant<kModeSplit, false>(a, g, grid, stream);
}

}  // namespace fa
