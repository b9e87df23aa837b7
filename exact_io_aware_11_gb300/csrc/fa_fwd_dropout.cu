// Forward pass with fused dropout (dense, causal, key-padded): the DROP
// variants of the fused forward kernel (fa_fwd_kernel.cuh), and a kernel that
// writes the keep decisions themselves, for callers that want to inspect or
// reuse the mask.
//
// Dropout is one of the stages of the attention computation that the method
// fuses into its single kernel, and the memory it needs does not depend on it
// (FlashAttention aggregator page, GPT-2 time-breakdown figure, which sets the
// separate matmul, mask, softmax, dropout and matmul steps against one fused
// kernel). The keep decisions come from a counter-based generator
// (fa_philox.cuh), so neither pass stores them.
#include "fa_fwd_kernel.cuh"

namespace fa {
namespace {

// keep[bh][i][j] = 1 if element (bh, i, j) is kept, else 0; one thread per
// (bh, i, 16-key group), grid-stride.
__global__ void __launch_bounds__(256) dropout_mask_kernel(DropoutParams dp, int BH, int N,
                                                           uint8_t* __restrict__ keep) {
  grid_dep_wait();
  grid_dep_launch();
  const int groups = (N + 15) >> 4;
  const long long total = static_cast<long long>(BH) * N * groups;
  const uint32_t t = dp.thresh4 & 0xffu;
  for (long long x = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; x < total;
       x += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int g = static_cast<int>(x % groups);
    const long long ri = x / groups;  // bh * N + i
    const int i = static_cast<int>(ri % N);
    const int bh = static_cast<int>(ri / N);
    const uint4 r = philox4x32_10(static_cast<uint32_t>(g), static_cast<uint32_t>(i),
                                  static_cast<uint32_t>(bh), dp.offset, dp.k0, dp.k1);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    uint8_t* dst = keep + ri * N + 16LL * g;
    const int n = min(16, N - 16 * g);
    for (int e = 0; e < n; ++e) dst[e] = ((w[e >> 2] >> (8 * (e & 3))) & 0xffu) >= t ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_fwd_plain_dropout(const FwdLaunch& a, const FwdGrid& g, int grid,
                                     cudaStream_t stream) {
  return launch_fwd_variant<true, kModePlain>(a, g, grid, stream);
}

cudaError_t launch_dropout_mask(const DropoutParams& drop, int BH, int N, uint8_t* keep,
                                cudaStream_t stream) {
  const long long threads = static_cast<long long>(BH) * N * ((N + 15) / 16);
  long long blocks = (threads + 255) / 256;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(dropout_mask_kernel, dim3(static_cast<unsigned>(blocks < 1 ? 1 : blocks)),
                    dim3(256), 0, stream, drop, BH, N, keep);
}

}  // namespace fa
