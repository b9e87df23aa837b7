// Backward pass of exact attention: the preprocess and dQ-conversion stages,
// the dense (causal or not, key-padded or not) variants of the main kernel
// (fa_bwd_kernel.cuh) and the watchdog self-test kernel. The block-sparse and
// dropout variants of the main kernel are compiled in fa_bwd_sparse.cu,
// fa_bwd_dropout.cu and fa_bwd_dropout_sparse.cu.
#include "fa_bwd_kernel.cuh"

namespace fa {
namespace {

__global__ void wait_selftest_kernel(int* status, long long limit) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Watchdog wd{limit, status, &abort_flag};
  // Nothing ever arrives on `bar`: the bounded wait must give up and report.
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, wd);
}

int grid_for(long long threads) {
  long long blocks = (threads + 255) / 256;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

template <int D, bool CAUSAL>
cudaError_t launch_bwd_t(const BwdLaunch& a, int stages, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int nt = (a.N + kBlock - 1) / kBlock;
  const int Npad = nt * kBlock;
  cudaError_t e = cudaSuccess;
  if (stages & kBwdStagePre) {
    e = launch_pdl(bwd_pre_kernel<D>, dim3(grid_for(static_cast<long long>(BH) * Npad * (D / 8))),
                   dim3(256), 0, stream, a.o, a.dout, a.lse, a.lse2, a.delta, a.dq_acc, BH, a.N,
                   Npad, a.st, a.H);
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdStageMain) {
    if (a.drop.enabled)
      e = launch_bwd_main_dropout(a, stream);
    else if (a.block_mask != nullptr)
      e = launch_bwd_main_sparse(a, stream);
    else
      e = launch_bwd_main_t<D, CAUSAL, false, false>(a, stream);
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdStageConvert) {
    e = launch_pdl(dq_convert_kernel<D>, dim3(grid_for(static_cast<long long>(BH) * a.N * (D / 8))),
                   dim3(256), 0, stream, a.dq_acc, a.dq, BH, a.N, Npad, a.st, a.H);
  }
  return e;
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunch& a, int stages, cudaStream_t stream) {
  const bool causal = a.causal != 0;
  if (a.d == 64)
    return causal ? launch_bwd_t<64, true>(a, stages, stream) : launch_bwd_t<64, false>(a, stages, stream);
  return causal ? launch_bwd_t<128, true>(a, stages, stream) : launch_bwd_t<128, false>(a, stages, stream);
}

cudaError_t launch_wait_selftest(int* status, long long limit_cycles, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_cycles);
  return cudaGetLastError();
}

}  // namespace fa
