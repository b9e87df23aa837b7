// Backward pass of exact attention: the preprocess and dQ-conversion stages,
// the planning of the main stage, the plain (dense, causal or not, key-padded
// or not) variants of the main kernel (fa_bwd_kernel.cuh) and the watchdog
// self-test kernel. The block-sparse, dropout and split variants of the main
// kernel are compiled in fa_bwd_sparse.cu, fa_bwd_dropout.cu,
// fa_bwd_dropout_sparse.cu and fa_bwd_split.cu.
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

// Blocks of 256 threads for a grid-stride kernel over `threads` work items:
// at most 16 resident blocks per SM.
int grid_for(long long threads) {
  long long blocks = (threads + 255) / 256;
  const long long cap = static_cast<long long>(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

template <int D>
cudaError_t launch_pre(const BwdLaunch& a, int BH, int Npad, cudaStream_t stream) {
  return launch_pdl(bwd_pre_kernel<D>, dim3(grid_for(static_cast<long long>(BH) * Npad * (D / 8))),
                    dim3(256), 0, stream, a.o, a.dout, a.lse, a.lse2, a.delta, a.dq_acc, BH, a.N,
                    Npad, a.st, a.H);
}

template <int D>
cudaError_t launch_convert(const BwdLaunch& a, int BH, int Npad, cudaStream_t stream) {
  return launch_pdl(dq_convert_kernel<D>, dim3(grid_for(static_cast<long long>(BH) * a.N * (D / 8))),
                    dim3(256), 0, stream, a.dq_acc, a.dq, BH, a.N, Npad, a.st, a.H);
}

// The main stage: plans the work (which items, whether the last wave is
// split) and launches the variant it needs.
cudaError_t launch_main(const BwdLaunch& a, cudaStream_t stream) {
  BwdGrid g{};
  g.H = a.H;
  g.N = a.N;
  g.nt = (a.N + kBlock - 1) / kBlock;
  g.BH = a.B * a.H;
  g.n_items = g.BH * g.nt;
  g.kv_len = a.kv_len;
  g.mask = a.block_mask;
  g.st = a.st;
  const int sms = sm_count();
  const BwdSplitWorkspace ws = bwd_split_layout(sms, a.d);
  const bool allowed = a.split_ws != nullptr && a.split_ws_bytes >= ws.total && a.kv_len == nullptr &&
                       a.block_mask == nullptr;
  g.plan = plan_bwd(a.B, a.H, a.N, a.d, a.causal != 0, sms, allowed);
  if (g.plan.whole < g.plan.n_items) {
    // Whole rounds on the plain kernel, then the tail on the split kernel.
    g.dkv_part = reinterpret_cast<float*>(static_cast<uint8_t*>(a.split_ws) + ws.dkv_off);
    if (g.plan.whole > 0) {
      const cudaError_t e = a.drop.enabled ? launch_bwd_main_dropout(a, g, sms, stream)
                                           : launch_bwd_main_plain(a, g, sms, stream);
      if (e != cudaSuccess) return e;
    }
    const int nt = g.nt, BH = g.BH;
    const bool causal = a.causal != 0;
    const MergeTable m =
        build_merge_table(g.plan, [&](int k) { return bwd_item_steps(nt, BH, causal, k); });
    return launch_bwd_main_split(a, g, g.plan.tail_ctas, m, stream);
  }
  const int grid = min(g.n_items, sms);
  if (a.block_mask != nullptr)
    return a.drop.enabled ? launch_bwd_main_dropout_sparse(a, g, grid, stream)
                          : launch_bwd_main_sparse(a, g, grid, stream);
  if (a.drop.enabled) return launch_bwd_main_dropout(a, g, grid, stream);
  return launch_bwd_main_plain(a, g, grid, stream);
}

}  // namespace

cudaError_t launch_bwd_main_plain(const BwdLaunch& a, const BwdGrid& g, int grid, cudaStream_t stream) {
  return launch_bwd_main_variant<kModePlain, false>(a, g, grid, stream);
}

cudaError_t launch_bwd(const BwdLaunch& a, int stages, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const int Npad = (a.N + kBlock - 1) / kBlock * kBlock;
  cudaError_t e = cudaSuccess;
  if (stages & kBwdStagePre) {
    e = a.d == 64 ? launch_pre<64>(a, BH, Npad, stream) : launch_pre<128>(a, BH, Npad, stream);
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdStageMain) {
    e = launch_main(a, stream);
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdStageConvert)
    e = a.d == 64 ? launch_convert<64>(a, BH, Npad, stream) : launch_convert<128>(a, BH, Npad, stream);
  return e;
}

cudaError_t launch_wait_selftest(int* status, long long limit_cycles, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_cycles);
  return cudaGetLastError();
}

}  // namespace fa
