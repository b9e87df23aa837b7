// Forward pass: plans the work of a call (which work items, whether the last
// wave is split) and launches the variant of the fused forward kernel
// (fa_fwd_kernel.cuh) it needs. This unit compiles the plain variants
// without dropout; the others have units of their own (fa_fwd_dropout.cu,
// fa_fwd_sparse.cu, fa_fwd_split.cu) so that they compile in parallel.
#include "fa_fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream) {
  FwdGrid g{};
  g.H = a.H;
  g.N = a.N;
  g.nqt = (a.N + kBlock - 1) / kBlock;
  g.npairs = (g.nqt + 1) / 2;
  g.n_items = a.B * a.H * g.npairs;
  g.kv_len = a.kv_len;
  g.block_mask = a.block_mask;
  g.st = a.st;
  const int sms = sm_count();
  const FwdSplitWorkspace ws = fwd_split_layout(sms, a.d);
  const bool allowed = a.split_ws != nullptr && a.split_ws_bytes >= ws.total && a.kv_len == nullptr &&
                       a.block_mask == nullptr;
  g.plan = plan_fwd(a.B, a.H, a.N, a.d, a.causal != 0, sms, allowed);
  if (g.plan.whole < g.plan.n_items) {
    // Whole rounds on the plain kernel, then the tail on the split kernel.
    uint8_t* w = static_cast<uint8_t*>(a.split_ws);
    g.m_part = reinterpret_cast<float*>(w + ws.m_off);
    g.l_part = reinterpret_cast<float*>(w + ws.l_off);
    g.o_part = reinterpret_cast<float*>(w + ws.o_off);
    if (g.plan.whole > 0) {
      const cudaError_t e = a.drop.enabled ? launch_fwd_plain_dropout(a, g, sms, stream)
                                           : launch_fwd_plain(a, g, sms, stream);
      if (e != cudaSuccess) return e;
    }
    const int nqt = g.nqt, npairs = g.npairs, BH = g.n_items / g.npairs;
    const bool causal = a.causal != 0;
    const MergeTable m = build_merge_table(
        g.plan, [&](int k) { return fwd_item_steps(nqt, npairs, BH, causal, k); });
    return launch_fwd_split(a, g, g.plan.tail_ctas, m, stream);
  }
  if (a.block_mask != nullptr) {
    // d = 64: items pair the same Q tile of two heads, which keep the same
    // block-mask row, so both Q slots visit every K/V step of the item.
    if (a.d == 64) g.n_items = a.B * ((a.H + 1) / 2) * g.nqt;
    g.plan = SplitPlan{g.n_items, g.n_items, 0, 0};  // every item whole
    return launch_fwd_sparse(a, g, min(g.n_items, sms), stream);
  }
  const int grid = min(g.n_items, sms);
  if (a.drop.enabled) return launch_fwd_plain_dropout(a, g, grid, stream);
  return launch_fwd_plain(a, g, grid, stream);
}

cudaError_t launch_fwd_plain(const FwdLaunch& a, const FwdGrid& g, int grid, cudaStream_t stream) {
  return launch_fwd_variant<false, kModePlain>(a, g, grid, stream);
}

}  // namespace fa
