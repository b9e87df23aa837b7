// Host-side launch descriptions shared by the C-ABI layer and the kernels'
// translation units. Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fa {

// Budget of one bounded device wait, in SM clock cycles (about a second).
constexpr long long kWaitLimitCycles = 2000000000LL;

// Rows of one Q tile and one K/V tile (the 128 x 128 block of the method).
constexpr int kBlock = 128;

// Element strides of the [B, H, N, d] tensors of one call (q, k, v, o, dout,
// dq, dk, dv share them): element (b, h, n, c) sits at b*b + h*h + n*n + c.
// [B, H, N, d] row-major is {H*N*d, N*d, d}; [B, N, H, d] is {N*H*d, d, H*d}.
// When head and batch merge into one problem axis bh = b*H + h of stride
// s_bh above the rows ([B, H, N, d] row-major, padded rows), the tensor maps
// are 3-D (d, N, B*H) and `merged` is set. Otherwise they are 4-D: d, then the
// row, head and batch axes in order of increasing stride, and pn, ph, pb give
// the positions (0..2 among dimensions 1..3) of those coordinates.
struct Strides {
  long long b, h, n;
  int pn, ph, pb;
  int merged;
  long long bh, n_map;  // merged maps: strides of the bh and row axes
};

// Coordinates (dimensions 1..3) of row n of head h in batch b.
__device__ __forceinline__ void row_coords(const Strides& s, int n, int h, int b, int& y0, int& y1,
                                           int& y2) {
  y0 = s.pn == 0 ? n : (s.ph == 0 ? h : b);
  y1 = s.pn == 1 ? n : (s.ph == 1 ? h : b);
  y2 = s.pn == 2 ? n : (s.ph == 2 ? h : b);
}

// Offset in elements of row n of problem bh = b*H + h.
__host__ __device__ __forceinline__ long long row_offset(const Strides& s, int H, int bh, int n) {
  return static_cast<long long>(bh / H) * s.b + static_cast<long long>(bh % H) * s.h +
         static_cast<long long>(n) * s.n;
}

// Dropout on the attention probabilities (inverted: kept entries are scaled
// by 1 / (1 - p')). Element (b, h, i, j) draws byte j mod 16 of the
// Philox4x32-10 block at counter (j / 16, i, b*H + h, offset) under key
// (k0, k1); it is kept iff that byte >= thresh (p' = thresh / 256).
struct DropoutParams {
  uint32_t k0, k1;    // seed low / high 32 bits
  uint32_t offset;    // fourth counter word
  uint32_t thresh4;   // thresh replicated into the four bytes
  float rescale;      // 256 / (256 - thresh)
  int enabled;        // 0: no dropout (the other fields are ignored)
};

struct FwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v;  // 4-D maps (d, N, H, B) with the call's strides, box 64 x 128 x 1 x 1, 128B swizzle
  void* o;
  float* lse;
  int B, H, N, d;
  Strides st;
  int causal;
  float scale;
  const int32_t* kv_len;      // device [B] or nullptr
  const uint8_t* block_mask;  // device [nb, nb] or nullptr
  DropoutParams drop;
  int* status;
  long long wait_limit;
};

struct BwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // as above (4-D, the call's strides)
  CUtensorMap tm_dqacc;  // fp32 [B*H, Npad, d] accumulator, box 32 x 128 x 1, 128B swizzle
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  int B, H, N, d;
  Strides st;
  int causal;
  float scale;
  const int32_t* kv_len;
  float* dq_acc;   // workspace: fp32 [B*H, Npad, d]
  float* lse2;     // workspace: fp32 [B*H, Npad]  (LSE * log2 e; +inf on padding rows)
  float* delta;    // workspace: fp32 [B*H, Npad]  (rowsum(dO * O); 0 on padding rows)
  const uint8_t* block_mask;  // device [nt][nt] (block-sparse backward) or nullptr
  DropoutParams drop;
  int* status;
  long long wait_limit;
};

// Workspace carving shared by fa_bwd_workspace_bytes and fa_bwd.
struct BwdWorkspace {
  size_t dq_off, lse2_off, delta_off, total;
};
BwdWorkspace bwd_workspace_layout(int B, int H, int N, int d);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Launches `kern` with programmatic dependent launch allowed: the grid may be
// set up while the previous kernel on the stream is still running, and every
// kernel of this library waits (griddepcontrol.wait) for its predecessor's
// completion before it touches global memory, then lets its own successor be
// set up (griddepcontrol.launch_dependents). This hides the launch gap between
// the kernels of a forward + backward pass.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream);
// Variants compiled in their own translation units: the forward kernel with
// dropout (a.drop.enabled != 0); the backward main kernel with a block mask,
// with dropout, and with both.
cudaError_t launch_fwd_dropout(const FwdLaunch& a, cudaStream_t stream);
cudaError_t launch_bwd_main_sparse(const BwdLaunch& a, cudaStream_t stream);
cudaError_t launch_bwd_main_dropout(const BwdLaunch& a, cudaStream_t stream);
cudaError_t launch_bwd_main_dropout_sparse(const BwdLaunch& a, cudaStream_t stream);
// Writes the keep decisions Z (1 = kept) of a.drop for [B*H, N, N] as bytes.
cudaError_t launch_dropout_mask(const DropoutParams& drop, int BH, int N, uint8_t* keep,
                                cudaStream_t stream);
// Backward stages (bit set): preprocess, main kernel, dQ conversion.
constexpr int kBwdStagePre = 1, kBwdStageMain = 2, kBwdStageConvert = 4, kBwdStageAll = 7;
cudaError_t launch_bwd(const BwdLaunch& a, int stages, cudaStream_t stream);
cudaError_t launch_wait_selftest(int* status, long long limit_cycles, cudaStream_t stream);

}  // namespace fa
