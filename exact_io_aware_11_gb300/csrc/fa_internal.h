// Host-side launch descriptions shared by the C-ABI layer and the kernels'
// translation units. Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
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

// How a persistent kernel's work items are shared out over its G CTAs
// (fa_sched.cuh). Items [0, whole) are handed out whole by the plain kernel,
// round r to CTA (r odd ? G-1-c : c) of item r G + c (a snake over an item
// list ordered heaviest first, so that CTAs get similar totals). When
// whole < n_items, the items [whole, n_items) form the tail: a second launch
// of the split kernel, with tail_ctas CTAs, lays them end to end as steps and
// gives each CTA an equal run; whole is then a multiple of G. When
// whole == n_items nothing is split and the last round may be short.
struct SplitPlan {
  int n_items;
  int whole;
  long long tail;  // steps of the tail items
  int tail_ctas;
};

// The part of the tail one CTA runs: steps o0.. of item t0 up to (but not
// including) step o1 of item t1; no tail work when t1 < t0.
struct TailRange {
  int t0, o0, t1, o1;
};

// Which workspace slots hold the parts of each item cut by a split plan, for
// the merge kernels (block i merges item[i] from the slots
// slot[first[i] .. first[i + 1])). Built on the host (fa_sched.cuh).
constexpr int kMaxSplitCtas = 256;
struct MergeTable {
  int n;
  int item[kMaxSplitCtas];
  short first[kMaxSplitCtas + 1];
  short slot[2 * kMaxSplitCtas];
};

// Compile-time variants of the persistent kernels: plain (whole items, dense
// tile ranges), sparse (tile lists from a block mask) and split (the last wave
// cut into parts whose partial results a merge kernel combines).
constexpr int kModePlain = 0, kModeSparse = 1, kModeSplit = 2;

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

// Workspace of a split forward (see fa_sched.cuh): per CTA of the split
// kernel two slots, each holding one partial result of a pair of Q tiles --
// per row the running maximum, the running sum and the unnormalised O
// (fp32). Regions are 256-byte aligned.
struct FwdSplitWorkspace {
  size_t m_off, l_off, o_off, total;
};
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline FwdSplitWorkspace fwd_split_layout(int G, int d) {
  FwdSplitWorkspace w{};
  const size_t slots = 2 * static_cast<size_t>(G);
  w.m_off = 0;
  w.l_off = w.m_off + align256(slots * 256 * 4);
  w.o_off = w.l_off + align256(slots * 256 * 4);
  w.total = w.o_off + align256(slots * 256 * static_cast<size_t>(d) * 4);
  return w;
}

// Extra workspace of a split backward, placed after the regions of
// BwdWorkspace: per slot a partial dV, dK (fp32, 128 key rows x d each, dK
// already multiplied by the scale).
struct BwdSplitWorkspace {
  size_t dkv_off, total;  // offsets from the start of the split area
};
inline BwdSplitWorkspace bwd_split_layout(int G, int d) {
  BwdSplitWorkspace w{};
  const size_t slots = 2 * static_cast<size_t>(G);
  w.dkv_off = 0;
  w.total = w.dkv_off + align256(slots * 2 * 128 * static_cast<size_t>(d) * 4);
  return w;
}

// Sets a kernel's dynamic shared-memory limit once per device: `done` holds
// one bit per device ordinal (a static of the caller, one per kernel).
inline cudaError_t set_smem_once(std::atomic<unsigned long long>& done, const void* kern, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit != 0ull && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0ull) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Forward work: items are pairs of 128-row Q tiles of one (batch, head).
struct FwdGrid {
  int H, N, nqt, npairs, n_items;
  Strides st;  // of q, k, v, o
  const int32_t* kv_len;
  const uint8_t* block_mask;
  SplitPlan plan;
  // split plans only: workspace slots of the partial results
  float* m_part;   // [2G][256] running maximum (log2 units) of each row
  float* l_part;   // [2G][256] running sum of each row
  float* o_part;   // [2G][d / 4][256][4] unnormalised O, column-group major
};

// Backward work: items are 128-key tiles of one (batch, head).
struct BwdGrid {
  int H, N, nt, BH, n_items;
  Strides st;  // of q, k, v, dout, dk, dv
  const int32_t* kv_len;
  const uint8_t* mask;  // block-sparse: uint8 [nt][nt], nonzero = (query tile, key tile) kept
  SplitPlan plan;
  float* dkv_part;  // split plans: [2G][2][d / 4][128][4] partial dV, dK (x scale)
};

struct FwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v;  // 4-D maps (d, N, H, B) with the call's strides, box 64 x 128 x 1 x 1, 128B swizzle
  CUtensorMap tm_o;              // O, the same layout, box 64 x 32 (one softmax warp's rows; d = 64 stores)
  void* split_ws;         // workspace for a split of the last wave, or nullptr
  size_t split_ws_bytes;
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
  CUtensorMap tm_dk, tm_dv;             // the outputs, same form (stores of whole tiles)
  CUtensorMap tm_dqacc;  // fp32 [B*H, Npad, d] accumulator; box 32 x 128 x 1, 128B swizzle
                         // (d = 64) or 16 x 32 x 1, 64B swizzle (d = 128)
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
  float* lse2;     // workspace: fp32 [B*H, Npad]  (-LSE * log2 e; -inf on padding rows)
  float* delta;    // workspace: fp32 [B*H, Npad]  (rowsum(dO * O); 0 on padding rows)
  const uint8_t* block_mask;  // device [nt][nt] (block-sparse backward) or nullptr
  void* split_ws;             // split area of the workspace (BwdSplitWorkspace), or nullptr
  size_t split_ws_bytes;
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

// Forward: plans the work (FwdGrid) and launches the variant it needs.
cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream);
// The forward variants, one translation unit each: plain without and with
// dropout, sparse (block mask) and split (with the merge kernel after it).
cudaError_t launch_fwd_plain(const FwdLaunch& a, const FwdGrid& g, int grid, cudaStream_t stream);
cudaError_t launch_fwd_plain_dropout(const FwdLaunch& a, const FwdGrid& g, int grid,
                                     cudaStream_t stream);
cudaError_t launch_fwd_sparse(const FwdLaunch& a, const FwdGrid& g, int grid, cudaStream_t stream);
cudaError_t launch_fwd_split(const FwdLaunch& a, const FwdGrid& g, int grid, const MergeTable& m,
                             cudaStream_t stream);
// The backward main kernel's variants, one translation unit each: plain
// (in fa_bwd.cu), sparse, plain with dropout, sparse with dropout, and split
// (with or without dropout; with the merge kernel after it).
cudaError_t launch_bwd_main_plain(const BwdLaunch& a, const BwdGrid& g, int grid, cudaStream_t stream);
cudaError_t launch_bwd_main_sparse(const BwdLaunch& a, const BwdGrid& g, int grid,
                                   cudaStream_t stream);
cudaError_t launch_bwd_main_dropout(const BwdLaunch& a, const BwdGrid& g, int grid,
                                    cudaStream_t stream);
cudaError_t launch_bwd_main_dropout_sparse(const BwdLaunch& a, const BwdGrid& g, int grid,
                                           cudaStream_t stream);
cudaError_t launch_bwd_main_split(const BwdLaunch& a, const BwdGrid& g, int grid,
                                  const MergeTable& m, cudaStream_t stream);
// Writes the keep decisions Z (1 = kept) of a.drop for [B*H, N, N] as bytes.
cudaError_t launch_dropout_mask(const DropoutParams& drop, int BH, int N, uint8_t* keep,
                                cudaStream_t stream);
// Backward stages (bit set): preprocess, main kernel, dQ conversion.
constexpr int kBwdStagePre = 1, kBwdStageMain = 2, kBwdStageConvert = 4, kBwdStageAll = 7;
cudaError_t launch_bwd(const BwdLaunch& a, int stages, cudaStream_t stream);
cudaError_t launch_wait_selftest(int* status, long long limit_cycles, cudaStream_t stream);

}  // namespace fa
