// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory -- code that runs where cudaMalloc is forbidden or unavailable, such
// as inside a CUDA-graph capture that may not allocate, under a framework
// that owns every allocation through its own pool, or in a plugin that is
// handed tensors but no allocator. Such a caller cannot provide the
// backward's workspace, so this entry point uses a fixed scratch buffer that
// lives in the library itself.
//
// The scratch is a file-scope __device__ array: every GPU that loads the
// library holds FA_NOALLOC_SCRATCH_BYTES of it until the process exits. Host
// code cannot use the array's name as a device address (on the host it names
// a stand-in), so the first call on each device looks up the real address
// with cudaGetSymbolAddress while that device is current and caches it.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (nullptr on error).
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, int causal, float scale,
                              const int32_t* kv_len, struct CUstream_st* stream) {
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (need == 0) {
    // invalid sizes: let fa_bwd report them exactly as it would
    return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, scale, kv_len, nullptr,
                  0, stream);
  }
  if (need > static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES)) return FA_ERR_INVALID_ARG;
  // Missing tensors are reported as fa_bwd reports them, before the scratch
  // lookup touches the device.
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  void* scratch = scratch_on_current_device();
  if (scratch == nullptr) return FA_ERR_CUDA;
  // fa_bwd ignores the workspace's previous contents: its first stage
  // rewrites every part of the scratch that the later stages read.
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, scale, kv_len, scratch,
                static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES), stream);
}
