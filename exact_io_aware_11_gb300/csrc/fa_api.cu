// C-ABI of libfa.so (declared in include/fa.h): argument validation, TMA
// descriptor encoding, workspace carving and dispatch to the kernels on the
// caller's stream. Holds no state beyond one device-side status word per
// device and a cached driver entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "fa_sched.cuh"

namespace fa {

__device__ int g_status_word;

namespace {

constexpr int kMaxDevices = 64;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Per-device: address of the status word and whether the device is sm_103.
struct DeviceInfo {
  int* status = nullptr;
  int supported = -1;  // -1 unknown
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mu;

int current_device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_devices_mu);
  DeviceInfo& info = g_devices[dev];
  if (info.supported < 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    info.supported = (major == 10 && minor == 3) ? 1 : 0;
  }
  if (!info.supported) return FA_ERR_UNSUPPORTED;
  if (info.status == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return FA_ERR_CUDA;
    info.status = static_cast<int*>(p);
  }
  *out = info;
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Validates the element strides (sb, sh, sn) of [B, H, N, d] tensors and
// orders the row, head and batch axes by increasing stride for the tensor
// maps. Requirements: strides >= 0 and multiples of 8 elements (16 bytes, the
// tensor-map rule), below 2^36, and rows that do not overlap -- sorted by
// stride, the smallest is >= d and each next one >= the previous stride times
// its extent. An axis of extent 1 is placed last whatever its stride.
bool make_strides(int B, int H, int N, int d, long long sb, long long sh, long long sn,
                  Strides* out) {
  const long long lim = 1LL << 36;
  const long long st[3] = {sn, sh, sb};
  const long long ext[3] = {N, H, B};
  long long top = d;
  for (int a = 0; a < 3; ++a) {
    if (st[a] < 0 || st[a] >= lim || (st[a] & 7)) return false;
    if (ext[a] > 1 && st[a] > lim / ext[a]) return false;  // span beyond 2^36 elements
    if (ext[a] > 1 && st[a] * ext[a] > top) top = st[a] * ext[a];
  }
  if (top >= lim) return false;
  long long key[3];
  int order[3] = {0, 1, 2};  // axes sorted by normalised stride (stable)
  for (int a = 0; a < 3; ++a) key[a] = ext[a] > 1 ? st[a] : top;
  for (int x = 0; x < 3; ++x)
    for (int y = 0; y + 1 < 3 - x; ++y)
      if (key[order[y]] > key[order[y + 1]]) {
        const int t = order[y];
        order[y] = order[y + 1];
        order[y + 1] = t;
      }
  long long need = d;  // the smallest stride a row may have without overlap
  for (int k = 0; k < 3; ++k) {
    const int a = order[k];
    if (ext[a] == 1) continue;
    if (key[a] < need) return false;
    need = key[a] * ext[a];
  }
  out->n = sn;
  out->h = sh;
  out->b = sb;
  for (int k = 0; k < 3; ++k) {
    if (order[k] == 0) out->pn = k;
    if (order[k] == 1) out->ph = k;
    if (order[k] == 2) out->pb = k;
  }
  // Head and batch merge into one axis bh = b*H + h when one stride serves
  // both (H = 1, B = 1, or sb = H * sh) and it lies above the rows.
  const long long sn_eff = N > 1 ? sn : d;
  long long sbh = -1;
  if (static_cast<long long>(B) * H == 1)
    sbh = static_cast<long long>(N) * sn_eff;
  else if (H == 1)
    sbh = sb;
  else if (B == 1 || sb == static_cast<long long>(H) * sh)
    sbh = sh;
  out->merged = (sbh >= 0 && sn_eff >= d && sbh >= static_cast<long long>(N) * sn_eff) ? 1 : 0;
  out->bh = sbh;
  out->n_map = sn_eff;
  return true;
}

// The row-major [B, H, N, d] strides (false if the tensor is too large).
bool dense_strides(int B, int H, int N, int d, Strides* s) {
  return make_strides(B, H, N, d, static_cast<long long>(H) * N * d, static_cast<long long>(N) * d,
                      d, s);
}

// Whether two bf16 [B, H, N, d] tensors with the same strides `s` share an
// element, their bases `a` and `b` (16-byte aligned) being given. Row starts
// form the set P = {i_b sb + i_h sh + i_n sn}; the tensors overlap iff the
// base difference (in elements) lies within d - 1 of some difference of two
// row starts, sum_a k_a s_a with |k_a| < extent_a. The axes' strides nest
// (each at least the one below times its extent, as make_strides requires),
// so for every axis, largest stride first, only the coefficients next to
// delta / stride can lead to a hit, and a search over those is exact. This
// accepts interleaved views such as q, k, v of one packed [B, N, 3, H, d]
// buffer, which a comparison of address spans would reject.
bool strided_overlap(const void* a, const void* b, int B, int H, int N, int d, const Strides& s) {
  const long long diff = static_cast<long long>(reinterpret_cast<uintptr_t>(b)) -
                         static_cast<long long>(reinterpret_cast<uintptr_t>(a));
  if (diff % 2 != 0) return true;  // not on the same element grid: be conservative
  const long long delta = diff / 2;
  long long st[3] = {s.n, s.h, s.b}, ext[3] = {N, H, B};
  // axes of extent 1 never step; sort the rest by stride, largest first
  int ord[3] = {0, 1, 2};
  for (int x = 0; x < 3; ++x)
    for (int y = 0; y + 1 < 3 - x; ++y)
      if (st[ord[y]] < st[ord[y + 1]]) {
        const int t = ord[y];
        ord[y] = ord[y + 1];
        ord[y + 1] = t;
      }
  struct Rec {
    static bool hit(const long long* st, const long long* ext, const int* ord, int lvl, long long r,
                    int d) {
      if (lvl == 3) return r > -d && r < d;
      const int ax = ord[lvl];
      if (ext[ax] <= 1 || st[ax] == 0) return hit(st, ext, ord, lvl + 1, r, d);
      const long long lim = ext[ax] - 1;
      long long k0 = r / st[ax];
      for (long long k = k0 - 1; k <= k0 + 1; ++k) {
        if (k < -lim || k > lim) continue;
        if (hit(st, ext, ord, lvl + 1, r - k * st[ax], d)) return true;
      }
      return false;
    }
  };
  return Rec::hit(st, ext, ord, 0, delta, d);
}

// Bytes from the first to one past the last element of a tensor with strides s.
size_t span_bytes(int B, int H, int N, int d, const Strides& s, size_t elem) {
  return static_cast<size_t>((B - 1) * s.b + (H - 1) * s.h + (N - 1) * s.n + d) * elem;
}

// A bf16 [B, H, N, d] tensor with strides `st` as a tensor map: 3-D (d, N,
// B*H) when st.merged, else 4-D with dimension 0 = d and dimensions 1..3 the
// row, head and batch axes in the order st gives; box = 64 columns (128 bytes)
// x box_rows rows (x 1 x 1), 128-byte swizzle, zero fill outside the tensor
// (ragged N); narrow = true: 32 columns (64 bytes) with the 64-byte swizzle.
bool encode_rows(CUtensorMap* map, const void* base, int B, int H, int N, int d,
                 const Strides& st, int box_rows = kBlock, bool narrow = false) {
  const cuuint32_t box_x = narrow ? 32u : 64u;
  const CUtensorMapSwizzle swz = narrow ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  if (st.merged) {  // 3-D (d, N, B*H)
    const cuuint64_t dims3[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                 static_cast<cuuint64_t>(B) * static_cast<cuuint64_t>(H)};
    const cuuint64_t strides3[2] = {static_cast<cuuint64_t>(st.n_map) * 2,
                                    static_cast<cuuint64_t>(st.bh) * 2};
    const cuuint32_t box3[3] = {box_x, static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t estr3[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims3, strides3,
              box3, estr3, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4];
  dims[0] = static_cast<cuuint64_t>(d);
  box[0] = box_x;
  const long long ext[3] = {N, H, B};
  const int pos[3] = {st.pn, st.ph, st.pb};
  const long long sv[3] = {st.n, st.h, st.b};
  long long top = d;  // the stride an axis of extent 1 is given (it is never stepped)
  for (int a = 0; a < 3; ++a)
    if (ext[a] > 1 && sv[a] * ext[a] > top) top = sv[a] * ext[a];
  for (int a = 0; a < 3; ++a) {
    dims[1 + pos[a]] = static_cast<cuuint64_t>(ext[a]);
    strides[pos[a]] = static_cast<cuuint64_t>(ext[a] > 1 ? sv[a] : top) * 2;
    box[1 + pos[a]] = a == 0 ? static_cast<cuuint32_t>(box_rows) : 1u;
  }
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [B*H, rows, d] as a 3-D tensor map; box = 32 columns (128 bytes) x 128
// rows x 1 head, 128-byte swizzle (the backward's dQ accumulator).
bool encode_f32_rows(CUtensorMap* map, const void* base, int BH, int rows, int d) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                 static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(d) * 4};
  // d = 64: 128 rows x 32 columns (128-byte rows, 128-byte swizzle); d = 128:
  // 32 rows x 16 columns (64-byte rows, 64-byte swizzle), one warp's box.
  const bool narrow = d == 128;
  const cuuint32_t box[3] = {narrow ? 16u : 32u, narrow ? 32u : static_cast<cuuint32_t>(kBlock), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            narrow ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The kernels count work items (B*H*ceil(N/128)), problems (B*H) and padded
// rows (N rounded up to 128) in 32-bit integers.
bool sizes_fit_int(int B, int H, int N) {
  if (N > INT_MAX - (kBlock - 1)) return false;
  const long long tiles = (static_cast<long long>(N) + kBlock - 1) / kBlock;
  return static_cast<long long>(B) * H * tiles <= INT_MAX;
}

int check_common(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (B > 65535 || H > 65535 || !sizes_fit_int(B, H, N)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Dropout parameters from the caller's probability, seed and offset: the drop
// threshold t = round(256 p) (at most 255) on one random byte per element,
// kept entries scaled by 256 / (256 - t). Returns false for p outside [0, 1).
bool make_dropout(float p, uint64_t seed, uint32_t offset, DropoutParams* out) {
  if (!std::isfinite(p) || p < 0.f || p >= 1.f) return false;
  int t = static_cast<int>(std::floor(256.0 * static_cast<double>(p) + 0.5));
  if (t > 255) t = 255;
  out->k0 = static_cast<uint32_t>(seed & 0xffffffffu);
  out->k1 = static_cast<uint32_t>(seed >> 32);
  out->offset = offset;
  out->thresh4 = static_cast<uint32_t>(t) * 0x01010101u;
  out->rescale = static_cast<float>(256.0 / (256.0 - t));
  out->enabled = 1;
  return true;
}

size_t tensor_bytes(int B, int H, int N, int d, size_t elem) {
  return static_cast<size_t>(B) * H * N * d * elem;
}

int fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int N, int d, int causal, float scale, const int32_t* kv_len,
               const uint8_t* block_mask, cudaStream_t stream,
               const DropoutParams* drop = nullptr, const Strides* strides = nullptr,
               void* split_ws = nullptr, size_t split_ws_bytes = 0) {
  int st = check_common(B, H, N, d, scale);
  if (st != FA_OK) return st;
  Strides lay{};
  if (strides)
    lay = *strides;
  else if (!dense_strides(B, H, N, d, &lay))
    return FA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return FA_ERR_INVALID_ARG;
  if (split_ws != nullptr && !aligned16(split_ws)) return FA_ERR_INVALID_ARG;
  const size_t tb = span_bytes(B, H, N, d, lay, 2), lb = tensor_bytes(B, H, N, 1, 4);
  const void* ins[3] = {q, k, v};
  for (const void* in : ins)
    if (strided_overlap(o, in, B, H, N, d, lay) || overlaps(lse, lb, in, tb) ||
        (split_ws && overlaps(split_ws, split_ws_bytes, in, tb)))
      return FA_ERR_INVALID_ARG;
  if (overlaps(o, tb, lse, lb)) return FA_ERR_INVALID_ARG;
  if (split_ws && (overlaps(split_ws, split_ws_bytes, o, tb) || overlaps(split_ws, split_ws_bytes, lse, lb)))
    return FA_ERR_INVALID_ARG;
  DeviceInfo dev;
  st = current_device_info(&dev);
  if (st != FA_OK) return st;
  FwdLaunch a;
  std::memset(&a, 0, sizeof(a));
  if (!encode_rows(&a.tm_q, q, B, H, N, d, lay) || !encode_rows(&a.tm_k, k, B, H, N, d, lay) ||
      !encode_rows(&a.tm_v, v, B, H, N, d, lay) || !encode_rows(&a.tm_o, o, B, H, N, d, lay, 32))
    return FA_ERR_CUDA;
  a.st = lay;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  a.kv_len = kv_len;
  a.block_mask = block_mask;
  if (drop) a.drop = *drop;
  a.split_ws = split_ws;
  a.split_ws_bytes = split_ws ? split_ws_bytes : 0;
  a.status = dev.status;
  a.wait_limit = kWaitLimitCycles;
  return launch_fwd(a, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

struct BwdPtrs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  void* ws;
};

// Validates and launches the requested backward stages. Pointers a stage does
// not use may be NULL; every pointer a stage uses must be non-NULL.
int bwd_common(int stages, const BwdPtrs& p, int B, int H, int N, int d, int causal, float scale,
               const int32_t* kv_len, size_t workspace_bytes, cudaStream_t stream,
               const uint8_t* block_mask = nullptr, const DropoutParams* drop = nullptr,
               const Strides* strides = nullptr) {
  int st = check_common(B, H, N, d, scale);
  if (st != FA_OK) return st;
  Strides lay{};
  if (strides)
    lay = *strides;
  else if (!dense_strides(B, H, N, d, &lay))
    return FA_ERR_INVALID_ARG;
  const bool pre = stages & kBwdStagePre, mainst = stages & kBwdStageMain,
             conv = stages & kBwdStageConvert;
  if (!p.ws) return FA_ERR_INVALID_ARG;
  if (pre && (!p.o || !p.dout || !p.lse)) return FA_ERR_INVALID_ARG;
  if (mainst && (!p.q || !p.k || !p.v || !p.dout || !p.dk || !p.dv)) return FA_ERR_INVALID_ARG;
  if (conv && !p.dq) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  const void* all[] = {p.q, p.k, p.v, p.o, p.dout, p.lse, p.dq, p.dk, p.dv, p.ws};
  for (const void* x : all)
    if (x && !aligned16(x)) return FA_ERR_INVALID_ARG;
  if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return FA_ERR_INVALID_ARG;
  const BwdWorkspace ws = bwd_workspace_layout(B, H, N, d);
  if (ws.total == 0 || workspace_bytes < ws.total) return FA_ERR_INVALID_ARG;
  // The split area (fa_bwd_split_workspace_bytes) follows the base regions;
  // the main kernel uses it only if it is complete.
  const size_t split_bytes = bwd_split_layout(sm_count(), d).total;
  const bool have_split = workspace_bytes - ws.total >= split_bytes;
  const size_t ws_used = ws.total + (have_split ? split_bytes : 0);
  const size_t tb = span_bytes(B, H, N, d, lay, 2), lb = tensor_bytes(B, H, N, 1, 4);
  const void* ins[] = {p.q, p.k, p.v, p.o, p.dout};
  void* outs[] = {p.dq, p.dk, p.dv};
  for (int x = 0; x < 3; ++x) {
    void* out = outs[x];
    if (!out) continue;
    for (const void* in : ins)
      if (in && strided_overlap(out, in, B, H, N, d, lay)) return FA_ERR_INVALID_ARG;
    if ((p.lse && overlaps(out, tb, p.lse, lb)) || overlaps(out, tb, p.ws, ws_used))
      return FA_ERR_INVALID_ARG;
    for (int y = x + 1; y < 3; ++y)
      if (outs[y] && strided_overlap(out, outs[y], B, H, N, d, lay)) return FA_ERR_INVALID_ARG;
  }
  for (const void* in : ins)
    if (in && overlaps(p.ws, ws_used, in, tb)) return FA_ERR_INVALID_ARG;
  if (p.lse && overlaps(p.ws, ws_used, p.lse, lb)) return FA_ERR_INVALID_ARG;
  DeviceInfo dev;
  st = current_device_info(&dev);
  if (st != FA_OK) return st;
  BwdLaunch a;
  std::memset(&a, 0, sizeof(a));
  uint8_t* wsb = static_cast<uint8_t*>(p.ws);
  const int npad = (N + kBlock - 1) / kBlock * kBlock;
  if (mainst && (!encode_rows(&a.tm_q, p.q, B, H, N, d, lay) ||
                 !encode_rows(&a.tm_k, p.k, B, H, N, d, lay) ||
                 !encode_rows(&a.tm_v, p.v, B, H, N, d, lay) ||
                 !encode_rows(&a.tm_do, p.dout, B, H, N, d, lay) ||
                 !encode_rows(&a.tm_dk, p.dk, B, H, N, d, lay, d == 128 ? 32 : kBlock, d == 128) ||
                 !encode_rows(&a.tm_dv, p.dv, B, H, N, d, lay, d == 128 ? 32 : kBlock, d == 128) ||
                 !encode_f32_rows(&a.tm_dqacc, wsb + ws.dq_off, B * H, npad, d)))
    return FA_ERR_CUDA;
  a.st = lay;
  a.o = p.o;
  a.dout = p.dout;
  a.lse = p.lse;
  a.dq = p.dq;
  a.dk = p.dk;
  a.dv = p.dv;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  a.kv_len = kv_len;
  a.block_mask = block_mask;
  if (drop) a.drop = *drop;
  a.split_ws = have_split ? wsb + ws.total : nullptr;
  a.split_ws_bytes = have_split ? split_bytes : 0;
  a.dq_acc = reinterpret_cast<float*>(wsb + ws.dq_off);
  a.lse2 = reinterpret_cast<float*>(wsb + ws.lse2_off);
  a.delta = reinterpret_cast<float*>(wsb + ws.delta_off);
  a.status = dev.status;
  a.wait_limit = kWaitLimitCycles;
  return launch_bwd(a, stages, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

BwdWorkspace bwd_workspace_layout(int B, int H, int N, int d) {
  BwdWorkspace w{};
  const size_t npad = (static_cast<size_t>(N) + kBlock - 1) / kBlock * kBlock;
  const size_t rows = static_cast<size_t>(B) * H * npad;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  w.dq_off = 0;
  w.lse2_off = up(rows * d * 4);
  w.delta_off = w.lse2_off + up(rows * 4);
  w.total = w.delta_off + up(rows * 4);
  return w;
}

int sm_count() {
  static int count[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (count[dev] == 0) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c < 1) c = 148;
    count[dev] = c;
  }
  return count[dev];
}

}  // namespace fa

using namespace fa;

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, int causal, float scale, struct CUstream_st* stream) {
  return fwd_common(q, k, v, o, lse, B, H, N, d, causal, scale, nullptr, nullptr, stream);
}

int fa_fwd_kpad(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int N, int d, int causal, float scale, const int32_t* kv_len,
                struct CUstream_st* stream) {
  return fwd_common(q, k, v, o, lse, B, H, N, d, causal, scale, kv_len, nullptr, stream);
}

int fa_blocksparse_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int N, int d, float scale, const uint8_t* block_mask, int block_size,
                       struct CUstream_st* stream) {
  if (block_mask == nullptr) return FA_ERR_INVALID_ARG;
  if (block_size != kBlock) return FA_ERR_UNSUPPORTED;
  return fwd_common(q, k, v, o, lse, B, H, N, d, 0, scale, nullptr, block_mask, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  if (B > 65535 || H > 65535 || !sizes_fit_int(B, H, N)) return 0;
  return bwd_workspace_layout(B, H, N, d).total;
}

size_t fa_bwd_split_workspace_bytes(int B, int H, int N, int d, int causal) {
  const size_t base = fa_bwd_workspace_bytes(B, H, N, d);
  if (base == 0 || (causal != 0 && causal != 1)) return 0;
  const int G = sm_count();
  const SplitPlan p = plan_bwd(B, H, N, d, causal != 0, G, true);
  return p.whole < p.n_items ? base + bwd_split_layout(G, d).total : base;
}

size_t fa_fwd_workspace_bytes(int B, int H, int N, int d, int causal) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || (causal != 0 && causal != 1)) return 0;
  if (B > 65535 || H > 65535 || !sizes_fit_int(B, H, N)) return 0;
  const int G = sm_count();
  const SplitPlan p = plan_fwd(B, H, N, d, causal != 0, G, true);
  return p.whole < p.n_items ? fwd_split_layout(G, d).total : 0;
}

int fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, int causal, float scale, const int32_t* kv_len, void* workspace,
                 size_t workspace_bytes, struct CUstream_st* stream) {
  if (workspace == nullptr && workspace_bytes != 0) return FA_ERR_INVALID_ARG;
  return fwd_common(q, k, v, o, lse, B, H, N, d, causal, scale, kv_len, nullptr, stream, nullptr,
                    nullptr, workspace, workspace_bytes);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
           float scale, const int32_t* kv_len, void* workspace, size_t workspace_bytes,
           struct CUstream_st* stream) {
  const BwdPtrs p{q, k, v, o, dout, lse, dq, dk, dv, workspace};
  return bwd_common(kBwdStageAll, p, B, H, N, d, causal, scale, kv_len, workspace_bytes, stream);
}

int fa_blocksparse_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                       int H, int N, int d, float scale, const uint8_t* block_mask, int block_size,
                       void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
  if (block_mask == nullptr) return FA_ERR_INVALID_ARG;
  if (block_size != kBlock) return FA_ERR_UNSUPPORTED;
  const BwdPtrs p{q, k, v, o, dout, lse, dq, dk, dv, workspace};
  return bwd_common(kBwdStageAll, p, B, H, N, d, 0, scale, nullptr, workspace_bytes, stream,
                    block_mask);
}

int fa_dropout_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int H, int N, int d, int causal, float scale, const int32_t* kv_len,
                   float dropout_p, uint64_t seed, uint32_t offset, struct CUstream_st* stream) {
  DropoutParams drop{};
  if (!make_dropout(dropout_p, seed, offset, &drop)) return FA_ERR_INVALID_ARG;
  return fwd_common(q, k, v, o, lse, B, H, N, d, causal, scale, kv_len, nullptr, stream, &drop);
}

int fa_dropout_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   int causal, float scale, const int32_t* kv_len, float dropout_p, uint64_t seed,
                   uint32_t offset, void* workspace, size_t workspace_bytes,
                   struct CUstream_st* stream) {
  DropoutParams drop{};
  if (!make_dropout(dropout_p, seed, offset, &drop)) return FA_ERR_INVALID_ARG;
  const BwdPtrs p{q, k, v, o, dout, lse, dq, dk, dv, workspace};
  return bwd_common(kBwdStageAll, p, B, H, N, d, causal, scale, kv_len, workspace_bytes, stream,
                    nullptr, &drop);
}

int fa_dropout_mask(int B, int H, int N, float dropout_p, uint64_t seed, uint32_t offset,
                    uint8_t* keep, struct CUstream_st* stream) {
  DropoutParams drop{};
  if (!make_dropout(dropout_p, seed, offset, &drop)) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1 || !keep) return FA_ERR_INVALID_ARG;
  if (B > 65535 || H > 65535 || !sizes_fit_int(B, H, N)) return FA_ERR_INVALID_ARG;
  DeviceInfo dev;
  const int st = current_device_info(&dev);
  if (st != FA_OK) return st;
  return launch_dropout_mask(drop, B * H, N, keep, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

namespace {

// Strides, dropout and the remaining checks of fa_attention_fwd / _bwd.
int attention_options(const fa_attention_options* opt, int B, int H, int N, int d, Strides* lay,
                      DropoutParams* drop, bool* use_drop) {
  if (opt == nullptr || B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (opt->stride_b == 0 && opt->stride_h == 0 && opt->stride_n == 0) {
    if (!dense_strides(B, H, N, d, lay)) return FA_ERR_INVALID_ARG;
  } else if (!make_strides(B, H, N, d, opt->stride_b, opt->stride_h, opt->stride_n, lay)) {
    return FA_ERR_INVALID_ARG;
  }
  if (opt->block_mask != nullptr && opt->block_size != kBlock) return FA_ERR_UNSUPPORTED;
  *use_drop = opt->dropout_p != 0.f;
  if (*use_drop && !make_dropout(opt->dropout_p, opt->dropout_seed, opt->dropout_offset, drop))
    return FA_ERR_INVALID_ARG;  // negative, NaN or >= 1
  return FA_OK;
}

}  // namespace

int fa_attention_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, const fa_attention_options* opt,
                     struct CUstream_st* stream) {
  Strides lay{};
  DropoutParams drop{};
  bool use_drop = false;
  const int st = attention_options(opt, B, H, N, d, &lay, &drop, &use_drop);
  if (st != FA_OK) return st;
  return fwd_common(q, k, v, o, lse, B, H, N, d, opt->causal, opt->scale, opt->kv_len,
                    opt->block_mask, stream, use_drop ? &drop : nullptr, &lay);
}

int fa_attention_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int N, int d, const fa_attention_options* opt,
                           void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
  Strides lay{};
  DropoutParams drop{};
  bool use_drop = false;
  const int st = attention_options(opt, B, H, N, d, &lay, &drop, &use_drop);
  if (st != FA_OK) return st;
  if (workspace == nullptr && workspace_bytes != 0) return FA_ERR_INVALID_ARG;
  return fwd_common(q, k, v, o, lse, B, H, N, d, opt->causal, opt->scale, opt->kv_len,
                    opt->block_mask, stream, use_drop ? &drop : nullptr, &lay, workspace,
                    workspace_bytes);
}

int fa_attention_bwd(const void* q, const void* k, const void* v, const void* o,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                     int H, int N, int d, const fa_attention_options* opt, void* workspace,
                     size_t workspace_bytes, struct CUstream_st* stream) {
  Strides lay{};
  DropoutParams drop{};
  bool use_drop = false;
  const int st = attention_options(opt, B, H, N, d, &lay, &drop, &use_drop);
  if (st != FA_OK) return st;
  const BwdPtrs p{q, k, v, o, dout, lse, dq, dk, dv, workspace};
  return bwd_common(kBwdStageAll, p, B, H, N, d, opt->causal, opt->scale, opt->kv_len,
                    workspace_bytes, stream, opt->block_mask, use_drop ? &drop : nullptr, &lay);
}

int fa_bwd_preprocess(const void* o, const void* dout, const float* lse, int B, int H, int N,
                      int d, void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
  const BwdPtrs p{nullptr, nullptr, nullptr, o, dout, lse, nullptr, nullptr, nullptr, workspace};
  return bwd_common(kBwdStagePre, p, B, H, N, d, 0, 1.f, nullptr, workspace_bytes, stream);
}

int fa_bwd_main(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                int B, int H, int N, int d, int causal, float scale, const int32_t* kv_len,
                void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
  const BwdPtrs p{q, k, v, nullptr, dout, nullptr, nullptr, dk, dv, workspace};
  return bwd_common(kBwdStageMain, p, B, H, N, d, causal, scale, kv_len, workspace_bytes, stream);
}

int fa_bwd_dq_convert(void* dq, int B, int H, int N, int d, void* workspace,
                      size_t workspace_bytes, struct CUstream_st* stream) {
  const BwdPtrs p{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dq, nullptr, nullptr,
                  workspace};
  return bwd_common(kBwdStageConvert, p, B, H, N, d, 0, 1.f, nullptr, workspace_bytes, stream);
}

int fa_device_status(void) {
  DeviceInfo dev;
  const int st = current_device_info(&dev);
  if (st != FA_OK) return st == FA_ERR_UNSUPPORTED ? FA_ERR_UNSUPPORTED : FA_ERR_CUDA;
  int value = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&value, g_status_word, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  return value;
}

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
    case FA_ERR_DEVICE_CHECK: return "FA_ERR_DEVICE_CHECK";
    default: return "FA_UNKNOWN_STATUS";
  }
}

int fa_selftest_wait_timeout(long long limit_cycles, struct CUstream_st* stream) {
  if (limit_cycles < 1) return FA_ERR_INVALID_ARG;
  DeviceInfo dev;
  const int st = current_device_info(&dev);
  if (st != FA_OK) return st;
  return launch_wait_selftest(dev.status, limit_cycles, stream) == cudaSuccess ? FA_OK
                                                                               : FA_ERR_CUDA;
}

}  // extern "C"
