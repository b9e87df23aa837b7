// Backward pass of exact attention as three sm_103a kernels.
//
// Method: the attention matrix is not read back from HBM; it is recomputed on
// chip, tile by tile, from Q, K and the per-row statistic saved by the forward
// pass (condensed paper sample_paper.md, section 3, "in the backward pass, the
// attention matrix is recomputed on-chip from stored statistics"; section 5,
// "tiling and recomputation"). With LSE the natural-log logsumexp:
//   P = exp(scale * Q K^T - LSE),   dV = P^T dO,   dP = dO V^T,
//   D = rowsum(dO * O) (= rowsum(P * dP)),   dS = P * (dP - D),
//   dQ = scale * dS K,   dK = scale * dS^T Q.
//
// 1. bwd_pre_kernel   D = rowsum(dO * O), LSE * log2(e), zero the fp32 dQ
//                     accumulator (bandwidth-bound, 16-byte accesses).
// 2. bwd_main_kernel  one CTA per 128-key tile of one (batch, head); it keeps
//                     K_j, V_j in shared memory and dK_j, dV_j in TMEM and
//                     loops over the Q tiles:
//                       S^T  = K_j Q_i^T        (TMEM, key rows on lanes)
//                       dP^T = V_j dO_i^T       (TMEM)
//                       P^T  = exp2(S^T * scale*log2e - LSE2_i)  -> smem bf16
//                       dV_j += P^T dO_i
//                       dS^T = P^T * (dP^T - D_i)                -> smem bf16
//                       dK_j += dS^T Q_i
//                       dQ_i  = dS K_j          (TMEM) -> fp32 atomics into the
//                                                        workspace, times scale
//                     warps 0-3 compute P / dS (thread t = key t = TMEM lane t),
//                     warp 4 issues TMA, warp 5 issues tcgen05.mma, warps 6-9
//                     drain dQ (thread = query row).
// 3. dq_convert_kernel  dQ bf16 = fp32 accumulator.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 320;
constexpr int kChunk = 128 * 128;  // one 128-row x 128-byte swizzled chunk
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdLayout {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kChunks * kChunk;
  static constexpr int kStages = (D == 64) ? 2 : 1;  // Q / dO / LSE2 / D stages
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;
  static constexpr int kDO = kQ + kStages * kTile;
  static constexpr int kStat = kDO + kStages * kTile;  // per stage: lse2[128], delta[128]
  static constexpr int kP = kStat + kStages * 1024;
  static constexpr int kDS = kP + 2 * kChunk;
  static constexpr int kBar = kDS + 2 * kChunk;
  static constexpr int kEnd = kBar + 256;
  static constexpr int kSmem = kEnd + 1024;
  // TMEM columns
  static constexpr uint32_t kTS = 0, kTDP = 128, kTDV = 256, kTDK = 256 + D;
  static constexpr uint32_t kTDQ = (D == 64) ? 384 : 0;  // d=128: dQ reuses the S^T columns
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

// ----------------------------------------------------------------- preprocess
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      const float* __restrict__ lse,
                                                      float* __restrict__ lse2,
                                                      float* __restrict__ delta,
                                                      float* __restrict__ dq_acc, int BH, int N,
                                                      int Npad) {
  constexpr int kPer = D / 8;  // threads per row (8 elements = 16 bytes each)
  const long long total = static_cast<long long>(BH) * Npad * kPer;
  const long long total32 = (total + 31) & ~31LL;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < total32;
       g += stride) {
    const bool in = g < total;
    const long long row = g / kPer;  // over [BH, Npad]
    const int part = static_cast<int>(g % kPer);
    const int bh = static_cast<int>(row / Npad);
    const int n = static_cast<int>(row % Npad);
    const bool valid = in && n < N;
    float acc = 0.f;
    if (valid) {
      const size_t off = (static_cast<size_t>(bh) * N + n) * D + part * 8;
      const uint4 a = *reinterpret_cast<const uint4*>(o + off);
      const uint4 b = *reinterpret_cast<const uint4*>(dout + off);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(a2[i]);
        const float2 y = __bfloat1622float2(b2[i]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
#pragma unroll
    for (int w = 1; w < kPer; w <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (in) {
      float4* z = reinterpret_cast<float4*>(dq_acc + static_cast<size_t>(row) * D + part * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (part == 0) {
        delta[row] = valid ? acc : 0.f;
        float l2 = INFINITY;  // padding rows and rows that saw no key get P = 0
        if (valid) {
          const float v = lse[static_cast<size_t>(bh) * N + n];
          if (v != -INFINITY) l2 = v * kLog2e;
        }
        lse2[row] = l2;
      }
    }
  }
}

// ----------------------------------------------------------------- dQ convert
template <int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ dq_acc,
                                                         __nv_bfloat16* __restrict__ dq, int BH,
                                                         int N, int Npad) {
  constexpr int kPer = D / 8;
  const long long total = static_cast<long long>(BH) * N * kPer;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
       g += stride) {
    const long long row = g / kPer;  // over [BH, N]
    const int part = static_cast<int>(g % kPer);
    const long long bh = row / N;
    const long long n = row % N;
    const float4* src = reinterpret_cast<const float4*>(dq_acc + (bh * Npad + n) * D + part * 8);
    const float4 a = src[0], b = src[1];
    uint4 w;
    w.x = pack_bf16(a.x, a.y);
    w.y = pack_bf16(a.z, a.w);
    w.z = pack_bf16(b.x, b.y);
    w.w = pack_bf16(b.z, b.w);
    *reinterpret_cast<uint4*>(dq + row * D + part * 8) = w;
  }
}

// ----------------------------------------------------------------- main kernel
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const float* __restrict__ lse2, const float* __restrict__ delta,
                    float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dk,
                    __nv_bfloat16* __restrict__ dv, int H, int N, int Npad, float scale,
                    const int32_t* __restrict__ kv_len, int* status, long long wait_limit) {
  using L = BwdLayout<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* bar_kv = bars + 0;
  uint64_t* bar_qfull = bars + 1;   // [S]
  uint64_t* bar_qempty = bars + 3;  // [S]
  uint64_t* bar_sfull = bars + 5;
  uint64_t* bar_dpfull = bars + 6;
  uint64_t* bar_pready = bars + 7;
  uint64_t* bar_pfree = bars + 8;
  uint64_t* bar_dsready = bars + 9;
  uint64_t* bar_dsfree = bars + 10;
  uint64_t* bar_dqfull = bars + 11;
  uint64_t* bar_dqfree = bars + 12;
  uint64_t* bar_final = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  int* abort_flag = reinterpret_cast<int*>(bars + 15);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nqt = (N + kBlock - 1) / kBlock;
  const int j = blockIdx.x;  // key tile
  const int bh = blockIdx.z * H + blockIdx.y;
  int kv_bound = N;
  if (kv_len != nullptr) kv_bound = min(N, max(0, kv_len[blockIdx.z]));
  const bool active = j * kBlock < kv_bound;
  const int i0 = CAUSAL ? j : 0;
  const int n_iter = active ? (nqt - i0) : 0;
  const float scale_log2 = scale * kLog2e;

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_qfull + s, 1);
      mbar_init(bar_qempty + s, 1);
    }
    mbar_init(bar_sfull, 1);
    mbar_init(bar_dpfull, 1);
    mbar_init(bar_pready, 4);
    mbar_init(bar_pfree, 1);
    mbar_init(bar_dsready, 4);
    mbar_init(bar_dsfree, 1);
    mbar_init(bar_dqfull, 1);
    mbar_init(bar_dqfree, 4);
    mbar_init(bar_final, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Watchdog wd{wait_limit, status, abort_flag};

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    int issued = 0;
    if (n_iter > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        mbar_expect_tx(bar_kv, 2 * L::kTile);
        for (int c = 0; c < L::kChunks; ++c) {
          tma_load_3d(smem + L::kK + c * kChunk, &tm_k, bar_kv, c * 64, j * kBlock, bh);
          tma_load_3d(smem + L::kV + c * kChunk, &tm_v, bar_kv, c * 64, j * kBlock, bh);
        }
      }
      for (int it = 0; it < n_iter; ++it) {
        const int s = it % S;
        const int i = i0 + it;
        if (it >= S && !mbar_wait_warp(bar_qempty + s, ((it / S) - 1) & 1, wd)) break;
        if (lane == 0) {
          mbar_expect_tx(bar_qfull + s, 2 * L::kTile + 1024);
          for (int c = 0; c < L::kChunks; ++c) {
            tma_load_3d(smem + L::kQ + s * L::kTile + c * kChunk, &tm_q, bar_qfull + s, c * 64,
                        i * kBlock, bh);
            tma_load_3d(smem + L::kDO + s * L::kTile + c * kChunk, &tm_do, bar_qfull + s, c * 64,
                        i * kBlock, bh);
          }
          const size_t roff = static_cast<size_t>(bh) * Npad + static_cast<size_t>(i) * kBlock;
          bulk_load(smem + L::kStat + s * 1024, lse2 + roff, 512, bar_qfull + s);
          bulk_load(smem + L::kStat + s * 1024 + 512, delta + roff, 512, bar_qfull + s);
        }
        __syncwarp();
        issued = it + 1;
      }
      if (lane == 0) {
        mbar_wait_drain(bar_kv, 0, wait_limit);
        for (int t = max(0, issued - S); t < issued; ++t)
          mbar_wait_drain(bar_qfull + (t % S), (t / S) & 1, wait_limit);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdSS = idesc_bf16(128, 128, false, false);  // S^T, dP^T
    constexpr uint32_t kIdKM = idesc_bf16(128, D, false, true);     // dV, dK: A K-major, B MN-major
    constexpr uint32_t kIdMM = idesc_bf16(128, D, true, true);      // dQ: A, B MN-major
    const uint32_t k_base = smem_u32(smem + L::kK);
    const uint32_t v_base = smem_u32(smem + L::kV);
    const uint32_t q_base0 = smem_u32(smem + L::kQ);
    const uint32_t do_base0 = smem_u32(smem + L::kDO);
    const uint32_t p_base = smem_u32(smem + L::kP);
    const uint32_t ds_base = smem_u32(smem + L::kDS);
    bool ok = n_iter > 0 && mbar_wait_warp(bar_kv, 0, wd);
    if (ok) tc_fence_after();
    for (int it = 0; ok && it < n_iter; ++it) {
      const int s = it % S;
      const uint32_t q_base = q_base0 + s * L::kTile;
      const uint32_t do_base = do_base0 + s * L::kTile;
      if (!mbar_wait_warp(bar_qfull + s, (it / S) & 1, wd)) { ok = false; break; }
      if (D == 128 && it >= 1 && !mbar_wait_warp(bar_dqfree, (it - 1) & 1, wd)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
          mma_ss(tmem + L::kTS, sdesc_sw128(k_base + off, 16, 1024),
                 sdesc_sw128(q_base + off, 16, 1024), kIdSS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_sfull);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
          mma_ss(tmem + L::kTDP, sdesc_sw128(v_base + off, 16, 1024),
                 sdesc_sw128(do_base + off, 16, 1024), kIdSS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_dpfull);
      }
      __syncwarp();
      if (!mbar_wait_warp(bar_pready, it & 1, wd)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          const uint64_t a = sdesc_sw128(p_base + (kk >> 2) * kChunk + (kk & 3) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(do_base + kk * 2048, kChunk, 1024);
          mma_ss(tmem + L::kTDV, a, b, kIdKM, (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar_pfree);
      }
      __syncwarp();
      if (!mbar_wait_warp(bar_dsready, it & 1, wd)) { ok = false; break; }
      if (D == 64 && it >= 1 && !mbar_wait_warp(bar_dqfree, (it - 1) & 1, wd)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          const uint64_t a = sdesc_sw128(ds_base + (kk >> 2) * kChunk + (kk & 3) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(q_base + kk * 2048, kChunk, 1024);
          mma_ss(tmem + L::kTDK, a, b, kIdKM, (it > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          const uint64_t a = sdesc_sw128(ds_base + kk * 2048, kChunk, 1024);
          const uint64_t b = sdesc_sw128(k_base + kk * 2048, kChunk, 1024);
          mma_ss(tmem + L::kTDQ, a, b, kIdMM, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_dqfull);
        mma_commit(bar_dsfree);
        mma_commit(bar_qempty + s);
      }
      __syncwarp();
    }
    if (lane == 0) {
      mma_commit(bar_final);
      mbar_wait_drain(bar_final, 0, wait_limit);
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ------------------------------------------------------------ dQ drain (warps 6-9)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row within the tile == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    for (int it = 0; it < n_iter; ++it) {
      const int i = i0 + it;
      if (!mbar_wait_warp(bar_dqfull, it & 1, wd)) break;
      tc_fence_after();
      uint32_t v[D / 32][32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(lane_base + L::kTDQ + c * 32, v[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) reg_fence(v[c]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dqfree);
      float4* dst = reinterpret_cast<float4*>(
          dq_acc + (static_cast<size_t>(bh) * Npad + static_cast<size_t>(i) * kBlock + r) * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 add = make_float4(__uint_as_float(v[c][4 * u + 0]) * scale,
                                         __uint_as_float(v[c][4 * u + 1]) * scale,
                                         __uint_as_float(v[c][4 * u + 2]) * scale,
                                         __uint_as_float(v[c][4 * u + 3]) * scale);
          atomicAdd(dst + c * 8 + u, add);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ P / dS (warps 0-3)
    const int t = threadIdx.x;  // key row within the tile == TMEM lane
    const int key = j * kBlock + t;
    const bool key_live = key < kv_bound;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t p_base = smem_u32(smem + L::kP);
    const uint32_t ds_base = smem_u32(smem + L::kDS);
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % S;
      const int i = i0 + it;
      const float* st_lse = reinterpret_cast<const float*>(smem + L::kStat + s * 1024);
      const float* st_delta = st_lse + 128;
      if (!mbar_wait_warp(bar_qfull + s, (it / S) & 1, wd)) { ok = false; break; }
      if (!mbar_wait_warp(bar_sfull, it & 1, wd)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + L::kTS + c * 32, r[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence(r[c]);
      float p[128];
#pragma unroll
      for (int c = 0; c < 128; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(st_lse + c);
        p[c + 0] = ex2(fmaf(__uint_as_float(r[c >> 5][(c + 0) & 31]), scale_log2, -l4.x));
        p[c + 1] = ex2(fmaf(__uint_as_float(r[c >> 5][(c + 1) & 31]), scale_log2, -l4.y));
        p[c + 2] = ex2(fmaf(__uint_as_float(r[c >> 5][(c + 2) & 31]), scale_log2, -l4.z));
        p[c + 3] = ex2(fmaf(__uint_as_float(r[c >> 5][(c + 3) & 31]), scale_log2, -l4.w));
      }
      if (!key_live) {
#pragma unroll
        for (int c = 0; c < 128; ++c) p[c] = 0.f;
      }
      if (CAUSAL && i == j) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c < t) p[c] = 0.f;  // query i*128+c < key j*128+t
      }
      if (it >= 1) {
        if (!mbar_wait_warp(bar_pfree, (it - 1) & 1, wd)) { ok = false; break; }
      }
      // P^T row t -> shared memory, K-major (queries along K), 128-byte swizzle.
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint32_t addr = p_base + (u >> 3) * kChunk + t * 128 + ((((u & 7) ^ (t & 7))) << 4);
        st_shared_v4(addr, pack_bf16(p[8 * u + 0], p[8 * u + 1]), pack_bf16(p[8 * u + 2], p[8 * u + 3]),
                     pack_bf16(p[8 * u + 4], p[8 * u + 5]), pack_bf16(p[8 * u + 6], p[8 * u + 7]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pready);

      if (!mbar_wait_warp(bar_dpfull, it & 1, wd)) { ok = false; break; }
      if (it >= 1) {
        if (!mbar_wait_warp(bar_dsfree, (it - 1) & 1, wd)) { ok = false; break; }
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t dp[32];
        tmem_ld32(lane_base + L::kTDP + c * 32, dp);
        tmem_wait_ld();
        reg_fence(dp);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q0 = c * 32 + u * 8;
          const float4 da = *reinterpret_cast<const float4*>(st_delta + q0);
          const float4 db = *reinterpret_cast<const float4*>(st_delta + q0 + 4);
          const float d0 = p[q0 + 0] * (__uint_as_float(dp[u * 8 + 0]) - da.x);
          const float d1 = p[q0 + 1] * (__uint_as_float(dp[u * 8 + 1]) - da.y);
          const float d2 = p[q0 + 2] * (__uint_as_float(dp[u * 8 + 2]) - da.z);
          const float d3 = p[q0 + 3] * (__uint_as_float(dp[u * 8 + 3]) - da.w);
          const float d4 = p[q0 + 4] * (__uint_as_float(dp[u * 8 + 4]) - db.x);
          const float d5 = p[q0 + 5] * (__uint_as_float(dp[u * 8 + 5]) - db.y);
          const float d6 = p[q0 + 6] * (__uint_as_float(dp[u * 8 + 6]) - db.z);
          const float d7 = p[q0 + 7] * (__uint_as_float(dp[u * 8 + 7]) - db.w);
          const int unit = q0 >> 3;  // 0..15
          const uint32_t addr =
              ds_base + (unit >> 3) * kChunk + t * 128 + ((((unit & 7) ^ (t & 7))) << 4);
          st_shared_v4(addr, pack_bf16(d0, d1), pack_bf16(d2, d3), pack_bf16(d4, d5),
                       pack_bf16(d6, d7));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dsready);
    }
    // ------------------------------------------------------------ epilogue: dV, dK
    bool have = ok && n_iter > 0;
    if (have) have = mbar_wait_warp(bar_final, 0, wd);
    if (have) tc_fence_after();
    const bool row_ok = key < N;
    const size_t roff = (static_cast<size_t>(bh) * N + key) * D;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint32_t col = which == 0 ? L::kTDV : L::kTDK;
      const float mul = which == 0 ? 1.f : scale;
      uint4* dst = reinterpret_cast<uint4*>((which == 0 ? dv : dk) + roff);
#pragma unroll
      for (int c0 = 0; c0 < D / 32; ++c0) {
        uint32_t v[32];
        if (have) {
          tmem_ld32(lane_base + col + c0 * 32, v);
          tmem_wait_ld();
          reg_fence(v);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = 0u;
        }
        if (row_ok) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(v[8 * u + 0]) * mul, __uint_as_float(v[8 * u + 1]) * mul);
            w.y = pack_bf16(__uint_as_float(v[8 * u + 2]) * mul, __uint_as_float(v[8 * u + 3]) * mul);
            w.z = pack_bf16(__uint_as_float(v[8 * u + 4]) * mul, __uint_as_float(v[8 * u + 5]) * mul);
            w.w = pack_bf16(__uint_as_float(v[8 * u + 6]) * mul, __uint_as_float(v[8 * u + 7]) * mul);
            dst[c0 * 4 + u] = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

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
  using L = BwdLayout<D>;
  const int BH = a.B * a.H;
  const int nt = (a.N + kBlock - 1) / kBlock;
  const int Npad = nt * kBlock;
  cudaError_t e = cudaSuccess;
  if (stages & kBwdStagePre) {
    bwd_pre_kernel<D><<<grid_for(static_cast<long long>(BH) * Npad * (D / 8)), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.lse,
        a.lse2, a.delta, a.dq_acc, BH, a.N, Npad);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdStageMain) {
    auto kern = bwd_main_kernel<D, CAUSAL>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(nt, a.H, a.B), kThreads, L::kSmem, stream>>>(
        a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.lse2, a.delta, a.dq_acc,
        static_cast<__nv_bfloat16*>(a.dk), static_cast<__nv_bfloat16*>(a.dv), a.H, a.N, Npad,
        a.scale, a.kv_len, a.status, a.wait_limit);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdStageConvert) {
    dq_convert_kernel<D><<<grid_for(static_cast<long long>(BH) * a.N * (D / 8)), 256, 0, stream>>>(
        a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), BH, a.N, Npad);
    e = cudaGetLastError();
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
