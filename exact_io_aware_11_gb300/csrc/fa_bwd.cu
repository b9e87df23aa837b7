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
// 2. bwd_main_kernel  one CTA per 128-key tile j of one (batch, head); K_j and
//                     V_j stay in shared memory, dK_j and dV_j accumulate in
//                     TMEM, and the CTA loops over the Q tiles i:
//                       S^T  = K_j Q_i^T    TMEM, key rows on lanes
//                       dP^T = V_j dO_i^T   TMEM
//                       P^T  = exp2(S^T * scale*log2e - LSE2_i), bf16, written
//                              back into the S^T columns and used from TMEM
//                       dV_j += P^T dO_i
//                       dS^T = P^T * (dP^T - D_i), bf16 -> shared memory
//                       dK_j += dS^T Q_i
//                       dQ_i  = dS K_j      TMEM -> shared memory (fp32) -> one
//                              TMA bulk reduce-add per 32-column chunk into the
//                              fp32 workspace accumulator
//                     Warps 0-7 compute P and dS (warps w and w+4 share the
//                     key rows of TMEM lane quarter w % 4 and split the 128
//                     query columns), warp 8 issues TMA, warp 9 issues
//                     tcgen05.mma, warps 10-13 drain dQ. S^T of tile i+1 is
//                     computed while dS of tile i is being formed.
// 3. dq_convert_kernel  dQ bf16 = fp32 accumulator.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 448;
constexpr int kChunk = 128 * 128;  // one 128-row x 128-byte swizzled chunk
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdLayout {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kChunks * kChunk;     // 128 x D bf16
  static constexpr int kQS = 2;                      // Q (+ LSE2 / D) stages
  static constexpr int kDS = (D == 64) ? 2 : 1;      // dO stages
  static constexpr int kDQChunks = (D == 64) ? 2 : 1;  // 128 x 32 fp32 chunks staged at once
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;
  static constexpr int kDO = kQ + kQS * kTile;
  static constexpr int kStat = kDO + kDS * kTile;    // per Q stage: lse2[128], delta[128]
  static constexpr int kDSb = kStat + kQS * 1024;    // dS^T, bf16, 2 chunks
  static constexpr int kDQ = kDSb + 2 * kChunk;      // dQ staging (fp32, 128-byte swizzle)
  static constexpr int kBar = kDQ + kDQChunks * kChunk;
  static constexpr int kEnd = kBar + 256;
  static constexpr int kSmem = kEnd + 1024;
  // TMEM columns
  static constexpr uint32_t kTS = 0, kTDP = 128, kTDV = 256, kTDK = 256 + D;
  static constexpr uint32_t kTDQ = (D == 64) ? 384 : 128;  // d=128: dQ reuses the dP^T columns
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

// D[tmem] (+)= A[tmem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int x,
                                                  int y, int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
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
                    const __grid_constant__ CUtensorMap tm_dqacc,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const float* __restrict__ lse2, const float* __restrict__ delta, int H, int N,
                    int Npad, float scale, const int32_t* __restrict__ kv_len, int* status,
                    long long wait_limit) {
  using L = BwdLayout<D>;
  constexpr int QS = L::kQS, DS = L::kDS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* bar_kv = bars + 0;
  uint64_t* bar_qfull = bars + 1;    // [QS]
  uint64_t* bar_qempty = bars + 3;   // [QS]
  uint64_t* bar_dofull = bars + 5;   // [DS]
  uint64_t* bar_doempty = bars + 7;  // [DS]
  uint64_t* bar_sfull = bars + 9;
  uint64_t* bar_dpfull = bars + 10;
  uint64_t* bar_pready = bars + 11;
  uint64_t* bar_dsready = bars + 12;
  uint64_t* bar_dsfree = bars + 13;
  uint64_t* bar_dqfull = bars + 14;
  uint64_t* bar_dqfree = bars + 15;
  uint64_t* bar_final = bars + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  int* abort_flag = reinterpret_cast<int*>(bars + 18);

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
    for (int s = 0; s < QS; ++s) {
      mbar_init(bar_qfull + s, 1);
      mbar_init(bar_qempty + s, 1);
    }
    for (int s = 0; s < DS; ++s) {
      mbar_init(bar_dofull + s, 1);
      mbar_init(bar_doempty + s, 1);
    }
    mbar_init(bar_sfull, 1);
    mbar_init(bar_dpfull, 1);
    mbar_init(bar_pready, 8);
    mbar_init(bar_dsready, 8);
    mbar_init(bar_dsfree, 1);
    mbar_init(bar_dqfull, 1);
    mbar_init(bar_dqfree, 4);
    mbar_init(bar_final, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Watchdog wd{wait_limit, status, abort_flag};

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer (one lane)
    if (lane == 0 && n_iter > 0) {
      int q_issued = 0, do_issued = 0;
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_dqacc);
      mbar_expect_tx(bar_kv, 2 * L::kTile);
      for (int c = 0; c < L::kChunks; ++c) {
        tma_load_3d(smem + L::kK + c * kChunk, &tm_k, bar_kv, c * 64, j * kBlock, bh);
        tma_load_3d(smem + L::kV + c * kChunk, &tm_v, bar_kv, c * 64, j * kBlock, bh);
      }
      for (int it = 0; it < n_iter; ++it) {
        const int i = i0 + it, qs = it % QS, ds = it % DS;
        if (it >= QS && !mbar_wait(bar_qempty + qs, ((it / QS) - 1) & 1, wd)) break;
        mbar_expect_tx(bar_qfull + qs, L::kTile + 1024);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(smem + L::kQ + qs * L::kTile + c * kChunk, &tm_q, bar_qfull + qs, c * 64,
                      i * kBlock, bh);
        const size_t roff = static_cast<size_t>(bh) * Npad + static_cast<size_t>(i) * kBlock;
        bulk_load(smem + L::kStat + qs * 1024, lse2 + roff, 512, bar_qfull + qs);
        bulk_load(smem + L::kStat + qs * 1024 + 512, delta + roff, 512, bar_qfull + qs);
        q_issued = it + 1;
        if (it >= DS && !mbar_wait(bar_doempty + ds, ((it / DS) - 1) & 1, wd)) break;
        mbar_expect_tx(bar_dofull + ds, L::kTile);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(smem + L::kDO + ds * L::kTile + c * kChunk, &tm_do, bar_dofull + ds, c * 64,
                      i * kBlock, bh);
        do_issued = it + 1;
      }
      mbar_wait_drain(bar_kv, 0, wait_limit);
      for (int t = max(0, q_issued - QS); t < q_issued; ++t)
        mbar_wait_drain(bar_qfull + (t % QS), (t / QS) & 1, wait_limit);
      for (int t = max(0, do_issued - DS); t < do_issued; ++t)
        mbar_wait_drain(bar_dofull + (t % DS), (t / DS) & 1, wait_limit);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer (one lane)
    // One thread on the critical path: it polls the barriers (test_wait) and
    // fences only after the waits that follow tcgen05.ld / tcgen05.st of
    // other threads (P^T ready, dS ready, dQ drained).
    if (lane == 0) {
      constexpr uint32_t kIdSS = idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t kIdKM = idesc_bf16(128, D, false, true);     // dV, dK: B MN-major
      constexpr uint32_t kIdMM = idesc_bf16(128, D, true, true);      // dQ: A, B MN-major
      // Descriptors built once; per MMA only a compile-time offset is added.
      const uint64_t k_kmaj = sdesc_sw128(smem_u32(smem + L::kK), 16, 1024);
      const uint64_t k_mn = sdesc_sw128(smem_u32(smem + L::kK), kChunk, 1024);
      const uint64_t v_kmaj = sdesc_sw128(smem_u32(smem + L::kV), 16, 1024);
      const uint64_t q_kmaj0 = sdesc_sw128(smem_u32(smem + L::kQ), 16, 1024);
      const uint64_t q_mn0 = sdesc_sw128(smem_u32(smem + L::kQ), kChunk, 1024);
      const uint64_t do_kmaj0 = sdesc_sw128(smem_u32(smem + L::kDO), 16, 1024);
      const uint64_t do_mn0 = sdesc_sw128(smem_u32(smem + L::kDO), kChunk, 1024);
      const uint64_t ds_kmaj = sdesc_sw128(smem_u32(smem + L::kDSb), 16, 1024);
      const uint64_t ds_mn = sdesc_sw128(smem_u32(smem + L::kDSb), kChunk, 1024);
      bool ok = n_iter > 0 && mbar_wait_spin(bar_kv, 0, wd);
      auto issue_s = [&](int it) -> bool {
        if (!mbar_wait_spin(bar_qfull + (it % QS), (it / QS) & 1, wd)) return false;
        const uint64_t qd = desc_adv(q_kmaj0, (it % QS) * L::kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
          mma_ss(tmem + L::kTS, desc_adv(k_kmaj, off), desc_adv(qd, off), kIdSS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_sfull);
        return true;
      };
      auto issue_dp = [&](int it) -> bool {
        if (!mbar_wait_spin(bar_dofull + (it % DS), (it / DS) & 1, wd)) return false;
        const uint64_t dd = desc_adv(do_kmaj0, (it % DS) * L::kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
          mma_ss(tmem + L::kTDP, desc_adv(v_kmaj, off), desc_adv(dd, off), kIdSS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_dpfull);
        return true;
      };
      if (ok) ok = issue_s(0) && issue_dp(0);
      for (int it = 0; ok && it < n_iter; ++it) {
        const uint64_t q_mn = desc_adv(q_mn0, (it % QS) * L::kTile);
        const uint64_t do_mn = desc_adv(do_mn0, (it % DS) * L::kTile);
        const uint32_t acc0 = it > 0 ? 1u : 0u;
        // dV += P^T dO: P^T (bf16) sits in the S^T columns [0,32) and [64,96)
        if (!mbar_wait_spin(bar_pready, it & 1, wd)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          const uint32_t a_col = L::kTS + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
          mma_ts(tmem + L::kTDV, tmem + a_col, desc_adv(do_mn, kk * 2048), kIdKM,
                 kk > 0 ? 1u : acc0);
        }
        mma_commit(bar_doempty + (it % DS));
        // S^T of the next Q tile while dS of this one is formed
        if (it + 1 < n_iter && !issue_s(it + 1)) { ok = false; break; }
        if (!mbar_wait_spin(bar_dsready, it & 1, wd)) { ok = false; break; }
        if (D == 64 && it >= 1 && !mbar_wait_spin(bar_dqfree, (it - 1) & 1, wd)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          mma_ss(tmem + L::kTDK, desc_adv(ds_kmaj, (kk >> 2) * kChunk + (kk & 3) * 32),
                 desc_adv(q_mn, kk * 2048), kIdKM, kk > 0 ? 1u : acc0);
        }
        mma_commit(bar_qempty + (it % QS));
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          mma_ss(tmem + L::kTDQ, desc_adv(ds_mn, kk * 2048), desc_adv(k_mn, kk * 2048), kIdMM,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_dqfull);
        mma_commit(bar_dsfree);
        if (it + 1 < n_iter) {
          // d = 128: dQ_i occupies the dP^T columns until the drain warps have it
          if (D == 128) {
            if (!mbar_wait_spin(bar_dqfree, it & 1, wd)) { ok = false; break; }
            tc_fence_after();
          }
          if (!issue_dp(it + 1)) { ok = false; break; }
        }
      }
      mma_commit(bar_final);
      mbar_wait_drain(bar_final, 0, wait_limit);
    }
    __syncwarp();
  } else if (warp >= 10) {
    // ------------------------------------------------------------ dQ drain (warps 10-13)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row within the tile == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint8_t* stage = smem + L::kDQ;
    const uint32_t st_base = smem_u32(stage);
    const bool issuer = (quarter == 0 && lane == 0);
    constexpr int kRounds = (D / 32) / L::kDQChunks;
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
#pragma unroll
      for (int round = 0; round < kRounds; ++round) {
#pragma unroll
        for (int cc = 0; cc < L::kDQChunks; ++cc) {
          const int c = round * L::kDQChunks + cc;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t addr = st_base + cc * kChunk + r * 128 + (((u ^ (r & 7))) << 4);
            st_shared_v4(addr, __float_as_uint(__uint_as_float(v[c][4 * u + 0]) * scale),
                         __float_as_uint(__uint_as_float(v[c][4 * u + 1]) * scale),
                         __float_as_uint(__uint_as_float(v[c][4 * u + 2]) * scale),
                         __float_as_uint(__uint_as_float(v[c][4 * u + 3]) * scale));
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(3, 128);
        if (issuer) {
#pragma unroll
          for (int cc = 0; cc < L::kDQChunks; ++cc)
            tma_reduce_add_3d(&tm_dqacc, stage + cc * kChunk, (round * L::kDQChunks + cc) * 32,
                              i * kBlock, bh);
          bulk_commit();
          bulk_wait_read0();
        }
        named_bar_sync(3, 128);
      }
    }
  } else {
    // ------------------------------------------------------------ P / dS (warps 0-7)
    const int wg = warp >> 2;             // query columns [64 wg, 64 wg + 64)
    const int quarter = warp & 3;
    const int kr = quarter * 32 + lane;   // key row within the tile == TMEM lane
    const int key = j * kBlock + kr;
    const bool key_live = key < kv_bound;
    const int qc0 = wg * 64;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t ds_base = smem_u32(smem + L::kDSb) + wg * kChunk;
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % QS;
      const int i = i0 + it;
      const float* st_lse = reinterpret_cast<const float*>(smem + L::kStat + s * 1024) + qc0;
      const float* st_delta = st_lse + 128;
      if (!mbar_wait_warp(bar_qfull + s, (it / QS) & 1, wd)) { ok = false; break; }
      if (!mbar_wait_warp(bar_sfull, it & 1, wd)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[2][32];
      tmem_ld32(lane_base + L::kTS + qc0, r[0]);
      tmem_ld32(lane_base + L::kTS + qc0 + 32, r[1]);
      tmem_wait_ld();
      reg_fence(r[0]);
      reg_fence(r[1]);
      // P is kept only as bf16 pairs (the form the dV MMA consumes); dS below
      // unpacks it, which halves the registers a compute thread holds.
      const bool diag = CAUSAL && i == j;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(st_lse + c);
        float p0 = ex2(fmaf(__uint_as_float(r[c >> 5][(c + 0) & 31]), scale_log2, -l4.x));
        float p1 = ex2(fmaf(__uint_as_float(r[c >> 5][(c + 1) & 31]), scale_log2, -l4.y));
        float p2 = ex2(fmaf(__uint_as_float(r[c >> 5][(c + 2) & 31]), scale_log2, -l4.z));
        float p3 = ex2(fmaf(__uint_as_float(r[c >> 5][(c + 3) & 31]), scale_log2, -l4.w));
        if (diag) {  // query i*128+qc0+c < key j*128+kr
          if (qc0 + c + 0 < kr) p0 = 0.f;
          if (qc0 + c + 1 < kr) p1 = 0.f;
          if (qc0 + c + 2 < kr) p2 = 0.f;
          if (qc0 + c + 3 < kr) p3 = 0.f;
        }
        pk[c / 2] = key_live ? pack_bf16(p0, p1) : 0u;
        pk[c / 2 + 1] = key_live ? pack_bf16(p2, p3) : 0u;
      }
      // P^T over the first 32 of this warpgroup's 64 S^T columns (already read)
      tmem_st32(lane_base + L::kTS + qc0, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pready);

      if (!mbar_wait_warp(bar_dpfull, it & 1, wd)) { ok = false; break; }
      if (it >= 1 && !mbar_wait_warp(bar_dsfree, (it - 1) & 1, wd)) { ok = false; break; }
      tc_fence_after();
      tmem_ld32(lane_base + L::kTDP + qc0, r[0]);
      tmem_ld32(lane_base + L::kTDP + qc0 + 32, r[1]);
      tmem_wait_ld();
      reg_fence(r[0]);
      reg_fence(r[1]);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int q0 = u * 8;
        const float4 da = *reinterpret_cast<const float4*>(st_delta + q0);
        const float4 db = *reinterpret_cast<const float4*>(st_delta + q0 + 4);
        const float dd[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
        float g[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t w = pk[(q0 + e) >> 1];
          const float pe = __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
          g[e] = pe * (__uint_as_float(r[(q0 + e) >> 5][(q0 + e) & 31]) - dd[e]);
        }
        const uint32_t addr = ds_base + kr * 128 + (((u ^ (kr & 7))) << 4);
        st_shared_v4(addr, pack_bf16(g[0], g[1]), pack_bf16(g[2], g[3]), pack_bf16(g[4], g[5]),
                     pack_bf16(g[6], g[7]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dsready);
    }
    // ------------------------------------------------------------ epilogue: dV (wg 0), dK (wg 1)
    bool have = ok && n_iter > 0;
    if (have) have = mbar_wait_warp(bar_final, 0, wd);
    if (have) tc_fence_after();
    const uint32_t col = wg == 0 ? L::kTDV : L::kTDK;
    const float mul = wg == 0 ? 1.f : scale;
    uint8_t* stage = smem + L::kQ + wg * L::kTile;  // Q stages are free now
    const uint32_t st_base = smem_u32(stage);
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
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int unit = c0 * 4 + u;
        const uint32_t addr = st_base + (unit >> 3) * kChunk + kr * 128 + (((unit & 7) ^ (kr & 7)) << 4);
        st_shared_v4(addr,
                     pack_bf16(__uint_as_float(v[8 * u + 0]) * mul, __uint_as_float(v[8 * u + 1]) * mul),
                     pack_bf16(__uint_as_float(v[8 * u + 2]) * mul, __uint_as_float(v[8 * u + 3]) * mul),
                     pack_bf16(__uint_as_float(v[8 * u + 4]) * mul, __uint_as_float(v[8 * u + 5]) * mul),
                     pack_bf16(__uint_as_float(v[8 * u + 6]) * mul, __uint_as_float(v[8 * u + 7]) * mul));
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1 + wg, 128);
    if (quarter == 0 && lane == 0) {
      const CUtensorMap* map = wg == 0 ? &tm_dv : &tm_dk;
      for (int c = 0; c < L::kChunks; ++c) tma_store_3d(map, stage + c * kChunk, c * 64, j * kBlock, bh);
      bulk_commit();
      bulk_wait_read0();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
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
        a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_dqacc, a.tm_dk, a.tm_dv, a.lse2, a.delta, a.H, a.N,
        Npad, a.scale, a.kv_len, a.status, a.wait_limit);
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
