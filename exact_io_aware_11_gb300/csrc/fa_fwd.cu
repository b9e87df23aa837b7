// Forward pass of exact attention (dense, causal, key-padded and block-sparse)
// as one fused sm_103a kernel.
//
// Method: FlashAttention's tiling with online softmax rescaling -- Q, K, V are
// split into blocks that are copied from HBM into on-chip memory, attention is
// computed block by block, the softmax normaliser is accumulated incrementally
// and the N x N matrices S and P are never written to HBM (condensed paper
// sample_paper.md, section 3 "Tiling" / "Softmax rescaling"; Medium article
// "No More Quadratic Complexity for Transformers", Figure 1). The pages put
// K/V in the outer loop; here each CTA owns one 128-row Q tile and streams
// the K/V tiles past it, which gives the same exact result and keeps the
// running statistics in registers.
//
// One CTA = one 128-row Q tile of one (batch, head); 6 warps:
//   warp 4      TMA producer: Q once, then K_j / V_j into a 2-stage ring
//   warp 5      MMA issuer:   S_j = Q K_j^T into TMEM (double-buffered),
//                             O += P_j V_j into a TMEM accumulator
//   warps 0-3   softmax:      thread t owns query row t (= TMEM lane t):
//                             masks, running max m / sum l, P_j = exp2(.) in
//                             bf16 to shared memory, O rescale in TMEM,
//                             epilogue O / l and LSE = (m + log2 l) ln 2.
// TMEM columns: [0,128) S buffer 0, [128,256) S buffer 1, [256,256+d) O.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr int kChunk = 128 * 128;  // bytes of one 128-row x 128-byte swizzled chunk (64 bf16 cols)
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct FwdLayout {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kChunks * kChunk;  // one 128 x D bf16 tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kP = kV + kStages * kTile;
  static constexpr int kBar = kP + 2 * kChunk;  // P: 128 rows x 128 keys bf16
  static constexpr int kEnd = kBar + 256;
  static constexpr int kSmem = kEnd + 1024;  // slack for 1024-byte alignment
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out,
               float* __restrict__ lse_out, int H, int N, float scale_log2,
               const int32_t* __restrict__ kv_len, const uint8_t* __restrict__ block_mask,
               int* status, long long wait_limit) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* bar_q = bars + 0;
  uint64_t* bar_kfull = bars + 1;    // [2]
  uint64_t* bar_vfull = bars + 3;    // [2]
  uint64_t* bar_kvempty = bars + 5;  // [2]
  uint64_t* bar_sfull = bars + 7;    // [2]
  uint64_t* bar_pfull = bars + 9;
  uint64_t* bar_odone = bars + 10;
  uint64_t* bar_final = bars + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
  int* abort_flag = reinterpret_cast<int*>(bars + 13);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nqt = (N + kBlock - 1) / kBlock;
  // Causal: heaviest tiles first so the tail of the grid is short.
  const int qt = CAUSAL ? (nqt - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const int bh = blockIdx.z * H + blockIdx.y;
  int kv_bound = N;
  if (kv_len != nullptr) kv_bound = min(N, max(0, kv_len[blockIdx.z]));
  int jend = (kv_bound + kBlock - 1) / kBlock;
  if (CAUSAL) jend = min(jend, qt + 1);
  const uint8_t* mrow = block_mask ? block_mask + static_cast<size_t>(qt) * nqt : nullptr;
  auto next_tile = [&](int j) {
    if (mrow != nullptr)
      while (j < jend && mrow[j] == 0) ++j;
    return j;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_kfull + s, 1);
      mbar_init(bar_vfull + s, 1);
      mbar_init(bar_kvempty + s, 1);
      mbar_init(bar_sfull + s, 1);
    }
    mbar_init(bar_pfull, 4);
    mbar_init(bar_odone, 1);
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
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_expect_tx(bar_q, L::kTile);
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_3d(smem + L::kQ + c * kChunk, &tm_q, bar_q, c * 64, qt * kBlock, bh);
    }
    int issued = 0;
    int jj = 0;
    for (int j = next_tile(0); j < jend; j = next_tile(j + 1), ++jj) {
      const int s = jj & 1;
      if (jj >= kStages && !mbar_wait_warp(bar_kvempty + s, ((jj >> 1) - 1) & 1, wd)) break;
      if (lane == 0) {
        mbar_expect_tx(bar_kfull + s, L::kTile);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(smem + L::kK + s * L::kTile + c * kChunk, &tm_k, bar_kfull + s, c * 64,
                      j * kBlock, bh);
        mbar_expect_tx(bar_vfull + s, L::kTile);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(smem + L::kV + s * L::kTile + c * kChunk, &tm_v, bar_vfull + s, c * 64,
                      j * kBlock, bh);
      }
      __syncwarp();
      issued = jj + 1;
    }
    // Let every copy already in flight land before the CTA can exit.
    if (lane == 0) {
      mbar_wait_drain(bar_q, 0, wait_limit);
      for (int t = max(0, issued - kStages); t < issued; ++t) {
        mbar_wait_drain(bar_kfull + (t & 1), (t >> 1) & 1, wait_limit);
        mbar_wait_drain(bar_vfull + (t & 1), (t >> 1) & 1, wait_limit);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);  // Q, K both K-major
    constexpr uint32_t kIdO = idesc_bf16(128, D, false, true);     // P K-major, V MN-major
    const uint32_t q_base = smem_u32(smem + L::kQ);
    const uint32_t k_base = smem_u32(smem + L::kK);
    const uint32_t v_base = smem_u32(smem + L::kV);
    const uint32_t p_base = smem_u32(smem + L::kP);
    auto issue_pv = [&](int t) -> bool {
      if (!mbar_wait_warp(bar_pfull, t & 1, wd)) return false;
      if (!mbar_wait_warp(bar_vfull + (t & 1), (t >> 1) & 1, wd)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t vb = v_base + (t & 1) * L::kTile;
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          // A = P (128 x 16 slice of keys), B = V (16 keys x D), MN-major.
          const uint64_t a = sdesc_sw128(p_base + (kk >> 2) * kChunk + (kk & 3) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(vb + kk * 2048, kChunk, 1024);
          mma_ss(tmem + 256, a, b, kIdO, (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar_kvempty + (t & 1));
        mma_commit(bar_odone);
      }
      __syncwarp();
      return true;
    };
    bool ok = mbar_wait_warp(bar_q, 0, wd);
    int jj = 0;
    if (ok) {
      tc_fence_after();
      for (int j = next_tile(0); j < jend; j = next_tile(j + 1), ++jj) {
        const int s = jj & 1;
        if (!mbar_wait_warp(bar_kfull + s, (jj >> 1) & 1, wd)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t kb = k_base + s * L::kTile;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
            mma_ss(tmem + s * 128, sdesc_sw128(q_base + off, 16, 1024),
                   sdesc_sw128(kb + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar_sfull + s);
        }
        __syncwarp();
        if (jj >= 1 && !issue_pv(jj - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && jj >= 1) issue_pv(jj - 1);
    }
    if (lane == 0) {
      mma_commit(bar_final);
      mbar_wait_drain(bar_final, 0, wait_limit);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (warps 0-3)
    const int t = threadIdx.x;  // row within the tile == TMEM lane
    const int row = qt * kBlock + t;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t p_base = smem_u32(smem + L::kP);
    float m = -INFINITY;  // running max of scale*log2(e)*s
    float l = 0.f;        // running sum of exp2(scale*log2(e)*s - m)
    bool ok = true;
    int jj = 0;
    for (int j = next_tile(0); j < jend; j = next_tile(j + 1), ++jj) {
      const int s = jj & 1;
      if (!mbar_wait_warp(bar_sfull + s, (jj >> 1) & 1, wd)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + s * 128 + c * 32, r[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence(r[c]);
      float sv[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) sv[c] = __uint_as_float(r[c >> 5][c & 31]);
      const bool edge = (j + 1) * kBlock > kv_bound || (CAUSAL && j == qt);
      if (edge) {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int key = j * kBlock + c;
          if (key >= kv_bound || (CAUSAL && key > row)) sv[c] = -INFINITY;
        }
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = sv[i];
#pragma unroll
      for (int c = 8; c < 128; ++c) mx[c & 7] = fmaxf(mx[c & 7], sv[c]);
      const float tile_max = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                   fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float m_new = fmaxf(m, tile_max * scale_log2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m - m_use);
      uint32_t pk[64];
      float ps[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) ps[i] = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = ex2(fmaf(sv[2 * c], scale_log2, -m_use));
        const float p1 = ex2(fmaf(sv[2 * c + 1], scale_log2, -m_use));
        pk[c] = pack_bf16(p0, p1);
        ps[c & 7] += p0 + p1;
      }
      const float tile_sum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      // P_{jj-1} V must be done before P is overwritten and O is rescaled.
      if (jj >= 1) {
        if (!mbar_wait_warp(bar_odone, (jj - 1) & 1, wd)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      // P -> shared memory, K-major with the 128-byte swizzle the MMA expects:
      // row t, 16-byte unit u of chunk (u / 8) lands at unit (u % 8) ^ (t % 8).
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint32_t addr =
            p_base + (u >> 3) * kChunk + t * 128 + ((((u & 7) ^ (t & 7))) << 4);
        st_shared_v4(addr, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
      if (jj >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c0 = 0; c0 < D / 32; ++c0) {
          uint32_t o[32];
          tmem_ld32(lane_base + 256 + c0 * 32, o);
          tmem_wait_ld();
          reg_fence(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(lane_base + 256 + c0 * 32, o);
        }
        tmem_wait_st();
      }
      l = l * alpha + tile_sum;
      m = m_new;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pfull);
    }
    // ------------------------------------------------------------ epilogue
    bool have = ok && jj > 0;
    if (have) have = mbar_wait_warp(bar_odone, (jj - 1) & 1, wd);
    if (have) tc_fence_after();
    const bool live = have && l > 0.f;
    const float inv = live ? 1.f / l : 0.f;
    const bool row_ok = row < N;
    uint4* orow = reinterpret_cast<uint4*>(out + (static_cast<size_t>(bh) * N + row) * D);
#pragma unroll
    for (int c0 = 0; c0 < D / 32; ++c0) {
      uint32_t o[32];
      if (have) {
        tmem_ld32(lane_base + 256 + c0 * 32, o);
        tmem_wait_ld();
        reg_fence(o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      if (row_ok) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
          w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
          w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
          w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
          orow[c0 * 4 + v] = w;
        }
      }
    }
    if (row_ok) lse_out[static_cast<size_t>(bh) * N + row] = live ? (m + log2f(l)) * kLn2 : -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_fwd_t(const FwdLaunch& a, cudaStream_t stream) {
  using L = FwdLayout<D>;
  auto kern = fwd_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
  if (e != cudaSuccess) return e;
  const int nqt = (a.N + kBlock - 1) / kBlock;
  const dim3 grid(nqt, a.H, a.B);
  const float scale_log2 = a.scale * 1.4426950408889634f;
  kern<<<grid, kThreads, L::kSmem, stream>>>(a.tm_q, a.tm_k, a.tm_v,
                                             static_cast<__nv_bfloat16*>(a.o), a.lse, a.H, a.N,
                                             scale_log2, a.kv_len, a.block_mask, a.status,
                                             a.wait_limit);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream) {
  const bool causal = a.causal != 0;
  if (a.d == 64) return causal ? launch_fwd_t<64, true>(a, stream) : launch_fwd_t<64, false>(a, stream);
  return causal ? launch_fwd_t<128, true>(a, stream) : launch_fwd_t<128, false>(a, stream);
}

}  // namespace fa
