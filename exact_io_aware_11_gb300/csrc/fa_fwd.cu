// Forward pass of exact attention (dense, causal, key-padded and block-sparse)
// as one fused sm_103a kernel.
//
// Method: FlashAttention's tiling with online softmax rescaling -- Q, K, V are
// split into blocks that are copied from HBM into on-chip memory, attention is
// computed block by block, the softmax normaliser is accumulated incrementally
// and the N x N matrices S and P are never written to HBM (condensed paper
// sample_paper.md, section 3 "Tiling" / "Softmax rescaling"; Medium article
// "No More Quadratic Complexity for Transformers", Figure 1). The pages put
// K/V in the outer loop; here each CTA keeps two 128-row Q tiles resident and
// streams the K/V tiles past them, which gives the same exact result, keeps
// the running statistics in registers and loads every K/V tile once for two
// Q tiles.
//
// One CTA = Q tiles A and B of one (batch, head); 10 warps:
//   warps 0-3   softmax of tile A: thread t owns query row t (= TMEM lane t)
//   warps 4-7   softmax of tile B
//   warp 8      TMA producer: Q_A, Q_B once; K_j, V_j through separate rings
//   warp 9      MMA issuer, in the order
//                 S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
//               so that the tensor core computes one tile's MMAs while the
//               other tile's softmax runs.
// TMEM columns: S_A [0,128), S_B [128,256) (fp32). After reading S_t the
// softmax writes P_t in bf16 over the first 64 columns of S_t and the PV MMA
// takes it from there as its A operand, so P never touches shared memory.
// O_A [256, 256+d), O_B [256+d, 256+2d): fp32 accumulators.
//
// Rescaling is lazy: a row's reference maximum m only moves when the new
// tile's maximum exceeds it by more than 8 (log2 units), so P <= 2^8 and O is
// rescaled in TMEM only on those rare tiles; the final O / l is exact because
// O and l always share the same m.
//
// CTA x holds Q tiles 2x and 2x+1, so both tiles are active on (almost)
// every K/V step and their softmax phases alternate on the tensor core;
// causal grids run the heaviest pairs first.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 320;
constexpr int kChunk = 128 * 128;  // bytes of one 128-row x 128-byte swizzled chunk (64 bf16 cols)
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 256

template <int D>
struct FwdLayout {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kChunks * kChunk;  // one 128 x D bf16 tile
  static constexpr int kKS = 3;                   // K ring slots
  static constexpr int kVS = (D == 128) ? 2 : 3;  // V ring slots
  static constexpr int kQ = 0;                    // Q_A, Q_B (reused to stage O)
  static constexpr int kK = kQ + 2 * kTile;
  static constexpr int kV = kK + kKS * kTile;
  static constexpr int kBar = kV + kVS * kTile;
  static constexpr int kEnd = kBar + 256;
  static constexpr int kSmem = kEnd + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t kTO = 256;       // O_A; O_B at kTO + D
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
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

// Which K/V tiles a Q tile visits: j < end, and the block-mask bit if any.
struct TileSet {
  int end;
  const uint8_t* mrow;
  __device__ bool has(int j) const { return j < end && (mrow == nullptr || mrow[j] != 0); }
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               float* __restrict__ lse_out, int H, int N, float scale_log2,
               const int32_t* __restrict__ kv_len, const uint8_t* __restrict__ block_mask,
               int* status, long long wait_limit) {
  using L = FwdLayout<D>;
  constexpr int KS = L::kKS, VS = L::kVS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* bar_q = bars + 0;
  uint64_t* bar_kfull = bars + 1;    // [KS]
  uint64_t* bar_kempty = bars + 4;   // [KS]
  uint64_t* bar_vfull = bars + 7;    // [VS]
  uint64_t* bar_vempty = bars + 10;  // [VS]
  uint64_t* bar_sfull = bars + 13;   // [2]
  uint64_t* bar_pfull = bars + 15;   // [2]
  uint64_t* bar_odone = bars + 17;   // [2]
  uint64_t* bar_final = bars + 19;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  int* abort_flag = reinterpret_cast<int*>(bars + 21);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nqt = (N + kBlock - 1) / kBlock;
  const int bh = blockIdx.z * H + blockIdx.y;
  // Q tiles of this CTA (B = -1 when there is none) and the K/V tiles each visits.
  // Adjacent tiles share a CTA, so both are active on (almost) every K/V step
  // and their softmax phases can alternate. Causal CTAs run heaviest first.
  const int pair = CAUSAL ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
  const int qtA = 2 * pair;
  const int qtB = 2 * pair + 1 < nqt ? 2 * pair + 1 : -1;
  int kv_bound = N;
  if (kv_len != nullptr) kv_bound = min(N, max(0, kv_len[blockIdx.z]));
  const int kv_tiles = (kv_bound + kBlock - 1) / kBlock;
  const TileSet tsA{CAUSAL ? min(kv_tiles, qtA + 1) : kv_tiles,
                    block_mask != nullptr ? block_mask + static_cast<size_t>(qtA) * nqt : nullptr};
  const TileSet tsB{qtB < 0 ? 0 : (CAUSAL ? min(kv_tiles, qtB + 1) : kv_tiles),
                    (block_mask != nullptr && qtB >= 0) ? block_mask + static_cast<size_t>(qtB) * nqt
                                                        : nullptr};
  const int uend = max(tsA.end, tsB.end);
  auto next_union = [&](int j) {
    while (j < uend && !tsA.has(j) && !tsB.has(j)) ++j;
    return j;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(bar_kfull + s, 1);
      mbar_init(bar_kempty + s, 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(bar_vfull + s, 1);
      mbar_init(bar_vempty + s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_sfull + t, 1);
      mbar_init(bar_pfull + t, 4);
      mbar_init(bar_odone + t, 1);
    }
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
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_o);
      mbar_expect_tx(bar_q, (qtB >= 0 ? 2 : 1) * L::kTile);
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_3d(smem + L::kQ + c * kChunk, &tm_q, bar_q, c * 64, qtA * kBlock, bh);
      if (qtB >= 0)
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(smem + L::kQ + L::kTile + c * kChunk, &tm_q, bar_q, c * 64, qtB * kBlock, bh);
      int k_issued = 0, v_issued = 0;
      int u = 0;
      for (int j = next_union(0); j < uend; j = next_union(j + 1), ++u) {
        const int ks = u % KS, vs = u % VS;
        if (u >= KS && !mbar_wait(bar_kempty + ks, ((u / KS) - 1) & 1, wd)) break;
        mbar_expect_tx(bar_kfull + ks, L::kTile);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(smem + L::kK + ks * L::kTile + c * kChunk, &tm_k, bar_kfull + ks, c * 64,
                      j * kBlock, bh);
        k_issued = u + 1;
        if (u >= VS && !mbar_wait(bar_vempty + vs, ((u / VS) - 1) & 1, wd)) break;
        mbar_expect_tx(bar_vfull + vs, L::kTile);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(smem + L::kV + vs * L::kTile + c * kChunk, &tm_v, bar_vfull + vs, c * 64,
                      j * kBlock, bh);
        v_issued = u + 1;
      }
      // Let every copy in flight land before the CTA can exit (bounded).
      mbar_wait_drain(bar_q, 0, wait_limit);
      for (int t = max(0, k_issued - KS); t < k_issued; ++t)
        mbar_wait_drain(bar_kfull + (t % KS), (t / KS) & 1, wait_limit);
      for (int t = max(0, v_issued - VS); t < v_issued; ++t)
        mbar_wait_drain(bar_vfull + (t % VS), (t / VS) & 1, wait_limit);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer (one lane)
    // The issuing thread sits on the critical path between the two softmax
    // warpgroups, so it runs alone, waits without warp-wide votes, and places
    // a tcgen05 fence only after waiting for P (the one cross-thread TMEM
    // dependency: P_t written by tcgen05.st, and S_t columns read by
    // tcgen05.ld before S_t(j+1) overwrites them).
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);  // Q, K both K-major
      constexpr uint32_t kIdO = idesc_bf16(128, D, false, true);     // P (TMEM), V MN-major
      // Descriptors built once; per MMA only a compile-time offset is added.
      const uint64_t q_desc = sdesc_sw128(smem_u32(smem + L::kQ), 16, 1024);     // K-major
      const uint64_t k_desc = sdesc_sw128(smem_u32(smem + L::kK), 16, 1024);     // K-major
      const uint64_t v_desc = sdesc_sw128(smem_u32(smem + L::kV), kChunk, 1024);  // MN-major
      int n_pvA = 0, n_pvB = 0;  // P V MMAs issued per tile
      bool ok = mbar_wait_spin(bar_q, 0, wd);
      auto issue_s = [&](int t, int u) -> bool {
        if (!mbar_wait_spin(bar_kfull + (u % KS), (u / KS) & 1, wd)) return false;
        const uint64_t qd = desc_adv(q_desc, t * L::kTile);
        const uint64_t kd = desc_adv(k_desc, (u % KS) * L::kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
          mma_ss(tmem + t * 128, desc_adv(qd, off), desc_adv(kd, off), kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_sfull + t);
        return true;
      };
      auto issue_pv = [&](int t, int u) -> bool {
        const int npv = t ? n_pvB : n_pvA;
        if (!mbar_wait_spin(bar_pfull + t, npv & 1, wd)) return false;
        if (!mbar_wait_spin(bar_vfull + (u % VS), (u / VS) & 1, wd)) return false;
        tc_fence_after();
        const uint64_t vd = desc_adv(v_desc, (u % VS) * L::kTile);
        const uint32_t acc0 = npv > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          // A = P (bf16 pairs in the first 64 columns of S_t), B = V, MN-major.
          mma_ts(tmem + L::kTO + t * D, tmem + t * 128 + kk * 8, desc_adv(vd, kk * 2048), kIdO,
                 kk > 0 ? 1u : acc0);
        }
        mma_commit(bar_odone + t);
        if (t) ++n_pvB; else ++n_pvA;
        return true;
      };
      if (ok) {
        int u = 0;
        int j = next_union(0);
        if (j < uend) {
          if (tsA.has(j)) ok = issue_s(0, 0);
          if (ok && tsB.has(j)) ok = issue_s(1, 0);
          if (ok) mma_commit(bar_kempty + 0);
        }
        while (ok && j < uend) {
          const int jn = next_union(j + 1);
          const int un = u + 1;
          // tile A: P_A(j) V_j, then S_A(j+1) over the columns P_A(j) just left
          if (tsA.has(j)) ok = issue_pv(0, u);
          if (ok && jn < uend && tsA.has(jn)) ok = issue_s(0, un);
          if (ok && tsB.has(j)) ok = issue_pv(1, u);
          if (ok) mma_commit(bar_vempty + (u % VS));
          if (ok && jn < uend && tsB.has(jn)) ok = issue_s(1, un);
          if (ok && jn < uend) mma_commit(bar_kempty + (un % KS));
          j = jn;
          u = un;
        }
      }
      mma_commit(bar_final);
      mbar_wait_drain(bar_final, 0, wait_limit);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int t = warp >> 2;              // which Q tile
    const int r = threadIdx.x & 127;      // row within the tile == TMEM lane
    const int qt = t ? qtB : qtA;
    if (qt >= 0) {
      const int row = qt * kBlock + r;
      const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
      const uint32_t s_col = t * 128;
      const uint32_t o_col = L::kTO + t * D;
      const TileSet my = t ? tsB : tsA;
      float m = -INFINITY;  // reference max, log2 units (scale folded in)
      float l = 0.f;        // sum of exp2(s * scale_log2 - m) over visited keys
      bool ok = true;
      int n = 0;
      for (int j = 0; j < my.end; ++j) {
        if (!my.has(j)) continue;
        if (!mbar_wait_warp(bar_sfull + t, n & 1, wd)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t rs[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + s_col + c * 32, rs[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence(rs[c]);
        float sv[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) sv[c] = __uint_as_float(rs[c >> 5][c & 31]);
        if ((j + 1) * kBlock > kv_bound || (CAUSAL && j == qt)) {
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const int key = j * kBlock + c;
            if (key >= kv_bound || (CAUSAL && key > row)) sv[c] = -INFINITY;
          }
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = max3(sv[i], sv[i + 8], sv[i + 16]);
#pragma unroll
        for (int c = 24; c < 128; c += 16) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            mx[i] = (c + 8 + i < 128) ? max3(mx[i], sv[c + i], sv[c + 8 + i]) : fmaxf(mx[i], sv[c + i]);
        }
        const float tmax =
            max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) *
            scale_log2;
        const bool grow = tmax > m + kRescaleThreshold;
        const float m_new = grow ? tmax : m;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = grow ? ex2(m - m_use) : 1.f;
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
        const float tsum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        // P_t over the first 64 columns of S_t (its fp32 values are already in registers)
        tmem_st32(lane_base + s_col, *reinterpret_cast<uint32_t(*)[32]>(pk));
        tmem_st32(lane_base + s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
        if (n >= 1 && __any_sync(0xffffffffu, grow)) {
          // O must be quiescent (P_t(n-1) V done) before it is rescaled.
          if (!mbar_wait_warp(bar_odone + t, (n - 1) & 1, wd)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D / 32; ++c0) {
            uint32_t o[32];
            tmem_ld32(lane_base + o_col + c0 * 32, o);
            tmem_wait_ld();
            reg_fence(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(lane_base + o_col + c0 * 32, o);
          }
        }
        tmem_wait_st();
        l = l * alpha + tsum;
        m = m_new;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pfull + t);
        ++n;
      }
      // ---------------------------------------------------------- epilogue
      bool have = ok && n > 0;
      if (have) have = mbar_wait_warp(bar_odone + t, (n - 1) & 1, wd);
      if (have) tc_fence_after();
      const bool live = have && l > 0.f;
      const float inv = live ? 1.f / l : 0.f;
      // O row -> the Q_t buffer (free now), same 128-byte swizzled layout as Q,
      // then one TMA store per 64-column chunk (rows >= N are clipped).
      uint8_t* stage = smem + L::kQ + t * L::kTile;
      const uint32_t st_base = smem_u32(stage);
#pragma unroll
      for (int c0 = 0; c0 < D / 32; ++c0) {
        uint32_t o[32];
        if (have) {
          tmem_ld32(lane_base + o_col + c0 * 32, o);
          tmem_wait_ld();
          reg_fence(o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int unit = c0 * 4 + v;  // 16-byte unit of the row (8 columns)
          const uint32_t addr = st_base + (unit >> 3) * kChunk + r * 128 + (((unit & 7) ^ (r & 7)) << 4);
          st_shared_v4(addr,
                       pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv),
                       pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv),
                       pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv),
                       pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv));
        }
      }
      if (row < N)
        lse_out[static_cast<size_t>(bh) * N + row] = live ? (m + log2f(l)) * kLn2 : -INFINITY;
      fence_proxy_async_smem();
      named_bar_sync(1 + t, 128);
      if (r == 0) {
        for (int c = 0; c < L::kChunks; ++c) tma_store_3d(&tm_o, stage + c * kChunk, c * 64, qt * kBlock, bh);
        bulk_commit();
        bulk_wait_read0();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
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
  const dim3 grid((nqt + 1) / 2, a.H, a.B);
  const float scale_log2 = a.scale * 1.4426950408889634f;
  kern<<<grid, kThreads, L::kSmem, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.lse, a.H, a.N,
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
