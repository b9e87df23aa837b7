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
// 1. bwd_pre_kernel   D = rowsum(dO * O), -LSE * log2(e), zero the fp32 dQ
//                     accumulator (bandwidth-bound, 16-byte accesses).
// 2. bwd_main_kernel  persistent, one CTA per SM; a work item is one 128-key
//                     tile j of one (batch, head). K_j and V_j stay in shared
//                     memory, dK_j and dV_j accumulate in TMEM, and the CTA
//                     loops over the Q tiles i:
//                       S^T  = K_j Q_i^T    TMEM, key rows on lanes
//                       dP^T = V_j dO_i^T   TMEM
//                       P^T  = exp2(S^T * scale*log2e - LSE2_i), bf16, written
//                              back into the S^T columns and used from TMEM
//                       dV_j += P^T dO_i
//                       dS^T = P^T * (dP^T - D_i), bf16 -> shared memory
//                       dK_j += dS^T Q_i
//                       dQ_i += scale dS K_j  TMEM -> shared memory (fp32) -> TMA
//                              bulk reduce-adds into the fp32 workspace
//                              accumulator
//                     Warps 0-7 compute P and dS (warps w and w+4 share the
//                     key rows of TMEM lane quarter w % 4 and split the 128
//                     query columns), warp 8 issues TMA, warp 9 issues
//                     tcgen05.mma, warps 10-13 drain dQ and, at the end of
//                     an item, write dK_j / dV_j from TMEM. S^T of tile i+1
//                     (also of the next item's first tile) is computed while
//                     dS of tile i is being formed.
// 3. dq_convert_kernel  dQ bf16 = fp32 accumulator.
#pragma once

#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_philox.cuh"
#include "fa_ptx.cuh"
#include "fa_sched.cuh"

namespace fa {
namespace {

constexpr int kThreads = 448;
constexpr int kChunk = 128 * 128;  // one 128-row x 128-byte swizzled chunk
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdLayout {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kChunks * kChunk;     // 128 x D bf16
  static constexpr int kKVS = (D == 64) ? 2 : 1;     // K/V stages (next item's K/V prefetched)
  static constexpr int kQS = 2;                      // Q (+ LSE2 / D) stages
  static constexpr int kDS = (D == 64) ? 2 : 1;      // dO stages
  static constexpr int kDQChunks = 2;  // d = 64: 128 x 32 fp32 chunks staged at once
  // d = 128: per drain warp a ring of kDQRing boxes of 32 rows x 16 fp32 columns
  static constexpr int kDQRing = 3, kDQBox = 32 * 64;
  static constexpr int kDQBytes = (D == 64) ? kDQChunks * kChunk : 4 * kDQRing * kDQBox;
  static constexpr int kKV = 0;                      // stage s: K at kKV + 2 s kTile, then V
  static constexpr int kQ = kKV + 2 * kKVS * kTile;
  static constexpr int kDO = kQ + kQS * kTile;
  static constexpr int kStat = kDO + kDS * kTile;    // per Q stage: lse2[128], delta[128]
  static constexpr int kDSb = kStat + kQS * 1024;    // dS^T, bf16, 2 chunks
  static constexpr int kDQ = kDSb + 2 * kChunk;      // dQ staging (fp32, swizzled)
  static constexpr int kBar = kDQ + kDQBytes;
  // barriers etc.; the producer's tile list; the cost-sorted group table
  static constexpr int kEnd = kBar + 512 + 128 + 2 * kOrderMax;
  static constexpr int kSmem = kEnd + 1024;
  static_assert(kSmem <= 227 * 1024, "shared memory of one CTA");
  // TMEM columns
  static constexpr uint32_t kTS = 0, kTDP = 128, kTDV = 256, kTDK = 256 + D;
  static constexpr uint32_t kTDQ = (D == 64) ? 384 : 128;  // d=128: dQ reuses the dP^T columns
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int x,
                                                  int y, int z) {
  if (FA_CHECK_FAILS((x & 3) == 0 && x >= 0 && y >= 0 && z >= 0 && (smem_u32(src) & 127u) == 0)) return;
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// ----------------------------------------------------------------- preprocess
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      const float* __restrict__ lse,
                                                      float* __restrict__ lse2,
                                                      float* __restrict__ delta,
                                                      float* __restrict__ dq_acc, int BH, int N,
                                                      int Npad, Strides st, int H) {
  constexpr int kPer = D / 8;  // threads per row (8 elements = 16 bytes each)
  grid_dep_wait();
  grid_dep_launch();
  const long long total = static_cast<long long>(BH) * Npad * kPer;
  const long long total32 = (total + 31) & ~31LL;
  // Row-major [B, H, N, d] (the common case) needs no division by H.
  const bool dense = st.n == D && st.h == static_cast<long long>(N) * D &&
                     st.b == static_cast<long long>(H) * N * D;
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
      const long long off = (dense ? (static_cast<long long>(bh) * N + n) * D
                                   : row_offset(st, H, bh, n)) + part * 8;
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
        float l2 = -INFINITY;  // padding rows and rows that saw no key get P = 0
        if (valid) {
          const float v = lse[static_cast<size_t>(bh) * N + n];
          if (v != -INFINITY) l2 = -(v * kLog2e);
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
                                                         int N, int Npad, Strides st, int H) {
  constexpr int kPer = D / 8;
  grid_dep_wait();
  grid_dep_launch();
  const long long total = static_cast<long long>(BH) * N * kPer;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const bool dense = st.n == D && st.h == static_cast<long long>(N) * D &&
                     st.b == static_cast<long long>(H) * N * D;
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
    const long long off = dense ? row * D : row_offset(st, H, static_cast<int>(bh), static_cast<int>(n));
    *reinterpret_cast<uint4*>(dq + off + part * 8) = w;
  }
}

// ----------------------------------------------------------------- work items
// One work unit: key tile j of one (batch, head), met by the Q tiles of
// steps [sb, se) of its item (Q tiles i0 + sb .. i0 + se - 1 without a block
// mask; with one, the kept Q tiles). A unit whose keys all lie beyond the
// valid length has no iterations; its dK and dV rows are written as zeros.
// `slot` >= 0: the unit is part of a split item and its dK, dV go to that
// workspace slot for the merge kernel.
struct BwdItem {
  int bh, j, n_iter, kv_bound, slot;
  TileSet ts;  // the Q tiles met
};

template <bool CAUSAL>
__host__ __device__ __forceinline__ int bwd_steps(const BwdGrid& g, int k) {
  return bwd_item_steps(g.nt, g.BH, CAUSAL, k);
}

// Unit u's item. With a block mask, counting the kept Q tiles is
// warp-collective, so every lane of the calling warp must take part.
// `order`: the cost-sorted group table (fa_sched.cuh) or null (index order).
template <bool CAUSAL, int MODE>
__device__ __forceinline__ BwdItem make_bwd_item(const BwdGrid& g, const Unit& u, const uint16_t* order) {
  constexpr bool SPARSE = MODE == kModeSparse;
  BwdItem x;
  if (!SPARSE || order == nullptr) {
    bwd_item_coords(g.nt, g.BH, CAUSAL, u.k, x.bh, x.j);
  } else {  // groups: key tiles; members: (batch, head)
    const int grp = u.k / g.BH;
    x.j = order[grp];
    x.bh = u.k - grp * g.BH;
  }
  x.slot = u.slot;
  x.kv_bound = g.N;
  if (g.kv_len != nullptr) x.kv_bound = min(g.N, max(0, g.kv_len[x.bh / g.H]));
  const int i0 = CAUSAL ? x.j : 0;
  x.ts = TileSet{i0 + u.sb, min(g.nt, i0 + u.se), SPARSE ? g.mask + x.j : nullptr, g.nt};
  int n = x.ts.end - x.ts.begin;
  if constexpr (SPARSE) {
    TileWalk<> w;
    w.init(x.ts);
    n = w.count();
  }
  x.n_iter = x.j * kBlock < x.kv_bound ? n : 0;
  return x;
}

// Position of the MMA issuer in this CTA's flattened sequence of iterations:
// iteration `it` of `n` of the t-th unit that has iterations, the g-th
// iteration overall (ring slots and barrier phases follow t and g).
template <bool CAUSAL, int MODE>
struct BwdCursor {
  int r = 0, it = 0, n = 0, t = 0, g = 0;
  bool valid = false;
  template <typename UnitFn>
  __device__ void seek(const BwdGrid& G, UnitFn unit, const uint16_t* order) {
    for (;; ++r) {
      const Unit u = unit(r);
      if (u.k < 0) {
        valid = false;
        return;
      }
      const int n_iter = make_bwd_item<CAUSAL, MODE>(G, u, order).n_iter;
      if (n_iter > 0) {
        n = n_iter;
        it = 0;
        valid = true;
        return;
      }
    }
  }
  template <typename UnitFn>
  __device__ void next(const BwdGrid& G, UnitFn unit, const uint16_t* order) {
    ++g;
    if (++it < n) return;
    ++t;
    ++r;
    seek(G, unit, order);
  }
};

// The cost-sorted item order of a block-sparse backward pass (fa_sched.cuh),
// built by the whole CTA before any TMA load: the groups are key tiles, each
// costing the Q tiles that keep it. `scratch` (>= 6656 bytes) is a tile
// buffer that no copy has written yet; every thread of the CTA takes part.
// (Key padding alone is not sorted: it gained 1-2 % on a BERT-like pass.)
template <bool CAUSAL>
__device__ __forceinline__ void bwd_sort_items(int nt, const int32_t* kv_len, const uint8_t* mask,
                                               uint8_t* scratch, uint64_t* bars) {
  const int G = kv_len == nullptr ? nt : 0;
  if (G == 0 || G > kOrderMax) return;  // uniform over the CTA
  int* cost = reinterpret_cast<int*>(scratch);
  int* hist = cost + kOrderMax;
  for (int i = threadIdx.x; i < G; i += blockDim.x) cost[i] = 0;
  __syncthreads();
  for_kept_blocks(mask, nt, [&](int i, int j) {
    if (!CAUSAL || i >= j) atomicAdd(&cost[j], 1);
  });
  __syncthreads();
  if ((threadIdx.x >> 5) == 0)
    sort_groups(cost, G, min(kCostMax, nt), hist, reinterpret_cast<uint16_t*>(bars + 64) + 64);
  fence_proxy_async_smem();  // the scratch tile is next written by TMA
  if (threadIdx.x == 0) *reinterpret_cast<volatile int*>(bars + kOrderFlagWord) = 1;
  __syncthreads();
}

// ----------------------------------------------------------------- main kernel
// Persistent: one CTA per SM walks its items; barrier phases run on across
// items, K/V of the next item are prefetched when shared memory holds two
// stages (d = 64), and dK/dV are written from TMEM by the dQ drain warps while
// the compute warps already form P of the next item.
// DROP: dropout (fa_philox.cuh) regenerated from the element indices: dV is
// accumulated from the dropped P^T (its 1 / (1 - p') applied when dV leaves
// TMEM) and dS = P * (Z dP_dropped / (1 - p') - D).
// MODE (kModePlain, kModeSparse, kModeSplit): the variant compiled -- dense
// Q-tile ranges over whole items, the Q tiles a block mask keeps, or dense
// ranges with the last wave's items cut into parts whose dK, dV go to the
// workspace for the merge kernel.
template <int D, bool CAUSAL, int MODE, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dqacc, const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv, __nv_bfloat16* __restrict__ dk,
                    __nv_bfloat16* __restrict__ dv, const float* __restrict__ lse2,
                    const float* __restrict__ delta, BwdGrid grid, int Npad, float scale,
                    DropoutParams dp, int* status, long long wait_limit) {
  using L = BwdLayout<D>;
  constexpr int QS = L::kQS, DS = L::kDS, KVS = L::kKVS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* bar_kvfull = bars + 0;    // [KVS]
  uint64_t* bar_kvempty = bars + 2;   // [KVS]
  uint64_t* bar_qfull = bars + 4;     // [QS]
  uint64_t* bar_qempty = bars + 6;    // [QS]
  uint64_t* bar_dofull = bars + 8;    // [DS]
  uint64_t* bar_doempty = bars + 10;  // [DS]
  uint64_t* bar_sfull = bars + 12;
  uint64_t* bar_dpfull = bars + 13;
  uint64_t* bar_pready = bars + 14;
  uint64_t* bar_dsready = bars + 15;
  uint64_t* bar_dsfree = bars + 16;
  uint64_t* bar_dqfull = bars + 17;
  uint64_t* bar_dqfree = bars + 18;
  uint64_t* bar_accfull = bars + 19;  // dV and dK of an item complete
  uint64_t* bar_dvempty = bars + 20;  // dV read out of TMEM
  uint64_t* bar_dkempty = bars + 21;  // dK read out of TMEM
  uint64_t* bar_final = bars + 22;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 23);
  int* abort_flag = reinterpret_cast<int*>(bars + 24);
  uint64_t* bar_dpfree = bars + 25;   // dP^T read out of TMEM (d = 64)
  TailRange* tail_sh = reinterpret_cast<TailRange*>(bars + 26);  // this CTA's share of a split tail
  uint8_t* walk_list = reinterpret_cast<uint8_t*>(bars + 64);     // [128] the producer's Q tiles of a window (sparse)
  // then [kOrderMax] cost-sorted groups from walk_list + 128 (item_order)
  // d = 64: dQ has TMEM columns of its own, so dP^T of the next Q tile can be
  // issued as soon as the compute warps have read dP^T of this one, ahead of
  // this tile's dK and dQ MMAs in the in-order tensor pipe.
  constexpr bool kEarlyDP = (D == 64);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  check_init(status);
  const int N = grid.N;
  const float scale_log2 = scale * kLog2e;

  if (threadIdx.x == 0) {
    for (int s = 0; s < KVS; ++s) {
      mbar_init(bar_kvfull + s, 1);
      mbar_init(bar_kvempty + s, 1);
    }
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
    mbar_init(bar_accfull, 1);
    mbar_init(bar_dvempty, 4);
    mbar_init(bar_dkempty, 4);
    mbar_init(bar_final, 1);
    mbar_init(bar_dpfree, 8);
    *abort_flag = 0;
    *reinterpret_cast<int*>(bars + kOrderFlagWord) = 0;  // index order unless sorted below
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  auto steps = [&](int k) { return bwd_steps<CAUSAL>(grid, k); };
  if constexpr (MODE == kModeSplit) {
    if (warp == 8) {
      const TailRange tr = tail_range(grid.plan, blockIdx.x, steps);
      if (lane == 0) *tail_sh = tr;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();  // the previous kernel's outputs (Q, K, V, O, ...) are complete
  grid_dep_launch();
  const Watchdog wd{wait_limit, status, abort_flag};
  // Cost-sorted item order with a block mask (bwd_sort_items).
  constexpr bool kSort = MODE == kModeSparse;
  if constexpr (kSort) bwd_sort_items<CAUSAL>(grid.nt, grid.kv_len, grid.mask, smem + L::kKV, bars);
  // The r-th unit of this CTA, or a unit with k < 0: the split kernel runs
  // the CTA's run of the tail; the others whole items [0, plan.whole) in a
  // snake over the item list.
  auto unit = [&](int r) -> Unit {
    if constexpr (MODE == kModeSplit) {
      return tail_unit(tail_sh, r, blockIdx.x, steps);
    } else {
      Unit u{-1, 0, 1 << 30, -1};
      const int G = gridDim.x, c = blockIdx.x;
      if (r * G >= grid.plan.whole) return u;
      const int k = r * G + ((r & 1) ? G - 1 - c : c);
      if (k < grid.plan.whole) u.k = k;
      return u;
    }
  };
  // The Q tiles of a unit, window by window: without a block mask one run
  // [begin, end); with one, each 128-tile window's kept tiles are listed in
  // the warp's shared-memory list. Returns the tiles of window w0 and sets
  // `base` (tile = base + idx) or lists them (tile = w0 + list[idx]).
  uint8_t* list = walk_list;  // the producer's (the only warp that lists tiles)

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    // Lane 0 waits for free ring slots and issues the copies (with a block
    // mask the whole warp first lists each window's Q tiles).
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_dqacc);
    }
    int t = 0, q_issued = 0, do_issued = 0;
    bool ok = true;
    // K_j, V_j of a unit into the next K/V stage (lane 0); false on an abort.
    auto load_kv = [&](const BwdItem& x) -> bool {
      const int kvs = t % KVS;
      if (t >= KVS && !mbar_wait(bar_kvempty + kvs, ((t / KVS) - 1) & 1, wd)) return false;
      mbar_expect_tx(bar_kvfull + kvs, 2 * L::kTile);
      uint8_t* kv = smem + L::kKV + kvs * 2 * L::kTile;
      for (int c = 0; c < L::kChunks; ++c) {
        tma_load_rows(kv + c * kChunk, &tm_k, bar_kvfull + kvs, c * 64, x.j * kBlock, x.bh, grid.H,
                      grid.st);
        tma_load_rows(kv + L::kTile + c * kChunk, &tm_v, bar_kvfull + kvs, c * 64, x.j * kBlock,
                      x.bh, grid.H, grid.st);
      }
      ++t;
      return true;
    };
    // Q_i (+ its LSE2 and D rows) and dO_i into the next stages (lane 0).
    auto load_q = [&](const BwdItem& x, int i) -> bool {
      const int gq = q_issued, qs = gq % QS, ds = gq % DS;
      if (gq >= QS && !mbar_wait(bar_qempty + qs, ((gq / QS) - 1) & 1, wd)) return false;
      mbar_expect_tx(bar_qfull + qs, L::kTile + 1024);
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_rows(smem + L::kQ + qs * L::kTile + c * kChunk, &tm_q, bar_qfull + qs, c * 64,
                      i * kBlock, x.bh, grid.H, grid.st);
      const size_t roff = static_cast<size_t>(x.bh) * Npad + static_cast<size_t>(i) * kBlock;
      bulk_load(smem + L::kStat + qs * 1024, lse2 + roff, 512, bar_qfull + qs);
      bulk_load(smem + L::kStat + qs * 1024 + 512, delta + roff, 512, bar_qfull + qs);
      q_issued = gq + 1;
      if (gq >= DS && !mbar_wait(bar_doempty + ds, ((gq / DS) - 1) & 1, wd)) return false;
      mbar_expect_tx(bar_dofull + ds, L::kTile);
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_rows(smem + L::kDO + ds * L::kTile + c * kChunk, &tm_do, bar_dofull + ds, c * 64,
                      i * kBlock, x.bh, grid.H, grid.st);
      do_issued = gq + 1;
      return true;
    };
    if constexpr (MODE == kModeSparse) {
      // The whole warp counts and lists the kept Q tiles window by window;
      // lane 0 issues the copies.
      for (int r = 0; ok; ++r) {
        const Unit un = unit(r);
        if (un.k < 0) break;
        const BwdItem x = make_bwd_item<CAUSAL, MODE>(grid, un, kSort ? item_order(bars) : nullptr);
        if (x.n_iter == 0) continue;
        if (lane == 0) ok = load_kv(x);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        for (int w0 = x.ts.begin & ~127; ok && w0 < x.ts.end; w0 += 128) {
          const int cnt = list_window(x.ts, w0, list);
          if (lane == 0)
            for (int idx = 0; ok && idx < cnt; ++idx) ok = load_q(x, w0 + list[idx]);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
      }
    } else if (lane == 0) {
      for (int r = 0; ok; ++r) {
        const Unit un = unit(r);
        if (un.k < 0) break;
        const BwdItem x = make_bwd_item<CAUSAL, MODE>(grid, un, kSort ? item_order(bars) : nullptr);
        if (x.n_iter == 0) continue;
        ok = load_kv(x);
        for (int it = 0; ok && it < x.n_iter; ++it) ok = load_q(x, x.ts.begin + it);
      }
    }
    // Copies still in flight (only after an abort) must land before exit.
    if (lane == 0) {
      for (int u = max(0, t - KVS); u < t; ++u)
        mbar_wait_drain(bar_kvfull + (u % KVS), (u / KVS) & 1, wait_limit);
      for (int u = max(0, q_issued - QS); u < q_issued; ++u)
        mbar_wait_drain(bar_qfull + (u % QS), (u / QS) & 1, wait_limit);
      for (int u = max(0, do_issued - DS); u < do_issued; ++u)
        mbar_wait_drain(bar_dofull + (u % DS), (u / DS) & 1, wait_limit);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer (whole warp)
    // On the critical path: the warp runs converged and an elected lane issues
    // each tcgen05.mma / commit; it polls the barriers (test_wait) and fences
    // only after the waits that follow tcgen05.ld / tcgen05.st of other
    // threads (P^T ready, dS ready, dQ drained, dV/dK read out).
    {
      constexpr uint32_t kIdSS = idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t kIdKM = idesc_bf16(128, D, false, true);     // dV, dK: B MN-major
      constexpr uint32_t kIdMM = idesc_bf16(128, D, true, true);      // dQ: A, B MN-major
      constexpr uint32_t kKVStride = 2 * L::kTile;
      // Descriptors built once; per MMA only an offset is added.
      const uint64_t k_kmaj0 = sdesc_sw128(smem_u32(smem + L::kKV), 16, 1024);
      const uint64_t k_mn0 = sdesc_sw128(smem_u32(smem + L::kKV), kChunk, 1024);
      const uint64_t v_kmaj0 = sdesc_sw128(smem_u32(smem + L::kKV + L::kTile), 16, 1024);
      const uint64_t q_kmaj0 = sdesc_sw128(smem_u32(smem + L::kQ), 16, 1024);
      const uint64_t q_mn0 = sdesc_sw128(smem_u32(smem + L::kQ), kChunk, 1024);
      const uint64_t do_kmaj0 = sdesc_sw128(smem_u32(smem + L::kDO), 16, 1024);
      const uint64_t do_mn0 = sdesc_sw128(smem_u32(smem + L::kDO), kChunk, 1024);
      const uint64_t ds_kmaj = sdesc_sw128(smem_u32(smem + L::kDSb), 16, 1024);
      const uint64_t ds_mn = sdesc_sw128(smem_u32(smem + L::kDSb), kChunk, 1024);
      using Cur = BwdCursor<CAUSAL, MODE>;
      auto kv_ready = [&](const Cur& c) -> bool {
        return mbar_wait_spin_w(bar_kvfull + (c.t % KVS), (c.t / KVS) & 1, wd);
      };
      auto issue_s = [&](const Cur& c) -> bool {
        if (!mbar_wait_spin_w(bar_qfull + (c.g % QS), (c.g / QS) & 1, wd)) return false;
        const uint64_t qd = desc_adv(q_kmaj0, (c.g % QS) * L::kTile);
        const uint64_t kd = desc_adv(k_kmaj0, (c.t % KVS) * kKVStride);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
          mma_ss_w(tmem + L::kTS, desc_adv(kd, off), desc_adv(qd, off), kIdSS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(bar_sfull);
        return true;
      };
      auto issue_dp = [&](const Cur& c) -> bool {
        if (!mbar_wait_spin_w(bar_dofull + (c.g % DS), (c.g / DS) & 1, wd)) return false;
        const uint64_t dd = desc_adv(do_kmaj0, (c.g % DS) * L::kTile);
        const uint64_t vd = desc_adv(v_kmaj0, (c.t % KVS) * kKVStride);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
          mma_ss_w(tmem + L::kTDP, desc_adv(vd, off), desc_adv(dd, off), kIdSS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(bar_dpfull);
        return true;
      };
      Cur cur;
      cur.seek(grid, unit, kSort ? item_order(bars) : nullptr);
      bool ok = cur.valid && kv_ready(cur) && issue_s(cur) && issue_dp(cur);
      while (ok && cur.valid) {
        Cur nx = cur;
        nx.next(grid, unit, kSort ? item_order(bars) : nullptr);
        const int gq = cur.g;
        const bool first = cur.it == 0, last = cur.it == cur.n - 1;
        const uint64_t q_mn = desc_adv(q_mn0, (gq % QS) * L::kTile);
        const uint64_t do_mn = desc_adv(do_mn0, (gq % DS) * L::kTile);
        const uint64_t k_mn = desc_adv(k_mn0, (cur.t % KVS) * kKVStride);
        const uint32_t acc0 = first ? 0u : 1u;
        // dV += P^T dO: P^T (bf16) sits in the S^T columns [0,32) and [64,96)
        if (!mbar_wait_spin_w(bar_pready, gq & 1, wd)) { ok = false; break; }
        if (first && cur.t >= 1 && !mbar_wait_spin_w(bar_dvempty, (cur.t - 1) & 1, wd)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          const uint32_t a_col = L::kTS + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
          mma_ts_w(tmem + L::kTDV, tmem + a_col, desc_adv(do_mn, kk * 2048), kIdKM,
                 kk > 0 ? 1u : acc0);
        }
        mma_commit_w(bar_doempty + (gq % DS));
        // S^T of the next Q tile while dS of this one is formed. Across items
        // with a single K/V stage it must wait until this item's dQ is issued.
        const bool hoist = nx.valid && (KVS > 1 || !last);
        if (hoist && !((nx.it > 0 || kv_ready(nx)) && issue_s(nx))) { ok = false; break; }
        if (kEarlyDP && nx.valid) {  // hoist is true here: KVS > 1 at d = 64
          if (!mbar_wait_spin_w(bar_dpfree, gq & 1, wd)) { ok = false; break; }
          tc_fence_after();
          if (!issue_dp(nx)) { ok = false; break; }
        }
        if (!mbar_wait_spin_w(bar_dsready, gq & 1, wd)) { ok = false; break; }
        if (D == 64 && gq >= 1 && !mbar_wait_spin_w(bar_dqfree, (gq - 1) & 1, wd)) { ok = false; break; }
        if (first && cur.t >= 1 && !mbar_wait_spin_w(bar_dkempty, (cur.t - 1) & 1, wd)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          mma_ss_w(tmem + L::kTDK, desc_adv(ds_kmaj, (kk >> 2) * kChunk + (kk & 3) * 32),
                 desc_adv(q_mn, kk * 2048), kIdKM, kk > 0 ? 1u : acc0);
        }
        mma_commit_w(bar_qempty + (gq % QS));
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          mma_ss_w(tmem + L::kTDQ, desc_adv(ds_mn, kk * 2048), desc_adv(k_mn, kk * 2048), kIdMM,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit_w(bar_dqfull);
        mma_commit_w(bar_dsfree);
        if (last) {
          mma_commit_w(bar_accfull);
          mma_commit_w(bar_kvempty + (cur.t % KVS));
        }
        if (nx.valid) {
          if (!hoist && !(kv_ready(nx) && issue_s(nx))) { ok = false; break; }
          // d = 128: dQ occupies the dP^T columns until the drain warps have it
          if (D == 128) {
            if (!mbar_wait_spin_w(bar_dqfree, gq & 1, wd)) { ok = false; break; }
            tc_fence_after();
          }
          if (!kEarlyDP && !issue_dp(nx)) { ok = false; break; }
        }
        cur = nx;
      }
      mma_commit_w(bar_final);
      mbar_wait_drain(bar_final, 0, wait_limit);
    }
    __syncwarp();
  } else if (warp >= 10) {
    // ------------------------------------------------------------ dQ drain, dK/dV out (warps 10-13)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // TMEM lane: query row of dQ, key row of dK / dV
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint8_t* stage = smem + L::kDQ;
    const uint32_t st_base = smem_u32(stage);
    // d = 128: every drain warp issues its own reduce-adds from its own ring
    uint8_t* ring = stage + quarter * (L::kDQRing * L::kDQBox);
    const uint32_t ring_base = smem_u32(ring);
    const bool issuer = lane == 0 && (D == 128 || quarter == 0);
    constexpr int kRounds = (D / 32) / L::kDQChunks;
    int gq = 0, t = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const Unit un = unit(r);
      if (un.k < 0) break;
      const BwdItem x = make_bwd_item<CAUSAL, MODE>(grid, un, kSort ? item_order(bars) : nullptr);
      const int key = x.j * kBlock + row;
      const long long out_off = row_offset(grid.st, grid.H, x.bh, key);
      if (x.n_iter == 0) {  // no valid key in this tile: zero gradients
        if (key < N) {
          uint4* a = reinterpret_cast<uint4*>(dk + out_off);
          uint4* b = reinterpret_cast<uint4*>(dv + out_off);
#pragma unroll
          for (int u = 0; u < D / 8; ++u) {
            a[u] = make_uint4(0u, 0u, 0u, 0u);
            b[u] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
      // block mask: the kept Q tiles one after the other (inext: the next one)
      int inext = MODE == kModeSparse ? next_kept(x.ts.mask, x.ts.stride, x.ts.begin, x.ts.end) : 0;
      for (int it = 0; it < x.n_iter; ++it, ++gq) {
        int i = x.ts.begin + it;
        if constexpr (MODE == kModeSparse) {
          i = inext;
          inext = next_kept(x.ts.mask, x.ts.stride, i + 1, x.ts.end);
        }
        if (!mbar_wait_warp(bar_dqfull, gq & 1, wd)) { ok = false; break; }
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
        if constexpr (D == 128) {
          // Each warp reduces its own 32 rows, in boxes of 16 columns staged
          // through a ring of kDQRing buffers of its own: a box is written
          // while the reduce-adds of the previous ones still read theirs, and
          // no barrier across warps is needed. Rows are 64 bytes with the
          // 64-byte swizzle (16-byte chunk u of row r at u ^ ((r >> 1) & 3)),
          // so each 8-lane phase of a 16-byte store covers all 32 banks.
          const uint32_t sw = (lane >> 1) & 3;
#pragma unroll
          for (int b = 0; b < D / 16; ++b) {
            // Slots 0,1,2,0,1,2,0,1 in every tile. Before box b the reduce-add
            // that last read its slot is done: box b-3 of this tile (two
            // later groups may still read), or box 6 / 7 of the previous
            // tile for boxes 0 / 1 (one later group may), or box 5 of the
            // previous tile for box 2 (four later groups may).
            const int slot = b % L::kDQRing;
            if (lane == 0) {
              if (b < 2)
                bulk_wait_read<1>();
              else
                bulk_wait_read<2>();
            }
            __syncwarp();
            const uint32_t* src = &v[b >> 1][(b & 1) * 16];
            const uint32_t dst = ring_base + slot * L::kDQBox + lane * 64;
#pragma unroll
            for (int u = 0; u < 4; ++u)
              st_shared_v4(dst + ((u ^ sw) << 4), __float_as_uint(__uint_as_float(src[4 * u]) * scale),
                           __float_as_uint(__uint_as_float(src[4 * u + 1]) * scale),
                           __float_as_uint(__uint_as_float(src[4 * u + 2]) * scale),
                           __float_as_uint(__uint_as_float(src[4 * u + 3]) * scale));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_3d(&tm_dqacc, ring + slot * L::kDQBox, b * 16, i * kBlock + quarter * 32, x.bh);
              bulk_commit();
            }
          }
          continue;
        }
#pragma unroll
        for (int round = 0; round < kRounds; ++round) {
#pragma unroll
          for (int cc = 0; cc < L::kDQChunks; ++cc) {
            const int c = round * L::kDQChunks + cc;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint32_t addr = st_base + cc * kChunk + row * 128 + (((u ^ (row & 7))) << 4);
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
                                i * kBlock, x.bh);
            bulk_commit();
            bulk_wait_read0();
          }
          named_bar_sync(3, 128);
        }
      }
      if (!ok) break;
      // dV (x1, or x 1 / (1 - p') with dropout) and dK (x scale) of the item,
      // 64 columns at a time: each accumulator is released as soon as it has
      // been read out of TMEM. At d = 64 the bf16 chunk is staged in the dQ
      // staging buffer (128-byte swizzle, free again after the last dQ round)
      // and one TMA store writes it -- whole 128-byte rows in full sectors,
      // rows past N clipped. Parts of split items write fp32 to their slot.
      if (!mbar_wait_warp(bar_accfull, t & 1, wd)) break;
      tc_fence_after();
      constexpr int kHalf = D / 64, kOut = 2 * kHalf;  // chunks of dV, then of dK
#pragma unroll
      for (int oc = 0; oc < kOut; ++oc) {
        const int which = oc / kHalf, h = oc % kHalf;
        const uint32_t col = (which == 0 ? L::kTDV : L::kTDK) + h * 64;
        const float mul = which == 0 ? (DROP ? dp.rescale : 1.f) : scale;
        uint32_t a[2][32];
        tmem_ld32(lane_base + col, a[0]);
        tmem_ld32(lane_base + col + 32, a[1]);
        tmem_wait_ld();
        reg_fence(a[0]);
        reg_fence(a[1]);
        if (h == kHalf - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(which == 0 ? bar_dvempty : bar_dkempty);
        }
        if (MODE == kModeSplit && x.slot >= 0) {
          // Part of a split item: fp32 into its workspace slot, column-group
          // major ([slot][dV, dK][D / 4][128 rows][4 floats]), so that the
          // 32 rows of a warp write 512 contiguous bytes per store.
          float4* part = reinterpret_cast<float4*>(grid.dkv_part) +
                         (static_cast<size_t>(x.slot) * 2 + which) * (D / 4) * kBlock + row;
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const uint32_t* s = &a[u >> 3][(u & 7) * 4];
            part[(h * 16 + u) * kBlock] =
                make_float4(__uint_as_float(s[0]) * mul, __uint_as_float(s[1]) * mul,
                            __uint_as_float(s[2]) * mul, __uint_as_float(s[3]) * mul);
          }
          continue;
        }
        if constexpr (D == 128) {
          // d = 128: two boxes of 32 rows x 32 columns (bf16, 64-byte rows,
          // 64-byte swizzle) per 64-column half, through the warp's dQ ring
          // with the same slot order as the dQ boxes (8 boxes an item: the
          // slots of the next tile's first boxes stay where its waits expect
          // them), each written with one TMA store.
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) {
            const int e = oc * 2 + bb;  // 0..7
            const int slot = e % L::kDQRing;
            if (lane == 0) {
              if (e < 2)
                bulk_wait_read<1>();
              else
                bulk_wait_read<2>();
            }
            __syncwarp();
            const uint32_t dst = ring_base + slot * L::kDQBox + lane * 64;
            const uint32_t sw = (lane >> 1) & 3;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t* s = &a[bb][u * 8];
              st_shared_v4(dst + ((u ^ sw) << 4),
                           pack_bf16(__uint_as_float(s[0]) * mul, __uint_as_float(s[1]) * mul),
                           pack_bf16(__uint_as_float(s[2]) * mul, __uint_as_float(s[3]) * mul),
                           pack_bf16(__uint_as_float(s[4]) * mul, __uint_as_float(s[5]) * mul),
                           pack_bf16(__uint_as_float(s[6]) * mul, __uint_as_float(s[7]) * mul));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_rows(which == 0 ? &tm_dv : &tm_dk, ring + slot * L::kDQBox, h * 64 + bb * 32,
                             x.j * kBlock + quarter * 32, x.bh, grid.H, grid.st);
              bulk_commit();
            }
          }
          continue;
        }
        const int cc = oc % L::kDQChunks;  // staging chunk of this output chunk
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t* s = &a[u >> 2][(u & 3) * 8];
          st_shared_v4(st_base + cc * kChunk + row * 128 + ((u ^ (row & 7)) << 4),
                       pack_bf16(__uint_as_float(s[0]) * mul, __uint_as_float(s[1]) * mul),
                       pack_bf16(__uint_as_float(s[2]) * mul, __uint_as_float(s[3]) * mul),
                       pack_bf16(__uint_as_float(s[4]) * mul, __uint_as_float(s[5]) * mul),
                       pack_bf16(__uint_as_float(s[6]) * mul, __uint_as_float(s[7]) * mul));
        }
        if (cc == L::kDQChunks - 1 || oc == kOut - 1) {  // staging full, or the last chunk
          fence_proxy_async_smem();
          named_bar_sync(3, 128);
          if (issuer) {
#pragma unroll
            for (int c2 = 0; c2 <= cc; ++c2) {
              const int o2 = oc - cc + c2;
              tma_store_rows(o2 < kHalf ? &tm_dv : &tm_dk, stage + c2 * kChunk, (o2 % kHalf) * 64,
                             x.j * kBlock, x.bh, grid.H, grid.st);
            }
            bulk_commit();
            bulk_wait_read0();
          }
          named_bar_sync(3, 128);
        }
      }
      ++t;
    }
    if (issuer) bulk_wait0();  // every dQ reduction and dK / dV store has completed
  } else {
    // ------------------------------------------------------------ P / dS (warps 0-7)
    const int wg = warp >> 2;             // query columns [64 wg, 64 wg + 64)
    const int quarter = warp & 3;
    const int kr = quarter * 32 + lane;   // key row within the tile == TMEM lane
    const int qc0 = wg * 64;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t ds_base = smem_u32(smem + L::kDSb) + wg * kChunk;
    int gq = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const Unit un = unit(r);
      if (un.k < 0) break;
      const BwdItem x = make_bwd_item<CAUSAL, MODE>(grid, un, kSort ? item_order(bars) : nullptr);
      const bool key_live = x.j * kBlock + kr < x.kv_bound;
      // block mask: the kept Q tiles one after the other (inext: the next one)
      int inext = MODE == kModeSparse ? next_kept(x.ts.mask, x.ts.stride, x.ts.begin, x.ts.end) : 0;
      for (int it = 0; it < x.n_iter; ++it, ++gq) {
        int i = x.ts.begin + it;  // the Q tile (causal diagonal, dropout draws)
        if constexpr (MODE == kModeSparse) {
          i = inext;
          inext = next_kept(x.ts.mask, x.ts.stride, i + 1, x.ts.end);
        }
        const int s = gq % QS;
        const float* st_lse = reinterpret_cast<const float*>(smem + L::kStat + s * 1024) + qc0;
        const float* st_delta = st_lse + 128;
        // Keep decisions of key kr against query columns qc0 + 32 h + e in
        // kb[h] (keep_bits32 layout). They do not depend on S, so they are
        // drawn before S^T is awaited, filling the wait for the MMA.
        uint32_t kb[2] = {~0u, ~0u};
        if constexpr (DROP) {
          // Lane (half h = lane / 16, p = lane % 16) draws the Philox blocks of
          // queries qc0 + 16 r + p (r = 0..3) for its half-warp's 16-key group;
          // a byte transpose across the half-warp leaves each lane the bytes of
          // its own key kr: byte b of kw[r][w] is query qc0 + 16 r + 4 w + b.
          const uint32_t c4 = 0x80808080u - (dp.thresh4 & 0x7f7f7f7fu);
          const uint32_t grp = static_cast<uint32_t>(x.j * kBlock + quarter * 32 + (lane & 16)) >> 4;
          const uint32_t qrow = static_cast<uint32_t>(i * kBlock + qc0 + (lane & 15));
          uint32_t kw[4][4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const uint4 v4 = philox4x32_10(grp, qrow + 16 * r, x.bh, dp.offset, dp.k0, dp.k1);
            kw[r][0] = v4.x;
            kw[r][1] = v4.y;
            kw[r][2] = v4.z;
            kw[r][3] = v4.w;
            transpose16_bytes(kw[r], lane);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h)
            kb[h] = keep_bits32(make_uint4(kw[2 * h][0], kw[2 * h][1], kw[2 * h][2], kw[2 * h][3]),
                                make_uint4(kw[2 * h + 1][0], kw[2 * h + 1][1], kw[2 * h + 1][2],
                                           kw[2 * h + 1][3]),
                                dp.thresh4, c4);
          asm volatile("" : "+r"(kb[0]), "+r"(kb[1]));
        }
        if (!mbar_wait_warp(bar_qfull + s, (gq / QS) & 1, wd)) { ok = false; break; }
        if (!mbar_wait_warp(bar_sfull, gq & 1, wd)) { ok = false; break; }
        tc_fence_after();
        uint32_t rr[2][32];
        tmem_ld32(lane_base + L::kTS + qc0, rr[0]);
        tmem_ld32(lane_base + L::kTS + qc0 + 32, rr[1]);
        tmem_wait_ld();
        reg_fence(rr[0]);
        reg_fence(rr[1]);
        // P is kept only as bf16 pairs (the form the dV MMA consumes); dS below
        // unpacks it, which halves the registers a compute thread holds.
        const bool diag = CAUSAL && i == x.j;
        uint32_t pk[32];
        const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(st_lse + c);  // -LSE2
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[c >> 5][(c + 0) & 31]),
                                   __uint_as_float(rr[c >> 5][(c + 1) & 31])),
                           sc2, f2_pack(l4.x, l4.y)),
                    x0, x1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[c >> 5][(c + 2) & 31]),
                                   __uint_as_float(rr[c >> 5][(c + 3) & 31])),
                           sc2, f2_pack(l4.z, l4.w)),
                    x2, x3);
          const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
          pk[c / 2] = key_live ? pack_bf16(p0, p1) : 0u;
          pk[c / 2 + 1] = key_live ? pack_bf16(p2, p3) : 0u;
        }
        if (diag) {
          // Causal diagonal tile: P = 0 where query i*128 + qc0 + c < key
          // j*128 + kr. Applied to the packed pairs (column c in the low half
          // of pk[c / 2] for even c) after the loop, which keeps the masking
          // out of the loop's registers.
          const int lim = kr - qc0;  // columns c < lim are masked
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            uint32_t m = 0xffffffffu;
            if (c < lim) m &= 0xffff0000u;
            if (c + 1 < lim) m &= 0x0000ffffu;
            pk[c / 2] &= m;
          }
        }
        // P^T over the first 32 of this warpgroup's 64 S^T columns (already read)
        if constexpr (DROP) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pd[16];  // dropped P^T pairs (query columns 32 h + 2 c, + 1)
#pragma unroll
            for (int c = 0; c < 16; ++c) pd[c] = pk[16 * h + c] & pair_mask_bits(kb[h], c);
            tmem_st16(lane_base + L::kTS + qc0 + 16 * h, pd);
          }
        } else {
          tmem_st32(lane_base + L::kTS + qc0, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pready);

        if (!mbar_wait_warp(bar_dpfull, gq & 1, wd)) { ok = false; break; }
        if (gq >= 1 && !mbar_wait_warp(bar_dsfree, (gq - 1) & 1, wd)) { ok = false; break; }
        tc_fence_after();
        tmem_ld32(lane_base + L::kTDP + qc0, rr[0]);
        tmem_ld32(lane_base + L::kTDP + qc0 + 32, rr[1]);
        tmem_wait_ld();
        reg_fence(rr[0]);
        reg_fence(rr[1]);
        if constexpr (kEarlyDP) {  // dP^T may be overwritten by the next tile's now
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dpfree);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int q0 = u * 8;
          const float4 da = *reinterpret_cast<const float4*>(st_delta + q0);
          const float4 db = *reinterpret_cast<const float4*>(st_delta + q0 + 4);
          const float dd[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
          float gv[8];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {  // pairs of columns (f32x2)
            const uint32_t w = pk[(q0 + e) >> 1];
            float dpe[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              dpe[h] = __uint_as_float(rr[(q0 + e + h) >> 5][(q0 + e + h) & 31]);
              if constexpr (DROP)
                dpe[h] = keep_bit(kb[(q0 + e + h) >> 5], (q0 + e + h) & 31) ? dpe[h] * dp.rescale : 0.f;
            }
            f2_unpack(f2_mul(f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)),
                             f2_sub(f2_pack(dpe[0], dpe[1]), f2_pack(dd[e], dd[e + 1]))),
                      gv[e], gv[e + 1]);
          }
          const uint32_t addr = ds_base + kr * 128 + (((u ^ (kr & 7))) << 4);
          st_shared_v4(addr, pack_bf16(gv[0], gv[1]), pack_bf16(gv[2], gv[3]),
                       pack_bf16(gv[4], gv[5]), pack_bf16(gv[6], gv[7]));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_dsready);
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

// Sums the parts of the backward items cut by a split plan: block (i, c)
// handles columns [32 c, 32 c + 32) of cut key tile i of the merge table, one
// thread per (dV or dK, key row), and writes dK = sum of the parts' dK
// (already scaled) and dV = sum of their dV, bf16. Every part covers a
// different run of Q tiles, so the sums are the whole accumulations
// dK_j = scale sum_i dS_ij^T Q_i and dV_j = sum_i P_ij^T dO_i.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(256) bwd_merge_kernel(BwdGrid g, const __grid_constant__ MergeTable m,
                                                        __nv_bfloat16* __restrict__ dk,
                                                        __nv_bfloat16* __restrict__ dv) {
  grid_dep_wait();  // the split kernel's parts are complete
  grid_dep_launch();
  const int i = blockIdx.x, c0 = blockIdx.y * 32;
  const int t = m.item[i], q0 = m.first[i], q1 = m.first[i + 1];
  int bh, j;
  bwd_item_coords(g.nt, g.BH, CAUSAL, t, bh, j);
  const int which = threadIdx.x >> 7, rr = threadIdx.x & 127;  // which: 0 dV, 1 dK
  float acc[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) acc[c] = 0.f;
  for (int q = q0; q < q1; ++q) {
    const float4* src = reinterpret_cast<const float4*>(g.dkv_part) +
                        ((static_cast<size_t>(m.slot[q]) * 2 + which) * (D / 4) + c0 / 4) * kBlock + rr;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 a = src[c * kBlock];
      acc[4 * c] += a.x;
      acc[4 * c + 1] += a.y;
      acc[4 * c + 2] += a.z;
      acc[4 * c + 3] += a.w;
    }
  }
  const int key = j * kBlock + rr;
  if (key >= g.N) return;
  uint4* dst = reinterpret_cast<uint4*>((which ? dk : dv) + row_offset(g.st, g.H, bh, key) + c0);
#pragma unroll
  for (int c = 0; c < 4; ++c)
    dst[c] = make_uint4(pack_bf16(acc[8 * c], acc[8 * c + 1]), pack_bf16(acc[8 * c + 2], acc[8 * c + 3]),
                        pack_bf16(acc[8 * c + 4], acc[8 * c + 5]), pack_bf16(acc[8 * c + 6], acc[8 * c + 7]));
}

// Launches bwd_main_kernel<D, CAUSAL, MODE, DROP> on `grid` CTAs.
template <int D, bool CAUSAL, int MODE, bool DROP>
cudaError_t launch_bwd_main_kernel(const BwdLaunch& a, const BwdGrid& g, int grid,
                                   cudaStream_t stream) {
  using L = BwdLayout<D>;
  auto kern = bwd_main_kernel<D, CAUSAL, MODE, DROP>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = set_smem_once(smem_set, reinterpret_cast<const void*>(kern), L::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), L::kSmem, stream, a.tm_q, a.tm_k, a.tm_v,
                    a.tm_do, a.tm_dqacc, a.tm_dk, a.tm_dv, a.dk, a.dv, a.lse2, a.delta, g,
                    g.nt * kBlock, a.scale,
                    a.drop, a.status, a.wait_limit);
}

// The split kernel over the tail on `grid` (= plan.tail_ctas) CTAs, then the
// merge kernel over the cut items of `m`.
template <int D, bool CAUSAL, bool DROP>
cudaError_t launch_bwd_tail(const BwdLaunch& a, const BwdGrid& g, int grid, const MergeTable& m,
                            cudaStream_t stream) {
  cudaError_t e = launch_bwd_main_kernel<D, CAUSAL, kModeSplit, DROP>(a, g, grid, stream);
  if (e != cudaSuccess || m.n == 0) return e;
  return launch_pdl(bwd_merge_kernel<D, CAUSAL>, dim3(m.n, D / 32), dim3(256), 0, stream, g, m,
                    static_cast<__nv_bfloat16*>(a.dk), static_cast<__nv_bfloat16*>(a.dv));
}

// The (d, causal) variants of one mode and dropout setting.
template <int MODE, bool DROP>
cudaError_t launch_bwd_main_variant(const BwdLaunch& a, const BwdGrid& g, int grid,
                                    cudaStream_t stream) {
  const bool causal = a.causal != 0;
  if (a.d == 64)
    return causal ? launch_bwd_main_kernel<64, true, MODE, DROP>(a, g, grid, stream)
                  : launch_bwd_main_kernel<64, false, MODE, DROP>(a, g, grid, stream);
  return causal ? launch_bwd_main_kernel<128, true, MODE, DROP>(a, g, grid, stream)
                : launch_bwd_main_kernel<128, false, MODE, DROP>(a, g, grid, stream);
}

}  // namespace
}  // namespace fa
