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
// The kernel is persistent: one CTA per SM walks a list of work items (Q
// tiles A = 2p and B = 2p + 1 of one (batch, head)); barrier phases continue
// across items, so the next item's Q and K/V loads overlap the current one's
// last steps and epilogue. 10 warps:
//   warp 0      MMA issuer (below)
//   warp 1      TMA producer: Q_A, Q_B per item; K_j, V_j through separate rings
//   warps 2-5   softmax of tile A: each thread owns one query row, the TMEM
//               lane of its warp's quarter (warp % 4)
//   warps 6-9   softmax of tile B
//   The MMA issuer runs, at d = 128, in the order
//                 S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
//               so that the tensor core computes one tile's MMAs while the
//               other tile's softmax runs.
// TMEM columns: S_A [0,128), S_B [128,256) (fp32); O_A [256, 256+d),
// O_B [256+d, 256+2d) (fp32 accumulators). The softmax writes P_t in bf16
// pairs to TMEM and the PV MMA takes it from there as its A operand, so P never
// touches shared memory. At d = 64, P_A and P_B have columns of their own
// ([384,448), [448,512)): S_t(j+1) is then issued as soon as the softmax has
// loaded S_t(j) into registers and is ready when P_t(j) is, and the issue
// order becomes S_A(j+1) S_B(j+1) PV_A(j) PV_B(j). At d = 128 TMEM is full and
// P_t goes over the first 64 columns of S_t. Each item ends with O / l stored
// straight from TMEM to global memory, one row per thread.
//
// Rescaling is lazy: a row's reference maximum m only moves when the new
// tile's maximum exceeds it by more than 8 (log2 units), so P <= 2^8 and O is
// rescaled in TMEM only on those rare tiles; the final O / l is exact because
// O and l always share the same m.
//
// An item pairs adjacent Q tiles, so both are active on (almost) every K/V
// step and their softmax phases alternate on the tensor core; causal items
// are handed out heaviest first, in a snake order across the CTAs.
#pragma once

#include <cuda_bf16.h>

#include <type_traits>

#include "fa_internal.h"
#include "fa_philox.cuh"
#include "fa_ptx.cuh"
#include "fa_sched.cuh"

namespace fa {
namespace {

// Warp roles: warp 0 issues MMAs (at d = 64 for Q tile slot A only, warp 2
// for slot B), warp 1 issues TMA copies, then four softmax warps per slot.
constexpr int kMmaWarp = 0, kLoadWarp = 1;
template <int D>
struct FwdWarps {
  static constexpr int kMmaB = (D == 64) ? 2 : -1;  // second MMA issuer (d = 64)
  static constexpr int kSoft0 = (D == 64) ? 3 : 2;  // first softmax warp
  static constexpr int kThreads = (kSoft0 + 8) * 32;
};
constexpr int kChunk = 128 * 128;  // bytes of one 128-row x 128-byte swizzled chunk (64 bf16 cols)
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 256

// kHP: items pair the same Q tile of two heads, each slot with a K/V ring
// of its own (block-sparse at d = 64, where the two heads visit the same K/V
// tiles); otherwise items pair adjacent Q tiles of one head, which share one
// K/V ring.
template <int D, bool kHP = false>
struct FwdLayout {
  // d = 64 leaves TMEM room for P in columns of its own: the next S of a tile
  // can then be computed while the softmax of the current one still runs.
  static constexpr bool kSepP = (D == 64);
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kChunks * kChunk;  // one 128 x D bf16 tile
  static constexpr int kRings = kHP ? 2 : 1;      // K/V rings (one per Q slot with kHP)
  static constexpr int kKS = kHP ? 2 : 3;         // K ring slots
  static constexpr int kVS = kHP ? 2 : ((D == 128) ? 2 : 3);  // V ring slots
  static constexpr int kQS = (D == 128) ? 1 : 2;  // Q stages per tile slot
  static constexpr int kQ = 0;                    // Q of slot t, stage s: kQ + (t kQS + s) kTile
  static constexpr int kK = kQ + 2 * kQS * kTile; // K of ring x, slot s: kK + (x kKS + s) kTile
  static constexpr int kV = kK + kRings * kKS * kTile;
  static constexpr int kBar = kV + kRings * kVS * kTile;
  // barriers, TMEM address, abort flag, tail range; then the producer's
  // 128-byte tile list and the cost-sorted group table
  static constexpr int kEnd = kBar + 512 + 128 + 2 * kOrderMax;
  // d = 64 (dense): per softmax warp a 32-row x 64-column bf16 box of O
  // (128-byte swizzle) for the epilogue's TMA store. The head-paired
  // block-sparse variant keeps row stores (measured slightly faster there).
  static constexpr bool kOStore = (D == 64 && !kHP);
  static constexpr int kOst = (kEnd + 1023) & ~1023, kOBox = 32 * 128;  // swizzle atoms: 1024-byte aligned
  static constexpr int kOBytes = kOStore ? 8 * kOBox : 0;
  static constexpr int kSmem = kOst + kOBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kSmem <= 227 * 1024, "shared memory of one CTA");
  static constexpr uint32_t kTO = 256;       // O_A; O_B at kTO + D
  // P_t (bf16 pairs, 64 columns): its own columns, or over the first 64 of S_t
  static constexpr uint32_t kTP = kSepP ? 256 + 2 * D : 0;
  __host__ __device__ static constexpr uint32_t p_col(int t) { return kSepP ? kTP + t * 64 : t * 128; }
  // barrier offsets (in 8-byte words from kBar)
  static constexpr int oKF = 8, oKE = kHP ? 12 : 11, oVF = kHP ? 16 : 14, oVE = kHP ? 20 : 17;
  static constexpr int oS = kHP ? 24 : 20;  // sfull [2], then pfull, odone, sfree, final [2 each]
  static constexpr int oTmem = oS + 10, oAbort = oS + 11, oTail = oS + 12;
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


// One work unit: Q tiles 2p and 2p+1 (qtB = -1 if absent) of one (batch,
// head), restricted to the K/V steps [sb, se) of the unit. Without a block
// mask or key padding, step j is K/V tile j, so a unit of a split item covers
// K/V tiles [sb, se); `slot` >= 0 names the workspace slot its partial result
// goes to (-1: the whole item, O and LSE written directly).
struct FwdItem {
  int k, bh, bhB, qtA, qtB, kv_bound, slot;  // bh, bhB: problems of Q tiles A and B
  TileSet tsA, tsB;
};

template <bool CAUSAL>
__host__ __device__ __forceinline__ int fwd_steps(const FwdGrid& g, int k) {
  return fwd_item_steps(g.nqt, g.npairs, g.n_items / g.npairs, CAUSAL, k);
}

// `order`: the cost-sorted group table (fa_sched.cuh) or null (index order).
// kAlt (causal, whole items): Q tile 2p + 1 sees one K/V tile more than 2p,
// so the slot that takes it alternates from one round of items to the next
// ((k / gridDim.x) odd: A = 2p + 1, B = 2p) -- otherwise slot B would carry
// one tile more per item and finish a CTA's items several tiles after A.
template <bool CAUSAL, bool kHP = false, bool kAlt = false>
__device__ FwdItem make_item(const FwdGrid& g, const Unit& u, const uint16_t* order) {
  FwdItem it;
  it.k = u.k;
  it.slot = u.slot;
  if constexpr (kHP) {
    // Q tile r of heads 2 hp and 2 hp + 1 of batch b: one mask row for both.
    // Sorted: the groups are mask rows, their members (batch, head pair).
    const int HP = (g.H + 1) / 2;
    int bhp, r;
    if (order != nullptr) {
      const int inner = g.n_items / g.nqt, grp = u.k / inner;
      r = order[grp];
      bhp = u.k - grp * inner;
    } else {
      bhp = u.k / g.nqt;
      r = u.k - bhp * g.nqt;
    }
    const int b = bhp / HP, hp = bhp - b * HP;
    it.bh = b * g.H + 2 * hp;
    it.bhB = 2 * hp + 1 < g.H ? it.bh + 1 : -1;
    it.qtA = r;
    it.qtB = it.bhB >= 0 ? r : -1;
  } else {
    int p;
    if (order == nullptr) {
      fwd_item_coords(g.npairs, g.n_items / g.npairs, CAUSAL, u.k, it.bh, p);
    } else {  // groups: pairs p; members: (batch, head)
      const int BH = g.n_items / g.npairs, grp = u.k / BH;
      p = order[grp];
      it.bh = u.k - grp * BH;
    }
    it.bhB = it.bh;
    it.qtA = 2 * p;
    it.qtB = 2 * p + 1 < g.nqt ? 2 * p + 1 : -1;
    if (kAlt && it.qtB >= 0 && ((u.k / static_cast<int>(gridDim.x)) & 1)) {
      it.qtA = 2 * p + 1;
      it.qtB = 2 * p;
    }
  }
  it.kv_bound = g.N;
  if (g.kv_len != nullptr) it.kv_bound = min(g.N, max(0, g.kv_len[it.bh / g.H]));
  const int kv_tiles = (it.kv_bound + kBlock - 1) / kBlock;
  const int endA = CAUSAL ? min(kv_tiles, it.qtA + 1) : kv_tiles;
  const int endB = it.qtB < 0 ? 0 : (CAUSAL ? min(kv_tiles, it.qtB + 1) : kv_tiles);
  const uint8_t* mA = g.block_mask != nullptr ? g.block_mask + static_cast<size_t>(it.qtA) * g.nqt : nullptr;
  const uint8_t* mB = (g.block_mask != nullptr && it.qtB >= 0)
                          ? g.block_mask + static_cast<size_t>(it.qtB) * g.nqt
                          : nullptr;
  it.tsA = TileSet{u.sb, min(endA, u.se), mA, 1};
  it.tsB = TileSet{u.sb, min(endB, u.se), mB, 1};
  return it;
}

// The next K/V tile >= j that Q tile A or B of an item visits (kNoTile if
// none), and which of the two visit it. Warp-collective.
__device__ __forceinline__ int next_pair_tile(TileWalk<>& wa, TileWalk<>& wb, int j, bool& hA, bool& hB) {
  const int a = wa.seek(j), b = wb.seek(j);
  const int m = min(a, b);
  hA = a == m;
  hB = b == m;
  return m;
}

// The cost-sorted item order of a block-sparse forward pass (fa_sched.cuh),
// built by the whole CTA before any TMA load: the groups are mask rows (kHP:
// d = 64, head-paired items) or pairs of rows, a group's cost the number of
// (Q tile, K/V tile) products of one of its items. `scratch` (>= 6656 bytes)
// is a tile buffer that no copy has written yet; every thread of the CTA
// takes part. (Key padding alone is not sorted: those items differ little in
// cost -- a BERT-like pass's items took 6.6-7.2 us whatever their length --
// and the sort's start-up cost more than it evened out.)
template <bool CAUSAL, bool kHP>
__device__ __forceinline__ void fwd_sort_items(int nqt, int npairs, const int32_t* kv_len,
                                               const uint8_t* block_mask, uint8_t* scratch,
                                               uint64_t* bars) {
  const int G = kv_len == nullptr ? (kHP ? nqt : npairs) : 0;
  if (G == 0 || G > kOrderMax) return;  // uniform over the CTA
  int* cost = reinterpret_cast<int*>(scratch);
  int* hist = cost + kOrderMax;
  for (int i = threadIdx.x; i < G; i += blockDim.x) cost[i] = 0;
  __syncthreads();
  for_kept_blocks(block_mask, nqt, [&](int r, int c) {
    if (!CAUSAL || c <= r) atomicAdd(&cost[kHP ? r : r >> 1], 1);
  });
  __syncthreads();
  if ((threadIdx.x >> 5) == 0)
    sort_groups(cost, G, min(kCostMax, 2 * nqt), hist, reinterpret_cast<uint16_t*>(bars + 64) + 64);
  fence_proxy_async_smem();  // the scratch tile is next written by TMA
  if (threadIdx.x == 0) *reinterpret_cast<volatile int*>(bars + kOrderFlagWord) = 1;
  __syncthreads();
}

// DROP: inverted dropout on P (fa_philox.cuh); the row sums and LSE use the
// undropped P, the PV product the dropped one, and O is scaled by 1 / (1 - p').
// MODE (kModePlain, kModeSparse, kModeSplit): the variant compiled. Plain
// walks dense ranges of K/V tiles and whole items; sparse walks the tile
// lists of a block mask; split also runs the parts of the last wave's items
// and writes their partial results. Keeping them apart at compile time leaves
// the plain kernel's hot loops exactly as tuned.
template <int D, bool CAUSAL, bool DROP, int MODE>
__global__ void __launch_bounds__(FwdWarps<D>::kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               __nv_bfloat16* __restrict__ out,
               float* __restrict__ lse_out, FwdGrid g, float scale_log2, DropoutParams dp,
               int* status, long long wait_limit) {
  // Block-sparse at d = 64: items pair one Q tile of two heads (same mask row),
  // each Q slot with a K/V ring of its own.
  constexpr bool kHP = (MODE == kModeSparse && D == 64);
  using L = FwdLayout<D, kHP>;
  constexpr int KS = L::kKS, VS = L::kVS, QS = L::kQS;
  constexpr bool kSepP = L::kSepP;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* bar_qfull = bars + 0;          // [2][QS] per Q slot (A, B) and stage
  uint64_t* bar_qempty = bars + 4;         // [2][QS]
  uint64_t* bar_kfull = bars + L::oKF;     // [rings][KS]
  uint64_t* bar_kempty = bars + L::oKE;    // [rings][KS]
  uint64_t* bar_vfull = bars + L::oVF;     // [rings][VS]
  uint64_t* bar_vempty = bars + L::oVE;    // [rings][VS]
  uint64_t* bar_sfull = bars + L::oS;      // [2]
  uint64_t* bar_pfull = bars + L::oS + 2;  // [2]
  uint64_t* bar_odone = bars + L::oS + 4;  // [2]
  uint64_t* bar_sfree = bars + L::oS + 6;  // [2] S_t read out of TMEM (separate-P layout)
  uint64_t* bar_final = bars + L::oS + 8;  // [2] one per MMA issuer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::oTmem);
  int* abort_flag = reinterpret_cast<int*>(bars + L::oAbort);
  TailRange* tail_sh = reinterpret_cast<TailRange*>(bars + L::oTail);  // this CTA's share of a split tail
  uint8_t* walk_list = reinterpret_cast<uint8_t*>(bars + 64);     // [128] the producer's kept tiles of a window (sparse)
  // then [kOrderMax] cost-sorted groups from walk_list + 128 (item_order)
  constexpr int kMmaB = FwdWarps<D>::kMmaB, kSoft0 = FwdWarps<D>::kSoft0;
  // arrivals that release a K or V ring slot: both issuers at d = 64 when the
  // slots share one ring, else the one issuer that uses it
  constexpr int kIssuers = (kSepP && !kHP) ? 2 : 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  check_init(status);

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      for (int q = 0; q < QS; ++q) {
        mbar_init(bar_qfull + t * QS + q, 1);
        mbar_init(bar_qempty + t * QS + q, 1);
      }
      mbar_init(bar_sfull + t, 1);
      mbar_init(bar_pfull + t, 4);
      mbar_init(bar_odone + t, 1);
      mbar_init(bar_sfree + t, 4);
    }
    for (int s = 0; s < L::kRings * KS; ++s) {
      mbar_init(bar_kfull + s, 1);
      mbar_init(bar_kempty + s, kIssuers);
    }
    for (int s = 0; s < L::kRings * VS; ++s) {
      mbar_init(bar_vfull + s, 1);
      mbar_init(bar_vempty + s, kIssuers);
    }
    mbar_init(bar_final, 1);
    mbar_init(bar_final + 1, 1);
    *abort_flag = 0;
    *reinterpret_cast<int*>(bars + kOrderFlagWord) = 0;  // index order unless sorted below
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  auto steps = [&](int k) { return fwd_steps<CAUSAL>(g, k); };
  if constexpr (MODE == kModeSplit) {
    if (warp == kLoadWarp) {
      const TailRange tr = tail_range(g.plan, blockIdx.x, steps);
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
  // Cost-sorted item order with a block mask (fwd_sort_items).
  constexpr bool kSort = MODE == kModeSparse;
  constexpr bool kAltSlots = CAUSAL && MODE == kModePlain;  // see make_item
  if constexpr (kSort) fwd_sort_items<CAUSAL, kHP>(g.nqt, g.npairs, g.kv_len, g.block_mask, smem + L::kQ, bars);
  // The r-th unit of this CTA, or a unit with k < 0: the split kernel runs
  // the CTA's run of the tail; the others whole items [0, plan.whole) in a
  // snake over the item list.
  auto unit = [&](int r) -> Unit {
    if constexpr (MODE == kModeSplit) {
      return tail_unit(tail_sh, r, blockIdx.x, steps);
    } else {
      Unit u{-1, 0, 1 << 30, -1};
      const int G = gridDim.x, c = blockIdx.x;
      if (r * G >= g.plan.whole) return u;
      const int k = r * G + ((r & 1) ? G - 1 - c : c);
      if (k < g.plan.whole) u.k = k;  // only the last round can run past the end
      return u;
    }
  };
  uint8_t* list = walk_list;  // the producer's (the only warp that lists tiles)

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    // Lane 0 waits for free ring slots and issues the copies (with a block
    // mask the whole warp first lists each window's tiles).
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    int nqA = 0, nqB = 0;  // Q loads issued per slot
    int k_issued = 0, v_issued = 0;
    int u = 0;           // position in the K/V rings, continued across items
    int uB = 0, kB_issued = 0, vB_issued = 0;  // ring B (head-paired items)
    bool ok = true;
    // Q loads of a unit's two tiles (lane 0); false on an abort.
    auto load_q = [&](const FwdItem& it, int lastA, int lastB) -> bool {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if ((t ? lastB : lastA) < 0) continue;
        int& nq = t ? nqB : nqA;
        const int qb = t * QS + nq % QS;
        if (nq >= QS && !mbar_wait(bar_qempty + qb, ((nq / QS) - 1) & 1, wd)) return false;
        mbar_expect_tx(bar_qfull + qb, L::kTile);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_rows(smem + L::kQ + qb * L::kTile + c * kChunk, &tm_q, bar_qfull + qb, c * 64,
                        (t ? it.qtB : it.qtA) * kBlock, kHP ? (t ? it.bhB : it.bh) : it.bh, g.H,
                        g.st);
        ++nq;
      }
      return true;
    };
    // K_j and V_j of problem bh into the next position uu of K/V ring `ring`
    // (lane 0); false on an abort.
    auto load_kv_r = [&](int ring, int bh, int j, int& uu, int& ki, int& vi) -> bool {
      const int ks = ring * KS + uu % KS, vs = ring * VS + uu % VS;
      if (uu >= KS && !mbar_wait(bar_kempty + ks, ((uu / KS) - 1) & 1, wd)) return false;
      mbar_expect_tx(bar_kfull + ks, L::kTile);
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_rows(smem + L::kK + ks * L::kTile + c * kChunk, &tm_k, bar_kfull + ks, c * 64,
                      j * kBlock, bh, g.H, g.st);
      ki = uu + 1;
      if (uu >= VS && !mbar_wait(bar_vempty + vs, ((uu / VS) - 1) & 1, wd)) return false;
      mbar_expect_tx(bar_vfull + vs, L::kTile);
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_rows(smem + L::kV + vs * L::kTile + c * kChunk, &tm_v, bar_vfull + vs, c * 64,
                      j * kBlock, bh, g.H, g.st);
      vi = uu + 1;
      ++uu;
      return true;
    };
    auto load_kv = [&](const FwdItem& it, int j) -> bool {
      return load_kv_r(0, it.bh, j, u, k_issued, v_issued);
    };
    if constexpr (kHP) {
      // Head-paired items: both Q tiles keep the same mask row. The whole warp
      // lists each 128-tile window's kept tiles; lane 0 loads each tile's K and
      // V of head A into ring A and of head B into ring B.
      for (int r = 0; ok; ++r) {
        const Unit un = unit(r);
        if (un.k < 0) break;
        const FwdItem it = make_item<CAUSAL, kHP, kAltSlots>(g, un, kSort ? item_order(bars) : nullptr);
        TileWalk<> wa;
        wa.init(it.tsA);
        const int lastA = wa.last(), lastB = it.bhB >= 0 ? lastA : -1;
        if (lane == 0) ok = load_q(it, lastA, lastB);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        for (int w0 = it.tsA.begin & ~127; ok && w0 < it.tsA.end; w0 += 128) {
          const int cnt = list_window(it.tsA, w0, list);
          if (lane == 0) {
            for (int idx = 0; ok && idx < cnt; ++idx) {
              const int j = w0 + list[idx];
              ok = load_kv_r(0, it.bh, j, u, k_issued, v_issued);
              if (ok && it.bhB >= 0) ok = load_kv_r(1, it.bhB, j, uB, kB_issued, vB_issued);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
      }
    } else if constexpr (MODE == kModeSparse) {
      // The whole warp lists each 128-tile window's tiles (union of the two Q
      // tiles' mask rows); lane 0 then issues their copies.
      for (int r = 0; ok; ++r) {
        const Unit un = unit(r);
        if (un.k < 0) break;
        const FwdItem it = make_item<CAUSAL, kHP, kAltSlots>(g, un, kSort ? item_order(bars) : nullptr);
        TileWalk<> wa, wb;
        wa.init(it.tsA);
        wb.init(it.tsB);
        const int lastA = wa.last(), lastB = wb.last();
        if (lane == 0) ok = load_q(it, lastA, lastB);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        const int uend = max(it.tsA.end, it.tsB.end);
        for (int w0 = it.tsA.begin & ~127; ok && w0 < uend; w0 += 128) {
          const int cnt = list_window2(it.tsA, it.tsB, w0, list);
          if (lane == 0)
            for (int idx = 0; ok && idx < cnt; ++idx) ok = load_kv(it, w0 + list[idx]);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
      }
    } else if (lane == 0) {
      // Dense ranges: K/V tiles [begin, max(end_A, end_B)) of every unit.
      for (int r = 0; ok; ++r) {
        const Unit un = unit(r);
        if (un.k < 0) break;
        const FwdItem it = make_item<CAUSAL, kHP, kAltSlots>(g, un, kSort ? item_order(bars) : nullptr);
        const int lastA = it.tsA.end > it.tsA.begin ? it.tsA.end - 1 : -1;
        const int lastB = it.tsB.end > it.tsB.begin ? it.tsB.end - 1 : -1;
        ok = load_q(it, lastA, lastB);
        const int uend = max(it.tsA.end, it.tsB.end);
        for (int j = it.tsA.begin; ok && j < uend; ++j) ok = load_kv(it, j);
      }
    }
    // Let every copy in flight land before the CTA can exit (bounded).
    if (lane == 0) {
      for (int t = 0; t < 2; ++t) {
        const int nq = t ? nqB : nqA;
        for (int q = max(0, nq - QS); q < nq; ++q)
          mbar_wait_drain(bar_qfull + t * QS + q % QS, (q / QS) & 1, wait_limit);
      }
      for (int t = max(0, k_issued - KS); t < k_issued; ++t)
        mbar_wait_drain(bar_kfull + (t % KS), (t / KS) & 1, wait_limit);
      for (int t = max(0, v_issued - VS); t < v_issued; ++t)
        mbar_wait_drain(bar_vfull + (t % VS), (t / VS) & 1, wait_limit);
      if constexpr (kHP) {
        for (int t = max(0, kB_issued - KS); t < kB_issued; ++t)
          mbar_wait_drain(bar_kfull + KS + (t % KS), (t / KS) & 1, wait_limit);
        for (int t = max(0, vB_issued - VS); t < vB_issued; ++t)
          mbar_wait_drain(bar_vfull + VS + (t % VS), (t / VS) & 1, wait_limit);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp || warp == kMmaB) {
    // ------------------------------------------------------------ MMA issuers (whole warps)
    // An issuer sits on the critical path between the softmax warpgroups. The
    // warp runs converged and an elected lane issues each tcgen05.mma /
    // commit; it polls the barriers and places a tcgen05 fence only after
    // waiting on another thread's TMEM access (P_t written by tcgen05.st; S_t
    // read by tcgen05.ld before S_t(j+1) overwrites it).
    if constexpr (kSepP) {
      // d = 64: one issuer per Q tile slot X, each walking every K/V tile of
      // its items. Both release each K and V ring slot (count 2): with an MMA
      // commit when slot X used the tile, else with a plain arrive once the
      // tile is known to be loaded, which keeps the ring's phases in order.
      const int X = (warp == kMmaWarp) ? 0 : 1;
      // With head-paired items slot X has K/V ring X and walks only its own
      // tiles; otherwise both walk the shared ring (see above).
      const int ring = kHP ? X : 0;
      uint64_t* const kfull = bar_kfull + ring * KS;
      uint64_t* const kempty = bar_kempty + ring * KS;
      uint64_t* const vfull = bar_vfull + ring * VS;
      uint64_t* const vempty = bar_vempty + ring * VS;
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);  // Q, K both K-major
      constexpr uint32_t kIdO = idesc_bf16(128, D, false, true);     // P (TMEM), V MN-major
      const uint64_t q_desc = sdesc_sw128(smem_u32(smem + L::kQ), 16, 1024);     // K-major
      const uint64_t k_desc =
          sdesc_sw128(smem_u32(smem + L::kK + ring * KS * L::kTile), 16, 1024);   // K-major
      const uint64_t v_desc =
          sdesc_sw128(smem_u32(smem + L::kV + ring * VS * L::kTile), kChunk, 1024);  // MN-major
      const uint32_t s_tm = tmem + X * 128, o_tm = tmem + L::kTO + X * D;
      const uint32_t p_tm = tmem + L::p_col(X);
      uint64_t* my_sfull = bar_sfull + X;
      uint64_t* my_sfree = bar_sfree + X;
      uint64_t* my_pfull = bar_pfull + X;
      uint64_t* my_odone = bar_odone + X;
      int npv = 0, nq = 0, ns = 0;  // P V MMAs, Q tiles, S tiles of this slot so far
      int u = 0;                    // position in the K/V rings
      int k_ready = -1, v_ready = -1;  // ring positions already seen loaded
      bool ok = true;
      auto k_wait = [&](int uu) -> bool {
        if (uu == k_ready) return true;
        if (!mbar_wait_spin_w(kfull + (uu % KS), (uu / KS) & 1, wd)) return false;
        k_ready = uu;
        return true;
      };
      auto v_wait = [&](int uu) -> bool {
        if (uu == v_ready) return true;
        if (!mbar_wait_spin_w(vfull + (uu % VS), (uu / VS) & 1, wd)) return false;
        v_ready = uu;
        return true;
      };
      for (int r = 0; ok; ++r) {
        const Unit un0 = unit(r);
        if (un0.k < 0) break;
        const FwdItem it = make_item<CAUSAL, kHP, kAltSlots>(g, un0, kSort ? item_order(bars) : nullptr);
        TileWalk<> wa, wb;  // block-mask walks (sparse)
        wa.init(it.tsA);
        wb.init(it.tsB);
        const int uend = max(it.tsA.end, it.tsB.end);
        // The next K/V tile >= j of the item and whether Q tiles A, B visit it.
        auto nxt = [&](int j, bool& hA, bool& hB) -> int {
          if constexpr (kHP) {  // only this slot's tiles, all of them its own
            hA = hB = true;
            return (X ? wb : wa).seek(j);
          } else if constexpr (MODE == kModeSparse) {
            return next_pair_tile(wa, wb, j, hA, hB);
          } else {
            hA = j < it.tsA.end;
            hB = j < it.tsB.end;
            return j < uend ? j : kNoTile;
          }
        };
        int last;  // the last K/V tile Q tile X visits (-1: none)
        if constexpr (MODE == kModeSparse) {
          last = X ? wb.last() : wa.last();
        } else {
          const TileSet& my = X ? it.tsB : it.tsA;
          last = my.end > my.begin ? my.end - 1 : -1;
        }
        bool needq = last >= 0;
        int loc = 0;  // P V MMAs of this item
        const int qb = X * QS + nq % QS;
        auto issue_s = [&](int uu, int j) -> bool {
          if (needq) {
            if (!mbar_wait_spin_w(bar_qfull + qb, (nq / QS) & 1, wd)) return false;
            needq = false;
          }
          if (!k_wait(uu)) return false;
          if (ns >= 1) {  // the softmax has read S_X(previous) out of TMEM
            if (!mbar_wait_spin_w(my_sfree, (ns - 1) & 1, wd)) return false;
            tc_fence_after();
          }
          ++ns;
          const uint64_t qd = desc_adv(q_desc, qb * L::kTile);
          const uint64_t kd = desc_adv(k_desc, (uu % KS) * L::kTile);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
            mma_ss_w(s_tm, desc_adv(qd, off), desc_adv(kd, off), kIdS, kk > 0 ? 1u : 0u);
          }
          mma_commit_w(my_sfull);
          if (j == last) {  // Q_X of this item is no longer needed
            mma_commit_w(bar_qempty + qb);
            ++nq;
          }
          return true;
        };
        auto issue_pv = [&](int uu) -> bool {
          if (!mbar_wait_spin_w(my_pfull, npv & 1, wd)) return false;
          if (!v_wait(uu)) return false;
          tc_fence_after();
          const uint64_t vd = desc_adv(v_desc, (uu % VS) * L::kTile);
          const uint32_t acc0 = loc > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < kBlock / 16; ++kk)
            mma_ts_w(o_tm, p_tm + kk * 8, desc_adv(vd, kk * 2048), kIdO, kk > 0 ? 1u : acc0);
          mma_commit_w(my_odone);
          ++npv;
          ++loc;
          return true;
        };
        auto release_k = [&](int uu, bool used) -> bool {
          if (used) {
            mma_commit_w(kempty + (uu % KS));
            return true;
          }
          if (!k_wait(uu)) return false;
          mbar_arrive_w(kempty + (uu % KS));
          return true;
        };
        auto release_v = [&](int uu, bool used) -> bool {
          if (used) {
            mma_commit_w(vempty + (uu % VS));
            return true;
          }
          if (!v_wait(uu)) return false;
          mbar_arrive_w(vempty + (uu % VS));
          return true;
        };
        bool jA, jB;
        int j = nxt(it.tsA.begin, jA, jB);
        if (j == kNoTile) continue;
        {
          const bool h = X ? jB : jA;
          if (h) ok = issue_s(u, j);
          if (ok) ok = release_k(u, h);
        }
        while (ok && j != kNoTile) {
          bool nA, nB;
          const int jn = nxt(j + 1, nA, nB);
          const int un = u + 1;
          // S_X(j+1) as soon as the softmax has read S_X(j), then P_X(j) V_j
          if (jn != kNoTile) {
            const bool h = X ? nB : nA;
            if (h) ok = issue_s(un, jn);
            if (ok) ok = release_k(un, h);
          }
          if (ok) {
            const bool h = X ? jB : jA;
            if (h) ok = issue_pv(u);
            if (ok) ok = release_v(u, h);
          }
          j = jn;
          jA = nA;
          jB = nB;
          u = un;
        }
      }
      mma_commit_w(bar_final + X);
      mbar_wait_drain(bar_final + X, 0, wait_limit);
    } else {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);  // Q, K both K-major
      constexpr uint32_t kIdO = idesc_bf16(128, D, false, true);     // P (TMEM), V MN-major
      // Descriptors built once; per MMA only a compile-time offset is added.
      const uint64_t q_desc = sdesc_sw128(smem_u32(smem + L::kQ), 16, 1024);     // K-major
      const uint64_t k_desc = sdesc_sw128(smem_u32(smem + L::kK), 16, 1024);     // K-major
      const uint64_t v_desc = sdesc_sw128(smem_u32(smem + L::kV), kChunk, 1024);  // MN-major
      // Per-slot state is kept in scalars and slots are compile-time constants
      // (generic lambdas over std::integral_constant), so nothing of this hot
      // loop lives in local memory.
      int npvA = 0, npvB = 0;  // P V MMAs issued per slot (pfull / odone phases)
      int nqA = 0, nqB = 0;    // Q tiles consumed per slot (qfull phases)
      int nsA = 0, nsB = 0;    // S tiles issued per slot (sfree phases)
      int u = 0;               // position in the K/V rings
      bool ok = true;
      using SlotA = std::integral_constant<int, 0>;
      using SlotB = std::integral_constant<int, 1>;
      for (int r = 0; ok; ++r) {
        const Unit un0 = unit(r);
        if (un0.k < 0) break;
        const FwdItem it = make_item<CAUSAL, kHP, kAltSlots>(g, un0, kSort ? item_order(bars) : nullptr);
        TileWalk<> wa, wb;  // block-mask walks (sparse)
        wa.init(it.tsA);
        wb.init(it.tsB);
        const int uend = max(it.tsA.end, it.tsB.end);
        auto nxt = [&](int j, bool& hA, bool& hB) -> int {
          if constexpr (MODE == kModeSparse) {
            return next_pair_tile(wa, wb, j, hA, hB);
          } else {
            hA = j < it.tsA.end;
            hB = j < it.tsB.end;
            return j < uend ? j : kNoTile;
          }
        };
        int lastA, lastB;
        if constexpr (MODE == kModeSparse) {
          lastA = wa.last();
          lastB = wb.last();
        } else {
          lastA = it.tsA.end > it.tsA.begin ? it.tsA.end - 1 : -1;
          lastB = it.tsB.end > it.tsB.begin ? it.tsB.end - 1 : -1;
        }
        bool needqA = lastA >= 0, needqB = lastB >= 0;
        int locA = 0, locB = 0;  // P V MMAs of this item per slot
        auto issue_s = [&](auto slot, int uu, int j) -> bool {
          constexpr int t = decltype(slot)::value;
          bool& needq = t ? needqB : needqA;
          int& nq = t ? nqB : nqA;
          int& ns = t ? nsB : nsA;
          const int qb = t * QS + nq % QS;
          if (needq) {
            if (!mbar_wait_spin_w(bar_qfull + qb, (nq / QS) & 1, wd)) return false;
            needq = false;
          }
          if (!mbar_wait_spin_w(bar_kfull + (uu % KS), (uu / KS) & 1, wd)) return false;
          if (kSepP && ns >= 1) {  // the softmax has read S_t(previous) out of TMEM
            if (!mbar_wait_spin_w(bar_sfree + t, (ns - 1) & 1, wd)) return false;
            tc_fence_after();
          }
          ++ns;
          const uint64_t qd = desc_adv(q_desc, qb * L::kTile);
          const uint64_t kd = desc_adv(k_desc, (uu % KS) * L::kTile);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
            mma_ss_w(tmem + t * 128, desc_adv(qd, off), desc_adv(kd, off), kIdS, kk > 0 ? 1u : 0u);
          }
          mma_commit_w(bar_sfull + t);
          if (j == (t ? lastB : lastA)) {  // Q_t of this item is no longer needed
            mma_commit_w(bar_qempty + qb);
            ++nq;
          }
          return true;
        };
        auto issue_pv = [&](auto slot, int uu) -> bool {
          constexpr int t = decltype(slot)::value;
          int& npv = t ? npvB : npvA;
          int& loc = t ? locB : locA;
          if (!mbar_wait_spin_w(bar_pfull + t, npv & 1, wd)) return false;
          if (!mbar_wait_spin_w(bar_vfull + (uu % VS), (uu / VS) & 1, wd)) return false;
          tc_fence_after();
          const uint64_t vd = desc_adv(v_desc, (uu % VS) * L::kTile);
          const uint32_t acc0 = loc > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < kBlock / 16; ++kk) {
            // A = P_t (bf16 pairs, from TMEM), B = V, MN-major.
            mma_ts_w(tmem + L::kTO + t * D, tmem + L::p_col(t) + kk * 8, desc_adv(vd, kk * 2048), kIdO,
                   kk > 0 ? 1u : acc0);
          }
          mma_commit_w(bar_odone + t);
          ++npv;
          ++loc;
          return true;
        };
        bool jA, jB;
        int j = nxt(it.tsA.begin, jA, jB);
        if (j == kNoTile) continue;
        if (jA) ok = issue_s(SlotA{}, u, j);
        if (ok && jB) ok = issue_s(SlotB{}, u, j);
        if (ok) mma_commit_w(bar_kempty + (u % KS));
        while (ok && j != kNoTile) {
          bool nA, nB;
          const int jn = nxt(j + 1, nA, nB);
          const bool more = jn != kNoTile;
          const int un = u + 1;
          if constexpr (kSepP) {
            // S_t(j+1) as soon as the softmax has read S_t(j), so that it is
            // ready when P_t(j) is; then P_A(j) V_j and P_B(j) V_j.
            if (more) {
              if (nA) ok = issue_s(SlotA{}, un, jn);
              if (ok && nB) ok = issue_s(SlotB{}, un, jn);
              if (ok) mma_commit_w(bar_kempty + (un % KS));
            }
            if (ok && jA) ok = issue_pv(SlotA{}, u);
            if (ok && jB) ok = issue_pv(SlotB{}, u);
            if (ok) mma_commit_w(bar_vempty + (u % VS));
          } else {
            // tile A: P_A(j) V_j, then S_A(j+1) over the columns P_A(j) just left
            if (jA) ok = issue_pv(SlotA{}, u);
            if (ok && more && nA) ok = issue_s(SlotA{}, un, jn);
            if (ok && jB) ok = issue_pv(SlotB{}, u);
            if (ok) mma_commit_w(bar_vempty + (u % VS));
            if (ok && more && nB) ok = issue_s(SlotB{}, un, jn);
            if (ok && more) mma_commit_w(bar_kempty + (un % KS));
          }
          j = jn;
          jA = nA;
          jB = nB;
          u = un;
        }
      }
      mma_commit_w(bar_final);
      mbar_wait_drain(bar_final, 0, wait_limit);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int t = (warp - kSoft0) >> 2;  // which Q slot
    const int r = (warp & 3) * 32 + lane;     // row within the tile == TMEM lane (quarter warp % 4)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_col = t * 128;
    const uint32_t p_col = L::p_col(t);
    const uint32_t o_col = L::kTO + t * D;
    int ns = 0;  // S tiles of this slot consumed so far (sfull / pfull / odone phases)
    bool ok = true;
    for (int ri = 0; ok; ++ri) {
      const Unit un0 = unit(ri);
      if (un0.k < 0) break;
      const FwdItem it = make_item<CAUSAL, kHP, kAltSlots>(g, un0, kSort ? item_order(bars) : nullptr);
      const int qt = t ? it.qtB : it.qtA;
      if (qt < 0) continue;
      const int jbeg = t ? it.tsB.begin : it.tsA.begin, jend = t ? it.tsB.end : it.tsA.end;
      const int kv_bound = it.kv_bound;
      const int row = qt * kBlock + r;
      const int bh = kHP ? (t ? it.bhB : it.bh) : it.bh;  // this slot's (batch, head)
      float m = -INFINITY;  // reference max, log2 units (scale folded in)
      float l = 0.f;        // sum of exp2(s * scale_log2 - m) over visited keys
      int n = 0;            // tiles of this item
      // One K/V tile j of this slot: S_t(j) from TMEM, the online softmax
      // update, P_t(j) to TMEM, then pfull. False when the CTA is aborting.
      auto tile = [&](const int j) -> bool {
        // Keep decisions of this row's 128 keys, one word per 32 keys
        // (keep_bits32). They do not depend on S, so they are drawn before
        // S_t(j) is awaited: the draws fill the wait for the MMA instead of
        // lengthening the softmax, which the next MMA waits for.
        uint32_t kb[4] = {0u, 0u, 0u, 0u};
        if constexpr (DROP) {
          const uint32_t c4 = 0x80808080u - (dp.thresh4 & 0x7f7f7f7fu);
          const uint32_t g0 = static_cast<uint32_t>(j * kBlock) >> 4;  // 16-key group of key j*128
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 ra = philox4x32_10(g0 + 2 * q, row, bh, dp.offset, dp.k0, dp.k1);
            const uint4 rb = philox4x32_10(g0 + 2 * q + 1, row, bh, dp.offset, dp.k0, dp.k1);
            kb[q] = keep_bits32(ra, rb, dp.thresh4, c4);
          }
          asm volatile("" : "+r"(kb[0]), "+r"(kb[1]), "+r"(kb[2]), "+r"(kb[3]));
        }
        if (!mbar_wait_warp<true>(bar_sfull + t, ns & 1, wd)) {
          return false;
        }
        tc_fence_after();
        uint32_t rs[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + s_col + c * 32, rs[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence(rs[c]);
        if constexpr (kSepP) {  // S_t may be overwritten by the next tile's S now
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_sfree + t);
        }
        float sv[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) sv[c] = __uint_as_float(rs[c >> 5][c & 31]);
        if ((j + 1) * kBlock > kv_bound || (CAUSAL && j == qt)) {
          if constexpr (CAUSAL && MODE != kModeSparse) {
            // Edge tile: this row's keys [0, lim) of the tile are visible (the
            // rest lie past the valid length or, on the diagonal, after the
            // query); one compare with a constant per column (GPT-2 forward
            // 35.5 -> 33.4 us against a compare of each key with both bounds).
            int lim = kv_bound - j * kBlock;
            if (j == qt) lim = min(lim, r + 1);
#pragma unroll
            for (int c = 0; c < 128; ++c) sv[c] = c < lim ? sv[c] : -INFINITY;
          } else {
            // The same in effect, one key at a time: this form measured faster
            // on the non-causal kernels (BERT-large forward 37.5 against
            // 39.6 us) and spills less in the causal block-sparse one.
#pragma unroll
            for (int c = 0; c < 128; ++c) {
              const int key = j * kBlock + c;
              if (key >= kv_bound || (CAUSAL && key > row)) sv[c] = -INFINITY;
            }
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
        if (kSepP && n >= 1) {
          // P_t's columns are free (and O quiescent) once this item's previous P V is done.
          if (!mbar_wait_warp<true>(bar_odone + t, (ns - 1) & 1, wd)) {
            return false;
          }
          tc_fence_after();
        }
        // P_t (bf16 pairs) goes to TMEM 16 columns at a time as soon as it is
        // formed -- in its own columns, or over the first 64 columns of S_t,
        // whose fp32 values are already in registers -- so that few packed
        // words are live at once.
        // At d = 128 the scale, shift and row sum work on pairs of columns
        // (f32x2: half the instructions; the d = 64 variants measured slower
        // with it, their register allocation being tighter).
        const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(-m_use, -m_use);
        uint64_t ps2[2] = {0ull, 0ull};  // (+0, +0)
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            if constexpr (D == 128) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(sv[2 * (c0 + c)], sv[2 * (c0 + c) + 1]), sc2, nm2), x0, x1);
              const float p0 = ex2(x0), p1 = ex2(x1);
              pk[c] = pack_bf16(p0, p1);
              ps2[c & 1] = f2_add(ps2[c & 1], f2_pack(p0, p1));
            } else {
              const float p0 = ex2(fmaf(sv[2 * (c0 + c)], scale_log2, -m_use));
              const float p1 = ex2(fmaf(sv[2 * (c0 + c) + 1], scale_log2, -m_use));
              pk[c] = pack_bf16(p0, p1);
              ps[c & 3] += p0 + p1;
            }
          }
          if constexpr (DROP) {  // keys j*128 + 2*c0 + [0, 32)
#pragma unroll
            for (int c = 0; c < 16; ++c) pk[c] &= pair_mask_bits(kb[c0 >> 4], c);
          }
          tmem_st16(lane_base + p_col + c0, pk);
        }
        if constexpr (D == 128) {
          f2_unpack(ps2[0], ps[0], ps[1]);
          f2_unpack(ps2[1], ps[2], ps[3]);
        }
        const float tsum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
        if (n >= 1 && __any_sync(0xffffffffu, grow)) {
          // O must be quiescent (this item's previous P V done) before it is rescaled.
          if (!kSepP) {
            if (!mbar_wait_warp<true>(bar_odone + t, (ns - 1) & 1, wd)) {
              return false;
            }
            tc_fence_after();
          }
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
        ++ns;
        return true;
      };
      if constexpr (MODE == kModeSparse) {
        // The mask row's kept tiles one after the other; only the current
        // tile and the next one stay live across the tile computation.
        const uint8_t* mrow = g.block_mask + static_cast<size_t>(qt) * g.nqt;
        for (int j = next_kept(mrow, 1, jbeg, jend); ok && j < jend;) {
          const int jn = next_kept(mrow, 1, j + 1, jend);
          ok = tile(j);
          j = jn;
        }
      } else {
        for (int j = jbeg; ok && j < jend; ++j) ok = tile(j);
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      // O / l straight from TMEM to global memory (one row per thread); the
      // next item's first P V overwrites O only after this thread's next P
      // arrives, i.e. after these loads.
      bool have = n > 0;
      if (have) {
        if (!mbar_wait_warp<true>(bar_odone + t, (ns - 1) & 1, wd)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (MODE == kModeSplit && it.slot >= 0) {
        // Part of a split item: the unnormalised O, the row's running maximum
        // and sum go to the item's workspace slot; the merge kernel combines
        // the parts into O and LSE.
        // O is stored column-group major ([slot][D / 4][256 rows][4 floats]),
        // so that the 32 rows of a warp write 512 contiguous bytes per store.
        const size_t prow = static_cast<size_t>(it.slot) * 256 + t * kBlock + r;
        g.m_part[prow] = m;
        g.l_part[prow] = l;
        if (have) {
          float4* dst = reinterpret_cast<float4*>(g.o_part) + static_cast<size_t>(it.slot) * (D / 4) * 256 +
                        t * kBlock + r;
#pragma unroll
          for (int c0 = 0; c0 < D / 32; ++c0) {
            uint32_t o[32];
            tmem_ld32(lane_base + o_col + c0 * 32, o);
            tmem_wait_ld();
            reg_fence(o);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[(c0 * 8 + v) * 256] =
                  make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                              __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3]));
          }
        }
        continue;
      }
      const bool live = have && l > 0.f;
      const float inv = live ? (DROP ? dp.rescale : 1.f) / l : 0.f;
      const bool row_ok = row < g.N;
      if constexpr (L::kOStore) {
        // The warp's 32 rows of O go to its shared-memory box (16-byte chunk
        // u of row r at u ^ (r & 7)) and leave with one TMA store: whole
        // 128-byte rows in full sectors, rows past N clipped.
        uint8_t* obox = smem + L::kOst + (warp - kSoft0) * L::kOBox;
        const uint32_t ob = smem_u32(obox) + lane * 128;
        if (lane == 0) bulk_wait_read<0>();  // the previous item's store has read the box
        __syncwarp();
#pragma unroll
        for (int c0 = 0; c0 < 2; ++c0) {
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
          for (int v = 0; v < 4; ++v)
            st_shared_v4(ob + (((c0 * 4 + v) ^ (lane & 7)) << 4),
                         pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv),
                         pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv),
                         pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv),
                         pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_rows(&tm_o, obox, 0, qt * kBlock + (warp & 3) * 32, bh, g.H, g.st);
          bulk_commit();
        }
        if (row_ok)
          lse_out[static_cast<size_t>(bh) * g.N + row] = live ? (m + log2f(l)) * kLn2 : -INFINITY;
        continue;
      }
      uint4* orow = reinterpret_cast<uint4*>(out + row_offset(g.st, g.H, bh, row));
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
      if (row_ok)
        lse_out[static_cast<size_t>(bh) * g.N + row] = live ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
    if constexpr (L::kOStore) {  // the O stores have read their boxes and written O
      if (lane == 0) bulk_wait0();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merges the parts of the items cut by a split plan. Block (i, c) handles
// columns [32 c, 32 c + 32) of cut item i of the merge table, one thread per
// row of its two Q tiles: with m_q, l_q, O_q the running maximum (log2
// units), sum and unnormalised output of part q of the row, M = max_q m_q and
//   O = r sum_q 2^(m_q - M) O_q / sum_q 2^(m_q - M) l_q,
//   LSE = (M + log2 sum_q 2^(m_q - M) l_q) ln 2,
// which is the online-softmax rescaling applied once more, across the parts
// (r = 1 / (1 - p') with dropout, else 1). Parts that saw no key (l = 0) do
// not contribute; a row with no part left gets O = 0 and LSE = -inf. The
// partial O is read column-group major (512 contiguous bytes per warp load)
// and each thread writes 64 contiguous bytes of its output row.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(256) fwd_merge_kernel(FwdGrid g, const __grid_constant__ MergeTable m,
                                                        __nv_bfloat16* __restrict__ out,
                                                        float* __restrict__ lse_out, float rescale) {
  grid_dep_wait();  // the split kernel's parts are complete
  grid_dep_launch();
  const int i = blockIdx.x, c0 = blockIdx.y * 32;
  const int t = m.item[i], q0 = m.first[i], q1 = m.first[i + 1];
  int bh, p;
  fwd_item_coords(g.npairs, g.n_items / g.npairs, CAUSAL, t, bh, p);
  const int x = threadIdx.x;  // row of the pair: tile x / 128, row x % 128
  const int qt = 2 * p + (x >> 7), row = qt * kBlock + (x & 127);
  float M = -INFINITY;
  for (int q = q0; q < q1; ++q) {
    const size_t pr = static_cast<size_t>(m.slot[q]) * 256 + x;
    if (g.l_part[pr] > 0.f) M = fmaxf(M, g.m_part[pr]);
  }
  float Lsum = 0.f;
  float acc[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) acc[c] = 0.f;
  for (int q = q0; q < q1; ++q) {
    const int sl = m.slot[q];
    const float l = g.l_part[static_cast<size_t>(sl) * 256 + x];
    const float w = l > 0.f ? exp2f(g.m_part[static_cast<size_t>(sl) * 256 + x] - M) : 0.f;
    Lsum += w * l;
    const float4* src = reinterpret_cast<const float4*>(g.o_part) +
                        (static_cast<size_t>(sl) * (D / 4) + c0 / 4) * 256 + x;
    if (w > 0.f) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 a = src[c * 256];
        acc[4 * c] += w * a.x;
        acc[4 * c + 1] += w * a.y;
        acc[4 * c + 2] += w * a.z;
        acc[4 * c + 3] += w * a.w;
      }
    }
  }
  if (qt >= g.nqt || row >= g.N) return;
  if (c0 == 0)
    lse_out[static_cast<size_t>(bh) * g.N + row] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
  const float inv = Lsum > 0.f ? rescale / Lsum : 0.f;
  uint4* dst = reinterpret_cast<uint4*>(out + row_offset(g.st, g.H, bh, row) + c0);
#pragma unroll
  for (int c = 0; c < 4; ++c)
    dst[c] = make_uint4(pack_bf16(acc[8 * c] * inv, acc[8 * c + 1] * inv),
                        pack_bf16(acc[8 * c + 2] * inv, acc[8 * c + 3] * inv),
                        pack_bf16(acc[8 * c + 4] * inv, acc[8 * c + 5] * inv),
                        pack_bf16(acc[8 * c + 6] * inv, acc[8 * c + 7] * inv));
}

// Launches fwd_kernel<D, CAUSAL, DROP, MODE> on `grid` CTAs.
template <int D, bool CAUSAL, bool DROP, int MODE>
cudaError_t launch_fwd_kernel(const FwdLaunch& a, const FwdGrid& g, int grid, cudaStream_t stream) {
  using L = FwdLayout<D, MODE == kModeSparse && D == 64>;
  auto kern = fwd_kernel<D, CAUSAL, DROP, MODE>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = set_smem_once(smem_set, reinterpret_cast<const void*>(kern), L::kSmem);
  if (e != cudaSuccess) return e;
  const float scale_log2 = a.scale * 1.4426950408889634f;
  return launch_pdl(kern, dim3(grid), dim3(FwdWarps<D>::kThreads), L::kSmem, stream, a.tm_q, a.tm_k,
                    a.tm_v, a.tm_o, a.o, a.lse, g, scale_log2, a.drop, a.status, a.wait_limit);
}

// The split kernel over the tail on `grid` (= plan.tail_ctas) CTAs, then the
// merge kernel over the cut items of `m`.
template <int D, bool CAUSAL, bool DROP>
cudaError_t launch_fwd_tail(const FwdLaunch& a, const FwdGrid& g, int grid, const MergeTable& m,
                            cudaStream_t stream) {
  cudaError_t e = launch_fwd_kernel<D, CAUSAL, DROP, kModeSplit>(a, g, grid, stream);
  if (e != cudaSuccess || m.n == 0) return e;
  return launch_pdl(fwd_merge_kernel<D, CAUSAL>, dim3(m.n, D / 32), dim3(256), 0, stream, g, m,
                    static_cast<__nv_bfloat16*>(a.o), a.lse, a.drop.enabled ? a.drop.rescale : 1.f);
}

// The (d, causal) variants of one dropout setting and mode.
template <bool DROP, int MODE>
cudaError_t launch_fwd_variant(const FwdLaunch& a, const FwdGrid& g, int grid, cudaStream_t stream) {
  const bool causal = a.causal != 0;
  if (a.d == 64)
    return causal ? launch_fwd_kernel<64, true, DROP, MODE>(a, g, grid, stream)
                  : launch_fwd_kernel<64, false, DROP, MODE>(a, g, grid, stream);
  return causal ? launch_fwd_kernel<128, true, DROP, MODE>(a, g, grid, stream)
                : launch_fwd_kernel<128, false, DROP, MODE>(a, g, grid, stream);
}

}  // namespace
}  // namespace fa
