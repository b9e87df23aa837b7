// Work scheduling shared by the persistent kernels: which K/V (or Q) tiles a
// work item visits, walked through warp-wide bitmaps of the block mask, and
// how the items are shared out over the CTAs, including the split of the
// last, partial wave of items into equal runs of tiles (stream-K).
//
// Tile sets. A Q tile of the forward visits the K/V tiles j in [begin, end)
// whose block-mask byte is non-zero (every j without a mask); a key tile of
// the backward visits the Q tiles i in [begin, end) whose mask row keeps it.
// The mask bytes of 128 consecutive tiles are read by one warp at once (each
// lane reads four independent bytes) and turned into a 128-bit bitmap with
// __ballot_sync, so a walk costs one round trip to L1/L2 per 128 tiles
// instead of one per tile.
//
// Split of the last wave (stream-K). With n items on G CTAs, whole rounds of
// G items leave a last round of n mod G items that keeps only part of the GPU
// busy. The items of that last round (the tail) are instead laid end to end
// as steps -- one step is one K/V tile of a forward item, one Q tile of a
// backward item -- and CTA c runs steps [c T / G, (c + 1) T / G) of them, so
// that every CTA ends at about the same time. An item cut between CTAs is
// computed in parts; each part leaves its partial result in a workspace slot
// (2c for the CTA's first tail item, 2c + 1 for its last), and a merge kernel
// combines the parts of each cut item. The plan is made on the host from the
// sizes alone, with a cost model that splits only when the estimated finish
// time falls.
#pragma once

#include <cstdint>

#include "fa_internal.h"

namespace fa {

// "No further tile" marker of the tile walks.
constexpr int kNoTile = 1 << 30;

// The tiles one Q tile (forward) or key tile (backward) visits: t in
// [begin, end) with mask[t * stride] != 0, or every t if mask is null.
struct TileSet {
  int begin, end;
  const uint8_t* mask;
  int stride;
};

// Bits of tiles [w0, w0 + 128) of `ts` (bit b of word b / 32 is tile w0 + b).
// Warp-collective: every lane returns the same words.
__device__ __forceinline__ void tile_window(const TileSet& ts, int w0, uint32_t (&bits)[4]) {
  const int l = threadIdx.x & 31;
  uint8_t v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int t = w0 + 32 * k + l;
    const bool in = t >= ts.begin && t < ts.end;
    v[k] = in ? (ts.mask == nullptr ? 1 : ts.mask[static_cast<long long>(t) * ts.stride]) : 0;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) bits[k] = __ballot_sync(0xffffffffu, v[k] != 0);
}

// Lowest set bit >= p (0 <= p <= 128) of a 128-bit map, or 128.
__device__ __forceinline__ int bits_next(const uint32_t (&b)[4], int p) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (p < 32 * (k + 1)) {
      const int sh = p - 32 * k;
      const uint32_t w = sh > 0 ? (b[k] & (~0u << sh)) : b[k];
      if (w != 0u) return 32 * k + __ffs(static_cast<int>(w)) - 1;
    }
  }
  return 128;
}

// Highest set bit of a 128-bit map, or -1.
__device__ __forceinline__ int bits_last(const uint32_t (&b)[4]) {
#pragma unroll
  for (int k = 3; k >= 0; --k)
    if (b[k] != 0u) return 32 * k + 31 - __clz(static_cast<int>(b[k]));
  return -1;
}

// Walks the tiles of a TileSet in increasing order. Without a mask the walk
// is plain arithmetic; with one it keeps the bitmap of one 128-tile window,
// in registers or -- for warps whose registers are all taken by the tile
// computation -- in four words of shared memory owned by the warp (kSmem).
// Every call is warp-collective and returns the same value on every lane.
template <bool kSmem = false>
struct TileWalk {
  TileSet ts;
  int w0;
  uint32_t b[kSmem ? 1 : 4];
  uint32_t* sb;  // kSmem: the warp's four words

  __device__ __forceinline__ void init(const TileSet& s, uint32_t* smem_words = nullptr) {
    ts = s;
    w0 = -1;
    sb = smem_words;
  }
  // The first tile >= j of the set, or kNoTile.
  __device__ __forceinline__ int seek(int j) {
    if (j < ts.begin) j = ts.begin;
    if (ts.mask == nullptr) return j < ts.end ? j : kNoTile;
    while (j < ts.end) {
      const int w = j & ~127;
      uint32_t bb[4];
      if (w != w0) {
        w0 = w;
        tile_window(ts, w, bb);
        if constexpr (kSmem) {
          if ((threadIdx.x & 31) == 0) {
            volatile uint32_t* v = sb;
            v[0] = bb[0];
            v[1] = bb[1];
            v[2] = bb[2];
            v[3] = bb[3];
          }
          __syncwarp();
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) b[k] = bb[k];
        }
      } else {
        if constexpr (kSmem) {
          const volatile uint32_t* v = sb;
          bb[0] = v[0];
          bb[1] = v[1];
          bb[2] = v[2];
          bb[3] = v[3];
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) bb[k] = b[k];
        }
      }
      const int p = bits_next(bb, j - w);
      if (p < 128) return w + p < ts.end ? w + p : kNoTile;
      j = w + 128;
    }
    return kNoTile;
  }
  // The last tile of the set, or -1 (leaves the cached window alone).
  __device__ __forceinline__ int last() const {
    if (ts.end <= ts.begin) return -1;
    if (ts.mask == nullptr) return ts.end - 1;
    for (int w = (ts.end - 1) & ~127; w >= (ts.begin & ~127); w -= 128) {
      uint32_t bb[4];
      tile_window(ts, w, bb);
      const int p = bits_last(bb);
      if (p >= 0) return w + p;
    }
    return -1;
  }
  // Number of tiles in the set.
  __device__ __forceinline__ int count() const {
    if (ts.end <= ts.begin) return 0;
    if (ts.mask == nullptr) return ts.end - ts.begin;
    int n = 0;
    for (int w = ts.begin & ~127; w < ts.end; w += 128) {
      uint32_t bb[4];
      tile_window(ts, w, bb);
      n += __popc(bb[0]) + __popc(bb[1]) + __popc(bb[2]) + __popc(bb[3]);
    }
    return n;
  }
};

// Lists the tiles of window [w0, w0 + 128) of `ts` as offsets from w0, in
// increasing order, in `list` (128 bytes of the warp's shared memory);
// returns how many. Warp-collective. Out of line: it runs once per window,
// and inlined into the loop nests of the tile computation its registers
// would add to theirs.
static __device__ __noinline__ int list_window(TileSet ts, int w0, uint8_t* list) {
  const int lane = threadIdx.x & 31;
  uint32_t bb[4];
  tile_window(ts, w0, bb);
  int base = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // lane l lists tile w0 + 32 q + l if it is in the set
    if ((bb[q] >> lane) & 1u) list[base + __popc(bb[q] & ((1u << lane) - 1u))] = 32 * q + lane;
    base += __popc(bb[q]);
  }
  __syncwarp();
  return base;
}

// The first tile >= j of [j, end) that the mask keeps (mask[c * stride] !=
// 0; stride 1 walks a mask row, the number of tiles a column), or `end`:
// 32 mask bytes per step, one per lane, and a ballot. Warp-collective. Out
// of line for the same reason as list_window: its caller keeps only j and
// the result live across the tile computation.
static __device__ __noinline__ int next_kept(const uint8_t* __restrict__ mask, int stride, int j, int end) {
  const int lane = threadIdx.x & 31;
  for (int b = j; b < end; b += 32) {
    const int c = b + lane;
    const bool keep = c < end && __ldg(mask + static_cast<size_t>(c) * stride) != 0;
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    if (bal != 0u) return b + __ffs(static_cast<int>(bal)) - 1;
  }
  return end;
}

// As list_window, for the union of two tile sets (the two Q tiles of a
// forward item share their K/V loads).
static __device__ __noinline__ int list_window2(TileSet a, TileSet b, int w0, uint8_t* list) {
  const int lane = threadIdx.x & 31;
  uint32_t ba[4], bb[4];
  tile_window(a, w0, ba);
  tile_window(b, w0, bb);
  int base = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t u = ba[q] | bb[q];
    if ((u >> lane) & 1u) list[base + __popc(u & ((1u << lane) - 1u))] = 32 * q + lane;
    base += __popc(u);
  }
  __syncwarp();
  return base;
}

// ------------------------------------------------------------------ cost-sorted item order
// With a block mask the items of a pass differ in cost, and dealing them out
// in index order can leave some SMs with far more tiles than others (3 to 12
// kept tiles per mask row: up to a third more than the average). Such items
// form groups of equal cost -- a mask row or pair of rows (forward), a key
// tile (backward) -- and at its start every CTA sorts the groups by
// decreasing cost, ties by increasing index, into a table in shared memory
// (the same table in every CTA); item k is then member k % inner of group
// order[k / inner], and the snake over the item list deals out the heaviest
// items first.
constexpr int kOrderMax = 640;  // groups a table holds; with more, index order
constexpr int kCostMax = 1023;  // costs above this sort as equal
// Both persistent kernels keep, in 64-bit words from their barrier area, a
// flag at word 40 (non-zero: the table is in use) and the table itself from
// byte 640 (after the producer's 128-byte tile list at word 64).
constexpr int kOrderFlagWord = 40;

// The CTA's group table, or null for index order. Read from shared memory at
// every item, so that no role keeps it live across its tile loops.
__device__ __forceinline__ const uint16_t* item_order(const uint64_t* bars) {
  const int on = *reinterpret_cast<const volatile int*>(bars + kOrderFlagWord);
  return on ? reinterpret_cast<const uint16_t*>(bars + 64) + 64 : nullptr;
}

// Warp-collective: order[0, G) = the groups 0 .. G-1 by decreasing cost[]
// (ties by increasing index); costs above maxc (<= kCostMax) count as maxc.
// `hist` is scratch of maxc + 1 ints. A counting sort: histogram of the
// costs, the first slot of every cost by a scan from the top, then the
// groups placed 32 at a time (lanes of equal cost ranked by __match_any_sync).
static __device__ __noinline__ void sort_groups(const int* cost, int G, int maxc, int* hist,
                                                uint16_t* order) {
  const int lane = threadIdx.x & 31;
  for (int v = lane; v <= maxc; v += 32) hist[v] = 0;
  __syncwarp();
  for (int i = lane; i < G; i += 32) atomicAdd(&hist[min(cost[i], maxc)], 1);
  __syncwarp();
  int run = 0;  // groups costing more than the current chunk's top
  for (int top = maxc; top >= 0; top -= 32) {
    const int v = top - lane;
    const int h = v >= 0 ? hist[v] : 0;
    int x = h;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    __syncwarp();
    if (v >= 0) hist[v] = run + x - h;
    run += __shfl_sync(0xffffffffu, x, 31);
  }
  __syncwarp();
  for (int base = 0; base < G; base += 32) {
    const int i = base + lane;
    const bool act = i < G;
    const int v = act ? min(cost[i], maxc) : -1 - lane;  // inactive lanes match nobody
    const unsigned peers = __match_any_sync(0xffffffffu, v);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int s = act ? hist[v] : 0;
    if (act) order[s + rank] = static_cast<uint16_t>(i);
    __syncwarp();
    if (act && rank == 0) hist[v] = s + __popc(peers);
    __syncwarp();
  }
}

// Block-wide: kept(r, c) for every non-zero byte mask[r n + c] of an n x n
// block mask (16-byte loads when the mask's address and n allow them).
template <typename Fn>
__device__ __forceinline__ void for_kept_blocks(const uint8_t* __restrict__ mask, int n, Fn kept) {
  if ((reinterpret_cast<uintptr_t>(mask) & 15u) == 0 && (n & 15) == 0) {
    const int per_row = n >> 4, total = n * per_row;
    const uint4* m4 = reinterpret_cast<const uint4*>(mask);
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
      const uint4 w = __ldg(m4 + idx);
      const int r = idx / per_row, c0 = (idx - r * per_row) * 16;
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // top bit of each byte: the byte is non-zero
        uint32_t nz = (((ws[q] & 0x7f7f7f7fu) + 0x7f7f7f7fu) | ws[q]) & 0x80808080u;
        while (nz != 0u) {
          const int b = (__ffs(static_cast<int>(nz)) - 1) >> 3;
          kept(r, c0 + 4 * q + b);
          nz &= nz - 1u;
        }
      }
    }
  } else {
    const int total = n * n;
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x)
      if (__ldg(mask + idx) != 0) kept(idx / n, idx % n);
  }
}

// ------------------------------------------------------------------ item plan
// Fewest tail steps a CTA is given: a part costs a partial-result write and
// the merge a read of it, which a part of one or two steps would not repay.
constexpr int kMinTailSteps = 4;

// Margin of the split decision: split when the estimated finish time falls
// below this share of the unsplit one. At 0.98 the 16K non-causal forward
// (estimate 0.976) splits: measured 1430 -> 1407 us; the 4K non-causal
// forward (estimate 1.02) measured 122 -> 129 us when forced to split.
#ifndef FA_SPLIT_MARGIN
#define FA_SPLIT_MARGIN 0.98
#endif


// Whole rounds of a plan.
__host__ __device__ __forceinline__ int plan_rounds(const SplitPlan& p, int G) {
  return p.whole < p.n_items ? p.whole / G : (p.n_items + G - 1) / G;
}

// Finds the tail range of CTA c of the split kernel (tail_ctas CTAs);
// steps(k) gives the steps of item k. Warp-collective (one warp), the tail
// items scanned 32 at once.
template <typename StepsFn>
__device__ TailRange tail_range(const SplitPlan& p, int c, StepsFn steps) {
  TailRange tr{0, 0, -1, 0};
  if (p.whole >= p.n_items || c >= p.tail_ctas) return tr;
  const long long s0 = p.tail * c / p.tail_ctas, s1 = p.tail * (c + 1) / p.tail_ctas;
  if (s1 <= s0) return tr;
  const int lane = threadIdx.x & 31;
  long long acc = 0;
  bool f0 = false;
  for (int base = p.whole; base < p.n_items; base += 32) {
    const int k = base + lane;
    const long long n = k < p.n_items ? static_cast<long long>(steps(k)) : 0;
    long long inc = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    const long long end_k = acc + inc, beg_k = end_k - n;
    const bool live = k < p.n_items && n > 0;
    const uint32_t m0 = __ballot_sync(0xffffffffu, live && beg_k <= s0 && s0 < end_k);
    if (!f0 && m0 != 0u) {
      const int l = __ffs(static_cast<int>(m0)) - 1;
      tr.t0 = base + l;
      tr.o0 = static_cast<int>(s0 - __shfl_sync(0xffffffffu, beg_k, l));
      f0 = true;
    }
    const uint32_t m1 = __ballot_sync(0xffffffffu, live && beg_k <= s1 - 1 && s1 - 1 < end_k);
    if (m1 != 0u) {
      const int l = __ffs(static_cast<int>(m1)) - 1;
      tr.t1 = base + l;
      tr.o1 = static_cast<int>(s1 - __shfl_sync(0xffffffffu, beg_k, l));
      break;
    }
    acc = __shfl_sync(0xffffffffu, end_k, 31);
  }
  return tr;
}

// One unit of a CTA's work: item k, steps [sb, se) of it, and the workspace
// slot of its partial result (-1: the whole item, results written directly).
struct Unit {
  int k, sb, se, slot;
};

// The r-th tail unit of CTA c of the split kernel (k = -1 when there is
// none). `trp` points to the CTA's TailRange in shared memory; it is read
// afresh at every call, so that callers short of registers do not keep it
// live. A cut item's part goes to slot 2c if it is the CTA's first tail
// item, else to slot 2c + 1.
template <typename StepsFn>
__device__ __forceinline__ Unit tail_unit(const TailRange* trp, int r, int c, StepsFn steps) {
  Unit u{-1, 0, 0, -1};
  const volatile TailRange* v = trp;
  const TailRange tr{v->t0, v->o0, v->t1, v->o1};
  const int t = tr.t0 + r;
  if (t > tr.t1) return u;
  const int n = steps(t);
  u.k = t;
  u.sb = t == tr.t0 ? tr.o0 : 0;
  u.se = t == tr.t1 ? tr.o1 : n;
  if (u.sb > 0 || u.se < n) u.slot = 2 * c + (t == tr.t0 ? 0 : 1);
  return u;
}

// The merge table of a split plan, from the same arithmetic as tail_range
// and tail_unit (host side).
template <typename StepsFn>
inline MergeTable build_merge_table(const SplitPlan& p, StepsFn steps) {
  MergeTable m{};
  m.n = 0;
  m.first[0] = 0;
  int np = 0, cur = -1;
  int t = p.whole;
  long long beg = 0;  // first tail step of item t
  auto add = [&](int item, int slot) {
    if (item != cur) {
      m.item[m.n] = item;
      m.first[m.n] = static_cast<short>(np);
      ++m.n;
      cur = item;
    }
    m.slot[np++] = static_cast<short>(slot);
    m.first[m.n] = static_cast<short>(np);
  };
  for (int c = 0; c < p.tail_ctas; ++c) {
    const long long s0 = p.tail * c / p.tail_ctas, s1 = p.tail * (c + 1) / p.tail_ctas;
    if (s1 <= s0) continue;
    while (beg + steps(t) <= s0) beg += steps(t++);
    const int t0 = t, o0 = static_cast<int>(s0 - beg);
    int t1 = t;
    long long b1 = beg;
    while (b1 + steps(t1) <= s1 - 1) b1 += steps(t1++);
    const int o1 = static_cast<int>(s1 - b1);
    if (o0 > 0 || (t1 == t0 && o1 < steps(t0))) add(t0, 2 * c);
    if (t1 != t0 && o1 < steps(t1)) add(t1, 2 * c + 1);
  }
  return m;
}

// ------------------------------------------------------------------ item lists
// Forward items are pairs of adjacent Q tiles (2p, 2p + 1) of one (batch,
// head), bh = b H + h. Causal lists are ordered heaviest first (pairs near
// the diagonal's end see the most K/V tiles); otherwise a head's pairs are
// consecutive. A forward step is one K/V tile.
__host__ __device__ __forceinline__ void fwd_item_coords(int npairs, int BH, bool causal, int k,
                                                         int& bh, int& p) {
  if (causal) {
    p = npairs - 1 - k / BH;
    bh = k % BH;
  } else {
    bh = k / npairs;
    p = k % npairs;
  }
}

// Steps of forward item k without key padding or block mask.
__host__ __device__ __forceinline__ int fwd_item_steps(int nqt, int npairs, int BH, bool causal,
                                                       int k) {
  if (!causal) return nqt;
  int bh, p;
  fwd_item_coords(npairs, BH, causal, k, bh, p);
  const int last_q = 2 * p + 1 < nqt ? 2 * p + 1 : 2 * p;
  return last_q + 1 < nqt ? last_q + 1 : nqt;
}

// Backward items are key tiles j of one (batch, head). Causal lists are
// ordered heaviest first (key tile j meets nt - j query tiles); otherwise a
// head's key tiles are consecutive. A backward step is one Q tile.
__host__ __device__ __forceinline__ void bwd_item_coords(int nt, int BH, bool causal, int k,
                                                         int& bh, int& j) {
  if (causal) {
    j = k / BH;
    bh = k - j * BH;
  } else {
    bh = k / nt;
    j = k - bh * nt;
  }
}

// Steps of backward item k without key padding or block mask.
__host__ __device__ __forceinline__ int bwd_item_steps(int nt, int BH, bool causal, int k) {
  if (!causal) return nt;
  int bh, j;
  bwd_item_coords(nt, BH, causal, k, bh, j);
  return nt - j;
}

// ------------------------------------------------------------------ host planning
// Estimated finish times (in steps) with and without the split: every item
// costs its steps plus `item_cost`; a split adds, per CTA, up to two partial
// results (`part_cost` each) and the merge (`merge_cost`). The split is taken
// only when it brings the estimate below FA_SPLIT_MARGIN of the unsplit one.
template <typename StepsFn>
inline SplitPlan plan_split(int n_items, int G, StepsFn steps, double item_cost, double part_cost,
                            double merge_cost, bool allowed) {
  SplitPlan p{n_items, n_items, 0, 0};
  if (!allowed || G < 2 || n_items < 1) return p;
  const int W = n_items / G, R = n_items % G;
  if (R == 0 || W >= 8 || G > 4096) return p;
  static thread_local double load[4096];
  for (int c = 0; c < G; ++c) load[c] = 0.0;
  auto add = [&](int k) {
    const int r = k / G, c = (r & 1) ? G - 1 - k % G : k % G;
    load[c] += steps(k) + item_cost;
  };
  auto peak = [&] {
    double m = 0.0;
    for (int c = 0; c < G; ++c) m = load[c] > m ? load[c] : m;
    return m;
  };
  for (int k = 0; k < W * G; ++k) add(k);
  const double whole_max = peak();
  for (int k = W * G; k < n_items; ++k) add(k);
  const double ms0 = peak();
  long long T = 0;
  for (int k = W * G; k < n_items; ++k) T += steps(k);
  long long Gt = T / kMinTailSteps;
  if (Gt > G) Gt = G;
  if (Gt > kMaxSplitCtas) Gt = kMaxSplitCtas;
  if (Gt < 1) Gt = 1;
  const double ms1 = whole_max + static_cast<double>(T) / Gt + 2.0 * (item_cost + part_cost) +
                     merge_cost;
  if (!(ms1 < FA_SPLIT_MARGIN * ms0)) return p;
  p.whole = W * G;
  p.tail = T;
  p.tail_ctas = static_cast<int>(Gt);
  return p;
}


// Split plans of the two passes on G CTAs. Costs in steps (one K/V tile of
// a forward item, one Q tile of a backward item), measured on GB300 by timing
// launches with exactly one and two items per SM: the start-up and epilogue an
// item adds beyond its steps (forward 2.6 steps at d = 128, 1 at d = 64;
// backward 3 and 1.6), a partial result's write (about one step), and the
// merge kernel with the extra launch of the split kernel. `allowed` is false
// when a workspace, key padding or a block mask rules the split out.
inline SplitPlan plan_fwd(int B, int H, int N, int d, bool causal, int G, bool allowed) {
  const int nqt = (N + 127) / 128, npairs = (nqt + 1) / 2, BH = B * H;
  const int n = BH * npairs;  // callers have checked that B H ceil(N / 128) fits in an int
  return plan_split(n, G,
                    [&](int k) { return fwd_item_steps(nqt, npairs, BH, causal, k); },
                    d == 128 ? 2.6 : 1.0, 1.0, d == 128 ? 7.0 : 8.0, allowed);
}

inline SplitPlan plan_bwd(int B, int H, int N, int d, bool causal, int G, bool allowed) {
  const int nt = (N + 127) / 128, BH = B * H;
  const int n = BH * nt;
  return plan_split(n, G, [&](int k) { return bwd_item_steps(nt, BH, causal, k); },
                    d == 128 ? 3.0 : 1.6, 1.0, d == 128 ? 3.5 : 5.0, allowed);
}

}  // namespace fa
