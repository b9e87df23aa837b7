// Thin inline-PTX layer for sm_103a: mbarriers, TMA bulk-tensor loads,
// Tensor Memory (TMEM) allocation / load / store, tcgen05 MMAs and their
// shared-memory and instruction descriptors, plus a bounded mbarrier wait.
//
// Every wait in the kernels goes through mbar_wait(), which gives up after a
// cycle budget, records FA_ERR_DEVICE_TIMEOUT in the caller-visible status
// word and raises a CTA-wide abort flag so that every other role stops
// waiting too. Nothing here traps.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "fa.h"
#include "fa_internal.h"

namespace fa {

// ------------------------------------------------------------------ basics
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31; }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ dependent launch
// Waits until the grids this one depends on (the previous kernel on the
// stream, when launched with programmatic dependent launch) have completed
// and their memory is visible; a no-op otherwise.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allows the next kernel on the stream to be set up now; it still waits for
// this grid's completion before it reads anything.
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Per-CTA watchdog: the cycle budget of one wait, the status word in global
// memory, and the CTA's abort flag in shared memory.
struct Watchdog {
  long long limit;
  int* status;
  volatile int* abort;
};

static __device__ __noinline__ void watchdog_fire(int* status, volatile int* abort) {
  *abort = 1;
  atomicCAS(status, FA_OK, FA_ERR_DEVICE_TIMEOUT);
}
// Same, inlined: for waits of threads that hold many live registers (the
// forward softmax), where the call's register saves cost more than the code.
static __device__ __forceinline__ void watchdog_fire_inline(int* status, volatile int* abort) {
  *abort = 1;
  atomicCAS(status, FA_OK, FA_ERR_DEVICE_TIMEOUT);
}

// Waits for the phase with the given parity to complete. Returns false if the
// CTA is aborting or the budget ran out (then the abort flag is raised).
template <bool kInlineFire = false>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Watchdog& wd) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*wd.abort) return false;
    if (clock64() - t0 > wd.limit) {
      if (kInlineFire)
        watchdog_fire_inline(wd.status, wd.abort);
      else
        watchdog_fire(wd.status, wd.abort);
      return false;
    }
  }
}

// Same, but ignores the abort flag: used only to drain copies already in
// flight before the CTA exits.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the MMA issuer: one non-blocking test_wait first (the
// phase has usually completed already), then try_wait, which lets the
// hardware park the warp instead of spinning; a spinning issuer warp takes
// issue slots from the compute warps that share its sub-partition.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity, const Watchdog& wd) {
  if (mbar_test_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*wd.abort) return false;
    if (clock64() - t0 > wd.limit) {
      watchdog_fire(wd.status, wd.abort);
      return false;
    }
  }
}

// mbar_wait_spin for a warp that issues through elect.sync: every lane polls
// and the verdict is made warp-uniform, so the warp stays converged.
__device__ __forceinline__ bool mbar_wait_spin_w(uint64_t* bar, uint32_t parity,
                                                 const Watchdog& wd) {
  const bool ok = mbar_wait_spin(bar, parity, wd);
  return __all_sync(0xffffffffu, ok);
}

// Warp-uniform wait: every lane waits, lane 0's verdict is broadcast.
template <bool kInlineFire = false>
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, const Watchdog& wd) {
  bool ok = mbar_wait<kInlineFire>(bar, parity, wd);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load (x = innermost, in elements) into shared memory; completion
// is signalled on `bar` as transaction bytes.
// Checked builds (compiled with -DFA_CHECKS=1; build(checked=True)): every
// TMA copy first checks its coordinates and addresses -- the innermost
// coordinate a multiple of 16 bytes, no negative coordinate for a store or a
// reduction, shared-memory addresses 128-byte aligned, bulk copies of whole
// 16-byte units. A failed check records FA_ERR_DEVICE_CHECK (5) in the status
// word and skips the copy; the wait for a skipped load then gives up, bounded,
// so the kernel returns instead of faulting. The kernels that issue TMA
// copies hand the status word's address to check_init at their start.
#ifndef FA_CHECKS
#define FA_CHECKS 0
#endif
#if FA_CHECKS
static __device__ int* g_check_status;  // one per translation unit
static __device__ __forceinline__ void check_init(int* status) {
  if (threadIdx.x == 0) g_check_status = status;  // before the kernel's first __syncthreads
}
static __device__ __noinline__ bool check_failed() {
  if (g_check_status != nullptr) atomicCAS(g_check_status, 0, 5);
  return true;
}
#define FA_CHECK_FAILS(cond) (!(cond) && check_failed())
#else
__device__ __forceinline__ void check_init(int*) {}
#define FA_CHECK_FAILS(cond) false
#endif

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
  if (FA_CHECK_FAILS((x & 7) == 0 && (smem_u32(dst) & 127u) == 0 && (smem_u32(bar) & 7u) == 0)) return;
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// 4-D tiled load (x = innermost, in elements) into shared memory.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z, int w) {
  if (FA_CHECK_FAILS((x & 7) == 0 && (smem_u32(dst) & 127u) == 0 && (smem_u32(bar) & 7u) == 0)) return;
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

// 128 rows (starting at `row`) x 64 columns (starting at `x`) of problem
// bh = b*H + h from a [B, H, N, d] tensor map laid out as `st` says.
__device__ __forceinline__ void tma_load_rows(void* dst, const CUtensorMap* map, uint64_t* bar,
                                              int x, int row, int bh, int H, const Strides& st) {
  if (st.merged) {
    tma_load_3d(dst, map, bar, x, row, bh);
  } else {
    int y0, y1, y2;
    row_coords(st, row, bh % H, bh / H, y0, y1, y2);
    tma_load_4d(dst, map, bar, x, y0, y1, y2);
  }
}

// 3-D / 4-D tiled stores shared -> global (bulk-group completion), the
// counterparts of the loads above: whole 128-byte rows leave in full sectors,
// and rows beyond the tensor's extent are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z) {
  if (FA_CHECK_FAILS((x & 7) == 0 && x >= 0 && y >= 0 && z >= 0 && (smem_u32(src) & 127u) == 0)) return;
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z, int w) {
  if (FA_CHECK_FAILS((x & 7) == 0 && x >= 0 && y >= 0 && z >= 0 && w >= 0 && (smem_u32(src) & 127u) == 0))
    return;
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
// 128 rows (from `row`) x 64 columns (from `x`) of problem bh of a [B, H, N, d]
// tensor map, from a 128-byte-swizzled shared-memory chunk.
__device__ __forceinline__ void tma_store_rows(const CUtensorMap* map, const void* src, int x, int row,
                                               int bh, int H, const Strides& st) {
  if (st.merged) {
    tma_store_3d(map, src, x, row, bh);
  } else {
    int y0, y1, y2;
    row_coords(st, row, bh % H, bh / H, y0, y1, y2);
    tma_store_4d(map, src, x, y0, y1, y2);
  }
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The shared-memory sources of every committed bulk group have been read.
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// At most N of the most recently committed bulk groups still read their
// shared-memory sources.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Every committed bulk group has completed (its global writes performed).
__device__ __forceinline__ void bulk_wait0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  if (FA_CHECK_FAILS((smem_u32(dst) & 15u) == 0 && (reinterpret_cast<uint64_t>(src) & 15u) == 0 &&
                     (bytes & 15u) == 0 && (smem_u32(bar) & 7u) == 0))
    return;
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: lane i of the warp reads TMEM lane
// (32 * (warp % 4) + i) -- the lane field of `taddr` must name that quarter.
// Pairs of fp32 values in one 64-bit register for the packed f32x2
// arithmetic of sm_100 and later (each half rounded like its scalar form).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Registers written by tcgen05.ld are only valid after tcgen05.wait::ld. This
// empty statement re-defines them after the wait so that no use can be
// scheduled between the load and the wait.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]));
}

// ------------------------------------------------------------------ tcgen05.mma
// Shared-memory matrix descriptor, 128-byte swizzle. `lbo`/`sbo` in bytes.
//  K-major operand: rows of 128 B (64 bf16 of K) in 8-row / 1024 B swizzle
//    atoms; sbo = distance between 8-row groups (1024 when packed); lbo unused.
//  MN-major operand: 64 contiguous MN elements x 8 K-rows per atom; lbo =
//    distance between 64-element MN groups, sbo = distance between 8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Advances a shared-memory descriptor by `bytes` (a multiple of 16). The start
// address field holds (address >> 4) in the low 14 bits, so the add is exact
// while the address stays inside shared memory; issuing threads build each
// operand's descriptor once and step it with compile-time offsets, which
// keeps the per-MMA issue cost to a single add.
__device__ __forceinline__ uint64_t desc_adv(uint64_t d, uint32_t bytes) {
  return d + static_cast<uint64_t>(bytes >> 4);
}

// Instruction descriptor, kind::f16: bf16 x bf16 -> f32 accumulate, dense.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                                    // D format: f32
         | (1u << 7)                                  // A format: bf16
         | (1u << 10)                                 // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)             // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)             // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)      // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);     // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
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

// Warp-wide forms: the whole (converged) warp executes them and elect.sync
// picks the one lane that issues. Issued this way an MMA costs the tensor
// pipe's own time, while a lone lane of a diverged warp needs more cycles per
// MMA than an N = 64 MMA takes to run, and more still when the neighbouring
// warps are busy. With every lane active the elected lane is always the same
// one, so a commit tracks every MMA issued before it.
__device__ __forceinline__ void mma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Plain (immediate) arrive by one elected lane of a converged warp.
__device__ __forceinline__ void mbar_arrive_w(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

}  // namespace fa
