// Inline-PTX building blocks for the sm_103a attention kernels: mbarriers
// with bounded waits, TMA tile copies, tcgen05 MMA / TMEM access and the
// shared-memory matrix descriptors the tensor core reads.
//
// Everything here is written from the public PTX ISA description of these
// instructions; nothing is taken from a vendor library.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "fa_internal.h"

namespace fa {

// ---------------------------------------------------------------------------
// Error word and bounded waits
// ---------------------------------------------------------------------------

// Sites recorded in the status word when a wait gives up (high byte = kernel).
enum : uint32_t {
  kSiteFwd = 0x100, kSiteDkdv = 0x200, kSiteDq = 0x300,
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared state every role of a CTA sees.  A wait that has not completed
// after limit_us is treated as a deadlock: the CTA records the site, raises its
// abort flag (ending every other wait of the CTA) and writes the launch's
// epoch to the abort word (ending the waits of the launch's other CTAs); all
// roles then unwind cleanly.  Only CTAs of the same launch (same epoch) react
// to the abort word, so a launch that gave up never cuts short another.
struct CtaGuard {
  volatile uint32_t* abort_flag;   // in shared memory
  unsigned int* status;            // device words: [0] status (first site wins), [1] abort epoch
  uint32_t epoch;                  // this launch's id (never 0)
  uint32_t limit_us;               // wait limit
};

__device__ __forceinline__ void guard_fail(const CtaGuard& g, uint32_t site) {
  *g.abort_flag = 1u;
  atomicCAS(g.status, 0u, site);
  atomicExch(g.status + 1, g.epoch);
}

// Has this CTA, or another CTA of the same launch, given up?
__device__ __forceinline__ bool guard_aborted(const CtaGuard& g) {
  return *g.abort_flag || *reinterpret_cast<volatile unsigned int*>(g.status + 1) == g.epoch;
}

__device__ __forceinline__ bool guard_expired(const CtaGuard& g, unsigned long long t0) {
  return global_ns() - t0 > static_cast<unsigned long long>(g.limit_us) * 1000ull;
}

// The polling loops run out of line by default: every wait site then shares
// one copy, which keeps the hot loops around them compact in the instruction
// cache.  A translation unit whose warps change their register budget with
// setmaxnreg (which out-of-line calls cannot follow) defines FA_INLINE_WAITS.
// Internal linkage either way: several translation units include this header.
#ifdef FA_INLINE_WAITS
#define FA_WAIT_LINKAGE static __forceinline__
#else
#define FA_WAIT_LINKAGE static __noinline__
#endif

// Wait for the phase of `bar` with the given parity.  Returns false (without
// waiting further) once the CTA is aborting or the wait limit is exceeded.
__device__ __forceinline__ bool mbar_poll(uint64_t* bar, uint32_t parity, const CtaGuard& g, uint32_t site) {
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      // this CTA or another of the launch gave up: unwind at once
      if (guard_aborted(g)) {
        *g.abort_flag = 1u;
        return false;
      }
      if (guard_expired(g, t0)) {
        guard_fail(g, site);
        return false;
      }
    }
  }
}

// Bounded wait that backs off between polls: for roles that wait a long time
// off the critical path (a loader waiting for the next unit), so that their
// polling does not take issue slots from the compute warps of the same SM
// sub-partition.
__device__ FA_WAIT_LINKAGE bool mbar_wait_backoff(uint64_t* bar, uint32_t parity, CtaGuard g, uint32_t site) {
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    __nanosleep(200);
    if ((it & 15u) == 0u) {
      if (guard_aborted(g)) {
        *g.abort_flag = 1u;
        return false;
      }
      if (guard_expired(g, t0)) {
        guard_fail(g, site);
        return false;
      }
    }
  }
}

__device__ FA_WAIT_LINKAGE bool mbar_wait_slow(uint64_t* bar, uint32_t parity, CtaGuard g, uint32_t site) {
  return mbar_poll(bar, parity, g, site);
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const CtaGuard& g,
                                          uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, g, site);
}

// Bounded wait that ignores the abort flag: used while unwinding, to let
// copies and MMAs already in flight land before shared memory / TMEM is freed.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > 100000000ull) return;  // 100 ms
  }
}

// Register reallocation between warpgroups (all four warps of a warpgroup
// execute the same instruction).  The counts must fit the registers the block
// was launched with; the launcher checks that before every launch.
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Tensors are viewed by TMA as 4-D {d, N, H, B} (any element strides, d
// contiguous): a tile of head bh is addressed by (x, row, h, b) with
// h = bh % H, b = bh / H, computed once per work unit.
struct HeadCoord {
  int h, b;
};
__device__ __forceinline__ HeadCoord head_coord(int bh, int H) { return HeadCoord{bh % H, bh / H}; }

// 4-D tile load of head `hc` into shared memory, completing bytes on `bar`.
__device__ __forceinline__ void tma_load_hd(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            HeadCoord hc) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(hc.h), "r"(hc.b)
      : "memory");
}

// Bring a 4-D tile of head `hc` into L2 ahead of its load.
__device__ __forceinline__ void tma_prefetch_l2_hd(const CUtensorMap* map, int x, int y, HeadCoord hc) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(hc.h), "r"(hc.b)
               : "memory");
}

// Work stealing (cluster launch control): ask the scheduler for a CTA of this
// grid that has not started yet; if it grants one, that CTA never launches and
// its work falls to the caller.  The 16-byte response lands at `resp` (16-byte
// aligned shared memory) and completes 16 transaction bytes on `bar`.  After a
// refusal no further request may be made.
__device__ __forceinline__ void clc_try_cancel(void* resp, uint64_t* bar) {
  asm volatile("clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];" ::"r"(
                   smem_u32(resp)),
               "r"(smem_u32(bar))
               : "memory");
}

// The granted CTA's x index, or -1 when the request was refused.
__device__ __forceinline__ int clc_decode(const void* resp) {
  uint32_t got, x;
  asm volatile(
      "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
      "mov.u32 %1, 0;\n\t"
      "ld.shared.b128 r, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
      : "=r"(got), "=r"(x)
      : "r"(smem_u32(resp))
      : "memory");
  return got ? static_cast<int>(x) : -1;
}

// 3-D tile store from shared memory (rows outside the tensor are clipped).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* smem_src, int x, int y,
                                             int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}

// 4-D tile store of head `hc` from shared memory (rows outside the tensor are clipped).
__device__ __forceinline__ void tma_store_hd(const CUtensorMap* map, const void* smem_src, int x, int y,
                                             HeadCoord hc) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(hc.h), "r"(hc.b)
               : "memory");
}

__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void tma_store_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until at most one bulk store group is still reading shared memory.
__device__ __forceinline__ void tma_store_wait_read_but_one() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make generic-proxy shared-memory writes visible to the async proxy (TMA store).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, fences
// ---------------------------------------------------------------------------

// Executed by one full warp.  Writes the TMEM base address to *smem_dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// tcgen05.mma kind::f16 (bf16 A/B, fp32 accumulate in TMEM), issued in
// warp-converged form: all 32 lanes execute the instruction with the same
// (warp-uniform) operands and one elected lane issues it.  Keeping the whole
// MMA warp converged lets the compiler hold descriptors and TMEM addresses in
// uniform registers, which is what the tensor-core instructions read.
// SS form: D(tmem) (+)= A(smem) * B(smem); TS form: A from TMEM.
__device__ __forceinline__ void tc_mma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// SS form issued only where `issue` is non-zero: the condition joins the
// elected lane's predicate, so a loop whose trip count is a run-time value
// (the head dim's 16-column steps) stays straight-line code.
__device__ __forceinline__ void tc_mma_ss_w_if(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate, uint32_t issue) {
  asm volatile(
      "{\n\t.reg .pred e, p, q;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.and.b32 q, %5, 0, e;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue)
      : "memory");
}

__device__ __forceinline__ void tc_mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// TS form issued only where `issue` is non-zero (see tc_mma_ss_w_if).
__device__ __forceinline__ void tc_mma_ts_w_if(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate, uint32_t issue) {
  asm volatile(
      "{\n\t.reg .pred e, p, q;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.and.b32 q, %5, 0, e;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by the
// issuing lane has completed.
__device__ __forceinline__ void tc_commit_w(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Bounded wait by a whole warp (every lane polls: measured faster than one
// polling lane, whose divergence costs more than the shared polls); every
// lane returns lane 0's verdict.
__device__ __forceinline__ bool mbar_wait_w(uint64_t* bar, uint32_t parity, const CtaGuard& g, uint32_t site) {
  const bool ok = mbar_wait(bar, parity, g, site);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// The polling loop of mbar_wait_either_w (out of line, like mbar_wait_slow).
__device__ FA_WAIT_LINKAGE int mbar_wait_either_slow(uint64_t* a, uint32_t pa, uint64_t* b, uint32_t pb, CtaGuard g,
                                                  uint32_t site) {
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, pa)) return 0;
    if (mbar_try_wait(b, pb)) return 1;
    if ((it & 63u) == 0u) {
      if (guard_aborted(g)) {
        *g.abort_flag = 1u;
        return -1;
      }
      if (guard_expired(g, t0)) {
        guard_fail(g, site);
        return -1;
      }
    }
  }
}

// Bounded wait, by a whole warp, for whichever of two barrier phases completes
// first: 0 for `a`, 1 for `b`, -1 if the CTA is aborting or the limit passed.
__device__ __forceinline__ int mbar_wait_either_w(uint64_t* a, uint32_t pa, uint64_t* b, uint32_t pb,
                                                  const CtaGuard& g, uint32_t site) {
  int which = -1;
  if ((threadIdx.x & 31) == 0) {
    if (mbar_try_wait(a, pa)) which = 0;
    else if (mbar_try_wait(b, pb)) which = 1;
    else which = mbar_wait_either_slow(a, pa, b, pb, g, site);
  }
  return __shfl_sync(0xffffffffu, which, 0);
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15 A major (1 = MN), 16 B major (1 = MN), 17-22 N>>3, 24-28 M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
//   bits 0-13 start address >> 4, 16-29 leading byte offset >> 4,
//   32-45 stride byte offset >> 4, 46-47 = 1 (tcgen05 descriptor),
//   49-51 base offset (0: atoms are 1024-byte aligned), 61-63 layout (2 = SW128).
// K-major operand: rows of 128 bytes, 8-row groups `sbo` apart, lbo unused.
// MN-major operand: 64-element MN blocks `lbo` apart, 8-row K groups `sbo` apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// ---------------------------------------------------------------------------
// TMEM <-> registers (32 lanes x 32-bit, one lane per thread)
// ---------------------------------------------------------------------------

#define FA_R8(r, o) "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), \
                    "=r"(r[o + 4]), "=r"(r[o + 5]), "=r"(r[o + 6]), "=r"(r[o + 7])
#define FA_W8(r, o) "r"(r[o + 0]), "r"(r[o + 1]), "r"(r[o + 2]), "r"(r[o + 3]), \
                    "r"(r[o + 4]), "r"(r[o + 5]), "r"(r[o + 6]), "r"(r[o + 7])
#define FA_T8(r, o) "+r"(r[o + 0]), "+r"(r[o + 1]), "+r"(r[o + 2]), "+r"(r[o + 3]), \
                    "+r"(r[o + 4]), "+r"(r[o + 5]), "+r"(r[o + 6]), "+r"(r[o + 7])

// Issue a load of 32 consecutive columns; results are valid only after
// tmem_ld_wait / tmem_ld_fence on the same registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : FA_R8(r, 0), FA_R8(r, 8), FA_R8(r, 16), FA_R8(r, 24)
      : "r"(taddr));
}

// Wait for all outstanding TMEM loads of this thread; the "+r" operands pin
// the loaded registers so no use of them is scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : FA_T8(r, 0), FA_T8(r, 8), FA_T8(r, 16), FA_T8(r, 24)::"memory");
}

// Further register groups loaded before the same wait: order after it.
__device__ __forceinline__ void tmem_ld_fence(uint32_t (&r)[32]) {
  asm volatile("" : FA_T8(r, 0), FA_T8(r, 8), FA_T8(r, 16), FA_T8(r, 24)::"memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      FA_W8(r, 0), FA_W8(r, 8), FA_W8(r, 16), FA_W8(r, 24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      FA_W8(r, 0), FA_W8(r, 8)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Work order
// ---------------------------------------------------------------------------

// CTA -> (head bh, work rank) for grids of BH heads x n_tiles tiles.  Heads
// are taken in bands of `band`; inside a band all rank-0 tiles come first,
// then rank 1, ...  Callers map rank 0 to their heaviest (causal) tile, so
// the last CTAs to start are the light ones, while the heads in flight stay
// few enough for their K/V (or Q/dO) to remain in L2.
__device__ __forceinline__ void banded_order(int cta, int n_tiles, int BH, int band, int& bh, int& rank) {
  const int per_band = band * n_tiles;
  const int b = cta / per_band;
  const int bh0 = b * band;
  const int width = min(band, BH - bh0);
  const int r = cta - b * per_band;
  rank = r / width;
  bh = bh0 + r % width;
}

// ---------------------------------------------------------------------------
// Dropout masks: Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel
// random numbers: as easy as 1, 2, 3", SC 2011) on a 4 x 4 (query, key) block
// per call: counter (key / 4, query / 4, head, offset), output word
// (query mod 4), byte (key mod 4) is the element's uniform byte; kept when the
// byte is at least the threshold t.
// ---------------------------------------------------------------------------

// Philox4x32-10 on counter (c0, c1, c2, c3); the round keys come from the
// kernel parameters (DropArgs::rk0/rk1), so each round is two widening
// multiplies and two three-way xors.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               const DropArgs& d) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c0;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ d.rk0[r];
    const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ d.rk1[r];
    c1 = static_cast<uint32_t>(p1);
    c3 = static_cast<uint32_t>(p0);
    c0 = n0;
    c2 = n2;
  }
  return make_uint4(c0, c1, c2, c3);
}

// Keep test of four uniform bytes at once, in byte-MSB form: bit 8b+7 of the
// result is set where byte b >= t; the other bits are don't-care.  SWAR
// compare (Hacker's Delight, multibyte arithmetic): z = (x | 0x80..) -
// (t & 0x7f..) cannot borrow across bytes and has a byte's MSB set where its
// low 7 bits are >= those of t; the MSBs of x and t then decide: x >= t is
// x_msb | z_msb when t < 128 and x_msb & z_msb otherwise, i.e. the majority
// of (x, z, maj) with maj = t < 128 ? ~0 : 0.
__device__ __forceinline__ uint32_t keep_msb4(uint32_t x, const DropArgs& d) {
  const uint32_t z = (x | 0x80808080u) - d.tlo4;
  return (x & z) | ((x | z) & d.maj);
}

// 0xFFFF in the half of a bf16x2 whose element is kept: elements b, b+1
// (b = 0 or 2) of a byte-MSB keep word (prmt replicating the bytes' sign bits).
__device__ __forceinline__ uint32_t keep_mask_pair(uint32_t ge, int b) {
  uint32_t m;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(m) : "r"(ge), "r"(b == 0 ? 0x9988u : 0xBBAAu));
  return m;
}

// All ones where element b (0..3) of a byte-MSB keep word is kept, else 0.
__device__ __forceinline__ uint32_t keep_mask_one(uint32_t ge, int b) {
  uint32_t m;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(m) : "r"(ge), "r"(0x1111u * (8u | static_cast<uint32_t>(b))));
  return m;
}

// Instruction descriptor for kind::f8f6f4 with e4m3 A and B (format 0), fp32
// D, both operands K-major: bits 4-5 D format (1 = f32), 7-9 A format, 10-12
// B format, 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_e4m3(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D (+)= A * B with A from TMEM (four e4m3 values per 32-bit column, K
// packed along the columns of each lane) and B from shared memory.
__device__ __forceinline__ void tc_mma_f8_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc_e4m3(128, 128)), "r"(accumulate)
      : "memory");
}

// D (+)= A * B, e4m3 operands from shared memory; converged warp, one elected lane.
__device__ __forceinline__ void tc_mma_f8_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc_e4m3(128, 128)), "r"(accumulate)
      : "memory");
}

// Two fp32 values to e4m3 (round to nearest even, saturating), lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return e4m3x2(a, b) | (e4m3x2(c, d) << 16);
}

// (M o dP) for columns c, c + 1 of keep words ge: dP where kept, else 0.
__device__ __forceinline__ float2 keep_pair_f(float2 v, const uint32_t* ge, int c) {
  return make_float2(__uint_as_float(__float_as_uint(v.x) & keep_mask_one(ge[c / 4], c % 4)),
                     __uint_as_float(__float_as_uint(v.y) & keep_mask_one(ge[c / 4], (c + 1) % 4)));
}

// Quad exchange: lane s of each quad holds y[k] = its word for lane (s + k)
// mod 4; returns z[m] = lane m's word for lane s.  Rotations are selects on
// the lane's position (branch-free); three shuffles.
__device__ __forceinline__ void quad_exchange(const uint32_t (&x)[4], uint32_t (&z)[4]) {
  const int lane = threadIdx.x & 31, s = lane & 3, qb = lane & ~3;
  // y[k] = x[(s + k) mod 4]: rotate left by s
  uint32_t y[4];
  {
    const bool r1 = s & 1, r2 = s & 2;
    uint32_t a0 = r1 ? x[1] : x[0], a1 = r1 ? x[2] : x[1], a2 = r1 ? x[3] : x[2], a3 = r1 ? x[0] : x[3];
    y[0] = r2 ? a2 : a0;
    y[1] = r2 ? a3 : a1;
    y[2] = r2 ? a0 : a2;
    y[3] = r2 ? a1 : a3;
  }
  // step k: receive from lane (s - k) mod 4 its y[k], which is meant for lane s
  uint32_t r[4];
  r[0] = y[0];
#pragma unroll
  for (int k = 1; k < 4; ++k) r[k] = __shfl_sync(0xffffffffu, y[k], qb + ((s - k) & 3));
  // z[m] = r[(s - m) mod 4]: with r'[j] = r[-j mod 4], z[m] = r'[(m - s) mod 4]
  const uint32_t q0 = r[0], q1 = r[3], q2 = r[2], q3 = r[1];
  const bool r1 = s & 1, r2 = s & 2;
  const uint32_t b0 = r1 ? q3 : q0, b1 = r1 ? q0 : q1, b2 = r1 ? q1 : q2, b3 = r1 ? q2 : q3;
  z[0] = r2 ? b2 : b0;
  z[1] = r2 ? b3 : b1;
  z[2] = r2 ? b0 : b2;
  z[3] = r2 ? b1 : b3;
}

// Keep words of query row i against keys j0 .. j0 + 16G - 1 (j0 a multiple of
// 16), for warps whose lanes hold consecutive rows: ge[c / 4] has element c's
// keep bit at bit 8 (c mod 4) + 7 (byte-MSB form).  Lane s of a quad draws the
// 4 x 4 blocks of keys j0 + 16g + 4s .. +3 for the quad's rows (all G calls
// first, independent chains), then the quad swaps words.
template <int G>
__device__ __forceinline__ void dropout_rows(const DropArgs& d, int bh, int i, int j0, uint32_t (&ge)[4 * G]) {
  const int s = threadIdx.x & 3;
  uint4 x[G];
#pragma unroll
  for (int g = 0; g < G; ++g)
    x[g] = philox4x32_10(static_cast<uint32_t>(j0 >> 2) + 4 * g + s, static_cast<uint32_t>(i >> 2),
                         static_cast<uint32_t>(bh), d.offset, d);
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint32_t w[4] = {keep_msb4(x[g].x, d), keep_msb4(x[g].y, d), keep_msb4(x[g].z, d),
                           keep_msb4(x[g].w, d)};
    uint32_t z[4];
    quad_exchange(w, z);   // word w of lane m = row 4q + w, keys 16g + 4m ..
#pragma unroll
    for (int m = 0; m < 4; ++m) ge[4 * g + m] = z[m];
  }
}

// Four byte-MSB keep words in one register: word k's MSBs moved to bit 7 - k
// of each byte (unpack_keep4 shifts them back; other bits are don't-care).
__device__ __forceinline__ uint32_t pack_keep4(uint32_t a, uint32_t b, uint32_t c, uint32_t e) {
  uint32_t r = a & 0x80808080u;
  r |= (b >> 1) & 0x40404040u;
  r |= (c >> 2) & 0x20202020u;
  r |= (e >> 3) & 0x10101010u;
  return r;
}
__device__ __forceinline__ uint32_t unpack_keep4(uint32_t r, int k) { return r << k; }

// Keep words of key j against queries i0 .. i0 + 16G - 1 (i0 a multiple of
// 16), for warps whose lanes hold consecutive keys: ge[c / 4] has the keep bit
// of query i0 + c at bit 8 (c mod 4) + 7.  Lane s of a quad draws the blocks
// of queries i0 + 16g + 4s .. +3 for the quad's keys, transposes its 4 x 4
// bytes (word w byte b -> word b byte w) and the quad swaps words.
template <int G>
__device__ __forceinline__ void dropout_cols(const DropArgs& d, int bh, int j, int i0, uint32_t (&ge)[4 * G]) {
  const int s = threadIdx.x & 3;
  uint4 x[G];
#pragma unroll
  for (int g = 0; g < G; ++g)
    x[g] = philox4x32_10(static_cast<uint32_t>(j >> 2), static_cast<uint32_t>(i0 >> 2) + 4 * g + s,
                         static_cast<uint32_t>(bh), d.offset, d);
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint32_t a = keep_msb4(x[g].x, d), b = keep_msb4(x[g].y, d), c = keep_msb4(x[g].z, d),
                   e = keep_msb4(x[g].w, d);
    const uint32_t lo01 = __byte_perm(a, b, 0x5140), hi01 = __byte_perm(a, b, 0x7362);
    const uint32_t lo23 = __byte_perm(c, e, 0x5140), hi23 = __byte_perm(c, e, 0x7362);
    const uint32_t w[4] = {__byte_perm(lo01, lo23, 0x5410), __byte_perm(lo01, lo23, 0x7632),
                           __byte_perm(hi01, hi23, 0x5410), __byte_perm(hi01, hi23, 0x7632)};
    uint32_t z[4];
    quad_exchange(w, z);   // word b of lane m = key 4(j/4) + b, queries 16g + 4m ..
#pragma unroll
    for (int m = 0; m < 4; ++m) ge[4 * g + m] = z[m];
  }
}

// ---------------------------------------------------------------------------
// Small numeric helpers
// ---------------------------------------------------------------------------

// 2^x on the special-function unit (approximate, flush-to-zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 16-byte shared-memory load (not volatile: the compiler may hoist it).
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

}  // namespace fa
