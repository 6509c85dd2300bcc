// Inline-PTX building blocks for sm_103a: mbarriers, TMA tile loads,
// 5th-generation tensor core (tcgen05) MMA, tensor memory (TMEM) allocation
// and loads/stores, and the shared-memory / instruction descriptors they take.
//
// Everything here is written from the public PTX ISA description of these
// instructions; no library code is involved.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {

// ---------------------------------------------------------------- status --
// Bits of the device status word a kernel sets when it gives up a wait.
enum : int {
  kStatusWaitTimeout = 1,   // an mbarrier wait ran past its cycle limit
  kStatusBadLaunch = 2,     // a kernel found its launch configuration inconsistent
};

// A healthy wait finishes in microseconds; this bound (about two seconds at
// the GB300's SM clock) only ends a wait that would otherwise never finish.
// The waits of the abort path (for copies and MMAs already issued, which
// always complete) use kDrainLimitCycles instead. A wait-limit test build of
// the library (FA_WAIT_TEST) shortens the first bound only and makes each
// kernel's MMA issuer start by waiting for a barrier phase that nothing
// completes, so that its bounded wait runs out and the kernel takes the
// abort path and reports kStatusWaitTimeout.
#ifdef FA_WAIT_LIMIT_CYCLES
constexpr long long kWaitLimitCycles = FA_WAIT_LIMIT_CYCLES;
#else
constexpr long long kWaitLimitCycles = 4000000000LL;
#endif
constexpr long long kDrainLimitCycles = 4000000000LL;

// ----------------------------------------------------------------- trace --
// Timeline tracing, compiled in only when FA_TRACE is defined (a separate
// trace build of the library). The first kTraceCtas CTAs of a launch record,
// per role, up to kTraceSlots events as (clock64 << 8 | event id) into the
// buffer passed in the kernel parameters. Without FA_TRACE the tracer is
// empty and costs nothing.
constexpr int kTraceCtas = 4, kTraceRoles = 4, kTraceSlots = 2048;
#ifdef FA_TRACE
struct Tracer {
  unsigned long long* base = nullptr;
  int n = 0;
  __device__ Tracer(unsigned long long* buf, int role) {
    if (buf && blockIdx.x < kTraceCtas)
      base = buf + (static_cast<size_t>(blockIdx.x) * kTraceRoles + role) * kTraceSlots;
  }
  __device__ void operator()(int ev) {
    if (base && n < kTraceSlots)
      base[n++] = (static_cast<unsigned long long>(clock64()) << 8) | static_cast<unsigned>(ev);
  }
};
// Every CTA of a launch (up to kTraceSpanCtas) also fills kTraceSpanSlots
// entries after the timeline region: its SM, its work count and clock64
// readings at points the kernel chooses (start, first step, last step, end).
constexpr int kTraceSpanCtas = 16384, kTraceSpanSlots = 8;
__device__ __forceinline__ void trace_span(unsigned long long* buf, int slot, unsigned long long v) {
  if (buf && blockIdx.x < kTraceSpanCtas)
    buf[static_cast<size_t>(kTraceCtas) * kTraceRoles * kTraceSlots +
        static_cast<size_t>(blockIdx.x) * kTraceSpanSlots + slot] = v;
}
__device__ __forceinline__ unsigned smid() {
  unsigned r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}
#else
struct Tracer {
  __device__ Tracer(unsigned long long*, int) {}
  __device__ void operator()(int) {}
};
__device__ __forceinline__ void trace_span(unsigned long long*, int, unsigned long long) {}
__device__ __forceinline__ unsigned smid() { return 0; }
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// -------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Test for completion of the phase with the given parity (the thread may be
// held briefly inside the instruction). No suspend-time hint is passed: on the
// critical paths here, a suspended waiter wakes later than a polling one.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed. Gives up (and
// returns false) when `abort_flag` is set by another warp or after
// kWaitLimitCycles; in the latter case it raises the abort flag and the
// status word so that every other role of the CTA stops too.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > kWaitLimitCycles) {
        *abort_flag = 1;
        atomicOr(status, kStatusWaitTimeout);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 3-D tiled load of one box into shared memory; completion is reported to
// `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Plain (untiled) bulk copy global -> shared; addresses 16-byte aligned and
// size a multiple of 16 bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// 3-D tiled reduce-add of one shared-memory box into global memory (fp32
// add for an fp32 map). Completion is tracked per issuing thread through
// bulk groups: commit after issuing, then wait until the source has been read
// (before overwriting it) or the whole group has completed.
__device__ __forceinline__ void tma_reduce_add_3d(const void* tmap, uint32_t src, int c0, int c1,
                                                  int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(tmap)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// 3-D tiled store of one box from shared memory; completion through the
// bulk group (rows past the tensor's extent are not written).
__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(tmap)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Prefetch one box of a tiled tensor into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_3d(const void* tmap, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Make generic-proxy writes to shared memory visible to the async proxy
// (TMA and the tensor core read shared memory through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------------------------- tcgen05 --
// Tensor memory: 128 lanes x 512 columns of 32 bit per SM. An address is
// (lane << 16) | column. Warp w of a CTA may only touch lanes
// 32*(w%4) .. 32*(w%4)+31.

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
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

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem], kind::f16 (bf16 or fp16 in, fp32 accumulate).
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16. A holds two 16-bit elements per
// 32-bit column, K-major (lane = row of A).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// ---- whole-product issue ---------------------------------------------------
// One 128 x N x (16*STEPS) product as STEPS tcgen05.mma instructions in a
// single asm block, with the per-step operand descriptors formed by adding
// compile-time offsets to descriptors computed once. A single issuing thread
// otherwise spends more time building descriptors than the tensor core spends
// on an N = 128 step, and the tensor core sits idle in between.
//
// Offset of K-step ks in descriptor units (16 bytes), 128-byte swizzle:
//   K-major:  32 bytes per step inside a 128-byte row, then the next
//             64-element chunk (kChunkBytes further) every 4 steps;
//   MN-major: 16 rows of 128 bytes (2048 bytes) per step.
template <bool kKMajor, int kChunkBytes>
__host__ __device__ constexpr int desc_step(int ks) {
  return kKMajor ? ((ks % 4) * 2 + (ks / 4) * (kChunkBytes >> 4)) : ks * 128;
}

// D (+)= A B, both operands in shared memory. `accumulate` applies to the
// first step; the remaining steps always accumulate.
template <int STEPS, bool kAK, int kAC, bool kBK, int kBC>
__device__ __forceinline__ void mma_ss_product(uint32_t d_tmem, uint64_t a0, uint64_t b0,
                                               uint32_t idesc, uint32_t accumulate) {
  static_assert(STEPS == 4 || STEPS == 8, "4 or 8 K-steps");
  if constexpr (STEPS == 4) {
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b64 a, b;\n\t"
        "setp.ne.b32 pf, %4, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
        "add.s64 a, %1, %5;\n\tadd.s64 b, %2, %6;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
        "add.s64 a, %1, %7;\n\tadd.s64 b, %2, %8;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
        "add.s64 a, %1, %9;\n\tadd.s64 b, %2, %10;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t}" ::"r"(d_tmem),
        "l"(a0), "l"(b0), "r"(idesc), "r"(accumulate),
        "n"(desc_step<kAK, kAC>(1)), "n"(desc_step<kBK, kBC>(1)),
        "n"(desc_step<kAK, kAC>(2)), "n"(desc_step<kBK, kBC>(2)),
        "n"(desc_step<kAK, kAC>(3)), "n"(desc_step<kBK, kBC>(3))
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b64 a, b;\n\t"
        "setp.ne.b32 pf, %4, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
        "add.s64 a, %1, %5;\n\tadd.s64 b, %2, %6;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
        "add.s64 a, %1, %7;\n\tadd.s64 b, %2, %8;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
        "add.s64 a, %1, %9;\n\tadd.s64 b, %2, %10;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
        "add.s64 a, %1, %11;\n\tadd.s64 b, %2, %12;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
        "add.s64 a, %1, %13;\n\tadd.s64 b, %2, %14;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
        "add.s64 a, %1, %15;\n\tadd.s64 b, %2, %16;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
        "add.s64 a, %1, %17;\n\tadd.s64 b, %2, %18;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t}" ::"r"(d_tmem),
        "l"(a0), "l"(b0), "r"(idesc), "r"(accumulate),
        "n"(desc_step<kAK, kAC>(1)), "n"(desc_step<kBK, kBC>(1)),
        "n"(desc_step<kAK, kAC>(2)), "n"(desc_step<kBK, kBC>(2)),
        "n"(desc_step<kAK, kAC>(3)), "n"(desc_step<kBK, kBC>(3)),
        "n"(desc_step<kAK, kAC>(4)), "n"(desc_step<kBK, kBC>(4)),
        "n"(desc_step<kAK, kAC>(5)), "n"(desc_step<kBK, kBC>(5)),
        "n"(desc_step<kAK, kAC>(6)), "n"(desc_step<kBK, kBC>(6)),
        "n"(desc_step<kAK, kAC>(7)), "n"(desc_step<kBK, kBC>(7))
        : "memory");
  }
}

// D (+)= A B with A in tensor memory (16-bit, two per column: step ks reads
// columns a_tmem + 8*ks, plus kAJump further for steps 4-7) and B in shared
// memory; 8 K-steps.
template <bool kBK, int kBC, int kAJump = 0>
__device__ __forceinline__ void mma_ts_product8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 b;\n\t.reg .b32 a;\n\t"
      "setp.ne.b32 pf, %4, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pf;\n\t"
      "add.s32 a, %1, 8;\n\tadd.s64 b, %2, %5;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, pt;\n\t"
      "add.s32 a, %1, 16;\n\tadd.s64 b, %2, %6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, pt;\n\t"
      "add.s32 a, %1, 24;\n\tadd.s64 b, %2, %7;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, pt;\n\t"
      "add.s32 a, %1, %12;\n\tadd.s64 b, %2, %8;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, pt;\n\t"
      "add.s32 a, %1, %13;\n\tadd.s64 b, %2, %9;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, pt;\n\t"
      "add.s32 a, %1, %14;\n\tadd.s64 b, %2, %10;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, pt;\n\t"
      "add.s32 a, %1, %15;\n\tadd.s64 b, %2, %11;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, pt;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b0), "r"(idesc), "r"(accumulate),
      "n"(desc_step<kBK, kBC>(1)), "n"(desc_step<kBK, kBC>(2)), "n"(desc_step<kBK, kBC>(3)),
      "n"(desc_step<kBK, kBC>(4)), "n"(desc_step<kBK, kBC>(5)), "n"(desc_step<kBK, kBC>(6)),
      "n"(desc_step<kBK, kBC>(7)), "n"(32 + kAJump), "n"(40 + kAJump), "n"(48 + kAJump),
      "n"(56 + kAJump)
      : "memory");
}

// ---- CTA pairs (cta_group::2) ----------------------------------------------
// A cluster of two CTAs on two SMs shares one instruction stream: the even
// CTA of the pair (the leader) issues M = 256 products whose D rows 0-127 land
// in its own tensor memory and rows 128-255 in its peer's, at the same column
// address; A rows come from each CTA's own shared memory (or tensor memory),
// and B's N columns are split, the first N/2 read from the leader's shared
// memory and the rest from the peer's, at the same offset. Tensor memory is
// allocated and freed jointly (one warp in each CTA), and every tcgen05
// instruction of a kernel that pairs uses the cta_group::2 form.

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of both CTAs; orders shared-memory and barrier set-up (and the
// final reads of the peer's memory) across the pair.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of another CTA of the cluster (release at cluster
// scope: this thread's prior writes and tensor-memory stores, fenced, are
// visible to the thread that observes the phase).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait for a phase that arrivals from the other CTA complete.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, int* status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > kWaitLimitCycles) {
        *abort_flag = 1;
        atomicOr(status, kStatusWaitTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Arrive once on the mbarrier at offset `bar` of every CTA in `cta_mask`
// (bit i = cluster rank i) when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// Pair forms of mma_ss_product (8 K-steps) and mma_ts_product8: M = 256 across
// the two CTAs.
template <bool kAK, int kAC, bool kBK, int kBC>
__device__ __forceinline__ void mma_pair_ss_product8(uint32_t d_tmem, uint64_t a0, uint64_t b0,
                                                     uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 a, b;\n\t"
      "setp.ne.b32 pf, %4, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, pf;\n\t"
      "add.s64 a, %1, %5;\n\tadd.s64 b, %2, %6;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, %7;\n\tadd.s64 b, %2, %8;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, %9;\n\tadd.s64 b, %2, %10;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, %11;\n\tadd.s64 b, %2, %12;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, %13;\n\tadd.s64 b, %2, %14;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, %15;\n\tadd.s64 b, %2, %16;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, %17;\n\tadd.s64 b, %2, %18;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t}" ::"r"(d_tmem),
      "l"(a0), "l"(b0), "r"(idesc), "r"(accumulate),
      "n"(desc_step<kAK, kAC>(1)), "n"(desc_step<kBK, kBC>(1)),
      "n"(desc_step<kAK, kAC>(2)), "n"(desc_step<kBK, kBC>(2)),
      "n"(desc_step<kAK, kAC>(3)), "n"(desc_step<kBK, kBC>(3)),
      "n"(desc_step<kAK, kAC>(4)), "n"(desc_step<kBK, kBC>(4)),
      "n"(desc_step<kAK, kAC>(5)), "n"(desc_step<kBK, kBC>(5)),
      "n"(desc_step<kAK, kAC>(6)), "n"(desc_step<kBK, kBC>(6)),
      "n"(desc_step<kAK, kAC>(7)), "n"(desc_step<kBK, kBC>(7))
      : "memory");
}

template <bool kBK, int kBC>
__device__ __forceinline__ void mma_pair_ts_product8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0,
                                                     uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 b;\n\t.reg .b32 a;\n\t"
      "setp.ne.b32 pf, %4, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, pf;\n\t"
      "add.s32 a, %1, 8;\n\tadd.s64 b, %2, %5;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, pt;\n\t"
      "add.s32 a, %1, 16;\n\tadd.s64 b, %2, %6;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, pt;\n\t"
      "add.s32 a, %1, 24;\n\tadd.s64 b, %2, %7;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, pt;\n\t"
      "add.s32 a, %1, 32;\n\tadd.s64 b, %2, %8;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, pt;\n\t"
      "add.s32 a, %1, 40;\n\tadd.s64 b, %2, %9;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, pt;\n\t"
      "add.s32 a, %1, 48;\n\tadd.s64 b, %2, %10;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, pt;\n\t"
      "add.s32 a, %1, 56;\n\tadd.s64 b, %2, %11;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [a], b, %3, pt;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b0), "r"(idesc), "r"(accumulate),
      "n"(desc_step<kBK, kBC>(1)), "n"(desc_step<kBK, kBC>(2)), "n"(desc_step<kBK, kBC>(3)),
      "n"(desc_step<kBK, kBC>(4)), "n"(desc_step<kBK, kBC>(5)), "n"(desc_step<kBK, kBC>(6)),
      "n"(desc_step<kBK, kBC>(7))
      : "memory");
}

// Instruction descriptor for kind::f16 with fp32 accumulation.
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format (0 = f16,
//   1 = bf16), 15 A major, 16 B major (0 = K-major, 1 = MN-major),
//   17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool bf16, bool a_mn, bool b_mn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
//   bits 0-13 start address >> 4, 16-29 leading-dimension byte offset >> 4,
//   32-45 stride-dimension byte offset >> 4, 46-48 fixed 0b001,
//   61-63 swizzle mode (2 = 128-byte swizzle).
// K-major, 128B swizzle: rows of 128 bytes (64 16-bit elements along K),
//   8-row groups `sbo` bytes apart; the leading offset is unused.
// MN-major, 128B swizzle: 128-byte rows hold 64 elements along M/N, one row
//   per K index, 8 K rows per 1024-byte atom; `lbo` = distance between atoms
//   adjacent along M/N, `sbo` = distance between atoms adjacent along K.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives lane
// (32*(warp%4) + t), columns [col, col+32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
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

// ------------------------------------------------------------- numerics --
// Hardware base-2 exponential (MUFU ex2, approximate, flush-to-zero);
// ex2(-inf) = +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pack two fp32 values into one 32-bit word of 16-bit elements, round to
// nearest even; `lo` goes to the low half.
template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (kBf16) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  }
  return r;
}

// Inverse of pack2 (exact): bf16 -> fp32 is a 16-bit shift; fp16 uses the
// hardware conversion.
template <bool kBf16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (kBf16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  } else {
    __half2 h;
    asm("mov.b32 %0, %1;" : "=r"(*reinterpret_cast<uint32_t*>(&h)) : "r"(w));
    return __half22float2(h);
  }
}

// Packed pairs of fp32 in one 64-bit register for the sm_100-family paired
// fp32 instructions (two results per issue, each rounded as its scalar form).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three (exact, so any grouping gives the same result)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }
__device__ __forceinline__ uint32_t warp_id() { return threadIdx.x >> 5; }

// 16-byte store to a shared-memory address
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Named barrier among `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace fa
