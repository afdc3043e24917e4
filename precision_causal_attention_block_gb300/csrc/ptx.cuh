// Thin inline-PTX wrappers for the Blackwell (sm_100 family) features the
// kernels use: mbarriers, TMA tensor loads, tcgen05 tensor-memory allocation,
// MMA, loads/stores and commits.  Written from the public PTX ISA.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace flamia {

// Every bounded wait gives up after this many nanoseconds and reports
// FLAMIA_DEV_TIMEOUT instead of spinning forever.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ORs an error bit into the caller's device status word (if one was given).
__device__ __forceinline__ void report(int* status, int bit) {
  if (status != nullptr) atomicOr(status, bit);
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

// One bounded wait: the thread waits in the hardware for the phase to
// complete, up to a system-dependent time limit.  (An explicit suspend-time
// hint measured slower: the woken warps resumed later.)
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

// Non-blocking: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if
// the wait ran past kWaitTimeoutNs (the caller records the timeout and
// unwinds without touching the barrier again).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
  }
}

// A bounded wait taken by every lane of a converged warp, with one outcome
// for the whole warp (so the lanes never take different paths).
__device__ __forceinline__ bool mbar_wait_w(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// mbar_wait that also gives up once *abort is set (another role of the CTA
// unwinding).  The flag is read only while the phase is incomplete, so a
// completed phase costs one try_wait and no extra shared-memory round trip.
__device__ __forceinline__ bool mbar_wait_ab(uint32_t bar, uint32_t parity,
                                             const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
  }
}

// The same for every lane of a converged warp, with one outcome for the warp.
__device__ __forceinline__ bool mbar_wait_w_ab(uint32_t bar, uint32_t parity,
                                               const volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait_ab(bar, parity, abort));
}

// ------------------------------------------------------------------ item ring
// Work items claimed by a CTA's producer thread are handed to the CTA's other
// roles in claim order through a small shared-memory ring: item number n
// (0, 1, ...) sits in slot n % kSlots.  `full` completes once per put, `empty`
// once every consumer role has taken the slot.

template <int kSlots>
struct ItemRing {
  int idx[kSlots];
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
};

template <int kSlots>
__device__ __forceinline__ void ring_init(ItemRing<kSlots>& r, int consumers) {
  for (int i = 0; i < kSlots; ++i) {
    mbar_init(smem_u32(&r.full[i]), 1);
    mbar_init(smem_u32(&r.empty[i]), consumers);
  }
}

// Producer: publishes item number n; false if the slot never came free.
template <int kSlots>
__device__ __forceinline__ bool ring_put(ItemRing<kSlots>& r, int n, int v) {
  const int s = n % kSlots;
  if (n >= kSlots && !mbar_wait(smem_u32(&r.empty[s]), ((n / kSlots) - 1) & 1)) return false;
  *static_cast<volatile int*>(&r.idx[s]) = v;
  mbar_arrive(smem_u32(&r.full[s]));  // release: the value is visible to the waiters
  return true;
}

// Consumer role: item number n, or -1 if it never arrived.  With `release`
// the caller's arrive frees the slot (one arrive per consumer role).
template <int kSlots>
__device__ __forceinline__ int ring_get(ItemRing<kSlots>& r, int n, bool release) {
  const int s = n % kSlots;
  if (!mbar_wait(smem_u32(&r.full[s]), (n / kSlots) & 1)) return -1;
  const int v = *static_cast<volatile int*>(&r.idx[s]);
  if (release) mbar_arrive(smem_u32(&r.empty[s]));
  return v;
}

// The next unclaimed item of a launch (items are claimed in list order, so
// the longest go first wherever a CTA is free).
__device__ __forceinline__ int claim_item(int* counter) { return atomicAdd(counter, 1); }

// Work distribution of the persistent kernels over their head-major,
// cost-sorted item list.  Dynamic: the next unclaimed item (claim_item; the
// review page, sec. 3.4 "Work scheduling", does this with cluster launch
// control).  Static: the snake over the list, CTA b taking item r P + b in
// even rounds r and r P + P - 1 - b in odd ones (P CTAs), which deals the
// longest items out first and needs no atomics.
enum : int { kSchedDynamic = 0, kSchedRule = 1, kSchedStatic = 2 };

// Static or dynamic for this launch.  kSchedRule is the pages' rule (review
// page, sec. 4.3 as the summary reports it): dynamic for causal calls; for
// non-causal calls only when the longest document is at least 4x the average
// length.  The list's first item carries the longest document's cost in
// 128-token tiles.
__device__ __forceinline__ bool static_schedule(int sched, int causal, const int4* items,
                                                int n_items, int T, int ndocs) {
  if (sched != kSchedRule) return sched == kSchedStatic;
  if (causal || n_items <= 0) return false;
  const long long longest = 128ll * items[0].w;
  return longest * ndocs < 4ll * T;
}

struct Claims {
  int* counter;
  bool snake;
  int round = 0;
  __device__ __forceinline__ int next() {
    if (!snake) return claim_item(counter);
    const int P = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
    const int idx = round * P + ((round & 1) ? P - 1 - b : b);
    ++round;
    return idx;
  }
};

// Called by thread 0 of every CTA as its last action: the last CTA of the
// launch resets the claim counter and the exit count for the next launch.
__device__ __forceinline__ void finish_claims(int* counter, int* exited) {
  __threadfence();
  if (atomicAdd(exited, 1) == static_cast<int>(gridDim.x) - 1) {
    atomicExch(counter, 0);
    atomicExch(exited, 0);
  }
}

// ------------------------------------------------------------------ proxies

// Generic-proxy writes to shared memory become visible to the async proxy
// (TMA, tensor core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Brings a 3-D box of a tensor into L2 (a hint: nothing waits for it).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1,
                                                   int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Bulk tensor reduce-add of a shared-memory box into global memory (the
// element type and the add come from the tensor map); completion is tracked
// with bulk async-groups of the issuing thread.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int c0,
                                                  int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until the sources of all committed bulk groups have been read.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until the sources of all but the most recent committed bulk group
// have been read.
__device__ __forceinline__ void bulk_wait_group_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Waits until all committed bulk groups have completed.
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------- ordered dQ turns
// In the deterministic dQ mode every 64- or 128-query tile of the float32 dQ
// accumulator has a turn counter (zeroed before the backward): a key tile
// adds its partial once the counter reads its turn (the number of key tiles
// that add before it) and raises the counter by one once its reduce-adds
// have completed, so the float32 sums run in one fixed order whatever the
// CTAs' timing.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Bounded wait until *turn >= want (false after kWaitTimeoutNs); the async
// proxy's later reduce-adds are ordered after the acquiring load.
__device__ __forceinline__ bool wait_turn(const int* turn, int want) {
  bool ok = ld_acquire_gpu(turn) >= want;
  if (!ok) {
    const uint64_t t0 = globaltimer_ns();
    while (!(ok = ld_acquire_gpu(turn) >= want)) {
      if (globaltimer_ns() - t0 > kWaitTimeoutNs) break;
      __nanosleep(32);
    }
  }
  fence_proxy_async_global();
  return ok;
}
// Passes the turn on: the caller's bulk reduce-adds have completed
// (bulk_wait_group0), their writes are ordered before the releasing add.
__device__ __forceinline__ void pass_turn(int* turn) {
  fence_proxy_async_global();
  asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(turn) : "memory");
}

// ------------------------------------------------------------------ tcgen05

// Allocation and deallocation are warp-wide (.sync.aligned): call from one
// full warp.  The allocated column base is written to shared memory.
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

// The mbarrier receives one arrive once every tcgen05 operation issued so far
// by this thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// ---------------------------------------------------------- warp-wide issue
// The *_w forms are executed by all 32 lanes of a converged warp (so their
// operands are warp-uniform values) and issued by one lane that elect.sync
// picks; the other lanes skip the instruction.

__device__ __forceinline__ void tc_commit_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

__device__ __forceinline__ void mma_f8_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_mxf8_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

__device__ __forceinline__ void mma_mxf8_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                              uint32_t idesc, uint32_t sfa_tmem,
                                              uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %2, %3, "
      "[%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

__device__ __forceinline__ void mma_nvf4_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// D (+)= A * B, E4M3 x E4M3 -> F32, operands in shared memory.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (+)= (A * 2^sfa) * (B * 2^sfb), E4M3 operands with one E8M0 scale per 32
// elements of the contraction, scale factors in tensor memory.
__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// D (+)= A * B, E4M3 x E4M3 -> F32, A read from tensor memory (row m in lane
// m, four elements per 32-bit column along K), B in shared memory.
__device__ __forceinline__ void mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same product with A read from tensor memory: row m of A in lane m,
// four E4M3 elements per 32-bit column along K (a_tmem = the first column of
// this K step's 32 elements).
__device__ __forceinline__ void mma_mxf8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// D (+)= (A * sfa) * (B * sfb), packed E2M1 operands with one E4M3 scale per
// 16 elements of the contraction (K = 64 per instruction).
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// 32 lanes x 32 columns of 32-bit words: thread t of the warp receives lane
// (base lane + t), columns [col, col + 32).
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

// As tmem_ld32 for float32 columns, also returning the largest of the 32
// values each thread receives (tcgen05.ld.red, sm_103: the row maximum comes
// with the load instead of 32 comparisons).
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, %32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=f"(mx)
      : "r"(taddr));
}

// 32 lanes x 8 columns: thread t receives lane (base + t), columns [col, col + 8).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
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

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ CTA pairs
// A cluster of two CTAs whose tensor cores run one product together
// (tcgen05 .cta_group::2): the even CTA's thread issues every product of the
// pair; A and D are split by M (each CTA its own 128 rows, in its own shared
// and tensor memory at the same addresses), B by N (each CTA supplies half of
// the columns from the same shared-memory address).  Every tcgen05
// instruction of such a kernel carries .cta_group::2.

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs; orders the CTAs' earlier memory operations
// (release) before the other's later ones (acquire).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// The shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive on an mbarrier of either CTA of the cluster (a shared::cluster
// address), releasing this thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cl_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_bar)
               : "memory");
}

// Bulk copy from this CTA's shared memory to the shared memory of a CTA of the
// cluster (async proxy); the destination CTA's mbarrier (a shared::cluster
// address) receives the bytes as transaction count.  Both addresses and the
// size are multiples of 16 bytes.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cl, uint32_t src, uint32_t bytes,
                                                     uint32_t bar_cl) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst_cl),
      "r"(src), "r"(bytes), "r"(bar_cl)
      : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cl_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cl_addr), "r"(v) : "memory");
}

// As mbar_wait, acquiring at cluster scope (for phases completed by the other
// CTA of the pair or by a pair product's commit).
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
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
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait_cl(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
  }
}
__device__ __forceinline__ bool mbar_wait_cl_w(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait_cl(bar, parity));
}

// One warp of each CTA of the pair allocates (and later frees) the same
// columns in both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// The mbarrier at this shared-memory offset in each CTA of `mask` receives
// one arrive once the pair products issued so far by this thread complete.
__device__ __forceinline__ void tc_commit2_w(uint32_t bar, uint16_t mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;\n\t}" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void mma2_f8_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma2_mxf8_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// ------------------------------------------------------------------ descriptors

// Shared-memory matrix descriptor layouts (tcgen05 encoding, bits 61..63).
enum : uint32_t {
  kLayoutNone = 0,
  kLayoutSW128 = 2,
  kLayoutSW64 = 4,
  kLayoutSW32 = 6,
};

// start address, leading- and stride-dimension byte offsets, layout.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version of the tcgen05 family
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

// Instruction descriptor, kind::f8f6f4: E4M3 x E4M3 -> F32.
__host__ __device__ constexpr uint32_t idesc_f8(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4)                                   // accumulator F32
         | (0u << 7) | (0u << 10)                    // A, B = E4M3
         | (static_cast<uint32_t>(a_mn_major) << 15) | (static_cast<uint32_t>(b_mn_major) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, kind::mxf8f6f4 block-scaled with E8M0 scales.
// sf ids pick the byte of the 32-bit scale word (one byte per 32-wide K block).
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int a_mn_major, int b_mn_major,
                                                 int sfa_id, int sfb_id) {
  return (static_cast<uint32_t>(sfb_id & 3) << 4) | (0u << 7) | (0u << 10) |
         (static_cast<uint32_t>(a_mn_major) << 15) | (static_cast<uint32_t>(b_mn_major) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23)  // scales are UE8M0
         | (static_cast<uint32_t>(M >> 4) << 24) | (static_cast<uint32_t>(sfa_id & 3) << 29);
}

// Instruction descriptor, kind::mxf4nvf4: E2M1 x E2M1, E4M3 scales, K-major.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10)  // A, B = E2M1
         | (static_cast<uint32_t>(N >> 3) << 17) | (0u << 23)  // scales are UE4M3
         | (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------ numerics

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Exact 2^k as a float for k in [-126, 127].
__device__ __forceinline__ float exp2i(int k) { return __int_as_float((k + 127) << 23); }

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two floats -> two E4M3 codes (round to nearest even, saturating);
// lo goes to bits 0..7, hi to bits 8..15.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four floats -> four E4M3 codes in one word (a in bits 0..7, ..., d in 24..31),
// each rounded to nearest even and saturated as cvt_e4m3x2 does.
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// Two E4M3 codes (bits 0..7 and 8..15) -> two exact floats.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(codes)));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// Two E2M1 codes (bits 0..3 and 4..7) -> two exact floats.
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t codes) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.u8.u32 t, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2)
      : "r"(codes & 0xFFu));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// Two floats -> two E2M1 codes (round to nearest even, saturating): lo in
// bits 0..3, hi in bits 4..7.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Round-up block exponent: smallest e with amax <= 448 * 2^e, clamped to
// [-127, 127]; amax == 0 (or below the normal range) gives -127.
// Unnormalised Sylvester-Hadamard butterflies (x H_d) on a row of N * P
// floats spread over P consecutive lanes: lane `part` (0 .. P-1 inside its
// aligned group of P lanes) holds elements [N part, N part + N).  Strides 1 ..
// N/2 run inside the lane, then N, 2N, .. N P / 2 across lanes (partner part ^
// stride / N), in increasing order; in each pair (i, i + s) the new values are
// (x_i + x_{i+s}, x_i - x_{i+s}) in float32.  All lanes of the warp must call
// it together when P > 1.
template <int N, int P>
__device__ __forceinline__ void fwht_row(float (&v)[N], int part) {
#pragma unroll
  for (int s = 1; s < N; s <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      if ((i & s) == 0) {
        const float a = v[i], b = v[i + s];
        v[i] = a + b;
        v[i + s] = a - b;
      }
    }
  }
#pragma unroll
  for (int dist = 1; dist < P; dist <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], dist);
      v[i] = (part & dist) ? o - v[i] : v[i] + o;
    }
  }
}

__device__ __forceinline__ int roundup_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int E = static_cast<int>((b >> 23) & 0xFF) - 127;
  const uint32_t man = b & 0x7FFFFFu;
  // amax = (1 + f) 2^E; (1 + f) <= 1.75  <=>  man <= 0.75 * 2^23
  int e = (man <= 0x600000u) ? E - 8 : E - 7;
  if (((b >> 23) & 0xFF) == 0) e = -127;
  return max(-127, min(127, e));
}

}  // namespace flamia
