// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tensor loads, tcgen05 (TMEM allocation, MMA, commit, loads/stores) and the
// shared-memory / instruction descriptors the MMA takes.
//
// Descriptor formats follow the public PTX ISA description of tcgen05
// (shared-memory matrix descriptor, instruction descriptor for .kind::f16).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {

// ----------------------------------------------------------------- status
// Device-wide status word. Kernels OR bits into it when a bounded wait gives
// up (or when the dynamic shared memory they were given is not 1024-byte
// aligned, which the swizzled layouts need); the host reads it through
// fa_device_status().
enum : uint32_t { kStatusTimeout = 1u, kStatusSmemMisaligned = 2u };

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool elect_one_sync() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .b32 r;\n .reg .pred p;\n"
      " elect.sync r|p, 0xffffffff;\n"
      " selp.b32 %0, 1, 0, p;\n}"
      : "=r"(pred));
  return pred != 0;
}

// -------------------------------------------- programmatic dependent launch
// Every kernel is launched with programmatic stream serialisation: the grid
// may be scheduled while the previous grid in the stream is still finishing.
// Each thread calls grid_wait_prior() after its prologue (barrier set-up and
// TMEM allocation, which touch no global memory) and before its first global
// load or store, and before it can exit; it returns once the previous grid has
// completed and its writes are visible (at once without such a dependency).
// So a grid's completion still implies that of every grid before it.
// grid_release_next() then lets the next grid be scheduled on the SMs this
// one frees; it only ever waits on this grid, never the reverse.
__device__ __forceinline__ void grid_wait_prior() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_release_next() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
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

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.b32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of phase `parity` (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.b32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// A wait bound below this many cycles (a test of the give-up path) also reads
// the clock after every failed try and never suspends, so the wait gives up
// at its first miss.
constexpr uint64_t kShortWaitCycles = 1024;

// As mbar_wait below, but polling with test_wait: for the single thread that
// issues MMAs, which must notice a completed phase at once.
__device__ __forceinline__ bool mbar_wait_poll(uint32_t bar, uint32_t parity,
                                               uint64_t timeout_cycles, volatile int* abort,
                                               uint32_t* status) {
  if (mbar_test_wait(bar, parity)) return true;
  const int tries = timeout_cycles < kShortWaitCycles ? 1 : 64;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < tries; ++i)
      if (mbar_test_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (static_cast<uint64_t>(clock64() - t0) > timeout_cycles) {
      if (abort != nullptr) *abort = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// Wait for phase `parity` of `bar` to complete, giving up after
// `timeout_cycles` SM clock cycles (clock64: cheap to read, unlike the global
// timer, so a waiter never misses a completion while reading the clock).
// On timeout the device status gets kStatusTimeout, `*abort` (a flag in shared
// memory, shared by the CTA) is raised, and the call returns false. Once the
// flag is up every later wait returns false at once, so all roles run to the
// common exit without blocking. `abort` may be null (a drain wait at exit that
// must not be cut short by an earlier abort).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_cycles,
                                          volatile int* abort, uint32_t* status) {
  // a bound below kShortWaitCycles tests without suspending (try_wait may hold
  // the thread until the phase completes, so such a wait would never miss)
  const bool short_bound = timeout_cycles < kShortWaitCycles;
  const int tries = short_bound ? 1 : 32;
#pragma unroll 1
  for (int i = 0; i < tries; ++i)
    if (short_bound ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < tries; ++i)
      if (short_bound ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (static_cast<uint64_t>(clock64() - t0) > timeout_cycles) {
      if (abort != nullptr) *abort = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// ------------------------------------------------------------------- fences
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load: box at coordinates (x, y, z), innermost first. x times the
// element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// L2 eviction policies for TMA loads (createpolicy): operands that many CTAs
// read again should stay in L2 (evict_last); operands read once should not
// push them out (evict_first).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 3-D tiled load with an L2 cache policy (see tma_load_3d).
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int x, int y, int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// 2-D tiled load (x innermost).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// ------------------------------------------------- cluster launch control
// Dynamic scheduling for persistent CTAs: a running CTA asks the hardware to
// cancel the launch of a CTA of its grid that has not started yet and takes
// over that CTA's work. The 16-byte response lands in shared memory at
// `resp` (16-byte aligned) and completes `bar` with 16 transaction bytes.
// Issued by one thread; not again once a response reported failure.
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint32_t bar) {
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128"
      " [%0], [%1];" ::"r"(resp), "r"(bar)
      : "memory");
}

// Decode a response: true, with the x index of the cancelled CTA, when a CTA
// was cancelled; false when the grid had none left to give.
__device__ __forceinline__ bool clc_query(uint32_t resp, int* ctaid_x) {
  uint32_t ok, x;
  asm volatile(
      "{\n .reg .b128 r;\n .reg .pred p;\n"
      " ld.shared.b128 r, [%2];\n"
      " clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n"
      " selp.u32 %0, 1, 0, p;\n"
      " clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n}"
      : "=r"(ok), "=r"(x)
      : "r"(resp)
      : "memory");
  *ctaid_x = static_cast<int>(x);
  return ok != 0;
}

// ------------------------------------------------------------------ tcgen05
// TMEM allocation: executed by one full warp. The allocated base address is
// written to the shared-memory word at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
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

// Shared-memory matrix descriptor. `swizzle`: 0 none, 2 = 128-byte swizzle,
// 4 = 64-byte, 6 = 32-byte. Byte offsets are encoded in 16-byte units.
// For K-major 128B-swizzled operands the leading offset is unused and the
// stride offset is the distance between 8-row groups (1024 bytes when rows are
// 128 bytes). For MN-major 128B-swizzled operands the leading offset is the
// distance between 64-element MN column blocks and the stride offset the
// distance between 8-row groups along K.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t swizzle) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16;
  d |= static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(swizzle & 7u) << 61;
  return d;
}

// Instruction descriptor for tcgen05.mma .kind::f16 with an fp32 accumulator.
// ab_bf16: operand type (0 = f16, 1 = bf16; A and B always share it).
// a_mn / b_mn: 1 when that operand is MN-major in shared memory.
__host__ __device__ constexpr uint32_t make_idesc_f16(uint32_t M, uint32_t N, uint32_t ab_bf16,
                                                      uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4)                 // D format: f32
         | (ab_bf16 << 7)          // A format
         | (ab_bf16 << 10)         // B format
         | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread t of the warp receives
// lane (base lane + t), columns [col, col + 16).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32"
      " [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32"
      " [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// ------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Split cluster barrier: every CTA of the cluster has started (its shared
// memory may be written by peers) once the wait returns.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Every thread of every CTA of the cluster arrives; release / acquire order
// the shared-memory writes before the barrier with the peers' reads after it.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address in CTA `rank`'s shared memory of the location at shared address
// `local` in this CTA's (the CTAs of a cluster share one layout).
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from this CTA's shared memory to a peer CTA's (addresses from peer_addr),
// completing the bytes on the peer's mbarrier `remote_bar`. The source must be
// made visible to the copy engine first (fence_proxy_async_smem by the threads
// that wrote it).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t remote_dst, uint32_t local_src,
                                                  uint32_t bytes, uint32_t remote_bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(remote_dst),
      "r"(local_src), "r"(bytes), "r"(remote_bar)
      : "memory");
}

// Arrive on an mbarrier in a peer CTA's shared memory (address from
// peer_addr) without ordering this thread's memory accesses: for a "buffer
// free" signal sent after the reads of the buffer have delivered their
// values.
__device__ __forceinline__ void mbar_arrive_peer_relaxed(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar)
               : "memory");
}

// As mbar_wait, for a barrier that peers arrive on: the acquire is at cluster
// scope, so the peers' stores announced by their arrivals are visible.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.b32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  uint64_t timeout_cycles, volatile int* abort,
                                                  uint32_t* status) {
  const int tries = timeout_cycles < kShortWaitCycles ? 1 : 32;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < tries; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (static_cast<uint64_t>(clock64() - t0) > timeout_cycles) {
      if (abort != nullptr) *abort = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// ------------------------------------------------------- register split
// Move registers between the warpgroups of a CTA. Every warp of a warpgroup
// executes the same call, and the code a warpgroup runs afterwards sits in the
// branch that made the call (the compiler allocates that branch against the
// new count). An increase waits until decreases elsewhere have returned enough
// registers, so the new counts must fit the launch's total (threads x
// registers per thread at launch); the host checks that before launching.
template <uint32_t N>
__device__ __forceinline__ void regs_release() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N) : "memory");
}
template <uint32_t N>
__device__ __forceinline__ void regs_claim() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ numerics
// 2^x with the hardware approximation (ex2.approx, flushes subnormals).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two-lane fp32 arithmetic (one instruction for both lanes; sm_100 family).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Pack two floats into one 32-bit word of 16-bit values (lo in bits 0-15).
template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kBF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// As pack2, with the bf16 rounding done on the integer pipe: round to nearest
// with ties away from zero by one integer add on each fp32 bit pattern, then a
// byte permute that keeps the two high halves (three integer instructions per
// pair instead of one cvt.rn.bf16x2.f32, which runs at 16 instructions per
// clock per SM on GB300, half the rate of ex2.approx). It differs from cvt.rn
// only on exact ties (low 16 bits 0x8000). fp16 keeps the conversion. Used
// for dS in the dQ kernel (4% faster there); in the forward and dK/dV softmax
// loops the extra integer instructions cost more than they save (measured).
template <bool kBF16>
__device__ __forceinline__ uint32_t pack2_rna(float lo, float hi) {
  if constexpr (kBF16) {
    return __byte_perm(__float_as_uint(lo) + 0x8000u, __float_as_uint(hi) + 0x8000u, 0x7632);
  } else {
    return pack2<false>(lo, hi);
  }
}

template <bool kBF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (kBF16) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w);
    return __bfloat1622float2(v);
  } else {
    __half2 v = *reinterpret_cast<__half2*>(&w);
    return __half22float2(v);
  }
}

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row` inside a tile
// laid out with 128-byte rows and the 128-byte swizzle (the layout TMA writes
// with CU_TENSOR_MAP_SWIZZLE_128B when the tile base is 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace fa
