// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tensor copies, and the tcgen05 tensor-core / tensor-memory instructions.
//
// Everything here follows the public PTX ISA (mbarrier, cp.async.bulk.tensor,
// tcgen05.*).  No CUTLASS or CuTe is used.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace rg {

// Device status bits (mirrors RG_DEV_* in rg.h).
constexpr unsigned int kDevBadOffsets = 0x1u;
constexpr unsigned int kDevTimeout = 0x2u;
constexpr unsigned int kDevLaunchConfig = 0x4u;
constexpr unsigned int kDevBounds = 0x8u;  // debug-bounds builds only

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- mbarrier

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

// Non-suspending test with cluster-scope acquire: for barriers that the peer
// CTA of a pair arrives on (remote arrives, multicast MMA commits).  A thread
// suspended in try_wait is not woken promptly by such arrivals, so these
// barriers are polled.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// ----------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its shared::cluster address (own or peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Shared state of the bounded waits of one CTA.
struct WaitGuard {
  unsigned int* status;   // device status word
  uint64_t limit_ns;      // bound on a single wait
  volatile int* abort;    // shared-memory flag: some wait of this CTA ran out
};

// Slow path of mbar_wait: spin with a deadline.
static __device__ __noinline__ bool mbar_wait_slow(const WaitGuard& g, uint32_t bar, uint32_t parity,
                                                   bool cluster_scope) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*g.abort) return false;
    if (globaltimer_ns() - t0 > g.limit_ns) {
      atomicOr(g.status, kDevTimeout);
      *g.abort = 1;
      return false;
    }
  }
}

// Wait until the phase of `bar` with the given parity has completed.  Returns
// false, without waiting further, once any wait of the CTA has run out; the
// wait that runs out sets kDevTimeout and raises the CTA's abort flag.
__device__ __forceinline__ bool mbar_wait(const WaitGuard& g, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(g, bar, parity, false);
}

// mbar_wait for barriers that the peer CTA of a CTA pair also arrives on.
__device__ __forceinline__ bool mbar_wait_cl(const WaitGuard& g, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  return mbar_wait_slow(g, bar, parity, true);
}

// Bounded wait, by one thread, for a barrier the peer CTA of a pair arrives
// on, sleeping `sleep_ns` between polls: for a wait whose latency hardly
// matters (an epilogue that waits out a whole mainloop), so that its polling
// does not compete with the copies and MMAs for the shared-memory pipe.
static __device__ __noinline__ bool mbar_wait_cl_sleep(const WaitGuard& g, uint32_t bar, uint32_t parity,
                                                       uint32_t sleep_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    __nanosleep(sleep_ns);
    if (*g.abort) return false;
    if (globaltimer_ns() - t0 > g.limit_ns) {
      atomicOr(g.status, kDevTimeout);
      *g.abort = 1;
      return false;
    }
  }
}

// Warp-wide bounded wait for an accumulator barrier, for epilogue warps that
// wait out a whole mainloop: with CTA pairs lane 0 alone polls, sleeping 1 us
// between polls, and the warp takes its answer (measured: the pair kernels'
// epilogues polling flat out cost the weight-gradient GEMM ~1%); single CTAs
// use the suspending wait.
template <int CG, uint32_t SLEEP_NS = 1000>
__device__ __forceinline__ bool warp_wait_acc(const WaitGuard& g, uint32_t bar, uint32_t parity) {
  if constexpr (CG == 1) {
    return __all_sync(0xffffffffu, mbar_wait(g, bar, parity)) != 0;
  } else {
    bool got = true;
    if ((threadIdx.x & 31) == 0) got = mbar_wait_cl_sleep(g, bar, parity, SLEEP_NS);
    return __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
  }
}

// Bound on each wait of the drain at a kernel's end.  Copies and MMAs that
// were issued always complete (their operands exist), within microseconds;
// the bound only keeps the wait finite, and it does not depend on the
// caller's pipeline-wait limit, which may be much shorter.
constexpr uint64_t kDrainLimitNs = 200000000ull;

// Bounded wait used while draining: ignores the abort flag.
static __device__ __noinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kDrainLimitNs) return false;
  }
}

// Count `bytes` of the current phase's expected transaction bytes as arrived
// (bytes of a copy that was armed for but will never be issued).
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// complete_tx on a barrier given by its shared::cluster address (own or peer
// CTA of a pair): the debug-bounds build counts the bytes of a copy it
// refused to issue, so that the stage completes without them.
__device__ __forceinline__ void mbar_complete_tx_cluster(uint32_t cluster_addr, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.relaxed.cluster.shared::cluster.b64 [%0], %1;" ::"r"(cluster_addr), "r"(bytes)
               : "memory");
}

// 32-bit load from the shared memory of a CTA of the cluster (address from mapa_shared).
__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}

// What each of a CTA's two producer threads last issued into each stage of
// its ring: the iteration of the (tile, block) walk (-1: nothing yet; stage
// = it % S, phase = it / S) and the bytes of this CTA's own copies.  Written
// by the producer that issues, read once at the kernel's end by the drain.
template <int S>
struct IssueLog {
  int it[2][S];
  uint32_t bytes[2][S];
};

template <int S>
__device__ __forceinline__ void issue_log_init(IssueLog<S>* log, uint32_t pid) {
#pragma unroll
  for (int s = 0; s < S; ++s) {
    log->it[pid][s] = -1;
    log->bytes[pid][s] = 0;
  }
}

// The drain at the end of a kernel, run by one thread of the CTA whose stage
// barriers receive every copy (the issuing CTA of a pair), once no producer
// of either CTA issues any more: wait, per stage, until the last phase that
// either CTA copied into has completed, so that no copy still writes into a
// CTA's shared memory when it exits.  `peer` is the shared::cluster address
// of the other CTA's log (0 for a single CTA).  The two CTAs of a pair are at
// most one phase apart on a stage (a stage is refilled only after both halves
// of its previous phase landed and were consumed), and a phase that only one
// of them reached is settled on the barrier: the peer's missing copy is
// counted as arrived (complete_tx), or the issuing CTA's missing arrival is
// made with the peer's bytes (arrive.expect_tx).  Waits are bounded by
// kDrainLimitNs.  After a normal run every last phase is already complete.
template <int S>
__device__ void drain_stages(uint32_t full_bar0, const IssueLog<S>* own, uint32_t peer) {
#pragma unroll 1
  for (int s = 0; s < S; ++s) {
    const int k0 = own->it[0][s] >= own->it[1][s] ? 0 : 1;
    const int i0 = own->it[k0][s];
    int i1 = -1;
    uint32_t b1 = 0;
    if (peer != 0) {
      const uint32_t f = peer + 4u * s;  // &log->it[0][s] in the peer CTA
      const int a = static_cast<int>(ld_shared_cluster_u32(f));
      const int b = static_cast<int>(ld_shared_cluster_u32(f + 4u * S));
      const int k1 = a >= b ? 0 : 1;
      i1 = k1 == 0 ? a : b;
      b1 = ld_shared_cluster_u32(peer + 8u * S + 4u * (k1 * S + s));
    } else {
      i1 = i0;
    }
    const uint32_t bar = full_bar0 + 8u * s;
    int last = i0;
    if (i0 > i1) {
      mbar_complete_tx(bar, own->bytes[k0][s]);  // the peer's half (same size as ours) never comes
    } else if (i1 > i0) {
      mbar_arrive_expect_tx(bar, b1);  // the peer copied into a phase we never armed
      last = i1;
    }
    if (last >= 0) mbar_wait_drain(bar, static_cast<uint32_t>(last / S) & 1u);
  }
}

// --------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Loads whose completion is signalled on an mbarrier of either CTA of a pair
// (`bar` is a shared::cluster address): the peer CTA's copies complete their
// bytes directly on the issuing CTA's barrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                                 int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                                 int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

template <int CG>
__device__ __forceinline__ void tma_load_2d_cg(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                               int32_t c0, int32_t c1) {
  if constexpr (CG == 1) tma_load_2d(dst, m, bar, c0, c1);
  else tma_load_2d_pair(dst, m, bar, c0, c1);
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t c0,
                                                 int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// The pair load with an L2 cache-policy hint (createpolicy).
__device__ __forceinline__ void tma_load_4d_pair_hint(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t c0,
                                                      int32_t c1, int32_t c2, int32_t c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
      : "memory");
}

// L2 eviction-priority policy for data that later copies will read again.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

template <int CG>
__device__ __forceinline__ void tma_load_4d_cg(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t c0,
                                               int32_t c1, int32_t c2, int32_t c3) {
  if constexpr (CG == 1) tma_load_4d(dst, m, bar, c0, c1, c2, c3);
  else tma_load_4d_pair(dst, m, bar, c0, c1, c2, c3);
}

template <int CG>
__device__ __forceinline__ void tma_load_3d_cg(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                               int32_t c0, int32_t c1, int32_t c2) {
  if constexpr (CG == 1) tma_load_3d(dst, m, bar, c0, c1, c2);
  else tma_load_3d_pair(dst, m, bar, c0, c1, c2);
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, uint32_t src, int32_t c0,
                                             int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int32_t c0,
                                             int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// dW[box] += smem box, fp32 add performed by the TMA unit (round to nearest).
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* m, uint32_t src, int32_t c0,
                                                  int32_t c1, int32_t c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// L2 eviction-priority policy for a stream written once and not read again
// by the kernel (createpolicy, fraction 1.0 of the accesses).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// The same stores / reduce-adds with an L2 cache-policy hint.
__device__ __forceinline__ void tma_store_3d_hint(const CUtensorMap* m, uint32_t src, int32_t c0,
                                                  int32_t c1, int32_t c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_reduce_add_3d_hint(const CUtensorMap* m, uint32_t src, int32_t c0,
                                                       int32_t c1, int32_t c2, uint64_t policy) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group.L2::cache_hint"
      " [%0, {%2, %3, %4}], [%1], %5;" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N committed bulk groups of this thread are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tensor cores).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's global-memory accesses through the async proxy (TMA
// stores, reduce-adds) with its accesses through the generic proxy.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Hand-over flags between CTAs (the K-grouped GEMM's chunk mode): a flag in
// global memory counts the chunks whose writes are complete.  publish raises
// it with release semantics at GPU scope; flag_wait_ge polls it with acquire
// semantics, bounded like every other wait (running out sets kDevTimeout and
// the CTA's abort flag), then orders the caller's later async-proxy accesses
// after what it saw.
__device__ __forceinline__ void flag_publish(int* flag, int value) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(flag), "r"(value) : "memory");
}

__device__ __forceinline__ bool flag_wait_ge(const WaitGuard& g, const int* flag, int target) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v >= target) {
      fence_proxy_async_global();
      return true;
    }
    __nanosleep(100);
    if (*g.abort) return false;
    if (globaltimer_ns() - t0 > g.limit_ns) {
      atomicOr(g.status, kDevTimeout);
      *g.abort = 1;
      return false;
    }
  }
}

// ----------------------------------------------------------------- tcgen05

// Tensor-memory allocation.  With CG == 2 one warp of each CTA of the pair
// executes these together; the allocation has the same address in both.
template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_relinquish() {
  if constexpr (CG == 1)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate.  With
// CG == 2 the issuing (even) CTA drives both tensor cores of the pair: A rows
// [0,M/2) and B rows [0,N/2) come from its shared memory, the other halves
// from the same addresses in the peer CTA, and each CTA's tensor memory
// receives its M/2 rows of D.
template <int CG>
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  if constexpr (CG == 1)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` (same shared-memory offset in every CTA of the pair
// when CG == 2) when all tcgen05 operations issued so far by this thread have
// completed.
template <int CG>
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  if constexpr (CG == 1) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
  } else {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
  }
}

// Arrive only on this CTA's `bar` (CG == 2: commit from the issuing CTA to
// its own barrier).
template <int CG>
__device__ __forceinline__ void umma_commit_local(uint32_t bar) {
  if constexpr (CG == 1) {
    umma_commit<1>(bar);
  } else {
    const uint16_t mask = 0x1;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
  }
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives
// columns [col, col+32) of TMEM lane (lane_base + t).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile whose
// swizzle atoms (8 rows x 128 B) start on 1024-byte boundaries.
//   K-major operand : rows of 128 B hold 64 consecutive K elements; LBO is not
//                     used; SBO = distance between groups of 8 rows (1024).
//   MN-major operand: rows of 128 B hold 64 consecutive M/N elements, one row
//                     per K index; LBO = distance between 64-wide M/N blocks,
//                     SBO = distance between groups of 8 K rows (1024).
// Bits: [0,14) start>>4, [16,30) LBO>>4, [32,46) SBO>>4, [46,48) = 1,
// [49,52) base offset 0, [61,64) swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A/B and fp32 D.
// Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B format
// (1 = bf16), 15 A major (1 = MN), 16 B major (1 = MN), [17,23) N>>3,
// [24,29) M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------- block-scaled (MXFP8)

// Untiled bulk copy global -> shared, completion on an mbarrier of this CTA.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// D[tmem] (+)= (A * 2^sfA) (B * 2^sfB)^T with FP8 E4M3 A/B in shared memory,
// fp32 accumulate, one E8M0 scale per row and 32-element K block read from
// tensor memory (kind::mxf8f6f4, block size 32, K = 32 per instruction).
// With CG == 2 the issuing CTA drives both tensor cores of the pair as in
// umma_bf16; the scale addresses name the same columns in both CTAs.
template <int CG = 1>
__device__ __forceinline__ void umma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  if constexpr (CG == 1)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Copy a 32-row x 16-byte matrix from shared memory (descriptor) into tensor
// memory columns [taddr, taddr+4) of lanes 0..31, replicated into each of the
// four 32-lane quarters.  With CG == 2, issued by the issuing CTA of a pair,
// each CTA's matrix (same shared-memory address) goes to its own tensor memory.
template <int CG = 1>
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
  else
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Descriptor of a contiguous, unswizzled K-major shared-memory matrix whose
// rows are 16 bytes: 8-row core matrices 128 bytes apart (SBO), one core
// matrix along K (LBO unused).  Layout type 0 (no swizzle).
__device__ __forceinline__ uint64_t sdesc_plain16(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(128u >> 4) << 16) |
         (static_cast<uint64_t>(128u >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor of tcgen05.mma kind::mxf8f6f4 with E4M3 A and B,
// E8M0 scales and fp32 D.  Bits: [4,6) B scale-factor id (byte of the scale
// word), [7,10) A format (0 = E4M3), [10,13) B format (0 = E4M3), 15 A major,
// 16 B major (1 = MN), [17,23) N>>3, 23 scale format (1 = E8M0), [24,29) M>>4,
// [29,31) A scale-factor id.
__host__ __device__ constexpr uint32_t idesc_mxf8_f32(int M, int N, bool a_mn, bool b_mn, uint32_t sf_id) {
  return ((sf_id & 3u) << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) |
         ((sf_id & 3u) << 29);
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_f32_bits, uint32_t hi_f32_bits) {
  __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo_f32_bits), __uint_as_float(hi_f32_bits));
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace rg
