// Thin inline-PTX wrappers for the sm_103a data path: mbarriers with bounded
// waits, TMA (tensor and plain bulk copies), and tcgen05 (TMEM allocation,
// MMA issue/commit, TMEM loads).  Written from the public PTX ISA.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace logra {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the thread sleep (up to ~20 us) until the phase
// completes instead of spinning, so waiting warps do not take issue slots
// from the warps doing work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; give up after `limit`
// clock64 ticks.  Returns false on timeout (the caller records the status).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity)) {
    if (static_cast<unsigned long long>(clock64() - t0) > limit) return false;
  }
  return true;
}

// Bounded wait with a CTA-wide abort flag: keeps waiting in slices while no
// other role has given up; past the limit it records LOGRA_ERR_TIMEOUT and
// raises the flag so every role leaves its loop.
template <class SH>
__device__ __forceinline__ bool wait_or_abort(SH* sh, uint64_t* bar, uint32_t parity, unsigned long long limit,
                                              Control* ctl) {
  const unsigned long long slice = limit / 8 + 1;
  unsigned long long spent = 0;
  while (!mbar_wait(bar, parity, slice)) {
    if (*reinterpret_cast<volatile int*>(&sh->abort)) return false;
    spent += slice;
    if (spent >= limit) {
      record_status(ctl, LOGRA_ERR_TIMEOUT);
      *reinterpret_cast<volatile int*>(&sh->abort) = 1;
      return false;
    }
  }
  return true;
}

// Warp-uniform version: lane 0 waits, the outcome is broadcast, and every lane
// then observes the completed phase itself (acquire) before touching the data.
template <class SH>
__device__ __forceinline__ bool warp_wait(SH* sh, uint64_t* bar, uint32_t parity, unsigned long long limit,
                                          Control* ctl) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_or_abort(sh, bar, parity, limit, ctl) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)mbar_try_wait(bar, parity);
  return ok != 0;
}

// try_wait with cluster-scope acquire: for a barrier whose phase is completed by
// another CTA of the cluster (a peer's copies or arrivals), so that what the
// peer wrote before its arrival is visible to this thread.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, unsigned long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (static_cast<unsigned long long>(clock64() - t0) > limit) return false;
  }
  return true;
}

// wait_or_abort for a barrier completed by the peer CTA of a pair.
template <class SH>
__device__ __forceinline__ bool wait_or_abort_cluster(SH* sh, uint64_t* bar, uint32_t parity,
                                                      unsigned long long limit, Control* ctl) {
  const unsigned long long slice = limit / 8 + 1;
  unsigned long long spent = 0;
  while (!mbar_wait_cluster(bar, parity, slice)) {
    if (*reinterpret_cast<volatile int*>(&sh->abort)) return false;
    spent += slice;
    if (spent >= limit) {
      record_status(ctl, LOGRA_ERR_TIMEOUT);
      *reinterpret_cast<volatile int*>(&sh->abort) = 1;
      return false;
    }
  }
  return true;
}

// try_wait with cluster-scope acquire and no suspend-time hint.
__device__ __forceinline__ bool mbar_try_wait_cluster_nohint(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// wait_or_abort / wait_or_abort_cluster for the single MMA-issuing thread:
// no suspend-time hint, so the thread resumes the moment its operands land
// (a suspended issuer wakes late and leaves the tensor pipe idle).  Bounded
// like the others: past `limit` it records LOGRA_ERR_TIMEOUT and raises the
// CTA's abort flag; it also gives up once another role has raised it.
template <bool kCluster, class SH>
__device__ __forceinline__ bool spin_or_abort(SH* sh, uint64_t* bar, uint32_t parity, unsigned long long limit,
                                              Control* ctl) {
  auto ready = [&]() { return kCluster ? mbar_try_wait_cluster_nohint(bar, parity) : mbar_try_wait(bar, parity); };
  if (ready()) return true;
  const long long t0 = clock64();
  for (unsigned n = 1;; ++n) {
    if (ready()) return true;
    if ((n & 63u) == 0) {
      if (*reinterpret_cast<volatile int*>(&sh->abort)) return false;
      if (static_cast<unsigned long long>(clock64() - t0) > limit) {
        record_status(ctl, LOGRA_ERR_TIMEOUT);
        *reinterpret_cast<volatile int*>(&sh->abort) = 1;
        return false;
      }
    }
  }
}

// warp_wait for a barrier completed from the other CTA of a pair.
// warp_wait with a polling lane 0 (spin_or_abort): for producers whose
// stage must be refilled the moment the MMAs release it (a suspended thread
// wakes late).  Every lane then observes the phase itself.
template <class SH>
__device__ __forceinline__ bool warp_spin_wait(SH* sh, uint64_t* bar, uint32_t parity, unsigned long long limit,
                                               Control* ctl) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = spin_or_abort<false>(sh, bar, parity, limit, ctl) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)mbar_try_wait(bar, parity);
  return ok != 0;
}

template <class SH>
__device__ __forceinline__ bool warp_wait_cluster(SH* sh, uint64_t* bar, uint32_t parity, unsigned long long limit,
                                                  Control* ctl) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_or_abort_cluster(sh, bar, parity, limit, ctl) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)mbar_try_wait_cluster(bar, parity);
  return ok != 0;
}

// ----------------------------------------------------------------- rings of shared-memory stages
struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++stage == n) { stage = 0; phase ^= 1u; }
  }
};

// Copies still in flight land before the CTA exits: wait (bounded) for the
// last phase issued on every stage of a ring; phases already consumed pass.
__device__ __forceinline__ void drain_ring(uint64_t* full, const Ring& rg, int n, unsigned long long limit) {
  for (int s = 0; s < n; ++s) mbar_wait(&full[s], (s < rg.stage) ? rg.phase : (rg.phase ^ 1u), limit);
}

// In a CTA pair the leader's MMA commits arrive on the other CTA's empty
// barriers from another SM, asynchronously: before a CTA releases its shared
// memory, its producer waits (bounded) until every stage it filled has been
// released, so that no such arrival is still on its way.  After an abort the
// consumer may never release a stage: each wait then gives up after a
// sixty-fourth of the limit.
template <class SH>
__device__ __forceinline__ void drain_empties(SH* sh, uint64_t* empty, const Ring& rg, int n,
                                              unsigned long long limit) {
  for (int s = 0; s < n; ++s) {
    const bool aborted = *reinterpret_cast<volatile int*>(&sh->abort) != 0;
    mbar_wait(&empty[s], (s < rg.stage) ? rg.phase : (rg.phase ^ 1u), aborted ? limit / 64 + 1 : limit);
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// ----------------------------------------------------------------- clusters (CTA pairs)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// shared::cluster address of the object at shared::cta address `saddr` in cluster CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Plain 32-bit store into another CTA's shared memory (shared::cluster address).
__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// Every thread of both CTAs; release/acquire at cluster scope.  The barrier is
// warp-aligned, so the warp first reconverges (its lanes may have split in
// lane-0 role loops).
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier of another CTA of the cluster (shared::cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// ----------------------------------------------------------------- fences
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Tensor copy into this CTA's shared memory whose completion is signalled on an
// mbarrier of either CTA of a pair (bar: shared::cluster address, e.g. the
// leader's barrier from mapa_shared).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int32_t x,
                                                 int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// Plain (non-tensor) bulk copy global -> shared; dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_addr(src))
               : "memory");
}

// global[box at (x, y)] += shared tile (fp32 add, performed by the TMA unit / L2).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* src, int32_t x, int32_t y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_addr(src))
               : "memory");
}

// Plain bulk copy shared -> global (bulk group); both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
               "r"(smem_addr(src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Programmatic dependent launch.  The pipeline kernels are launched with
// programmatic stream serialization, which lets the hardware have the next
// kernel ready while the current one finishes.  None of them signals its
// dependents early (griddepcontrol.launch_dependents): that signal only
// promises the dependents the writes made before it, and measured with the
// signal at kernel start the dependents read unfinished results.  So the
// dependent is released when this grid completes, and grid_dependency_wait(),
// called by every CTA after its prologue and before any global access, waits
// for that completion and its memory.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor (tcgen05 format): start address, leading /
// stride byte offsets (16-byte units), the fixed version bits 46..48 = 0b001,
// base offset 0 (atoms aligned to the swizzle repeat) and the swizzle mode.
enum Swizzle : uint32_t { kSwNone = 0, kSw128 = 2, kSw64 = 4, kSw32 = 6 };

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes, Swizzle sw) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(sw) << 61;
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A and B, fp32 accumulator.
// a_mn / b_mn: operand is MN-major (1) or K-major (0).
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4)            // D format: f32
         | (1u << 7)          // A format: bf16
         | (1u << 10)         // B format: bf16
         | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Block barrier for kernels whose warps split into lane-0 role loops: bar.sync
// is warp-aligned, so a warp whose lanes arrive apart is undefined behaviour
// (lanes that come early can be released before the rest of the block).  The
// warp reconverges first.
__device__ __forceinline__ void cta_sync() {
  __syncwarp();
  __syncthreads();
}

// TMEM allocation: one full warp executes these (.sync.aligned: reconverged first).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  __syncwarp();
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  __syncwarp();
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  __syncwarp();
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// CTA-pair forms (cta_group::2): one warp of EACH CTA of the pair executes the
// allocation, relinquish and deallocation together; both receive the same
// column address.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  __syncwarp();
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  __syncwarp();
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  __syncwarp();
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T across a CTA pair, issued by one thread of the
// even CTA: M = 256 rows, rows 0..127 of A (and of D) in the even CTA, 128..255
// in the odd one; B's N columns split in halves, the first in the even CTA.
// Both CTAs' operands sit at the same shared-memory offsets.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at `bar`'s offset in every CTA of `mask` when all
// pair MMAs issued so far by this thread complete.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(mask)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one thread issues.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives
// lane (quadrant*32 + t), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Eight +-1 bf16 values from eight sign bits (bit set -> -1.0), as four
// packed bf16x2 words: bit 2q goes to the low half of word q, bit 2q+1 to the
// high half.  0x3F80 is bf16(+1); the sign bit is bit 15 of each half.
__device__ __forceinline__ uint4 signs8_to_bf16(uint32_t byte) {
  uint4 o;
  o.x = ((((byte >> 0) & 3u) * 0x40008000u) & 0x80008000u) | 0x3F803F80u;
  o.y = ((((byte >> 2) & 3u) * 0x40008000u) & 0x80008000u) | 0x3F803F80u;
  o.z = ((((byte >> 4) & 3u) * 0x40008000u) & 0x80008000u) | 0x3F803F80u;
  o.w = ((((byte >> 6) & 3u) * 0x40008000u) & 0x80008000u) | 0x3F803F80u;
  return o;
}

}  // namespace tc

// Host: encode a 2-D tiled tensor map (driver entry point fetched through the
// runtime, so the library needs no link-time dependency on libcuda).
int make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint32_t elem_bytes, uint64_t inner,
                 uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swizzle);

}  // namespace logra
