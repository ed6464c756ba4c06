// h3q_tc_ptx.cuh -- inline-PTX wrappers for the sm_103a tensor-core path:
// mbarriers with bounded waits, TMA tile loads, TMEM allocation, tcgen05 MMA,
// commit, loads/stores and fences.
#pragma once

#include <cstdint>

namespace h3q {
namespace ptx {

// A bounded wait gives up after this much global time and reports a timeout.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// --- mbarrier -------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Single-thread bounded wait.  Returns false (and records `code` in *err) on
// timeout or when another role has already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* err, uint32_t code) {
  const uint32_t a = smem_u32(bar);
  if (mbar_test(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test(a, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitTimeoutNs) {
        atomicOr(err, code);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Warp-collective bounded wait: every lane observes the phase (acquire), and
// the give-up decision is lane 0's, broadcast, so the warp stays converged.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity,
                                               volatile int* abort_flag, uint32_t* err,
                                               uint32_t code) {
  const uint32_t a = smem_u32(bar);
  const unsigned full = 0xFFFFFFFFu;
  if (__all_sync(full, mbar_test(a, parity))) return true;
  uint64_t t0 = 0;
  if ((threadIdx.x & 31) == 0) t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (__all_sync(full, mbar_test(a, parity))) return true;
    if ((i & 255u) == 0) {
      int give_up = 0;
      if ((threadIdx.x & 31) == 0) {
        if (*abort_flag) {
          give_up = 1;
        } else if (globaltimer() - t0 > kWaitTimeoutNs) {
          atomicOr(err, code);
          *abort_flag = 1;
          give_up = 1;
        }
      }
      if (__shfl_sync(full, give_up, 0)) return false;
    }
  }
}

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Arrive on an mbarrier of any CTA of the cluster (address from mapa_shared).
// The release is at CTA scope: what the arrival publishes here is TMEM
// contents (ordered by the tcgen05 fences around the barrier) and the
// completion of this CTA's own TMA copies, not generic-memory writes, and a
// cluster-scope release costs about a microsecond per arrival.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait for a barrier that other CTAs of the cluster arrive on: the
// acquire is at cluster scope.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, uint32_t* err,
                                                  uint32_t code) {
  const uint32_t a = smem_u32(bar);
  if (mbar_test_cluster(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test_cluster(a, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitTimeoutNs) {
        atomicOr(err, code);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Store to a 64-bit word in the shared memory of any CTA of the cluster
// (address from mapa_shared).
__device__ __forceinline__ void st_cluster_u64(uint32_t cluster_addr, uint64_t v) {
  asm volatile("st.relaxed.cluster.shared::cluster.u64 [%0], %1;" ::"r"(cluster_addr), "l"(v)
               : "memory");
}

__device__ __forceinline__ void fence_acq_rel_cluster() {
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
}

// mbar_arrive_cluster with a cluster-scope release: publishes this thread's
// generic-memory writes to a waiter in another CTA (about a microsecond).
__device__ __forceinline__ void mbar_arrive_cluster_release(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// --- programmatic dependent launch ----------------------------------------------------

// Wait until the grids this one depends on have completed and their memory
// writes are visible.  Without the launch attribute this returns at once.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Let the next grid on the stream be scheduled before this one finishes (it
// still waits for this grid's completion in grid_dependency_wait).
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --- TMA ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 2-D tiled load into CTA shared memory; completion is counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, uint64_t* bar, int x,
                                            int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Untiled bulk copy of `bytes` contiguous bytes from global memory into this
// CTA's shared memory, completing that many transaction bytes on `bar`.  Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tiled load into this CTA's shared memory.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, uint64_t* bar, int x,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Elects one lane of the (converged) calling warp: 1 on that lane, 0 on the
// others; its lane id goes to *leader_lane if given.  A loop that the whole
// warp runs, with one elected lane issuing the asynchronous copies or MMAs,
// keeps its waits, addresses and descriptors warp-uniform; the same loop run
// by one lane alone was measured to lose most of its issue rate to busy warps
// on its SM sub-partition.
__device__ __forceinline__ uint32_t elect_one(uint32_t* leader_lane = nullptr) {
  uint32_t l, is;
  asm volatile("{\n.reg .pred p;\nelect.sync %0|p, 0xffffffff;\nselp.u32 %1, 1, 0, p;\n}"
               : "=r"(l), "=r"(is));
  if (leader_lane) *leader_lane = l;
  return is;
}

// --- clusters -------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// All threads of every CTA in the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// --- TMEM and tcgen05 -------------------------------------------------------------------

// Whole warp.  Writes the TMEM base address to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16, one CTA.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (base_lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
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
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// --- the CTA-pair forms (cta_group::2): TMEM is allocated in both CTAs of the
// pair at the same address, by one warp of each; an MMA issued by one thread
// of the even CTA computes M = 256 rows, 128 in each CTA's TMEM, from A in each
// CTA's TMEM and B split along N between the two CTAs' shared memory.

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void mma_f16_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` in every CTA of `mask` once the pair MMAs issued so far are done.
__device__ __forceinline__ void mma_commit_pair_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart.  The tile base is 1024-aligned.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);      // start address (>> 4)
  d |= static_cast<uint64_t>(1) << 16;                       // leading offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;               // stride offset: 8 rows
  d |= static_cast<uint64_t>(1) << 46;                       // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                       // SWIZZLE_128B
  return d;
}

// Instruction descriptor for kind::f16: FP16 A and B (both K-major), FP32 D.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n) {
  return (1u << 4)                                   // D format: F32
         | (0u << 7) | (0u << 10)                    // A, B format: F16
         | (static_cast<uint32_t>(n >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);    // M / 16
}

// INT8 x4 (one 32-bit word) -> two FP16x2 words holding the same integers,
// exactly: bias each byte to b = q + 128 (XOR 0x80), splice it under the FP16
// exponent of 1024 (0x64xx encodes 1024 + b), subtract 1152.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4)                                   // D format: F32
         | (1u << 7) | (1u << 10)                    // A, B format: BF16
         | (static_cast<uint32_t>(n >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);    // M / 16
}

// Four unsigned 8-bit codes -> four BF16 values a q + b (a and b the same in
// both halves of a2 and b2): each byte, placed under the exponent of 2^23 by a
// byte permute (selector nibbles 7, 6, 5 take the constant's upper bytes, the
// last one the code's byte), becomes the FP32 2^23 + q (exact),
// minus 2^23 (exact), one FMA (one rounding), then BF16 (round to nearest
// even).  lo holds codes 0 and 1, hi codes 2 and 3, the first in the low half.
__device__ __forceinline__ void u8x4_affine_to_bf16x4(uint32_t w, uint64_t a2, uint64_t b2,
                                                      uint32_t& lo, uint32_t& hi) {
  const uint32_t base = 0x4B000000u;                  // FP32 2^23
  uint32_t f0, f1, f2, f3;
  asm("prmt.b32 %0, %1, %2, 0x7650;" : "=r"(f0) : "r"(w), "r"(base));
  asm("prmt.b32 %0, %1, %2, 0x7651;" : "=r"(f1) : "r"(w), "r"(base));
  asm("prmt.b32 %0, %1, %2, 0x7652;" : "=r"(f2) : "r"(w), "r"(base));
  asm("prmt.b32 %0, %1, %2, 0x7653;" : "=r"(f3) : "r"(w), "r"(base));
  const uint64_t two23 = 0x4B0000004B000000ull;
  const uint64_t p01 = (uint64_t(f1) << 32) | f0, p23 = (uint64_t(f3) << 32) | f2;
  uint64_t q01, q23, r01, r23;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(q01) : "l"(p01), "l"(two23));
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(q23) : "l"(p23), "l"(two23));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r01) : "l"(q01), "l"(a2), "l"(b2));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r23) : "l"(q23), "l"(a2), "l"(b2));
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
      : "=r"(lo)
      : "f"(__uint_as_float(uint32_t(r01 >> 32))), "f"(__uint_as_float(uint32_t(r01))));
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
      : "=r"(hi)
      : "f"(__uint_as_float(uint32_t(r23 >> 32))), "f"(__uint_as_float(uint32_t(r23))));
}

__device__ __forceinline__ void s8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t t = w ^ 0x80808080u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(a) : "r"(t), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x5342;" : "=r"(b) : "r"(t), "r"(0x64646464u));
  const uint32_t magic = 0x64806480u;                 // FP16 1152, 1152
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(magic));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(magic));
}

}  // namespace ptx
}  // namespace h3q
