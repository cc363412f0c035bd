// Inline-PTX wrappers for kernels that run as a pair of CTAs on the two SMs
// of one TPC (a cluster of 2) and share one tcgen05 MMA between them
// (`.cta_group::2`): cluster rank and barrier, addresses in the peer CTA's
// shared memory, remote mbarrier arrivals, TMA copies that signal the lead
// CTA's mbarrier, tensor-memory allocation for the pair, pair MMAs (M = 256:
// each CTA holds 128 rows of A and half of B, and receives its 128 rows of
// D in its own tensor memory) and their commits, multicast to both CTAs.
// Each wrapper is one PTX instruction (or a short fixed sequence) written
// from the PTX ISA descriptions of these instructions.
#pragma once

#include <stdint.h>

#include "msa_common.cuh"
#include "tc_ptx.cuh"

namespace msa {
namespace pair {

__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Both CTAs of the cluster: every thread arrives, then waits for all.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Address, in the cluster's shared window, of the variable at local shared
// address `a` in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

// Arrive once on an mbarrier given by its cluster-window address (this CTA's
// or the peer's).  Default semantics (release, CTA scope): what the waiting
// thread reads after it is tensor memory, ordered by the tcgen05 fences on
// both sides of the arrive/wait pair.
__device__ __forceinline__ void arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

// The same, executed by a whole converged warp: one elected lane arrives
// (predicated inside one asm block, so the compiler sees no divergent
// branch around values the warp keeps live).
__device__ __forceinline__ void arrive_cluster_w(uint32_t cluster_bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.shared::cluster.b64 _, [%0];\n\t}" ::"r"(cluster_bar)
      : "memory");
}

// Wait probes of this CTA's mbarrier (arrivals may come from the peer CTA
// too).  Cluster-scope release/acquire on these measured about 1400 cycles
// per handoff against about 40 with the defaults.
__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
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
__device__ __forceinline__ bool test_wait_cluster(uint32_t bar, uint32_t parity) {
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

// 3-D tiled tensor copy global -> this CTA's shared memory whose completion
// (bytes) is signalled on an mbarrier of either CTA of the pair, given by its
// cluster-window address.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* desc, uint32_t cluster_bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(x), "r"(y), "r"(z), "r"(cluster_bar)
      : "memory");
}

// Tensor memory for the pair: executed by one warp in each CTA.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Arrive once on the mbarrier at local offset `bar` in BOTH CTAs when every
// pair MMA this warp issued before has completed (elected lane).
__device__ __forceinline__ void commit_both(uint32_t bar) {
  const uint16_t both = 3;  // CTA mask: ranks 0 and 1
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(bar), "h"(both)
      : "memory");
}

// Eight pair SS MMAs over K = 128 (steps of 16) from one elect.sync: A is
// each CTA's 128 x 128 K-major SW128 tile (64-column chunks `kAChunk`
// descriptor units apart), B each CTA's half of the N = 128 rows (64 rows,
// chunks `kBChunk` apart).  Step kk reads chunk kk / 4, 32 bytes x (kk % 4)
// into it.  The first MMA overwrites D unless `accumulate`.
template <uint32_t kAChunk, uint32_t kBChunk>
__device__ __forceinline__ void mma_ss_x8(uint32_t d, uint32_t a_lo, uint32_t b_lo,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p0;\n\t.reg .b64 da, db;\n\t.reg .b32 al, bl;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\t"
      "mov.b64 da, {%1, %5};\n\tmov.b64 db, {%2, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, p0;\n\t"
      "add.u32 al, %1, 2;\n\tadd.u32 bl, %2, 2;\n\t"
      "mov.b64 da, {al, %5};\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, 1;\n\t"
      "add.u32 al, %1, 4;\n\tadd.u32 bl, %2, 4;\n\t"
      "mov.b64 da, {al, %5};\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, 1;\n\t"
      "add.u32 al, %1, 6;\n\tadd.u32 bl, %2, 6;\n\t"
      "mov.b64 da, {al, %5};\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, 1;\n\t"
      "add.u32 al, %1, %6;\n\tadd.u32 bl, %2, %7;\n\t"
      "mov.b64 da, {al, %5};\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, 1;\n\t"
      "add.u32 al, al, 2;\n\tadd.u32 bl, bl, 2;\n\t"
      "mov.b64 da, {al, %5};\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, 1;\n\t"
      "add.u32 al, al, 2;\n\tadd.u32 bl, bl, 2;\n\t"
      "mov.b64 da, {al, %5};\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, 1;\n\t"
      "add.u32 al, al, 2;\n\tadd.u32 bl, bl, 2;\n\t"
      "mov.b64 da, {al, %5};\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, 1;\n\t}" ::"r"(d),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(ptx::kDescHiSw128), "n"(kAChunk),
      "n"(kBChunk)
      : "memory");
}

// Eight pair TS MMAs over K = 128: A (128 rows per CTA) from each CTA's
// tensor memory, columns a + 8 kk; B each CTA's half of N, an MN-major
// SW128 tile of 128 K rows, 16 rows (2048 bytes) per step.
__device__ __forceinline__ void mma_ts_x8(uint32_t d, uint32_t a_tmem, uint32_t b_lo,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p0;\n\t.reg .b64 db;\n\t.reg .b32 at, bl;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\t"
      "mov.b64 db, {%2, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], db, %3, p0;\n\t"
      "mov.b32 at, %1;\n\tmov.b32 bl, %2;\n\t"
      "add.u32 at, at, 8;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t"
      "add.u32 at, at, 8;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t"
      "add.u32 at, at, 8;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t"
      "add.u32 at, at, 8;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t"
      "add.u32 at, at, 8;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t"
      "add.u32 at, at, 8;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t"
      "add.u32 at, at, 8;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t}" ::"r"(d),
      "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(ptx::kDescHiSw128)
      : "memory");
}

// Eight pair TS MMAs over K = 128 whose A operand sits in tensor memory as
// four 32-column chunks, each holding its 16 packed bf16 pairs in the
// chunk's first 16 columns (steps at a, a + 8, a + 32, a + 40, ...); B each
// CTA's half of N, an MN-major SW128 tile, 16 rows (2048 bytes) per step.
__device__ __forceinline__ void mma_ts_chunked_x8(uint32_t d, uint32_t a_tmem, uint32_t b_lo,
                                                  uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p0;\n\t.reg .b64 db;\n\t.reg .b32 at, bl;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\t"
      "mov.b64 db, {%2, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], db, %3, p0;\n\t"
      "add.u32 at, %1, 8;\n\tadd.u32 bl, %2, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t"
      "add.u32 at, %1, 32;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t"
      "add.u32 at, %1, 40;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t"
      "add.u32 at, %1, 64;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t"
      "add.u32 at, %1, 72;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t"
      "add.u32 at, %1, 96;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t"
      "add.u32 at, %1, 104;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [at], db, %3, 1;\n\t}" ::"r"(d),
      "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(ptx::kDescHiSw128)
      : "memory");
}

}  // namespace pair

// Bounded waits of a CTA pair.  Each CTA has an abort flag in its shared
// memory; a wait also gives up when the peer's flag is set, so both CTAs
// leave their loops together.
struct PairWait {
  volatile int* abort;       // this CTA's flag
  uint32_t peer_abort;       // the peer's flag (cluster address)
  int* status;
  uint64_t limit;
};

__device__ __forceinline__ int peer_flag(uint32_t a) {
  int v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

// Bounded wait on phase `parity` of one of this CTA's mbarriers.  Returns
// false when the pair is aborting (this CTA's or the peer's flag set, or
// this wait ran out).  The first probe does not block; a limit of at most
// 1 ns makes every wait that this probe does not find complete run out.
// The peer's flag (a load from the other SM) is read every 8th round only.
// `backoff_ns` > 0 (the producer, whose ring gives it slack) sleeps between
// probes, leaving the issue slots of its SM sub-partition to the softmax.
__device__ __forceinline__ bool wait_pair(uint32_t bar, uint32_t parity, const PairWait& c,
                                          uint32_t backoff_ns = 0) {
  if (pair::test_wait_cluster(bar, parity)) return true;
  if (c.limit > 1) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t round = 0;; ++round) {
      if (backoff_ns) {
        __nanosleep(backoff_ns);
        if (pair::test_wait_cluster(bar, parity)) return true;
      } else if (pair::try_wait_cluster(bar, parity)) {
        return true;
      }
      if (*c.abort || ((round & 7) == 7 && peer_flag(c.peer_abort))) {
        *c.abort = 1;
        return false;
      }
      if (ptx::globaltimer() - t0 > c.limit) break;
    }
  } else if (*c.abort || peer_flag(c.peer_abort)) {
    *c.abort = 1;
    return false;
  }
  *c.abort = 1;
  record_status(c.status, MSA_ERR_TIMEOUT);
  return false;
}

// The same for a whole warp: every lane probes, so the warp's control flow
// stays converged (waits taken by one lane in a divergent branch measured
// far slower: branch-resolution stalls), with one result for all lanes.
__device__ __forceinline__ bool wait_pair_w(uint32_t bar, uint32_t parity, const PairWait& c) {
  return __all_sync(0xffffffffu, wait_pair(bar, parity, c));
}

// Wait used while draining: ignores the abort flags, limit `ns`.
__device__ __forceinline__ void drain_for(uint32_t bar, uint32_t parity, int* status,
                                          uint64_t ns) {
  if (pair::try_wait_cluster(bar, parity)) return;
  const uint64_t t0 = ptx::globaltimer();
  while (!pair::try_wait_cluster(bar, parity)) {
    if (ptx::globaltimer() - t0 > ns) {
      record_status(status, MSA_ERR_TIMEOUT);
      return;
    }
  }
}

}  // namespace msa
