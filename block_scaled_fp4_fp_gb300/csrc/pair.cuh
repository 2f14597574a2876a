// pair.cuh -- cluster and CTA-pair (tcgen05 cta_group::2) helpers shared by
// the kernels that run on two SMs per tile: PTX for the cluster rank, shared
// memory addresses of the peer CTA, cluster barriers, remote and
// cluster-scope mbarrier operations, TMA loads that complete on either CTA's
// barrier, and the commit that frees a barrier in both CTAs.
#pragma once
#include "common.cuh"

namespace fp4 {
namespace {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa_u32(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrivals on an mbarrier of another CTA of the cluster (shared::cluster
// address).  Neither carries a cluster-scope release: such a release waits for
// the memory traffic still in flight on the arriving SM (measured: on the qqmm
// pair kernel it held each epilogue warp ~0.7 us a tile while the next tile's
// TMA loads landed; on the W4A16 pair kernel's stage forwarding it capped
// NVFP4 at ~1370 TFLOP/s, ~1750 without it).
//
// Relaxed: for a signal that publishes no memory, "this thread's
// tensor-memory reads are complete" (after tcgen05.wait::ld and
// tcgen05.fence::before_thread_sync), which frees the accumulator for the next
// tile's MMAs.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t caddr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" :: "r"(caddr) : "memory");
}
// Release at CTA scope: orders this CTA's prior shared-memory writes (already
// made visible to the async proxy by fence.proxy.async), the operands that the
// pair's MMAs read from this CTA's own shared memory.
__device__ __forceinline__ void mbar_arrive_remote_cta(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" :: "r"(caddr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(bar_addr), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait (as mbar_wait) on a barrier that other CTAs of the cluster arrive at.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, unsigned* err, bool& failed) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_cluster(a, parity)) return true;
  if (failed) return false;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_cluster(a, parity)) return true;
    if (clock64() - t0 > kWaitLimitCycles) {
      record_error(err, kErrTimeout);
      failed = true;
      return false;
    }
  }
}
__device__ __forceinline__ void tma2_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];"
      :: "r"(dst), "l"(tmap), "r"(bar), "r"(x), "r"(y) : "memory");
}
// Commit this thread's tcgen05 operations to `bar` in both CTAs of the pair.
__device__ __forceinline__ void tc2_commit_both(uint64_t* bar) {
  const uint16_t mask = 0x3;
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               :: "r"(smem_u32(bar)), "h"(mask) : "memory");
}

}  // namespace
}  // namespace fp4
