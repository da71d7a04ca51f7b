// Thread-block-cluster and programmatic-launch helpers (inline PTX, sm_103a)
// shared by the CTA-pair decode kernels: cluster rank and id, the address of
// a shared-memory location in the peer CTA, the split cluster barrier,
// remote mbarrier arrivals and waits at cluster scope, remote stores, and
// griddepcontrol.
#pragma once

#include "wq_device.cuh"

namespace wq {
namespace cl {

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
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_peer(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// The cluster barrier in two halves: every thread arrives once, early (after
// its CTA's mbarriers exist), and waits only before its first access to the
// peer's shared memory.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a barrier that the peer CTA arrives on (cluster scope).
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}
// Remote 16-byte store into the peer's shared memory that counts its bytes
// on the peer's mbarrier (complete_tx): the peer's wait on that barrier
// returns once every such store has landed, with no release/arrive round
// trip on the sending side.
__device__ __forceinline__ void st_async_peer_v4(uint32_t cluster_addr, float4 v, uint32_t cluster_mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   cluster_addr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(cluster_mbar)
               : "memory");
}
// Programmatic dependent launch: let the next kernel of the stream start
// launching, and wait for the previous one (both no-ops without such a
// neighbour).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// The 32 activations of a staged job, from their raw bf16 words.
__device__ __forceinline__ void raw_to_float(const uint4 (&r)[4], float (&v)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t wv[4] = {r[c].x, r[c].y, r[c].z, r[c].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[8 * c + 2 * e] = __uint_as_float(wv[e] << 16);
      v[8 * c + 2 * e + 1] = __uint_as_float(wv[e] & 0xFFFF0000u);
    }
  }
}
}  // namespace cl
}  // namespace wq
