// Inline-PTX helpers for kernels that run on 2-CTA clusters with
// tcgen05 cta_group::2 (one MMA spans both SMs of the pair): cluster rank and
// barrier, shared::cluster addressing, TMA loads that complete on the leader
// CTA's mbarrier, pair MMAs, multicast commits and remote arrivals. Written
// from the PTX ISA descriptions of these instructions.
#pragma once
#include <cuda_bf16.h>

#include "sm100_ptx.cuh"

namespace moe {
namespace pair {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cta address -> shared::cluster address of the same variable in CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m, int x, int y,
                                                 uint32_t leader_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(leader_bar)
      : "memory");
}

__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at `bar` (same offset) in every CTA of `mask`
// when all previously issued pair MMAs of this thread complete.
__device__ __forceinline__ void commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster. Used by the epilogue warps to
// hand a TMEM accumulator back to the MMA issuer: the tcgen05 loads are complete
// (tcgen05.wait::ld) and ordered by tcgen05.fence::before_thread_sync, so only
// CTA-scope release is needed; a cluster-scope release would also wait for the
// epilogue's global stores to drain before every hand-back.
__device__ __forceinline__ void arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}


// Shared-memory descriptor for an MN-major operand as a 128-byte-swizzled TMA
// box of 64 MN elements x 64 K rows writes it: 8-row K groups 1024 bytes
// apart (stride byte offset), 64-element MN blocks `mn_block_bytes` apart
// (leading byte offset), version 1, layout type 2. One K=16 step of the MMA
// covers two K groups, so its start address advances by 2048 bytes.
__device__ __forceinline__ uint64_t sdesc_mn128(uint32_t saddr, uint32_t mn_block_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((mn_block_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16, D f32, A and B bf16; a_mn / b_mn select
// MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16_f32_major(int M, int N, int a_mn, int b_mn) {
  return ptx::idesc_bf16_f32(M, N) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16);
}

}  // namespace pair
}  // namespace moe
