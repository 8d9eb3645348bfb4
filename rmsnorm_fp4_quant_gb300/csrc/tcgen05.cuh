// tcgen05.cuh - the sm_100-family tensor-core primitives used by the FP4 GEMM:
// tensor-memory allocation, shared-memory matrix descriptors, the block-scaled
// MMA of kind mxf4nvf4, scale-factor copies into tensor memory, commit to an
// mbarrier, tensor-memory loads, the tiled TMA load and PDL grid control.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "async_copy.cuh"

namespace fp4q {

// --- tensor memory ----------------------------------------------------------
// Allocation is warp-wide; the address (lane 0, first column) lands in shared
// memory.  ncols: a power of two, 32..512.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_addr(slot)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// --- shared-memory matrix descriptors ----------------------------------------
// Bits 0-13 start address, 16-29 leading-dimension byte offset, 32-45 stride
// byte offset (all in 16-byte units), 46-47 descriptor version (1 on the
// sm_100 family), 61-63 swizzle mode.
constexpr uint32_t kSwizzleNone = 0;
constexpr uint32_t kSwizzle128B = 2;
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(swizzle) << 61);
}

// --- MMA ----------------------------------------------------------------------
// D[tmem] (+)= A[smem] * B[smem]^T with E2M1 operands (K = 64 per instruction)
// and block scales read from tensor memory at sfa / sfb: NVFP4 (MX = false),
// one E4M3 scale per 16 elements (4 per row per instruction), or MXFP4 (MX =
// true), one UE8M0 scale per 32 elements (2 per row per instruction, the byte
// pair chosen by the instruction descriptor).
template <bool MX>
__device__ __forceinline__ void mma_fp4_block_scaled(uint32_t d_tmem, uint64_t adesc,
                                                     uint64_t bdesc, uint32_t idesc,
                                                     uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                     uint32_t accumulate) {
  if constexpr (MX) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X "
        "[%0], %1, %2, %3, [%5], [%6], p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem),
           "r"(sfb_tmem)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
        "[%0], %1, %2, %3, [%5], [%6], p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem),
           "r"(sfb_tmem)
        : "memory");
  }
}

// 32 rows x 16 bytes of shared memory into 32 lanes x 4 columns of tensor
// memory, repeated in each of the four 32-lane quarters.
__device__ __forceinline__ void tmem_copy_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc)
               : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued
// before it has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(smem_addr(bar)) : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 lanes (one lane per thread),
// waited for in the same statement so no use can move above the wait.
__device__ __forceinline__ void tmem_load_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// --- shared memory across the cluster -----------------------------------------
// Makes this thread's generic-proxy writes to its CTA's shared memory visible
// to the async proxy (bulk copies issued after a later barrier read them).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Shared -> shared bulk copy (TMA engine) into a CTA of the cluster: dst and
// bar are shared::cluster addresses (mapa), src is this CTA's; both 16-byte
// aligned, bytes a multiple of 16; completion counted on bar, in dst's CTA.
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst, uint32_t src, uint32_t bytes,
                                               uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst), "r"(src), "r"(bytes), "r"(bar) : "memory");
}

// --- TMA ----------------------------------------------------------------------
// Tiled 2-D load of the box at (x, y) of `map` (x in elements of the innermost
// dimension, a multiple of 16 bytes) into shared memory, counted on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];"
      :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
         "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace fp4q
