// Fifth-generation tensor cores (tcgen05, sm_100 family): tensor-memory
// allocation, shared-memory operand and instruction descriptors, MMA issue,
// completion and loads from tensor memory, and TMA tensor copies.  Inline PTX
// only, written from the PTX ISA's description of these instructions.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "ptx.cuh"

namespace mkv {

// ---- tensor memory (TMEM) ---------------------------------------------------
// Allocation and release are warp-wide (.sync.aligned): the whole warp calls.
// The allocated base address is written to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Order tensor-core work around a thread barrier.
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// ---- descriptors --------------------------------------------------------------
// Shared-memory operand descriptor of a K-major tile in the 128-byte swizzled
// layout: rows of 128 bytes (64 fp16 along K), 16-byte chunks of row r placed
// at chunk ^ (r mod 8) inside 1024-byte atoms of 8 rows, atoms 1024 bytes
// apart along M (or N).  The tile must start on a 1024-byte boundary; the K
// steps inside an atom are taken by adding 32 bytes per 16 elements to the
// start address.  Fields: start address / 16 (bits 0-13), leading byte offset
// / 16 (16-29; unused by swizzled K-major layouts, set to 1), stride byte
// offset / 16 (32-45: 1024 B), descriptor version 1 (46-47), swizzle mode 2 =
// 128-byte (61-63).
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16 with fp16 A and B (both K-major), fp32
// accumulation, M x N: D format F32 = 1 (bits 4-5), A and B format F16 = 0
// (7-9, 10-12), no negation or transposition (13-16), N / 8 (17-22), M / 16
// (24-28).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---- MMA ----------------------------------------------------------------------
// D[tmem] = A * B (+ D when accumulate != 0); one thread issues.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// One arrive on `bar` once every MMA issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ---- loads from TMEM ----------------------------------------------------------
// Warp w (of a warpgroup) reads TMEM lanes 32 (w % 4) .. +31: lane i of the
// warp gets 16 consecutive 32-bit columns of TMEM lane (base lane + i),
// starting at the address's column.  Complete with tmem_ld_wait().
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t r[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// ---- TMA tensor copies ----------------------------------------------------------
// 3-D tiled copy global -> shared completing on `bar` (expect-tx bytes set by
// the caller).  The innermost coordinate must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace mkv
