// Fifth-generation tensor-core (tcgen05) and tensor-memory helpers for the
// dense single-adapter fold (sm_103a), as thin inline-PTX wrappers.
//
// Operand tiles live in shared memory in the K-major swizzled layouts that TMA
// writes: rows of W bytes (W = 128, 64 or 32: the swizzle width), 16-byte chunk
// c of row r stored at chunk c ^ f(r), with f(r) = r & 7 (128-byte swizzle),
// (r >> 1) & 3 (64-byte) or (r >> 2) & 1 (32-byte); groups of 8 rows are 8 * W
// bytes apart and every tile starts on a 1024-byte boundary. Accumulators live
// in tensor memory (TMEM): for M = 128, row i of the tile is TMEM lane i and
// column j is column base + j, fp32.
#pragma once

#include <stdint.h>

#include "dense_types.h"   // idesc_bf16_f32

namespace glora {

// ---- tensor-memory allocation (one full warp executes these) ---------------
// Allocate `ncols` TMEM columns (a power of two >= 32) for this CTA and write
// their base address to shared memory at dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

// Order tcgen05 operations across a thread synchronization (barrier or
// mbarrier): `before` ahead of the arrive, `after` behind the wait.
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// ---- shared-memory matrix descriptors ---------------------------------------
enum class Swz : uint32_t { k32 = 6, k64 = 4, k128 = 2 };   // descriptor layout codes

// Descriptor of a K-major operand tile at shared address `addr` (16-byte
// aligned, its swizzle atom 1024-byte aligned): start address >> 4 in bits
// 0-13, leading-byte offset (unused by swizzled K-major tiles; 16 bytes) in
// 16-29, stride-byte offset (between 8-row groups) >> 4 in 32-45, the
// descriptor version 1 in bits 46-47, base offset 0, layout code in 61-63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t sbo_bytes, Swz swz) {
  uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(swz) << 61;
  return d;
}

// ---- MMA issue (one thread) --------------------------------------------------
// D[tmem] (+)= A[smem] * B[smem]^T over one K = 16 step; `accumulate` = 0 overwrites D.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on mbarrier `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
               : "memory");
}

// ---- TMEM -> registers -------------------------------------------------------
// 16 consecutive fp32 columns of this thread's lane (warp w reads lanes
// 32 * (w % 4) ..; taddr carries that lane base in bits 16-31). Values are valid
// after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// ---- TMA tile store and bulk groups -----------------------------------------
// 2-D TMA tile store of the box at shared address src to tensor map `map` at
// (c0 innermost, c1); parts outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const void* map, int c0, int c1, uint32_t src_smem) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];\n" ::"l"(map), "r"(c0),
               "r"(c1), "r"(src_smem)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
// Wait until this thread's bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
// Wait until this thread's bulk stores are complete (written to global memory).
__device__ __forceinline__ void bulk_wait0() {
  asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}
// Make this thread's generic-proxy writes to shared memory of the cluster
// visible to later async-proxy (tensor core, TMA) reads.
__device__ __forceinline__ void fence_proxy_async_cluster() {
  asm volatile("fence.proxy.async.shared::cluster;\n" ::: "memory");
}

}  // namespace glora
