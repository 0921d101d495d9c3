// Device helpers shared by the bgmv and MoE fold kernels (sm_103a).
//
// Everything here is a thin inline-PTX wrapper: mbarriers (with bounded
// waits), 1-D TMA bulk copies global->shared (cp.async.bulk), 16-byte
// asynchronous copies (cp.async.cg), shared-memory matrix loads (ldmatrix),
// BF16 tensor-core MMA with fp32 accumulation (mma.sync m16n8k16 / m16n8k8),
// and programmatic-dependent-launch controls (griddepcontrol).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fold_types.h"

namespace glora {

constexpr int kThreads = (kConsumerWarps + kProducerWarps) * 32;
constexpr int kWarps = kThreads / 32;
constexpr long long kWaitLimitCycles = 4000000000LL;  // give up on an mbarrier after ~2 s
constexpr long long kDrainLimitCycles = 200000000LL;  // ~0.1 s for in-flight copies after a give-up

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- asynchronous copies ---------------------------------------------------
// 16 bytes global -> shared, L2-only (.cg): adapter and activation rows are
// read once per CTA, so they should not displace L1.
__device__ __forceinline__ void cp_async16(uint32_t dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst_smem), "l"(src) : "memory");
}
// 16 zero bytes into shared memory through the same asynchronous path (no
// global read: the source size is 0).
__device__ __forceinline__ void cp_async16_zero(uint32_t dst_smem, const void* any_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, 0;\n" ::"r"(dst_smem), "l"(any_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
// Wait until at most `n` of this thread's most recent copy groups are pending.
__device__ __forceinline__ void cp_async_wait(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;\n" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;\n" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;\n" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;\n" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;\n" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;\n" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;\n" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;\n" ::: "memory"); break;
  }
}

// ---- mbarriers and TMA bulk copies -----------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
// Arrive on `bar` once all of this thread's earlier cp.async copies have landed
// (the arrival is counted in the barrier's initial count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_count(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
// Test phase `parity` of an mbarrier. If it is not complete the thread is
// suspended in hardware until it completes or `hint_ns` elapse, so waiting
// warps do not spin on issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}
// Wait for phase `parity` of an mbarrier; false after `limit` SM clocks
// (kWaitLimitCycles for the folds) without it. The limit is measured with the
// SM-local cycle counter: reading the global nanosecond timer costs about half
// a microsecond.
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity, long long limit) {
  constexpr uint32_t kHintNs = 1000000;
  if (mbar_try_wait(bar, parity, kHintNs)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity, kHintNs)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  return mbar_wait_limit(bar, parity, kWaitLimitCycles);
}

// 1-D TMA copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// from global to this CTA's shared memory, completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
               ::"r"(dst_smem), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// 2-D TMA tile load: the box of the tensor map `map` (a CUtensorMap in global or
// parameter memory) at coordinates (c0 innermost, c1) into shared memory at dst,
// completing on mbarrier `bar`. c0 * element size must be a multiple of 16 bytes;
// out-of-range parts of the box are filled with zeros and still count as bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst_smem, const void* map, int c0, int c1, uint32_t bar) {
  asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n"
               ::"r"(dst_smem), "l"(map), "r"(c0), "r"(c1), "r"(bar)
               : "memory");
}
// Start fetching a tensor map (in global memory) into the descriptor cache
// ahead of its first use by tma_load_2d.
__device__ __forceinline__ void prefetch_tensormap(const void* map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(map) : "memory");
}
// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
// Barrier among the CW consumer warps only (named barrier 1).
template <int CW = kConsumerWarps>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(CW * 32) : "memory");
}

// ---- shared-memory matrix fragments ----------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x1(uint32_t addr, uint32_t& r0) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x1.shared.b16 {%0}, [%1];\n" : "=r"(r0) : "r"(addr));
}

// Transposing forms: with .trans, lane (g = lane/4, q = lane%4) exchanges the
// pair [row 2q][col g], [row 2q+1][col g] of each 8x8 matrix (low half first),
// which is the accumulator layout of an m16n8 tile whose N index is the row.
// ---- BF16 tensor-core MMA, fp32 accumulate ----------------------------------
// D[16x8] += A[16xK] * B[Kx8]; A row-major (K contiguous per row of A), B
// "col" (K contiguous per column of B). Accumulator layout per lane
// (g = lane/4, q = lane%4): d0 (g, 2q), d1 (g, 2q+1), d2 (g+8, 2q), d3 (g+8, 2q+1).
__device__ __forceinline__ void mma_k16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_k8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// One K step (16, or 8 for a ragged tail) of a 16x8 output tile:
//   a_row_addr: shared address of the A row this lane feeds to ldmatrix,
//               i.e. A tile row (lane & 15), at the step's first column;
//   b_row_addr: shared address of the B row (lane & 7), at the step's first column.
// Column offsets of the second 8-wide half are added here.
__device__ __forceinline__ void mma_step(float (&acc)[4], uint32_t a_row_addr, uint32_t b_row_addr,
                                         int kstep, int lane) {
  if (kstep == 16) {
    uint32_t a0, a1, a2, a3, b0, b1;
    ldsm_x4(a_row_addr + ((lane >> 4) << 4), a0, a1, a2, a3);
    ldsm_x2(b_row_addr + (((lane >> 3) & 1) << 4), b0, b1);
    mma_k16(acc, a0, a1, a2, a3, b0, b1);
  } else {
    uint32_t a0, a1, b0;
    ldsm_x2(a_row_addr, a0, a1);
    ldsm_x1(b_row_addr, b0);
    mma_k8(acc, a0, a1, b0);
  }
}

// ---- programmatic dependent launch -----------------------------------------
// Wait until the preceding grid on the stream has completed and its memory is
// visible (no-op when the launch carried no programmatic dependency), then let
// the next grid start launching its CTAs.
__device__ __forceinline__ void pdl_wait_then_release() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Two fp32 values -> one BF16 pair (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The fold of two elements packed as BF16 pairs (low half first): per
// element bf16( fma(scale, bf16(acc), out) ), with both roundings done as
// pair conversions.
__device__ __forceinline__ uint32_t fold_pair(float acc_lo, float acc_hi, float scale, uint32_t out2) {
  const uint32_t d2 = pack_bf16x2(acc_lo, acc_hi);
  const float d_lo = __uint_as_float(d2 << 16), d_hi = __uint_as_float(d2 & 0xffff0000u);
  const float o_lo = __uint_as_float(out2 << 16), o_hi = __uint_as_float(out2 & 0xffff0000u);
  return pack_bf16x2(__fmaf_rn(scale, d_lo, o_lo), __fmaf_rn(scale, d_hi, o_hi));
}


// Block-wide inclusive sum over all kThreads threads (warp shuffles + one
// partial per warp in `warp_sums` shared scratch). Must be called by all threads.
__device__ __forceinline__ int block_inclusive_sum(int v, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) warp_sums[warp] = v;
  __syncthreads();
  int before = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) before += (w < warp) ? warp_sums[w] : 0;
  __syncthreads();
  return v + before;
}

}  // namespace glora
