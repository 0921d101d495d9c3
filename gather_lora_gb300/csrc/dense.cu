// Dense single-adapter fold on the fifth-generation tensor cores (sm_103a).
//
// The pages' apply_lora_delta ("lora_delta.rs", apply_lora_delta: the
// tensor-core path for larger m, dense_gemm_tc then the fused
// dense_gemm_tc_scaled_acc) computes, for one adapter pair and every row i < m,
//   xa[i, :]  = bf16( x[i, :] @ A^T )                       (fp32 accumulate)
//   out[i, :] = bf16( fma(scale, bf16( xa[i, :] @ B^T ), out[i, :]) ).
// Here both contractions run as tcgen05 MMAs (M = 128 rows per tile) with fp32
// accumulators in tensor memory; every operand tile arrives by TMA in the
// swizzled K-major layout the MMA reads directly.
//
// One tile of 128 rows is spread over a cluster of cl CTAs (1, 2, 4 or 8):
//   shrink   CTA c contracts the 64-wide k-chunks c, c + cl, ... of x and A into
//            an fp32 partial of xa [128, max_rank] (TMEM columns 0 ..);
//   exchange the partials go to shared memory, CTA c sums rows
//            [c * 128 / cl, (c + 1) * 128 / cl) over the cluster in rank order,
//            rounds them to BF16 and writes them into every CTA's xa tile (and
//            to the optional global xa);
//   expand   CTA c takes the 128-column output chunks c, c + cl, ...: D = xa @ B^T
//            into one of two TMEM accumulators (columns 128 and 256), while the
//            epilogue warps fold the other one with the staged output tile and
//            store it back by TMA.
// Warp roles: warps 0-7 read TMEM and fold (two warpgroups: lanes 32 * (w % 4)
// .., even / odd 16-column groups), warp 8 issues TMA, warp 9 allocates TMEM
// and issues the MMAs. Every wait on an mbarrier is bounded; a timeout sets a
// status bit, skips the output stores and lets the CTA reach its exit.
#include <cooperative_groups.h>

#include "common.cuh"
#include "dense_types.h"
#include "tc05.cuh"

namespace cg = cooperative_groups;

namespace glora {

__device__ unsigned int g_dense_status = 0;
constexpr unsigned kDenseTimeoutBit = 0x2u;   // the fold kernels' timeout bit

namespace {

constexpr int kEpiThreads = kDenseEpiWarps * 32;
constexpr int kTmaWarp = kDenseEpiWarps;
constexpr int kMmaWarp = kDenseEpiWarps + 1;

struct DenseCtl {
  unsigned long long full[kDenseMaxRing];
  unsigned long long empty[kDenseMaxRing];
  unsigned long long ofull[2], oempty[2];       // staged output tiles
  unsigned long long d1_full;                   // the xa partial is in TMEM
  unsigned long long d2_full[2], d2_empty[2];   // expand accumulators
  uint32_t tmem_base;
  int failed;
};
static_assert(sizeof(DenseCtl) <= kDenseControl, "control block");

__device__ __forceinline__ void dense_timeout(DenseCtl& c) {
  c.failed = 1;
  atomicOr(&g_dense_status, kDenseTimeoutBit);
}

// Barrier among the epilogue warps only (named barrier 1).
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(kEpiThreads) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Byte offset, inside the xa tile [128 rows, max_rank] (the expand's A
// operand), of the 16-byte chunk holding columns [8c, 8c + 8) of row i.
// max_rank >= 64: 128-byte swizzle, atoms of 64 columns 16 KB apart;
// 32: 64-byte swizzle; 16: 32-byte swizzle.
__device__ __forceinline__ uint32_t xa_chunk(int i, int c, int max_rank) {
  if (max_rank >= 64) return (c >> 3) * (kDenseRows * 128) + i * 128 + (((c & 7) ^ (i & 7)) << 4);
  if (max_rank == 32) return i * 64 + ((c ^ ((i >> 1) & 3)) << 4);
  return i * 32 + ((c ^ ((i >> 2) & 1)) << 4);
}

// Byte offset of the fp32 partial of xa, row i, 16-byte chunk c (columns
// [4c, 4c + 4)): rows of max_rank floats, chunks permuted by the row so that
// the 32 rows of a warp store to different banks.
__device__ __forceinline__ uint32_t part_chunk(int i, int c, int max_rank) {
  return i * max_rank * 4 + ((c ^ (i & (max_rank / 4 - 1))) << 4);
}

}  // namespace

__global__ void __launch_bounds__(kDenseThreads, 1) lora_dense_fold_kernel(const __grid_constant__ DenseArgs p) {
  extern __shared__ unsigned char dense_smem_raw[];
  const uint32_t raw = smem_u32(dense_smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  unsigned char* base = dense_smem_raw + pad;
  const uint32_t base_u32 = raw + pad;
  const int R = p.max_rank, ns = p.ns, CL = p.cl;
  const uint32_t ring = base_u32;
  const uint32_t outr = ring + ns * p.stage_bytes;          // two output stages / the fp32 partial
  const uint32_t xa_s = outr + 2 * kDenseOutStage;          // BF16 xa tile
  DenseCtl& ctl = *reinterpret_cast<DenseCtl*>(base + (xa_s - base_u32) + kDenseRows * R * 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const cg::cluster_group cluster = cg::this_cluster();
  const int crank = static_cast<int>(cluster.block_rank());
  const int row0 = static_cast<int>(blockIdx.x / CL) * kDenseRows;
  const int nkc = (p.k_in + kDenseKChunk - 1) / kDenseKChunk;
  const int njc = (p.n_out + kDenseJChunk - 1) / kDenseJChunk;
  const int n_sh = crank < nkc ? (nkc - 1 - crank) / CL + 1 : 0;   // this CTA's shrink items
  const int n_ex = crank < njc ? (njc - 1 - crank) / CL + 1 : 0;   // and expand chunks
  const int n_items = n_sh + n_ex;

  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(smem_u32(&ctl.full[s]), 1);
      mbar_init(smem_u32(&ctl.empty[s]), 1);
    }
    for (int o = 0; o < 2; ++o) {
      mbar_init(smem_u32(&ctl.ofull[o]), 1);
      mbar_init(smem_u32(&ctl.oempty[o]), 1);
      mbar_init(smem_u32(&ctl.d2_full[o]), 1);
      mbar_init(smem_u32(&ctl.d2_empty[o]), kEpiThreads);
    }
    mbar_init(smem_u32(&ctl.d1_full), 1);
    ctl.failed = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&ctl.tmem_base), kDenseTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;

  pdl_wait_then_release();

  if (warp == kTmaWarp) {
    // ============================ TMA producer ============================
    // Ring items in order: the shrink items (x box [128 x 64] then A box
    // [max_rank x 64]), then the expand items (B [128 x max_rank] as boxes of
    // at most 64 columns). Items whose stage is freed by shrink MMAs go out
    // before the exchange; output tiles only after it (they overwrite the
    // partials).
    const int pre = min(n_items, n_sh + ns);
    auto produce = [&](int it) {
      const int s = it % ns;
      if (it >= ns && !mbar_wait(smem_u32(&ctl.empty[s]), ((it / ns) - 1) & 1)) dense_timeout(ctl);
      const uint32_t st = ring + s * p.stage_bytes, fb = smem_u32(&ctl.full[s]);
      if (it < n_sh) {
        const int k0 = (crank + it * CL) * kDenseKChunk;
        mbar_arrive_expect_tx(fb, (kDenseRows + R) * kDenseKChunk * 2);
        tma_load_2d(st, &p.map_x, k0, row0, fb);
        tma_load_2d(st + kDenseRows * kDenseKChunk * 2, &p.map_a, k0, 0, fb);
      } else {
        const int j0 = (crank + (it - n_sh) * CL) * kDenseJChunk;
        const int natoms = R >= 64 ? R / 64 : 1;
        mbar_arrive_expect_tx(fb, kDenseJChunk * R * 2);
        for (int a = 0; a < natoms; ++a) tma_load_2d(st + a * (kDenseJChunk * 128), &p.map_b, a * 64, j0, fb);
      }
    };
    auto produce_out = [&](int e) {
      const int o = e & 1;
      if (e >= 2 && !mbar_wait(smem_u32(&ctl.oempty[o]), ((e >> 1) - 1) & 1)) dense_timeout(ctl);
      const int j0 = (crank + e * CL) * kDenseJChunk;
      const uint32_t ob = smem_u32(&ctl.ofull[o]), dst = outr + o * kDenseOutStage;
      mbar_arrive_expect_tx(ob, kDenseOutStage);
      tma_load_2d(dst, &p.map_out, j0, row0, ob);
      tma_load_2d(dst + kDenseOutStage / 2, &p.map_out, j0 + 64, row0, ob);
    };
    if (lane == 0)
      for (int it = 0; it < pre; ++it) produce(it);
    __syncwarp();
    cluster.sync();   // partials written
    cluster.sync();   // partials summed: the output stages are free
    if (lane == 0) {
      int it = pre;
      for (int e = 0; e < n_ex; ++e) {
        produce_out(e);
        for (const int lim = min(n_items, n_sh + e + ns); it < lim; ++it) produce(it);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ============================ MMA issuer ==============================
    if (lane == 0) {
      const uint32_t id1 = idesc_bf16_f32(kDenseRows, R);
      for (int it = 0; it < n_sh; ++it) {
        const int s = it % ns;
        if (!mbar_wait(smem_u32(&ctl.full[s]), (it / ns) & 1)) dense_timeout(ctl);
        tc_fence_after();
        const uint32_t sx = ring + s * p.stage_bytes, sa = sx + kDenseRows * kDenseKChunk * 2;
#pragma unroll
        for (int kk = 0; kk < kDenseKChunk / 16; ++kk)
          umma_bf16(tmem, smem_desc(sx + kk * 32, 1024, Swz::k128), smem_desc(sa + kk * 32, 1024, Swz::k128), id1,
                    (it | kk) != 0);
        umma_commit(smem_u32(&ctl.empty[s]));
      }
      if (n_sh > 0) umma_commit(smem_u32(&ctl.d1_full));
    }
    __syncwarp();
    cluster.sync();
    cluster.sync();   // xa is in every CTA's shared memory
    if (lane == 0) {
      fence_proxy_async_smem();
      tc_fence_after();
      const uint32_t id2 = idesc_bf16_f32(kDenseRows, kDenseJChunk);
      const Swz swz = R >= 64 ? Swz::k128 : (R == 32 ? Swz::k64 : Swz::k32);
      const uint32_t sbo = 8u * (R >= 64 ? 128u : 2u * R);   // bytes between 8-row groups
      for (int e = 0; e < n_ex; ++e) {
        const int b = e & 1, it = n_sh + e, s = it % ns;
        if (e >= 2 && !mbar_wait(smem_u32(&ctl.d2_empty[b]), ((e >> 1) - 1) & 1)) dense_timeout(ctl);
        if (!mbar_wait(smem_u32(&ctl.full[s]), (it / ns) & 1)) dense_timeout(ctl);
        tc_fence_after();
        const uint32_t sb = ring + s * p.stage_bytes;
        for (int ks = 0; ks < R / 16; ++ks) {
          // k-step ks: 32 bytes further inside a swizzle row; 64-column atoms are separate tiles
          const uint32_t oa = R >= 64 ? (ks >> 2) * (kDenseRows * 128) + (ks & 3) * 32 : ks * 32;
          const uint32_t ob = R >= 64 ? (ks >> 2) * (kDenseJChunk * 128) + (ks & 3) * 32 : ks * 32;
          umma_bf16(tmem + 128 + 128 * b, smem_desc(xa_s + oa, sbo, swz), smem_desc(sb + ob, sbo, swz), id2, ks != 0);
        }
        umma_commit(smem_u32(&ctl.empty[s]));
        umma_commit(smem_u32(&ctl.d2_full[b]));
      }
    }
    __syncwarp();
  } else {
    // ========================= epilogue warps =============================
    const int wg = warp >> 2, quad = warp & 3, row = quad * 32 + lane;   // tile row = TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    // 1. this CTA's fp32 partial of xa -> shared memory
    if (n_sh > 0) {
      if (!mbar_wait(smem_u32(&ctl.d1_full), 0)) dense_timeout(ctl);
      tc_fence_after();
      for (int g = wg; g < R / 16; g += 2) {
        uint32_t v[16];
        tmem_ld16(lane_addr + g * 16, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j)
          sts128(outr + part_chunk(row, g * 4 + j, R), make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
      }
    } else {   // no k-chunk reached this CTA: its partial is zero
      for (int g = wg; g < R / 16; g += 2)
#pragma unroll
        for (int j = 0; j < 4; ++j) sts128(outr + part_chunk(row, g * 4 + j, R), make_uint4(0, 0, 0, 0));
    }
    cluster.sync();
    // 2. rows [crank * 128 / cl, ..) summed over the cluster in rank order,
    //    rounded to BF16, written into every CTA's xa tile (and to global xa)
    const int rows_per = kDenseRows / CL, c8n = R / 8;
    const float* part = reinterpret_cast<const float*>(base + (outr - base_u32));
    unsigned char* xa_tile = base + (xa_s - base_u32);
    for (int item = tid; item < rows_per * c8n; item += kEpiThreads) {
      const int i = crank * rows_per + item / c8n, c8 = item - (item / c8n) * c8n;
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.f;
      for (int q = 0; q < CL; ++q) {
        const unsigned char* pq = reinterpret_cast<const unsigned char*>(cluster.map_shared_rank(part, q));
        const float4 lo = *reinterpret_cast<const float4*>(pq + part_chunk(i, 2 * c8, R));
        const float4 hi = *reinterpret_cast<const float4*>(pq + part_chunk(i, 2 * c8 + 1, R));
        acc[0] += lo.x; acc[1] += lo.y; acc[2] += lo.z; acc[3] += lo.w;
        acc[4] += hi.x; acc[5] += hi.y; acc[6] += hi.z; acc[7] += hi.w;
      }
      const uint4 packed = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                      pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
      const uint32_t off = xa_chunk(i, c8, R);
      for (int q = 0; q < CL; ++q)
        *reinterpret_cast<uint4*>(cluster.map_shared_rank(xa_tile, q) + off) = packed;
      if (p.xa && row0 + i < p.m)
        *reinterpret_cast<uint4*>(p.xa + static_cast<long long>(row0 + i) * R + c8 * 8) = packed;
    }
    fence_proxy_async_cluster();
    cluster.sync();
    // 3. expand + fold: chunk e of this CTA is output columns
    //    [(crank + e * cl) * 128, + 128); lane = row, 16-column groups alternate
    //    between the two warpgroups. The staged tile is two 64-column boxes
    //    with the 128-byte swizzle.
    const float scale = p.scale;
    for (int e = 0; e < n_ex; ++e) {
      const int b = e & 1;
      if (!mbar_wait(smem_u32(&ctl.d2_full[b]), (e >> 1) & 1)) dense_timeout(ctl);
      if (!mbar_wait(smem_u32(&ctl.ofull[b]), (e >> 1) & 1)) dense_timeout(ctl);
      tc_fence_after();
      const uint32_t ost = outr + b * kDenseOutStage;
      for (int g = wg; g < kDenseJChunk / 16; g += 2) {
        uint32_t v[16];
        tmem_ld16(lane_addr + 128 + 128 * b + g * 16, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = (g & 3) * 2 + j;
          const uint32_t addr = ost + (g >> 2) * (kDenseOutStage / 2) + row * 128 + ((c ^ (row & 7)) << 4);
          uint4 o = lds128(addr);
          const uint32_t* d = v + 8 * j;
          o.x = fold_pair(__uint_as_float(d[0]), __uint_as_float(d[1]), scale, o.x);
          o.y = fold_pair(__uint_as_float(d[2]), __uint_as_float(d[3]), scale, o.y);
          o.z = fold_pair(__uint_as_float(d[4]), __uint_as_float(d[5]), scale, o.z);
          o.w = fold_pair(__uint_as_float(d[6]), __uint_as_float(d[7]), scale, o.w);
          sts128(addr, o);
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&ctl.d2_empty[b]));
      fence_proxy_async_smem();
      epi_sync();
      if (tid == 0) {
        if (!ctl.failed) {
          const int j0 = (crank + e * CL) * kDenseJChunk;
          tma_store_2d(&p.map_out, j0, row0, ost);
          tma_store_2d(&p.map_out, j0 + 64, row0, ost + kDenseOutStage / 2);
          bulk_commit_group();
        }
        bulk_wait_read0();
        mbar_arrive(smem_u32(&ctl.oempty[b]));
      }
    }
    if (tid == 0) bulk_wait0();
  }

  // After a timeout, let this CTA's own loads still in flight land (bounded)
  // before its shared memory is released.
  if (warp == kTmaWarp && lane == 0 && ctl.failed) {
    for (int it = max(0, n_items - ns); it < n_items; ++it) mbar_wait(smem_u32(&ctl.full[it % ns]), (it / ns) & 1);
    for (int e = max(0, n_ex - 2); e < n_ex; ++e) mbar_wait(smem_u32(&ctl.ofull[e & 1]), (e >> 1) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kDenseTmemCols);
  }
}

int launch_dense(const DenseArgs& a, void* stream) {
  // (set on every call: the attribute belongs to the current device, like the launch)
  const cudaError_t set = cudaFuncSetAttribute(lora_dense_fold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               a.smem_bytes);
  if (set != cudaSuccess) return static_cast<int>(set);
  const int tiles = (a.m + kDenseRows - 1) / kDenseRows;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * a.cl), 1, 1);
  cfg.blockDim = dim3(kDenseThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(a.smem_bytes);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = static_cast<unsigned>(a.cl);
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, lora_dense_fold_kernel, a);
  return static_cast<int>(e);
}

int read_dense_status(void* stream, uint32_t* out, int clear) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t err = cudaMemcpyFromSymbolAsync(&v, g_dense_status, sizeof v, 0, cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess && clear) {
    static const uint32_t z = 0;
    err = cudaMemcpyToSymbolAsync(g_dense_status, &z, sizeof z, 0, cudaMemcpyHostToDevice, s);
  }
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  *out = v;
  return static_cast<int>(err);
}

}  // namespace glora
