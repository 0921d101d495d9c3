// Launch description of the dense single-adapter fold (shared by the host
// launcher and the kernel; no CUDA types: host code includes it after
// cuda_runtime.h, which defines __host__ / __device__).
//
// One adapter (A [max_rank, k_in], B [n_out, max_rank], scale) folded into
// every one of m rows:
//   out[i, :] = bf16( fma(scale, bf16( bf16(x[i, :] @ A^T) @ B^T ), out[i, :]) ).
// Work unit: a tile of kDenseRows rows, spread over a cluster of `cl` CTAs:
// CTA c contracts the k-chunks c, c + cl, ... into an fp32 partial of
// xa (tensor cores, TMEM), the cluster sums the partials in rank order and
// rounds them to BF16, then CTA c expands and folds the output-column chunks
// c, c + cl, ...
#pragma once

#include <stdint.h>

namespace glora {

constexpr int kDenseRows = 128;       // rows per tile: the M of every MMA
constexpr int kDenseKChunk = 64;      // k per shrink ring item: one 128-byte swizzle atom of BF16
constexpr int kDenseJChunk = 128;     // output columns per expand accumulator: the N of the expand MMA
constexpr int kDenseEpiWarps = 8;     // two warpgroups read TMEM and fold (lanes 32 * (w % 4) ..)
constexpr int kDenseThreads = (kDenseEpiWarps + 2) * 32;   // + one TMA warp + one MMA warp
constexpr int kDenseTmemCols = 512;   // xa partial at column 0, two expand accumulators at 128 and 256
constexpr int kDenseMaxRing = 8;

// A CUtensorMap, as opaque bytes (the kernel only passes its address to TMA).
struct alignas(64) TensorMapBytes {
  unsigned char bytes[128];
};

struct DenseArgs {
  TensorMapBytes map_x;     // x [m, k_in], box {64, 128}, 128-byte swizzle
  TensorMapBytes map_a;     // A [max_rank, k_in], box {64, max_rank}, 128-byte swizzle
  TensorMapBytes map_b;     // B [n_out, max_rank], box {min(max_rank, 64), 128}, swizzle = min(2 * max_rank, 128) bytes
  TensorMapBytes map_out;   // base_out [m, n_out], box {64, 128}, 128-byte swizzle
  uint16_t* xa;             // optional [m, max_rank] BF16 output of the shrink
  float scale;
  int m, k_in, n_out, max_rank;
  int cl;                   // CTAs per cluster: 1, 2, 4 or 8
  int ns;                   // ring stages
  int stage_bytes;          // bytes per ring stage (multiple of 1024)
  int smem_bytes;           // dynamic shared memory per CTA (with 1 KB of alignment slack)
};

// Shared-memory plan (offsets from the 1024-byte aligned base):
//   [0, ns * stage_bytes)            ring: shrink items (x box, then A box) or expand items (B boxes)
//   out region: 2 * 32 KB            two staged output tiles [128 rows x 128 cols]; also the
//                                    fp32 partial of xa [128 x max_rank] during the exchange
//   xa region: 128 * max_rank * 2    the BF16 xa tile, the expand's A operand
//   control: 1 KB                    mbarriers and the TMEM base address
constexpr int kDenseOutStage = kDenseRows * kDenseJChunk * 2;
constexpr int kDenseControl = 1024;

__host__ __device__ constexpr int dense_stage_bytes(int max_rank) {
  const int shrink = kDenseRows * kDenseKChunk * 2 + max_rank * kDenseKChunk * 2;
  const int expand = kDenseJChunk * max_rank * 2;
  const int s = shrink > expand ? shrink : expand;
  return (s + 1023) / 1024 * 1024;
}

// Instruction descriptor of tcgen05.mma kind::f16 with BF16 A and B, an fp32
// accumulator, both operands K-major: D format (F32 = 1) in bits 4-5, A format
// (BF16 = 1) in 7-9, B format in 10-12, N >> 3 in 17-22, M >> 4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

int launch_dense(const DenseArgs& a, void* stream);
// OR of the dense kernel's device status bits since the last clear (synchronizes `stream`).
int read_dense_status(void* stream, uint32_t* out, int clear);

}  // namespace glora
