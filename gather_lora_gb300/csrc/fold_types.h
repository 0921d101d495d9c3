// Plain structs shared by the host launcher (abi.cpp) and the kernels.
#pragma once

#include <stdint.h>

namespace glora {

constexpr int kMaxGroupRows = 16;  // rows of one group (one adapter's rows folded together)
constexpr int kMaxRows = 64;        // rows (positions) per pass of a work unit
constexpr int kMaxTilesPerWarp = 4; // 16x8 shrink tiles a warp may own: MT * NT <= 32
constexpr int kPlanBytes = 4096;    // shared memory reserved for the work-unit plan
constexpr int kMoeMaxDesc = 128;    // MoE: (expert, adapter) groups (runs) one CTA plans per round
#ifndef GLORA_MOE_ROUND_ROWS
#define GLORA_MOE_ROUND_ROWS 512
#endif
constexpr int kMoeMaxPos = GLORA_MOE_ROUND_ROWS;   // MoE: rows one CTA scans (so at most folds) per round
constexpr int kMoeMaxBins = 4096;   // MoE: (expert, adapter) groups of a window (num_experts * adapters)
#ifndef GLORA_CONSUMER_WARPS
#define GLORA_CONSUMER_WARPS 8
#endif
#ifndef GLORA_PRODUCER_WARPS
#define GLORA_PRODUCER_WARPS 4
#endif
constexpr int kConsumerWarps = GLORA_CONSUMER_WARPS;   // tensor-core / fold warps per CTA (routed folds)
constexpr int kProducerWarps = GLORA_PRODUCER_WARPS;   // TMA-issuing warps per CTA
constexpr int kMaxWarps = 16;                                 // most warps of any fold CTA

// The MoE fold's CTA shapes (FoldGeometry::moe_cfg): 0 = one CTA per SM with
// 12 consumer and 4 producer warps; 1 = two CTAs per SM with 8 consumer and 2
// producer warps (more CTAs in flight, half the ring each).
template <int CFG> struct MoeShape;
template <> struct MoeShape<0> { static constexpr int cw = 12, pw = 4, ctas = 1, threads = (cw + pw) * 32; };
template <> struct MoeShape<1> { static constexpr int cw = 8, pw = 2, ctas = 2, threads = (cw + pw) * 32; };
constexpr int moe_cw(int cfg) { return cfg ? MoeShape<1>::cw : MoeShape<0>::cw; }
constexpr int moe_ctas_per_sm(int cfg) { return cfg ? MoeShape<1>::ctas : MoeShape<0>::ctas; }

// Launch geometry and shared-memory layout of one fold launch. Every CTA of a
// cluster of `cl` CTAs owns one k-slice of the shrink (ksl columns of A / x)
// and one j-slice of the expand (jsl rows of B / columns of out). Inputs
// stream through a ring of `ns` stages of `stage_bytes`.
struct FoldGeometry {
  int cl;           // CTAs per cluster
  int rt;           // rows per pass of a work unit (<= kMaxRows)
  int ksl, jsl;     // k-slice / j-slice per CTA (multiples of 16)
  int kch, jch;     // k columns / B rows per ring stage (multiples of 16)
  int ns;           // ring depth (>= 2)
  int gmax;         // most rows in one group (<= 32; MT * ceil(gmax/8) <= 8 * maxt shrink tiles)
  int maxt;         // shrink tiles per consumer warp the kernel instance holds (1, 2, 4)
  int group_parallel;  // 1: each consumer warp owns whole groups; 0: warps split every item's tiles
  int ksplit;       // tile-parallel: k-phases the consumer warps form (1, 2, 4, 8; partial planes of part_s)
  int direct;       // bgmv: unit s < max_loras is tile 0 of slot s (max_loras <= rows)
  int gather;       // exchange by all-gather of fp32 partials into cl planes after the k-phase planes
  int a_tiled;      // shrink stages hold A as 2-D TMA boxes (kch/64 boxes of mr16 rows x 128 B,
                    // 128-byte swizzle) ahead of the padded x rows; 0: padded A rows
  int tc;           // bgmv shrink on tcgen05 (a_tiled, mr16 == 128, gmax == 16): the x rows are
                    // placed as 128-byte-swizzled 64-column atoms of gmax rows after the A boxes
  int mr16;         // max_rank rounded up to 16
  int pitch_k;      // bytes per A or x row in a shrink stage (kch*2 + 16)
  int pitch_b;      // bytes per B row in an expand stage
  int pitch_out;    // bytes per staged out row (jsl*2 + 16)
  int pitch_part;   // floats per partial-sum row (max_rank + 4)
  int pitch_xa;     // bytes per xa row (max_rank*2 + 16)
  int stage_bytes;
  int off_ring, off_out, off_part, off_xa, smem_bytes;
  int off_mplan;    // MoE: the CTA's planned row runs and rows (MoePlan), before the ring
  int moe_cfg;      // MoE: the CTA shape (MoeShape)
  int clusters;     // grid = clusters * cl CTAs
};

struct BgmvArgs {
  const uint16_t* x;
  long long x_stride;
  uint16_t* out;
  long long out_stride;
  const void* a_maps;        // [max_loras] 128-byte A tensor maps (a_tiled), or NULL
  const int32_t* seq_slot;   // slot per row, or NULL: derived from the MoE decode routing below
  int single;                // 1: every row uses slot 0, whose entries are one_a / one_b / one_scale
  const uint16_t* one_a;
  const uint16_t* one_b;
  float one_scale;
  int n;
  const int32_t* indices;    // MoE decode rows: expert per row
  const int32_t* row_adapter;  // [num_tokens] adapter per token (NULL: adapter 0)
  int top_k, num_tokens, num_experts;
  const uint16_t* const* a_table;
  const uint16_t* const* b_table;
  const float* scale_table;
  int max_loras;
  int max_rank, k_in, n_out;
  uint16_t* xa;
  int late;                  // 1: wait for the previous grid only before touching base_out or xa
  FoldGeometry g;
};

struct MoeArgs {
  const uint16_t* x;
  long long x_stride;
  uint16_t* out;
  long long out_stride;
  const int32_t* expert_offsets;
  int num_experts;
  const int32_t* sorted_token_ids;
  const int32_t* row_adapter;
  int num_tokens;
  int x_gather;     // 1: x is token-major; sorted row r reads row sorted_token_ids[r]
  int row_offset, row_end;
  int adapters;     // adapters the routing distinguishes: max_loras with a row_adapter, else 1
  int late;         // 1: wait for the previous grid only before touching base_out or xa
  const uint16_t* const* a_table;
  const uint16_t* const* b_table;
  const float* scale_table;
  int max_loras;
  int max_rank, k_in, n_out;
  uint16_t* xa;
  FoldGeometry g;
};

// MoE fold: one run of an (expert, adapter) group's rows planned for a CTA, and
// the CTA's plan of one round (its runs and their rows, run after run).
struct MoeDesc {
  int e, a;                // expert, adapter
  int n;                   // its rows
  int pos0;                // first position of the run in the CTA's row list
  float scale;
  const uint16_t* A;       // NULL: entry NULL or misaligned (the rows stay unchanged)
  const uint16_t* B;
};
struct MoePlan {
  int nd, npos;
  MoeDesc desc[kMoeMaxDesc];
  int pos_row[kMoeMaxPos];     // sorted row of each position
  int pos_tok[kMoeMaxPos];     // its token (the x row of the gate/up form)
  short pos_desc[kMoeMaxPos];  // its run
};

// Launchers (kernels.cu). Return 0 or a cudaError_t value.
int launch_bgmv(const BgmvArgs& a, void* stream);
int launch_moe(const MoeArgs& a, void* stream);
int read_device_status(void* stream, uint32_t* out, int clear);
int launch_wait_selftest(long long limit_cycles, void* stream);

}  // namespace glora
