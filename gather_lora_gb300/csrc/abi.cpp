// C ABI of the routed multi-LoRA fold (include/gather_lora.h): argument checks,
// launch geometry, error text, and the pure host helpers. Every check runs
// before any CUDA call, so a rejected call launches nothing.
#include "../../include/gather_lora.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "dense_types.h"
#include "fold_types.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_err[0] = '\0';
  return LORA_OK;
}

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
inline int round_up(int a, int m) { return (a + m - 1) / m * m; }
inline int round_down(int a, int m) { return a / m * m; }
inline int pow2_floor(int v) {
  int p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SMs of the current device, or `fallback` without one (host-only geometry queries).
int device_sm_count_or(int fallback) {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      v <= 0) {
    cudaGetLastError();   // clear the sticky "no device" error of the query
    return fallback;
  }
  return v;
}

// Shared-memory budgets: two CTAs per SM, or one when the fixed part is large.
// The tuning constants can be overridden at build time for measurement sweeps.
#ifndef GLORA_BUDGET_TWO_PER_SM
#define GLORA_BUDGET_TWO_PER_SM (112 * 1024)
#endif
#ifndef GLORA_STAGE_TARGET
#define GLORA_STAGE_TARGET (42 * 1024)
#endif
#ifndef GLORA_MOE_STAGE_TARGET
#define GLORA_MOE_STAGE_TARGET (56 * 1024)
#endif
#ifndef GLORA_UNIT_ROWS
#define GLORA_UNIT_ROWS 16
#endif
#ifndef GLORA_GATHER_UNIT_ROWS
#define GLORA_GATHER_UNIT_ROWS 8
#endif
#ifndef GLORA_GATHER_MAX_CL
#define GLORA_GATHER_MAX_CL 1
#endif
#ifndef GLORA_TMAP_MIN_RANK
#define GLORA_TMAP_MIN_RANK LORA_TMAP_MIN_RANK
#endif
#ifndef GLORA_DIRECT_UNITS
#define GLORA_DIRECT_UNITS 1
#endif
#ifndef GLORA_TC_SHRINK
#define GLORA_TC_SHRINK 1
#endif
#ifndef GLORA_MIN_STAGE
#define GLORA_MIN_STAGE (24 * 1024)
#endif
#ifndef GLORA_MAX_CLUSTER
#define GLORA_MAX_CLUSTER 8
#endif
#ifndef GLORA_MOE_TILE_SHRINK
#define GLORA_MOE_TILE_SHRINK 0
#endif
#ifndef GLORA_MOE_TWO_PER_SM
#define GLORA_MOE_TWO_PER_SM 1   // MoE folds with k_in > n_out use the two-CTAs-per-SM shape
#endif
#ifndef GLORA_MOE_GROUP_ROWS
#define GLORA_MOE_GROUP_ROWS 16
#endif
constexpr int kBudgetTwoPerSm = GLORA_BUDGET_TWO_PER_SM;
constexpr int kBudgetOnePerSm = 225 * 1024;
constexpr int kStageTarget = GLORA_STAGE_TARGET;
#ifndef GLORA_CLUSTER_CAP_HIGH_RANK
#define GLORA_CLUSTER_CAP_HIGH_RANK 4
#endif
constexpr int kClusterCapRank = 64;
// Rows per bgmv work unit. Measured on GB300 against 32 (rank <= 64) and 8:
// decode q_proj 10.2 -> 8.5 us, qkv 28.3 -> 25.1 us at 16; the decode gather
// fold, whose table entries hold about one row each, 27.9 -> 22.8 us at 8.
constexpr int kUnitRows = GLORA_UNIT_ROWS;
constexpr int kGatherUnitRows = GLORA_GATHER_UNIT_ROWS;
static_assert(kUnitRows <= glora::kMaxGroupRows && kGatherUnitRows <= glora::kMaxGroupRows &&
                  GLORA_MOE_GROUP_ROWS <= glora::kMaxGroupRows,
              "groups wider than the kernels' row tiles (kMaxGroupRows)");
constexpr int kClusterCapHighRank = GLORA_CLUSTER_CAP_HIGH_RANK;
// MoE groups are small and many: larger items (a whole k_in of 768 in one shrink
// item, which also lets each consumer warp own whole groups) measured 7% faster
// on the MoE down fold; the bgmv folds measured best at kStageTarget.
constexpr int kMoeStageTarget = GLORA_MOE_STAGE_TARGET;
constexpr int kMinStage = GLORA_MIN_STAGE;
constexpr int kMaxStages = 8;
constexpr int kGatherBytes = 24 * 1024;                  // largest all-gather buffer of the exchange

// Split `total` into equal chunks of at most `cap` (multiples of 16).
int balanced_chunk(int total, int cap) {
  cap = std::max(16, round_down(cap, 16));
  const int n = static_cast<int>(ceil_div(total, cap));
  return std::min(cap, round_up(static_cast<int>(ceil_div(total, n)), 16));
}

// Launch geometry. Depends only on the shapes (never on n, the routing or the
// window), so a row's arithmetic — the k-slices, k-chunks and summation order —
// is the same in every call with the same (k_in, n_out, max_rank).
bool make_geometry_at(bool moe, int rows, int max_loras, int planner_ints, int max_rank, int k_in,
                      int n_out, glora::FoldGeometry& g, int max_cl, bool a_tiled, int target, int unit_rows,
                      int cw = glora::kConsumerWarps) {
  g = glora::FoldGeometry{};
  // bgmv: a cluster splits each unit's k (shrink) and n_out (expand); MoE units
  // are many and small, so one CTA folds whole groups.
  // Clusters of at most 4 from max_rank 64 up: per k-slice a CTA then moves
  // more adapter bytes per fixed cost (planning, exchange). Measured on GB300:
  // qkv (rank 64) 33.5 -> 28.4 us and ffn (rank 128) 69.4 -> 63.4 us at 4
  // instead of 8, decode (rank 16) 10.2 -> 12.3 us. The cap depends on the
  // shapes only (a row's k-split never depends on the batch).
  if (max_rank >= kClusterCapRank) max_cl = std::min(max_cl, kClusterCapHighRank);
  g.cl = moe ? 1 : pow2_floor(std::min(max_cl, std::max(1, std::max(k_in, n_out) / 512)));
  g.mr16 = round_up(max_rank, 16);
  const int mt = g.mr16 / 16;
  const int tile_rows_cap = 8 * (glora::kMaxTilesPerWarp * cw / mt);
  if (moe) {
    g.rt = LORA_MOE_M_TILE;
    g.gmax = std::min(std::min(GLORA_MOE_GROUP_ROWS, glora::kMaxGroupRows), tile_rows_cap);
  } else {
    g.rt = unit_rows;
    g.gmax = std::min(g.rt, tile_rows_cap);
  }
  g.ksl = round_up(static_cast<int>(ceil_div(k_in, g.cl)), 16);
  g.jsl = round_up(static_cast<int>(ceil_div(n_out, g.cl)), 16);
  const int srows = g.mr16 + g.gmax;
  int kcap = g.ksl;
  if (srows * (kcap * 2 + 16) > target) {
    kcap = 16;
    static const int kCands[] = {1024, 768, 512, 384, 256, 128, 64, 32, 16};
    for (int c : kCands)
      if (c <= g.ksl && srows * (c * 2 + 16) <= target) { kcap = c; break; }
  }
  g.kch = balanced_chunk(g.ksl, kcap);
  // A as 2-D TMA boxes of 64 columns: k-chunks are whole boxes (a chunk may
  // reach past its k-slice; those columns are loaded and not used).
  g.a_tiled = a_tiled ? 1 : 0;
  if (a_tiled) g.kch = round_up(g.kch, 64);
  // A unit's items either each go to the one consumer warp that owns their
  // ring slot (many small MoE groups whose shrink is a single k-chunk: the
  // latency chains of several items overlap) or are split tile by tile over
  // all consumer warps in order (one bgmv group, or larger groups).
  const int tiles = mt * static_cast<int>(ceil_div(g.gmax, 8));
  g.group_parallel = (moe && !GLORA_MOE_TILE_SHRINK && tiles <= 4 && g.kch >= g.ksl) ? 1 : 0;
  // With cluster peers and small fp32 partials, the exchange is an all-gather
  // (one cluster barrier; each CTA adds the slots itself). Tile-parallel groups
  // of few tiles also split k over the consumer warps (ksplit k-phases of
  // kConsumerWarps / ksplit warps each) when there are no peers or the exchange
  // is an all-gather; with a reduce-scatter the extra planes would lengthen it.
  g.gather = (g.cl > 1 && g.cl * g.rt * (max_rank + 4) * 4 <= kGatherBytes) ? 1 : 0;
  // (slot-parallel groups: two warps may share a slot, each with its own plane)
  g.ksplit = g.group_parallel ? 2 : 1;
  if (!g.group_parallel && (g.cl == 1 || g.gather))
    while (g.ksplit < cw && cw % (2 * g.ksplit) == 0 && (cw / (2 * g.ksplit)) >= tiles) g.ksplit *= 2;
  g.maxt = 1;
  if (g.group_parallel) {
    while (g.maxt < tiles) g.maxt *= 2;
  } else {
    while (g.maxt * (cw / g.ksplit) < tiles) g.maxt *= 2;
  }
  // The bgmv shrink runs on tcgen05 when A comes as TMA boxes of 128 rows and
  // a unit has at most 16 rows: M = 128 (A rows), N = 16 (the unit's x rows).
  g.tc = (!moe && a_tiled && g.mr16 == 128 && g.gmax == 16 && g.ksplit == 1 && !g.group_parallel) ? GLORA_TC_SHRINK : 0;
  g.pitch_k = g.kch * 2 + 16;
  g.pitch_b = max_rank * 2 + (max_rank >= 32 ? 16 : 0);
  const int shrink_stage = a_tiled ? g.mr16 * g.kch * 2 + g.gmax * g.pitch_k : srows * g.pitch_k;
  const int S = std::max(shrink_stage, kMinStage);
  const int jcap = (S - 16 * g.gmax) / (g.pitch_b + 2 * g.gmax);
  g.jch = balanced_chunk(g.jsl, std::min(jcap, g.jsl));
  const int expand_stage = g.jch * g.pitch_b + g.gmax * (g.jch * 2 + 16);
  // (stages of tiled launches start on the 1024-byte atom of the 128-byte swizzle)
  g.stage_bytes = round_up(std::max(shrink_stage, expand_stage), a_tiled ? 1024 : 128);
  g.pitch_part = max_rank + 4;
  g.pitch_xa = max_rank * 2 + 16;
  const int planes = g.ksplit + (g.gather ? g.cl : 0);   // partial planes (+ the all-gather slots)
  const int fixed = glora::kPlanBytes + planes * g.rt * g.pitch_part * 4 + g.rt * g.pitch_xa;
  int ns = (kBudgetTwoPerSm - fixed) / g.stage_bytes;
  if (ns < 2) ns = (kBudgetOnePerSm - fixed) / g.stage_bytes;
  ns = std::min(ns, kMaxStages);
  if (ns < 2) return false;
  // the ring doubles as planning scratch (bgmv rows + slot counts / MoE offsets)
  while (ns * g.stage_bytes < planner_ints * 4 && ns < kMaxStages) ++ns;
  if (ns * g.stage_bytes < planner_ints * 4)
    g.stage_bytes = round_up(static_cast<int>(ceil_div(planner_ints * 4, ns)), a_tiled ? 1024 : 128);
  g.ns = ns;
  g.off_ring = glora::kPlanBytes;
  g.off_out = 0;
  g.off_part = g.off_ring + ns * g.stage_bytes;
  g.off_xa = g.off_part + planes * g.rt * g.pitch_part * 4;
  g.smem_bytes = g.off_xa + g.rt * g.pitch_xa;
  if (g.smem_bytes > kBudgetOnePerSm + 2048) return false;
  if (moe) {
    g.clusters = 0;   // the persistent grid and layout: moe_geometry()
  } else {
    // Direct numbering (unit s = tile 0 of slot s) plans fastest, but its empty
    // units (slots without rows) sit between the real ones in launch order.
    // When the grid is more than one wave of CTAs (two per SM) and slots are
    // many for the rows (likely empty), number the units slot by slot instead:
    // the real units come first. Both give the same rows per unit. Measured on
    // GB300: qkv (256 rows, 128 slots, 576 CTAs) 24.6 -> 21.0 us slot by slot;
    // decode (one wave) and ffn (64 slots for 512 rows) stay faster with direct
    // numbering.
    const long long units = rows / g.rt + std::min(rows, max_loras);
    const int sms = device_sm_count_or(152);
    const bool sparse_slots = 4LL * max_loras > rows && units * g.cl > 2LL * sms;
    g.direct = (GLORA_DIRECT_UNITS && max_loras <= rows && !sparse_slots) ? 1 : 0;
    g.clusters = rows <= 0 ? 0 : rows / g.rt + std::min(rows, max_loras);
  }
  return true;
}

// MoE takes the larger stage target when its geometry still fits two CTAs per
// SM (the gate/up form at k_in 2048 would drop to one and measured slower).
bool make_geometry(bool moe, int rows, int max_loras, int planner_ints, int max_rank, int k_in,
                   int n_out, glora::FoldGeometry& g, int max_cl = GLORA_MAX_CLUSTER, bool a_tiled = false,
                   int unit_rows = kUnitRows) {
  if (moe && make_geometry_at(moe, rows, max_loras, planner_ints, max_rank, k_in, n_out, g, max_cl, a_tiled,
                              kMoeStageTarget, unit_rows) &&
      g.smem_bytes <= kBudgetTwoPerSm)
    return true;
  return make_geometry_at(moe, rows, max_loras, planner_ints, max_rank, k_in, n_out, g, max_cl, a_tiled,
                          kStageTarget, unit_rows);
}

// The MoE fold's launch: the arithmetic (k chunks, shrink mode, row tiles) from
// the shapes alone, as for every fold, so a row's bits never depend on the
// window; then the persistent layout: the CTA's plan (MoePlan) before the ring,
// as many ring stages as fit the CTA shape's CTAs per SM, and a grid of one such
// CTA set per SM (fewer for small windows, at least 16 rows per CTA). Each CTA
// plans its units in the ring before its first fold (offsets, its units, the
// counts of their groups).
//
// CTA shape: two CTAs per SM of 8 + 2 warps when the shrink is the larger half
// (k_in > n_out), else one CTA per SM of 12 + 4 warps. Measured on GB300 with
// inputs-ready windows: the gate/up form (k_in 2048, n_out 768) 93.7 -> 79.6 us,
// the down form (k_in 768, n_out 2048) 86.1 -> 89.7 us.
bool moe_geometry_cfg(int cfg, int window, int adapters, int num_experts, int max_rank, int k_in, int n_out,
                      int sms, glora::FoldGeometry& g) {
  // The largest stage target whose ring still gets two stages beside the plan.
  const int budget = glora::moe_ctas_per_sm(cfg) == 1 ? kBudgetOnePerSm : kBudgetTwoPerSm;
  const int off_ring = round_up(glora::kPlanBytes + static_cast<int>(sizeof(glora::MoePlan)), 1024);
  int ns = 0, tail = 0;
  for (int target : {kMoeStageTarget, kStageTarget, kMinStage}) {
    if (!make_geometry_at(true, window, adapters, 0, max_rank, k_in, n_out, g, GLORA_MAX_CLUSTER, false, target,
                          kUnitRows, glora::moe_cw(cfg)))
      continue;
    const int planes = g.ksplit + (g.gather ? g.cl : 0);
    tail = planes * g.rt * g.pitch_part * 4 + g.rt * g.pitch_xa;
    ns = std::min(kMaxStages, (budget - off_ring - tail) / g.stage_bytes);
    if (ns >= 2) break;
  }
  if (ns < 2) return false;
  const int planes = g.ksplit + (g.gather ? g.cl : 0);
  g.moe_cfg = cfg;
  g.off_mplan = glora::kPlanBytes;
  g.off_ring = off_ring;
  g.ns = ns;
  g.off_part = g.off_ring + ns * g.stage_bytes;
  g.off_xa = g.off_part + planes * g.rt * g.pitch_part * 4;
  g.smem_bytes = g.off_xa + g.rt * g.pitch_xa;
  const long long bins = static_cast<long long>(num_experts) * adapters;
  // planner scratch: offsets, four unit arrays, the groups of a round
  const long long scratch = ((num_experts + 4) & ~3) * 4LL + (4LL * 64 + 4) * 4 +
                            ((static_cast<long long>(std::max(glora::kMoeMaxDesc, adapters)) + 4) & ~3LL) * 4;
  const long long ring = static_cast<long long>(ns) * g.stage_bytes;
  if (bins > glora::kMoeMaxBins || scratch > ring) return false;
  g.clusters = static_cast<int>(std::max<long long>(
      1, std::min<long long>(static_cast<long long>(sms) * glora::moe_ctas_per_sm(cfg), ceil_div(window, 16))));
  return true;
}

bool moe_geometry(int window, int adapters, int num_experts, int max_rank, int k_in, int n_out, int sms,
                  glora::FoldGeometry& g) {
  if (k_in > n_out && GLORA_MOE_TWO_PER_SM &&
      moe_geometry_cfg(1, window, adapters, num_experts, max_rank, k_in, n_out, sms, g))
    return true;
  return moe_geometry_cfg(0, window, adapters, num_experts, max_rank, k_in, n_out, sms, g);
}

// cuTensorMapEncodeTiled from the driver, looked up once (NULL without a driver).
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Launch geometry for a fold call, with A as tensor-map boxes when maps are given
// and max_rank >= LORA_TMAP_MIN_RANK (falls back to padded A rows otherwise, or
// when the tiled layout does not fit). Measured on GB300: at rank 16 the boxes
// (16 rows of 128 bytes) made decode-sized folds about 5% slower than one copy
// per 512-byte row, while at ranks 64 and 128 they made the folds 6-11% faster.
bool fold_geometry(bool moe, int rows, int max_loras, int planner_ints, int max_rank, int k_in, int n_out,
                   glora::FoldGeometry& g, int max_cl, const void* a_tmaps, int unit_rows = kUnitRows) {
  if (a_tmaps && max_rank >= GLORA_TMAP_MIN_RANK &&
      make_geometry(moe, rows, max_loras, planner_ints, max_rank, k_in, n_out, g, max_cl, true, unit_rows))
    return true;
  return make_geometry(moe, rows, max_loras, planner_ints, max_rank, k_in, n_out, g, max_cl, false, unit_rows);
}

int check_shape(int32_t max_rank, int32_t k_in, int32_t n_out, int64_t xs, int64_t os) {
  if (max_rank < 8 || max_rank > LORA_MAX_RANK) return fail(LORA_ERR_SIZE, "max_rank %d outside [8, %d]", max_rank, LORA_MAX_RANK);
  if (k_in < 8 || k_in > LORA_MAX_K_IN) return fail(LORA_ERR_SIZE, "k_in %d outside [8, %d]", k_in, LORA_MAX_K_IN);
  if (n_out < 8 || n_out > LORA_MAX_N_OUT) return fail(LORA_ERR_SIZE, "n_out %d outside [8, %d]", n_out, LORA_MAX_N_OUT);
  if (xs < k_in) return fail(LORA_ERR_STRIDE, "x_row_stride %lld < k_in %d", (long long)xs, k_in);
  if (os < n_out) return fail(LORA_ERR_STRIDE, "out_row_stride %lld < n_out %d", (long long)os, n_out);
  if (max_rank % 8 || k_in % 8 || n_out % 8)
    return fail(LORA_ERR_ALIGN, "max_rank, k_in and n_out must be multiples of 8 (%d, %d, %d)", max_rank, k_in, n_out);
  if (xs % 8 || os % 8)
    return fail(LORA_ERR_ALIGN, "row strides must be multiples of 8 elements (%lld, %lld)", (long long)xs, (long long)os);
  return LORA_OK;
}

int cuda_fail(int err, const char* what) {
  return fail(LORA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(static_cast<cudaError_t>(err)));
}

// ---- dense single-adapter delta ----------------------------------------------
static_assert(glora::idesc_bf16_f32(128, 64) == 0x08100490u, "instruction descriptor bit layout");

// Ranks the tensor-core path takes: the expand's K (= max_rank) is one 32- or
// 64-byte swizzle row, or whole 64-column atoms of the 128-byte swizzle, and the
// shrink's N (= max_rank) fits the TMEM partial (128 columns).
bool dense_rank(int r) { return r == 16 || r == 32 || r == 64 || r == 128; }

struct DenseGeom {
  int dense, cl, ns, stage, smem;
  long long ctas;
};

// The tensor-core launch for m rows, or false (the routed engine takes the call).
// cl: the largest power of two <= 8 with tiles * cl <= the SM count (one CTA
// per SM) and at least one k-chunk per CTA; the ring takes what shared memory
// is left (at most kDenseMaxRing stages).
bool dense_geometry(int m, int r, int k_in, int sms, DenseGeom& g) {
  g = DenseGeom{};
  if (!dense_rank(r) || m < LORA_DELTA_DENSE_MIN_ROWS) return false;
  const long long tiles = ceil_div(m, glora::kDenseRows);
  const int nkc = static_cast<int>(ceil_div(k_in, glora::kDenseKChunk));
  int cl = 1;
  while (cl < 8 && tiles * cl * 2 <= std::max(sms, 1) && cl * 2 <= nkc) cl *= 2;
  const int stage = glora::dense_stage_bytes(r);
  const int fixed = 2 * glora::kDenseOutStage + glora::kDenseRows * r * 2 + glora::kDenseControl + 1024;
  const int ns = std::min(glora::kDenseMaxRing, (227 * 1024 - fixed) / stage);
  if (ns < 2) return false;
  g.dense = 1;
  g.cl = cl;
  g.ns = ns;
  g.stage = stage;
  g.smem = fixed + ns * stage;
  g.ctas = tiles * cl;
  return true;
}

int device_sm_count() { return device_sm_count_or(0); }

// One 2-D BF16 tensor map: `inner` x `outer` elements, rows `row_bytes` apart.
int encode_map(glora::TensorMapBytes* out, const void* ptr, uint64_t inner, uint64_t outer, uint64_t row_bytes,
               uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz, const char* what) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled();
  if (!enc) return fail(LORA_ERR_CUDA, "cuTensorMapEncodeTiled is not available (no CUDA driver)");
  static_assert(sizeof(glora::TensorMapBytes) == sizeof(CUtensorMap), "tensor map size");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(reinterpret_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr),
                         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LORA_OK : fail(LORA_ERR_CUDA, "cuTensorMapEncodeTiled failed for %s (%d)", what, static_cast<int>(r));
}

}  // namespace

extern "C" {

const char* lora_last_error(void) { return g_err; }

int lora_bgmv(const lora_bf16_t* x, int64_t x_row_stride, lora_bf16_t* base_out, int64_t out_row_stride,
              const int32_t* seq_slot, int32_t n, const lora_bf16_t* const* a_table,
              const lora_bf16_t* const* b_table, const float* scale_table, int32_t max_loras,
              int32_t max_rank, int32_t k_in, int32_t n_out, lora_bf16_t* xa, const void* a_tmaps,
              uint32_t flags, void* stream) {
  if (flags & ~LORA_INPUTS_READY) return fail(LORA_ERR_FLAGS, "unknown flags 0x%x", flags);
  if (n < 0 || n > LORA_MAX_ROWS) return fail(LORA_ERR_SIZE, "n %d outside [0, %d]", n, LORA_MAX_ROWS);
  if (max_loras < 1 || max_loras > LORA_MAX_LORAS)
    return fail(LORA_ERR_SIZE, "max_loras %d outside [1, %d]", max_loras, LORA_MAX_LORAS);
  int rc = check_shape(max_rank, k_in, n_out, x_row_stride, out_row_stride);
  if (rc) return rc;
  if (n == 0) return ok();
  if (!x || !base_out || !seq_slot || !a_table || !b_table || !scale_table)
    return fail(LORA_ERR_NULL, "a required pointer is NULL (x, base_out, seq_slot, a_table, b_table, scale_table)");
  if (!aligned16(x) || !aligned16(base_out) || (xa && !aligned16(xa)))
    return fail(LORA_ERR_ALIGN, "x, base_out and xa must be 16-byte aligned");
  glora::BgmvArgs a{};
  if (a_tmaps && (reinterpret_cast<uintptr_t>(a_tmaps) & 63u))
    return fail(LORA_ERR_ALIGN, "a_tmaps must be 64-byte aligned");
  if (!fold_geometry(false, n, max_loras, ((n + 3) & ~3) + max_loras, max_rank, k_in, n_out, a.g, GLORA_MAX_CLUSTER, a_tmaps))
    return fail(LORA_ERR_SIZE, "no launch geometry fits shared memory for max_rank %d, k_in %d, n_out %d", max_rank, k_in, n_out);
  a.a_maps = a.g.a_tiled ? a_tmaps : nullptr;
  a.x = x;
  a.x_stride = x_row_stride;
  a.out = base_out;
  a.out_stride = out_row_stride;
  a.seq_slot = seq_slot;
  a.n = n;
  a.a_table = a_table;
  a.b_table = b_table;
  a.scale_table = scale_table;
  a.max_loras = max_loras;
  a.max_rank = max_rank;
  a.k_in = k_in;
  a.n_out = n_out;
  a.xa = xa;
  a.late = (flags & LORA_INPUTS_READY) ? 1 : 0;
  rc = glora::launch_bgmv(a, stream);
  return rc ? cuda_fail(rc, "lora_bgmv launch") : ok();
}

int lora_moe_grouped_fold(const lora_bf16_t* x, int64_t x_row_stride, int32_t x_gather,
                          lora_bf16_t* base_out, int64_t out_row_stride, const int32_t* expert_offsets, int32_t num_experts,
                          const int32_t* sorted_token_ids, int32_t te, const int32_t* row_adapter,
                          int32_t num_tokens, int32_t row_offset, int32_t row_end,
                          const lora_bf16_t* const* a_table, const lora_bf16_t* const* b_table,
                          const float* scale_table, int32_t max_loras, int32_t max_rank, int32_t k_in,
                          int32_t n_out, lora_bf16_t* xa, int32_t xa_rows, uint32_t flags, void* stream) {
  if (flags & ~LORA_INPUTS_READY) return fail(LORA_ERR_FLAGS, "unknown flags 0x%x", flags);
  if (num_experts < 1 || num_experts > LORA_MAX_EXPERTS)
    return fail(LORA_ERR_SIZE, "num_experts %d outside [1, %d]", num_experts, LORA_MAX_EXPERTS);
  if (max_loras < 1 || max_loras > LORA_MAX_LORAS)
    return fail(LORA_ERR_SIZE, "max_loras %d outside [1, %d]", max_loras, LORA_MAX_LORAS);
  if (static_cast<int64_t>(max_loras) * num_experts > LORA_MAX_LORAS)
    return fail(LORA_ERR_SIZE, "max_loras %d x num_experts %d outside [1, %d] table entries", max_loras,
                num_experts, LORA_MAX_LORAS);
  if (te < 0 || num_tokens < 0) return fail(LORA_ERR_SIZE, "te %d and num_tokens %d must be >= 0", te, num_tokens);
  if (row_offset < 0 || row_end < row_offset || row_end > te)
    return fail(LORA_ERR_WINDOW, "window [%d, %d) outside [0, te=%d]", row_offset, row_end, te);
  int rc = check_shape(max_rank, k_in, n_out, x_row_stride, out_row_stride);
  if (rc) return rc;
  if (!x || !base_out || !expert_offsets || !a_table || !b_table || !scale_table)
    return fail(LORA_ERR_NULL, "a required pointer is NULL (x, base_out, expert_offsets, a_table, b_table, scale_table)");
  if ((row_adapter || x_gather) && !sorted_token_ids)
    return fail(LORA_ERR_NULL, "sorted_token_ids is required with row_adapter or x_gather");
  if (xa && (xa_rows < 0 || xa_rows < row_end - row_offset))
    return fail(LORA_ERR_SIZE, "xa holds %d rows, the window [%d, %d) writes %d", xa_rows, row_offset, row_end,
                row_end - row_offset);
  if (!aligned16(x) || !aligned16(base_out) || (xa && !aligned16(xa)))
    return fail(LORA_ERR_ALIGN, "x, base_out and xa must be 16-byte aligned");
  glora::MoeArgs a{};
  const int adapters = row_adapter ? max_loras : 1;
  if (!moe_geometry(row_end - row_offset, adapters, num_experts, max_rank, k_in, n_out, device_sm_count_or(152), a.g))
    return fail(LORA_ERR_SIZE, "no launch geometry for %d experts x %d adapters at max_rank %d, k_in %d, n_out %d "
                "(shared memory)", num_experts, adapters, max_rank, k_in, n_out);
  a.adapters = adapters;
  a.x = x;
  a.x_stride = x_row_stride;
  a.out = base_out;
  a.out_stride = out_row_stride;
  a.expert_offsets = expert_offsets;
  a.num_experts = num_experts;
  a.sorted_token_ids = sorted_token_ids;
  a.row_adapter = row_adapter;
  a.num_tokens = num_tokens;
  a.x_gather = x_gather ? 1 : 0;
  a.row_offset = row_offset;
  a.row_end = row_end;
  a.a_table = a_table;
  a.b_table = b_table;
  a.scale_table = scale_table;
  a.max_loras = max_loras;
  a.max_rank = max_rank;
  a.k_in = k_in;
  a.n_out = n_out;
  a.xa = xa;
  a.late = (flags & LORA_INPUTS_READY) ? 1 : 0;
  rc = glora::launch_moe(a, stream);
  return rc ? cuda_fail(rc, "lora_moe_grouped_fold launch") : ok();
}

int lora_moe_gather_bgmv(const lora_bf16_t* x, int64_t x_row_stride, lora_bf16_t* base_out,
                         int64_t out_row_stride, const int32_t* indices, int32_t n_rows, int32_t top_k,
                         const int32_t* row_adapter, int32_t num_tokens, int32_t num_experts,
                         const lora_bf16_t* const* a_table, const lora_bf16_t* const* b_table,
                         const float* scale_table, int32_t max_loras, int32_t max_rank, int32_t k_in,
                         int32_t n_out, lora_bf16_t* xa, const void* a_tmaps, uint32_t flags, void* stream) {
  if (flags & ~LORA_INPUTS_READY) return fail(LORA_ERR_FLAGS, "unknown flags 0x%x", flags);
  if (n_rows < 0 || n_rows > LORA_MAX_ROWS) return fail(LORA_ERR_SIZE, "n_rows %d outside [0, %d]", n_rows, LORA_MAX_ROWS);
  if (top_k < 1) return fail(LORA_ERR_SIZE, "top_k %d < 1", top_k);
  if (num_tokens < 0) return fail(LORA_ERR_SIZE, "num_tokens %d < 0", num_tokens);
  if (num_experts < 1 || num_experts > LORA_MAX_EXPERTS)
    return fail(LORA_ERR_SIZE, "num_experts %d outside [1, %d]", num_experts, LORA_MAX_EXPERTS);
  if (max_loras < 1 || static_cast<int64_t>(max_loras) * num_experts > LORA_MAX_LORAS)
    return fail(LORA_ERR_SIZE, "max_loras %d x num_experts %d outside [1, %d] table entries", max_loras,
                num_experts, LORA_MAX_LORAS);
  int rc = check_shape(max_rank, k_in, n_out, x_row_stride, out_row_stride);
  if (rc) return rc;
  if (n_rows == 0) return ok();
  if (!x || !base_out || !indices || !a_table || !b_table || !scale_table)
    return fail(LORA_ERR_NULL, "a required pointer is NULL (x, base_out, indices, a_table, b_table, scale_table)");
  if (!aligned16(x) || !aligned16(base_out) || (xa && !aligned16(xa)))
    return fail(LORA_ERR_ALIGN, "x, base_out and xa must be 16-byte aligned");
  const int tables = max_loras * num_experts;
  glora::BgmvArgs a{};
  // Decode MoE rows spread over many (adapter, expert) entries of about one row
  // each: one CTA per unit (no cluster split) keeps the grid near one wave.
  if (a_tmaps && (reinterpret_cast<uintptr_t>(a_tmaps) & 63u))
    return fail(LORA_ERR_ALIGN, "a_tmaps must be 64-byte aligned");
  if (!fold_geometry(false, n_rows, tables, ((n_rows + 3) & ~3) + tables, max_rank, k_in, n_out, a.g, GLORA_GATHER_MAX_CL, a_tmaps,
                     kGatherUnitRows))
    return fail(LORA_ERR_SIZE, "no launch geometry fits shared memory for max_rank %d, k_in %d, n_out %d", max_rank, k_in, n_out);
  a.x = x;
  a.x_stride = x_row_stride;
  a.out = base_out;
  a.out_stride = out_row_stride;
  a.seq_slot = nullptr;
  a.a_maps = a.g.a_tiled ? a_tmaps : nullptr;
  a.n = n_rows;
  a.indices = indices;
  a.row_adapter = row_adapter;
  a.top_k = top_k;
  a.num_tokens = num_tokens;
  a.num_experts = num_experts;
  a.a_table = a_table;
  a.b_table = b_table;
  a.scale_table = scale_table;
  a.max_loras = tables;
  a.max_rank = max_rank;
  a.k_in = k_in;
  a.n_out = n_out;
  a.xa = xa;
  a.late = (flags & LORA_INPUTS_READY) ? 1 : 0;
  rc = glora::launch_bgmv(a, stream);
  return rc ? cuda_fail(rc, "lora_moe_gather_bgmv launch") : ok();
}

int lora_delta(const lora_bf16_t* x, int64_t x_row_stride, lora_bf16_t* base_out, int64_t out_row_stride,
               int32_t m, const lora_bf16_t* a, const lora_bf16_t* b, float scale, int32_t max_rank,
               int32_t k_in, int32_t n_out, lora_bf16_t* xa, void* stream) {
  if (m < 0 || m > LORA_MAX_DELTA_ROWS) return fail(LORA_ERR_SIZE, "m %d outside [0, %d]", m, LORA_MAX_DELTA_ROWS);
  int rc = check_shape(max_rank, k_in, n_out, x_row_stride, out_row_stride);
  if (rc) return rc;
  if (m == 0) return ok();
  if (!x || !base_out || !a || !b) return fail(LORA_ERR_NULL, "a required pointer is NULL (x, base_out, a, b)");
  if (!aligned16(x) || !aligned16(base_out) || !aligned16(a) || !aligned16(b) || (xa && !aligned16(xa)))
    return fail(LORA_ERR_ALIGN, "x, base_out, a, b and xa must be 16-byte aligned");
  DenseGeom dg;
  if (dense_geometry(m, max_rank, k_in, device_sm_count(), dg)) {
    glora::DenseArgs d{};
    const CUtensorMapSwizzle bswz = max_rank >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                    : (max_rank == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    if ((rc = encode_map(&d.map_x, x, k_in, m, x_row_stride * 2, 64, glora::kDenseRows, CU_TENSOR_MAP_SWIZZLE_128B, "x")) ||
        (rc = encode_map(&d.map_a, a, k_in, max_rank, static_cast<uint64_t>(k_in) * 2, 64, max_rank,
                         CU_TENSOR_MAP_SWIZZLE_128B, "A")) ||
        (rc = encode_map(&d.map_b, b, max_rank, n_out, static_cast<uint64_t>(max_rank) * 2, std::min(max_rank, 64),
                         glora::kDenseJChunk, bswz, "B")) ||
        (rc = encode_map(&d.map_out, base_out, n_out, m, out_row_stride * 2, 64, glora::kDenseRows,
                         CU_TENSOR_MAP_SWIZZLE_128B, "base_out")))
      return rc;
    d.xa = xa;
    d.scale = scale;
    d.m = m;
    d.k_in = k_in;
    d.n_out = n_out;
    d.max_rank = max_rank;
    d.cl = dg.cl;
    d.ns = dg.ns;
    d.stage_bytes = dg.stage;
    d.smem_bytes = dg.smem;
    rc = glora::launch_dense(d, stream);
    return rc ? cuda_fail(rc, "lora_delta launch") : ok();
  }
  // Small m, or a rank the tensor-core path does not take: the routed engine
  // with every row on one slot (one launch per LORA_MAX_ROWS rows).
  for (int32_t r0 = 0; r0 < m; r0 += LORA_MAX_ROWS) {
    const int32_t n = std::min<int32_t>(LORA_MAX_ROWS, m - r0);
    glora::BgmvArgs g{};
    if (!fold_geometry(false, n, 1, ((n + 3) & ~3) + 1, max_rank, k_in, n_out, g.g, GLORA_MAX_CLUSTER, nullptr))
      return fail(LORA_ERR_SIZE, "no launch geometry fits shared memory for max_rank %d, k_in %d, n_out %d", max_rank, k_in, n_out);
    g.x = x + static_cast<long long>(r0) * x_row_stride;
    g.x_stride = x_row_stride;
    g.out = base_out + static_cast<long long>(r0) * out_row_stride;
    g.out_stride = out_row_stride;
    g.single = 1;
    g.one_a = a;
    g.one_b = b;
    g.one_scale = scale;
    g.n = n;
    g.max_loras = 1;
    g.max_rank = max_rank;
    g.k_in = k_in;
    g.n_out = n_out;
    g.xa = xa ? xa + static_cast<long long>(r0) * max_rank : nullptr;
    rc = glora::launch_bgmv(g, stream);
    if (rc) return cuda_fail(rc, "lora_delta launch");
  }
  return ok();
}

int lora_delta_geometry(int32_t m, int32_t max_rank, int32_t k_in, int32_t n_out, int32_t sm_count, int64_t out[6]) {
  if (!out) return fail(LORA_ERR_NULL, "out is NULL");
  if (m < 0 || m > LORA_MAX_DELTA_ROWS) return fail(LORA_ERR_SIZE, "m %d outside [0, %d]", m, LORA_MAX_DELTA_ROWS);
  const int rc = check_shape(max_rank, k_in, n_out, k_in, n_out);
  if (rc) return rc;
  DenseGeom dg;
  const int sms = sm_count > 0 ? sm_count : device_sm_count();
  int64_t v[6] = {0, 0, 0, 0, 0, 0};
  if (dense_geometry(m, max_rank, k_in, sms, dg)) {
    v[0] = 1; v[1] = dg.cl; v[2] = dg.ns; v[3] = dg.stage; v[4] = dg.smem; v[5] = dg.ctas;
  } else {
    glora::FoldGeometry g{};
    const int n = std::max(1, std::min<int32_t>(m, LORA_MAX_ROWS));
    if (!fold_geometry(false, n, 1, ((n + 3) & ~3) + 1, max_rank, k_in, n_out, g, GLORA_MAX_CLUSTER, nullptr))
      return fail(LORA_ERR_SIZE, "no launch geometry fits shared memory");
    v[1] = g.cl; v[2] = g.ns; v[3] = g.stage_bytes; v[4] = g.smem_bytes; v[5] = static_cast<int64_t>(g.clusters) * g.cl;
  }
  std::memcpy(out, v, sizeof v);
  return ok();
}

int lora_selftest_wait_timeout(int64_t limit_cycles, void* stream) {
  if (limit_cycles < 1 || limit_cycles > (int64_t{1} << 32))
    return fail(LORA_ERR_SIZE, "limit_cycles %lld outside [1, 2^32]", static_cast<long long>(limit_cycles));
  const int rc = glora::launch_wait_selftest(limit_cycles, stream);
  return rc ? cuda_fail(rc, "lora_selftest_wait_timeout launch") : ok();
}

int lora_read_device_status(void* stream, uint32_t* status_out, int clear) {
  if (!status_out) return fail(LORA_ERR_NULL, "status_out is NULL");
  uint32_t a = 0, b = 0;
  int rc = glora::read_device_status(stream, &a, clear);
  if (!rc) rc = glora::read_dense_status(stream, &b, clear);
  *status_out = a | b;
  return rc ? cuda_fail(rc, "lora_read_device_status") : ok();
}

int lora_launch_geometry(int moe, int32_t rows, int32_t max_loras, int32_t max_rank, int32_t k_in,
                         int32_t n_out, int64_t out[12]) {
  if (!out) return fail(LORA_ERR_NULL, "out is NULL");
  int rc = check_shape(max_rank, k_in, n_out, k_in, n_out);
  if (rc) return rc;
  glora::FoldGeometry g{};
  const int kind = moe & 15;
  const bool grouped = kind == 1;
  // stands for a tensor-map array (only its presence matters); the grouped fold takes none
  static const char kAnyMaps = 0;
  if (grouped ? !moe_geometry(std::max(rows, 0), max_loras, 1, max_rank, k_in, n_out, device_sm_count_or(152), g)
              : !fold_geometry(false, rows, max_loras, ((rows + 3) & ~3) + max_loras, max_rank, k_in, n_out, g,
                               kind == 2 ? GLORA_GATHER_MAX_CL : GLORA_MAX_CLUSTER,
                               (moe & 16) ? &kAnyMaps : nullptr, kind == 2 ? kGatherUnitRows : kUnitRows))
    return fail(LORA_ERR_SIZE, "no launch geometry fits shared memory and the grid size");
  const int64_t v[12] = {g.cl, g.rt, g.ksl, g.jsl, g.kch, g.jch, g.ns, g.clusters, g.smem_bytes, g.a_tiled, g.tc,
                         grouped ? g.moe_cfg : g.direct};
  std::memcpy(out, v, sizeof v);
  return ok();
}

int32_t lora_grouped_down_wc(int32_t row_offset, int32_t row_end) {
  if (row_end < row_offset) return -1;
  const int64_t span = static_cast<int64_t>(row_end) - row_offset;
  return static_cast<int32_t>(std::max<int64_t>(1, (span + LORA_MOE_M_TILE - 1) / LORA_MOE_M_TILE));
}

int32_t lora_gather_row_token(int32_t row, int32_t top_k) {
  if (row < 0 || top_k < 1) return -1;
  return row / top_k;
}

int lora_gather_bgmv_grids(int32_t max_rank, int32_t n_out, int32_t n_slots, int32_t shrink[3],
                           int32_t expand[3]) {
  if (max_rank < 1 || n_out < 1 || n_slots < 0 || !shrink || !expand) return -1;
  shrink[0] = (max_rank + 3) / 4;
  shrink[1] = n_slots;
  shrink[2] = 1;
  expand[0] = static_cast<int32_t>((static_cast<int64_t>(n_out) + 3) / 4);
  expand[1] = n_slots;
  expand[2] = 1;
  return 0;
}

int lora_encode_a_tmaps(const uint64_t* a_ptrs, int32_t count, int32_t max_rank, int32_t k_in,
                        void* maps_out) {
  if (count < 0) return fail(LORA_ERR_SIZE, "count %d < 0", count);
  if (max_rank < 8 || max_rank > LORA_MAX_RANK) return fail(LORA_ERR_SIZE, "max_rank %d outside [8, %d]", max_rank, LORA_MAX_RANK);
  if (k_in < 8 || k_in > LORA_MAX_K_IN) return fail(LORA_ERR_SIZE, "k_in %d outside [8, %d]", k_in, LORA_MAX_K_IN);
  if (k_in % 8) return fail(LORA_ERR_ALIGN, "k_in %d must be a multiple of 8", k_in);
  if (count == 0) return ok();
  if (!a_ptrs || !maps_out) return fail(LORA_ERR_NULL, "a_ptrs and maps_out are required");
  if (reinterpret_cast<uintptr_t>(maps_out) & 63u) return fail(LORA_ERR_ALIGN, "maps_out must be 64-byte aligned");
  const PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled();
  if (!enc) return fail(LORA_ERR_CUDA, "cuTensorMapEncodeTiled is not available (no CUDA driver)");
  const int mr16 = (max_rank + 15) / 16 * 16;
  auto* maps = static_cast<CUtensorMap*>(maps_out);
  for (int32_t i = 0; i < count; ++i) {
    std::memset(&maps[i], 0, sizeof(CUtensorMap));
    if (a_ptrs[i] == 0) continue;
    if (a_ptrs[i] & 15u) return fail(LORA_ERR_ALIGN, "A pointer %d is not 16-byte aligned", i);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k_in), static_cast<cuuint64_t>(max_rank)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(k_in) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(mr16)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(&maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, reinterpret_cast<void*>(a_ptrs[i]), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LORA_ERR_CUDA, "cuTensorMapEncodeTiled failed for A pointer %d (%d)", i, static_cast<int>(r));
  }
  return ok();
}

int32_t lora_grouped_down_windows(int32_t total_rows, int32_t cap, int32_t* starts, int32_t* ends,
                                  int32_t max_windows) {
  if (cap < 1 || total_rows < 0) return -1;
  const int64_t count = (static_cast<int64_t>(total_rows) + cap - 1) / cap;
  if (count > max_windows) return -2;
  if (count > 0 && (!starts || !ends)) return -1;
  for (int64_t w = 0; w < count; ++w) {
    starts[w] = static_cast<int32_t>(w * cap);
    ends[w] = static_cast<int32_t>(std::min<int64_t>(static_cast<int64_t>(total_rows), (w + 1) * cap));
  }
  return static_cast<int32_t>(count);
}

int lora_pack_expert_tables(const int32_t* expert_ids, const uint64_t* a_addrs, const uint64_t* b_addrs,
                            const float* scales, int32_t n_entries, uint64_t* a_table, uint64_t* b_table,
                            float* scale_table, int32_t table_len, int32_t* n_experts_out) {
  if (!n_experts_out) return -1;
  *n_experts_out = 0;
  if (n_entries <= 0) return 1;
  if (!expert_ids || !a_addrs || !b_addrs || !scales || !a_table || !b_table || !scale_table) return -1;
  int32_t n_experts = 0;
  for (int32_t i = 0; i < n_entries; ++i) {
    if (expert_ids[i] < 0) return -1;
    n_experts = std::max(n_experts, expert_ids[i] + 1);
  }
  if (table_len < n_experts) return -2;
  for (int32_t e = 0; e < n_experts; ++e) {
    a_table[e] = 0;
    b_table[e] = 0;
    scale_table[e] = 0.0f;
  }
  for (int32_t i = 0; i < n_entries; ++i) {  // later entries replace earlier ones
    a_table[expert_ids[i]] = a_addrs[i];
    b_table[expert_ids[i]] = b_addrs[i];
    scale_table[expert_ids[i]] = scales[i];
  }
  *n_experts_out = n_experts;
  return 0;
}

}  // extern "C"
