// Fold kernels for sm_103a: routed bgmv and MoE grouped fold.
//
// Method (pages): "Function apply_lora_bgmv" rustdoc (spark_model lora_delta) —
// per row, shrink x @ A_s^T to BF16 xa, expand xa @ B_s^T, round the delta to
// BF16, then out += scale_s * delta in fp32; "Module moe_lora_grouped" rustdoc —
// the same fold over expert-sorted rows of a window, keyed by expert and gated
// per token by moe_row_adapter.
//
// GB300 design (one launch per call, no global scratch):
//   * A cluster of `cl` CTAs owns one WORK UNIT: bgmv, up to 16 rows of one
//     slot (8 for the decode gather fold); MoE, the rows of one adapter in a
//     tile of 64-256 sorted rows, folded in passes and split into groups of
//     one expert. CTA c of the cluster takes k-slice c of the shrink and
//     j-slice c of the expand; every CTA builds the same plan from the routing
//     data.
//   * A producer warpgroup per CTA streams the unit's data into a ring of
//     shared-memory stages (full / empty mbarriers): rows by 1-D TMA bulk
//     copies (16-byte cp.async below kTmaRowBytes), A as 2-D swizzled TMA
//     boxes when tensor maps are given. Each item's copies are spread over
//     the four warps, because the request rate of one issuing warp, not HBM,
//     limits small copies: first [group, k-chunk] items (A of this CTA's
//     k-slice and the group's x rows), then [group, j-chunk] items (B rows of
//     this CTA's j-slice and the matching out-row segments).
//   * Eight consumer warps contract each shrink item on the tensor cores:
//     mma.sync BF16 with fp32 accumulation, or (A boxes of 128 rows, units of
//     at most 16 rows) one tcgen05.mma per k-step into TMEM. The fp32
//     partials of the cl k-slices are combined in distributed shared memory
//     in rank order (an all-gather when they are small, else a reduce-scatter
//     whose BF16 result is pushed to every CTA) and rounded to BF16 once.
//   * For each expand item the consumers compute d = bf16(xa @ B^T), fold
//     out = bf16(fma(scale, d, out)) against the staged out segment in
//     registers, and store the result straight to global memory (the stage is
//     only read, so it can be refilled by TMA without a proxy fence).
// A row's fp32 summation order is fixed by (k_in, max_rank, cl, k chunking):
// it never depends on which other rows share its launch, group or tile.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <limits.h>

#include "common.cuh"
#include "tc05.cuh"

#include <type_traits>
#include "fold_types.h"

namespace cg = cooperative_groups;

// Device status word (LORA_DEV_* bits), read and cleared through read_device_status().
__device__ unsigned int g_lora_status = 0;

// Phase trace (diagnostic builds only, -DGLORA_TRACE=1; gather_lora_gb300/phase_trace.py):
// one row of SM-clock stamps per CTA, written by one thread at each phase
// boundary. Slots: 0 entry, 1 past the entry wait, 2 planned (engine entry),
// 3 the producer's first item issued, 4 shrink done, 5 exchange done, 6 first
// expand data, 7 expand done, 8 exit; 9/10 global timer (ns) at entry/exit;
// 11 rows the CTA's last pass folded. A later pass of the same CTA overwrites
// its engine stamps.
#ifndef GLORA_TRACE
#define GLORA_TRACE 0
#endif
#if GLORA_TRACE
constexpr int kTraceCtas = 4096, kTraceSlots = 12;
__device__ unsigned long long g_lora_trace[kTraceCtas][kTraceSlots];
#define GLORA_STAMP(cond, slot)                                                                  \
  do {                                                                                           \
    if ((cond) && blockIdx.x < kTraceCtas) g_lora_trace[blockIdx.x][slot] = clock64();          \
  } while (0)
#define GLORA_GTIME(cond, slot)                                                                  \
  do {                                                                                           \
    if ((cond) && blockIdx.x < kTraceCtas) {                                                     \
      unsigned long long t_;                                                                     \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                                     \
      g_lora_trace[blockIdx.x][slot] = t_;                                                       \
    }                                                                                            \
  } while (0)
#define GLORA_NOTE(cond, slot, v)                                                                \
  do {                                                                                           \
    if ((cond) && blockIdx.x < kTraceCtas) g_lora_trace[blockIdx.x][slot] = (v);                 \
  } while (0)
extern "C" int lora_trace_copy(void* dst, int bytes) {
  return static_cast<int>(cudaMemcpyFromSymbol(dst, g_lora_trace, bytes));
}
extern "C" int lora_trace_clear(void) {
  static unsigned long long zero[kTraceCtas][kTraceSlots];
  return static_cast<int>(cudaMemcpyToSymbol(g_lora_trace, zero, sizeof zero));
}
#else
#define GLORA_STAMP(cond, slot) do { } while (0)
#define GLORA_GTIME(cond, slot) do { } while (0)
#define GLORA_NOTE(cond, slot, v) do { } while (0)
#endif

namespace glora {

constexpr unsigned kDevMisaligned = 0x1u;
constexpr unsigned kDevTimeout = 0x2u;
constexpr int kMaxStages = 8;
// Rows of at least kTmaRowBytes go by 1-D TMA, shorter ones by 16-byte
// cp.async (measured on GB300: moving the 1 KB decode rows to cp.async made the
// decode fold 8.5 -> 9.4 us).
#ifndef GLORA_TMA_ROW_BYTES
#define GLORA_TMA_ROW_BYTES 128
#endif
constexpr int kTmaRowBytes = GLORA_TMA_ROW_BYTES;

// Work-unit plan, identical in every CTA of a cluster.
struct Plan {
  unsigned long long full[kMaxStages];   // mbarriers: stage filled (TMA bytes landed)
  unsigned long long empty[kMaxStages];  // mbarriers: stage released by the consumer warps
  int G;                           // groups (0: nothing to do)
  int NV;                          // valid positions (sum of group sizes)
  int failed;                      // an mbarrier wait gave up: no further stores
  int warp_sums[kMaxWarps];
  int found_slot, found_tile;      // bgmv planning scratch
  int members[kMaxRows];           // positions, grouped, ascending within a group
  int gstart[kMaxRows + 1];        // group g = members[gstart[g] .. gstart[g+1])
  int grow[kMaxRows];              // position -> row of base_out
  int xsrc[kMaxRows];              // position -> row of x
  int xarow[kMaxRows];             // position -> row of xa
  int flag[kMaxRows];              // MoE: the expert where a position starts a group, else -1
  unsigned ballots[2];
  float gscale[kMaxRows];
  const uint16_t* gA[kMaxRows];
  const uint16_t* gB[kMaxRows];
  const void* gmap[kMaxRows];      // the group's A tensor map (a_tiled launches)
  unsigned long long tc_done;      // tcgen05 shrink: the unit's partial is in TMEM
  uint32_t tmem;                   // tcgen05 shrink: TMEM base address
};

static_assert(sizeof(Plan) <= kPlanBytes, "plan does not fit its shared-memory reservation");

struct EngineArgs {
  const uint16_t* x;
  long long x_stride;
  uint16_t* out;
  long long out_stride;
  uint16_t* xa;
  int max_rank, k_in, n_out;
  int late;   // wait for the previous grid on the stream only before base_out or xa is touched
};

__device__ __forceinline__ void record_timeout(Plan& pl) {
  atomicOr(&g_lora_status, kDevTimeout);
  pl.failed = 1;
}

// Launches with A as swizzled TMA boxes need the ring on a 1024-byte boundary
// (the 128-byte swizzle atom). If the dynamic shared memory were placed
// otherwise, fold nothing and report it instead of issuing the copies.
__device__ __forceinline__ bool tiled_smem_ok(const FoldGeometry& g, const unsigned char* smem) {
  if (!g.a_tiled || ((smem_u32(smem) + g.off_ring) & 1023u) == 0) return true;
  if (threadIdx.x == 0) atomicOr(&g_lora_status, kDevMisaligned);
  return false;
}

// The ring's mbarriers, initialized once per CTA; passes of a work unit keep
// counting ring items from where the previous pass stopped. Called by all threads.
template <int CW = kConsumerWarps, int PW = kProducerWarps>
__device__ __forceinline__ void ring_init(Plan& pl, int ns) {
  fence_proxy_async_smem();   // planning scratch in the ring: generic accesses before TMA writes
  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(smem_u32(&pl.full[s]), PW * 32);
      mbar_init(smem_u32(&pl.empty[s]), CW);
    }
    pl.failed = 0;
    mbar_fence_init();
  }
  __syncthreads();
}

// Shrink, cluster exchange, expand + fold for one planned pass of a work unit.
// Called by all kThreads threads of every CTA of the cluster, after
// ring_init(); `it0` ring items were used by earlier passes. Returns the ring
// items this pass used. MAXT bounds the 16x8 shrink tiles one consumer warp
// owns (MT * ceil(group rows / 8) <= 8 * MAXT). TILED: A comes as TMA boxes
// (launches with g.a_tiled); each instance has one A layout. TC: the shrink
// runs on tcgen05 (launches with g.tc; one group per pass, TMEM allocated by
// the caller at pl.tmem).
template <int MAXT, bool TILED, bool TC = false, int CW = kConsumerWarps, int PW = kProducerWarps, int RK = 0>
__device__ __forceinline__ int fold_engine(const EngineArgs& p, const FoldGeometry& g, Plan& pl,
                                           unsigned char* smem, const cg::cluster_group& cluster,
                                           int crank, int it0) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned char* ring = smem + g.off_ring;
  const uint32_t ring_u32 = smem_u32(ring);
  float* part_s = reinterpret_cast<float*>(smem + g.off_part);
  uint16_t* xa_s = reinterpret_cast<uint16_t*>(smem + g.off_xa);
  const int G = pl.G, NV = pl.NV;
  const int ns = g.ns;

  const int k_lo = crank * g.ksl, k_hi = min(k_lo + g.ksl, p.k_in);
  const int j_lo = crank * g.jsl, j_hi = min(j_lo + g.jsl, p.n_out);
  const int nk = k_hi > k_lo ? (k_hi - k_lo + g.kch - 1) / g.kch : 0;
  const int nj = j_hi > j_lo ? (j_hi - j_lo + g.jch - 1) / g.jch : 0;
  const int n_shrink = G * nk, n_items = G * (nk + nj);
  const int out_region = g.jch * g.pitch_b;   // byte offset of the out rows inside an expand stage
  const int pitch_o = g.jch * 2 + 16;
  // Barrier of the exchange: a cluster barrier when the cluster has peers;
  // otherwise only the consumer warps take part (the producer never touches
  // the partials or xa, so it keeps filling the ring meanwhile).
  auto unit_sync = [&]() {
    if (g.cl > 1) cluster.sync(); else consumer_sync<CW>();
  };

  if (warp >= CW) {
    // ===================== producer warpgroup =====================
    // All four producer warps serve every item, in item order (an mbarrier
    // parity wait only tells the current phase from the one before it). Rows
    // of at least kTmaRowBytes go by 1-D TMA (copy q to warp q % 4, since one
    // warp serializes its TMA requests); shorter rows go as 16-byte cp.async
    // chunks spread over all 128 producer threads. Every producer thread first
    // registers the TMA bytes it issues, then arrives on the item's full
    // barrier once its own cp.async chunks have landed.
    const int pw = warp - CW;
    const int pt = tid - CW * 32;          // 0 .. 127
    constexpr int kP = PW * 32;
    const int q0 = pw + PW * lane;         // this thread's first TMA copy
    bool dead = false;   // this thread gave up on a stage: it issues no further copies
    // part 0: the whole item. An expand item may also go in two parts around
    // the wait for the previous grid: part 1 its adapter (B) rows, which no
    // earlier kernel writes, part 2 its out rows and this thread's arrival.
    auto produce = [&](int it, int part = 0) {
      const int ri = it0 + it, s = ri % ns;   // ring item
      const uint32_t full = smem_u32(&pl.full[s]);
      if (part != 2 && !dead && ri >= ns && !mbar_wait(smem_u32(&pl.empty[s]), ((ri / ns) - 1) & 1)) {
        if (lane == 0) record_timeout(pl);
        dead = true;
      }
      if (dead) {   // no copies into a stage that may still be read; the phase completes
        if (part != 1) cp_async_arrive_noinc(full);
        return;
      }
      const uint32_t st = ring_u32 + s * g.stage_bytes;
      // An item is two row sets. Set 0: the adapter rows (A rows of this
      // k-chunk, or B rows of this j-chunk: one copy when B is unpadded), at a
      // fixed stride. Set 1: the group's activation rows (x, shrink) or output
      // rows (out, expand), gathered through the plan. Row r of a set goes from
      // src + row(r) * stride (elements) to dst + r * pitch (bytes).
      const uint16_t* src0;
      const uint16_t* src1;
      long long stride0, stride1;
      uint32_t dst0, dst1;
      int n0, bytes0, pitch0, n1, bytes1, pitch1, m0;
      const void* amap = nullptr;   // a_tiled shrink item: A comes as kch/64 boxes of this map
      int k0 = 0;
      if (it < n_shrink) {
        const int gi = it / nk, kc = it - gi * nk;
        k0 = k_lo + kc * g.kch;
        const int bytes = min(g.kch, k_hi - k0) * 2;
        m0 = pl.gstart[gi];
        src0 = pl.gA[gi] + k0; stride0 = p.k_in; dst0 = st; n0 = p.max_rank; bytes0 = bytes; pitch0 = g.pitch_k;
        src1 = p.x + k0; stride1 = p.x_stride; dst1 = st + g.mr16 * g.pitch_k; n1 = pl.gstart[gi + 1] - m0;
        bytes1 = bytes; pitch1 = g.pitch_k;
        if (TILED && g.a_tiled) {
          amap = pl.gmap[gi];
          n0 = 0;
          dst1 = st + g.mr16 * g.kch * 2;
        }
      } else {
        const int e = it - n_shrink, gi = e / nj, jc = e - gi * nj;
        const int j0 = j_lo + jc * g.jch, jlen = min(g.jch, j_hi - j0);
        const int brow = p.max_rank * 2;
        m0 = pl.gstart[gi];
        src0 = pl.gB[gi] + (long long)j0 * p.max_rank; stride0 = p.max_rank; dst0 = st; pitch0 = g.pitch_b;
        if (g.pitch_b == brow) { n0 = 1; bytes0 = jlen * brow; } else { n0 = jlen; bytes0 = brow; }
        src1 = p.out + j0; stride1 = p.out_stride; dst1 = st + out_region; n1 = pl.gstart[gi + 1] - m0;
        bytes1 = jlen * 2; pitch1 = pitch_o;
      }
      // TMA bytes this thread issues (rows q0, q0 + kP, ... of each TMA set)
      const int mine0 = bytes0 >= kTmaRowBytes && q0 < n0 ? (n0 - 1 - q0) / kP + 1 : 0;
      const int mine1 = bytes1 >= kTmaRowBytes && q0 < n1 && !(TC && it < n_shrink) ? (n1 - 1 - q0) / kP + 1 : 0;
      const int nbox = g.kch >> 6, a_box = g.mr16 * 128;
      const int tx = (part != 2 ? mine0 * bytes0 : 0) + (part != 1 ? mine1 * bytes1 : 0) +
                     (amap && pt == 0 ? nbox * a_box : 0);
      if (tx) mbar_expect_tx(full, static_cast<uint32_t>(tx));
      if (amap && pt == 0) {
#pragma unroll 1
        for (int b = 0; b < nbox; ++b) tma_load_2d(st + b * a_box, amap, k0 + 64 * b, 0, full);
      }
#pragma unroll 1
      for (int set = part == 2 ? 1 : 0; set < (part == 1 ? 1 : 2); ++set) {
        const uint16_t* src = set ? src1 : src0;
        const long long stride = set ? stride1 : stride0;
        const uint32_t dst = set ? dst1 : dst0;
        const int n = set ? n1 : n0, bytes = set ? bytes1 : bytes0, pitch = set ? pitch1 : pitch0;
        const int* rmap = it < n_shrink ? pl.xsrc : pl.grow;   // gathered rows: x (shrink) or base_out
        if (TC && set == 1 && it < n_shrink) {
          // x rows for the tensor core: 16-byte chunk ch of row q goes to atom
          // ch / 8 (gmax rows x 128 B), chunk (ch % 8) ^ (q % 8); the chunks of
          // the last 16-wide k-step past the data are zeros.
          const int cpr = bytes >> 4, cpr16 = ((bytes + 31) >> 5) << 1;
#pragma unroll 1
          for (int c = pt; c < n * cpr16; c += kP) {
            const int q = c / cpr16, ch = c - q * cpr16;
            const uint32_t d = dst + (ch >> 3) * (g.gmax * 128) + q * 128 + (((ch & 7) ^ (q & 7)) << 4);
            const char* srow = reinterpret_cast<const char*>(src + static_cast<long long>(rmap[pl.members[m0 + q]]) * stride);
            if (ch < cpr) cp_async16(d, srow + ch * 16); else cp_async16_zero(d, srow);
          }
        } else if (bytes >= kTmaRowBytes) {
#pragma unroll 1
          for (int q = q0; q < n; q += kP) {
            const int row = set ? rmap[pl.members[m0 + q]] : q;
            bulk_g2s(dst + q * pitch, src + row * stride, bytes, full);
          }
        } else {   // short rows: 16-byte cp.async chunks over all producer threads
          const int cpr = bytes >> 4;
#pragma unroll 1
          for (int c = pt; c < n * cpr; c += kP) {
            const int q = c / cpr, ch = c - q * cpr;
            const int row = set ? rmap[pl.members[m0 + q]] : q;
            cp_async16(dst + q * pitch + ch * 16, reinterpret_cast<const char*>(src + row * stride) + ch * 16);
          }
        }
      }
      if (part != 1) cp_async_arrive_noinc(full);
    };
    // Items whose stage is freed by shrink work can be issued before the
    // cluster exchange; the rest only after it (their stages are released by
    // expand work, which needs the exchanged xa).
    // With a late wait (inputs ready), the out rows of expand items, which
    // are base_out, are read only after the previous grid on the stream has
    // completed: before the wait go the shrink items and, in cluster units,
    // the B rows of the expand items that the shrink's stages free (measured
    // on GB300: qkv 21.3 -> 21.0 us; the single-CTA MoE units were slower).
    const int pre = p.late ? n_shrink : g.cl > 1 ? min(n_items, n_shrink + ns) : n_items;
    const int early = (p.late && g.cl > 1) ? min(n_items, n_shrink + ns) : n_shrink;   // items [n_shrink, early) in two parts
    for (int it = 0; it < pre; ++it) {
      produce(it);
      GLORA_STAMP(it == 0 && tid == CW * 32, 3);
    }
    for (int it = n_shrink; it < early; ++it) produce(it, 1);
    if (g.cl > 1) {
      cluster.sync();
      if (!g.gather) cluster.sync();
    }
    if (p.late) pdl_wait_then_release();
    for (int it = n_shrink; it < early; ++it) produce(it, 2);
    for (int it = max(pre, early); it < n_items; ++it) produce(it);
    if (*reinterpret_cast<volatile int*>(&pl.failed)) {
      // A wait gave up somewhere: before the CTA can exit, let this thread's own
      // copies land (cp.async groups; TMA bytes complete the stages' full phases).
      cp_async_wait(0);
      for (int it = max(0, n_items - ns); it < n_items; ++it) {
        const int ri = it0 + it;
        mbar_wait_limit(smem_u32(&pl.full[ri % ns]), (ri / ns) & 1, kDrainLimitCycles);
      }
    }
    return n_items;
  }

  // ========================= consumer warps =========================
  // Shrink items are either tile-parallel (one group per unit, bgmv): every
  // consumer warp takes part in every item, in order, splitting its tiles; or
  // slot-parallel (many small MoE groups whose shrink is one k-chunk): the KSG
  // consumer warps of ring slot s (warps s, s + ns, ...) alone serve it, each
  // taking alternate k-steps of every shrink item in it into its own partial
  // plane, and release the slot with CW / KSG arrivals each, so the latency
  // chains of several groups overlap while every slot keeps in-order consumers.
  // Expand items are always tile-parallel.
  // Tile-parallel items with few tiles are also split over k: the consumer
  // warps form KS k-phases of TW warps; phase kp takes k-steps kp, kp + KS, ...
  // of every chunk and keeps its partial sums in its own plane of part_s, and
  // the exchange adds the planes in phase order.
  const bool gpar = g.group_parallel != 0;
  // Slot-parallel: group gi's one shrink item is ring item it0 + gi, in slot
  // (it0 + gi) % ns, served by KSG warps (warps s, s + ns, ...) that take
  // alternate k-steps into their own partial planes.
  const int KSG = gpar ? max(1, min(g.ksplit, CW / ns)) : 1;
  const bool idle = gpar && warp >= ns * KSG;   // slot-parallel with fewer slots than warps
  const int g_first = gpar ? (((warp % ns) - it0 % ns) + ns) % ns : 0, g_step = gpar ? ns : 1;
  const int KS = gpar ? KSG : g.ksplit, TW = CW / KS;
  const int kp = gpar ? warp / ns : warp / TW;
  const int t_first = gpar ? 0 : warp % TW, t_step = gpar ? 1 : TW;
  const int MT = g.mr16 >> 4;
  const int plane = g.rt * g.pitch_part;         // floats per k-phase plane of part_s
  // The shrink of one group, compiled per A layout (padded rows, or swizzled TMA boxes).
  auto shrink_group = [&](int gi, auto tiled_c) {
    const int m0 = pl.gstart[gi], R = pl.gstart[gi + 1] - m0, NT = (R + 7) >> 3, ntiles = MT * NT;
    // Independent accumulator chains per tile (k-steps dealt round-robin over
    // the chains within each chunk) when a warp holds few tiles, so consecutive
    // MMAs do not wait on each other; the chains are added once per group, in
    // a fixed order. When all of a warp's tiles share one A row block (the
    // warp stride is a multiple of MT), its A fragment is loaded once per k-step.
    constexpr int kChains = MAXT == 1 ? 4 : (MAXT == 2 ? 2 : 1);
    const bool share_a = !gpar && (TW % MT) == 0;
    // A fragment rows: padded rows (pitch_k), or 128-byte swizzled rows of
    // 64-column TMA boxes (a_tiled: 16-byte chunk c of row r sits at chunk
    // c ^ (r & 7)); the x rows follow the A region, padded.
    constexpr bool tiled = decltype(tiled_c)::value;
    const int a_box = g.mr16 * 128;                  // bytes per A box
    const uint32_t x_base = tiled ? g.mr16 * g.kch * 2 : g.mr16 * g.pitch_k;
    int a_row[MAXT];
    uint32_t a_off[MAXT], x_off[MAXT];
    float acc[kChains][MAXT][4];
#pragma unroll
    for (int i = 0; i < MAXT; ++i) {
      const int t = t_first + i * t_step;
      const int mt = t % MT, nt = t / MT;
      a_row[i] = mt * 16 + (lane & 15);
      a_off[i] = a_row[i] * (tiled ? 128 : g.pitch_k);
      x_off[i] = x_base + (nt * 8 + (lane & 7)) * g.pitch_k;
#pragma unroll
      for (int ch = 0; ch < kChains; ++ch) acc[ch][i][0] = acc[ch][i][1] = acc[ch][i][2] = acc[ch][i][3] = 0.f;
    }
    // this lane's ldmatrix address of A tile i at k-step kk (x4 for k16: lanes
    // 16..31 take the second 8 columns; x2 for the k8 tail)
    auto a_addr = [&](uint32_t st, int i, int kk, bool k16) -> uint32_t {
      if constexpr (tiled) {
        const int c = ((kk & 63) >> 3) + (k16 ? (lane >> 4) : 0);
        return st + (kk >> 6) * a_box + a_off[i] + ((c ^ (a_row[i] & 7)) << 4);
      } else {
        return st + a_off[i] + kk * 2 + (k16 ? ((lane >> 4) << 4) : 0);
      }
    };
    // one k-step (16, or an 8-wide tail) of every tile of this warp into chain `ch`
    auto step = [&](uint32_t st, int kk, int kstep, float (&ac)[MAXT][4]) {
      if (!tiled && !share_a) {
#pragma unroll
        for (int i = 0; i < MAXT; ++i) {
          if (t_first + i * t_step < ntiles)
            mma_step(ac[i], st + a_off[i] + kk * 2, st + x_off[i] + kk * 2, kstep, lane);
        }
      } else if (kstep == 16) {
        uint32_t a0, a1, a2, a3;
        if (share_a) ldsm_x4(a_addr(st, 0, kk, true), a0, a1, a2, a3);
#pragma unroll
        for (int i = 0; i < MAXT; ++i) {
          if (t_first + i * t_step < ntiles) {
            if (!share_a) ldsm_x4(a_addr(st, i, kk, true), a0, a1, a2, a3);
            uint32_t b0, b1;
            ldsm_x2(st + x_off[i] + kk * 2 + (((lane >> 3) & 1) << 4), b0, b1);
            mma_k16(ac[i], a0, a1, a2, a3, b0, b1);
          }
        }
      } else {
        uint32_t a0, a1;
        if (share_a) ldsm_x2(a_addr(st, 0, kk, false), a0, a1);
#pragma unroll
        for (int i = 0; i < MAXT; ++i) {
          if (t_first + i * t_step < ntiles) {
            if (!share_a) ldsm_x2(a_addr(st, i, kk, false), a0, a1);
            uint32_t b0;
            ldsm_x1(st + x_off[i] + kk * 2, b0);
            mma_k8(ac[i], a0, a1, b0);
          }
        }
      }
    };
    for (int kc = 0; kc < nk; ++kc) {
      const int ri = it0 + gi * nk + kc, s = ri % ns;
      if (!mbar_wait(smem_u32(&pl.full[s]), (ri / ns) & 1) && lane == 0) record_timeout(pl);
      const uint32_t st = ring_u32 + s * g.stage_bytes;
      const int klen = min(g.kch, k_hi - (k_lo + kc * g.kch));
      const int nst = (klen + 15) >> 4, nfull = klen >> 4;   // k-steps of this chunk (the last may be 8 wide)
      int si = kp;
      for (; si + KS * (kChains - 1) < nfull; si += KS * kChains) {
#pragma unroll
        for (int ch = 0; ch < kChains; ++ch) step(st, (si + ch * KS) * 16, 16, acc[ch]);
      }
      for (; si < nst; si += KS) step(st, si * 16, min(16, klen - si * 16), acc[0]);   // the rest on chain 0
      __syncwarp();
      if (lane == 0) mbar_arrive_count(smem_u32(&pl.empty[s]), gpar ? CW / KSG : 1);
    }
#pragma unroll
    for (int ch = 1; ch < kChains; ++ch)
#pragma unroll
      for (int i = 0; i < MAXT; ++i)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[0][i][v] += acc[ch][i][v];
    // group complete: this k-slice's partial sums -> shared memory
#pragma unroll
    for (int i = 0; i < MAXT; ++i) {
      const int t = t_first + i * t_step;
      if (t < ntiles) {
        const int mt = t % MT, nt = t / MT;
        const int c0 = mt * 16 + (lane >> 2), r0 = nt * 8 + 2 * (lane & 3);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int c = c0 + (v >> 1) * 8, r = r0 + (v & 1);
          if (c < p.max_rank && r < R) part_s[kp * plane + pl.members[m0 + r] * g.pitch_part + c] = acc[0][i][v];
        }
      }
    }
  };
  if constexpr (TC) {
    // tcgen05 shrink of the pass's one group: consumer warp 0 issues the MMAs
    // D[A rows (rank) x x rows] += A x^T into TMEM (M = 128, N = gmax = 16),
    // and releases each stage through the commit plus the other seven
    // consumer arrivals; warps 0-3 then move the fp32 partial from their TMEM
    // lanes (lane = rank index, column = row) to part_s. One pass per launch:
    // tc_done completes once (phase 0).
    if (nk > 0) {
      const int m0 = pl.gstart[0], R = pl.gstart[1] - m0;
      if (warp == 0 && lane == 0) {
        const uint32_t idesc = idesc_bf16_f32(128, 16);
        const int a_box = g.mr16 * 128, x_atom = g.gmax * 128;
        for (int kc = 0; kc < nk; ++kc) {
          const int ri = it0 + kc, s = ri % ns;
          if (!mbar_wait(smem_u32(&pl.full[s]), (ri / ns) & 1)) record_timeout(pl);
          tc_fence_after();
          const uint32_t st = ring_u32 + s * g.stage_bytes, xt = st + g.mr16 * g.kch * 2;
          const int klen = min(g.kch, k_hi - (k_lo + kc * g.kch)), nst = (klen + 15) >> 4;
          for (int s16 = 0; s16 < nst; ++s16) {
            const uint32_t off = (s16 & 3) * 32;
            umma_bf16(pl.tmem, smem_desc(st + (s16 >> 2) * a_box + off, 1024, Swz::k128),
                      smem_desc(xt + (s16 >> 2) * x_atom + off, 1024, Swz::k128), idesc, (kc | s16) != 0);
          }
          umma_commit(smem_u32(&pl.empty[s]));
          mbar_arrive_count(smem_u32(&pl.empty[s]), CW - 1);   // the phase still waits for the commit
        }
        umma_commit(smem_u32(&pl.tc_done));
      }
      __syncwarp();
      if (!mbar_wait(smem_u32(&pl.tc_done), 0) && lane == 0) record_timeout(pl);
      tc_fence_after();
      if (warp < 4) {
        uint32_t v[16];
        tmem_ld16(pl.tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
        tmem_ld_wait();
        const int c = warp * 32 + lane;
        if (c < p.max_rank) {
#pragma unroll
          for (int r = 0; r < 16; ++r)
            if (r < R) part_s[pl.members[m0 + r] * g.pitch_part + c] = __uint_as_float(v[r]);
        }
      }
      tc_fence_before();
    }
  } else {
    for (int gi = g_first; gi < G && nk > 0 && !idle; gi += g_step) {
      shrink_group(gi, std::integral_constant<bool, TILED>{});
    }
  }
  if (nk == 0) {  // empty k-slice: the partials are zero
    for (int e = tid; e < KS * NV * p.max_rank; e += CW * 32) {
      const int ph = e / (NV * p.max_rank), r = e - ph * NV * p.max_rank;
      const int mi = r / p.max_rank, c = r - mi * p.max_rank;
      part_s[ph * plane + pl.members[mi] * g.pitch_part + c] = 0.f;
    }
  }

  GLORA_STAMP(tid == 0, 4);
  GLORA_NOTE(tid == 0, 11, NV);
  // ---- exchange: xa = bf16(sum of the partials: cluster ranks in order, and
  //      k-phase planes in order within a rank) ----
  const int xa_pitch_el = g.pitch_xa >> 1;
  // xa is written here, or after the expand with a late wait (it may still be
  // in use by the previous grid until then).
  const bool store_xa = p.xa != nullptr && pl.failed == 0 && !p.late;
  if (g.gather) {
    // All-gather: each CTA adds its k-phase planes and stores the result into
    // slot crank of every peer's gather buffer (one cluster barrier); then every
    // CTA adds the cl slots in rank order itself.
    float* gath = part_s + KS * plane;
    consumer_sync<CW>();
    for (int e = tid; e < NV * p.max_rank; e += CW * 32) {
      const int mi = e / p.max_rank, c = e - mi * p.max_rank;
      const int off = pl.members[mi] * g.pitch_part + c;
      float v = part_s[off];
      for (int ph = 1; ph < KS; ++ph) v += part_s[ph * plane + off];
      for (int q = 0; q < g.cl; ++q) cluster.map_shared_rank(gath, q)[crank * plane + off] = v;
    }
    unit_sync();
    for (int e = tid; e < NV * p.max_rank; e += CW * 32) {
      const int mi = e / p.max_rank, c = e - mi * p.max_rank, pos = pl.members[mi];
      const int off = pos * g.pitch_part + c;
      float sum = gath[off];
      for (int q = 1; q < g.cl; ++q) sum += gath[q * plane + off];
      const uint16_t xb = f32_to_bf16_bits(sum);
      xa_s[pos * xa_pitch_el + c] = xb;
      if (store_xa && e % g.cl == crank) p.xa[(long long)pl.xarow[pos] * p.max_rank + c] = xb;
    }
    consumer_sync<CW>();
  } else {
    // Reduce-scatter: CTA crank adds its share of the elements over the ranks'
    // partials (each rank first folds its own k-phase planes) and pushes the
    // BF16 result to every CTA of the cluster.
    if (KS > 1 && g.cl > 1) {
      consumer_sync<CW>();
      for (int e = tid; e < NV * p.max_rank; e += CW * 32) {
        const int mi = e / p.max_rank, c = e - mi * p.max_rank;
        const int off = pl.members[mi] * g.pitch_part + c;
        float v = part_s[off];
        for (int ph = 1; ph < KS; ++ph) v += part_s[ph * plane + off];
        part_s[off] = v;
      }
    }
    unit_sync();
    const int E = NV * p.max_rank, per = (E + g.cl - 1) / g.cl;
    const int e_lo = crank * per, e_hi = min(e_lo + per, E);
    for (int e = e_lo + tid; e < e_hi; e += CW * 32) {
      const int mi = e / p.max_rank, c = e - mi * p.max_rank, pos = pl.members[mi];
      const int off = pos * g.pitch_part + c;
      float sum;
      if (g.cl > 1) {
        sum = cluster.map_shared_rank(part_s, 0)[off];
        for (int q = 1; q < g.cl; ++q) sum += cluster.map_shared_rank(part_s, q)[off];
      } else {
        sum = part_s[off];
        for (int ph = 1; ph < KS; ++ph) sum += part_s[ph * plane + off];
      }
      const uint16_t xb = f32_to_bf16_bits(sum);
      const int xoff = pos * xa_pitch_el + c;
      for (int q = 0; q < g.cl; ++q) cluster.map_shared_rank(xa_s, q)[xoff] = xb;
      if (store_xa) p.xa[(long long)pl.xarow[pos] * p.max_rank + c] = xb;
    }
    unit_sync();
  }

  // ---- expand + fold over this CTA's j-slice ---------------------------------
  // Work comes in 16-column blocks of two 16x8 tensor-core tiles (16 group rows
  // x 8 consecutive output columns each), with the xa rows as the A operand:
  // their fragments are loaded once per group at max_rank 16 and 32, per
  // block at other ranks. Lane (g, q)
  // holds columns 2q, 2q+1 of each tile for rows g and g + 8; it folds them
  // with the staged old values in registers, and one exchange with lane q ^ 1
  // leaves it four adjacent columns, so each row leaves as one full 32-byte
  // sector of 8-byte stores. The TMA-filled stage is only read. Consumer warp
  // w takes blocks w, w + CW, ...
  if (p.late) pdl_wait_then_release();   // base_out (and xa) only after the previous grid
  GLORA_STAMP(tid == 0, 5);
  const uint32_t xa_base = smem_u32(xa_s);
  const int gq = lane >> 2, q = lane & 3;
  const bool odd = (q & 1) != 0;
  const int scol = odd ? 2 * q + 6 : 2 * q;                            // first stored column
  const int brow4 = (lane >> 4) * 8 + (lane & 7), bk4 = ((lane >> 3) & 1) << 4;   // ldmatrix.x4 of B
  const int brow2 = ((lane >> 3) & 1) * 8 + (lane & 7);                // ldmatrix.x2 of B (k8 tail)
  for (int gi = 0; gi < G; ++gi) {
    const int m0 = pl.gstart[gi], R = pl.gstart[gi + 1] - m0;
    const float scale = pl.gscale[gi];
    // Per group: xa row (lane & 15) of each 16-row tile (rows past R repeat the
    // last one), and for rows gq + 8 * hh the offset of the staged old values
    // inside a stage (rows past R read the last row, in bounds) and the output
    // row (NULL past R).
    constexpr int kRT = (kMaxGroupRows + 15) / 16;   // 16-row tiles of a group
    uint32_t a_row[kRT], rowoff[2 * kRT];
    uint16_t* obase[2 * kRT];
#pragma unroll
    for (int mr = 0; mr < kRT; ++mr) a_row[mr] = xa_base + pl.members[m0 + min(mr * 16 + (lane & 15), R - 1)] * g.pitch_xa;
#pragma unroll
    for (int hh = 0; hh < 2 * kRT; ++hh) {
      const int r = hh * 8 + gq;
      rowoff[hh] = out_region + min(r, R - 1) * pitch_o + 4 * q;
      obase[hh] = r < R ? p.out + (long long)pl.grow[pl.members[m0 + r]] * p.out_stride + scol : nullptr;
    }
    // The group's expand items, compiled per row-tile count MR (up to kRT) and
    // per KS, the k16 steps whose xa fragments stay in registers (1: max_rank
    // 16, 2: max_rank 32; 0: any max_rank, fragments loaded per step, k8 tail).
    auto items = [&](auto mr_c, auto ks_c) {
      constexpr int MR = decltype(mr_c)::value, KS = decltype(ks_c)::value;
      uint32_t af[MR][KS > 0 ? KS : 1][4];
      if (KS > 0) {
#pragma unroll
        for (int mr = 0; mr < MR; ++mr)
#pragma unroll
          for (int ks = 0; ks < (KS > 0 ? KS : 1); ++ks)
            ldsm_x4(a_row[mr] + ks * 32 + ((lane >> 4) << 4), af[mr][ks][0], af[mr][ks][1], af[mr][ks][2], af[mr][ks][3]);
      }
      for (int jc = 0; jc < nj; ++jc) {
        const int ri = it0 + n_shrink + gi * nj + jc, s = ri % ns;
        if (!mbar_wait(smem_u32(&pl.full[s]), (ri / ns) & 1) && lane == 0) record_timeout(pl);
        GLORA_STAMP(tid == 0 && gi == 0 && jc == 0, 6);
        const uint32_t st = ring_u32 + s * g.stage_bytes;
        const int j0 = j_lo + jc * g.jch, jlen = min(g.jch, j_hi - j0), NCB = (jlen + 15) >> 4;
        const bool store = pl.failed == 0;
        // One 16-column block: both 16x8 tiles of every 16-row tile of the group.
        auto block_mma = [&](int cb, float (&d)[MR][2][4]) {
#pragma unroll
          for (int mr = 0; mr < MR; ++mr)
#pragma unroll
            for (int t = 0; t < 2; ++t) d[mr][t][0] = d[mr][t][1] = d[mr][t][2] = d[mr][t][3] = 0.f;
          const uint32_t bblk = st + cb * 16 * g.pitch_b;
          if (KS > 0) {
#pragma unroll
            for (int ks = 0; ks < (KS > 0 ? KS : 1); ++ks) {
              uint32_t b0, b1, b2, b3;
              ldsm_x4(bblk + brow4 * g.pitch_b + ks * 32 + bk4, b0, b1, b2, b3);
#pragma unroll
              for (int mr = 0; mr < MR; ++mr) {
                mma_k16(d[mr][0], af[mr][ks][0], af[mr][ks][1], af[mr][ks][2], af[mr][ks][3], b0, b1);
                mma_k16(d[mr][1], af[mr][ks][0], af[mr][ks][1], af[mr][ks][2], af[mr][ks][3], b2, b3);
              }
            }
          } else {
            int kk = 0;
            for (; kk + 16 <= p.max_rank; kk += 16) {
              uint32_t b0, b1, b2, b3;
              ldsm_x4(bblk + brow4 * g.pitch_b + kk * 2 + bk4, b0, b1, b2, b3);
#pragma unroll
              for (int mr = 0; mr < MR; ++mr) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(a_row[mr] + kk * 2 + ((lane >> 4) << 4), a0, a1, a2, a3);
                mma_k16(d[mr][0], a0, a1, a2, a3, b0, b1);
                mma_k16(d[mr][1], a0, a1, a2, a3, b2, b3);
              }
            }
            if (kk < p.max_rank) {                     // k8 tail (max_rank % 16 == 8)
              uint32_t b0, b1;
              ldsm_x2(bblk + brow2 * g.pitch_b + kk * 2, b0, b1);
#pragma unroll
              for (int mr = 0; mr < MR; ++mr) {
                uint32_t a0, a1;
                ldsm_x2(a_row[mr] + kk * 2, a0, a1);
                mma_k8(d[mr][0], a0, a1, b0);
                mma_k8(d[mr][1], a0, a1, b1);
              }
            }
          }
        };
        // The staged old values of a block's rows (rows past R read the last
        // row: in bounds, never stored).
        auto block_old = [&](int cb, uint32_t (&o)[2 * MR][2]) {
          const int c0 = cb * 16;
#pragma unroll
          for (int hh = 0; hh < 2 * MR; ++hh) {
            if (hh == 0 || hh * 8 < R) {                // warp-uniform: this row half has rows
              asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(o[hh][0]) : "r"(st + rowoff[hh] + c0 * 2));
              asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(o[hh][1]) : "r"(st + rowoff[hh] + c0 * 2 + 16));
            }
          }
        };
        // Fold and store a block: lane (g, q) folds columns 2q, 2q+1 of both
        // tiles for rows g and g + 8; one exchange with lane q ^ 1 leaves it
        // four adjacent columns (a full 8-byte store; each row's 32 bytes
        // leave as one sector).
        auto block_fold = [&](int cb, const float (&d)[MR][2][4], const uint32_t (&o)[2 * MR][2]) {
          const int c0 = cb * 16;
          const bool col_ok = c0 + scol < jlen;         // the last block may hold only 8 columns
#pragma unroll
          for (int hh = 0; hh < 2 * MR; ++hh) {
            const int mr = hh >> 1, h = hh & 1;
            if (hh == 0 || hh * 8 < R) {
              const uint32_t f0 = fold_pair(d[mr][0][2 * h], d[mr][0][2 * h + 1], scale, o[hh][0]);
              const uint32_t f1 = fold_pair(d[mr][1][2 * h], d[mr][1][2 * h + 1], scale, o[hh][1]);
              const uint32_t recv = __shfl_xor_sync(0xffffffffu, odd ? f0 : f1, 1);
              uint16_t* ob = obase[hh];
              if (ob && store && col_ok) {
                const uint32_t lo = odd ? recv : f0, hi = odd ? f1 : recv;
                asm volatile("st.global.v2.b32 [%0], {%1, %2};\n" ::"l"(ob + j0 + c0), "r"(lo), "r"(hi) : "memory");
              }
            }
          }
        };
        // Two blocks per step (cb and cb + CW): both blocks' loads and MMAs are
        // issued before either block's dependent fold.
        int cb = warp;
        for (; cb + CW < NCB; cb += 2 * CW) {
          float da[MR][2][4], db[MR][2][4];
          uint32_t oa[2 * MR][2], ob2[2 * MR][2];
          block_mma(cb, da);
          block_mma(cb + CW, db);
          block_old(cb, oa);
          block_old(cb + CW, ob2);
          block_fold(cb, da, oa);
          block_fold(cb + CW, db, ob2);
        }
        if (cb < NCB) {
          float da[MR][2][4];
          uint32_t oa[2 * MR][2];
          block_mma(cb, da);
          block_old(cb, oa);
          block_fold(cb, da, oa);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&pl.empty[s]));
      }
    };
    using I1 = std::integral_constant<int, 1>;
    using I2 = std::integral_constant<int, 2>;
    using I0 = std::integral_constant<int, 0>;
    // The expand loop is compiled for the launch's rank class only (RK: 1 =
    // max_rank 16 and 2 = max_rank 32, xa fragments held in registers; 0 = any
    // max_rank, fragments loaded per step): one variant per kernel keeps its
    // code small (measured on GB300: MoE down fold 86.4 -> 84.8 us, decode
    // 8.6 -> 8.3 us with waiting calls).
    auto by_rank = [&](auto mr_c) {
      if constexpr (RK == 1) items(mr_c, I1{});
      else if constexpr (RK == 2) items(mr_c, I2{});
      else items(mr_c, I0{});
    };
    if constexpr (kRT > 1) {
      if (R <= 16) by_rank(I1{}); else by_rank(I2{});
    } else {
      by_rank(I1{});
    }
  }
  GLORA_STAMP(tid == 0, 7);
  // With a late wait xa leaves last: after the exchange every CTA of the
  // cluster holds all of it in xa_s; CTA crank writes rows crank, crank + cl,
  // ... in 4-byte pairs.
  if (p.late && p.xa != nullptr && pl.failed == 0) {
    const int half = p.max_rank >> 1, mine = NV > crank ? (NV - crank + g.cl - 1) / g.cl : 0;
    for (int e = tid; e < mine * half; e += CW * 32) {
      const int mi = crank + (e / half) * g.cl, c2 = e - (e / half) * half, pos = pl.members[mi];
      const uint32_t v = *reinterpret_cast<const uint32_t*>(xa_s + pos * xa_pitch_el + 2 * c2);
      *reinterpret_cast<uint32_t*>(p.xa + static_cast<long long>(pl.xarow[pos]) * p.max_rank + 2 * c2) = v;
    }
  }
  return n_items;
}

// ============================================================================
// Routed bgmv: work unit = up to rt rows of one slot, in ascending row order.
// Direct numbering (max_loras <= n): unit s < max_loras is tile 0 of slot s, so
// its table entries are loaded at once, beside seq_slot; units from max_loras
// on are the further tiles (1, 2, ...) of slots with more than rt rows, in slot
// order. Otherwise units are numbered slot by slot over every slot that has
// rows. Either way the static grid bound is n/rt + min(n, max_loras) units; a
// unit that finds no rows, or whose slot has a NULL table entry, does nothing.
// The decode-path MoE fold runs here too: its "slot" is the table entry
// a * E + e of the row's expert and its token's adapter, and max_loras is the
// table count. So does the single-adapter delta at small m (`single`): every
// row is slot 0 of a one-entry table passed by value.
// ============================================================================
template <int MAXT, bool TILED, bool TC, int RK>
__global__ void __launch_bounds__(kThreads, 2) lora_bgmv_fold_kernel(const __grid_constant__ BgmvArgs p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const FoldGeometry& g = p.g;
  const cg::cluster_group cluster = cg::this_cluster();
  const int crank = static_cast<int>(cluster.block_rank());
  const int unit = static_cast<int>(blockIdx.x) / g.cl;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Plan& pl = *reinterpret_cast<Plan*>(smem);
  GLORA_STAMP(tid == 0, 0);
  GLORA_GTIME(tid == 0, 9);

  // Without a late wait, nothing is read before the previous grid on the
  // stream has completed. With one, the engine waits before it touches base_out
  // or xa; a CTA that folds nothing leaves at once, except CTA 0, which waits,
  // so that this grid never completes before the previous one.
  if (!p.late) pdl_wait_then_release();
  GLORA_STAMP(tid == 0, 1);
  auto leave = [&]() {
    if (p.late && blockIdx.x == 0) pdl_wait_then_release();
  };
  if (!tiled_smem_ok(g, smem)) return leave();

  const bool first_tile = g.direct && unit < p.max_loras;
  int slot = first_tile ? unit : -1, tile = 0;
  const uint16_t* tab_a = nullptr;  // table entries: the loads overlap the scans below
  const uint16_t* tab_b = nullptr;
  float tab_s = 0.f;
  // the slot's A tensor map (a_tiled launches); its descriptor fetch overlaps the scans
  auto a_map = [&](int s) { return static_cast<const char*>(p.a_maps) + 128 * static_cast<long long>(s); };
  if (first_tile && tid == 0) {
    if (TILED) prefetch_tensormap(a_map(slot));
    tab_a = p.single ? p.one_a : p.a_table[slot];
    tab_b = p.single ? p.one_b : p.b_table[slot];
    tab_s = p.single ? p.one_scale : p.scale_table[slot];
  }
  // seq_slot (and the per-slot row counts) live in the not-yet-used ring.
  int* ss = reinterpret_cast<int*>(smem + g.off_ring);
  int* cnt = ss + ((p.n + 3) & ~3);
  for (int i = tid; i < p.n; i += kThreads) {
    int sl;
    if (p.single) {
      sl = 0;
    } else if (p.seq_slot) {
      sl = p.seq_slot[i];
    } else {   // MoE decode rows: table a * E + e from the row's expert and its token's adapter
      const int e = p.indices[i], t = i / p.top_k;
      const int a = p.row_adapter ? (t < p.num_tokens ? p.row_adapter[t] : -1) : 0;
      sl = (e >= 0 && e < p.num_experts && a >= 0 && a < p.max_loras / p.num_experts) ? a * p.num_experts + e : -1;
    }
    ss[i] = sl;
  }
  if (!first_tile) {
    for (int s = tid; s < p.max_loras; s += kThreads) cnt[s] = 0;
    if (tid == 0) pl.found_slot = -1;
    __syncthreads();
    for (int i = tid; i < p.n; i += kThreads) {
      const int s = ss[i];
      if (s >= 0 && s < p.max_loras) atomicAdd(&cnt[s], 1);
    }
    __syncthreads();
    // Tiles per slot (direct numbering: only the tiles after the first), prefix
    // over slots, locate this cluster's (slot, tile).
    const int v = g.direct ? unit - p.max_loras : unit, t0 = g.direct ? 1 : 0;
    const int per = (p.max_loras + kThreads - 1) / kThreads;
    const int lo = min(tid * per, p.max_loras), hi = min(lo + per, p.max_loras);
    int local = 0;
    for (int s = lo; s < hi; ++s) local += max(0, (cnt[s] + g.rt - 1) / g.rt - t0);
    int run = block_inclusive_sum(local, pl.warp_sums) - local;
    for (int s = lo; s < hi; ++s) {
      const int t = max(0, (cnt[s] + g.rt - 1) / g.rt - t0);
      if (v >= run && v < run + t) {
        pl.found_slot = s;
        pl.found_tile = t0 + v - run;
      }
      run += t;
    }
    __syncthreads();
    slot = pl.found_slot;
    if (slot < 0) return leave();  // every CTA of the cluster takes this branch together
    tile = pl.found_tile;
    if (tid == 0) {
      if (TILED) prefetch_tensormap(a_map(slot));
      tab_a = p.single ? p.one_a : p.a_table[slot];
      tab_b = p.single ? p.one_b : p.b_table[slot];
      tab_s = p.single ? p.one_scale : p.scale_table[slot];
    }
  } else {
    __syncthreads();
  }
  // Rows of this slot in ascending order; keep ranks [want_lo, want_lo + rt).
  const int want_lo = tile * g.rt;
  int R;
  {
    int base = 0;
    for (int i0 = 0; i0 < p.n; i0 += kThreads) {
      const int i = i0 + tid;
      const bool f = (i < p.n) && (ss[i] == slot);
      const unsigned bal = __ballot_sync(0xffffffffu, f);
      if (lane == 0) pl.warp_sums[warp] = __popc(bal);
      __syncthreads();
      int before = 0, total = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const int c = pl.warp_sums[w];
        before += (w < warp) ? c : 0;
        total += c;
      }
      const int rank = base + before + __popc(bal & ((1u << lane) - 1u));
      if (f && rank >= want_lo && rank < want_lo + g.rt) {
        const int pos = rank - want_lo;
        pl.members[pos] = pos;
        pl.grow[pos] = i;
        pl.xsrc[pos] = i;
        pl.xarow[pos] = i;
      }
      base += total;
      __syncthreads();
    }
    R = min(g.rt, base - want_lo);
  }
  if (R <= 0) return leave();  // no rows for this unit (every thread computed the same count)
  if (tid == 0) {
    pl.gA[0] = tab_a;
    pl.gmap[0] = TILED ? a_map(slot) : nullptr;
    pl.gB[0] = tab_b;
    pl.gscale[0] = tab_s;
    const uintptr_t a = reinterpret_cast<uintptr_t>(tab_a), b = reinterpret_cast<uintptr_t>(tab_b);
    int G = 1;
    if (a == 0 || b == 0) {
      G = 0;
    } else if ((a | b) & 15u) {
      G = 0;
      if (crank == 0) atomicOr(&g_lora_status, kDevMisaligned);
    }
    pl.G = G;
    pl.NV = R;
    pl.gstart[0] = 0;
    pl.gstart[1] = R;
  }
  __syncthreads();
  if (pl.G == 0) return leave();  // NULL or misaligned adapter: rows stay unchanged

  if constexpr (TC) {   // the shrink's accumulator: 32 TMEM columns (16 used)
    if (warp == 0) {
      tmem_alloc(smem_u32(&pl.tmem), 32);
      tmem_relinquish();
    }
    if (tid == 0) mbar_init(smem_u32(&pl.tc_done), 1);   // ring_init fences and synchronizes
    tc_fence_before();
  }
  ring_init(pl, g.ns);
  if constexpr (TC) tc_fence_after();
  const EngineArgs ea{p.x, p.x_stride, p.out, p.out_stride, p.xa, p.max_rank, p.k_in, p.n_out, p.late};
  GLORA_STAMP(tid == 0, 2);
  fold_engine<MAXT, TILED, TC, kConsumerWarps, kProducerWarps, RK>(ea, g, pl, smem, cluster, crank, 0);
  if constexpr (TC) {
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(pl.tmem, 32);
    }
  }
  GLORA_STAMP(tid == 0, 8);
  GLORA_GTIME(tid == 0, 10);
}

// ============================================================================
// MoE grouped fold: persistent CTAs over units of the window's (expert,
// adapter) groups.
//
// The rows of a window are sorted by expert; the rows of one (expert e,
// adapter a) group share A and B, so each group should be read once. A unit
// is one expert of the window and a chunk of `ac` adapters: its groups are
// (e, a) for a in the chunk. The chunk size follows the window's expert count
// (about kMoeUnitsPerCta units per CTA), and CTA b of G takes units b, b + G,
// ... A CTA plans only its own units: it reads the expert offsets, then the
// token and adapter of each row of its units' experts (two memory round trips,
// the units' table entries loaded beside them), and numbers each routed row
// within its group with one shared-memory atomic. Which rows share a group of
// the fold never changes a row's arithmetic, so that order may vary.
// Rows are taken kMoeRoundRows at a time (rounds) from the CTA's units' rows,
// folded in passes of up to kMaxRows rows, split into groups of at most gmax
// rows of one (expert, adapter) pair, each folded over the full k_in and n_out.
// ============================================================================
#ifndef GLORA_MOE_UNITS_PER_CTA
#define GLORA_MOE_UNITS_PER_CTA 3
#endif
constexpr int kMoeUnitsPerCta = GLORA_MOE_UNITS_PER_CTA;   // target units per CTA (sets the chunk size)
constexpr int kMoeRoundRows = kMoeMaxPos;    // rows of the units' experts scanned per round
constexpr int kMoeMaxMyUnits = 64;           // units of one CTA planned per round

template <int MAXT, int CFG, int RK>
__global__ void __launch_bounds__(MoeShape<CFG>::threads, MoeShape<CFG>::ctas) lora_moe_fold_kernel(const __grid_constant__ MoeArgs p) {
  constexpr int CW = MoeShape<CFG>::cw, PW = MoeShape<CFG>::pw, kMoeThreads = MoeShape<CFG>::threads;
  constexpr int kMoeRowsPerThread = (kMoeRoundRows + kMoeThreads - 1) / kMoeThreads;
  extern __shared__ __align__(128) unsigned char smem[];
  const FoldGeometry& g = p.g;
  const cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Plan& pl = *reinterpret_cast<Plan*>(smem);
  MoePlan& mp = *reinterpret_cast<MoePlan*>(smem + g.off_mplan);
  const int E = p.num_experts, A = p.adapters;
  const bool need_token = p.row_adapter != nullptr || p.x_gather != 0;
  const int G = gridDim.x, b = blockIdx.x;

  // Planning scratch in the ring (free until the first fold): the expert
  // offsets and, per round, the CTA's units (expert, first adapter, rows) and
  // the counts of their groups.
  unsigned char* ring = smem + g.off_ring;
  int* offs = reinterpret_cast<int*>(ring);
  int* u_e = offs + ((E + 4) & ~3);            // [kMoeMaxMyUnits] expert of each unit of the round
  int* u_a0 = u_e + kMoeMaxMyUnits;            // first adapter of its chunk
  int* u_lo = u_a0 + kMoeMaxMyUnits;           // its rows in the window: [u_lo, u_hi)
  int* u_row0 = u_lo + kMoeMaxMyUnits;         // prefix of the units' rows (+1 entry)
  int* bcnt = u_row0 + kMoeMaxMyUnits + 4;     // [units * ac] rows of each group in the round
  // The planning inputs read first: the expert offsets.
  auto load_inputs = [&]() {
    for (int i = tid; i <= E; i += kMoeThreads) offs[i] = p.expert_offsets[i];
  };

  // The ring's mbarriers read no input: they are set up while the previous
  // grid on the stream may still be running.
  if (tid == 0) {
    for (int s = 0; s < g.ns; ++s) {
      mbar_init(smem_u32(&pl.full[s]), PW * 32);
      mbar_init(smem_u32(&pl.empty[s]), CW);
    }
    pl.failed = 0;
    mbar_fence_init();
  }
  GLORA_STAMP(tid == 0, 0);
  GLORA_GTIME(tid == 0, 9);
  // Without a late wait nothing is read before the previous grid on the stream
  // has completed; with one, the engine waits before it touches base_out or xa,
  // and a CTA that folds nothing leaves at once, except CTA 0, which waits, so
  // that this grid never completes before the previous one.
  if (!p.late) pdl_wait_then_release();
  GLORA_STAMP(tid == 0, 1);
  auto leave = [&]() {
    if (p.late && blockIdx.x == 0) pdl_wait_then_release();
  };

  // Expert of sorted row r (-1 outside the spans): the largest e with offs[e] <= r.
  auto expert_of = [&](int r) -> int {
    if (r < offs[0] || r >= offs[E]) return -1;
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (offs[mid] <= r) lo = mid; else hi = mid;
    }
    return (offs[lo] <= r && r < offs[lo + 1]) ? lo : -1;
  };

  load_inputs();
  __syncthreads();
  const int lo_w = max(p.row_offset, offs[0]), hi_w = min(p.row_end, offs[E]);
  if (hi_w <= lo_w) return leave();              // every thread agrees
  int e_first = expert_of(lo_w), e_last = expert_of(hi_w - 1);
  if (e_first < 0 || e_last < e_first) { e_first = 0; e_last = E - 1; }   // offsets out of order: all experts
  const int E_w = e_last - e_first + 1;
  const int n_chunks0 = min(A, max(1, (kMoeUnitsPerCta * G) / E_w));
  const int ac = (A + n_chunks0 - 1) / n_chunks0, n_chunks = (A + ac - 1) / ac;
  const int n_units = E_w * n_chunks;   // <= num_experts * adapters <= kMoeMaxBins
  const int my_units = n_units > b ? (n_units - b + G - 1) / G : 0;

  const EngineArgs ea{p.x, p.x_stride, p.out, p.out_stride, p.xa, p.max_rank, p.k_in, p.n_out, p.late};
  int it0 = 0;
  bool ring_ready = false;
  // Rounds over the CTA's units: units [v0, v1) of its list and, within their
  // concatenated rows, rows [row_cur, row_cur + kMoeRoundRows).
  int v0 = 0, row_cur = 0;
  // Rows scanned per round: kMoeRoundRows, or kMoeMaxDesc when one unit's chunk
  // alone has more groups than a round holds runs (each row at most one run).
  const int round_rows = ac > kMoeMaxDesc ? kMoeMaxDesc : kMoeRoundRows;
  while (v0 < my_units) {
    if (ring_ready) {   // the ring holds the last round's stages: reload the planning inputs
      load_inputs();
      __syncthreads();
    }
    // at most kMoeMaxDesc groups (so runs) per round, or one unit
    const int v1 = min(my_units, v0 + min(kMoeMaxMyUnits, max(1, kMoeMaxDesc / ac)));
    const int nu = v1 - v0;
    if (tid < nu) {
      const int u = b + (v0 + tid) * G;
      const int e = e_first + u / n_chunks;
      u_e[tid] = e;
      u_a0[tid] = (u % n_chunks) * ac;
      u_lo[tid] = max(offs[e], lo_w);
      u_row0[tid] = max(0, min(offs[e + 1], hi_w) - max(offs[e], lo_w));
    }
    for (int i = tid; i < nu * ac; i += kMoeThreads) bcnt[i] = 0;
    // The table entries of the round's groups (at most kMoeMaxDesc, one per
    // thread): loaded into registers here, consumed after the row scan, so the
    // round trip overlaps it. Groups past the adapters are never routed.
    const bool cached = nu * ac <= kMoeMaxDesc;
    const uint16_t* tA = nullptr;
    const uint16_t* tB = nullptr;
    float tS = 0.f;
    if (cached && tid < nu * ac) {
      const int v = tid / ac, u = b + (v0 + v) * G;
      const int a = (u % n_chunks) * ac + (tid - v * ac), e = e_first + u / n_chunks;
      if (a < A) {
        tA = p.a_table[a * E + e];
        tB = p.b_table[a * E + e];
        tS = p.scale_table[a * E + e];
      }
    }
    __syncthreads();
    if (tid == 0) {   // prefix of the units' rows
      int run = 0;
      for (int v = 0; v < nu; ++v) {
        const int c = u_row0[v];
        u_row0[v] = run;
        run += c;
      }
      u_row0[nu] = run;
    }
    __syncthreads();
    const int rows_all = u_row0[nu];
    // this planning round: rows [row_cur, row_end) of the units' concatenated rows
    const int row_end = min(rows_all, row_cur + round_rows);
    // Each thread takes up to kMoeRowsPerThread rows of the round: their unit,
    // token and adapter (all token loads, then all adapter loads); a routed row
    // of its unit's chunk takes a rank in its group.
    int rr[kMoeRowsPerThread], tk[kMoeRowsPerThread], grp[kMoeRowsPerThread], rank[kMoeRowsPerThread];
    int uv[kMoeRowsPerThread];
#pragma unroll
    for (int j = 0; j < kMoeRowsPerThread; ++j) {
      const int q = row_cur + tid + j * kMoeThreads;
      rr[j] = -1;
      tk[j] = 0;
      uv[j] = 0;
      if (q < row_end) {
        int v = 0;
        while (u_row0[v + 1] <= q) ++v;
        uv[j] = v;
        rr[j] = u_lo[v] + (q - u_row0[v]);
        tk[j] = need_token ? p.sorted_token_ids[rr[j]] : 0;
      }
    }
#pragma unroll
    for (int j = 0; j < kMoeRowsPerThread; ++j) {
      grp[j] = -1;
      rank[j] = 0;
      if (rr[j] >= 0) {
        const int v = uv[j], t = tk[j];
        const bool tok_ok = !need_token || (t >= 0 && t < p.num_tokens);
        const int a = (tok_ok && p.row_adapter) ? p.row_adapter[t] : 0;
        if (tok_ok && expert_of(rr[j]) == u_e[v] && a >= u_a0[v] && a < min(A, u_a0[v] + ac)) {
          grp[j] = v * ac + (a - u_a0[v]);
          rank[j] = atomicAdd(&bcnt[grp[j]], 1);
        }
      }
    }
    __syncthreads();
    // Groups with rows become the round's runs (in group order); positions follow.
    if (warp == 0) {
      int carry_pos = 0, carry_run = 0;
      for (int c0 = 0; c0 < nu * ac; c0 += 32) {
        const int k = c0 + lane;
        const int n = k < nu * ac ? bcnt[k] : 0;
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const unsigned has = __ballot_sync(0xffffffffu, n > 0);
        const int d = carry_run + __popc(has & ((1u << lane) - 1u));
        if (n > 0) {
          MoeDesc& dd = mp.desc[d];
          const int v = k / ac;
          dd.e = u_e[v];
          dd.a = u_a0[v] + (k - v * ac);
          dd.n = n;
          dd.pos0 = carry_pos + incl - n;
          bcnt[k] = (d << 16) | 1;   // group k has rows, in run d (positions are pos0 + rank)
        }
        carry_pos += __shfl_sync(0xffffffffu, incl, 31);
        carry_run += __popc(has);
      }
      if (lane == 0) {
        mp.nd = carry_run;
        mp.npos = carry_pos;
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kMoeRowsPerThread; ++j) {
      if (grp[j] >= 0) {
        const int d = bcnt[grp[j]] >> 16;
        const int qpos = mp.desc[d].pos0 + rank[j];
        mp.pos_row[qpos] = rr[j];
        mp.pos_tok[qpos] = p.x_gather ? tk[j] : rr[j];
        mp.pos_desc[qpos] = static_cast<short>(d);
      }
    }
    const int nd = mp.nd, npos = mp.npos;
    // table entries of the runs
    auto set_entries = [&](MoeDesc& d, const uint16_t* Ap, const uint16_t* Bp, float sc) {
      const uintptr_t ua = reinterpret_cast<uintptr_t>(Ap), ub = reinterpret_cast<uintptr_t>(Bp);
      const bool usable = ua != 0 && ub != 0 && ((ua | ub) & 15u) == 0;
      if (ua != 0 && ub != 0 && !usable) atomicOr(&g_lora_status, kDevMisaligned);
      d.A = usable ? Ap : nullptr;
      d.B = Bp;
      d.scale = usable ? sc : 0.f;
    };
    if (cached) {   // the thread of each group with rows fills in its run
      if (tid < nu * ac && (bcnt[tid] & 1)) set_entries(mp.desc[bcnt[tid] >> 16], tA, tB, tS);
    } else {
      for (int k = tid; k < nd; k += kMoeThreads) {
        MoeDesc& d = mp.desc[k];
        const int idx = d.a * E + d.e;
        set_entries(d, p.a_table[idx], p.b_table[idx], p.scale_table[idx]);
      }
    }
    // next round
    if (row_end >= rows_all) {
      v0 = v1;
      row_cur = 0;
    } else {
      row_cur = row_end;
    }
    // the planner's generic writes to the ring before the ring's TMA writes
    fence_proxy_async_smem();
    __syncthreads();
    ring_ready = true;

    // ---- passes of up to kMaxRows positions ----
    for (int P0 = 0; P0 < npos; P0 += kMaxRows) {
      const int P = min(kMaxRows, npos - P0);
      if (tid < kMaxRows) {
        bool start = false;
        int k = -1;
        if (tid < P) {
          const int q = P0 + tid;
          k = mp.pos_desc[q];
          const int run = q - max(P0, mp.desc[k].pos0);   // rows of the run before this one in the pass
          start = (run % g.gmax) == 0;
          const int r = mp.pos_row[q];
          pl.members[tid] = tid;
          pl.grow[tid] = r;
          pl.xsrc[tid] = mp.pos_tok[q];
          pl.xarow[tid] = r - p.row_offset;
        }
        const unsigned sb = __ballot_sync(0xffffffffu, start);
        if (lane == 0) pl.ballots[tid >> 5] = sb;
        pl.flag[tid] = start ? k : -1;
      }
      __syncthreads();
      bool usable = true;   // this thread's group (if it starts one) has its adapter matrices
      if (tid < P) {
        const unsigned s0 = pl.ballots[0], s1 = pl.ballots[1];
        const unsigned below = tid < 32 ? (s0 & ((1u << tid) - 1u)) : s0;
        const int gid = __popc(below) + (tid < 32 ? 0 : __popc(s1 & ((1u << (tid - 32)) - 1u)));
        const int k = pl.flag[tid];
        if (k >= 0) {
          const MoeDesc& d = mp.desc[k];
          pl.gstart[gid] = tid;
          pl.gA[gid] = d.A;
          pl.gB[gid] = d.B;
          pl.gscale[gid] = d.scale;
          usable = d.A != nullptr;
        }
        if (tid == 0) {
          const int G0 = __popc(s0) + __popc(s1);
          pl.G = G0;
          pl.gstart[G0] = P;
        }
      }
      // Groups whose adapter matrices are NULL or misaligned are dropped (their
      // rows stay unchanged); the common case, every group usable, needs no
      // compaction. (The vote is also the barrier after the group table.)
      const bool all_usable = __syncthreads_and(usable) != 0;
      if (all_usable) {
        if (tid == 0) pl.NV = P;
      } else if (tid == 0) {
        int G1 = 0, nvk = 0;
        const int G0 = pl.G;
        for (int gi = 0; gi < G0; ++gi) {
          const int a0 = pl.gstart[gi], a1 = pl.gstart[gi + 1];
          if (pl.gA[gi] == nullptr) continue;
          const uint16_t* Ap = pl.gA[gi];
          const uint16_t* Bp = pl.gB[gi];
          const float sc = pl.gscale[gi];
          for (int i = a0; i < a1; ++i) pl.members[nvk + (i - a0)] = pl.members[i];
          pl.gstart[G1] = nvk;
          pl.gA[G1] = Ap;
          pl.gB[G1] = Bp;
          pl.gscale[G1] = sc;
          nvk += a1 - a0;
          ++G1;
        }
        pl.gstart[G1] = nvk;
        pl.G = G1;
        pl.NV = nvk;
      }
      __syncthreads();
      GLORA_STAMP(tid == 0, 2);
      if (pl.G > 0) it0 += fold_engine<MAXT, false, false, CW, PW, RK>(ea, g, pl, smem, cluster, 0, it0);
      __syncthreads();   // the next pass rewrites the plan
    }
    // Another round: the ring serves as planning scratch again (every item of
    // the last pass has been consumed).
  }
  leave();
  GLORA_STAMP(tid == 0, 8);
  GLORA_GTIME(tid == 0, 10);
}

// ============================================================================
// Launchers
// ============================================================================
template <typename Args>
static int launch_fold(void (*kernel)(Args), const Args& a, void* stream, int threads = kThreads) {
  const FoldGeometry& g = a.g;
  if (g.clusters <= 0) return 0;
  if (g.ns > kMaxStages) return static_cast<int>(cudaErrorInvalidValue);
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_bytes);
  if (err != cudaSuccess) return static_cast<int>(err);
  if (g.cl > 8) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return static_cast<int>(err);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(g.clusters * g.cl), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(g.smem_bytes);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = static_cast<unsigned>(g.cl);
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  err = cudaLaunchKernelEx(&cfg, kernel, a);
  return static_cast<int>(err);
}

// Rank class of a launch (the expand loop's variant): 1 = max_rank 16, 2 = 32,
// 0 = any other (the general variant, correct for every max_rank).
static int rank_class(int max_rank) { return max_rank == 16 ? 1 : max_rank == 32 ? 2 : 0; }

// maxt 4 needs more than one 16-row tile of rank (max_rank > 16): no rank-16 instance.
template <bool TILED, bool TC, int RK>
static int launch_bgmv_rk(const BgmvArgs& a, void* stream) {
  switch (a.g.maxt) {
    case 1: return launch_fold(lora_bgmv_fold_kernel<1, TILED, TC, RK>, a, stream);
    case 2: return launch_fold(lora_bgmv_fold_kernel<2, TILED, TC, RK>, a, stream);
    case 4:
      if constexpr (RK != 1) return launch_fold(lora_bgmv_fold_kernel<4, TILED, TC, RK>, a, stream);
      else return launch_fold(lora_bgmv_fold_kernel<4, TILED, TC, 0>, a, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}
int launch_bgmv(const BgmvArgs& a, void* stream) {
  const int rk = rank_class(a.max_rank);
  // tcgen05 shrink: max_rank in (112, 128]; A tensor maps: max_rank >= 32
  if (a.g.tc) return launch_bgmv_rk<true, true, 0>(a, stream);
  if (a.g.a_tiled) return rk == 2 ? launch_bgmv_rk<true, false, 2>(a, stream) : launch_bgmv_rk<true, false, 0>(a, stream);
  if (rk == 1) return launch_bgmv_rk<false, false, 1>(a, stream);
  if (rk == 2) return launch_bgmv_rk<false, false, 2>(a, stream);
  return launch_bgmv_rk<false, false, 0>(a, stream);
}

template <int CFG, int RK>
static int launch_moe_rk(const MoeArgs& a, void* stream) {
  constexpr int threads = MoeShape<CFG>::threads;
  switch (a.g.maxt) {
    case 1: return launch_fold(lora_moe_fold_kernel<1, CFG, RK>, a, stream, threads);
    case 2: return launch_fold(lora_moe_fold_kernel<2, CFG, RK>, a, stream, threads);
    case 4:
      if constexpr (RK != 1) return launch_fold(lora_moe_fold_kernel<4, CFG, RK>, a, stream, threads);
      else return launch_fold(lora_moe_fold_kernel<4, CFG, 0>, a, stream, threads);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}
template <int CFG>
static int launch_moe_cfg(const MoeArgs& a, void* stream) {
  switch (rank_class(a.max_rank)) {
    case 1: return launch_moe_rk<CFG, 1>(a, stream);
    case 2: return launch_moe_rk<CFG, 2>(a, stream);
    default: return launch_moe_rk<CFG, 0>(a, stream);
  }
}
int launch_moe(const MoeArgs& a, void* stream) {
  return a.g.moe_cfg ? launch_moe_cfg<1>(a, stream) : launch_moe_cfg<0>(a, stream);
}

// Self-test of the bounded wait every fold relies on: one thread waits on an
// mbarrier that nothing arrives at, with a limit of `limit_cycles` SM clocks;
// giving up sets the timeout bit of the device status word, as in the folds.
__global__ void lora_wait_selftest_kernel(long long limit_cycles) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_limit(smem_u32(&bar), 0, limit_cycles)) atomicOr(&g_lora_status, kDevTimeout);
}

int launch_wait_selftest(long long limit_cycles, void* stream) {
  lora_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_cycles);
  return static_cast<int>(cudaGetLastError());
}

int read_device_status(void* stream, uint32_t* out, int clear) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  cudaError_t err = cudaMemcpyFromSymbolAsync(&v, g_lora_status, sizeof v, 0, cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  if (err == cudaSuccess && clear) {
    const unsigned int z = 0;
    err = cudaMemcpyToSymbolAsync(g_lora_status, &z, sizeof z, 0, cudaMemcpyHostToDevice, s);
    if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  }
  if (out) *out = v;
  return static_cast<int>(err);
}

}  // namespace glora
