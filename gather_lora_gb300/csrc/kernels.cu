// Fold kernels for sm_103a: routed bgmv and MoE grouped fold.
//
// Method (pages): "Function apply_lora_bgmv" rustdoc (spark_model lora_delta) —
// per row, shrink x @ A_s^T to BF16 xa, expand xa @ B_s^T, round the delta to
// BF16, then out += scale_s * delta in fp32; "Module moe_lora_grouped" rustdoc —
// the same fold over expert-sorted rows of a window, keyed by expert and gated
// per token by moe_row_adapter.
//
// GB300 design (one launch per call, no global scratch):
//   * A cluster of `cl` CTAs owns one WORK UNIT: up to 64 rows split into
//     groups that share one adapter (bgmv: rows of one slot; MoE: the
//     (adapter, expert) groups of a 64-row tile of sorted rows). Every CTA of
//     the cluster builds the same plan from the routing data.
//   * Shrink: CTA `rank` contracts its k-slice [rank*ksl, +ksl) of every
//     group's A with the group's x rows on the tensor cores (mma.sync BF16,
//     fp32 accumulate), adapter and activation chunks streaming through a
//     cp.async ring so each adapter byte is read once per unit.
//   * The fp32 partials of the cl k-slices are reduced in distributed shared
//     memory in rank order (reduce-scatter), rounded to BF16 once, and the
//     BF16 xa is pushed to every CTA of the cluster.
//   * Expand + fold: CTA `rank` takes its j-slice of every group's B (streamed
//     through the same ring, prefetched while the shrink finishes), computes
//     d = bf16(xa @ B^T) on the tensor cores and folds
//     out = bf16(fma(scale, d, out)) into a staged copy of the out rows, which
//     is written back with 16-byte stores.
// A row's fp32 summation order is fixed by (k_in, max_rank, cl): it never
// depends on which other rows share its launch, group or tile.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <limits.h>

#include "common.cuh"
#include "fold_types.h"

namespace cg = cooperative_groups;

// Device status word (LORA_DEV_* bits), read and cleared through read_device_status().
__device__ unsigned int g_lora_status = 0;

namespace glora {

constexpr unsigned kDevMisaligned = 0x1u;

// Work-unit plan, identical in every CTA of a cluster.
struct Plan {
  int G;                           // groups (0: nothing to do)
  int NV;                          // valid positions (sum of group sizes)
  int warp_sums[kWarps];
  int found_slot, found_tile, found_rows;  // bgmv planning scratch
  int members[kMaxRows];           // positions, grouped, ascending within a group
  int gstart[kMaxRows + 1];        // group g = members[gstart[g] .. gstart[g+1])
  int grow[kMaxRows];              // position -> row of x / base_out
  int xarow[kMaxRows];             // position -> row of xa
  int key[kMaxRows];               // MoE: table index of the position (INT_MAX: skipped)
  float gscale[kMaxRows];
  float pscale[kMaxRows];
  const uint16_t* gA[kMaxRows];
  const uint16_t* gB[kMaxRows];
  const uint16_t* pA[kMaxRows];
  const uint16_t* pB[kMaxRows];
};

static_assert(sizeof(Plan) <= kPlanBytes, "plan does not fit its shared-memory reservation");

struct EngineArgs {
  const uint16_t* x;
  long long x_stride;
  uint16_t* out;
  long long out_stride;
  uint16_t* xa;
  int max_rank, k_in, n_out;
};

// Shrink, cluster exchange, expand + fold for one planned work unit.
__device__ __forceinline__ void fold_engine(const EngineArgs& p, const FoldGeometry& g, const Plan& pl,
                                            unsigned char* smem, const cg::cluster_group& cluster,
                                            int crank) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned char* ring = smem + g.off_ring;
  unsigned char* out_s = smem + g.off_out;
  float* part_s = reinterpret_cast<float*>(smem + g.off_part);
  uint16_t* xa_s = reinterpret_cast<uint16_t*>(smem + g.off_xa);
  const int G = pl.G, NV = pl.NV;
  const int xa_pitch_el = g.pitch_xa >> 1;

  const int k_lo = crank * g.ksl, k_hi = min(k_lo + g.ksl, p.k_in);
  const int j_lo = crank * g.jsl, j_hi = min(j_lo + g.jsl, p.n_out);
  const int nk = k_hi > k_lo ? (k_hi - k_lo + g.kch - 1) / g.kch : 0;
  const int nj = j_hi > j_lo ? (j_hi - j_lo + g.jch - 1) / g.jch : 0;
  const int n_shrink = G * nk, n_items = G * (nk + nj);
  const int jw = max(j_hi - j_lo, 0);

  // Prologue: this CTA's out segment of every valid row (needed at the end).
  {
    const int cpr = jw >> 3;
    for (int q = tid; q < NV * cpr; q += kThreads) {
      const int mi = q / cpr, c = q - mi * cpr, pos = pl.members[mi];
      cp_async16(smem_u32(out_s + pos * g.pitch_out + c * 16),
                 p.out + (long long)pl.grow[pos] * p.out_stride + j_lo + c * 8);
    }
    cp_async_commit();
  }

  // Ring items: [group g, k-chunk] for the shrink, then [group g, j-chunk] for
  // the expand. Item `it` lives in stage it % ns. Always commits a group so
  // that the wait counts stay uniform.
  auto issue = [&](int it) {
    if (it < n_items) {
      unsigned char* st = ring + (it % g.ns) * g.stage_bytes;
      if (it < n_shrink) {
        const int gi = it / nk, kc = it - gi * nk;
        const int k0 = k_lo + kc * g.kch, klen = min(g.kch, k_hi - k0), cpr = klen >> 3;
        const int m0 = pl.gstart[gi], R = pl.gstart[gi + 1] - m0;
        const uint16_t* A = pl.gA[gi];
        const int na = p.max_rank * cpr, tot = na + R * cpr;
        for (int q = tid; q < tot; q += kThreads) {
          if (q < na) {
            const int c = q / cpr, ch = q - c * cpr;
            cp_async16(smem_u32(st + c * g.pitch_k + ch * 16), A + (long long)c * p.k_in + k0 + ch * 8);
          } else {
            const int qq = q - na, r = qq / cpr, ch = qq - r * cpr;
            cp_async16(smem_u32(st + (g.mr16 + r) * g.pitch_k + ch * 16),
                       p.x + (long long)pl.grow[pl.members[m0 + r]] * p.x_stride + k0 + ch * 8);
          }
        }
      } else {
        const int e = it - n_shrink, gi = e / nj, jc = e - gi * nj;
        const int j0 = j_lo + jc * g.jch, jlen = min(g.jch, j_hi - j0), cpr = p.max_rank >> 3;
        const uint16_t* B = pl.gB[gi];
        for (int q = tid; q < jlen * cpr; q += kThreads) {
          const int j = q / cpr, ch = q - j * cpr;
          cp_async16(smem_u32(st + j * g.pitch_b + ch * 16), B + (long long)(j0 + j) * p.max_rank + ch * 8);
        }
      }
    }
    cp_async_commit();
  };
  for (int it = 0; it < g.ns - 1; ++it) issue(it);

  // ---- shrink: fp32 partial xa of this k-slice ------------------------------
  const int MT = g.mr16 >> 4;
  float acc[kMaxTilesPerWarp][4];
#pragma unroll
  for (int i = 0; i < kMaxTilesPerWarp; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  if (nk == 0) {  // empty k-slice: the partials are zero
    for (int e = tid; e < NV * p.max_rank; e += kThreads) {
      const int mi = e / p.max_rank, c = e - mi * p.max_rank;
      part_s[pl.members[mi] * g.pitch_part + c] = 0.f;
    }
  }
  for (int it = 0; it < n_shrink; ++it) {
    cp_async_wait(g.ns - 2);
    __syncthreads();
    issue(it + g.ns - 1);
    const int gi = it / nk, kc = it - gi * nk;
    const int m0 = pl.gstart[gi], R = pl.gstart[gi + 1] - m0, NT = (R + 7) >> 3, ntiles = MT * NT;
    const int k0 = k_lo + kc * g.kch, klen = min(g.kch, k_hi - k0);
    const uint32_t st_a = smem_u32(ring + (it % g.ns) * g.stage_bytes);
    const uint32_t st_x = st_a + g.mr16 * g.pitch_k;
    for (int kk = 0; kk < klen; kk += 16) {
      const int kstep = min(16, klen - kk);
#pragma unroll
      for (int i = 0; i < kMaxTilesPerWarp; ++i) {
        const int t = warp + i * kWarps;
        if (t < ntiles) {
          const int mt = t % MT, nt = t / MT;
          mma_step(acc[i], st_a + (mt * 16 + (lane & 15)) * g.pitch_k + kk * 2,
                   st_x + (nt * 8 + (lane & 7)) * g.pitch_k + kk * 2, kstep, lane);
        }
      }
    }
    if (kc == nk - 1) {  // group complete: partials -> shared memory
#pragma unroll
      for (int i = 0; i < kMaxTilesPerWarp; ++i) {
        const int t = warp + i * kWarps;
        if (t < ntiles) {
          const int mt = t % MT, nt = t / MT;
          const int c0 = mt * 16 + (lane >> 2), r0 = nt * 8 + 2 * (lane & 3);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int c = c0 + (v >> 1) * 8, r = r0 + (v & 1);
            if (c < p.max_rank && r < R) part_s[pl.members[m0 + r] * g.pitch_part + c] = acc[i][v];
          }
        }
        acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
      }
    }
  }

  // ---- cluster exchange: xa = bf16(sum of the cl partials, in rank order) ----
  cluster.sync();
  {
    const int E = NV * p.max_rank, per = (E + g.cl - 1) / g.cl;
    const int e_lo = crank * per, e_hi = min(e_lo + per, E);
    for (int e = e_lo + tid; e < e_hi; e += kThreads) {
      const int mi = e / p.max_rank, c = e - mi * p.max_rank, pos = pl.members[mi];
      const int off = pos * g.pitch_part + c;
      float s = cluster.map_shared_rank(part_s, 0)[off];
      for (int q = 1; q < g.cl; ++q) s += cluster.map_shared_rank(part_s, q)[off];
      const uint16_t xb = f32_to_bf16_bits(s);
      const int xoff = pos * xa_pitch_el + c;
      for (int q = 0; q < g.cl; ++q) cluster.map_shared_rank(xa_s, q)[xoff] = xb;
      if (p.xa) p.xa[(long long)pl.xarow[pos] * p.max_rank + c] = xb;
    }
  }
  cluster.sync();

  // ---- expand + fold over this CTA's j-slice ---------------------------------
  const uint32_t xa_base = smem_u32(xa_s);
  for (int it = n_shrink; it < n_items; ++it) {
    cp_async_wait(g.ns - 2);
    __syncthreads();
    issue(it + g.ns - 1);
    const int e = it - n_shrink, gi = e / nj, jc = e - gi * nj;
    const int m0 = pl.gstart[gi], R = pl.gstart[gi + 1] - m0, NT = (R + 7) >> 3;
    const int j0 = j_lo + jc * g.jch, jlen = min(g.jch, j_hi - j0), MTj = (jlen + 15) >> 4;
    const int tiles = MTj * NT;
    const float scale = pl.gscale[gi];
    const uint32_t st_b = smem_u32(ring + (it % g.ns) * g.stage_bytes);
    for (int t = warp; t < tiles; t += kWarps) {
      const int mt = t % MTj, nt = t / MTj;
      const int bpos = pl.members[m0 + min(nt * 8 + (lane & 7), R - 1)];
      float d4[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kk = 0; kk < p.max_rank; kk += 16) {
        mma_step(d4, st_b + (mt * 16 + (lane & 15)) * g.pitch_b + kk * 2,
                 xa_base + bpos * g.pitch_xa + kk * 2, min(16, p.max_rank - kk), lane);
      }
      const int jj0 = mt * 16 + (lane >> 2), rr0 = nt * 8 + 2 * (lane & 3);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int jj = jj0 + (v >> 1) * 8, rr = rr0 + (v & 1);
        if (jj < jlen && rr < R) {
          uint16_t* o = reinterpret_cast<uint16_t*>(out_s + pl.members[m0 + rr] * g.pitch_out) + (j0 - j_lo) + jj;
          *o = fold_one(d4[v], scale, *o);
        }
      }
    }
  }
  cp_async_wait(0);
  __syncthreads();

  // ---- write the folded out segments back -----------------------------------
  {
    const int cpr = jw >> 3;
    for (int q = tid; q < NV * cpr; q += kThreads) {
      const int mi = q / cpr, c = q - mi * cpr, pos = pl.members[mi];
      const uint4 v = *reinterpret_cast<const uint4*>(out_s + pos * g.pitch_out + c * 16);
      *reinterpret_cast<uint4*>(p.out + (long long)pl.grow[pos] * p.out_stride + j_lo + c * 8) = v;
    }
  }
}

// ============================================================================
// Routed bgmv: work unit = up to rt rows of one slot, in ascending row order.
// Units are numbered slot by slot (ascending slot, then ascending tile), so the
// static grid bound is n/rt + min(n, max_loras) units.
// ============================================================================
__global__ void __launch_bounds__(kThreads, 2) lora_bgmv_fold_kernel(const __grid_constant__ BgmvArgs p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const FoldGeometry& g = p.g;
  const cg::cluster_group cluster = cg::this_cluster();
  const int crank = static_cast<int>(cluster.block_rank());
  const int unit = static_cast<int>(blockIdx.x) / g.cl;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Plan& pl = *reinterpret_cast<Plan*>(smem);

  pdl_wait_then_release();

  // Routed rows per slot (histogram in the not-yet-used ring).
  int* cnt = reinterpret_cast<int*>(smem + g.off_ring);
  for (int s = tid; s < p.max_loras; s += kThreads) cnt[s] = 0;
  if (tid == 0) pl.found_slot = -1;
  __syncthreads();
  for (int i = tid; i < p.n; i += kThreads) {
    const int s = p.seq_slot[i];
    if (s >= 0 && s < p.max_loras) atomicAdd(&cnt[s], 1);
  }
  __syncthreads();
  for (int s = tid; s < p.max_loras; s += kThreads) {
    if (cnt[s] > 0) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(p.a_table[s]);
      const uintptr_t b = reinterpret_cast<uintptr_t>(p.b_table[s]);
      if (a == 0 || b == 0) {
        cnt[s] = 0;
      } else if ((a | b) & 15u) {
        cnt[s] = 0;
        if (unit == 0 && crank == 0) atomicOr(&g_lora_status, kDevMisaligned);
      }
    }
  }
  __syncthreads();
  // Units per slot, prefix over slots, locate this cluster's (slot, tile).
  {
    const int per = (p.max_loras + kThreads - 1) / kThreads;
    const int lo = min(tid * per, p.max_loras), hi = min(lo + per, p.max_loras);
    int local = 0;
    for (int s = lo; s < hi; ++s) local += (cnt[s] + g.rt - 1) / g.rt;
    int run = block_inclusive_sum(local, pl.warp_sums) - local;
    for (int s = lo; s < hi; ++s) {
      const int t = (cnt[s] + g.rt - 1) / g.rt;
      if (unit >= run && unit < run + t) {
        pl.found_slot = s;
        pl.found_tile = unit - run;
        pl.found_rows = min(g.rt, cnt[s] - (unit - run) * g.rt);
      }
      run += t;
    }
  }
  __syncthreads();
  const int slot = pl.found_slot;
  if (slot < 0) return;  // every CTA of the cluster takes this branch together
  const int R = pl.found_rows, want_lo = pl.found_tile * g.rt;

  // Rows of this slot in ascending order; keep ranks [want_lo, want_lo + R).
  {
    int base = 0;
    for (int i0 = 0; i0 < p.n; i0 += kThreads) {
      const int i = i0 + tid;
      const bool f = (i < p.n) && (p.seq_slot[i] == slot);
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
      if (f && rank >= want_lo && rank < want_lo + R) {
        const int pos = rank - want_lo;
        pl.members[pos] = pos;
        pl.grow[pos] = i;
        pl.xarow[pos] = i;
      }
      base += total;
      __syncthreads();
    }
  }
  if (tid == 0) {
    pl.G = 1;
    pl.NV = R;
    pl.gstart[0] = 0;
    pl.gstart[1] = R;
    pl.gA[0] = p.a_table[slot];
    pl.gB[0] = p.b_table[slot];
    pl.gscale[0] = p.scale_table[slot];
  }
  __syncthreads();

  const EngineArgs ea{p.x, p.x_stride, p.out, p.out_stride, p.xa, p.max_rank, p.k_in, p.n_out};
  fold_engine(ea, g, pl, smem, cluster, crank);
}

// ============================================================================
// MoE grouped fold: work unit = one 64-row tile of the window's sorted rows,
// split into (adapter, expert) groups; grid = ceil(window / 64) tiles (>= 1).
// ============================================================================
__global__ void __launch_bounds__(kThreads, 2) lora_moe_fold_kernel(const __grid_constant__ MoeArgs p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const FoldGeometry& g = p.g;
  const cg::cluster_group cluster = cg::this_cluster();
  const int crank = static_cast<int>(cluster.block_rank());
  const int tile = static_cast<int>(blockIdx.x) / g.cl;
  const int tid = threadIdx.x;
  Plan& pl = *reinterpret_cast<Plan*>(smem);
  const int E = p.num_experts;

  pdl_wait_then_release();

  const int r0 = p.row_offset + tile * g.rt;
  const int T = min(g.rt, p.row_end - r0);
  int* offs = reinterpret_cast<int*>(smem + g.off_ring);  // expert_offsets copy (ring not yet used)
  for (int i = tid; i <= E; i += kThreads) offs[i] = p.expert_offsets[i];
  __syncthreads();

  // Per position: expert by binary search, adapter gate, table entry.
  if (tid < g.rt) {
    int key = INT_MAX;
    const int r = r0 + tid;
    if (tid < T && r >= offs[0] && r < offs[E]) {
      int lo = 0, hi = E;  // largest e in [0, E) with offs[e] <= r
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offs[mid] <= r) lo = mid; else hi = mid;
      }
      const int e = lo;
      if (offs[e] <= r && r < offs[e + 1]) {
        int a = 0;
        bool ok = true;
        if (p.row_adapter) {
          const int t = p.sorted_token_ids[r];
          if (t < 0 || t >= p.num_tokens) ok = false; else a = p.row_adapter[t];
        }
        if (ok && a >= 0 && a < p.max_loras) {
          const int idx = a * E + e;
          const uint16_t* A = p.a_table[idx];
          const uint16_t* B = p.b_table[idx];
          const uintptr_t ua = reinterpret_cast<uintptr_t>(A), ub = reinterpret_cast<uintptr_t>(B);
          if (ua != 0 && ub != 0) {
            if ((ua | ub) & 15u) {
              atomicOr(&g_lora_status, kDevMisaligned);
            } else {
              key = idx;
              pl.pA[tid] = A;
              pl.pB[tid] = B;
              pl.pscale[tid] = p.scale_table[idx];
            }
          }
        }
      }
    }
    pl.key[tid] = key;
    pl.grow[tid] = r;
    pl.xarow[tid] = r - p.row_offset;
  }
  __syncthreads();
  // Stable sort of the valid positions by table index.
  int nv = 0;
  {
    int k = INT_MAX;
    if (tid < g.rt) {
      k = pl.key[tid];
      int rank = 0;
      for (int u = 0; u < g.rt; ++u) {
        const int ku = pl.key[u];
        rank += (ku < k) || (ku == k && u < tid);
      }
      if (k != INT_MAX) pl.members[rank] = tid;
    }
    nv = __syncthreads_count(tid < g.rt && k != INT_MAX);
  }
  if (nv == 0) return;  // every CTA of the cluster takes this branch together
  if (tid == 0) {
    int G = 0, prev = INT_MAX;
    for (int i = 0; i < nv; ++i) {
      const int pos = pl.members[i], k = pl.key[pos];
      if (i == 0 || k != prev || i - pl.gstart[G - 1] >= g.gmax) {
        pl.gstart[G] = i;
        pl.gA[G] = pl.pA[pos];
        pl.gB[G] = pl.pB[pos];
        pl.gscale[G] = pl.pscale[pos];
        ++G;
        prev = k;
      }
    }
    pl.gstart[G] = nv;
    pl.G = G;
    pl.NV = nv;
  }
  __syncthreads();

  const EngineArgs ea{p.x, p.x_stride, p.out, p.out_stride, p.xa, p.max_rank, p.k_in, p.n_out};
  fold_engine(ea, g, pl, smem, cluster, crank);
}

// ============================================================================
// Launchers
// ============================================================================
template <typename Args>
static int launch_fold(void (*kernel)(Args), const Args& a, void* stream) {
  const FoldGeometry& g = a.g;
  if (g.clusters <= 0) return 0;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_bytes);
  if (err != cudaSuccess) return static_cast<int>(err);
  if (g.cl > 8) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return static_cast<int>(err);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(g.clusters * g.cl), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
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

int launch_bgmv(const BgmvArgs& a, void* stream) { return launch_fold(lora_bgmv_fold_kernel, a, stream); }
int launch_moe(const MoeArgs& a, void* stream) { return launch_fold(lora_moe_fold_kernel, a, stream); }

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
