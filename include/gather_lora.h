/*
 * gather_lora.h — C ABI of the routed multi-LoRA fold for NVIDIA GB300 (sm_103a).
 *
 * Four folds, each one kernel launch on the caller's stream (lora_delta on
 * its row-by-row path: one per LORA_MAX_ROWS rows):
 *
 *   lora_bgmv             per-request routed LoRA delta over n rows
 *   lora_moe_grouped_fold the same fold over expert-sorted MoE rows of one window
 *   lora_moe_gather_bgmv  the decode-path MoE fold over flat (token, slot) rows
 *   lora_delta            one adapter pair folded into every row (prefill)
 *
 * plus lora_encode_a_tmaps (TMA tensor maps of the A matrices, encoded once on
 * the host), diagnostics (status word, geometry queries, a bounded-wait self
 * test) and five pure host helpers (no GPU needed) for the MoE windows, grids
 * and tables.
 *
 * Conventions for every entry point
 *   - BF16 values are raw 16-bit patterns (lora_bf16_t); f32 is IEEE float.
 *   - Every pointer argument of the folds is DEVICE memory owned by the
 *     caller; the library allocates, frees and synchronizes nothing, and
 *     returns as soon as the launch is queued.
 *   - Strides are in ELEMENTS, not bytes.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Return value: LORA_OK (0), or a negative lora_status. Every argument
 *     check runs on the host BEFORE any launch: a negative return other than
 *     LORA_ERR_CUDA means nothing was launched. LORA_ERR_CUDA means the launch
 *     itself failed; lora_last_error() gives the text (per host thread).
 *   - Bad DEVICE data is never a fault: a slot outside [0, max_loras), a NULL
 *     table entry, a token or adapter out of range, a row outside the expert
 *     spans all mean "this row gets no delta". A table entry that is not
 *     16-byte aligned is skipped too and sets LORA_DEV_MISALIGNED in the
 *     device status word (lora_read_device_status).
 *   - Every fold is capture-safe: the launch shape depends only on the host
 *     integers passed in, so a CUDA graph captured once replays correctly
 *     when only device buffer CONTENTS (seq_slot, row_adapter, offsets, x,
 *     base_out) change.
 *
 * Alignment (this library's own restriction; the method states none): x,
 * base_out and xa must be 16-byte aligned; k_in, n_out, max_rank and both row
 * strides must be multiples of 8; adapter matrices must be 16-byte aligned.
 * Otherwise the call returns LORA_ERR_ALIGN (there is no fallback path).
 *
 * Numerics (the rounding order of the method): per row, fp32 accumulation of
 * BF16 products; xa rounded to BF16 (RNE); the expand sum rounded to BF16
 * (RNE); then out = bf16_rn(fmaf(scale, delta, out)). The fp32 summation
 * order is fixed by (k_in, max_rank) alone, so a row's result never depends
 * on which or how many other rows share the call (batch invariance).
 */
#ifndef GATHER_LORA_H
#define GATHER_LORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t lora_bf16_t;

enum lora_status {
    LORA_OK = 0,
    LORA_ERR_NULL = -1,        /* a required pointer is NULL */
    LORA_ERR_SIZE = -2,        /* a size or count is outside its supported range */
    LORA_ERR_STRIDE = -3,      /* a row stride is smaller than the row width */
    LORA_ERR_ALIGN = -4,       /* a pointer, stride or width breaks the alignment rule */
    LORA_ERR_WINDOW = -5,      /* MoE window outside [0, te] or row_end < row_offset */
    LORA_ERR_CUDA = -6,        /* the CUDA launch (or a device query) failed */
    LORA_ERR_UNSUPPORTED = -7, /* the current device cannot run these kernels */
    LORA_ERR_FLAGS = -8        /* an unknown bit is set in `flags` */
};

/*
 * Call flags (the `flags` argument of lora_bgmv, lora_moe_grouped_fold and
 * lora_moe_gather_bgmv; 0 = none).
 *
 * LORA_INPUTS_READY: the caller promises that every input of the call other
 * than base_out and xa (x, the routing arrays, the tables and the adapter
 * matrices they point to) is written by no kernel that may still be running
 * when this call's kernel starts. The kernels of this library let the next
 * launch on the stream start once they themselves have waited for the one
 * before them, so for a stream of calls of this library the promise reads:
 * the kernel launched just before this call does not write those inputs (as
 * for successive windows of one MoE layer, or a fold right after the base
 * GEMM that writes base_out). The kernel then plans, loads and runs its shrink
 * while the previous kernel finishes, and waits for it only before it reads
 * or writes base_out or writes xa. Without the flag it waits before reading
 * anything. The results are the same bits either way. The overlap is CUDA's
 * programmatic dependent launch, which relaxes only the order between two
 * kernel launches: copies and event waits before the call on the stream are
 * waited for as usual.
 */
#define LORA_INPUTS_READY 0x1u

/* Device status bits, set by kernels, read with lora_read_device_status(). */
#define LORA_DEV_MISALIGNED 0x1u   /* an adapter table entry was not 16-byte aligned */
#define LORA_DEV_TIMEOUT 0x2u      /* a kernel gave up waiting for its own copies (~2 s); its
                                      results were not stored */

/* Supported ranges, checked on every call. */
#define LORA_MAX_RANK 256          /* max_rank in [8, 256], multiple of 8 */
#define LORA_MAX_K_IN (1 << 20)    /* k_in in [8, 2^20], multiple of 8 */
#define LORA_MAX_N_OUT (1 << 20)   /* n_out in [8, 2^20], multiple of 8 */
#define LORA_MAX_ROWS 8192         /* n of lora_bgmv in [0, 8192] */
#define LORA_MAX_LORAS 4096        /* max_loras of lora_bgmv in [1, 4096] */
#define LORA_MAX_EXPERTS 1024      /* num_experts of the MoE fold in [1, 1024] */
#define LORA_TMAP_MIN_RANK 32      /* a_tmaps are used from this max_rank up */
#define LORA_MAX_DELTA_ROWS (1 << 20)      /* m of lora_delta in [0, 2^20] */
#define LORA_DELTA_DENSE_MIN_ROWS 256      /* lora_delta takes the tensor-core path from this m up */
#define LORA_MOE_M_TILE 64         /* sorted rows per MoE m-tile (window tile count; rows per fold pass) */

/*
 * lora_bgmv — per-request routed LoRA delta over n rows.
 *
 * Defines: "Function apply_lora_bgmv" (spark_model::layers::ops::lora_delta
 * rustdoc), the summary, BYTE-IDENTICAL, STRIDES and GRAPH-SAFE paragraphs;
 * lora_delta.rs (metrale source listing), `LoraRoute` and `LoraPair`.
 *
 * For every row i in [0, n) with s = seq_slot[i], 0 <= s < max_loras and both
 * a_table[s] and b_table[s] non-NULL:
 *     xa[i, c]  = bf16( sum_k x[i, k] * A_s[c, k] )          c < max_rank
 *     d[j]      = bf16( sum_c xa[i, c] * B_s[j, c] )         j < n_out
 *     out[i, j] = bf16( fmaf(scale_table[s], d[j], out[i, j]) )
 * Every other row, and every element outside out[i, 0:n_out), is left
 * byte-for-byte unchanged.
 *
 *   x            [n rows, x_row_stride] BF16; row i's input is x[i*x_row_stride .. +k_in)
 *   base_out     [n rows, out_row_stride] BF16, folded IN PLACE; row i's segment is
 *                base_out[i*out_row_stride .. +n_out). To fold into the K part of an
 *                interleaved [Q|K|V] row, pass base_out = qkv + q_width and
 *                out_row_stride = q_width + k_width + v_width.
 *   seq_slot     [n] int32 adapter slot per row (< 0 = no delta)
 *   a_table      [max_loras] device pointers to A_s, [max_rank, k_in] row-major BF16
 *   b_table      [max_loras] device pointers to B_s, [n_out, max_rank] row-major BF16
 *                (rank-padded: rows of A / columns of B past the adapter's rank are 0)
 *   scale_table  [max_loras] f32 per-slot scale (alpha/r, or alpha/sqrt(r) for rsLoRA)
 *   xa           optional [n, max_rank] BF16 output of the shrink (routed rows only
 *                are written); NULL skips it
 *   a_tmaps      optional device array of [max_loras] 128-byte TMA tensor maps of the
 *                A matrices, written by lora_encode_a_tmaps for the same a_table
 *                pointers, max_rank and k_in, 64-byte aligned. Given and max_rank >=
 *                LORA_TMAP_MIN_RANK, A is loaded as 2-D boxes (far fewer copy
 *                requests); NULL, or a smaller max_rank, loads A row by row (boxes
 *                of under 32 rows measured slower than the row copies on GB300).
 *                The results are the same bits either way. The caller keeps the
 *                maps in step with a_table (adapters are load-time fixed); an entry
 *                used by a routed row must describe that adapter.
 *   flags        0 or LORA_INPUTS_READY (above); other bits give LORA_ERR_FLAGS
 *   n == 0 is a no-op (returns LORA_OK, nothing launched).
 */
int lora_bgmv(const lora_bf16_t* x, int64_t x_row_stride,
              lora_bf16_t* base_out, int64_t out_row_stride,
              const int32_t* seq_slot, int32_t n,
              const lora_bf16_t* const* a_table, const lora_bf16_t* const* b_table,
              const float* scale_table, int32_t max_loras,
              int32_t max_rank, int32_t k_in, int32_t n_out,
              lora_bf16_t* xa, const void* a_tmaps, uint32_t flags, void* stream);

/*
 * lora_moe_grouped_fold — the fold over expert-sorted MoE rows of one window.
 *
 * Defines: "Module moe_lora_grouped" (atlas rustdoc), the module summary and the
 * `moe_lora_grouped_down`, `MoeExpertRoute` and `MLG_M_TILE` entries. Down
 * (x_gather == 0): x is the sorted [te, k_in] activation and row r of it feeds
 * sorted row r. Gate/up (x_gather != 0): x is the token-major [num_tokens, k_in]
 * expert input and sorted row r reads row sorted_token_ids[r] of it.
 *
 * For every sorted row r in [row_offset, row_end):
 *   e = the expert with expert_offsets[e] <= r < expert_offsets[e+1]
 *       (rows outside [expert_offsets[0], expert_offsets[num_experts]) are skipped);
 *   t = sorted_token_ids[r] (read with a row_adapter or x_gather; skipped if t
 *       is outside [0, num_tokens));
 *   a = row_adapter ? row_adapter[t] : 0 (skipped if a is outside [0, max_loras));
 *   t = a * num_experts + e (adapter-major tables); skipped if a_table[t] or
 *       b_table[t] is NULL; otherwise the fold of lora_bgmv is applied to
 *       x[xr*x_row_stride ..] (xr = x_gather ? t : r) and
 *       base_out[r*out_row_stride ..] with A_t, B_t, scale_table[t].
 *
 *   expert_offsets    [num_experts + 1] int32 prefix sum (non-decreasing; offsets out
 *                     of order are bad data that fold no row twice, for windows under
 *                     2^25 rows: the planner sums its units' spans in 32 bits)
 *   sorted_token_ids  [te] int32 sorted row -> token; may be NULL when row_adapter is
 *                     NULL and x_gather == 0
 *   row_adapter       [num_tokens] int32 (< 0 = no delta), or NULL: every row uses adapter 0
 *   a_table, b_table, scale_table   [max_loras * num_experts], index a*num_experts + e
 *   xa                optional [xa_rows, max_rank] BF16 shrink output, written at the
 *                     LOCAL row r - row_offset (routed rows only); NULL skips it
 *   xa_rows           rows the caller allocated for xa. The window writes local rows
 *                     [0, row_end - row_offset), so xa != NULL with xa_rows < row_end -
 *                     row_offset (or < 0) is rejected with LORA_ERR_SIZE before any
 *                     launch; ignored when xa is NULL ("Module moe_lora_grouped",
 *                     `moe_lora_grouped_down`: the caller needs at least the window's rows)
 *   flags             0 or LORA_INPUTS_READY (above); other bits give LORA_ERR_FLAGS.
 *                     Successive windows of one layer may all pass it: each window
 *                     then plans and shrinks while the previous one finishes (xa
 *                     is written only after that wait, so the windows may share it)
 * The window must satisfy 0 <= row_offset <= row_end <= te (else LORA_ERR_WINDOW);
 * the tables may hold at most LORA_MAX_LORAS entries (max_loras * num_experts),
 * else LORA_ERR_SIZE (so is a shape whose stages do not fit shared memory). The
 * launch grid is persistent and static: one CTA per SM, or two smaller ones when
 * the shrink is the larger half of the work (k_in > n_out), fewer for windows
 * under 16 rows per CTA (at least 1), so it depends only on the shapes, the
 * window size and the device. Each CTA takes a fixed share of the window's units
 * (one expert and a chunk of adapters) and folds the rows of their (expert,
 * adapter) groups; which rows share a group never changes a row's bits. Calls
 * over windows [0, cap), [cap, 2cap), ... give the same base_out as one call
 * over [0, te). The fold never reads xa back, so a caller whose xa holds all te
 * rows, or who passes NULL, can make that one call: it also spares the wait of
 * each window for the previous one's last CTA.
 */
int lora_moe_grouped_fold(const lora_bf16_t* x, int64_t x_row_stride, int32_t x_gather,
                          lora_bf16_t* base_out, int64_t out_row_stride,
                          const int32_t* expert_offsets, int32_t num_experts,
                          const int32_t* sorted_token_ids, int32_t te,
                          const int32_t* row_adapter, int32_t num_tokens,
                          int32_t row_offset, int32_t row_end,
                          const lora_bf16_t* const* a_table, const lora_bf16_t* const* b_table,
                          const float* scale_table, int32_t max_loras,
                          int32_t max_rank, int32_t k_in, int32_t n_out,
                          lora_bf16_t* xa, int32_t xa_rows, uint32_t flags, void* stream);

/*
 * lora_moe_gather_bgmv — the decode-path MoE fold over flat, unsorted
 * (token, slot) rows.
 *
 * Defines: "Module moe_lora_grouped" (atlas rustdoc), `moe_lora_gather_bgmv`
 * entry (the unsorted, slot-major analogue of `moe_lora_grouped_down`).
 *
 * For every row r in [0, n_rows):
 *   e = indices[r] (skipped if outside [0, num_experts));
 *   t = r / top_k (skipped if t >= num_tokens);
 *   a = row_adapter ? row_adapter[t] : 0 (skipped if outside [0, max_loras));
 *   entry a * num_experts + e of the adapter-major tables; skipped if its A or B
 *   pointer is NULL; otherwise the fold of lora_bgmv is applied to
 *   x[r*x_row_stride ..] and base_out[r*out_row_stride ..].
 *
 *   indices      [n_rows] int32 expert per row (row = token * top_k + slot)
 *   row_adapter  [num_tokens] int32 (< 0 = no delta), or NULL: adapter 0
 *   a_table, b_table, scale_table  [max_loras * num_experts], index a*num_experts + e
 *                (max_loras * num_experts <= LORA_MAX_LORAS)
 *   xa           optional [n_rows, max_rank] BF16 shrink output at row r (routed rows)
 *   a_tmaps      optional [max_loras * num_experts] A tensor maps, as for lora_bgmv
 *   flags        0 or LORA_INPUTS_READY, as for lora_bgmv
 * Rows of one table entry share a work unit; the launch grid depends only on
 * n_rows and the table count (capture-safe). Errors, alignment and ownership as
 * for lora_bgmv.
 */
int lora_moe_gather_bgmv(const lora_bf16_t* x, int64_t x_row_stride,
                         lora_bf16_t* base_out, int64_t out_row_stride,
                         const int32_t* indices, int32_t n_rows, int32_t top_k,
                         const int32_t* row_adapter, int32_t num_tokens, int32_t num_experts,
                         const lora_bf16_t* const* a_table, const lora_bf16_t* const* b_table,
                         const float* scale_table, int32_t max_loras,
                         int32_t max_rank, int32_t k_in, int32_t n_out,
                         lora_bf16_t* xa, const void* a_tmaps, uint32_t flags, void* stream);

/*
 * lora_delta — one adapter pair folded into every row: the pages' apply_lora_delta
 * ("lora_delta.rs", apply_lora_delta; "Module lora_delta", LoraPair), for m rows
 *   xa[i, :]  = bf16( x[i, :] @ a^T )                          fp32 accumulate
 *   out[i, :] = bf16( fma(scale, bf16( xa[i, :] @ b^T ), out[i, :]) ),  i < m.
 * Pages' m == 1 GEMV, small-m per-row and large-m tensor-core GEMM paths are one
 * call here, with the same rounding points as lora_bgmv:
 *   - m >= LORA_DELTA_DENSE_MIN_ROWS and max_rank in {16, 32, 64, 128}: one
 *     launch of the tcgen05 tensor-core kernel (tiles of 128 rows, a cluster of
 *     CTAs splits k_in and n_out; TMA tensor maps are encoded on the host per call);
 *   - otherwise the routed engine of lora_bgmv with every row on one slot (one
 *     launch per LORA_MAX_ROWS rows).
 * The fp32 summation order depends on (k_in, max_rank) and, on the tensor-core
 * path, on the cluster size, which follows the number of 128-row tiles: unlike
 * lora_bgmv, results may differ in the last bit between calls of different m
 * (each within the oracle's tolerance).
 *   x         [m, x_row_stride] BF16 rows (k_in used), 16-byte aligned
 *   base_out  [m, out_row_stride] BF16, columns [0, n_out) folded in place; other
 *             bytes are not touched
 *   a         [max_rank, k_in] row-major BF16 (rank-padded with zero rows)
 *   b         [n_out, max_rank] row-major BF16 (rank-padded with zero columns)
 *   scale     f32 (alpha/r, or alpha/sqrt(r) for rsLoRA)
 *   xa        optional [m, max_rank] BF16 output of the shrink; NULL skips it
 * Shapes, strides and alignment as for lora_bgmv (a and b 16-byte aligned, too);
 * m == 0 is a no-op. No allocation, no synchronization: capture-safe.
 */
int lora_delta(const lora_bf16_t* x, int64_t x_row_stride, lora_bf16_t* base_out, int64_t out_row_stride,
               int32_t m, const lora_bf16_t* a, const lora_bf16_t* b, float scale, int32_t max_rank,
               int32_t k_in, int32_t n_out, lora_bf16_t* xa, void* stream);

/*
 * lora_delta_geometry — the launch lora_delta would make for m rows on a device
 * with sm_count SMs (0: the current device). Writes [dense (1: tensor-core
 * kernel, 0: routed engine), cluster, ring_stages, stage_bytes, smem_bytes, ctas
 * (of one launch)] to out[0..5]. No counterpart in the pages (tests, benchmarks).
 */
int lora_delta_geometry(int32_t m, int32_t max_rank, int32_t k_in, int32_t n_out, int32_t sm_count,
                        int64_t out[6]);

/*
 * lora_encode_a_tmaps — host helper run once when adapters are loaded: writes,
 * for each of `count` A matrices ([max_rank, k_in] row-major BF16 at the device
 * address a_ptrs[i]; 0 = none), the 128-byte TMA tensor map the folds use to
 * load 64-column boxes of all its rank rows (128-byte swizzle). maps_out is
 * HOST memory of count * 128 bytes, 64-byte aligned; entries of 0 pointers are
 * zeroed. Copy it to device memory and pass it as a_tmaps. Needs the CUDA driver
 * (no GPU work is done); returns LORA_ERR_CUDA without one.
 * No counterpart in the pages: it prepares the TMA copies of this library.
 */
int lora_encode_a_tmaps(const uint64_t* a_ptrs, int32_t count, int32_t max_rank, int32_t k_in,
                        void* maps_out);

/*
 * lora_selftest_wait_timeout — diagnostic: launches one CTA whose thread waits on
 * an mbarrier that nothing arrives at, through the same bounded wait the folds
 * use, with a limit of limit_cycles SM clocks (in [1, 2^32]); giving up sets
 * LORA_DEV_TIMEOUT in the device status word, as a fold that timed out would.
 * The kernel then returns normally: the context stays usable. No counterpart in
 * the pages (it tests the failure path of this library without a GPU fault).
 */
int lora_selftest_wait_timeout(int64_t limit_cycles, void* stream);

/* Text of the last error returned on this host thread ("" if none). */
const char* lora_last_error(void);

/*
 * Device status word: OR of LORA_DEV_* bits set by kernels on the current
 * device since the last clear. Synchronizes `stream` (a test/diagnostic call,
 * not for the hot path). clear != 0 resets the word after reading.
 */
int lora_read_device_status(void* stream, uint32_t* status_out, int clear);

/*
 * Launch geometry that lora_bgmv / lora_moe_grouped_fold / lora_moe_gather_bgmv
 * would use (for tests and benchmarks). moe == 0: bgmv with `rows` = n; moe == 1:
 * MoE grouped fold with `rows` = row_end - row_offset and max_loras = the number
 * of adapters the grid covers (max_loras with a row_adapter, 1 without); moe ==
 * 2: decode gather fold with `rows` = n_rows and max_loras = the table count
 * (adapters x experts). Add 16 to `moe` for the geometry of a call given
 * a_tmaps. Writes [cluster,
 * rows_per_tile, k_slice, j_slice, k_chunk, j_chunk, ring_stages, clusters,
 * smem_bytes, a_tiled (1 when A is loaded through the tensor maps), tc (1 when the shrink
 * runs on the tcgen05 tensor cores), direct (1: unit s is tile 0 of slot s; 0: units are
 * numbered slot by slot over the slots with rows; for the MoE grouped fold: its CTA
 * shape, 0 = one CTA of 12 + 4 warps per SM, 1 = two CTAs of 8 + 2 warps per SM,
 * taken when k_in > n_out)] to out[0..11]. The unit numbering and the MoE grid also
 * depend on the current device's SM count (152 without a device).
 */
int lora_launch_geometry(int moe, int32_t rows, int32_t max_loras, int32_t max_rank,
                         int32_t k_in, int32_t n_out, int64_t out[12]);

/* ---- pure host helpers (no GPU) ------------------------------------------ */

/*
 * lora_grouped_down_wc — m-tile count of one window: max(1, ceil((row_end -
 * row_offset) / LORA_MOE_M_TILE)), the method's tile grid of a window (the
 * fold itself launches the persistent grid described at lora_moe_grouped_fold).
 * Defines: "Module moe_lora_grouped" rustdoc, `grouped_down_wc` entry.
 * Returns -1 if row_end < row_offset.
 */
int32_t lora_grouped_down_wc(int32_t row_offset, int32_t row_end);

/*
 * lora_gather_row_token — the token owning flat (token, slot) row `row` of the
 * decode gather fold: row / top_k (the rule lora_moe_gather_bgmv applies).
 * Returns -1 if row < 0 or top_k < 1.
 * Defines: "Module moe_lora_grouped" rustdoc, `gather_row_token` entry.
 */
int32_t lora_gather_row_token(int32_t row, int32_t top_k);

/*
 * lora_gather_bgmv_grids — the pages' exact launch grids of their decode gather
 * fold: shrink = [ceil(max_rank / 4), n_slots, 1], expand = [ceil(n_out / 4),
 * n_slots, 1], each with a (256, 1, 1) block (one 64-lane group per output, four
 * outputs per block). Reading: the shrink's outputs are the max_rank xa columns.
 * This library's own kernel uses lora_launch_geometry's grid instead; the helper
 * states the pages' arithmetic. Writes shrink[0..2] and expand[0..2]; returns 0,
 * or -1 if max_rank or n_out < 1, n_slots < 0, or a pointer is NULL.
 * Defines: "Module moe_lora_grouped" rustdoc, `gather_bgmv_grids` entry.
 */
int lora_gather_bgmv_grids(int32_t max_rank, int32_t n_out, int32_t n_slots,
                           int32_t shrink[3], int32_t expand[3]);

/*
 * lora_grouped_down_windows — contiguous [start, end) windows of `cap` rows
 * covering 0..total_rows (the last may be shorter). Writes up to max_windows
 * pairs into starts/ends (host arrays) and returns the number of windows, or
 * -1 if cap < 1 or total_rows < 0, or -2 if max_windows is too small.
 * total_rows == 0 gives 0 windows.
 * Defines: "Module moe_lora_grouped" rustdoc, `grouped_down_windows` entry.
 */
int32_t lora_grouped_down_windows(int32_t total_rows, int32_t cap,
                                  int32_t* starts, int32_t* ends, int32_t max_windows);

/*
 * lora_pack_expert_tables — dense per-expert tables from (expert_id, a, b,
 * scale) entries: a_table[e], b_table[e], scale_table[e] for e < n_experts =
 * max expert_id + 1, with 0 / 0 / 0.0f at experts without an entry; a later
 * entry for the same expert replaces an earlier one. All arrays are host
 * memory; table arrays hold table_len entries. Writes n_experts to
 * *n_experts_out and returns 0; returns 1 (nothing written, *n_experts_out = 0)
 * when n_entries == 0; -1 on a negative expert id or NULL argument; -2 when
 * table_len < n_experts.
 * Defines: "Module moe_lora_grouped" rustdoc, `pack_expert_tables` and
 * `ExpertTables` entries.
 */
int lora_pack_expert_tables(const int32_t* expert_ids, const uint64_t* a_addrs,
                            const uint64_t* b_addrs, const float* scales, int32_t n_entries,
                            uint64_t* a_table, uint64_t* b_table, float* scale_table,
                            int32_t table_len, int32_t* n_experts_out);

#ifdef __cplusplus
}
#endif

#endif /* GATHER_LORA_H */
