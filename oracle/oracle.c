/*
 * CPU oracle for the routed multi-LoRA fold. TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and the CPU-baseline leg of bench.py may
 * load this library. The product path (gather_lora_gb300, libgather_lora.so)
 * never calls it and shares no code, header or helper with it.
 *
 * What it computes is the plain per-row definition of the operations, with the
 * rounding points that the pages fix and nothing else:
 *
 *   Function apply_lora_bgmv page (spark_model::layers::ops::lora_delta rustdoc),
 *   summary and "BYTE-IDENTICAL" paragraph:
 *     out[i,:] += scale_s * (x[i,:] @ A_s^T) @ B_s^T, s = seq_slot[i]; s < 0 or a
 *     NULL table entry means no delta.  The shrink emits BF16 xa; the expand
 *     rounds the delta to BF16; the per-slot scale is applied in fp32 after that
 *     rounding; both stages contract at max_rank (pad rows/cols are zero).
 *   lora_delta.rs page (metrale source listing), LoraPair doc comment:
 *     a = [max_rank, k_in] row-major BF16, b = [n_out, max_rank] row-major BF16.
 *   Module moe_lora_grouped page (atlas rustdoc), moe_lora_grouped_down entry:
 *     expert-sorted rows of one window [row_offset, row_end), expert e from the
 *     device expert_offsets prefix sum, token from sorted_token_ids, adapter gate
 *     from moe_row_adapter[token] (< 0 = base, NULL table = every row adapter 0),
 *     xa indexed at the LOCAL row r - row_offset; same fold math as the bgmv.
 *     Down (x_gather == 0): x is the sorted [te, k_in] activation at row r;
 *     gate/up (x_gather == 1): x is token-major and sorted row r reads row
 *     sorted_token_ids[r] of it.
 *   Same page, moe_lora_gather_bgmv entry: the decode-path twin over flat,
 *     unsorted (token, slot) rows; expert from indices[row], adapter gate from
 *     row_adapter[row / top_k].
 *   lora_delta.rs page, apply_lora_delta: one LoraPair over all m rows
 *     (base_out[m, n_out] += scale * (x @ a^T) @ b^T), every row adapted; the
 *     same per-row fold as the bgmv.
 *
 * Readings where the pages are silent:
 *   - fp32 -> BF16 is round-to-nearest-even.
 *   - fp32 accumulation is a plain sequential sum in index order (k, then c).
 *     Products of two BF16 values are exact in fp32, so fused or unfused
 *     multiply-add give the same sum; the file is built with -ffp-contract=off.
 *   - the fold is ONE fused multiply-add in fp32 (fmaf), then BF16 RNE.
 *   - a row is skipped when its slot is < 0 or >= max_loras, or when the A OR
 *     the B table entry is NULL. MoE: also when the row is outside
 *     [off[0], off[E]), when its token is outside [0, num_tokens), or when its
 *     adapter is < 0 or >= max_loras.
 *   - MoE tables are [max_loras * num_experts], adapter-major (index a*E + e);
 *     with row_adapter == NULL every row uses adapter 0.
 *
 * Variants: mode 0 = fp32 accumulation (the pages' arithmetic); mode 1 = the
 * same rounding points with fp64 sums (a brute-force twin used to bound the
 * fp32 summation error in the pins).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#include "oracle.h"

/* ---- BF16 <-> fp32 --------------------------------------------------------- */

float ora_f32_of_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest-even of an fp32 to BF16 (keep the top 16 bits after adding
 * half an ulp, with ties going to the even neighbour). */
uint16_t ora_bf16_of_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)          /* NaN stays a quiet NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xffffu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;                               /* carries into the exponent */
    return (uint16_t)upper;
}

/* Round-to-nearest-even of an fp64 straight to BF16 (no intermediate fp32
 * rounding, which could round twice). Works on the exact binary value: the
 * result keeps 8 significant bits, or fewer in BF16's subnormal range. */
uint16_t ora_bf16_of_f64(double v)
{
    if (v != v) return 0x7fc0u;
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);              /* a = m * 2^e, m in [0.5, 1) */
    int q_exp = e - 8;               /* 8 significant bits: ulp = 2^(e-8) */
    if (q_exp < -133) q_exp = -133;  /* BF16 subnormal ulp is 2^-133 */
    double scaled = ldexp(a, -q_exp);             /* exact (power-of-two scaling) */
    double fl = floor(scaled);
    double frac = scaled - fl;                    /* exact */
    double q = fl;
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0)) q = fl + 1.0;
    double r = ldexp(q, q_exp);                   /* exact, representable in fp32 */
    if (r > 3.3895313892515355e38) return (uint16_t)(sign | 0x7f80u); /* > max BF16 */
    float rf = (float)r;                          /* exact */
    uint32_t u;
    memcpy(&u, &rf, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* ---- one routed row: shrink, expand, fold --------------------------------- */

static void fold_one_row(const uint16_t* xrow, uint16_t* orow,
                         const uint16_t* A, const uint16_t* B, float scale,
                         int32_t max_rank, int32_t k_in, int32_t n_out,
                         uint16_t* xa_row, uint16_t* d_row, int32_t mode)
{
    /* shrink: xa[c] = bf16( sum_k x[k] * A[c][k] ), A row-major [max_rank, k_in] */
    for (int32_t c = 0; c < max_rank; ++c) {
        const uint16_t* arow = A + (int64_t)c * k_in;
        if (mode == 0) {
            float acc = 0.0f;
            for (int32_t k = 0; k < k_in; ++k)
                acc = acc + ora_f32_of_bf16(xrow[k]) * ora_f32_of_bf16(arow[k]);
            xa_row[c] = ora_bf16_of_f32(acc);
        } else {
            double acc = 0.0;
            for (int32_t k = 0; k < k_in; ++k)
                acc = acc + (double)ora_f32_of_bf16(xrow[k]) * (double)ora_f32_of_bf16(arow[k]);
            xa_row[c] = ora_bf16_of_f64(acc);
        }
    }
    /* expand + fold: d[j] = bf16( sum_c xa[c] * B[j][c] ), B row-major [n_out, max_rank];
     * out[j] = bf16( fmaf(scale, d[j], out[j]) ) */
    for (int32_t j = 0; j < n_out; ++j) {
        const uint16_t* brow = B + (int64_t)j * max_rank;
        uint16_t d;
        if (mode == 0) {
            float acc = 0.0f;
            for (int32_t c = 0; c < max_rank; ++c)
                acc = acc + ora_f32_of_bf16(xa_row[c]) * ora_f32_of_bf16(brow[c]);
            d = ora_bf16_of_f32(acc);
        } else {
            double acc = 0.0;
            for (int32_t c = 0; c < max_rank; ++c)
                acc = acc + (double)ora_f32_of_bf16(xa_row[c]) * (double)ora_f32_of_bf16(brow[c]);
            d = ora_bf16_of_f64(acc);
        }
        if (d_row) d_row[j] = d;
        float folded = fmaf(scale, ora_f32_of_bf16(d), ora_f32_of_bf16(orow[j]));
        orow[j] = ora_bf16_of_f32(folded);
    }
}

/* ---- routed bgmv ----------------------------------------------------------- */

int ora_lora_bgmv(const uint16_t* x, int64_t x_row_stride,
                  uint16_t* base_out, int64_t out_row_stride,
                  const int32_t* seq_slot, int32_t n,
                  const uint16_t* const* a_table, const uint16_t* const* b_table,
                  const float* scale_table, int32_t max_loras,
                  int32_t max_rank, int32_t k_in, int32_t n_out,
                  uint16_t* xa, uint16_t* d_out, int32_t mode)
{
    if (n < 0 || max_rank <= 0 || k_in <= 0 || n_out <= 0 || max_loras < 0) return -1;
    if (x_row_stride < k_in || out_row_stride < n_out) return -1;
    uint16_t xa_tmp[4096];
    if (max_rank > 4096) return -1;
    for (int32_t i = 0; i < n; ++i) {
        int32_t s = seq_slot[i];
        if (s < 0 || s >= max_loras) continue;
        const uint16_t* A = a_table[s];
        const uint16_t* B = b_table[s];
        if (A == NULL || B == NULL) continue;
        uint16_t* xa_row = xa ? xa + (int64_t)i * max_rank : xa_tmp;
        uint16_t* d_row = d_out ? d_out + (int64_t)i * n_out : NULL;
        fold_one_row(x + (int64_t)i * x_row_stride, base_out + (int64_t)i * out_row_stride,
                     A, B, scale_table[s], max_rank, k_in, n_out, xa_row, d_row, mode);
    }
    return 0;
}

/* ---- one adapter pair over every row ---------------------------------------
 * "lora_delta.rs", apply_lora_delta: base_out[m, n_out] += scale * (x @ a^T) @ b^T
 * for one LoraPair, with the same rounding points as the routed fold (xa and the
 * delta rounded to BF16, then one fp32 fma and a BF16 rounding). Every row is
 * adapted; there is no routing. */
int ora_lora_delta(const uint16_t* x, int64_t x_row_stride,
                   uint16_t* base_out, int64_t out_row_stride, int32_t m,
                   const uint16_t* a, const uint16_t* b, float scale,
                   int32_t max_rank, int32_t k_in, int32_t n_out,
                   uint16_t* xa, uint16_t* d_out, int32_t mode)
{
    if (m < 0 || max_rank <= 0 || k_in <= 0 || n_out <= 0) return -1;
    if (x_row_stride < k_in || out_row_stride < n_out || a == NULL || b == NULL) return -1;
    uint16_t xa_tmp[4096];
    if (max_rank > 4096) return -1;
    for (int32_t row = 0; row < m; ++row) {
        uint16_t* xa_row = xa ? xa + (int64_t)row * max_rank : xa_tmp;
        uint16_t* d_row = d_out ? d_out + (int64_t)row * n_out : NULL;
        const uint16_t* x_row = x + (int64_t)row * x_row_stride;
        uint16_t* out_row = base_out + (int64_t)row * out_row_stride;
        fold_one_row(x_row, out_row, a, b, scale, max_rank, k_in, n_out, xa_row, d_row, mode);
    }
    return 0;
}

/* ---- MoE grouped fold over one window of expert-sorted rows --------------- */

int ora_lora_moe_grouped_fold(const uint16_t* x, int64_t x_row_stride, int32_t x_gather,
                              uint16_t* base_out, int64_t out_row_stride,
                              const int32_t* expert_offsets, int32_t num_experts,
                              const int32_t* sorted_token_ids, int32_t te,
                              const int32_t* row_adapter, int32_t num_tokens,
                              int32_t row_offset, int32_t row_end,
                              const uint16_t* const* a_table, const uint16_t* const* b_table,
                              const float* scale_table, int32_t max_loras,
                              int32_t max_rank, int32_t k_in, int32_t n_out,
                              uint16_t* xa, uint16_t* d_out, int32_t mode)
{
    if (num_experts <= 0 || max_rank <= 0 || k_in <= 0 || n_out <= 0 || max_loras < 0) return -1;
    if (row_offset < 0 || row_end < row_offset || row_end > te) return -1;
    if (x_row_stride < k_in || out_row_stride < n_out) return -1;
    uint16_t xa_tmp[4096];
    if (max_rank > 4096) return -1;
    const int32_t lo = expert_offsets[0], hi = expert_offsets[num_experts];
    for (int32_t r = row_offset; r < row_end; ++r) {
        if (r < lo || r >= hi) continue;
        int32_t e = -1;
        for (int32_t k = 0; k < num_experts; ++k) {         /* the expert whose span holds r */
            if (expert_offsets[k] <= r && r < expert_offsets[k + 1]) { e = k; break; }
        }
        if (e < 0) continue;
        /* the row's token: needed for the adapter gate and for the gate/up
           input (x_gather: x is token-major, row t of it feeds sorted row r) */
        int32_t t = -1;
        if (row_adapter || x_gather) {
            t = sorted_token_ids[r];
            if (t < 0 || t >= num_tokens) continue;
        }
        int32_t a = row_adapter ? row_adapter[t] : 0;
        if (a < 0 || a >= max_loras) continue;
        int64_t ti = (int64_t)a * num_experts + e;
        const uint16_t* A = a_table[ti];
        const uint16_t* B = b_table[ti];
        if (A == NULL || B == NULL) continue;
        int64_t local = r - row_offset;
        uint16_t* xa_row = xa ? xa + local * max_rank : xa_tmp;
        uint16_t* d_row = d_out ? d_out + (int64_t)r * n_out : NULL;
        const int64_t xr = x_gather ? t : r;
        fold_one_row(x + xr * x_row_stride, base_out + (int64_t)r * out_row_stride,
                     A, B, scale_table[ti], max_rank, k_in, n_out, xa_row, d_row, mode);
    }
    return 0;
}

/*
 * Decode-path MoE fold over flat, unsorted (token, slot) rows ("Module
 * moe_lora_grouped", moe_lora_gather_bgmv): row r takes its expert from
 * indices[r] and its adapter from row_adapter[r / top_k] (< 0: no delta;
 * row_adapter == NULL: adapter 0). The table entry is a * num_experts + e as
 * for the grouped fold; rows with an expert outside [0, num_experts), a token
 * outside [0, num_tokens), an adapter outside [0, max_loras) or a NULL entry
 * are skipped. x and base_out are [n_rows, .] at row r; xa [n_rows, max_rank]
 * and d_out [n_rows, n_out] at row r.
 */
int ora_lora_moe_gather_bgmv(const uint16_t* x, int64_t x_row_stride,
                             uint16_t* base_out, int64_t out_row_stride,
                             const int32_t* indices, int32_t n_rows, int32_t top_k,
                             const int32_t* row_adapter, int32_t num_tokens, int32_t num_experts,
                             const uint16_t* const* a_table, const uint16_t* const* b_table,
                             const float* scale_table, int32_t max_loras,
                             int32_t max_rank, int32_t k_in, int32_t n_out,
                             uint16_t* xa, uint16_t* d_out, int32_t mode)
{
    if (num_experts <= 0 || top_k <= 0 || max_rank <= 0 || k_in <= 0 || n_out <= 0 || max_loras < 0) return -1;
    if (n_rows < 0 || x_row_stride < k_in || out_row_stride < n_out) return -1;
    uint16_t xa_tmp[4096];
    if (max_rank > 4096) return -1;
    for (int32_t r = 0; r < n_rows; ++r) {
        const int32_t e = indices[r];
        if (e < 0 || e >= num_experts) continue;
        const int32_t t = r / top_k;
        if (t >= num_tokens) continue;
        const int32_t a = row_adapter ? row_adapter[t] : 0;
        if (a < 0 || a >= max_loras) continue;
        const int64_t entry = (int64_t)a * num_experts + e;
        const uint16_t* A = a_table[entry];
        const uint16_t* B = b_table[entry];
        if (A == NULL || B == NULL) continue;
        uint16_t* xa_row = xa ? xa + (int64_t)r * max_rank : xa_tmp;
        uint16_t* d_row = d_out ? d_out + (int64_t)r * n_out : NULL;
        fold_one_row(x + (int64_t)r * x_row_stride, base_out + (int64_t)r * out_row_stride,
                     A, B, scale_table[entry], max_rank, k_in, n_out, xa_row, d_row, mode);
    }
    return 0;
}
