/*
 * Declarations of the CPU oracle (oracle.c). TEST INFRASTRUCTURE ONLY: the
 * product library never includes this header and shares nothing with it.
 *
 * All BF16 values are raw uint16 bit patterns. Pointers are host pointers.
 * a_table / b_table are host arrays of host pointers (NULL = no adapter).
 * xa (optional) receives the BF16 shrink output of every routed row:
 *   bgmv: [n, max_rank] at row i;  MoE: [row_end-row_offset, max_rank] at r-row_offset.
 * d_out (optional) receives the BF16-rounded delta of every routed row:
 *   bgmv: [n, n_out] at row i;     MoE: [te, n_out] at sorted row r.
 * mode 0 = fp32 sequential sums (the method), mode 1 = fp64 sums, same roundings.
 * Return 0, or -1 on an argument the oracle does not accept.
 */
#ifndef GATHER_LORA_ORACLE_H
#define GATHER_LORA_ORACLE_H
#include <stdint.h>

float ora_f32_of_bf16(uint16_t h);
uint16_t ora_bf16_of_f32(float f);
uint16_t ora_bf16_of_f64(double v);

int ora_lora_bgmv(const uint16_t* x, int64_t x_row_stride,
                  uint16_t* base_out, int64_t out_row_stride,
                  const int32_t* seq_slot, int32_t n,
                  const uint16_t* const* a_table, const uint16_t* const* b_table,
                  const float* scale_table, int32_t max_loras,
                  int32_t max_rank, int32_t k_in, int32_t n_out,
                  uint16_t* xa, uint16_t* d_out, int32_t mode);

/* One adapter pair (a [max_rank, k_in], b [n_out, max_rank], scale) over all m rows. */
int ora_lora_delta(const uint16_t* x, int64_t x_row_stride,
                   uint16_t* base_out, int64_t out_row_stride, int32_t m,
                   const uint16_t* a, const uint16_t* b, float scale,
                   int32_t max_rank, int32_t k_in, int32_t n_out,
                   uint16_t* xa, uint16_t* d_out, int32_t mode);

/* x_gather != 0: x is token-major [num_tokens, .] and sorted row r reads row
   sorted_token_ids[r] of it (gate/up); 0: x is [te, .] at row r (down). */
int ora_lora_moe_grouped_fold(const uint16_t* x, int64_t x_row_stride, int32_t x_gather,
                              uint16_t* base_out, int64_t out_row_stride,
                              const int32_t* expert_offsets, int32_t num_experts,
                              const int32_t* sorted_token_ids, int32_t te,
                              const int32_t* row_adapter, int32_t num_tokens,
                              int32_t row_offset, int32_t row_end,
                              const uint16_t* const* a_table, const uint16_t* const* b_table,
                              const float* scale_table, int32_t max_loras,
                              int32_t max_rank, int32_t k_in, int32_t n_out,
                              uint16_t* xa, uint16_t* d_out, int32_t mode);

int ora_lora_moe_gather_bgmv(const uint16_t* x, int64_t x_row_stride,
                             uint16_t* base_out, int64_t out_row_stride,
                             const int32_t* indices, int32_t n_rows, int32_t top_k,
                             const int32_t* row_adapter, int32_t num_tokens, int32_t num_experts,
                             const uint16_t* const* a_table, const uint16_t* const* b_table,
                             const float* scale_table, int32_t max_loras,
                             int32_t max_rank, int32_t k_in, int32_t n_out,
                             uint16_t* xa, uint16_t* d_out, int32_t mode);

#endif
