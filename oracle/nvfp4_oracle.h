/*
 * nvfp4_oracle.h -- declarations of the CPU oracle (test infrastructure only).
 *
 * The oracle is the slow, obviously correct reference for the NVFP4 paged KV
 * cache; only tests, the smoke check and the benchmark's CPU-baseline leg use
 * it.  It has no GPU dependency and shares nothing with the CUDA library.
 * All pointers are host pointers.  Functions that walk page tables return 0,
 * or 1 when an out-of-range slot, page id or length was skipped or clamped.
 */
#ifndef NVFP4_ORACLE_H
#define NVFP4_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4_ORACLE_BLOCK 16 /* values sharing one E4M3 block scale */

typedef struct {
  uint8_t* k_data;  /* [num_pages][num_kv_heads][page_size][head_dim/2]  */
  uint8_t* v_data;
  uint8_t* k_scale; /* [num_pages][num_kv_heads][page_size][head_dim/16] */
  uint8_t* v_scale;
  int64_t num_pages;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  float k_global_scale;
  float v_global_scale;
} nvfp4_oracle_cache;

double nvfp4_oracle_e2m1_value(uint8_t code);
double nvfp4_oracle_e4m3_value(uint8_t code);
uint8_t nvfp4_oracle_e2m1_encode(float y);
uint8_t nvfp4_oracle_e4m3_encode(float z);
float nvfp4_oracle_bf16_to_float(uint16_t bits);

void nvfp4_oracle_quantize_block(const float x[NVFP4_ORACLE_BLOCK], float g,
                                 uint8_t packed[NVFP4_ORACLE_BLOCK / 2], uint8_t* scale);
double nvfp4_oracle_dequant_value(uint8_t code, uint8_t scale, float g);
void nvfp4_oracle_demo_fake_quant(const double* x, int64_t n, int64_t block, double* out);

int64_t nvfp4_oracle_row_bytes(int head_dim);
int64_t nvfp4_oracle_row_scale_bytes(int head_dim);

int nvfp4_oracle_quantize_append(const nvfp4_oracle_cache* c, const uint16_t* k_bf16,
                                 const uint16_t* v_bf16, const int64_t* slot_mapping,
                                 int64_t num_tokens);
int nvfp4_oracle_decode_attention(const nvfp4_oracle_cache* c, const uint16_t* q_bf16,
                                  const int32_t* page_table, int32_t max_pages,
                                  const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                  double softmax_scale, double* out);
int nvfp4_oracle_decode_attention_heads(const nvfp4_oracle_cache* c, const uint16_t* q_bf16,
                                        const int32_t* page_table, int32_t max_pages,
                                        const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                        double softmax_scale, int32_t head_begin, int32_t head_end,
                                        double* out);
/* Largest |x| over n bf16 values (0 for n == 0), as a float (exact: a bf16
 * value).  The calibration statistic of a tensor's global scale. */
float nvfp4_oracle_tensor_amax(const uint16_t* x_bf16, int64_t n);
/* Calibrated global scale g = amax / (6 * 448), one binary32 division, so the
 * tensor's largest value maps onto E2M1's 6 times E4M3's 448; 1 when amax is 0. */
float nvfp4_oracle_calibrated_global_scale(float amax);

int nvfp4_oracle_dequant_to_fp8_workspace(const nvfp4_oracle_cache* c, const int32_t* page_table,
                                          int32_t max_pages, const int32_t* prefix_lens,
                                          const int64_t* cu_prefix, int32_t batch,
                                          float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                                          uint8_t* ws_v);

/* Format variants (MXFP4 blocks of 32 with an E8M0 scale; stochastic rounding
 * of the E2M1 codes from input random bytes; the orthonormal Walsh-Hadamard
 * rotation in binary32 butterflies). */
double nvfp4_oracle_e8m0_value(uint8_t code);
void nvfp4_oracle_mxfp4_quantize_block(const float x[32], uint8_t packed[16], uint8_t* scale);
double nvfp4_oracle_mxfp4_dequant_value(uint8_t code, uint8_t scale);
uint8_t nvfp4_oracle_e2m1_encode_sr(float y, uint8_t r);
void nvfp4_oracle_quantize_block_sr(const float x[NVFP4_ORACLE_BLOCK], float g, const uint8_t r[NVFP4_ORACLE_BLOCK],
                                    uint8_t packed[NVFP4_ORACLE_BLOCK / 2], uint8_t* scale);
int nvfp4_oracle_hadamard(const float* x, int n, float* y);

/* Decode attention over a variant's cache: format 0 NVFP4, 1 NVFP4 of
 * Hadamard-rotated rows (rotated back before the attention), 2 MXFP4 (scale
 * pools of head_dim/32 E8M0 bytes per row). */
int nvfp4_oracle_decode_attention_format(const nvfp4_oracle_cache* c, int format, const uint16_t* q_bf16,
                                         const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                                         int32_t batch, int32_t num_q_heads, double softmax_scale, double* out);

/* Extend over the FP8 workspace.  The chunk's K/V rows enter the workspace
 * from bf16 (w = E4M3(fp32(x) / s_ws), signed); ws_rows[t] < 0 skips token t.
 * Extend attention evaluates, in binary64, the output rows named by pairs
 * (global query token i, query head h): sequence b of token i attends from
 * chunk position t = i - cu_q[b] over keys 0 .. prefix_lens[b] + t, key j
 * being workspace row cu_prefix[b] + j, dequantised as E4M3val(w) * s_ws. */
int nvfp4_oracle_bf16_to_fp8_workspace(const uint16_t* k_bf16, const uint16_t* v_bf16,
                                       const int64_t* ws_rows, int64_t num_tokens,
                                       int32_t num_kv_heads, int32_t head_dim, int64_t total_rows,
                                       float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                                       uint8_t* ws_v);
int nvfp4_oracle_extend_attention_rows(const uint8_t* ws_k, const uint8_t* ws_v, int64_t total_rows,
                                       int32_t num_kv_heads, int32_t head_dim, float k_ws_scale,
                                       float v_ws_scale, const uint16_t* q_bf16, int32_t num_q_heads,
                                       const int64_t* cu_q, const int64_t* cu_prefix,
                                       const int32_t* prefix_lens, int32_t batch,
                                       double softmax_scale, const int64_t* pairs, int64_t num_pairs,
                                       double* out);

#ifdef __cplusplus
}
#endif

#endif
