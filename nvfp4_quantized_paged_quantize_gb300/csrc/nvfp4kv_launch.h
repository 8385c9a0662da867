// nvfp4kv_launch.h -- internal launchers shared by the kernels' translation
// units and the C ABI layer (api.cu).  Arguments are already validated.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "nvfp4kv.h"

namespace nvfp4kv {

cudaError_t launch_quantize_append(const nvfp4kv_cache& c, const uint16_t* k, const uint16_t* v,
                                   const int64_t* slot_mapping, int64_t num_tokens,
                                   int32_t* device_status, int num_sms, cudaStream_t stream);

cudaError_t launch_dequant_fp8(const nvfp4kv_cache& c, const int32_t* page_table, int32_t max_pages,
                               const int32_t* prefix_lens, const int64_t* cu_prefix, int32_t batch,
                               int64_t total_rows, float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                               uint8_t* ws_v, int32_t* device_status, int num_sms, cudaStream_t stream);

// Quantize-append plus the FP8 workspace rows of the same tokens, one pass.
cudaError_t launch_quantize_append_fp8(const nvfp4kv_cache& c, const uint16_t* k, const uint16_t* v,
                                       const int64_t* slot_mapping, int64_t num_tokens, const int64_t* ws_rows,
                                       int64_t total_rows, float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                                       uint8_t* ws_v, int32_t* device_status, int num_sms, cudaStream_t stream);

// Quantize-append of a format variant (NVFP4KV_VARIANT_*).
cudaError_t launch_quantize_variant(int variant, const nvfp4kv_cache& c, const uint16_t* k, const uint16_t* v,
                                    const int64_t* slot_mapping, int64_t num_tokens, const uint8_t* rand_k,
                                    const uint8_t* rand_v, int32_t* device_status, cudaStream_t stream);

// The chunk's bf16 K/V rows -> FP8 workspace rows ws_rows[t] (< 0: skipped).
cudaError_t launch_chunk_to_ws(const uint16_t* k, const uint16_t* v, const int64_t* ws_rows, int64_t num_tokens,
                               int32_t num_kv_heads, int64_t total_rows, float k_ws_scale, float v_ws_scale,
                               uint8_t* ws_k, uint8_t* ws_v, int32_t* device_status, int num_sms,
                               cudaStream_t stream);

// Causal extend attention of the chunk's queries over the FP8 workspace
// (group = num_q_heads / num_kv_heads a power of two <= 128).
cudaError_t launch_extend_attention(const uint16_t* q, const int64_t* cu_q, int32_t max_q_len, const uint8_t* ws_k,
                                    const uint8_t* ws_v, const int64_t* cu_prefix, const int32_t* prefix_lens,
                                    int32_t batch, int64_t total_rows, int32_t num_q_heads, int32_t num_kv_heads,
                                    float k_ws_scale, float v_ws_scale, float softmax_scale, float* out,
                                    int32_t* device_status, cudaStream_t stream);

// Largest |x| of n bf16 values into the device float *amax (zeroed first
// unless accumulate, which folds into the value already there).
cudaError_t launch_tensor_amax(const uint16_t* x, int64_t n, float* amax, bool accumulate, int num_sms,
                               cudaStream_t stream);

// Split-K decode: how many CTAs the decode launches on a device with num_sms
// SMs, and the workspace layout that goes with it.
int decode_num_ctas(int num_sms);
size_t decode_workspace_bytes(int num_ctas, int32_t batch, int32_t num_kv_heads);

cudaError_t launch_decode(const nvfp4kv_cache& c, const uint16_t* q, float* out,
                          const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                          int32_t batch, int32_t num_q_heads, float softmax_scale, void* workspace,
                          int32_t* device_status, int num_sms, cudaStream_t stream,
                          bool after_kernel = false);

}  // namespace nvfp4kv
