// nvfp4kv_launch.h -- internal launchers shared by the kernels' translation
// units and the C ABI layer (api.cu).  Arguments are already validated.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "nvfp4kv.h"

namespace nvfp4kv {

// A set-up step that must run once on every device before a kernel is
// launched there (a function attribute such as the dynamic shared-memory
// limit belongs to the function as loaded on the current device).  run()
// calls set_up() with the device current the first time that device is seen
// and caches the success; concurrent first calls from several host threads
// serialise on the mutex.  Devices past kMaxDevices run the set-up every time.
class PerDeviceOnce {
 public:
  template <class F>
  cudaError_t run(F set_up) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return set_up();
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = set_up();
    if (e == cudaSuccess) done_[dev].store(true, std::memory_order_release);
    return e;
  }

 private:
  static constexpr int kMaxDevices = 64;
  std::atomic<bool> done_[kMaxDevices] = {};
  std::mutex mu_;
};

cudaError_t launch_quantize_append(const nvfp4kv_cache& c, const uint16_t* k, const uint16_t* v,
                                   const int64_t* slot_mapping, int64_t num_tokens,
                                   int32_t* device_status, int num_sms, cudaStream_t stream);

cudaError_t launch_dequant_fp8(const nvfp4kv_cache& c, const int32_t* page_table, int32_t max_pages,
                               const int32_t* prefix_lens, const int64_t* cu_prefix, int32_t batch,
                               int64_t total_rows, float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                               uint8_t* ws_v, int32_t* device_status, cudaStream_t stream);

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
// SMs, and the workspace it needs there (two split records per warp of the
// launch, whatever the batch).
int decode_num_ctas(int num_sms);
size_t decode_workspace_bytes(int num_sms, int32_t batch, int32_t num_kv_heads);
// An upper bound of decode_workspace_bytes over every KV-head count that
// divides num_q_heads.
size_t decode_workspace_bound(int num_sms, int32_t batch, int32_t num_q_heads);

// The decode's memory stream with no math (NVFP4KV_PROBE_* modes).
cudaError_t launch_stream_probe(const nvfp4kv_cache& c, const int32_t* page_table, int32_t max_pages,
                                const int32_t* seq_lens, int32_t batch, int mode, uint32_t* sink,
                                int32_t* device_status, int num_sms, cudaStream_t stream);

// The decode over a format variant's cache (NVFP4KV_VARIANT_*): SR pages are
// NVFP4; Hadamard pages hold NVFP4 of rotated rows; MXFP4 its own page-heads.
cudaError_t launch_decode_variant(int variant, const nvfp4kv_cache& c, const uint16_t* q, float* out,
                                  const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                                  int32_t batch, int32_t num_q_heads, float softmax_scale, void* workspace,
                                  int32_t* device_status, int num_sms, cudaStream_t stream);

cudaError_t launch_decode(const nvfp4kv_cache& c, const uint16_t* q, float* out,
                          const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                          int32_t batch, int32_t num_q_heads, float softmax_scale, void* workspace,
                          int32_t* device_status, int num_sms, cudaStream_t stream,
                          bool after_kernel = false);

}  // namespace nvfp4kv
