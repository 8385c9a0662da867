// api.cu -- the C ABI of libnvfp4kv.so (declared in include/nvfp4kv.h): host
// validation, size queries and kernel launches.  Nothing here allocates device
// memory or synchronises; every launch goes to the caller's stream.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "nvfp4kv.h"
#include "nvfp4kv_launch.h"

namespace {

constexpr int kHeadDim = 128;

constexpr int kPageSize = 16;
constexpr int kMaxDevices = 64;
std::atomic<int> g_num_sms[kMaxDevices];  // 0 = not queried yet

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool positive_finite(float x) { return std::isfinite(x) && x > 0.0f; }

// SM count of the current device (cached; the query is a host call).
int current_num_sms(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4KV_ERR_CUDA;
  if (dev >= 0 && dev < kMaxDevices) {
    int cached = g_num_sms[dev].load(std::memory_order_relaxed);
    if (cached > 0) {
      *num_sms = cached;
      return NVFP4KV_OK;
    }
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return NVFP4KV_ERR_CUDA;
  if (dev >= 0 && dev < kMaxDevices) g_num_sms[dev].store(n, std::memory_order_relaxed);
  *num_sms = n;
  return NVFP4KV_OK;
}

// Shape and pointer checks common to every call that reads or writes the pool.
int check_cache(const nvfp4kv_cache* c) {
  if (c == nullptr) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (c->head_dim != kHeadDim || c->page_size != kPageSize) return NVFP4KV_ERR_UNSUPPORTED;
  if (c->num_pages <= 0 || c->num_kv_heads <= 0) return NVFP4KV_ERR_INVALID_ARGUMENT;
  // row indices (page * heads + head) * page_size stay below 2^31
  if (c->num_pages * (int64_t)c->num_kv_heads * kPageSize >= (int64_t(1) << 31))
    return NVFP4KV_ERR_UNSUPPORTED;
  if (!c->pages || !aligned(c->pages, 16)) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (!positive_finite(c->k_global_scale) || !positive_finite(c->v_global_scale))
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  return NVFP4KV_OK;
}

// the last CUDA error a call of this thread returned NVFP4KV_ERR_CUDA for
thread_local cudaError_t last_cuda_error = cudaSuccess;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return NVFP4KV_OK;
  last_cuda_error = e;
  return NVFP4KV_ERR_CUDA;
}

}  // namespace

extern "C" {

int nvfp4kv_cache_bytes(int64_t num_pages, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                        size_t* pool_bytes) {
  if (pool_bytes == nullptr) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (num_pages <= 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || head_dim % 16 != 0)
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  // rows of K (and of V), each head_dim / 2 data bytes and head_dim / 16 scale bytes
  const int64_t row_bytes = 2 * (int64_t)(head_dim / 2 + head_dim / 16);
  if (num_pages > INT64_MAX / num_kv_heads / page_size / row_bytes) return NVFP4KV_ERR_UNSUPPORTED;
  *pool_bytes = (size_t)(num_pages * num_kv_heads * (int64_t)page_size * row_bytes);
  return NVFP4KV_OK;
}

// Host checks of quantize-append arguments (nothing is enqueued).
static int check_append(const nvfp4kv_cache* cache, const void* k, const void* v, const int64_t* slot_mapping,
                        int64_t num_tokens, int32_t* device_status) {
  int st = check_cache(cache);
  if (st != NVFP4KV_OK) return st;
  if (num_tokens < 0) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return NVFP4KV_OK;
  if (num_tokens * (int64_t)cache->num_kv_heads >= (int64_t(1) << 31)) return NVFP4KV_ERR_UNSUPPORTED;
  if (!k || !v || !slot_mapping) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8)) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (device_status && !aligned(device_status, 4)) return NVFP4KV_ERR_INVALID_ARGUMENT;
  return NVFP4KV_OK;
}

int nvfp4kv_quantize_append(const nvfp4kv_cache* cache, const void* k, const void* v,
                            const int64_t* slot_mapping, int64_t num_tokens, int32_t* device_status,
                            nvfp4kv_stream_t stream) {
  int st = check_append(cache, k, v, slot_mapping, num_tokens, device_status);
  if (st != NVFP4KV_OK || num_tokens == 0) return st;
  int nsm = 0;
  if ((st = current_num_sms(&nsm)) != NVFP4KV_OK) return st;
  return cuda_status(nvfp4kv::launch_quantize_append(
      *cache, static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), slot_mapping, num_tokens,
      device_status, nsm, reinterpret_cast<cudaStream_t>(stream)));
}

int nvfp4kv_quantize_append_fp8(const nvfp4kv_cache* cache, const void* k, const void* v,
                                const int64_t* slot_mapping, int64_t num_tokens, const int64_t* ws_rows,
                                int64_t total_rows, float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                                uint8_t* ws_v, int32_t* device_status, nvfp4kv_stream_t stream) {
  int st = check_append(cache, k, v, slot_mapping, num_tokens, device_status);
  if (st != NVFP4KV_OK) return st;
  if (total_rows < 0 || !std::isfinite(k_ws_scale) || !std::isfinite(v_ws_scale) || k_ws_scale <= 0.0f ||
      v_ws_scale <= 0.0f)
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return NVFP4KV_OK;
  if (!ws_rows || !ws_k || !ws_v || !aligned(ws_rows, 8) || !aligned(ws_k, 16) || !aligned(ws_v, 16))
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  int nsm = 0;
  if ((st = current_num_sms(&nsm)) != NVFP4KV_OK) return st;
  return cuda_status(nvfp4kv::launch_quantize_append_fp8(
      *cache, static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), slot_mapping, num_tokens, ws_rows,
      total_rows, k_ws_scale, v_ws_scale, ws_k, ws_v, device_status, nsm, reinterpret_cast<cudaStream_t>(stream)));
}

int nvfp4kv_quantize_append_variant(int variant, const nvfp4kv_cache* cache, const void* k, const void* v,
                                    const int64_t* slot_mapping, int64_t num_tokens, const uint8_t* rand_k,
                                    const uint8_t* rand_v, int32_t* device_status, nvfp4kv_stream_t stream) {
  if (variant != NVFP4KV_VARIANT_SR && variant != NVFP4KV_VARIANT_HADAMARD && variant != NVFP4KV_VARIANT_MXFP4)
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  const int st = check_append(cache, k, v, slot_mapping, num_tokens, device_status);
  if (st != NVFP4KV_OK || num_tokens == 0) return st;
  if (variant == NVFP4KV_VARIANT_SR && (!rand_k || !rand_v || !aligned(rand_k, 16) || !aligned(rand_v, 16)))
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  return cuda_status(nvfp4kv::launch_quantize_variant(variant, *cache, static_cast<const uint16_t*>(k),
                                                      static_cast<const uint16_t*>(v), slot_mapping, num_tokens,
                                                      rand_k, rand_v, device_status,
                                                      reinterpret_cast<cudaStream_t>(stream)));
}

int nvfp4kv_decode_workspace_size(const nvfp4kv_cache* cache, int32_t batch, int32_t num_q_heads,
                                  size_t* bytes) {
  if (bytes == nullptr || cache == nullptr) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (cache->num_kv_heads <= 0 || batch < 0 || num_q_heads <= 0) return NVFP4KV_ERR_INVALID_ARGUMENT;
  int nsm = 0;
  int st = current_num_sms(&nsm);
  if (st != NVFP4KV_OK) return st;
  *bytes = nvfp4kv::decode_workspace_bytes(nsm, batch, cache->num_kv_heads);
  return NVFP4KV_OK;
}

size_t nvfp4kv_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t max_seq_len, int32_t num_sms) {
  (void)max_seq_len;  // the split is over pages of all sequences together: lengths do not size it
  if (batch < 0 || num_q_heads <= 0 || num_sms <= 0) return 0;
  // the KV-head count divides num_q_heads (num_q_heads = G * num_kv_heads)
  return nvfp4kv::decode_workspace_bound(num_sms, batch, num_q_heads);
}

// Host checks of decode arguments (nothing is enqueued); *nsm gets the
// current device's SM count when batch > 0.
static int check_decode(const nvfp4kv_cache* cache, const void* q, float* out, const int32_t* page_table,
                        int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                        float softmax_scale, void* workspace, size_t workspace_bytes, int32_t* device_status,
                        int* nsm) {
  int st = check_cache(cache);
  if (st != NVFP4KV_OK) return st;
  if (batch < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (num_q_heads % cache->num_kv_heads != 0) return NVFP4KV_ERR_INVALID_ARGUMENT;
  const int group = num_q_heads / cache->num_kv_heads;
  if (group > 8) return NVFP4KV_ERR_UNSUPPORTED;
  if (!positive_finite(softmax_scale)) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (batch == 0) return NVFP4KV_OK;
  // global page-head indices (sequence pages times KV heads) stay below 2^31
  if ((int64_t)batch * max_pages_per_seq * cache->num_kv_heads >= (int64_t(1) << 31) ||
      (int64_t)max_pages_per_seq * kPageSize >= (int64_t(1) << 31))
    return NVFP4KV_ERR_UNSUPPORTED;
  if (!q || !out || !page_table || !seq_lens) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(page_table, 4) || !aligned(seq_lens, 4))
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (device_status && !aligned(device_status, 4)) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if ((st = current_num_sms(nsm)) != NVFP4KV_OK) return st;
  const size_t need = nvfp4kv::decode_workspace_bytes(*nsm, batch, cache->num_kv_heads);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)) return NVFP4KV_ERR_WORKSPACE;
  return NVFP4KV_OK;
}

int nvfp4kv_decode_attention(const nvfp4kv_cache* cache, const void* q, float* out,
                             const int32_t* page_table, int32_t max_pages_per_seq, const int32_t* seq_lens,
                             int32_t batch, int32_t num_q_heads, float softmax_scale, void* workspace,
                             size_t workspace_bytes, int32_t* device_status, nvfp4kv_stream_t stream) {
  int nsm = 0;
  const int st = check_decode(cache, q, out, page_table, max_pages_per_seq, seq_lens, batch, num_q_heads,
                              softmax_scale, workspace, workspace_bytes, device_status, &nsm);
  if (st != NVFP4KV_OK || batch == 0) return st;
  return cuda_status(nvfp4kv::launch_decode(*cache, static_cast<const uint16_t*>(q), out, page_table,
                                            max_pages_per_seq, seq_lens, batch, num_q_heads, softmax_scale,
                                            workspace, device_status, nsm,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

int nvfp4kv_decode_attention_variant(int variant, const nvfp4kv_cache* cache, const void* q, float* out,
                                     const int32_t* page_table, int32_t max_pages_per_seq, const int32_t* seq_lens,
                                     int32_t batch, int32_t num_q_heads, float softmax_scale, void* workspace,
                                     size_t workspace_bytes, int32_t* device_status, nvfp4kv_stream_t stream) {
  if (variant != NVFP4KV_VARIANT_SR && variant != NVFP4KV_VARIANT_HADAMARD && variant != NVFP4KV_VARIANT_MXFP4)
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  int nsm = 0;
  const int st = check_decode(cache, q, out, page_table, max_pages_per_seq, seq_lens, batch, num_q_heads,
                              softmax_scale, workspace, workspace_bytes, device_status, &nsm);
  if (st != NVFP4KV_OK || batch == 0) return st;
  return cuda_status(nvfp4kv::launch_decode_variant(variant, *cache, static_cast<const uint16_t*>(q), out, page_table,
                                                    max_pages_per_seq, seq_lens, batch, num_q_heads, softmax_scale,
                                                    workspace, device_status, nsm,
                                                    reinterpret_cast<cudaStream_t>(stream)));
}

int nvfp4kv_append_decode_attention(const nvfp4kv_cache* cache, const void* k, const void* v,
                                    const int64_t* slot_mapping, int64_t num_tokens, const void* q, float* out,
                                    const int32_t* page_table, int32_t max_pages_per_seq,
                                    const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                    float softmax_scale, void* workspace, size_t workspace_bytes,
                                    int32_t* device_status, nvfp4kv_stream_t stream) {
  int st = check_append(cache, k, v, slot_mapping, num_tokens, device_status);
  if (st != NVFP4KV_OK) return st;
  int nsm = 0;
  st = check_decode(cache, q, out, page_table, max_pages_per_seq, seq_lens, batch, num_q_heads, softmax_scale,
                    workspace, workspace_bytes, device_status, &nsm);
  if (st != NVFP4KV_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (num_tokens > 0) {
    int asm_ = nsm;
    if (asm_ == 0 && (st = current_num_sms(&asm_)) != NVFP4KV_OK) return st;
    st = cuda_status(nvfp4kv::launch_quantize_append(*cache, static_cast<const uint16_t*>(k),
                                                     static_cast<const uint16_t*>(v), slot_mapping, num_tokens,
                                                     device_status, asm_, s));
    if (st != NVFP4KV_OK) return st;
  }
  if (batch == 0) return NVFP4KV_OK;
  return cuda_status(nvfp4kv::launch_decode(*cache, static_cast<const uint16_t*>(q), out, page_table,
                                            max_pages_per_seq, seq_lens, batch, num_q_heads, softmax_scale,
                                            workspace, device_status, nsm, s, num_tokens > 0));
}

int nvfp4kv_bf16_to_fp8_workspace(const void* k_bf16, const void* v_bf16, const int64_t* ws_rows,
                                   int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                   int64_t total_rows, float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                                   uint8_t* ws_v, int32_t* device_status, nvfp4kv_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || total_rows < 0) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (head_dim != 128) return NVFP4KV_ERR_UNSUPPORTED;
  if (!std::isfinite(k_ws_scale) || !std::isfinite(v_ws_scale) || k_ws_scale <= 0.0f || v_ws_scale <= 0.0f)
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (device_status && !aligned(device_status, 4)) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return NVFP4KV_OK;
  if (!k_bf16 || !v_bf16 || !ws_rows || !ws_k || !ws_v) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (!aligned(k_bf16, 16) || !aligned(v_bf16, 16) || !aligned(ws_rows, 8) || !aligned(ws_k, 16) ||
      !aligned(ws_v, 16))
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (num_tokens > (INT64_MAX / 2) / ((int64_t)num_kv_heads * 16)) return NVFP4KV_ERR_UNSUPPORTED;
  int nsm = 0;
  const int st = current_num_sms(&nsm);
  if (st != NVFP4KV_OK) return st;
  return cuda_status(nvfp4kv::launch_chunk_to_ws(static_cast<const uint16_t*>(k_bf16),
                                                 static_cast<const uint16_t*>(v_bf16), ws_rows, num_tokens,
                                                 num_kv_heads, total_rows, k_ws_scale, v_ws_scale, ws_k, ws_v,
                                                 device_status, nsm, reinterpret_cast<cudaStream_t>(stream)));
}

int nvfp4kv_extend_attention(const void* q_bf16, const int64_t* cu_q, int32_t max_q_len, const uint8_t* ws_k,
                             const uint8_t* ws_v, const int64_t* cu_prefix, const int32_t* prefix_lens,
                             int32_t batch, int64_t total_rows, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, float k_ws_scale, float v_ws_scale, float softmax_scale,
                             float* out, int32_t* device_status, nvfp4kv_stream_t stream) {
  if (batch < 0 || max_q_len < 0 || total_rows < 0 || num_q_heads <= 0 || num_kv_heads <= 0)
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (num_q_heads % num_kv_heads != 0) return NVFP4KV_ERR_INVALID_ARGUMENT;
  const int32_t group = num_q_heads / num_kv_heads;
  if (head_dim != 128 || group > 128 || (group & (group - 1)) != 0 || batch > 65535 || num_kv_heads > 65535)
    return NVFP4KV_ERR_UNSUPPORTED;
  for (float sc : {k_ws_scale, v_ws_scale, softmax_scale})
    if (!std::isfinite(sc) || sc <= 0.0f) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (device_status && !aligned(device_status, 4)) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (batch == 0 || max_q_len == 0) return NVFP4KV_OK;
  if (!q_bf16 || !cu_q || !ws_k || !ws_v || !cu_prefix || !prefix_lens || !out)
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (!aligned(q_bf16, 16) || !aligned(out, 16) || !aligned(ws_k, 16) || !aligned(ws_v, 16) || !aligned(cu_q, 8) ||
      !aligned(cu_prefix, 8) || !aligned(prefix_lens, 4))
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  if ((int64_t)max_q_len * group > (int64_t)INT32_MAX) return NVFP4KV_ERR_UNSUPPORTED;
  return cuda_status(nvfp4kv::launch_extend_attention(
      static_cast<const uint16_t*>(q_bf16), cu_q, max_q_len, ws_k, ws_v, cu_prefix, prefix_lens, batch,
      total_rows, num_q_heads, num_kv_heads, k_ws_scale, v_ws_scale, softmax_scale, out, device_status,
      reinterpret_cast<cudaStream_t>(stream)));
}

int nvfp4kv_tensor_amax(const void* x_bf16, int64_t n, float* amax, int accumulate,
                        nvfp4kv_stream_t stream) {
  if (n < 0 || amax == nullptr || !aligned(amax, 4)) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (n > 0 && (x_bf16 == nullptr || !aligned(x_bf16, 16))) return NVFP4KV_ERR_INVALID_ARGUMENT;
  int nsm = 0;
  const int st = current_num_sms(&nsm);
  if (st != NVFP4KV_OK) return st;
  return cuda_status(nvfp4kv::launch_tensor_amax(static_cast<const uint16_t*>(x_bf16), n, amax, accumulate != 0,
                                                 nsm, reinterpret_cast<cudaStream_t>(stream)));
}

int nvfp4kv_calibrated_global_scale(float amax, float* g) {
  if (g == nullptr || !std::isfinite(amax) || amax < 0.0f) return NVFP4KV_ERR_INVALID_ARGUMENT;
  *g = amax == 0.0f ? 1.0f : amax / (6.0f * 448.0f);  // one binary32 division
  return NVFP4KV_OK;
}

int nvfp4kv_dequant_to_fp8_workspace(const nvfp4kv_cache* cache, const int32_t* page_table,
                                     int32_t max_pages_per_seq, const int32_t* prefix_lens,
                                     const int64_t* cu_prefix, int32_t batch, int64_t total_rows,
                                     float k_ws_scale, float v_ws_scale, uint8_t* ws_k, uint8_t* ws_v,
                                     int32_t* device_status, nvfp4kv_stream_t stream) {
  int st = check_cache(cache);
  if (st != NVFP4KV_OK) return st;
  if (batch < 0 || total_rows < 0 || max_pages_per_seq <= 0) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (!positive_finite(k_ws_scale) || !positive_finite(v_ws_scale)) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (batch == 0 || total_rows == 0) return NVFP4KV_OK;
  if ((int64_t)max_pages_per_seq * kPageSize >= (int64_t(1) << 31)) return NVFP4KV_ERR_UNSUPPORTED;
  if (total_rows * cache->num_kv_heads >= (int64_t(1) << 40)) return NVFP4KV_ERR_UNSUPPORTED;
  if (!page_table || !prefix_lens || !cu_prefix || !ws_k || !ws_v) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (!aligned(page_table, 4) || !aligned(prefix_lens, 4) || !aligned(cu_prefix, 8) || !aligned(ws_k, 16) ||
      !aligned(ws_v, 16))
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (device_status && !aligned(device_status, 4)) return NVFP4KV_ERR_INVALID_ARGUMENT;
  return cuda_status(nvfp4kv::launch_dequant_fp8(*cache, page_table, max_pages_per_seq, prefix_lens, cu_prefix,
                                                 batch, total_rows, k_ws_scale, v_ws_scale, ws_k, ws_v,
                                                 device_status, reinterpret_cast<cudaStream_t>(stream)));
}

int nvfp4kv_stream_probe(const nvfp4kv_cache* cache, const int32_t* page_table, int32_t max_pages_per_seq,
                         const int32_t* seq_lens, int32_t batch, int mode, uint32_t* sink, int32_t* device_status,
                         nvfp4kv_stream_t stream) {
  int st = check_cache(cache);
  if (st != NVFP4KV_OK) return st;
  if (mode != NVFP4KV_PROBE_DECODE_PATTERN && mode != NVFP4KV_PROBE_WHOLE_PAGES) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (batch < 0 || max_pages_per_seq <= 0) return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (mode == NVFP4KV_PROBE_WHOLE_PAGES && cache->num_kv_heads > 16) return NVFP4KV_ERR_UNSUPPORTED;
  if (batch == 0) return NVFP4KV_OK;
  if ((int64_t)batch * max_pages_per_seq * cache->num_kv_heads >= (int64_t(1) << 31) ||
      (int64_t)max_pages_per_seq * kPageSize >= (int64_t(1) << 31))
    return NVFP4KV_ERR_UNSUPPORTED;
  if (!page_table || !seq_lens || !sink || !aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(sink, 4))
    return NVFP4KV_ERR_INVALID_ARGUMENT;
  if (device_status && !aligned(device_status, 4)) return NVFP4KV_ERR_INVALID_ARGUMENT;
  int nsm = 0;
  if ((st = current_num_sms(&nsm)) != NVFP4KV_OK) return st;
  return cuda_status(nvfp4kv::launch_stream_probe(*cache, page_table, max_pages_per_seq, seq_lens, batch, mode,
                                                  sink, device_status, nsm, reinterpret_cast<cudaStream_t>(stream)));
}

const char* nvfp4kv_last_cuda_error(void) {
  return last_cuda_error == cudaSuccess ? "no CUDA error" : cudaGetErrorString(last_cuda_error);
}

const char* nvfp4kv_status_string(int status) {
  switch (status) {
    case NVFP4KV_OK: return "ok";
    case NVFP4KV_ERR_INVALID_ARGUMENT: return "invalid argument";
    case NVFP4KV_ERR_UNSUPPORTED: return "unsupported configuration";
    case NVFP4KV_ERR_CUDA: return "CUDA error (see cudaGetLastError)";
    case NVFP4KV_ERR_WORKSPACE: return "workspace null, too small or misaligned";
    default: return "unknown status";
  }
}

}  // extern "C"
