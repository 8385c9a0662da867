// decode_no_alloc.cu -- paged decode attention for callers that cannot
// allocate device memory.
//
// nvfp4kv_decode_attention needs a caller-provided device workspace for its
// split-K pieces.  Some callers cannot provide one: code
// running inside a host allocator hook, a plug-in loaded by a runtime that
// owns all device memory, or a process that must never call cudaMalloc on its
// hot path.  nvfp4kv_decode_attention_static serves them by using a fixed
// scratch array that lives in this library's device image instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds NVFP4KV_STATIC_SCRATCH_BYTES of device memory until the
// process exits.  Its device address is looked up once per device with
// cudaGetSymbolAddress (the host-side symbol is only a stand-in and must never
// be handed to a kernel).  Each call runs the ordinary decode through
// nvfp4kv_decode_attention, which writes every part of the workspace it later
// reads, so the scratch needs no clearing; nothing in this file allocates or
// frees memory.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "nvfp4kv.h"

namespace {

constexpr size_t kScratchBytes = NVFP4KV_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself: one copy per device context that loads the library.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Device address of g_decode_scratch per device (nullptr until resolved).
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Resolve (once per device, with that device current) the scratch address.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4KV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return NVFP4KV_ERR_UNSUPPORTED;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return NVFP4KV_ERR_CUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return NVFP4KV_OK;
}

}  // namespace

extern "C" int nvfp4kv_decode_attention_static(const nvfp4kv_cache* cache, const void* q, float* out,
                                               const int32_t* page_table, int32_t max_pages_per_seq,
                                               const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                               float softmax_scale, int32_t* device_status,
                                               nvfp4kv_stream_t stream) {
  if (cache == nullptr || num_q_heads <= 0 || batch < 0) return NVFP4KV_ERR_INVALID_ARGUMENT;
  size_t need = 0;
  int st = nvfp4kv_decode_workspace_size(cache, batch, num_q_heads, &need);
  if (st != NVFP4KV_OK) return st;
  if (need > kScratchBytes) return NVFP4KV_ERR_WORKSPACE;  // batch too large for the fixed scratch
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != NVFP4KV_OK) return st;
  return nvfp4kv_decode_attention(cache, q, out, page_table, max_pages_per_seq, seq_lens, batch, num_q_heads,
                                  softmax_scale, scratch, kScratchBytes, device_status, stream);
}
