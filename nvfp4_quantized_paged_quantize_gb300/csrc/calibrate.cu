// calibrate.cu -- the per-tensor amax that a calibrated global scale is made
// from ("nvfp4-kv-cache-memory-wall", section 2: the FP32 per-tensor scale is
// left at 1 by the uncalibrated public setting; a calibrated one maps the
// tensor's largest magnitude onto E2M1 6 x E4M3 448, g = amax / 2688).
//
// A grid-stride pass over 16-byte vectors of bf16: magnitudes are the bit
// patterns with the sign cleared, and non-negative bf16 patterns order like
// unsigned integers, so the maximum is taken on integers (two lanes of 16 bits
// per instruction) and is exact.  Each warp folds its maximum into the result
// with one atomicMax on the fp32 bit pattern (bf16 bits << 16), which orders
// like the value for non-negative floats.  HBM-bound: 2 bytes read per value.
#include "nvfp4kv_device.cuh"
#include "nvfp4kv_launch.h"

namespace nvfp4kv {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // 16-byte loads in flight per thread

__device__ __forceinline__ uint32_t abs_max2(const uint4& w) {
  const uint32_t m = 0x7FFF7FFFu;
  return __vmaxu2(__vmaxu2(w.x & m, w.y & m), __vmaxu2(w.z & m, w.w & m));
}

__global__ void __launch_bounds__(kThreads) tensor_amax_kernel(const uint16_t* x, int64_t n, uint32_t* out) {
  const int64_t nvec = n >> 3;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t m2 = 0;  // two 16-bit lanes of magnitude maxima
  int64_t v = first;
  for (; v + (kUnroll - 1) * stride < nvec; v += kUnroll * stride) {
    uint4 w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) w[u] = __ldg(xv + v + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) m2 = __vmaxu2(m2, abs_max2(w[u]));
  }
  for (; v < nvec; v += stride) m2 = __vmaxu2(m2, abs_max2(__ldg(xv + v)));
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  for (int64_t t = nvec * 8 + first; t < n; t += stride) m = max(m, (uint32_t)(__ldg(x + t) & 0x7FFFu));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(out, m << 16);
}

}  // namespace

cudaError_t launch_tensor_amax(const uint16_t* x, int64_t n, float* amax, bool accumulate, int num_sms,
                               cudaStream_t stream) {
  if (!accumulate) {
    const cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), stream);  // +0.0f
    if (e != cudaSuccess) return e;
  }
  if (n == 0) return cudaSuccess;
  const int64_t vec = (n + 7) / 8;
  int64_t blocks = (vec + (int64_t)kThreads * kUnroll - 1) / ((int64_t)kThreads * kUnroll);
  const int64_t max_blocks = (int64_t)num_sms * (2048 / kThreads);
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  tensor_amax_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(x, n, reinterpret_cast<uint32_t*>(amax));
  return cudaGetLastError();
}

}  // namespace nvfp4kv
