// quantize_append.cu -- NVFP4 quantize-on-append of new K/V tokens into the
// paged cache ("nvfp4-kv-cache-memory-wall", section 3: new K/V are quantised
// to NVFP4 on the way into the cache; section 2: two-level scaling).
//
// One warp handles one (token, KV head) row of K (lanes 0-15) and of V (lanes
// 16-31) per step; each lane owns 8 consecutive values (one 16-byte load), two
// lanes form a 16-value block.  Per block:
//   amax = max |x|                       (exact; inputs are bf16)
//   sb   = E4M3(amax / (6 g))            (IEEE division, RNE, saturating)
//   den  = E4M3val(sb) * g
//   code = E2M1(x / den)                 (x / den rounded to nearest, RNE, saturating)
// A block with den == 0 stores signed zeros.  The row's 64 data bytes and 8
// scale bytes go to slot slot_mapping[token].  HBM-bound: 2 B read and 9/16 B
// written per value.
#include "nvfp4kv_device.cuh"
#include "nvfp4kv_launch.h"

namespace nvfp4kv {
namespace {

struct QuantParams {
  const uint16_t* k;
  const uint16_t* v;
  const int64_t* slots;
  int32_t rows;  // num_tokens * num_kv_heads (< 2^31, checked on the host)
  int32_t hkv;
  int64_t capacity;  // num_pages * page_size
  uint8_t* k_data;
  uint8_t* v_data;
  uint8_t* k_scale;
  uint8_t* v_scale;
  float gk, gv;
  int32_t* status;
};

constexpr int kThreads = 256;
constexpr int kRowsPerStep = 2;  // rows whose loads are in flight together per warp

__device__ __forceinline__ void unpack_bf16x8(const uint4& x, float f[8]) {
  f[0] = bf16_to_f32(x.x & 0xFFFFu); f[1] = bf16_to_f32(x.x >> 16);
  f[2] = bf16_to_f32(x.y & 0xFFFFu); f[3] = bf16_to_f32(x.y >> 16);
  f[4] = bf16_to_f32(x.z & 0xFFFFu); f[5] = bf16_to_f32(x.z >> 16);
  f[6] = bf16_to_f32(x.w & 0xFFFFu); f[7] = bf16_to_f32(x.w >> 16);
}

__global__ void __launch_bounds__(kThreads) quantize_append_kernel(QuantParams p) {
  const int lane = threadIdx.x & 31;
  const int tensor = lane >> 4;  // 0: K, 1: V
  const int sub = lane & 15;     // values [8 sub, 8 sub + 8) of the row
  const uint16_t* src = tensor ? p.v : p.k;
  uint8_t* data = tensor ? p.v_data : p.k_data;
  uint8_t* scale = tensor ? p.v_scale : p.k_scale;
  const float g = tensor ? p.gv : p.gk;
  const float t6 = __fmul_rn(6.0f, g);  // the block amax maps onto E2M1's 6
  const int warp = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  const int nwarps = (int)((gridDim.x * (unsigned)blockDim.x) >> 5);

  for (int r0 = warp * kRowsPerStep; r0 < p.rows; r0 += nwarps * kRowsPerStep) {
    uint4 x[kRowsPerStep];
    int64_t slot[kRowsPerStep];
#pragma unroll
    for (int u = 0; u < kRowsPerStep; ++u) {
      const int r = r0 + u;
      slot[u] = -1;
      if (r < p.rows) {
        slot[u] = __ldg(p.slots + r / p.hkv);
        x[u] = __ldg(reinterpret_cast<const uint4*>(src + (int64_t)r * kHeadDim) + sub);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsPerStep; ++u) {
      const int r = r0 + u;
      // slot[u] and r are the same in every lane: the branches are warp-uniform
      if (r >= p.rows || slot[u] < 0) continue;
      if (slot[u] >= p.capacity) {
        if (lane == 0) flag_error(p.status, NVFP4KV_DEVERR_SLOT);
        continue;
      }
      const int h = r % p.hkv;
      const int64_t row = ((slot[u] >> 4) * p.hkv + h) * kPage + (slot[u] & (kPage - 1));
      float f[8];
      unpack_bf16x8(x[u], f);
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      const uint32_t sb = e4m3_from_f32(__fdiv_rn(amax, t6));
      const float den = __fmul_rn(e4m3_to_f32(sb), g);
      // x / den rounded to nearest: one correctly rounded reciprocal per block,
      // then per value q0 = x*r and Markstein's correction q0 + r*(x - den*q0)
      // (two FMAs), which gives the correctly rounded quotient while den, 1/den
      // and every quotient of the block stay well inside the normal range (a
      // saturated block scale can push quotients towards overflow); otherwise
      // IEEE division.
      const float rcp = __frcp_rn(den);
      const bool fast = den >= 0x1p-100f && den <= 0x1p+100f && __fmul_rn(amax, rcp) < 0x1p+64f;
      float y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (den == 0.0f) {
          y[i] = copysignf(0.0f, f[i]);
        } else if (fast) {
          const float q0 = __fmul_rn(f[i], rcp);
          const float rem = __fmaf_rn(-q0, den, f[i]);
          // a quotient that rounds to zero can come out as +0 for negative x;
          // the sign of x / den is the sign of x (den > 0)
          y[i] = copysignf(__fmaf_rn(rem, rcp, q0), f[i]);
        } else {
          y[i] = __fdiv_rn(f[i], den);
        }
      }
      uint32_t packed = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) packed |= e2m1x2_from_f32(y[2 * k], y[2 * k + 1]) << (8 * k);
      reinterpret_cast<uint32_t*>(data + row * kRowBytes)[sub] = packed;
      if ((sub & 1) == 0) scale[row * kRowScales + (sub >> 1)] = (uint8_t)sb;
    }
  }
}

}  // namespace

cudaError_t launch_quantize_append(const nvfp4kv_cache& c, const uint16_t* k, const uint16_t* v,
                                   const int64_t* slot_mapping, int64_t num_tokens,
                                   int32_t* device_status, int num_sms, cudaStream_t stream) {
  QuantParams p;
  p.k = k;
  p.v = v;
  p.slots = slot_mapping;
  p.rows = (int32_t)(num_tokens * c.num_kv_heads);
  p.hkv = c.num_kv_heads;
  p.capacity = c.num_pages * (int64_t)c.page_size;
  p.k_data = c.k_data;
  p.v_data = c.v_data;
  p.k_scale = c.k_scale;
  p.v_scale = c.v_scale;
  p.gk = c.k_global_scale;
  p.gv = c.v_global_scale;
  p.status = device_status;
  const int warps_needed = (p.rows + kRowsPerStep - 1) / kRowsPerStep;
  const int warps_per_block = kThreads / 32;
  int blocks = (warps_needed + warps_per_block - 1) / warps_per_block;
  const int max_blocks = num_sms * (2048 / kThreads);
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  quantize_append_kernel<<<blocks, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nvfp4kv
