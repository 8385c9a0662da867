// dequant_fp8.cu -- NVFP4 prefix -> FP8 E4M3 workspace for chunked prefill /
// extend ("nvfp4-kv-cache-memory-wall", section 3, item 2: the cached NVFP4
// prefix is dequantised into one FP8 workspace pair that all layers reuse).
//
//   ws[cu_prefix[b] + t][h][d] = E4M3(fp32(fp32(e2m1 * E4M3val(sb)) * g) / s_ws)
//
// Each thread owns 32 values (two 16-value blocks) of one (row, head) in both
// K and V: a 16-byte data load and a 2-byte scale load per tensor, two 16-byte
// stores per tensor.  With g = s_ws = 1 the product e2m1 * E4M3val(sb) is
// exact in f16 and is rounded straight to E4M3 (cvt e2m1x2 -> f16x2, one
// f16x2 multiply, cvt f16x2 -> e4m3x2); otherwise the fp32 steps are taken as
// written.  HBM-bound: 9/16 B read and 1 B written per value.
#include "nvfp4kv_device.cuh"
#include "nvfp4kv_launch.h"

namespace nvfp4kv {
namespace {

struct DequantParams {
  const uint8_t* k_data;
  const uint8_t* v_data;
  const uint8_t* k_scale;
  const uint8_t* v_scale;
  int64_t num_pages;
  int32_t hkv;
  const int32_t* page_table;
  int32_t max_pages;
  const int32_t* prefix_lens;
  const int64_t* cu_prefix;
  int32_t batch;
  int64_t items;  // total_rows * hkv
  float gk, gv, sk, sv;
  uint8_t* ws_k;
  uint8_t* ws_v;
  int32_t* status;
};

constexpr int kThreads = 256;

// The sequence whose row range holds `row`: the largest b with cu[b] <= row.
__device__ __forceinline__ int find_seq(const int64_t* cu, int batch, int64_t row) {
  int lo = 0, hi = batch;  // invariant: cu[lo] <= row (when row >= cu[0])
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(cu + mid) <= row) lo = mid; else hi = mid;
  }
  return lo;
}

// 16 data bytes + 2 scale bytes (32 values) -> 32 E4M3 bytes, unit scales.
__device__ __forceinline__ void convert_unit(const uint4& d, uint32_t scales2, uint4 out[2]) {
  const uint32_t s2 = e4m3x2_to_f16x2(scales2);  // (block 0 scale, block 1 scale)
  const uint32_t s_lo = __byte_perm(s2, 0, 0x1010);
  const uint32_t s_hi = __byte_perm(s2, 0, 0x3232);
  const uint32_t w[4] = {d.x, d.y, d.z, d.w};
  uint32_t o[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t s = j < 2 ? s_lo : s_hi;
    const uint32_t b0 = e4m3x2_from_f16x2(hmul2(e2m1x2_to_f16x2<0>(w[j]), s));
    const uint32_t b1 = e4m3x2_from_f16x2(hmul2(e2m1x2_to_f16x2<1>(w[j]), s));
    const uint32_t b2 = e4m3x2_from_f16x2(hmul2(e2m1x2_to_f16x2<2>(w[j]), s));
    const uint32_t b3 = e4m3x2_from_f16x2(hmul2(e2m1x2_to_f16x2<3>(w[j]), s));
    o[2 * j] = b0 | (b1 << 16);
    o[2 * j + 1] = b2 | (b3 << 16);
  }
  out[0] = make_uint4(o[0], o[1], o[2], o[3]);
  out[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

template <int K>
__device__ __forceinline__ uint32_t convert_pair_general(uint32_t w, uint32_t s, float g, float sws) {
  const uint32_t h2 = hmul2(e2m1x2_to_f16x2<K>(w), s);  // exact e2m1 * E4M3val(sb)
  const float v0 = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
  const float v1 = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
  const float z0 = __fdiv_rn(__fmul_rn(v0, g), sws);
  const float z1 = __fdiv_rn(__fmul_rn(v1, g), sws);
  return e4m3x2_from_f32(z0, z1);
}

// Same, any global scale g and workspace scale s_ws.
__device__ __forceinline__ void convert_general(const uint4& d, uint32_t scales2, float g, float sws,
                                                uint4 out[2]) {
  const uint32_t s2 = e4m3x2_to_f16x2(scales2);
  const uint32_t s_lo = __byte_perm(s2, 0, 0x1010);
  const uint32_t s_hi = __byte_perm(s2, 0, 0x3232);
  const uint32_t w[4] = {d.x, d.y, d.z, d.w};
  uint32_t o[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t s = j < 2 ? s_lo : s_hi;
    o[2 * j] = convert_pair_general<0>(w[j], s, g, sws) | (convert_pair_general<1>(w[j], s, g, sws) << 16);
    o[2 * j + 1] = convert_pair_general<2>(w[j], s, g, sws) | (convert_pair_general<3>(w[j], s, g, sws) << 16);
  }
  out[0] = make_uint4(o[0], o[1], o[2], o[3]);
  out[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

template <bool kUnit>
__global__ void __launch_bounds__(kThreads) dequant_fp8_kernel(DequantParams p) {
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  const int64_t total = p.items * 4;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += nthreads) {
    const int64_t item = idx >> 2;
    const int q = (int)(idx & 3);  // values [32 q, 32 q + 32)
    const int64_t row = item / p.hkv;
    const int h = (int)(item - row * p.hkv);
    if (row < __ldg(p.cu_prefix)) continue;
    const int b = find_seq(p.cu_prefix, p.batch, row);
    const int64_t t = row - __ldg(p.cu_prefix + b);
    int32_t L = __ldg(p.prefix_lens + b);
    if (L < 0 || L > p.max_pages * kPage) {
      flag_error(p.status, NVFP4KV_DEVERR_LENGTH);
      L = L < 0 ? 0 : p.max_pages * kPage;
    }
    if (t >= L) continue;  // a row between this prefix and the next sequence
    const int32_t page = __ldg(p.page_table + (int64_t)b * p.max_pages + (t >> 4));
    uint4* dst_k = reinterpret_cast<uint4*>(p.ws_k + (item * kHeadDim + 32 * q));
    uint4* dst_v = reinterpret_cast<uint4*>(p.ws_v + (item * kHeadDim + 32 * q));
    if (page < 0 || page >= p.num_pages) {
      flag_error(p.status, NVFP4KV_DEVERR_PAGE);
      const uint4 z = make_uint4(0, 0, 0, 0);
      dst_k[0] = z; dst_k[1] = z; dst_v[0] = z; dst_v[1] = z;
      continue;
    }
    const int64_t src_row = ((int64_t)page * p.hkv + h) * kPage + (t & (kPage - 1));
    const uint4 kd = __ldg(reinterpret_cast<const uint4*>(p.k_data + src_row * kRowBytes) + q);
    const uint4 vd = __ldg(reinterpret_cast<const uint4*>(p.v_data + src_row * kRowBytes) + q);
    const uint32_t ks = __ldg(reinterpret_cast<const uint16_t*>(p.k_scale + src_row * kRowScales) + q);
    const uint32_t vs = __ldg(reinterpret_cast<const uint16_t*>(p.v_scale + src_row * kRowScales) + q);
    uint4 ok[2], ov[2];
    if constexpr (kUnit) {
      convert_unit(kd, ks, ok);
      convert_unit(vd, vs, ov);
    } else {
      convert_general(kd, ks, p.gk, p.sk, ok);
      convert_general(vd, vs, p.gv, p.sv, ov);
    }
    dst_k[0] = ok[0]; dst_k[1] = ok[1];
    dst_v[0] = ov[0]; dst_v[1] = ov[1];
  }
}

}  // namespace

cudaError_t launch_dequant_fp8(const nvfp4kv_cache& c, const int32_t* page_table, int32_t max_pages,
                               const int32_t* prefix_lens, const int64_t* cu_prefix, int32_t batch,
                               int64_t total_rows, float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                               uint8_t* ws_v, int32_t* device_status, int num_sms, cudaStream_t stream) {
  DequantParams p;
  p.k_data = c.k_data;
  p.v_data = c.v_data;
  p.k_scale = c.k_scale;
  p.v_scale = c.v_scale;
  p.num_pages = c.num_pages;
  p.hkv = c.num_kv_heads;
  p.page_table = page_table;
  p.max_pages = max_pages;
  p.prefix_lens = prefix_lens;
  p.cu_prefix = cu_prefix;
  p.batch = batch;
  p.items = total_rows * c.num_kv_heads;
  p.gk = c.k_global_scale;
  p.gv = c.v_global_scale;
  p.sk = k_ws_scale;
  p.sv = v_ws_scale;
  p.ws_k = ws_k;
  p.ws_v = ws_v;
  p.status = device_status;
  const int64_t threads_needed = p.items * 4;
  int64_t blocks = (threads_needed + kThreads - 1) / kThreads;
  const int64_t max_blocks = (int64_t)num_sms * (2048 / kThreads);
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  const bool unit = c.k_global_scale == 1.0f && c.v_global_scale == 1.0f && k_ws_scale == 1.0f &&
                    v_ws_scale == 1.0f;
  if (unit)
    dequant_fp8_kernel<true><<<(unsigned)blocks, kThreads, 0, stream>>>(p);
  else
    dequant_fp8_kernel<false><<<(unsigned)blocks, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nvfp4kv
