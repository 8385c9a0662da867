// dequant_fp8.cu -- NVFP4 prefix -> FP8 E4M3 workspace for chunked prefill /
// extend ("nvfp4-kv-cache-memory-wall", section 3, item 2: the cached NVFP4
// prefix is dequantised into one FP8 workspace pair that all layers reuse).
//
//   ws[cu_prefix[b] + t][h][d] = E4M3(fp32(fp32(e2m1 * E4M3val(sb)) * g) / s_ws)
//
// One warp converts one page-head (16 rows of one KV head of one sequence) of
// K or of V, reading its 1 KiB of data contiguously.  K: lane l loads row
// l / 2, values [64 (l % 2), 64 (l % 2) + 64) -- two 16-byte data loads and
// one 4-byte scale load -- then trades blocks with the row's other lane so
// that each store of the pair fills a 32-byte sector.  V (stored by token
// pair): lane l loads dimensions [32 (l % 4), 32 (l % 4) + 32) of token pair
// l / 4, each byte one dimension of both tokens, which one conversion turns
// into the two tokens' values (lane l takes blocks l % 4 and l % 4 + 4, so
// that the four lanes of a pair fill 64 contiguous bytes of each output row
// with each store); the two tokens' scales of a block are one 16-bit load.
// The page-table lookup and the row arithmetic are done once per page-head; a
// block takes four page-heads (K and V warps), and the grid holds every block,
// so the block scheduler keeps each SM full of independent loads.  With g = s_ws = 1 the product e2m1 * E4M3val(sb) is exact
// in f16 and is rounded straight to E4M3 (cvt e2m1x2 -> f16x2, one f16x2
// multiply, cvt f16x2 -> e4m3x2); otherwise the fp32 steps are taken as
// written.  HBM-bound: 9/16 B read and 1 B written per value.
#include "nvfp4kv_device.cuh"
#include "nvfp4kv_launch.h"

namespace nvfp4kv {
namespace {

struct DequantParams {
  const uint8_t* pages;  // [num_pages][hkv][kPageHeadBytes]
  int64_t num_pages;
  int32_t hkv;
  const int32_t* page_table;
  int32_t max_pages;
  const int32_t* prefix_lens;
  const int64_t* cu_prefix;
  int32_t batch;
  int64_t total_rows;
  int32_t chunks_per_seq;  // blocks per sequence: ceil(max_pages * hkv / kHeadsPerBlock)
  float gk, gv, sk, sv;
  float rsk, rsv;          // RN(1 / s_ws)
  bool sk_fast, sv_fast;   // s_ws and 1 / s_ws well inside the normal range
  uint8_t* ws_k;
  uint8_t* ws_v;
  int32_t* status;
};

constexpr int kThreads = 256;
constexpr int kHeadsPerBlock = kThreads / 64;  // page-heads per block: a K warp and a V warp each

// 8 data bytes (16 values of one block) -> 16 E4M3 bytes with unit scales:
// cvt e2m1x2 -> f16x2, one f16x2 multiply by the block scale (exact), cvt
// f16x2 -> e4m3x2 (the one rounding).
__device__ __forceinline__ uint4 convert_block_unit(uint32_t w0, uint32_t w1, uint32_t s16x2) {
  uint32_t o[4];
  const uint32_t w[2] = {w0, w1};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t b0 = e4m3x2_from_f16x2(hmul2(e2m1x2_to_f16x2<0>(w[j]), s16x2));
    const uint32_t b1 = e4m3x2_from_f16x2(hmul2(e2m1x2_to_f16x2<1>(w[j]), s16x2));
    const uint32_t b2 = e4m3x2_from_f16x2(hmul2(e2m1x2_to_f16x2<2>(w[j]), s16x2));
    const uint32_t b3 = e4m3x2_from_f16x2(hmul2(e2m1x2_to_f16x2<3>(w[j]), s16x2));
    o[2 * j] = b0 | (b1 << 16);
    o[2 * j + 1] = b2 | (b3 << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// fp32(fp32(v * g) / sws) rounded to E4M3, for the two halves of an exact f16x2 product.
template <int K>
__device__ __forceinline__ uint32_t convert_pair_general(uint32_t w, uint32_t s16x2, float g, float sws, float rs,
                                                         bool fast) {
  const uint32_t h2 = hmul2(e2m1x2_to_f16x2<K>(w), s16x2);  // exact e2m1 * E4M3val(sb)
  const float a0 = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))), g);
  const float a1 = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(h2 >> 16))), g);
  float z0, z1;
  const float q0 = __fmul_rn(a0, rs), q1 = __fmul_rn(a1, rs);
  if (fast && fabsf(q0) < 0x1p+64f && fabsf(q1) < 0x1p+64f) {
    // correctly rounded a / sws (Markstein) while the first quotient stays far from
    // overflow; the sign of a zero quotient is the sign of a
    z0 = copysignf(__fmaf_rn(__fmaf_rn(-q0, sws, a0), rs, q0), a0);
    z1 = copysignf(__fmaf_rn(__fmaf_rn(-q1, sws, a1), rs, q1), a1);
  } else {
    z0 = __fdiv_rn(a0, sws);
    z1 = __fdiv_rn(a1, sws);
  }
  return e4m3x2_from_f32(z0, z1);
}

__device__ __forceinline__ uint4 convert_block_general(uint32_t w0, uint32_t w1, uint32_t s16x2, float g, float sws,
                                                       float rs, bool fast) {
  uint32_t o[4];
  const uint32_t w[2] = {w0, w1};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    o[2 * j] = convert_pair_general<0>(w[j], s16x2, g, sws, rs, fast) |
               (convert_pair_general<1>(w[j], s16x2, g, sws, rs, fast) << 16);
    o[2 * j + 1] = convert_pair_general<2>(w[j], s16x2, g, sws, rs, fast) |
                   (convert_pair_general<3>(w[j], s16x2, g, sws, rs, fast) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// 32 data bytes + 4 scale bytes (64 values, 4 blocks) -> 64 E4M3 bytes.
template <bool kUnit>
__device__ __forceinline__ void convert_half_row(const uint4& d0, const uint4& d1, uint32_t sc4, float g, float sws,
                                                 float rs, bool fast, uint4 out[4]) {
  const uint32_t s01 = e4m3x2_to_f16x2(sc4 & 0xFFFFu);  // (block 0, block 1) scales as f16
  const uint32_t s23 = e4m3x2_to_f16x2(sc4 >> 16);
  const uint32_t sc[4] = {__byte_perm(s01, 0, 0x1010), __byte_perm(s01, 0, 0x3232), __byte_perm(s23, 0, 0x1010),
                          __byte_perm(s23, 0, 0x3232)};
  const uint32_t w[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if constexpr (kUnit)
      out[k] = convert_block_unit(w[2 * k], w[2 * k + 1], sc[k]);
    else
      out[k] = convert_block_general(w[2 * k], w[2 * k + 1], sc[k], g, sws, rs, fast);
  }
}

// Unit scales fit 32 registers (full occupancy); the general path takes up to 48
// (no spills).
template <bool kUnit>
__global__ void __launch_bounds__(kThreads, kUnit ? 8 : 5) dequant_fp8_kernel(DequantParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tensor = warp & 1;  // 0: K, 1: V
  const int r = lane >> 1, half = lane & 1;
  uint8_t* ws = tensor ? p.ws_v : p.ws_k;
  const float g = tensor ? p.gv : p.gk, sws = tensor ? p.sv : p.sk, rs = tensor ? p.rsv : p.rsk;
  const bool fast = tensor ? p.sv_fast : p.sk_fast;
  const int64_t units = (int64_t)p.batch * p.chunks_per_seq;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int b = (int)(u / p.chunks_per_seq);
    const int ph = (int)(u - (int64_t)b * p.chunks_per_seq) * kHeadsPerBlock + (warp >> 1);  // page * hkv + h
    const int pg = ph / p.hkv, h = ph - pg * p.hkv;
    if (pg >= p.max_pages) continue;
    // the page id, the length and the row base are loaded together
    const int32_t page = __ldg(p.page_table + (int64_t)b * p.max_pages + pg);
    int32_t L = __ldg(p.prefix_lens + b);
    const int64_t base = __ldg(p.cu_prefix + b);
    if (L < 0 || L > p.max_pages * kPage) {
      if (lane == 0 && ph == 0 && tensor == 0) flag_error(p.status, NVFP4KV_DEVERR_LENGTH);
      L = L < 0 ? 0 : p.max_pages * kPage;
    }
    if (pg * kPage >= L) continue;  // a page past this prefix
    const bool page_ok = page >= 0 && page < p.num_pages;
    const uint8_t* phd = p.pages + ((int64_t)(page_ok ? page : 0) * p.hkv + h) * kPageHeadBytes;
    if (tensor == 1) {
      // V: token pair q = lane / 4, blocks c and c + 4 (dimensions 16 c .., 64 + 16 c ..)
      const int q = lane >> 2, c = lane & 3;
      const int te = pg * kPage + 2 * q;  // the pair's tokens te, te + 1 of the prefix
      const int64_t orow = base + te;
      const bool live_e = te < L && orow >= 0 && orow < p.total_rows;
      const bool live_o = te + 1 < L && orow + 1 >= 0 && orow + 1 < p.total_rows;
      uint4* dst_e = reinterpret_cast<uint4*>(ws + (orow * p.hkv + h) * kHeadDim) + c;
      uint4* dst_o = reinterpret_cast<uint4*>(ws + ((orow + 1) * p.hkv + h) * kHeadDim) + c;
      if (!page_ok) {
        if (lane == 0) flag_error(p.status, NVFP4KV_DEVERR_PAGE);
        const uint4 z = make_uint4(0, 0, 0, 0);
        if (live_e) dst_e[0] = dst_e[4] = z;
        if (live_o) dst_o[0] = dst_o[4] = z;
        continue;
      }
      if (!live_e && !live_o) continue;
      const uint4* src = reinterpret_cast<const uint4*>(phd + kOffVData + q * kVPairBytes) + c;
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        // block c + 4 hb: 16 bytes, and the (token te, token te + 1) scales as f16x2
        const uint4 d = __ldg(src + 4 * hb);
        const uint32_t sc =
            e4m3x2_to_f16x2(__ldg(reinterpret_cast<const uint16_t*>(phd + v_scale_offset(2 * q, c + 4 * hb))));
        const uint32_t w[4] = {d.x, d.y, d.z, d.w};
        uint32_t oe[4], oo[4];  // the two tokens' output bytes, 4 dimensions per word
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t r[4];  // dimension 4k + i of the block: low byte token te, high byte token te + 1
          if constexpr (kUnit) {
            r[0] = e4m3x2_from_f16x2(hmul2(e2m1x2_to_f16x2<0>(w[k]), sc));
            r[1] = e4m3x2_from_f16x2(hmul2(e2m1x2_to_f16x2<1>(w[k]), sc));
            r[2] = e4m3x2_from_f16x2(hmul2(e2m1x2_to_f16x2<2>(w[k]), sc));
            r[3] = e4m3x2_from_f16x2(hmul2(e2m1x2_to_f16x2<3>(w[k]), sc));
          } else {
            r[0] = convert_pair_general<0>(w[k], sc, g, sws, rs, fast);
            r[1] = convert_pair_general<1>(w[k], sc, g, sws, rs, fast);
            r[2] = convert_pair_general<2>(w[k], sc, g, sws, rs, fast);
            r[3] = convert_pair_general<3>(w[k], sc, g, sws, rs, fast);
          }
          const uint32_t x01 = r[0] | (r[1] << 16), x23 = r[2] | (r[3] << 16);
          oe[k] = __byte_perm(x01, x23, 0x6420);
          oo[k] = __byte_perm(x01, x23, 0x7531);
        }
        if (live_e) dst_e[4 * hb] = make_uint4(oe[0], oe[1], oe[2], oe[3]);
        if (live_o) dst_o[4 * hb] = make_uint4(oo[0], oo[1], oo[2], oo[3]);
      }
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(phd + kOffKData + r * kRowBytes) + 2 * half;
    const uint4 d0 = __ldg(src), d1 = __ldg(src + 1);  // blocks 4 half .. 4 half + 3
    // the scales of blocks 4 half .. 4 half + 3 of row r: 4 adjacent bytes
    const uint32_t sc4 = __ldg(reinterpret_cast<const uint32_t*>(phd + k_scale_offset(r, 4 * half)));
    const int t = pg * kPage + r;   // this lane's token of the prefix
    const int64_t orow = base + t;  // its workspace row
    const bool live = t < L && orow >= 0 && orow < p.total_rows;
    // 16-byte output chunk k of this lane goes to block 2k + half of the row, so the
    // two lanes of a row fill whole 32-byte sectors with each store
    uint4* dst = reinterpret_cast<uint4*>(ws + (orow * p.hkv + h) * kHeadDim) + half;
    if (!page_ok) {
      if (lane == 0) flag_error(p.status, NVFP4KV_DEVERR_PAGE);
      if (live) {
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[2 * k] = z;
      }
      continue;
    }
    // trade blocks with the row's other lane: half 0 ends up with blocks 0, 2, 4, 6
    // and half 1 with blocks 1, 3, 5, 7 (8 data bytes and 1 scale byte per block)
    const uint32_t x0 = __shfl_xor_sync(0xFFFFFFFFu, half ? d0.x : d0.z, 1);
    const uint32_t x1 = __shfl_xor_sync(0xFFFFFFFFu, half ? d0.y : d0.w, 1);
    const uint32_t x2 = __shfl_xor_sync(0xFFFFFFFFu, half ? d1.x : d1.z, 1);
    const uint32_t x3 = __shfl_xor_sync(0xFFFFFFFFu, half ? d1.y : d1.w, 1);
    const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, sc4, 1);
    const uint4 e0 = half ? make_uint4(x0, x1, x2, x3) : make_uint4(d0.x, d0.y, d1.x, d1.y);
    const uint4 e1 = half ? make_uint4(d0.z, d0.w, d1.z, d1.w) : make_uint4(x0, x1, x2, x3);
    const uint32_t esc = __byte_perm(sc4, other, half ? 0x3175 : 0x6420);
    if (!live) continue;
    uint4 o[4];
    convert_half_row<kUnit>(e0, e1, esc, g, sws, rs, fast, o);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[2 * k] = o[k];
  }
}

}  // namespace

cudaError_t launch_dequant_fp8(const nvfp4kv_cache& c, const int32_t* page_table, int32_t max_pages,
                               const int32_t* prefix_lens, const int64_t* cu_prefix, int32_t batch,
                               int64_t total_rows, float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                               uint8_t* ws_v, int32_t* device_status, cudaStream_t stream) {
  DequantParams p;
  p.pages = c.pages;
  p.num_pages = c.num_pages;
  p.hkv = c.num_kv_heads;
  p.page_table = page_table;
  p.max_pages = max_pages;
  p.prefix_lens = prefix_lens;
  p.cu_prefix = cu_prefix;
  p.batch = batch;
  p.total_rows = total_rows;
  p.chunks_per_seq = (int32_t)(((int64_t)max_pages * c.num_kv_heads + kHeadsPerBlock - 1) / kHeadsPerBlock);
  p.gk = c.k_global_scale;
  p.gv = c.v_global_scale;
  p.sk = k_ws_scale;
  p.sv = v_ws_scale;
  p.rsk = 1.0f / k_ws_scale;  // host IEEE division: RN(1 / s_ws)
  p.rsv = 1.0f / v_ws_scale;
  p.sk_fast = k_ws_scale >= 0x1p-100f && k_ws_scale <= 0x1p+100f;
  p.sv_fast = v_ws_scale >= 0x1p-100f && v_ws_scale <= 0x1p+100f;
  p.ws_k = ws_k;
  p.ws_v = ws_v;
  p.status = device_status;
  const int64_t units = (int64_t)batch * p.chunks_per_seq;
  int64_t blocks = units;  // one unit per block: the block scheduler overlaps them
  if (blocks > (1LL << 30)) blocks = 1LL << 30;
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
