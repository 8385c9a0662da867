// quantize_variants.cu -- the quantize-on-append of the format variants the
// pages compare with NVFP4:
//  - stochastic rounding of the E2M1 codes ("NVFP4: breaking the memory wall",
//    quantisation techniques: 2.3 -> 2 with 70 %, -> 3 with 30 %), one input
//    random byte per value, read as the uniform (r + 0.5) / 256;
//  - a Hadamard rotation of each 128-value head vector before the NVFP4 block
//    quantisation (same page: an orthogonal transform spreads an outlier):
//    the orthonormal Walsh-Hadamard transform as seven binary32 butterfly
//    passes (h = 1, 2, 4, ..., 64) and one multiplication by RN(1 / sqrt(128));
//  - MXFP4 ("NVIDIA NVFP4: LLM memory doubled, inference 3x", figure 6; "NVFP4:
//    breaking the memory wall", technical breakdown): blocks of 32 values with
//    a power-of-two scale, an E8M0 byte e + 127 with e = floor(log2 amax) - 2,
//    elements E2M1(x * 2^-e); its scale pool holds 4 bytes per row.
// SR and Hadamard write the NVFP4 page-heads; MXFP4 writes its own page-heads
// (the same 64 data bytes per row, 4 scale bytes per row).
//
// Eight lanes own one (token, head) row of K or of V, 16 values each; a warp
// takes the rows of one token pair (2q, 2q + 1) of one KV head: K of token 2q,
// K of token 2q + 1, V of token 2q, V of token 2q + 1, so that V's token-pair
// bytes can be written whole when the two slots are 2m and 2m + 1.  Block
// scales and quotients are correctly rounded (a reciprocal and one Markstein
// correction, IEEE division outside its range), as in the NVFP4 append.
#include "nvfp4kv_device.cuh"
#include "nvfp4kv_launch.h"

namespace nvfp4kv {
namespace {

struct VariantParams {
  const uint16_t* k;
  const uint16_t* v;
  const int64_t* slots;
  const uint8_t* rand_k;  // stochastic rounding: one byte per value, [tokens][hkv][128]
  const uint8_t* rand_v;
  int64_t units;  // token pairs * hkv: one warp each
  int64_t ntok;
  int32_t hkv;
  int64_t capacity;
  uint8_t* pages;  // [num_pages][hkv][page-head bytes of the variant's layout]
  float gk, gv;
  int32_t* status;
};

constexpr int kThreads = 256;

// E2M1 code of |y| < 6 (grid neighbours a <= |y| < b) rounded up with
// probability (|y| - a) / (b - a): up iff 2 r + 1 < 512 (|y| - a) / (b - a).
// The grid's segments [0, 2), [2, 4), [4, 6) have gaps 0.5, 1, 2: with t =
// (|y| - segment start) / gap, a is the segment start plus floor(t) gaps and
// the scaled fraction is 512 (t - floor(t)), every step exact.  No branches.
__device__ __forceinline__ uint32_t e2m1_code_sr(float y, uint32_t r) {
  const float m = fabsf(y);
  const bool s1 = m >= 2.0f, s2 = m >= 4.0f;
  const float inv_gap = s2 ? 0.5f : (s1 ? 1.0f : 2.0f);
  const float start = s2 ? 4.0f : (s1 ? 2.0f : 0.0f);
  const uint32_t c0 = s2 ? 6u : (s1 ? 4u : 0u);
  const float t = (m - start) * inv_gap;
  const float k = floorf(t);
  uint32_t c = c0 + (uint32_t)k + (((float)(2 * r + 1) < (t - k) * 512.0f) ? 1u : 0u);
  c = m >= 6.0f ? 7u : c;
  return c | (__float_as_uint(y) >> 31 << 3);
}

template <int kVariant>
__global__ void __launch_bounds__(kThreads) quantize_variant_kernel(VariantParams p) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;  // values [16 sub, 16 sub + 16) of the row
  const int tensor = lane >> 4, which = (lane >> 3) & 1;
  // every lane stays to the end (the rotation and MXFP4 exchange values across
  // the row's lanes with full-warp shuffles, and V's two tokens meet); lanes
  // without a row work on row 0 and store nothing
  const int64_t unit = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t q = unit / p.hkv;
  const int h0 = (int)(unit - q * p.hkv);
  const int64_t token0 = 2 * q + which;
  const bool live = unit < p.units && token0 < p.ntok;
  const int64_t token = live ? token0 : 0;
  const int h = live ? h0 : 0;
  const int64_t th = token * p.hkv + h;  // the input row
  const uint16_t* src = (tensor ? p.v : p.k) + th * kHeadDim + 16 * sub;
  const uint4 xa = __ldg(reinterpret_cast<const uint4*>(src));
  const uint4 xb = __ldg(reinterpret_cast<const uint4*>(src) + 1);
  const uint32_t w[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
  float f[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = bf16_to_f32(w[i] & 0xFFFFu);
    f[2 * i + 1] = bf16_to_f32(w[i] >> 16);
  }
  if constexpr (kVariant == NVFP4KV_VARIANT_HADAMARD) {
    // passes h = 1, 2, 4, 8 inside the lane, then 16, 32, 64 across the row's lanes
#pragma unroll
    for (int hh = 1; hh < 16; hh *= 2)
#pragma unroll
      for (int i = 0; i < 16; i += 2 * hh)
#pragma unroll
        for (int j = i; j < i + hh; ++j) {
          const float a = f[j], b = f[j + hh];
          f[j] = a + b;
          f[j + hh] = a - b;
        }
#pragma unroll
    for (int x = 1; x < 8; x *= 2) {
      const bool upper = (sub & x) != 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float o = __shfl_xor_sync(0xFFFFFFFFu, f[i], x);
        f[i] = upper ? o - f[i] : f[i] + o;  // lower: a + b; upper: a - b (a from the lower lane)
      }
    }
    const float c = 0x1.6a09e6p-4f;  // RN(1 / sqrt(128)) = RN(sqrt(2)) / 16
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = __fmul_rn(f[i], c);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));

  uint32_t lo = 0, hi = 0, sbyte;
  if constexpr (kVariant == NVFP4KV_VARIANT_MXFP4) {
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));  // the block of 32 spans a lane pair
    int e = -127;
    if (amax > 0.0f) {
      const int be = (int)((__float_as_uint(amax) >> 23) & 0xFFu);  // 0 for subnormals: floor(log2) <= -127
      e = be == 0 ? -127 : be - 127 - 2;
      e = e < -127 ? -127 : (e > 127 ? 127 : e);
    }
    sbyte = (uint32_t)(e + 127);
    // 2^-e (e <= 125 since amax < 2^128, so 2^-e is a normal float): each
    // product rounds once, as the exact quotient x / 2^e does
    const float sc = __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      lo |= e2m1x2_from_f32(__fmul_rn(f[2 * k], sc), __fmul_rn(f[2 * k + 1], sc)) << (8 * k);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      hi |= e2m1x2_from_f32(__fmul_rn(f[8 + 2 * k], sc), __fmul_rn(f[8 + 2 * k + 1], sc)) << (8 * k);
  } else {
    const float g = tensor ? p.gv : p.gk;
    const float t6 = __fmul_rn(6.0f, g), r6 = __frcp_rn(t6);
    // Markstein while t6 and the first product stay well inside the normal range
    // (a quotient below 2^-11 encodes as 0 either way)
    const bool t6_ok = t6 >= 0x1p-100f && t6 <= 0x1p+100f && __fmul_rn(amax, r6) < 0x1p+64f;
    sbyte = e4m3_from_f32(t6_ok ? div_markstein(amax, t6, r6) : __fdiv_rn(amax, t6));
    const float den = __fmul_rn(e4m3_to_f32(sbyte), g);
    const float rcp = __frcp_rn(den);
    // the sign of x / den is the sign of x (den > 0): restored where a quotient
    // rounding to zero came out as +0
    const bool fast = den >= 0x1p-100f && den <= 0x1p+100f && __fmul_rn(amax, rcp) < 0x1p+64f;
    auto quot = [&](float x) { return fast ? copysignf(div_markstein(x, den, rcp), x) : __fdiv_rn(x, den); };
    if (den == 0.0f) {
#pragma unroll
      for (int i = 0; i < 8; ++i) lo |= (__float_as_uint(f[i]) >> 31) << (4 * i + 3);
#pragma unroll
      for (int i = 0; i < 8; ++i) hi |= (__float_as_uint(f[8 + i]) >> 31) << (4 * i + 3);
    } else if constexpr (kVariant == NVFP4KV_VARIANT_SR) {
      const uint8_t* rs = (tensor ? p.rand_v : p.rand_k) + th * kHeadDim + 16 * sub;
      const uint4 r4 = __ldg(reinterpret_cast<const uint4*>(rs));
      const uint32_t rw[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
        lo |= e2m1_code_sr(quot(f[i]), (rw[i >> 2] >> (8 * (i & 3))) & 0xFFu) << (4 * i);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        hi |= e2m1_code_sr(quot(f[8 + i]), (rw[2 + (i >> 2)] >> (8 * (i & 3))) & 0xFFu) << (4 * i);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        lo |= e2m1x2_from_f32(quot(f[2 * k]), quot(f[2 * k + 1])) << (8 * k);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        hi |= e2m1x2_from_f32(quot(f[8 + 2 * k]), quot(f[8 + 2 * k + 1])) << (8 * k);
    }
  }
  const int64_t slot = live ? __ldg(p.slots + token) : -1;
  // V: the other token of the pair (lane ^ 8 holds the same block of it)
  const uint32_t plo = __shfl_xor_sync(0xFFFFFFFFu, lo, 8);
  const uint32_t phi = __shfl_xor_sync(0xFFFFFFFFu, hi, 8);
  const int64_t pslot = __shfl_xor_sync(0xFFFFFFFFu, slot, 8);
  if (slot < 0) return;  // padding, or no row
  if (slot >= p.capacity) {
    if (sub == 0) flag_error(p.status, NVFP4KV_DEVERR_SLOT);
    return;
  }
  const int rin = (int)(slot & (kPage - 1));  // the slot's row in its page-head
  const int64_t se = which ? pslot : slot, so = which ? slot : pslot;
  const bool paired = (se & 1) == 0 && so == se + 1;  // the two tokens fill one V pair row
  const bool mx = kVariant == NVFP4KV_VARIANT_MXFP4;
  uint8_t* ph = p.pages + ((slot >> 4) * p.hkv + h) * (mx ? kMxPageHeadBytes : kPageHeadBytes);
  if (tensor == 0) {
    reinterpret_cast<uint2*>(ph + kOffKData + rin * kRowBytes)[sub] = make_uint2(lo, hi);
  } else {
    uint8_t* vdata = ph + (mx ? kMxOffVData : kOffVData);
    if (paired) {
      if (which == 0) v_store_block_pair(vdata, rin >> 1, sub, lo, hi, plo, phi);
    } else {
      v_store_block_one(vdata, rin, sub, lo, hi);
    }
  }
  if constexpr (kVariant == NVFP4KV_VARIANT_MXFP4) {
    if ((sub & 1) == 0) ph[tensor ? mx_v_scale_offset(rin, sub >> 1) : mx_k_scale_offset(rin, sub >> 1)] = (uint8_t)sbyte;
  } else {
    ph[tensor ? v_scale_offset(rin, sub) : k_scale_offset(rin, sub)] = (uint8_t)sbyte;
  }
}

}  // namespace

cudaError_t launch_quantize_variant(int variant, const nvfp4kv_cache& c, const uint16_t* k, const uint16_t* v,
                                    const int64_t* slot_mapping, int64_t num_tokens, const uint8_t* rand_k,
                                    const uint8_t* rand_v, int32_t* device_status, cudaStream_t stream) {
  VariantParams p;
  p.k = k;
  p.v = v;
  p.slots = slot_mapping;
  p.rand_k = rand_k;
  p.rand_v = rand_v;
  p.units = (num_tokens + 1) / 2 * c.num_kv_heads;
  p.ntok = num_tokens;
  p.hkv = c.num_kv_heads;
  p.capacity = c.num_pages * (int64_t)c.page_size;
  p.pages = c.pages;
  p.gk = c.k_global_scale;
  p.gv = c.v_global_scale;
  p.status = device_status;
  const int64_t blocks = (p.units * 32 + kThreads - 1) / kThreads;
  if (blocks == 0) return cudaSuccess;
  if (variant == NVFP4KV_VARIANT_SR)
    quantize_variant_kernel<NVFP4KV_VARIANT_SR><<<(unsigned)blocks, kThreads, 0, stream>>>(p);
  else if (variant == NVFP4KV_VARIANT_HADAMARD)
    quantize_variant_kernel<NVFP4KV_VARIANT_HADAMARD><<<(unsigned)blocks, kThreads, 0, stream>>>(p);
  else
    quantize_variant_kernel<NVFP4KV_VARIANT_MXFP4><<<(unsigned)blocks, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nvfp4kv
