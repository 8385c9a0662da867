// quantize_append.cu -- NVFP4 quantize-on-append of new K/V tokens into the
// paged cache ("nvfp4-kv-cache-memory-wall", section 3: new K/V are quantised
// to NVFP4 on the way into the cache; section 2: two-level scaling).
//
// One lane quantises one 16-value block (two 16-byte loads).  Per step a warp
// takes two (token, KV head) rows of K (lanes 0-7 and 8-15) and the two
// tokens of a token pair of one KV head of V (lanes 16-23: token 2q, lanes
// 24-31: token 2q + 1), so the per-block work (amax, the scale's division,
// the reciprocal) is done once per block.  Per block:
//   amax = max |x|                       (exact; inputs are bf16)
//   sb   = E4M3(amax / (6 g))            (correctly rounded quotient, RNE, saturating)
//   den  = E4M3val(sb) * g
//   code = E2M1(x / den)                 (correctly rounded quotient, RNE, saturating)
// A block with den == 0 stores signed zeros.  A token's codes and scales go
// to slot slot_mapping[token]: row slot % 16 of the page-head (slot / 16,
// head).  V data is stored by token pair (byte d of pair row p: dimension d of
// tokens 2p and 2p + 1): when the two tokens of a step land in the two rows
// of one pair row (the usual case: consecutive slots from an even one), one
// lane writes both tokens' bytes; otherwise each token's nibbles are merged
// into their bytes with atomic XORs.  HBM-bound: 2 B read and 9/16 B
// written per value.
#include "fp8_quotient.cuh"
#include "nvfp4kv_device.cuh"
#include "nvfp4kv_launch.h"

namespace nvfp4kv {
namespace {

struct QuantParams {
  const uint16_t* k;
  const uint16_t* v;
  const int64_t* slots;
  int32_t rows;  // num_tokens * num_kv_heads (< 2^31, checked on the host)
  int32_t ntok;  // num_tokens
  int32_t hkv;
  int64_t capacity;  // num_pages * page_size
  uint8_t* pages;  // [num_pages][hkv][kPageHeadBytes]
  float gk, gv;
  int32_t* status;
  // FP8 workspace rows written in the same pass (the fused prefill / extend write)
  const int64_t* ws_rows;
  int64_t ws_total_rows;
  uint8_t* ws_k;
  uint8_t* ws_v;
  float sk, sv, rsk, rsv;
  bool sk_fast, sv_fast, ws_unit;
};

constexpr int kThreads = 256;
constexpr int kRowsPerWarp = 2;  // (token, head) rows of K and of V per warp and step

// The (token, KV head) a lane quantises, walked without a division per step:
// K lanes walk the rows r = token * hkv + head, V lanes the token pairs
// u = q * hkv + head (their token is 2q or 2q + 1), both by a fixed stride.
struct RowWalk {
  int32_t major;  // K: token; V: token pair q
  int32_t head;
  int32_t dmajor, dhead;  // the stride as (major, head) steps
  int32_t hkv;

  __device__ __forceinline__ void init(int32_t start, int32_t stride, int32_t h) {
    hkv = h;
    major = start / h;
    head = start - major * h;
    dmajor = stride / h;
    dhead = stride - dmajor * h;
  }
  __device__ __forceinline__ void next() {
    major += dmajor;
    head += dhead;
    if (head >= hkv) {
      head -= hkv;
      ++major;
    }
  }
};

__device__ __forceinline__ void unpack_bf16x8(const uint4& x, float* f) {
  f[0] = bf16_to_f32(x.x & 0xFFFFu); f[1] = bf16_to_f32(x.x >> 16);
  f[2] = bf16_to_f32(x.y & 0xFFFFu); f[3] = bf16_to_f32(x.y >> 16);
  f[4] = bf16_to_f32(x.z & 0xFFFFu); f[5] = bf16_to_f32(x.z >> 16);
  f[6] = bf16_to_f32(x.w & 0xFFFFu); f[7] = bf16_to_f32(x.w >> 16);
}

// kWs: also write each row's FP8 workspace row, E4M3(fp32(x) / s_ws), at
// ws_rows[token] (< 0: none) from the same registers.
template <bool kWs>
__global__ void __launch_bounds__(kThreads) quantize_append_kernel(QuantParams p) {
  // a decode launched behind this append (nvfp4kv_append_decode_attention) may
  // start its set-up now; it waits for this grid before reading any page
  asm volatile("griddepcontrol.launch_dependents;");
  const int lane = threadIdx.x & 31;
  const int tensor = lane >> 4;  // 0: K, 1: V
  const int sub = lane & 7;      // block j = sub of the row: values [16 j, 16 j + 16)
  const int which = (lane >> 3) & 1;  // first or second row of the step
  const uint16_t* src = tensor ? p.v : p.k;
  const float g = tensor ? p.gv : p.gk;
  const float t6 = __fmul_rn(6.0f, g);  // the block amax maps onto E2M1's 6
  const float r6 = __frcp_rn(t6);
  const bool t6_ok = t6 >= 0x1p-100f && t6 <= 0x1p+100f;  // t6 and 1/t6 well inside the normal range
  const int warp = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  const int nwarps = (int)((gridDim.x * (unsigned)blockDim.x) >> 5);
  // steps cover the K rows and the V token pairs: (ntok rounded up to even) * hkv,
  // an even count, so the two halves of a warp run the same number of steps
  const int64_t steps_end = (int64_t)(p.ntok + (p.ntok & 1)) * p.hkv;

  // software pipeline: the next step's row (two 16-byte loads, its slot and,
  // for V, the slot of the pair's other token) is in flight while this step's
  // block is quantised
  const int64_t stride = (int64_t)nwarps * kRowsPerWarp;
  int64_t r = (int64_t)warp * kRowsPerWarp + which;
  RowWalk walk;
  if (tensor == 0)
    walk.init(warp * kRowsPerWarp + which, nwarps * kRowsPerWarp, p.hkv);
  else
    walk.init(warp, nwarps, p.hkv);
  // the lane's token at the walk's position (V: 2q + which)
  auto token_of = [&](const RowWalk& w) { return tensor == 0 ? w.major : 2 * w.major + which; };
  uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
  int64_t slot = -1, pslot = -1, wrow = -1;
  int tok = token_of(walk), head = walk.head;
  if (r < steps_end && tok < p.ntok) {
    const uint4* xs = reinterpret_cast<const uint4*>(src + ((int64_t)tok * p.hkv + head) * kHeadDim) + 2 * sub;
    xa = __ldg(xs);
    xb = __ldg(xs + 1);
    slot = __ldg(p.slots + tok);
    if (tensor && (tok ^ 1) < p.ntok) pslot = __ldg(p.slots + (tok ^ 1));
    if constexpr (kWs) wrow = __ldg(p.ws_rows + tok);
  }
  for (; r < steps_end; r += stride) {
    const int64_t rn = r + stride;
    const int ctok = tok, h = head;
    walk.next();
    tok = token_of(walk);
    head = walk.head;
    uint4 na = make_uint4(0, 0, 0, 0), nb = na;
    int64_t nslot = -1, npslot = -1, nwrow = -1;
    if (rn < steps_end && tok < p.ntok) {
      const uint4* xs = reinterpret_cast<const uint4*>(src + ((int64_t)tok * p.hkv + head) * kHeadDim) + 2 * sub;
      na = __ldg(xs);
      nb = __ldg(xs + 1);
      nslot = __ldg(p.slots + tok);
      if (tensor && (tok ^ 1) < p.ntok) npslot = __ldg(p.slots + (tok ^ 1));
      if constexpr (kWs) nwrow = __ldg(p.ws_rows + tok);
    }
    const uint4 ca = xa, cb = xb;
    const bool cvalid = ctok < p.ntok;
    const int64_t cslot = cvalid ? slot : -1, cpslot = pslot;
    xa = na;
    xb = nb;
    slot = nslot;
    pslot = npslot;
    if constexpr (kWs) {
      const int64_t cw = cvalid ? wrow : -1;
      wrow = nwrow;
      if (cw >= p.ws_total_rows) {
        flag_error(p.status, NVFP4KV_DEVERR_ROW);
      } else if (cw >= 0) {
        // this lane's 16 values -> 16 E4M3 bytes of the workspace row
        const uint32_t w[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
        const float s = tensor ? p.sv : p.sk, rs = tensor ? p.rsv : p.rsk;
        const bool fast = tensor ? p.sv_fast : p.sk_fast;
        uint32_t e[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          e[i] = e4m3x2_from_quotients(bf16_to_f32(w[i] & 0xFFFFu), bf16_to_f32(w[i] >> 16), s, rs, fast, p.ws_unit);
        uint8_t* ws = tensor ? p.ws_v : p.ws_k;
        reinterpret_cast<uint4*>(ws + (cw * p.hkv + h) * kHeadDim)[sub] =
            make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
      }
    }
    float f[16];
    unpack_bf16x8(ca, f);
    unpack_bf16x8(cb, f + 8);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
    // the block scale's quotient: Markstein while the first product stays far
    // from overflow (a quotient below 2^-11 encodes as 0 either way)
    const float sq = (t6_ok && __fmul_rn(amax, r6) < 0x1p+64f) ? div_markstein(amax, t6, r6) : __fdiv_rn(amax, t6);
    const uint32_t sb = e4m3_from_f32(sq);
    const float den = __fmul_rn(e4m3_to_f32(sb), g);
    uint32_t lo = 0, hi = 0;
    if (den == 0.0f) {
      // signed zeros: code 8 for negative inputs
#pragma unroll
      for (int i = 0; i < 8; ++i) lo |= (__float_as_uint(f[i]) >> 31) << (4 * i + 3);
#pragma unroll
      for (int i = 0; i < 8; ++i) hi |= (__float_as_uint(f[8 + i]) >> 31) << (4 * i + 3);
    } else {
      const float rcp = __frcp_rn(den);
      float y[16];
      if (den >= 0x1p-100f && den <= 0x1p+100f && __fmul_rn(amax, rcp) < 0x1p+64f) {
        // a quotient that rounds to zero can come out as +0 for negative x;
        // the sign of x / den is the sign of x (den > 0)
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = copysignf(div_markstein(f[i], den, rcp), f[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = __fdiv_rn(f[i], den);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) lo |= e2m1x2_from_f32(y[2 * k], y[2 * k + 1]) << (8 * k);
#pragma unroll
      for (int k = 0; k < 4; ++k) hi |= e2m1x2_from_f32(y[8 + 2 * k], y[8 + 2 * k + 1]) << (8 * k);
    }
    // V: the other token of the pair (lane ^ 8 holds the same block of it);
    // every lane takes part in the exchange
    const uint32_t plo = __shfl_xor_sync(0xFFFFFFFFu, lo, 8);
    const uint32_t phi = __shfl_xor_sync(0xFFFFFFFFu, hi, 8);
    if (cslot < 0) continue;  // padding, or no such row
    if (cslot >= p.capacity) {
      flag_error(p.status, NVFP4KV_DEVERR_SLOT);
      continue;
    }
    uint8_t* ph = p.pages + ((cslot >> 4) * p.hkv + h) * kPageHeadBytes;  // the slot's page-head
    const int rin = (int)(cslot & (kPage - 1));                            // its row there
    if (tensor == 0) {
      reinterpret_cast<uint2*>(ph + kOffKData + rin * kRowBytes)[sub] = make_uint2(lo, hi);
      ph[k_scale_offset(rin, sub)] = (uint8_t)sb;
    } else {
      // the step's two tokens fill one pair row when their slots are 2m and 2m + 1
      const int64_t se = which ? cpslot : cslot, so = which ? cslot : cpslot;
      const bool paired = (se & 1) == 0 && so == se + 1;
      if (paired) {
        if (which == 0) v_store_block_pair(ph + kOffVData, rin >> 1, sub, lo, hi, plo, phi);
      } else {
        v_store_block_one(ph + kOffVData, rin, sub, lo, hi);
      }
      ph[v_scale_offset(rin, sub)] = (uint8_t)sb;
    }
  }
}

}  // namespace

namespace {

template <bool kWs>
cudaError_t launch_quantize(QuantParams& p, int num_sms, cudaStream_t stream) {
  const int warps_needed = (int)(((int64_t)(p.ntok + (p.ntok & 1)) * p.hkv) / kRowsPerWarp);
  const int warps_per_block = kThreads / 32;
  int blocks = (warps_needed + warps_per_block - 1) / warps_per_block;
  // a persistent grid: as many blocks as fit on the device at once (more
  // blocks, each doing less, measured slower)
  static const int per_sm = [] {  // once per instantiation, thread-safely
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_append_kernel<kWs>, kThreads, 0) != cudaSuccess ||
        n < 1)
      n = 1;
    return n;
  }();
  const int max_blocks = num_sms * per_sm;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  quantize_append_kernel<kWs><<<blocks, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

QuantParams cache_params(const nvfp4kv_cache& c, const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                         int64_t num_tokens, int32_t* device_status) {
  QuantParams p = {};
  p.k = k;
  p.v = v;
  p.slots = slot_mapping;
  p.rows = (int32_t)(num_tokens * c.num_kv_heads);
  p.ntok = (int32_t)num_tokens;
  p.hkv = c.num_kv_heads;
  p.capacity = c.num_pages * (int64_t)c.page_size;
  p.pages = c.pages;
  p.gk = c.k_global_scale;
  p.gv = c.v_global_scale;
  p.status = device_status;
  return p;
}

}  // namespace

cudaError_t launch_quantize_append(const nvfp4kv_cache& c, const uint16_t* k, const uint16_t* v,
                                   const int64_t* slot_mapping, int64_t num_tokens,
                                   int32_t* device_status, int num_sms, cudaStream_t stream) {
  QuantParams p = cache_params(c, k, v, slot_mapping, num_tokens, device_status);
  return launch_quantize<false>(p, num_sms, stream);
}

cudaError_t launch_quantize_append_fp8(const nvfp4kv_cache& c, const uint16_t* k, const uint16_t* v,
                                       const int64_t* slot_mapping, int64_t num_tokens, const int64_t* ws_rows,
                                       int64_t total_rows, float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                                       uint8_t* ws_v, int32_t* device_status, int num_sms, cudaStream_t stream) {
  QuantParams p = cache_params(c, k, v, slot_mapping, num_tokens, device_status);
  p.ws_rows = ws_rows;
  p.ws_total_rows = total_rows;
  p.ws_k = ws_k;
  p.ws_v = ws_v;
  p.sk = k_ws_scale;
  p.sv = v_ws_scale;
  p.rsk = 1.0f / k_ws_scale;  // host IEEE division: RN(1 / s_ws)
  p.rsv = 1.0f / v_ws_scale;
  p.sk_fast = k_ws_scale >= 0x1p-100f && k_ws_scale <= 0x1p+100f;
  p.sv_fast = v_ws_scale >= 0x1p-100f && v_ws_scale <= 0x1p+100f;
  p.ws_unit = k_ws_scale == 1.0f && v_ws_scale == 1.0f;
  return launch_quantize<true>(p, num_sms, stream);
}

}  // namespace nvfp4kv
