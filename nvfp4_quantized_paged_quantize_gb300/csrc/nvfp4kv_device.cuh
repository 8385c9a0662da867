// nvfp4kv_device.cuh -- device-side building blocks of the NVFP4 paged KV cache
// (sm_103a): format conversions through the hardware cvt instructions, mbarrier
// set-up, and bounded waits.
//
// Format ("nvfp4-kv-cache-memory-wall", section 2; "NVFP4: breaking the memory
// wall", technical breakdown): E2M1 data (+-{0,0.5,1,1.5,2,3,4,6}), one E4M3
// scale per 16 consecutive values, one FP32 global scale per tensor.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "nvfp4kv.h"

namespace nvfp4kv {

constexpr int kHeadDim = 128;                          // supported head_dim
constexpr int kPage = 16;                              // tokens per page
constexpr int kBlock = 16;                             // values per E4M3 block scale
constexpr int kRowBytes = kHeadDim / 2;                // 64: packed E2M1 of one (token, head)
constexpr int kRowScales = kHeadDim / kBlock;          // 8: E4M3 scales of one (token, head)
constexpr int kPageDataBytes = kPage * kRowBytes;      // 1024: one head's page of data
constexpr int kPageScaleBytes = kPage * kRowScales;    // 128: one head's page of scales
constexpr int kDevErrTimeout = 8;                      // a bounded wait gave up

// One page-head (16 tokens of one KV head) of the pool: K data, K scales,
// V data, V scales, contiguous; the page-heads of a page follow one another.
// K data is token-major: 16 rows of 64 bytes, value 2k of a row in the low
// nibble of its byte k.  V data is stored by token pair: 8 rows of 128
// bytes, byte d of row p holding dimension d of token 2p (low nibble) and of
// token 2p + 1 (high nibble) -- the decode's P.V product contracts over
// tokens, and its f16 operands pair two tokens of one dimension, which one
// E2M1 conversion of such a byte gives directly.  K scales are token-major
// (the 8 scales of a token row together), V scales block-major (the 16
// tokens' scales of one 16-value block together): the decode reads K scales
// by token and V scales by token pair within a block.
constexpr int kOffKData = 0;
constexpr int kOffKScale = kPageDataBytes;                        // 1024
constexpr int kOffVData = kPageDataBytes + kPageScaleBytes;       // 1152
constexpr int kOffVScale = 2 * kPageDataBytes + kPageScaleBytes;  // 2176
constexpr int kPageHeadBytes = 2 * (kPageDataBytes + kPageScaleBytes);  // 2304
static_assert(kPageHeadBytes == NVFP4KV_PAGE_HEAD_BYTES, "page-head size");
// The MXFP4 variant's page-head: 4 E8M0 scale bytes per row.
constexpr int kMxRowScales = kHeadDim / 32;                       // 4
constexpr int kMxOffKScale = kPageDataBytes;                      // 1024
constexpr int kMxOffVData = kPageDataBytes + kPage * kMxRowScales;  // 1088
constexpr int kMxOffVScale = 2 * kPageDataBytes + kPage * kMxRowScales;  // 2112
constexpr int kMxPageHeadBytes = 2 * (kPageDataBytes + kPage * kMxRowScales);  // 2176
static_assert(kMxPageHeadBytes == NVFP4KV_MXFP4_PAGE_HEAD_BYTES, "MXFP4 page-head size");

constexpr int kVPairBytes = 2 * kRowBytes;  // 128: one token pair of V data

// Byte offset, within a page-head, of the scale of block j of token row r.
__host__ __device__ constexpr int k_scale_offset(int r, int j) { return kOffKScale + r * kRowScales + j; }
__host__ __device__ constexpr int v_scale_offset(int r, int j) { return kOffVScale + j * kPage + r; }
__host__ __device__ constexpr int mx_k_scale_offset(int r, int j) { return kMxOffKScale + r * kMxRowScales + j; }
__host__ __device__ constexpr int mx_v_scale_offset(int r, int j) { return kMxOffVScale + j * kPage + r; }

// ---------------------------------------------------------------------------
// E2M1 / E4M3 conversions (round to nearest even, saturating, as the
// satfinite cvt forms do).
// ---------------------------------------------------------------------------

// Two fp32 -> one byte of two E2M1 codes; `lo` goes to the low nibble.
__device__ __forceinline__ uint32_t e2m1x2_from_f32(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// One non-negative fp32 -> E4M3 byte.
__device__ __forceinline__ uint32_t e4m3_from_f32(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;
}

// Two E4M3 bytes (low byte -> low half) -> f16x2.  Exact: every E4M3 value is
// an f16 normal number.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("{ .reg .b16 h; cvt.u16.u32 h, %1; cvt.rn.f16x2.e4m3x2 %0, h; }" : "=r"(r) : "r"(two_bytes));
  return r;
}

// One E4M3 byte -> fp32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  uint32_t h2 = e4m3x2_to_f16x2(byte & 0xFFu);
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Byte K of w (two E2M1 codes, element 2i in the low nibble) -> f16x2 with the
// low nibble in the low half.  Exact: every E2M1 value is an f16 number.
template <int K>
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t w) {
  uint32_t r;
  if constexpr (K == 0)
    asm("{ .reg .b8 a, b, c, d; mov.b32 {a, b, c, d}, %1; cvt.rn.f16x2.e2m1x2 %0, a; }" : "=r"(r) : "r"(w));
  else if constexpr (K == 1)
    asm("{ .reg .b8 a, b, c, d; mov.b32 {a, b, c, d}, %1; cvt.rn.f16x2.e2m1x2 %0, b; }" : "=r"(r) : "r"(w));
  else if constexpr (K == 2)
    asm("{ .reg .b8 a, b, c, d; mov.b32 {a, b, c, d}, %1; cvt.rn.f16x2.e2m1x2 %0, c; }" : "=r"(r) : "r"(w));
  else
    asm("{ .reg .b8 a, b, c, d; mov.b32 {a, b, c, d}, %1; cvt.rn.f16x2.e2m1x2 %0, d; }" : "=r"(r) : "r"(w));
  return r;
}

// f16x2 (low half first) -> two E4M3 bytes (low half -> low byte).
__device__ __forceinline__ uint32_t e4m3x2_from_f16x2(uint32_t h2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
  return r;
}

// Two fp32 -> two E4M3 bytes; `lo` goes to the low byte.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Correctly rounded a / b from r = RN(1 / b): q0 = RN(a r), then Markstein's
// correction RN(q0 + r RN(a - b q0)) (two FMAs).  Valid while b, 1 / b and
// the quotient stay well inside the normal range; the caller checks.
__device__ __forceinline__ float div_markstein(float a, float b, float r) {
  const float q0 = __fmul_rn(a, r);
  const float rem = __fmaf_rn(-q0, b, a);
  return __fmaf_rn(rem, r, q0);
}

// ---------------------------------------------------------------------------
// V data by token pair
// ---------------------------------------------------------------------------

// Eight E2M1 codes of token 2p (e: value i in nibble i) and the same eight
// values of token 2p + 1 (o) -> the 8 bytes of the pair row, in value order
// (byte i: value i of e in the low nibble, of o in the high one).
__device__ __forceinline__ uint2 v_pair_bytes(uint32_t e, uint32_t o) {
  const uint32_t ev = (e & 0x0F0F0F0Fu) | ((o << 4) & 0xF0F0F0F0u);         // byte k: values 2k
  const uint32_t od = ((e >> 4) & 0x0F0F0F0Fu) | (o & 0xF0F0F0F0u);         // byte k: values 2k + 1
  return make_uint2(__byte_perm(ev, od, 0x5140), __byte_perm(ev, od, 0x7362));
}

// Store one 16-value block (codes lo: values 0-7, hi: 8-15) of both tokens of
// a pair (e: token 2p, o: token 2p + 1) at block j of pair row p of V data.
__device__ __forceinline__ void v_store_block_pair(uint8_t* vdata, int p, int j, uint32_t elo, uint32_t ehi,
                                                   uint32_t olo, uint32_t ohi) {
  const uint2 a = v_pair_bytes(elo, olo), b = v_pair_bytes(ehi, ohi);
  reinterpret_cast<uint4*>(vdata + p * kVPairBytes)[j] = make_uint4(a.x, a.y, b.x, b.y);
}

// Store one 16-value block of token row r alone: its nibbles of the 16 bytes,
// leaving the other token's (which another thread may be writing in the same
// launch) untouched.  Each word gets XORed with the difference between the
// codes it holds and the new ones, restricted to this token's nibbles, so
// concurrent updates of the two tokens of a pair commute.
__device__ __forceinline__ void v_store_block_one(uint8_t* vdata, int r, int j, uint32_t lo, uint32_t hi) {
  const bool odd = r & 1;
  const uint2 a = odd ? v_pair_bytes(0u, lo) : v_pair_bytes(lo, 0u);
  const uint2 b = odd ? v_pair_bytes(0u, hi) : v_pair_bytes(hi, 0u);
  const uint32_t mask = odd ? 0xF0F0F0F0u : 0x0F0F0F0Fu;
  uint32_t* w = reinterpret_cast<uint32_t*>(vdata + (r >> 1) * kVPairBytes + 16 * j);
  const uint4 old = __ldcg(reinterpret_cast<const uint4*>(w));
  const uint32_t nw[4] = {a.x, a.y, b.x, b.y}, ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t d = (nw[k] ^ ow[k]) & mask;
    if (d) atomicXor(w + k, d);
  }
}

// ---------------------------------------------------------------------------
// shared memory and mbarriers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the asynchronous proxy (the
// cp.async arrivals).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait until the mbarrier phase with the given parity has completed.  Gives up
// after about `limit_ns` of wall time and returns false (the caller records a
// device error and stops using the stage).
// Each try_wait may suspend the thread (up to the hinted 1 ms) until the phase
// completes, so a warp waiting for data sleeps instead of spinning.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = 1000000000ull) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(done) : "r"(bar), "r"(parity), "r"(1000000u) : "memory");
  if (done) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(done) : "r"(bar), "r"(parity), "r"(1000000u) : "memory");
    if (done) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void flag_error(int32_t* status, int bit) {
  if (status != nullptr) atomicOr(status, bit);
}

}  // namespace nvfp4kv
