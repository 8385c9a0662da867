// fp8_quotient.cuh -- FP8 E4M3 workspace bytes of fp32(a / s_ws), the last
// step of every workspace row ("nvfp4-kv-cache-memory-wall", section 3, item
// 2: the FP8 workspace of chunked prefill / extend).
#pragma once

#include "nvfp4kv_device.cuh"

namespace nvfp4kv {

// Two fp32 -> two E4M3 bytes of fp32(a / s), sign kept, saturating (`lo` to the
// low byte).  unit: s == 1, no division.  Otherwise the correctly rounded
// quotient from rs = RN(1 / s) with Markstein's correction while s is well
// inside the normal range (fast) and the first quotient stays below 2^64, and
// an IEEE division elsewhere; a zero quotient keeps the sign of a.
__device__ __forceinline__ uint32_t e4m3x2_from_quotients(float a0, float a1, float s, float rs, bool fast,
                                                          bool unit) {
  if (!unit) {
    const float q0 = __fmul_rn(a0, rs), q1 = __fmul_rn(a1, rs);
    if (fast && fabsf(q0) < 0x1p+64f && fabsf(q1) < 0x1p+64f) {
      a0 = copysignf(__fmaf_rn(__fmaf_rn(-q0, s, a0), rs, q0), a0);
      a1 = copysignf(__fmaf_rn(__fmaf_rn(-q1, s, a1), rs, q1), a1);
    } else {
      a0 = __fdiv_rn(a0, s);
      a1 = __fdiv_rn(a1, s);
    }
  }
  return e4m3x2_from_f32(a0, a1);
}

}  // namespace nvfp4kv
