// MXFP8 block arithmetic shared by the quantisers and the block-scaled GEMM's
// epilogue: E4M3 codes with one E8M0 scale per 32 elements.
//
// Scale rule (the reading used throughout): e = the smallest integer with
// amax <= 448 * 2^e, clamped to [-127, 127], stored as the byte e + 127 (an
// all-zero block gets e = -127); codes = RNE_E4M3(v * 2^-e), saturating.  It is
// exact: frexp gives amax = F * 2^q with F in [0.5, 1) and 448 = 0.875 * 2^9,
// so e = q - 9 when F <= 0.875 and q - 8 otherwise.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {
namespace mx {

__device__ __forceinline__ int block_exponent(float amax) {
  if (!(amax > 0.f)) return -127;
  int q;
  const float F = frexpf(amax, &q);
  const int e = (F <= 0.875f) ? q - 9 : q - 8;
  return max(-127, min(127, e));
}

// 2^-e as an exact fp32 (e in [-127, 127]; 2^-127 is the subnormal 0x00400000)
__device__ __forceinline__ float inv_scale(int e) {
  return e <= 126 ? __int_as_float((127 - e) << 23) : __int_as_float(0x00400000);
}

// four fp32 values -> four E4M3 codes (RNE, saturating), first value in the low byte
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

}  // namespace mx
}  // namespace moe
