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

// ------------------------------------------------------------ scale atoms
// The block-scaled MMA reads its E8M0 scale factors from tensor memory, where
// tcgen05.cp (.32x128b.warpx4) puts them from 512-byte shared-memory atoms:
// 32 rows of 16 bytes, byte 4j + q of row r holding the scale of row (or
// output column) 32j + r of a 128-row block for the q-th 32-element block of
// a 128-deep k-block.  The GEMMs fetch whole atoms by TMA, so the scales they
// read are kept in HBM in atom order (GEMM scratch, rebuilt from the
// row-major tables):
//  * activations [R][K] in expert-sorted rows: every expert starts a fresh
//    128-row block.  Row r of expert e is scale row
//      s = r - offsets[e] + 128 * (ceil(offsets[e] / 128) + e)
//    (segments cannot overlap: s < offsets[e+1] + 128 (e + 1) - 1 <= the next
//    expert's first scale row), and (block s / 128, k-block kb) is atom
//    (s / 128) * (K / 128) + kb; (ceil(R / 128) + E) * K / 128 atoms.
//  * weights, per expert, column tile and k-block two atoms (tile columns
//    0-127 and 128-191): the up-projection's tiles are 96 rows of W1 then the
//    same 96 rows of W3 (ceil(h / 96) tiles, K = d), the down-projection's
//    192 rows of W2 (ceil(d / 192) tiles, K = h); columns past N hold 0.
constexpr int kAtomBytes = 512;
constexpr int kUpCols = 96, kDownCols = 192;

__host__ __device__ inline long long act_atom_blocks(long long R, int E) { return (R + 127) / 128 + E; }
__host__ __device__ inline long long act_atom_bytes(long long R, int E, int K) {
  return act_atom_blocks(R, E) * (K / 128) * kAtomBytes;
}
__host__ __device__ inline int up_tiles(int h) { return (h + kUpCols - 1) / kUpCols; }
__host__ __device__ inline int down_tiles(int d) { return (d + kDownCols - 1) / kDownCols; }
// weight atoms: the up-projection's, then the down-projection's
__host__ __device__ inline long long up_atom_count(int E, int d, int h) {
  return (long long)E * up_tiles(h) * (d / 128) * 2;
}
__host__ __device__ inline long long weight_atom_bytes(int E, int d, int h) {
  return (up_atom_count(E, d, h) + (long long)E * down_tiles(d) * (h / 128) * 2) * kAtomBytes;
}
// first 128-row block of expert e's scale rows
__host__ __device__ inline int act_block0(int offset_e, int e) { return (offset_e + 127) / 128 + e; }

}  // namespace mx
}  // namespace moe
