// MXFP8 quantisation: E4M3 elements with one E8M0 scale per 32 consecutive
// elements along the GEMM reduction dimension.
//
// "OLMo-core 3：MoE 训练栈让专家池越大、吞吐不再越慢", section "一个低精度格式，同时压三
// 个地方": 8-bit E4M3 values share a power-of-two E8M0 scale per 32-element
// block, taken from the FP32 exponent bits; 448 is the largest E4M3 value and
// the block maximum must just fit; the scale is block-local (no scale
// all-reduce).  The page's list of the three scale steps did not survive; the
// reading implemented here: e = the smallest integer with amax <= 448 * 2^e,
// clamped to [-127, 127], scale byte = e + 127 (e = -127 for an all-zero
// block), codes = RNE_E4M3(v * 2^-e) with saturation (never reached); see
// mx_common.cuh for the exact exponent computation.
#include "common.cuh"
#include "mx_common.cuh"

namespace moe {
namespace {

using mx::block_exponent;
using mx::e4m3x4;
using mx::inv_scale;

// rows x K (row-major, K contiguous) -> codes rows x K and scales rows x K/32.
// One thread per 32-element block.
__global__ void quantize_rows_kernel(const uint16_t* __restrict__ src, long long nblocks, int K,
                                     uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
  pdl_enter();
  const long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (b >= nblocks) return;
  const uint16_t* p = src + b * 32;
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 w = ld_nc_v4(p + 8 * i);
    v[8 * i + 0] = bf16_lo(w.x); v[8 * i + 1] = bf16_hi(w.x);
    v[8 * i + 2] = bf16_lo(w.y); v[8 * i + 3] = bf16_hi(w.y);
    v[8 * i + 4] = bf16_lo(w.z); v[8 * i + 5] = bf16_hi(w.z);
    v[8 * i + 6] = bf16_lo(w.w); v[8 * i + 7] = bf16_hi(w.w);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int e = block_exponent(amax);
  const float inv = inv_scale(e);
  uint4 o[2];
  uint32_t* w = reinterpret_cast<uint32_t*>(o);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = e4m3x4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
  st_v4(q + b * 32, o[0]);
  st_v4(q + b * 32 + 16, o[1]);
  s[b] = (uint8_t)(e + 127);
}

// One weight column's 32-element block along K (values v, fp32) -> its 32
// codes at wq[e][n][32kb..] and its scale byte at ws[e][n][kb].
__device__ __forceinline__ void store_weight_block(const float (&v)[32], uint8_t* __restrict__ wq,
                                                   uint8_t* __restrict__ ws, int e, int n, int kb,
                                                   int K, int N) {
  float amax = 0.f;
#pragma unroll
  for (int r = 0; r < 32; ++r) amax = fmaxf(amax, fabsf(v[r]));
  const int ex = block_exponent(amax);
  const float inv = inv_scale(ex);
  uint4 o[2];
  uint32_t* w = reinterpret_cast<uint32_t*>(o);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = e4m3x4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
  uint8_t* dst = wq + ((size_t)e * N + n) * K + (size_t)kb * 32;
  st_v4(dst, o[0]);
  st_v4(dst + 16, o[1]);
  ws[((size_t)e * N + n) * (K / 32) + kb] = (uint8_t)(ex + 127);
}

// W[E][K][N] (bf16) -> Wq[E][N][K] codes and Ws[E][N][K/32] scales: blocks of
// 32 along K for every (e, n).  CTA = (32 K-rows, 128 columns); the slab is
// staged in shared memory and every thread quantises one column's block.
__global__ void __launch_bounds__(128)
quantize_weights_kernel(const uint16_t* __restrict__ W, int K, int N, uint8_t* __restrict__ wq,
                        uint8_t* __restrict__ ws) {
  pdl_enter();
  __shared__ uint16_t tile[32][128 + 8];
  const int e = blockIdx.z, kb = blockIdx.y, n0 = blockIdx.x * 128;
  const uint16_t* src = W + ((size_t)e * K + (size_t)kb * 32) * N + n0;
  const int t = threadIdx.x;
  // 32 rows x 128 columns: each thread loads 8 columns (16 bytes) of 4 rows
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = (t >> 4) + 8 * i, c = (t & 15) * 8;
    const uint4 v = ld_nc_v4(src + (size_t)r * N + c);
    *reinterpret_cast<uint4*>(&tile[r][c]) = v;
  }
  __syncthreads();
  float v[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) v[r] = __uint_as_float((uint32_t)tile[r][t] << 16);
  store_weight_block(v, wq, ws, e, n0 + t, kb, K, N);
}

// The same from fp32 master weights: one rounding, fp32 -> E4M3 (the scaled
// value v * 2^-e is exact in fp32 wherever it can round to a non-zero code).
// Row pitch 132 floats: 16-byte aligned rows, and a warp reading one column
// slot per row touches 32 different banks.
__global__ void __launch_bounds__(128)
quantize_weights_f32_kernel(const float* __restrict__ W, int K, int N, uint8_t* __restrict__ wq,
                            uint8_t* __restrict__ ws) {
  pdl_enter();
  __shared__ float tile[32][128 + 4];
  const int e = blockIdx.z, kb = blockIdx.y, n0 = blockIdx.x * 128;
  const float* src = W + ((size_t)e * K + (size_t)kb * 32) * N + n0;
  const int t = threadIdx.x;
  // 32 rows x 128 columns: each thread loads 4 columns (16 bytes) of 8 rows
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = (t >> 5) + 4 * i, c = (t & 31) * 4;
    *reinterpret_cast<uint4*>(&tile[r][c]) = ld_nc_v4(src + (size_t)r * N + c);
  }
  __syncthreads();
  float v[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) v[r] = tile[r][t];
  store_weight_block(v, wq, ws, e, n0 + t, kb, K, N);
}

// E4M3 code -> its value in fp32 (exact): sign, 4 exponent bits (bias 7), 3
// mantissa bits; exponent field 0 holds the subnormals m * 2^-9.  The two NaN
// codes (S.1111.111) never come out of the quantisers here.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t ex = (c >> 3) & 0xFu, m = c & 0x7u;
  const float mag = ex == 0 ? (float)m * 0.001953125f                      // m * 2^-9
                            : __uint_as_float(((ex + 120u) << 23) | (m << 20));
  return (c & 0x80u) ? -mag : mag;
}

// q[rows][K] codes + scale[rows][K/32] -> out[rows][K] bf16: value = code *
// 2^(byte - 127), exact in fp32, then rounded to bf16 (RNE; exact unless it
// falls into bf16's subnormal range).  One thread per 32-element block.
__global__ void dequantize_rows_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                                       long long nblocks, uint16_t* __restrict__ out) {
  pdl_enter();
  const long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (b >= nblocks) return;
  const uint4 c0 = ld_nc_v4(q + b * 32), c1 = ld_nc_v4(q + b * 32 + 16);
  const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const int ex = (int)__ldg(s + b) - 127;
  // 2^ex as an exact fp32 (2^-127 is the subnormal 0x00400000)
  const float scale = ex >= -126 ? __uint_as_float((uint32_t)(ex + 127) << 23) : __uint_as_float(0x00400000u);
  uint4 o[4];
  uint32_t* w = reinterpret_cast<uint32_t*>(o);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t word = cw[i >> 1], sh = (i & 1) * 16;
    w[i] = pack_bf16x2(e4m3_value((word >> sh) & 0xFFu) * scale,
                       e4m3_value((word >> (sh + 8)) & 0xFFu) * scale);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) st_v4(out + b * 32 + 8 * i, o[i]);
}

// Rowwise dispatch with quantisation: every token row is quantised once
// (blocks of 32 along d) and its codes and scales written to the k rows
// row_of_slot[t*k+j] of xq / xs; the bf16 row also goes to xp when given
// (the backward stays bf16).  One warp per token; 4 lanes share a block.
__global__ void __launch_bounds__(256)
dispatch_mxfp8_kernel(const uint16_t* __restrict__ x, int T, int d, int k,
                      const int32_t* __restrict__ row_of_slot, uint8_t* __restrict__ xq,
                      uint8_t* __restrict__ xs, uint16_t* __restrict__ xp) {
  pdl_enter();
  const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int rows[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) rows[j] = j < k ? __ldg(row_of_slot + (size_t)t * k + j) : -1;
  const int R = T * k;
  const uint16_t* src = x + (size_t)t * d;
  // 8 elements per lane, 256 per warp and step; all lanes take every step so
  // the shuffles below always see the full warp (d is a multiple of 32, so a
  // 32-element block is either wholly inside or wholly outside the row)
  for (int base = 0; base < d; base += 256) {
    const int c0 = base + lane * 8;
    const bool act = c0 < d;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (act) w = ld_nc_v4(src + c0);
    float v[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                  bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if (!act) continue;
    const int e = block_exponent(amax);
    const float inv = inv_scale(e);
    uint2 o;
    o.x = e4m3x4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
    o.y = e4m3x4(v[4] * inv, v[5] * inv, v[6] * inv, v[7] * inv);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (row_ok(rows[j], R)) {
        const size_t r = (size_t)rows[j];
        *reinterpret_cast<uint2*>(xq + r * d + c0) = o;
        if ((lane & 3) == 0) xs[r * (d / 32) + c0 / 32] = (uint8_t)(e + 127);
        if (xp) st_v4(xp + r * d + c0, w);
      }
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_mxfp8_quantize_rows(const moe_bf16_t* src, int rows, int K, uint8_t* q, uint8_t* scale,
                            moe_stream_t stream) {
  MOE_CHECK_ARG(rows >= 0 && K > 0);
  if (K % 32 != 0) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  MOE_CHECK_PTR(src); MOE_CHECK_PTR(q);
  if (scale == nullptr) return MOE_ERR_INVALID_ARG;
  const long long nb = (long long)rows * (K / 32);
  (void)launch_pdl(quantize_rows_kernel, (unsigned)((nb + 255) / 256), 256, 0, (cudaStream_t)stream, src, nb, K, q, scale);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

int moe_mxfp8_quantize_weights(const moe_bf16_t* W, int E, int K, int N, uint8_t* wq, uint8_t* ws,
                               moe_stream_t stream) {
  MOE_CHECK_ARG(E >= 1 && K > 0 && N > 0);
  if (K % 32 != 0 || N % 128 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_CHECK_PTR(W); MOE_CHECK_PTR(wq);
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (K / 32 > 65535 || E > 65535) return MOE_ERR_UNSUPPORTED;
  dim3 grid(N / 128, K / 32, E);
  (void)launch_pdl(quantize_weights_kernel, grid, 128, 0, (cudaStream_t)stream, W, K, N, wq, ws);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

int moe_mxfp8_quantize_weights_f32(const float* W, int E, int K, int N, uint8_t* wq, uint8_t* ws,
                                   moe_stream_t stream) {
  MOE_CHECK_ARG(E >= 1 && K > 0 && N > 0);
  if (K % 32 != 0 || N % 128 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_CHECK_PTR(W); MOE_CHECK_PTR(wq);
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (K / 32 > 65535 || E > 65535) return MOE_ERR_UNSUPPORTED;
  dim3 grid(N / 128, K / 32, E);
  (void)launch_pdl(quantize_weights_f32_kernel, grid, 128, 0, (cudaStream_t)stream, W, K, N, wq, ws);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

int moe_mxfp8_dequantize_rows(const uint8_t* q, const uint8_t* scale, int rows, int K,
                              moe_bf16_t* out, moe_stream_t stream) {
  MOE_CHECK_ARG(rows >= 0 && K > 0);
  if (K % 32 != 0) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  MOE_CHECK_PTR(q); MOE_CHECK_PTR(out);
  if (scale == nullptr) return MOE_ERR_INVALID_ARG;
  const long long nb = (long long)rows * (K / 32);
  (void)launch_pdl(dequantize_rows_kernel, (unsigned)((nb + 255) / 256), 256, 0, (cudaStream_t)stream, q, scale, nb, out);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

int moe_dispatch_rows_mxfp8(const moe_bf16_t* x, int T, int d, int k, const int32_t* row_of_slot,
                            uint8_t* xq, uint8_t* xs, moe_bf16_t* xp, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && d > 0 && k >= 1 && k <= kMaxTopK);
  if (d % 32 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  MOE_CHECK_PTR(x); MOE_CHECK_PTR(row_of_slot); MOE_CHECK_PTR(xq);
  if (xs == nullptr) return MOE_ERR_INVALID_ARG;
  if (xp && !aligned16(xp)) return MOE_ERR_INVALID_ARG;
  dim3 grid((T + 7) / 8);
  (void)launch_pdl(dispatch_mxfp8_kernel, grid, 256, 0, (cudaStream_t)stream, x, T, d, k, row_of_slot, xq, xs, xp);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

}  // extern "C"
