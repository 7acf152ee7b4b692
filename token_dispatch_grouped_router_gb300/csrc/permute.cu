// Rowwise dispatch and combine (and the combine backward): 16-byte vectorised
// row copies between token order and the expert-contiguous buffer.
//
// "OLMo-core 3：MoE 训练栈让专家池越大、吞吐不再越慢", section "rowwise EP：用
// NVSHMEM 一端直写": no pack/permute stages; every routed row is written
// directly into its destination expert buffer by a route-table lookup, and
// combine brings the expert outputs back (the page's Table 7 puts dispatch at
// 2.298 ms and combine at 2.423 ms per trace on the multi-GPU stack).  On one
// GPU the NVSHMEM one-sided put becomes a plain HBM store.
//
// One warp per token; each lane moves 16-byte vectors (8 bf16), U of them in
// flight, so one token row is read once and written k times (dispatch) or k
// rows are read and one written (combine).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int U>
__global__ void __launch_bounds__(kThreads)
dispatch_kernel(const uint16_t* __restrict__ x, int T, int d, int k,
                const int32_t* __restrict__ row_of_slot, int R, uint16_t* __restrict__ xp) {
  pdl_enter();
  const int t = (int)((blockIdx.x * (size_t)kThreads + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int nvec = d >> 3;
  int rows[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) rows[j] = j < k ? __ldg(row_of_slot + (size_t)t * k + j) : -1;
  const uint16_t* src = x + (size_t)t * d;
  for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
    uint4 val[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      int v = v0 + 32 * u;
      if (v < nvec) val[u] = ld_nc_v4(src + (size_t)v * 8);
    }
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (row_ok(rows[j], R)) {
        uint16_t* dst = xp + (size_t)rows[j] * d;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          int v = v0 + 32 * u;
          if (v < nvec) st_v4(dst + (size_t)v * 8, val[u]);
        }
      }
    }
  }
}

__device__ __forceinline__ void fma8(float (&acc)[8], float g, uint4 v) {
  acc[0] = fmaf(g, bf16_lo(v.x), acc[0]); acc[1] = fmaf(g, bf16_hi(v.x), acc[1]);
  acc[2] = fmaf(g, bf16_lo(v.y), acc[2]); acc[3] = fmaf(g, bf16_hi(v.y), acc[3]);
  acc[4] = fmaf(g, bf16_lo(v.z), acc[4]); acc[5] = fmaf(g, bf16_hi(v.z), acc[5]);
  acc[6] = fmaf(g, bf16_lo(v.w), acc[6]); acc[7] = fmaf(g, bf16_hi(v.w), acc[7]);
}

// out[t] = sum_j g[t,j] * yp[row(t,j)] in slot order, fp32, one rounding
// (g = 1 without gates: the unpermute-sum).  k is a template parameter so
// that all K x U row loads of a pass are in flight before the first FMA (6 to
// 16 vectors of 16 bytes a lane; a generic copy loading one row at a time ran
// at 0.88-0.89 of the HBM copy rate, this one at 0.93-0.95); slots with no
// row read row 0 and add nothing.
template <int K, int U>
__global__ void __launch_bounds__(kThreads)
combine_k_kernel(const uint16_t* __restrict__ yp, int R, const int32_t* __restrict__ row_of_slot,
                 const float* __restrict__ gate, int T, int d, uint16_t* __restrict__ out) {
  pdl_enter();
  const int t = (int)((blockIdx.x * (size_t)kThreads + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int nvec = d >> 3;
  int rows[K];
  float g[K];
  bool ok[K];
#pragma unroll
  for (int j = 0; j < K; ++j) {
    rows[j] = __ldg(row_of_slot + (size_t)t * K + j);
    ok[j] = row_ok(rows[j], R);
    if (!ok[j]) rows[j] = 0;
    g[j] = gate ? __ldg(gate + (size_t)t * K + j) : 1.f;
  }
  uint16_t* dst = out + (size_t)t * d;
  for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
    uint4 val[K][U];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const uint16_t* src = yp + (size_t)rows[j] * d;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        if (v < nvec) val[j][u] = ld_nc_v4(src + (size_t)v * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v < nvec) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
        for (int j = 0; j < K; ++j)
          if (ok[j]) fma8(acc, g[j], val[j][u]);
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        st_v4(dst + (size_t)v * 8, o);
      }
    }
  }
}

template <int K>
void launch_combine_k(dim3 grid, cudaStream_t s, const uint16_t* yp, int R, const int32_t* row_of_slot,
                      const float* gate, int T, int d, uint16_t* out) {
  // two 16-byte vectors a row from k = 3 up: at k = 4, 64 registers instead of
  // 100 (twice the blocks an SM holds, 2 us faster at T = 16384, d = 2048, and
  // room for two blocks beside a CTA-pair GEMM's block)
  constexpr int U = K <= 2 ? 8 : 2;
  (void)launch_pdl(combine_k_kernel<K, U>, grid, kThreads, 0, s, yp, R, row_of_slot, gate, T, d, out);
}

void combine_switch(dim3 grid, cudaStream_t s, const moe_bf16_t* yp, int R, const int32_t* row_of_slot,
                    const float* gate, int T, int k, int d, moe_bf16_t* out) {
  switch (k) {
    case 1: launch_combine_k<1>(grid, s, yp, R, row_of_slot, gate, T, d, out); break;
    case 2: launch_combine_k<2>(grid, s, yp, R, row_of_slot, gate, T, d, out); break;
    case 3: launch_combine_k<3>(grid, s, yp, R, row_of_slot, gate, T, d, out); break;
    case 4: launch_combine_k<4>(grid, s, yp, R, row_of_slot, gate, T, d, out); break;
    case 5: launch_combine_k<5>(grid, s, yp, R, row_of_slot, gate, T, d, out); break;
    case 6: launch_combine_k<6>(grid, s, yp, R, row_of_slot, gate, T, d, out); break;
    case 7: launch_combine_k<7>(grid, s, yp, R, row_of_slot, gate, T, d, out); break;
    default: launch_combine_k<8>(grid, s, yp, R, row_of_slot, gate, T, d, out); break;
  }
}

__device__ __forceinline__ float dot8(uint4 a, uint4 b, float acc) {
  acc = fmaf(bf16_lo(a.x), bf16_lo(b.x), acc); acc = fmaf(bf16_hi(a.x), bf16_hi(b.x), acc);
  acc = fmaf(bf16_lo(a.y), bf16_lo(b.y), acc); acc = fmaf(bf16_hi(a.y), bf16_hi(b.y), acc);
  acc = fmaf(bf16_lo(a.z), bf16_lo(b.z), acc); acc = fmaf(bf16_hi(a.z), bf16_hi(b.z), acc);
  acc = fmaf(bf16_lo(a.w), bf16_lo(b.w), acc); acc = fmaf(bf16_hi(a.w), bf16_hi(b.w), acc);
  return acc;
}

__device__ __forceinline__ uint4 scale8(uint4 a, float g) {
  uint4 o;
  o.x = pack_bf16x2(g * bf16_lo(a.x), g * bf16_hi(a.x));
  o.y = pack_bf16x2(g * bf16_lo(a.y), g * bf16_hi(a.y));
  o.z = pack_bf16x2(g * bf16_lo(a.z), g * bf16_hi(a.z));
  o.w = pack_bf16x2(g * bf16_lo(a.w), g * bf16_hi(a.w));
  return o;
}

// dyp[row(t,j)] = g[t,j] * dout[t];  dg[t,j] = <dout[t], yp[row(t,j)]>
// K (= k) is a template parameter so that all K x U row loads of a pass are
// issued before the first use (the scaled stores would otherwise order each
// slot's loads after the previous slot's stores).
template <int K, int U>
__global__ void __launch_bounds__(kThreads)
combine_bwd_kernel(const uint16_t* __restrict__ dout, const uint16_t* __restrict__ yp, int R,
                   const int32_t* __restrict__ row_of_slot, const float* __restrict__ gate,
                   int T, int d, uint16_t* __restrict__ dyp, float* __restrict__ dgate) {
  pdl_enter();
  const int t = (int)((blockIdx.x * (size_t)kThreads + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int nvec = d >> 3;
  int rows[K];
  float g[K], dot[K];
  bool ok[K];
#pragma unroll
  for (int j = 0; j < K; ++j) {
    rows[j] = __ldg(row_of_slot + (size_t)t * K + j);
    ok[j] = row_ok(rows[j], R);
    if (!ok[j]) rows[j] = 0;                   // read a valid row; store and dot skipped
    g[j] = __ldg(gate + (size_t)t * K + j);
    dot[j] = 0.f;
  }
  const uint16_t* src = dout + (size_t)t * d;
  for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
    uint4 dv[U], yv[K][U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v < nvec) dv[u] = ld_nc_v4(src + (size_t)v * 8);
    }
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const uint16_t* yr = yp + (size_t)rows[j] * d;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        if (v < nvec) yv[j][u] = ld_nc_v4(yr + (size_t)v * 8);
      }
    }
#pragma unroll
    for (int j = 0; j < K; ++j) {
      uint16_t* dr = dyp + (size_t)rows[j] * d;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        if (v < nvec && ok[j]) {
          dot[j] = dot8(dv[u], yv[j][u], dot[j]);
          st_v4(dr + (size_t)v * 8, scale8(dv[u], g[j]));
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < K; ++j) {
    const float s = warp_sum(dot[j]);
    if (lane == 0) dgate[(size_t)t * K + j] = s;
  }
}

template <int K>
void launch_combine_bwd(dim3 grid, cudaStream_t s, const uint16_t* dout, const uint16_t* yp, int R,
                        const int32_t* row_of_slot, const float* gate, int T, int d, uint16_t* dyp,
                        float* dgate) {
  // 8 to 16 row vectors of 16 bytes in flight a lane
  constexpr int U = K <= 2 ? 8 : (K <= 4 ? 4 : 2);
  (void)launch_pdl(combine_bwd_kernel<K, U>, grid, kThreads, 0, s, dout, yp, R, row_of_slot, gate, T, d, dyp,
                   dgate);
}

// Zero the rows of a capacity-padded buffer [E*C][d] that hold no routed
// row: rows [e*C + counts[e], (e+1)*C) of every expert.  Warp per row.
__global__ void __launch_bounds__(kThreads)
zero_pad_rows_kernel(const int32_t* __restrict__ counts, int E, int C, int d, uint16_t* __restrict__ buf) {
  pdl_enter();
  const long long r = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= (long long)E * C) return;
  const int e = (int)(r / C), j = (int)(r - (long long)e * C);
  if (j < __ldg(counts + e)) return;
  uint16_t* p = buf + (size_t)r * d;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int v = lane; v < (d >> 3); v += 32) st_v4(p + (size_t)v * 8, z);
}

int launch_zero_pad_rows(const int32_t* counts, int E, int C, int d, uint16_t* buf, cudaStream_t s) {
  const long long rows = (long long)E * C;
  (void)launch_pdl(zero_pad_rows_kernel, (unsigned)((rows + kWarps - 1) / kWarps), kThreads, 0, s, counts, E,
                   C, d, buf);
  return 1;
}

void combine_bwd_switch(dim3 grid, cudaStream_t s, const moe_bf16_t* dout, const moe_bf16_t* yp, int R,
                        const int32_t* row_of_slot, const float* gate, int T, int k, int d, moe_bf16_t* dyp,
                        float* dgate) {
  switch (k) {
    case 1: launch_combine_bwd<1>(grid, s, dout, yp, R, row_of_slot, gate, T, d, dyp, dgate); break;
    case 2: launch_combine_bwd<2>(grid, s, dout, yp, R, row_of_slot, gate, T, d, dyp, dgate); break;
    case 3: launch_combine_bwd<3>(grid, s, dout, yp, R, row_of_slot, gate, T, d, dyp, dgate); break;
    case 4: launch_combine_bwd<4>(grid, s, dout, yp, R, row_of_slot, gate, T, d, dyp, dgate); break;
    case 5: launch_combine_bwd<5>(grid, s, dout, yp, R, row_of_slot, gate, T, d, dyp, dgate); break;
    case 6: launch_combine_bwd<6>(grid, s, dout, yp, R, row_of_slot, gate, T, d, dyp, dgate); break;
    case 7: launch_combine_bwd<7>(grid, s, dout, yp, R, row_of_slot, gate, T, d, dyp, dgate); break;
    default: launch_combine_bwd<8>(grid, s, dout, yp, R, row_of_slot, gate, T, d, dyp, dgate); break;
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_dispatch_rows(const moe_bf16_t* x, int T, int d, int k, const int32_t* row_of_slot,
                      moe_bf16_t* xp, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && d > 0 && d % 8 == 0 && k >= 1 && k <= kMaxTopK);
  if (T == 0) return MOE_OK;
  MOE_CHECK_PTR(x); MOE_CHECK_PTR(row_of_slot); MOE_CHECK_PTR(xp);
  dim3 grid((T + kWarps - 1) / kWarps);
  (void)launch_pdl(dispatch_kernel<8>, grid, kThreads, 0, (cudaStream_t)stream, x, T, d, k, row_of_slot, T * k,
                   xp);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

int moe_combine(const moe_bf16_t* yp, const int32_t* row_of_slot, const float* gate, int T, int k,
                int d, moe_bf16_t* out, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && d > 0 && d % 8 == 0 && k >= 1 && k <= kMaxTopK);
  if (T == 0) return MOE_OK;
  MOE_CHECK_PTR(yp); MOE_CHECK_PTR(row_of_slot); MOE_CHECK_PTR(out);
  if (gate && !aligned16(gate)) return MOE_ERR_INVALID_ARG;
  dim3 grid((T + kWarps - 1) / kWarps);
  combine_switch(grid, (cudaStream_t)stream, yp, T * k, row_of_slot, gate, T, k, d, out);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

int moe_combine_bwd(const moe_bf16_t* dout, const moe_bf16_t* yp, const int32_t* row_of_slot,
                    const float* gate, int T, int k, int d, moe_bf16_t* dyp, float* dgate,
                    moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && d > 0 && d % 8 == 0 && k >= 1 && k <= kMaxTopK);
  if (T == 0) return MOE_OK;
  MOE_CHECK_PTR(dout); MOE_CHECK_PTR(yp); MOE_CHECK_PTR(row_of_slot); MOE_CHECK_PTR(gate);
  MOE_CHECK_PTR(dyp); MOE_CHECK_PTR(dgate);
  dim3 grid((T + kWarps - 1) / kWarps);
  const cudaStream_t s = (cudaStream_t)stream;
  combine_bwd_switch(grid, s, dout, yp, T * k, row_of_slot, gate, T, k, d, dyp, dgate);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

// ------------------------------------------------- capacity-padded layer

int moe_dispatch_rows_capacity(const moe_bf16_t* x, int T, int d, int k, const int32_t* row_of_slot,
                               const int32_t* counts, int E, int C, moe_bf16_t* xp,
                               moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && d > 0 && d % 8 == 0 && k >= 1 && k <= kMaxTopK && E >= 1 && C >= 1);
  MOE_CHECK_ARG((long long)E * C <= 0x7fffffffLL && (long long)T * k <= 0x7fffffffLL);
  MOE_CHECK_PTR(counts); MOE_CHECK_PTR(xp);
  const cudaStream_t s = (cudaStream_t)stream;
  int n = 0;
  if (T > 0) {
    MOE_CHECK_PTR(x); MOE_CHECK_PTR(row_of_slot);
    (void)launch_pdl(dispatch_kernel<8>, dim3((T + kWarps - 1) / kWarps), kThreads, 0, s, x, T, d, k,
                     row_of_slot, E * C, xp);
    n = 1;
  }
  n += launch_zero_pad_rows(counts, E, C, d, xp, s);
  MOE_LAUNCH_CHECK(n);
  return MOE_OK;
}

int moe_combine_capacity(const moe_bf16_t* yp, int E, int C, const int32_t* row_of_slot, const float* gate,
                         int T, int k, int d, moe_bf16_t* out, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && d > 0 && d % 8 == 0 && k >= 1 && k <= kMaxTopK && E >= 1 && C >= 1);
  MOE_CHECK_ARG((long long)E * C <= 0x7fffffffLL);
  if (T == 0) return MOE_OK;
  MOE_CHECK_PTR(yp); MOE_CHECK_PTR(row_of_slot); MOE_CHECK_PTR(out);
  if (gate && !aligned16(gate)) return MOE_ERR_INVALID_ARG;
  combine_switch(dim3((T + kWarps - 1) / kWarps), (cudaStream_t)stream, yp, E * C, row_of_slot, gate, T, k, d, out);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

int moe_combine_bwd_capacity(const moe_bf16_t* dout, const moe_bf16_t* yp, int E, int C,
                             const int32_t* row_of_slot, const int32_t* counts, const float* gate,
                             int T, int k, int d, moe_bf16_t* dyp, float* dgate, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && d > 0 && d % 8 == 0 && k >= 1 && k <= kMaxTopK && E >= 1 && C >= 1);
  MOE_CHECK_ARG((long long)E * C <= 0x7fffffffLL);
  MOE_CHECK_PTR(counts); MOE_CHECK_PTR(dyp);
  const cudaStream_t s = (cudaStream_t)stream;
  int n = 0;
  if (T > 0) {
    MOE_CHECK_PTR(dout); MOE_CHECK_PTR(yp); MOE_CHECK_PTR(row_of_slot); MOE_CHECK_PTR(gate);
    MOE_CHECK_PTR(dgate);
    combine_bwd_switch(dim3((T + kWarps - 1) / kWarps), s, dout, yp, E * C, row_of_slot, gate, T, k, d, dyp,
                       dgate);
    n = 1;
  }
  n += launch_zero_pad_rows(counts, E, C, d, dyp, s);
  MOE_LAUNCH_CHECK(n);
  return MOE_OK;
}

}  // extern "C"
