// Router: logits GEMM (fp32 on CUDA cores), warp-per-token top-k with shuffle
// arg-max, renormalised softmax gates, and the backward of both.
//
// The pages ("Ai2 Olmo-core 3: The Secret Behind 2.7x MoE Training
// Throughput", section "The Capacity Tax") only say that a routing function
// picks a few experts (e.g. 4 of 128) per token.  The function implemented
// here is the benchmark specification's: softmax over the E logits, top-k,
// ties to the lower expert id, gates renormalised over the selection.  The
// router stays in fp32 (the OLMo-core 3 tutorial's DeepSeek-V3 paragraph in
// section "一个低精度格式，同时压三个地方" keeps gating in high precision).
#include <math.h>

#include "common.cuh"
#include "router_bwd.cuh"

namespace moe {
namespace {

// ----------------------------------------------------------- SIMT fp32 GEMM
// out[m][n] = sum_k A(m,k) * B(k,n), 64x64 tiles, BK = 16, 256 threads with a
// 4x4 register block each.  Used only for the router's small GEMMs (N = E).

enum class Lay { RowMK, ColMK };   // A: RowMK = a[m*ld+k], ColMK = a[k*ld+m]
enum class LayB { RowKN, ColKN };  // B: RowKN = b[k*ld+n], ColKN = b[n*ld+k]
enum class Epi { StoreBias, AddBf16, StorePartial };

template <typename TA> __device__ __forceinline__ float ldf(const TA* p);
template <> __device__ __forceinline__ float ldf<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

constexpr int SB = 64, SK = 16;

template <typename TA, Lay LA, LayB LB, Epi EP>
__global__ void __launch_bounds__(256)
simt_gemm_kernel(const TA* __restrict__ A, int lda, const float* __restrict__ B, int ldb,
                 int M, int N, int K, int k_per_split,
                 float* __restrict__ outf, __nv_bfloat16* __restrict__ outb, int ldo,
                 const float* __restrict__ bias) {
  pdl_enter();
  __shared__ float As[SK][SB + 4];
  __shared__ float Bs[SK][SB + 4];
  const int tid = threadIdx.x;
  const int m0 = blockIdx.x * SB, n0 = blockIdx.y * SB;
  const int split = blockIdx.z;
  const int kbeg = split * k_per_split;
  const int kend = min(K, kbeg + k_per_split);
  const int tm = (tid / 16) * 4, tn = (tid % 16) * 4;
  float acc[4][4] = {};
  for (int k0 = kbeg; k0 < kend; k0 += SK) {
#pragma unroll
    for (int i = 0; i < (SK * SB) / 256; ++i) {
      int e = tid + i * 256;
      int kk, mm;
      if (LA == Lay::RowMK) { kk = e % SK; mm = e / SK; } else { mm = e % SB; kk = e / SB; }
      int gm = m0 + mm, gk = k0 + kk;
      float v = 0.f;
      if (gm < M && gk < kend)
        v = (LA == Lay::RowMK) ? ldf(A + (size_t)gm * lda + gk) : ldf(A + (size_t)gk * lda + gm);
      As[kk][mm] = v;
    }
#pragma unroll
    for (int i = 0; i < (SK * SB) / 256; ++i) {
      int e = tid + i * 256;
      int kk, nn;
      if (LB == LayB::RowKN) { nn = e % SB; kk = e / SB; } else { kk = e % SK; nn = e / SK; }
      int gn = n0 + nn, gk = k0 + kk;
      float v = 0.f;
      if (gn < N && gk < kend)
        v = (LB == LayB::RowKN) ? __ldg(B + (size_t)gk * ldb + gn) : __ldg(B + (size_t)gn * ldb + gk);
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = As[kk][tm + i]; b[i] = Bs[kk][tn + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int gm = m0 + tm + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int gn = n0 + tn + j;
      if (gn >= N) continue;
      if (EP == Epi::StoreBias) {
        outf[(size_t)gm * ldo + gn] = acc[i][j] + (bias ? __ldg(bias + gn) : 0.f);
      } else if (EP == Epi::AddBf16) {
        __nv_bfloat16* p = outb + (size_t)gm * ldo + gn;
        *p = __float2bfloat16_rn(__bfloat162float(*p) + acc[i][j]);
      } else {
        outf[((size_t)split * M + gm) * ldo + gn] = acc[i][j];
      }
    }
  }
}

// dW_r[m][n] = sum over splits of the partials (fixed order: deterministic)
__global__ void reduce_splits_kernel(const float* __restrict__ part, int splits, int MN,
                                     float* __restrict__ out) {
  pdl_enter();
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= MN) return;
  float s = 0.f;
  for (int p = 0; p < splits; ++p) s += part[(size_t)p * MN + i];
  out[i] = s;
}

// db[e] = sum_t dz[t][e]: one block per expert, fixed-order block reduction
__global__ void column_sum_kernel(const float* __restrict__ dz, int T, int E, float* __restrict__ db) {
  pdl_enter();
  __shared__ float red[256];
  int e = blockIdx.x;
  float s = 0.f;
  for (int t = threadIdx.x; t < T; t += 256) s += dz[(size_t)t * E + e];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) db[e] = red[0];
}

// ----------------------------------------------------------------- top-k
// One warp per token.  Lane l holds logits l, l+32, ... (VPL per lane).  Each
// of the k rounds takes every lane's best untaken logit and reduces them with
// a butterfly arg-max whose order is (value desc, id asc), so every lane ends
// with the same winner; the owner lane marks it taken.

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  // candidate (v, i) precedes (bv, bi); bi < 0 means "no candidate yet"
  return i >= 0 && (bi < 0 || v > bv || (v == bv && i < bi));
}

template <int VPL>
__global__ void __launch_bounds__(256)
topk_kernel(const float* __restrict__ logits, int T, int E, int k,
            int32_t* __restrict__ idx_out, float* __restrict__ gate_out) {
  pdl_enter();
  const int warp = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* row = logits + (size_t)warp * E;
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    int e = lane + 32 * i;
    v[i] = e < E ? __ldg(row + e) : 0.f;
  }
  uint32_t taken = 0;
  float zsel[kMaxTopK];
  int isel[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    zsel[j] = 0.f; isel[j] = 0;
    if (j < k) {
      float bv = 0.f; int bi = -1;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && better(v[i], e, bv, bi)) { bv = v[i]; bi = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      zsel[j] = bv; isel[j] = bi;
    }
  }
  if (lane == 0) {
    // renormalised softmax over the selection; zsel[0] is the maximum
    float ex[kMaxTopK], s = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k) { ex[j] = expf(zsel[j] - zsel[0]); s += ex[j]; }
    }
    float inv = 1.f / s;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k) {
        idx_out[(size_t)warp * k + j] = isel[j];
        gate_out[(size_t)warp * k + j] = ex[j] * inv;
      }
    }
  }
}

__global__ void gates_kernel(const float* __restrict__ sel, int T, int k, float* __restrict__ gate) {
  pdl_enter();
  int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const float* z = sel + (size_t)t * k;
  float m = z[0];
  for (int j = 1; j < k; ++j) m = fmaxf(m, z[j]);
  float ex[kMaxTopK], s = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k) { ex[j] = expf(z[j] - m); s += ex[j]; }
  }
  float inv = 1.f / s;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (j < k) gate[(size_t)t * k + j] = ex[j] * inv;
}

// dz[t, idx_j] = g_j (dg_j - sum_l g_l dg_l); zero elsewhere.  Warp per token.
__global__ void __launch_bounds__(256)
topk_bwd_kernel(const float* __restrict__ gate, const float* __restrict__ dgate,
                const int32_t* __restrict__ idx, int T, int E, int k, float* __restrict__ dz) {
  pdl_enter();
  const int warp = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  float g[kMaxTopK], dg[kMaxTopK];
  int id[kMaxTopK];
  float inner = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    g[j] = 0.f; dg[j] = 0.f; id[j] = -1;
    if (j < k) {
      g[j] = __ldg(gate + (size_t)warp * k + j);
      dg[j] = __ldg(dgate + (size_t)warp * k + j);
      id[j] = __ldg(idx + (size_t)warp * k + j);
      inner = fmaf(g[j], dg[j], inner);
    }
  }
  float* row = dz + (size_t)warp * E;
  for (int e = lane; e < E; e += 32) {
    float val = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k && id[j] == e) val = g[j] * (dg[j] - inner);
    row[e] = val;
  }
}

// ------------------------------------------- backward through the top-k only
// The gates are a softmax over the k selected logits, so d_logits is zero
// outside the selection (moe_router_topk_bwd writes it so) and the router
// GEMMs' backward reduces to k rows of W_r^T per token (dx) and, per expert,
// a sum over the rows routed to it (dW_r, db), taken in the route map's
// token order so that the result does not depend on timing.

// W [d][E] -> WT [E][d] through 32 x 32 shared-memory tiles
__global__ void transpose_kernel(const float* __restrict__ W, int d, int E, float* __restrict__ WT) {
  pdl_enter();
  __shared__ float tile[32][33];
  const int e0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int k = k0 + i, e = e0 + threadIdx.x;
    tile[i][threadIdx.x] = (k < d && e < E) ? __ldg(W + (size_t)k * E + e) : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int e = e0 + i, k = k0 + threadIdx.x;
    if (e < E && k < d) WT[(size_t)e * d + k] = tile[threadIdx.x][i];
  }
}

// Chunks of at most kRouterChunk rows of every expert's segment, numbered
// expert-major: units[u] = (expert, first row, rows); estart / ecount give
// each expert's first chunk and chunk count; *total the number of chunks.
// One block of 1024 threads, thread = expert.
__global__ void __launch_bounds__(1024)
router_units_kernel(const int32_t* __restrict__ offsets, int E, int R, int4* __restrict__ units,
                    int* __restrict__ estart, int* __restrict__ ecount, int* __restrict__ total) {
  pdl_enter();
  __shared__ int wsum[32];
  const int e = threadIdx.x, lane = e & 31, w = e >> 5;
  int lo = 0, hi = 0, n = 0;
  if (e < E) {
    lo = max(0, min(__ldg(offsets + e), R));
    hi = max(lo, min(__ldg(offsets + e + 1), R));
    n = (hi - lo + kRouterChunk - 1) / kRouterChunk;
  }
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int v = wsum[lane];
    int iv = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, iv, o);
      if (lane >= o) iv += u;
    }
    wsum[lane] = iv - v;                 // exclusive prefix of the warp sums
    if (lane == 31) *total = iv;
  }
  __syncthreads();
  if (e < E) {
    const int base = wsum[w] + incl - n;
    estart[e] = base;
    ecount[e] = n;
    for (int c = 0; c < n; ++c)
      units[base + c] = make_int4(e, lo + c * kRouterChunk, min(kRouterChunk, hi - lo - c * kRouterChunk), 0);
  }
}

// Chunk u of expert e: part[u][:] = sum over its rows r (in order) of
// dz[t_r, e] * x[t_r][:], pbias[u] = sum of those dz.  The chunk's token ids
// and gradients are staged in shared memory first, so the x rows are loaded
// without a chain of dependent reads in front of each.  Thread = 8 columns.
__global__ void __launch_bounds__(256)
router_dw_partial_kernel(const uint16_t* __restrict__ x, const float* __restrict__ dz,
                         const int32_t* __restrict__ slot_of_row, const int4* __restrict__ units,
                         const int* __restrict__ total, int d, int E, int k, int R,
                         float* __restrict__ part, float* __restrict__ pbias) {
  pdl_enter();
  __shared__ int s_t[kRouterChunk];
  __shared__ float s_g[kRouterChunk];
  const int u = blockIdx.x;
  if (u >= __ldg(total)) return;
  const int4 un = units[u];
  const int e = un.x, r0 = un.y, rows = un.z;
  for (int i = threadIdx.x; i < rows; i += blockDim.x) {
    // a slot outside [0, T*k) (a row that holds no slot) adds nothing
    const int sl = __ldg(slot_of_row + r0 + i);
    const bool ok = row_ok(sl, R);
    const int t = ok ? sl / k : 0;
    s_t[i] = t;
    s_g[i] = ok ? __ldg(dz + (size_t)t * E + e) : 0.f;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float gs = 0.f;
    for (int r = 0; r < rows; ++r) gs += s_g[r];
    pbias[u] = gs;
  }
  for (int c0 = threadIdx.x * 8; c0 < d; c0 += 256 * 8) {
    float acc[8] = {};
    // groups of 8 rows: the 8 row loads are issued before their 64 FMAs
    for (int r0g = 0; r0g < rows; r0g += 8) {
      const int n = min(8, rows - r0g);
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        v[i] = i < n ? ld_nc_v4(x + (size_t)s_t[r0g + i] * d + c0) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i >= n) break;
        const float g = s_g[r0g + i];
        acc[0] = fmaf(g, bf16_lo(v[i].x), acc[0]); acc[1] = fmaf(g, bf16_hi(v[i].x), acc[1]);
        acc[2] = fmaf(g, bf16_lo(v[i].y), acc[2]); acc[3] = fmaf(g, bf16_hi(v[i].y), acc[3]);
        acc[4] = fmaf(g, bf16_lo(v[i].z), acc[4]); acc[5] = fmaf(g, bf16_hi(v[i].z), acc[5]);
        acc[6] = fmaf(g, bf16_lo(v[i].w), acc[6]); acc[7] = fmaf(g, bf16_hi(v[i].w), acc[7]);
      }
    }
    float* p = part + (size_t)u * d + c0;
    *reinterpret_cast<float4*>(p) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// dW_r[n][e] = sum of expert e's chunk partials in chunk order (zero for an
// empty expert); db[e] likewise.  Block = (256 columns, expert).
__global__ void __launch_bounds__(256)
router_dw_reduce_kernel(const float* __restrict__ part, const float* __restrict__ pbias,
                        const int* __restrict__ estart, const int* __restrict__ ecount, int d, int E,
                        float* __restrict__ dW, float* __restrict__ db) {
  pdl_enter();
  const int e = blockIdx.y, n = blockIdx.x * 256 + threadIdx.x;
  const int s0 = __ldg(estart + e), cnt = __ldg(ecount + e);
  if (n < d) {
    float acc = 0.f;
    for (int c = 0; c < cnt; ++c) acc += __ldg(part + (size_t)(s0 + c) * d + n);
    dW[(size_t)n * E + e] = acc;
  }
  if (db && blockIdx.x == 0 && threadIdx.x == 0) {
    float b = 0.f;
    for (int c = 0; c < cnt; ++c) b += __ldg(pbias + s0 + c);
    db[e] = b;
  }
}

// dx[t] += sum_j dz[t, e_j] * WT[e_j] (j in slot order), rounded once to
// bf16.  Warp per token, 8 columns per lane and step.
__global__ void __launch_bounds__(256)
router_dx_topk_kernel(const float* __restrict__ dz, const int32_t* __restrict__ idx,
                      const float* __restrict__ WT, int T, int d, int E, int k,
                      uint16_t* __restrict__ dx) {
  pdl_enter();
  const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int ee[kMaxTopK];
  float gg[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    ee[j] = -1; gg[j] = 0.f;
    if (j < k) {
      const int e = __ldg(idx + (size_t)t * k + j);
      if ((unsigned)e < (unsigned)E) { ee[j] = e; gg[j] = __ldg(dz + (size_t)t * E + e); }
    }
  }
  for (int c0 = lane * 8; c0 < d; c0 += 256) {
    float acc[8] = {};
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (ee[j] < 0) continue;
      const float* w = WT + (size_t)ee[j] * d + c0;
      const float4 a = __ldg(reinterpret_cast<const float4*>(w));
      const float4 b = __ldg(reinterpret_cast<const float4*>(w + 4));
      acc[0] = fmaf(gg[j], a.x, acc[0]); acc[1] = fmaf(gg[j], a.y, acc[1]);
      acc[2] = fmaf(gg[j], a.z, acc[2]); acc[3] = fmaf(gg[j], a.w, acc[3]);
      acc[4] = fmaf(gg[j], b.x, acc[4]); acc[5] = fmaf(gg[j], b.y, acc[5]);
      acc[6] = fmaf(gg[j], b.z, acc[6]); acc[7] = fmaf(gg[j], b.w, acc[7]);
    }
    uint4* p = reinterpret_cast<uint4*>(dx + (size_t)t * d + c0);
    uint4 v = *p;
    v.x = pack_bf16x2(bf16_lo(v.x) + acc[0], bf16_hi(v.x) + acc[1]);
    v.y = pack_bf16x2(bf16_lo(v.y) + acc[2], bf16_hi(v.y) + acc[3]);
    v.z = pack_bf16x2(bf16_lo(v.z) + acc[4], bf16_hi(v.z) + acc[5]);
    v.w = pack_bf16x2(bf16_lo(v.w) + acc[6], bf16_hi(v.w) + acc[7]);
    *p = v;
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_router_logits_bwd_topk(const moe_bf16_t* x, const float* W_r, const float* d_logits,
                               const int32_t* topk_idx, const int32_t* offsets,
                               const int32_t* slot_of_row, int T, int d, int E, int k,
                               moe_bf16_t* dx, float* dW_r, float* db, void* ws, size_t ws_bytes,
                               moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && d > 0 && E > 0 && E <= kMaxExperts && k >= 1 && k <= kMaxTopK && k <= E);
  if (d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_CHECK_PTR(W_r); MOE_CHECK_PTR(dW_r);
  if (db && !aligned16(db)) return MOE_ERR_INVALID_ARG;
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (T == 0) {
    if (cudaMemsetAsync(dW_r, 0, sizeof(float) * (size_t)d * E, s) != cudaSuccess ||
        (db && cudaMemsetAsync(db, 0, sizeof(float) * (size_t)E, s) != cudaSuccess)) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }
  MOE_CHECK_PTR(x); MOE_CHECK_PTR(d_logits); MOE_CHECK_PTR(topk_idx); MOE_CHECK_PTR(offsets);
  MOE_CHECK_PTR(slot_of_row); MOE_CHECK_PTR(dx);
  const long long R = (long long)T * k;
  const RouterTopkScratch L = router_topk_scratch(R, E, d);
  if (ws_bytes < L.end) return MOE_ERR_WORKSPACE;
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* WT = reinterpret_cast<float*>(base + L.wt);
  int4* units = reinterpret_cast<int4*>(base + L.units);
  int* estart = reinterpret_cast<int*>(base + L.estart);
  int* ecount = reinterpret_cast<int*>(base + L.ecount);
  int* total = reinterpret_cast<int*>(base + L.total);
  float* part = reinterpret_cast<float*>(base + L.part);
  float* pbias = reinterpret_cast<float*>(base + L.pbias);
  (void)launch_pdl(transpose_kernel, dim3((E + 31) / 32, (d + 31) / 32), dim3(32, 8), 0, s, W_r, d, E, WT);
  (void)launch_pdl(router_units_kernel, 1, 1024, 0, s, offsets, E, (int)R, units, estart, ecount, total);
  (void)launch_pdl(router_dw_partial_kernel, (unsigned)L.max_units, 256, 0, s,
                   reinterpret_cast<const uint16_t*>(x), d_logits, slot_of_row, units, total, d, E, k,
                   (int)R, part, pbias);
  (void)launch_pdl(router_dw_reduce_kernel, dim3((d + 255) / 256, E), 256, 0, s, part, pbias, estart,
                   ecount, d, E, dW_r, db);
  (void)launch_pdl(router_dx_topk_kernel, (unsigned)((T + 7) / 8), 256, 0, s, d_logits, topk_idx, WT,
                   T, d, E, k, reinterpret_cast<uint16_t*>(dx));
  MOE_LAUNCH_CHECK(5);
  return MOE_OK;
}

int moe_router_logits(const moe_bf16_t* x, const float* W_r, const float* b, int T, int d, int E,
                      float* logits, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && d > 0 && E > 0);
  if (T == 0) return MOE_OK;
  MOE_CHECK_PTR(x); MOE_CHECK_PTR(W_r); MOE_CHECK_PTR(logits);
  if (b && !aligned16(b)) return MOE_ERR_INVALID_ARG;
  dim3 grid((T + SB - 1) / SB, (E + SB - 1) / SB, 1);
  (void)launch_pdl(simt_gemm_kernel<__nv_bfloat16, Lay::RowMK, LayB::RowKN, Epi::StoreBias>, grid, 256, 0, (cudaStream_t)stream, 
          reinterpret_cast<const __nv_bfloat16*>(x), d, W_r, E, T, E, d, d,
          logits, nullptr, E, b);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

int moe_router_topk(const float* logits, int T, int E, int k, int32_t* topk_idx,
                    float* topk_gate, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && E > 0 && E <= kMaxExperts && k >= 1 && k <= kMaxTopK && k <= E);
  if (T == 0) return MOE_OK;
  MOE_CHECK_PTR(logits); MOE_CHECK_PTR(topk_idx); MOE_CHECK_PTR(topk_gate);
  const int threads = 256, warps = threads / 32;
  dim3 grid((T + warps - 1) / warps);
  cudaStream_t s = (cudaStream_t)stream;
  int vpl = (E + 31) / 32;
  if (vpl <= 1) (void)launch_pdl(topk_kernel<1>, grid, threads, 0, s, logits, T, E, k, topk_idx, topk_gate);
  else if (vpl <= 2) (void)launch_pdl(topk_kernel<2>, grid, threads, 0, s, logits, T, E, k, topk_idx, topk_gate);
  else if (vpl <= 4) (void)launch_pdl(topk_kernel<4>, grid, threads, 0, s, logits, T, E, k, topk_idx, topk_gate);
  else if (vpl <= 8) (void)launch_pdl(topk_kernel<8>, grid, threads, 0, s, logits, T, E, k, topk_idx, topk_gate);
  else if (vpl <= 16) (void)launch_pdl(topk_kernel<16>, grid, threads, 0, s, logits, T, E, k, topk_idx, topk_gate);
  else (void)launch_pdl(topk_kernel<32>, grid, threads, 0, s, logits, T, E, k, topk_idx, topk_gate);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

int moe_router_gates(const float* sel_logits, int T, int k, float* topk_gate, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && k >= 1 && k <= kMaxTopK);
  if (T == 0) return MOE_OK;
  MOE_CHECK_PTR(sel_logits); MOE_CHECK_PTR(topk_gate);
  (void)launch_pdl(gates_kernel, (T + 255) / 256, 256, 0, (cudaStream_t)stream, sel_logits, T, k, topk_gate);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

int moe_router_topk_bwd(const float* topk_gate, const float* d_gate, const int32_t* topk_idx,
                        int T, int E, int k, float* d_logits, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && E > 0 && E <= kMaxExperts && k >= 1 && k <= kMaxTopK && k <= E);
  if (T == 0) return MOE_OK;
  MOE_CHECK_PTR(topk_gate); MOE_CHECK_PTR(d_gate); MOE_CHECK_PTR(topk_idx); MOE_CHECK_PTR(d_logits);
  dim3 grid((T + 7) / 8);
  (void)launch_pdl(topk_bwd_kernel, grid, 256, 0, (cudaStream_t)stream, topk_gate, d_gate, topk_idx, T, E, k, d_logits);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

int moe_router_logits_bwd(const moe_bf16_t* x, const float* W_r, const float* d_logits, int T,
                          int d, int E, moe_bf16_t* dx, float* dW_r, float* db, void* ws,
                          size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && d > 0 && E > 0 && E <= kMaxExperts);
  MOE_CHECK_PTR(x); MOE_CHECK_PTR(W_r); MOE_CHECK_PTR(dW_r);
  if (db && !aligned16(db)) return MOE_ERR_INVALID_ARG;
  if (T > 0) { MOE_CHECK_PTR(d_logits); MOE_CHECK_PTR(dx); }
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  if (ws_bytes < router_scratch_end(E, d)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  if (T == 0) {
    if (cudaMemsetAsync(dW_r, 0, sizeof(float) * (size_t)d * E, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (db && cudaMemsetAsync(db, 0, sizeof(float) * (size_t)E, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  // dx += dz @ W_r^T : M = T, N = d, K = E; B(k=e, n) = W_r[n*E + e]
  {
    dim3 grid((T + SB - 1) / SB, (d + SB - 1) / SB, 1);
    (void)launch_pdl(simt_gemm_kernel<float, Lay::RowMK, LayB::ColKN, Epi::AddBf16>, grid, 256, 0, s, 
        d_logits, E, W_r, E, T, d, E, E, nullptr, reinterpret_cast<__nv_bfloat16*>(dx), d, nullptr);
  }
  // dW_r = x^T @ dz : M = d, N = E, K = T, split into kRouterSplits partials
  float* part = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + kStatusBytes);
  {
    int kps = (T + kRouterSplits - 1) / kRouterSplits;
    kps = (kps + SK - 1) / SK * SK;
    dim3 grid((d + SB - 1) / SB, (E + SB - 1) / SB, kRouterSplits);
    (void)launch_pdl(simt_gemm_kernel<__nv_bfloat16, Lay::ColMK, LayB::RowKN, Epi::StorePartial>, grid, 256, 0, s, 
        reinterpret_cast<const __nv_bfloat16*>(x), d, d_logits, E, d, E, T, kps, part, nullptr, E,
        nullptr);
    int MN = d * E;
    (void)launch_pdl(reduce_splits_kernel, (MN + 255) / 256, 256, 0, s, part, kRouterSplits, MN, dW_r);
  }
  int n = 3;
  if (db) { (void)launch_pdl(column_sum_kernel, E, 256, 0, s, d_logits, T, E, db); ++n; }
  MOE_LAUNCH_CHECK(n);
  return MOE_OK;
}

}  // extern "C"
