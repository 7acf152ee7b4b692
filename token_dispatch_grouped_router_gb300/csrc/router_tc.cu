// Router logits z = x W_r + b on the tcgen05 tensor cores at fp32 accuracy.
//
// The router stays in high precision (OLMo-core 3 tutorial, section
// "一个低精度格式，同时压三个地方": DeepSeek-V3 keeps its gating in high
// precision), so the logits must be the fp32 product of the bf16 tokens x and
// the fp32 router weights W_r.  x is exact in bf16; W_r is split exactly into
// three bf16 parts, W_r = W0 + W1 + W2 with W0 = RNE_bf16(W_r),
// W1 = RNE_bf16(W_r - W0), W2 = RNE_bf16(W_r - W0 - W1) (each residual is
// exact in fp32 and holds at most 8 significant bits after two steps, so the
// three parts carry all 24 bits of a normal fp32 value).  Every product of a
// bf16 x with a bf16 part is exact in fp32, and the MMA accumulates them in
// fp32: z = x W0 + x W1 + x W2 + b, a reduction over 3d terms instead of d.
//
// Kernel: one 128 x 128 output tile per CTA (grid = row tiles x expert
// tiles), warp 0 streams k-blocks of 64 by TMA (the x tile once, the three
// weight parts beside it: 64 KB a stage, 3 stages), warp 1 issues
// tcgen05.mma kind::f16 M = 128, N = 128, K = 16 into one TMEM accumulator
// (12 MMAs a stage), warps 2-5 add the bias and store fp32 rows.  Rows past T
// and experts past E are TMA zero fill and are not stored.
#include "gemm_common.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace gemm;

constexpr int RM = 128, RN = 128, RBK = 64, RSTAGES = 3, RPARTS = 3;
constexpr int R_A = RM * RBK * 2;                    // 16 KB of x
constexpr int R_B = RN * RBK * 2;                    // 16 KB of one weight part
constexpr int R_STAGE = R_A + RPARTS * R_B;          // 64 KB
constexpr int R_THREADS = 192;                       // producer, MMA, 4 epilogue warps
constexpr int R_TMEM_COLS = 128;

struct RouterShared {
  uint64_t full[RSTAGES], empty[RSTAGES], tfull, drain;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t router_smem_bytes() { return 1024 + (size_t)RSTAGES * R_STAGE + sizeof(RouterShared); }

inline int round64(int v) { return (v + 63) / 64 * 64; }

// W_r [d][E] fp32 -> w3 [E][3][dp] bf16, dp = d rounded up to 64, zeros in
// columns d..dp-1 of every part.  Thread per (e, k): consecutive threads
// write consecutive k of one expert row.
__global__ void router_split_kernel(const float* __restrict__ W, int d, int E, int dp,
                                    uint16_t* __restrict__ w3) {
  pdl_enter();
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= (long long)E * dp) return;
  const int e = (int)(i / dp), k = (int)(i % dp);
  float w = k < d ? __ldg(W + (size_t)k * E + e) : 0.f;
  uint16_t part[RPARTS];
#pragma unroll
  for (int p = 0; p < RPARTS; ++p) {
    const __nv_bfloat16 b = __float2bfloat16_rn(w);
    part[p] = *reinterpret_cast<const uint16_t*>(&b);
    w -= __bfloat162float(b);                        // exact: the residual of an RNE rounding
  }
  uint16_t* row = w3 + (size_t)e * RPARTS * dp + k;
#pragma unroll
  for (int p = 0; p < RPARTS; ++p) row[(size_t)p * dp] = part[p];
}

__global__ void __launch_bounds__(R_THREADS, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 const float* __restrict__ bias, int T, int E, int dp, float* __restrict__ logits,
                 int* __restrict__ status) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  RouterShared* sh = reinterpret_cast<RouterShared*>(smem + RSTAGES * R_STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * RM, n0 = blockIdx.y * RN;
  const int nkb = dp / RBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RSTAGES; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    mbar_init(smem_u32(&sh->tfull), 1);
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sh->tmem_base), R_TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) { prefetch_tmap(&tmX); prefetch_tmap(&tmW); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0, issued = 0, last_par = 0;
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
      if (!bounded_wait(smem_u32(&sh->empty[stage]), phase ^ 1u, &sh->abort_flag, status)) { ok = false; break; }
      if (lane == 0) {
        const uint32_t fb = smem_u32(&sh->full[stage]);
        const uint32_t sa = smem_u32(smem + stage * R_STAGE);
        mbar_arrive_expect_tx(fb, R_STAGE);
        tma_load_2d(sa, &tmX, fb, kb * RBK, m0);
#pragma unroll
        for (int p = 0; p < RPARTS; ++p) tma_load_2d(sa + R_A + p * R_B, &tmW, fb, p * dp + kb * RBK, n0);
      }
      __syncwarp();
      issued |= 1u << stage;
      last_par = (last_par & ~(1u << stage)) | (phase << stage);
      if (++stage == RSTAGES) { stage = 0; phase ^= 1u; }
    }
    if (!ok && lane == 0) {
      for (int s = 0; s < RSTAGES; ++s)
        if (issued & (1u << s)) drain_wait(smem_u32(&sh->full[s]), (last_par >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16(RM, RN, false, false);   // both operands K-major
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true, issued_any = false;
    for (int kb = 0; kb < nkb; ++kb) {
      if (!bounded_wait(smem_u32(&sh->full[stage]), phase, &sh->abort_flag, status)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sa = smem_u32(smem + stage * R_STAGE);
#pragma unroll
        for (int p = 0; p < RPARTS; ++p)
#pragma unroll
          for (int kk = 0; kk < RBK / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sa + R_A + p * R_B + kk * 32, 16, 1024);
            mma_f16(tmem, ad, bd, idesc, (kb > 0 || p > 0 || kk > 0) ? 1u : 0u);
          }
        mma_commit(smem_u32(&sh->empty[stage]));
      }
      issued_any = true;
      __syncwarp();
      if (++stage == RSTAGES) { stage = 0; phase ^= 1u; }
    }
    if (ok && lane == 0) mma_commit(smem_u32(&sh->tfull));
    if (!ok && issued_any && lane == 0) {
      mma_commit(smem_u32(&sh->drain));
      drain_wait(smem_u32(&sh->drain), 0);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------------- epilogue
    const int lane_q = warp & 3;                     // TMEM lane quarter of this warp
    if (bounded_wait(smem_u32(&sh->tfull), 0, &sh->abort_flag, status)) {
      tc_fence_after();
      const int m = m0 + 32 * lane_q + lane;
      const bool vec = (E & 3) == 0;
#pragma unroll 1
      for (int c = 0; c < RN / 32; ++c) {
        const int n = n0 + 32 * c;
        if (n >= E) break;                           // warp-uniform
        uint32_t q[32];
        tmem_ld32(tmem + ((uint32_t)(32 * lane_q) << 16) + 32 * c, q);
        tmem_ld_wait();
        if (m >= T) continue;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(q[i]) + (bias && n + i < E ? __ldg(bias + n + i) : 0.f);
        float* row = logits + (size_t)m * E + n;
        if (vec && n + 32 <= E) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(row + 4 * i) = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        } else {
          for (int i = 0; i < 32 && n + i < E; ++i) row[i] = v[i];
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, R_TMEM_COLS);
  }
}

}  // namespace
}  // namespace moe

using namespace moe;
using namespace moe::gemm;

extern "C" int moe_router_logits_tc(const moe_bf16_t* x, const float* W_r, const float* b, int T,
                                    int d, int E, float* logits, void* ws, size_t ws_bytes,
                                    moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && d > 0 && E > 0 && E <= kMaxExperts);
  if (d % 8 != 0) return MOE_ERR_UNSUPPORTED;            // 16-byte rows of x for TMA
  if (ws == nullptr || ws_bytes < kStatusBytes) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  MOE_CHECK_PTR(x); MOE_CHECK_PTR(W_r); MOE_CHECK_PTR(logits);
  if (b && !aligned16(b)) return MOE_ERR_INVALID_ARG;
  const int dp = round64(d);
  const size_t split_bytes = (size_t)E * RPARTS * dp * 2;
  if (ws_bytes < kStatusBytes + split_bytes) return MOE_ERR_WORKSPACE;
  uint16_t* w3 = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + kStatusBytes);
  cudaStream_t s = (cudaStream_t)stream;
  const long long n_split = (long long)E * dp;
  (void)launch_pdl(router_split_kernel, (unsigned)((n_split + 255) / 256), 256, 0, s, W_r, d, E, dp, w3);
  MOE_LAUNCH_CHECK(1);
  CUtensorMap mx, mw;
  if (!map2d(&mx, x, d, T, RBK, RM) || !map2d(&mw, w3, (uint64_t)RPARTS * dp, E, RBK, RN))
    return MOE_ERR_CUDA;
  auto kern = router_tc_kernel;
  static bool attr_done[64] = {false};
  if (ensure_smem_attr(kern, router_smem_bytes(), attr_done) != MOE_OK) return MOE_ERR_CUDA;
  dim3 grid((T + RM - 1) / RM, (E + RN - 1) / RN);
  (void)launch_pdl(kern, grid, R_THREADS, router_smem_bytes(), s, mx, mw, b, T, E, dp, logits,
                   reinterpret_cast<int*>(ws));
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}
