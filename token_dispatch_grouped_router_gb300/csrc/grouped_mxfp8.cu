// MXFP8 forward of the unpadded grouped SwiGLU FFN on block-scaled tcgen05
// tensor cores (kind::mxf8f6f4, E4M3 x E4M3, E8M0 scale per 32 along K).
//
// "OLMo-core 3：MoE 训练栈让专家池越大、吞吐不再越慢", section "一个低精度格式，同时压三
// 个地方": the GEMMs run in MXFP8 (the page also quantises saved activations
// and dispatch payloads); the FP32 master weights stay authoritative and the
// low-precision copies are re-made after each optimizer step.  Here the
// forward GEMMs take E4M3 operands with per-32 E8M0 scales along K and
// accumulate in fp32; outputs are bf16 (the backward stays bf16).
//
// Two modes of one persistent kernel, same warp roles as the bf16 kernel:
//   UP8  : [h1 | h3] = Xq_e @ [W1q[e] | W3q[e]]  (96 + 96 columns per tile);
//          epilogue writes h1, h3, a = silu(h1) * h3 (bf16) and quantises a
//          (one 32-column block per thread: Aq codes + As scale bytes)
//   DOWN8: yp = Aq_e @ W2q[e]
// Tiles are 128 x 192 with BK = 128 fp8 (one 128-byte swizzled row per
// operand row), 4 pipeline stages.  Operands are K-major: activations
// [R][K], weights [E][N][K] (moe_mxfp8_quantize_weights transposes).
// Issue rates of block-scaled MMAs with their per-k-block scale copies,
// measured on the GB300 with operands resident in shared memory: N = 256 runs
// at the full fp8 rate, N = 192 at 93% and N = 128 at 65-68%.  Two 192-column
// fp32 accumulators (at TMEM columns 0 and 256) leave room for the scale
// factors, so the epilogue of one tile overlaps the next tile's mainloop
// (a 256-column tile would fit only one accumulator).
// Scale factors: per stage 512-byte atoms, byte (r, 4j + k) = scale of row
// (or column) 32j + r of the atom for the stage's k-th 32-element block, one
// for A and two for B (columns 0-127 and 128-191), gathered by the producer
// warp with zero-filling cp.async (row-major scales in HBM) and moved to
// tensor memory with tcgen05.cp .32x128b.warpx4 (which replicates an atom
// into the four lane quarters).  The MMA then reads row m's A scale at lane
// m, column base + m/32, and column n's B scale at lane n%32 of the issuing
// quarter, column base + n/32, byte = the MMA's scale-factor id (0..3).
#include "gemm_common.cuh"
#include "mx_common.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace gemm;

enum Mode8 : int { kUp8 = 0, kDown8 = 1 };

constexpr int BM = 128, BN = 192, BK = 128, STAGES = 4;
constexpr int A_STAGE = BM * BK;                // 16 KB of E4M3
constexpr int B_STAGE = BN * BK;                // 24 KB
constexpr int SF_STAGE = 1536;                  // A atom + two B atoms
constexpr int kAccStride = 256;                 // accumulators at TMEM columns 0 and 256
constexpr int kSfCol0 = 448;                    // stage s: A at +12s, B at +12s+4 (8 columns)
constexpr int kTmemCols = 512;
constexpr int kMaxExperts8 = 768;               // shared-memory tile table bound

struct Args8 {
  const int32_t* offsets;
  int E, R, d, h;
  int n_tiles;
  int kb_total;                 // K / 128
  int K;                        // reduction length of this GEMM
  const uint8_t* sfa;           // activation scales [R][K/32]
  const uint8_t* sfb0;          // weight scales [E][N][K/32] (UP8: W1)
  const uint8_t* sfb1;          // UP8: W3 scales
  int N;                        // rows of one weight matrix (UP8: h, DOWN8: d)
  uint16_t* out0;               // UP8: h1 / DOWN8: yp
  uint16_t* out1;               // UP8: h3
  uint16_t* out2;               // UP8: a
  uint8_t* aq;                  // UP8: quantised a [R][h]
  uint8_t* as;                  // UP8: scales of a [R][h/32]
  int* status;
};

using Shared = PipeShared<STAGES>;

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_cp_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of the block-scaled MMA: E4M3 A and B (format 0),
// E8M0 scales (bit 23), N >> 3 at bits 17-22, M >> 4 at bits 24-28, the
// scale-factor byte id of B at bits 4-5 and of A at bits 29-30.
__device__ __forceinline__ uint32_t idesc_mxf8(int M, int N, int sf_id) {
  return ((uint32_t)sf_id << 4) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(M >> 4) << 24) | ((uint32_t)sf_id << 29);
}

// no-swizzle descriptor of a 32-row x 16-byte scale atom (8-row groups 128 B apart)
__device__ __forceinline__ uint64_t sdesc_atom(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Whole 32-row slices of the bf16 outputs leave by TMA store (o0..o2: UP8
// h1, h3, a; DOWN8 yp; see store_chunk_tma); a slice cut by the end of an
// expert's rows, and the fp8 codes of a, by coalesced stores of its own rows.
template <int MODE>
__device__ __forceinline__ void epilogue8(const RowTile& rt, int n0, uint32_t tacc, int lane_q,
                                          int half, int lane, uint8_t* stg, const Args8& a,
                                          const CUtensorMap* o0, const CUtensorMap* o1,
                                          const CUtensorMap* o2) {
  const uint32_t tbase = tacc + ((uint32_t)(lane_q * 32) << 16);
  const int nrows = min(32, rt.rows - lane_q * 32);
  const size_t r0 = (size_t)rt.row0 + (nrows > 0 ? lane_q * 32 : 0);
  const bool whole = nrows == 32;
  if constexpr (MODE == kUp8) {
    // columns 0..95: h1[:, n0..n0+95]; 96..191: h3[:, n0..n0+95]; three
    // 32-column chunks, two for the first half of the warps, one for the second
#pragma unroll 1
    for (int c = half * 2; c < min(half * 2 + 2, 3); ++c) {
      const int col = n0 + c * 32;
      if (col >= a.h) break;                      // warp-uniform
      uint32_t q1[32], q3[32];
      tmem_ld32(tbase + c * 32, q1);
      tmem_ld32(tbase + 96 + c * 32, q3);
      tmem_ld_wait();
      float h1[32], h3[32], av[32];
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        h1[i] = __uint_as_float(q1[i]);
        h3[i] = __uint_as_float(q3[i]);
        av[i] = silu_f(h1[i]) * h3[i];
        amax = fmaxf(amax, fabsf(av[i]));
      }
      // (a caller that keeps only the quantised a passes no bf16 a)
      if (whole) {
        store_chunk_tma(stg, h1, lane, o0, col, (int)r0);
        store_chunk_tma(stg, h3, lane, o1, col, (int)r0);
        if (a.out2) store_chunk_tma(stg, av, lane, o2, col, (int)r0);
      } else {
        stg_acquire(lane);
        store_chunk(stg, h1, lane, a.out0 + r0 * a.h + col, a.h, nrows);
        store_chunk(stg, h3, lane, a.out1 + r0 * a.h + col, a.h, nrows);
        if (a.out2) store_chunk(stg, av, lane, a.out2 + r0 * a.h + col, a.h, nrows);
      }
      // quantise this row's 32-column block of a (fp32 values, before rounding)
      const int ex = mx::block_exponent(amax);
      const float inv = mx::inv_scale(ex);
      uint4 o[2];
      uint32_t* w = reinterpret_cast<uint32_t*>(o);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = mx::e4m3x4(av[4 * i] * inv, av[4 * i + 1] * inv, av[4 * i + 2] * inv, av[4 * i + 3] * inv);
      stg_acquire(lane);
      store_chunk_bytes32(stg, o, lane, a.aq + r0 * a.h + col, a.h, nrows);
      if (lane < nrows) a.as[(r0 + lane) * (a.h / 32) + col / 32] = (uint8_t)(ex + 127);
    }
  } else {
#pragma unroll 1
    for (int c = half * 3; c < half * 3 + 3; ++c) {
      const int col = n0 + c * 32;
      if (col >= a.d) break;                      // warp-uniform
      uint32_t q[32];
      tmem_ld32(tbase + c * 32, q);
      tmem_ld_wait();
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(q[i]);
      if (whole) {
        store_chunk_tma(stg, v, lane, o0, col, (int)r0);
      } else {
        stg_acquire(lane);
        store_chunk(stg, v, lane, a.out0 + r0 * a.d + col, a.d, nrows);
      }
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
grouped_mxfp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                     const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmO0,
                     const __grid_constant__ CUtensorMap tmO1, const __grid_constant__ CUtensorMap tmO2,
                     const Args8 args) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + STAGES * A_STAGE;
  uint8_t* sSF = sB + STAGES * B_STAGE;                      // STAGES x 1 KB
  uint8_t* sStage = sSF + STAGES * SF_STAGE;                 // kEpiWarps x kStageBytes
  Shared* sh = reinterpret_cast<Shared*>(sStage + kEpiWarps * kStageBytes);
  int* s_off = reinterpret_cast<int*>(sh + 1);
  int* s_ts = s_off + (args.E + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i <= args.E; i += kThreads) s_off[i] = __ldg(args.offsets + i);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1 + 32);     // TMA arrival + one cp.async arrival per lane
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) { mbar_init(smem_u32(&sh->tfull[s]), 1); mbar_init(smem_u32(&sh->tempty[s]), kEpiWarps); }
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    const int n = build_row_tile_table(s_off, s_ts, args.E, args.R, args.n_tiles, lane);
    if (lane == 0) sh->total_tiles = n;
  }
  __syncthreads();
  const int total = sh->total_tiles;
  if ((int)blockIdx.x >= total) return;

  if (warp == 1) {
    tmem_alloc(smem_u32(&sh->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA); prefetch_tmap(&tmB0); prefetch_tmap(&tmB1);
    prefetch_tmap(&tmO0); prefetch_tmap(&tmO1); prefetch_tmap(&tmO2);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  const int ksf = args.K / 32;                               // scale bytes per row

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0, issued = 0, last_par = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const RowTile rt = decode_row_tile(t, args.E, args.R, s_off, s_ts);
      const int n0 = rt.n_idx * (MODE == kUp8 ? BN / 2 : BN);
      for (int kb = 0; kb < args.kb_total; ++kb) {
        if (!bounded_wait(smem_u32(&sh->empty[stage]), phase ^ 1u, &sh->abort_flag, args.status)) { ok = false; break; }
        const uint32_t fb = smem_u32(&sh->full[stage]);
        const uint32_t sa = smem_u32(sA + stage * A_STAGE), sb = smem_u32(sB + stage * B_STAGE);
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, A_STAGE + B_STAGE);
          tma_load_2d(sa, &tmA, fb, kb * BK, rt.row0);
          if constexpr (MODE == kUp8) {
            // 96 rows of W1 then the same 96 rows of W3
            tma_load_3d(sb, &tmB0, fb, kb * BK, n0, rt.e);
            tma_load_3d(sb + 96 * BK, &tmB1, fb, kb * BK, n0, rt.e);
          } else {
            tma_load_3d(sb, &tmB0, fb, kb * BK, n0, rt.e);
          }
        }
        // scale atoms: this lane gathers rows 32j + lane (j = 0..3) of A and
        // columns 128hb + 32j + lane (< 192) of B
        const uint32_t sfa_s = smem_u32(sSF + stage * SF_STAGE);
        const uint32_t sfb_s = sfa_s + 512;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int row = rt.row0 + 32 * j + lane;
          const bool v = row < args.R;
          cp_async4(sfa_s + 16 * lane + 4 * j,
                    args.sfa + (size_t)(v ? row : 0) * ksf + kb * 4, v);
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const int c = 128 * hb + 32 * j + lane;               // tile column
            const uint8_t* tab = args.sfb0;
            int n = n0 + c;
            if constexpr (MODE == kUp8) {
              if (c >= BN / 2) { tab = args.sfb1; n -= BN / 2; }  // W3 half
            }
            const bool bv = c < BN && n < args.N;
            cp_async4(sfb_s + 512 * hb + 16 * lane + 4 * j,
                      tab + ((size_t)rt.e * args.N + (bv ? n : 0)) * ksf + kb * 4, bv);
          }
        }
        cp_async_arrive_noinc(fb);
        __syncwarp();
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) drain_wait(smem_u32(&sh->full[s]), (last_par >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true, issued_any = false;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      if (!bounded_wait(smem_u32(&sh->tempty[acc]), acc_phase ^ 1u, &sh->abort_flag, args.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t dt = tmem + (uint32_t)(acc * kAccStride);
      for (int kb = 0; kb < args.kb_total; ++kb) {
        if (!bounded_wait(smem_u32(&sh->full[stage]), phase, &sh->abort_flag, args.status)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          // the scale bytes were written by cp.async (generic proxy); make them
          // visible to the tensor core's async proxy before tcgen05.cp reads them
          fence_proxy_async_smem();
          const uint32_t sfa_t = tmem + kSfCol0 + 12 * stage, sfb_t = sfa_t + 4;
          const uint32_t sf_s = smem_u32(sSF + stage * SF_STAGE);
          tmem_cp_warpx4(sfa_t, sdesc_atom(sf_s));
          tmem_cp_warpx4(sfb_t, sdesc_atom(sf_s + 512));          // B columns 0..127
          tmem_cp_warpx4(sfb_t + 4, sdesc_atom(sf_s + 1024));     // B columns 128..191
          const uint32_t sa = smem_u32(sA + stage * A_STAGE), sb = smem_u32(sB + stage * B_STAGE);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint64_t ad = sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sb + kk * 32, 16, 1024);
            mma_mxf8(dt, ad, bd, idesc_mxf8(BM, BN, kk), sfa_t, sfb_t, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&sh->empty[stage]));
        }
        issued_any = true;
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(smem_u32(&sh->tfull[acc]));
      __syncwarp();
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (!ok && issued_any && lane == 0) {
      mma_commit(smem_u32(&sh->drain));
      drain_wait(smem_u32(&sh->drain), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int lane_q = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stg = sStage + (warp - 2) * kStageBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const RowTile rt = decode_row_tile(t, args.E, args.R, s_off, s_ts);
      const int n0 = rt.n_idx * (MODE == kUp8 ? BN / 2 : BN);
      if (!bounded_wait(smem_u32(&sh->tfull[acc]), acc_phase, &sh->abort_flag, args.status)) break;
      tc_fence_after();
      epilogue8<MODE>(rt, n0, tmem + (uint32_t)(acc * kAccStride), lane_q, half, lane, stg, args,
                      &tmO0, &tmO1, &tmO2);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[acc]));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    stg_finish(lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

constexpr size_t smem_bytes8(int E) {
  return 1024 + (size_t)STAGES * (A_STAGE + B_STAGE + SF_STAGE) + (size_t)kEpiWarps * kStageBytes +
         sizeof(Shared) + 2 * (size_t)(E + 1) * 4;
}

template <int MODE>
int launch8(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& o0,
            const CUtensorMap& o1, const CUtensorMap& o2, const Args8& args, int grid, cudaStream_t s) {
  auto kern = grouped_mxfp8_kernel<MODE>;
  static bool attr_done[64] = {false};
  if (ensure_smem_attr(kern, smem_bytes8(kMaxExperts8), attr_done) != MOE_OK) return MOE_ERR_CUDA;
  (void)launch_pdl(kern, grid, kThreads, smem_bytes8(args.E), s, a, b0, b1, o0, o1, o2, args);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;
using namespace moe::gemm;

extern "C" int moe_grouped_swiglu_fwd_mxfp8(
    const uint8_t* xq, const uint8_t* xs, const int32_t* offsets, int R, int E, int d, int h,
    const uint8_t* w1q, const uint8_t* w1s, const uint8_t* w3q, const uint8_t* w3s,
    const uint8_t* w2q, const uint8_t* w2s, moe_bf16_t* h1, moe_bf16_t* h3, moe_bf16_t* a,
    uint8_t* aq, uint8_t* as, moe_bf16_t* yp, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (R < 0 || E < 1 || E > kMaxExperts || d <= 0 || h <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 128 != 0 || h % 128 != 0 || E > kMaxExperts8) return MOE_ERR_UNSUPPORTED;
  if (ws == nullptr || ws_bytes < kStatusBytes) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (R == 0) return MOE_OK;
  MOE_CHECK_PTR(xq); MOE_CHECK_PTR(offsets); MOE_CHECK_PTR(w1q); MOE_CHECK_PTR(w3q);
  MOE_CHECK_PTR(w2q); MOE_CHECK_PTR(h1); MOE_CHECK_PTR(h3); MOE_CHECK_PTR(aq);
  MOE_CHECK_PTR(yp);
  if (a != nullptr && !aligned16(a)) return MOE_ERR_INVALID_ARG;      // a may be NULL
  // scale tables are read 4 bytes at a time
  auto al4 = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!al4(xs) || !al4(w1s) || !al4(w3s) || !al4(w2s) || as == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUtensorMap mx, mw1, mw3, ma, mw2;
  if (!map2d(&mx, xq, d, R, BK, BM, U8, 1) || !map3d(&mw1, w1q, d, h, E, BK, BN / 2, U8, 1) ||
      !map3d(&mw3, w3q, d, h, E, BK, BN / 2, U8, 1) || !map2d(&ma, aq, h, R, BK, BM, U8, 1) ||
      !map3d(&mw2, w2q, h, d, E, BK, BN, U8, 1))
    return MOE_ERR_CUDA;
  Args8 g{};
  g.offsets = offsets; g.E = E; g.R = R; g.d = d; g.h = h; g.status = reinterpret_cast<int*>(ws);
  // up-projection: K = d, 96 columns of W1 and of W3 per tile
  g.K = d; g.kb_total = d / BK; g.n_tiles = (h + BN / 2 - 1) / (BN / 2); g.N = h;
  g.sfa = xs; g.sfb0 = w1s; g.sfb1 = w3s;
  g.out0 = h1; g.out1 = h3; g.out2 = a; g.aq = aq; g.as = as;
  CUtensorMap mo_h1, mo_h3, mo_a, mo_yp;
  if (!map2d_out(&mo_h1, h1, h, R, h) || !map2d_out(&mo_h3, h3, h, R, h) ||
      !map2d_out(&mo_a, a ? a : h1, h, R, h) || !map2d_out(&mo_yp, yp, d, R, d))
    return MOE_ERR_CUDA;
  int st = launch8<kUp8>(mx, mw1, mw3, mo_h1, mo_h3, mo_a, g, row_grid_upper(R, E, g.n_tiles), s);
  if (st != MOE_OK) return st;
  // down-projection: K = h
  Args8 g2 = g;
  g2.K = h; g2.kb_total = h / BK; g2.n_tiles = (d + BN - 1) / BN; g2.N = d;
  g2.sfa = as; g2.sfb0 = w2s; g2.sfb1 = w2s;
  g2.out0 = yp; g2.out1 = nullptr; g2.out2 = nullptr; g2.aq = nullptr; g2.as = nullptr;
  return launch8<kDown8>(ma, mw2, mw2, mo_yp, mo_yp, mo_yp, g2, row_grid_upper(R, E, g2.n_tiles), s);
}
