// Unpadded grouped SwiGLU GEMMs on tcgen05 tensor cores (forward and backward).
//
// "OLMo-core 3：MoE 训练栈让专家池越大、吞吐不再越慢", section "另外两处税：主机同步
// 与 padding": all small expert GEMMs are merged into one kernel schedule that
// runs every expert on exactly the row count the device route map gives, with
// no padding to a common capacity (no wasted FLOPs, no per-expert host
// launches).  The same page's layer map puts this in a CUTLASS grouped GEMM on
// B300; nothing here comes from CUTLASS: the kernel is written directly
// against tcgen05/TMEM/TMA for sm_103a.  The expert network (SwiGLU,
// W2(silu(x W1) * (x W3))) is the benchmark specification's reading; the
// pages only say "FFN".  The backward GEMMs are the Dgrad and Wgrad GEMMs
// named in the tutorial's DeepSeek-V3 paragraph (section "一个低精度格式，同时压三个地方").
//
// One persistent kernel template, five modes:
//   UP : [h1 | h3] = xp_e @ [W1[e] | W3[e]],  epilogue a = silu(h1) * h3
//   DOWN: yp = a_e @ W2[e]
//   DA : dA = dyp_e @ W2[e]^T, epilogue dh1 = dA*h3*silu'(h1), dh3 = dA*silu(h1)
//   DX : dxp = [dh1 | dh3]_e @ [W1[e] | W3[e]]^T   (K = 2h)
//   WG : dW1[e] = xp_e^T dh1_e, dW3[e] = xp_e^T dh3_e, dW2[e] = a_e^T dyp_e
//        (the reduction runs over the expert's own rows; K = n_e varies)
//
// Single-CTA tiles are 128 x 256 (BM x BN) with BK = 64; every CTA loops over
// tiles t = blockIdx.x, blockIdx.x + gridDim.x, ... in expert-major order
// (column blocks fastest, see decode_row_tile).  The row groups come from
// `offsets` read on the device: nothing is padded and the host never learns
// the row counts.  The CTA-pair kernel further down takes 256-row tiles.
//
// Warp roles (320 threads): warp 0 issues TMA loads into a 4-stage shared
// memory ring; warp 1 allocates 512 TMEM columns (two 128x256 fp32
// accumulators) and one of its lanes issues tcgen05.mma; warps 2-9 drain a
// finished accumulator (tcgen05.ld, two warps per TMEM lane quarter) while
// the next tile accumulates into the other one.  Every mbarrier wait is
// bounded: on timeout the kernel records MOE_DEV_WAIT_TIMEOUT, waits
// (bounded) for its own in-flight copies and MMAs, frees TMEM and returns.
#include "gemm_common.cuh"
#include "mx_common.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace gemm;

enum Mode : int { kUp = 0, kDown = 1, kDA = 2, kDX = 3, kWG = 4 };

constexpr int BM = 128, BN = 256, BK = 64;
// 4 k-block slots of A and B; a stage (one barrier wait and one commit on the
// MMA lane) holds KPS1 of them.  Two k-blocks a stage leave this kernel only
// two stages, and the lost latency cover costs more than the waits it saves
// (measured: DX at T = 16384, E = 128 410 -> 449 us), so one.
constexpr int SLOTS = 4, KPS1 = 1, STAGES = SLOTS / KPS1;
constexpr int A_STAGE = BM * BK * 2;            // 16 KB
constexpr int B_STAGE = BN * BK * 2;            // 32 KB
constexpr int SUB = 64 * 64 * 2;                // one 64x64 bf16 TMA box (8 KB)
constexpr int kTmemCols = 512;
struct GemmArgs {
  const int32_t* offsets;   // [E+1], device
  int E, R, d, h;
  int n_tiles;              // N tiles per expert (row-grouped modes)
  int kb_total;             // k-blocks per tile (row-grouped modes)
  int kb_split;             // DX: k-blocks taken from (dh1, W1) before (dh3, W3)
  uint16_t* out0;
  uint16_t* out1;
  uint16_t* out2;
  const uint16_t* in0;      // DA: h1
  const uint16_t* in1;      // DA: h3
  int ldo;                  // row stride (elements) of the row-grouped outputs
  int* status;
  // DA: when set, dh1 / dh3 also leave quantised along h for the MXFP8 dgrad
  // (E4M3 codes [R][h], E8M0 scales [R][h/32]; the blocks of the stored bf16)
  uint8_t* q0;
  uint8_t* q1;
  uint8_t* qs0;
  uint8_t* qs1;
  int wg_t1, wg_t2;         // WG: tiles per expert of dW1 (= dW3) and of dW2
  int wg_mt1, wg_mt2;       // WG: M tiles of dW1 and dW2
  const CUtensorMap* wg_maps;  // WG: [E][5] descriptors of xp, a, dh1, dh3, dyp
                               //     whose row extent ends at the expert's last row
  // WG on CTA pairs: the tile plan wgrad_maps_kernel writes from the offsets
  // (head words, then the order of the experts with rows, deepest first, then
  // the experts without rows).  Work unit u < whole is tile u of that order
  // (per tiles an expert); unit whole + v is k-chunk v % split of tile
  // whole + v / split, accumulated in fp32 into wg_part[v] (256 x 256).
  const int* wg_plan;
  float* wg_part;
};

struct Tile {
  int e, row0, rows, m0, n0, nkb, which, krow0, krows;
  int part;                 // WG pair units: fp32 partial slot, or -1 for a whole tile
};

using Shared = PipeShared<STAGES>;

// Row tiles of the single-CTA kernel (the weight-gradient GEMM runs on CTA
// pairs only, decode_pair_tile below).
template <int MODE>
__device__ __forceinline__ Tile decode_tile(int t, const GemmArgs& a, const int* s_off,
                                            const int* s_ts) {
  static_assert(MODE != kWG, "the weight-gradient GEMM runs on CTA pairs only");
  Tile tl{};
  const RowTile r = decode_row_tile(t, a.E, a.R, s_off, s_ts);
  tl.e = r.e;
  tl.row0 = r.row0;
  tl.rows = r.rows;
  tl.n0 = r.n_idx * (MODE == kUp ? BN / 2 : BN);
  tl.nkb = a.kb_total;
  return tl;
}

// wgrad only: MMAs for k-block kb of an expert, one per 16-row group that
// holds any of its rows.  The expert's own descriptors end at its last row,
// so TMA fills the rest of the last block with zeros.
__device__ __forceinline__ int wg_groups(const Tile& tl, int kb) {
  const int valid = tl.krows - kb * BK;
  return valid >= BK ? BK / 16 : (valid + 15) >> 4;
}

// wgrad only: the k-block a pair processes at loop step kb of its i-th unit.
// Every other deep tile of a pair (i odd; 32 k-blocks or more) runs its
// k-blocks from the last to the first, so a tile starts on the expert rows its
// predecessor read last, which the L2 still holds: dense_e8's wgrad reads 1128
// instead of 1209 MB from DRAM, in the same time.  (Shallow tiles' rows fit
// in the L2 anyway; reversing them cost 0.5%.)
__device__ __forceinline__ int wg_kblock(const Tile& tl, int i, int kb) {
  return (tl.nkb >= 32 && (i & 1)) ? tl.nkb - 1 - kb : kb;
}

// The i-th work unit of a pair.  WG deals its units (deepest experts first)
// in snake order, round i running over the pairs forwards when i is even and
// backwards when odd, so every pair's sum of tile depths comes out nearly the
// same (skew_e128: largest pair 1.03x the mean, against 1.18x round-robin in
// expert order); the row-grouped modes deal round-robin.
template <int MODE>
__device__ __forceinline__ int pair_unit(int i, int pair, int npairs) {
  if constexpr (MODE == kWG) return i * npairs + ((i & 1) ? npairs - 1 - pair : pair);
  else return i * npairs + pair;
}

template <int MODE>
__device__ __forceinline__ void issue_loads(const Tile& tl, int kb, uint32_t sa, uint32_t sb,
                                            uint32_t bar, const CUtensorMap* a0,
                                            const CUtensorMap* a1, const CUtensorMap* b0,
                                            const CUtensorMap* b1, const CUtensorMap* b2,
                                            const GemmArgs& a) {
  if constexpr (MODE == kUp) {
    tma_load_2d(sa, a0, bar, kb * BK, tl.row0);
    tma_load_3d(sb + 0 * SUB, b0, bar, tl.n0, kb * BK, tl.e);
    tma_load_3d(sb + 1 * SUB, b0, bar, tl.n0 + 64, kb * BK, tl.e);
    tma_load_3d(sb + 2 * SUB, b1, bar, tl.n0, kb * BK, tl.e);
    tma_load_3d(sb + 3 * SUB, b1, bar, tl.n0 + 64, kb * BK, tl.e);
  } else if constexpr (MODE == kDown) {
    tma_load_2d(sa, a0, bar, kb * BK, tl.row0);
#pragma unroll
    for (int c = 0; c < 4; ++c) tma_load_3d(sb + c * SUB, b0, bar, tl.n0 + 64 * c, kb * BK, tl.e);
  } else if constexpr (MODE == kDA) {
    tma_load_2d(sa, a0, bar, kb * BK, tl.row0);
    tma_load_3d(sb, b0, bar, kb * BK, tl.n0, tl.e);
  } else {  // kDX
    static_assert(MODE == kDX, "the weight-gradient GEMM runs on CTA pairs only");
    const bool second = kb >= a.kb_split;
    const int kk = (second ? kb - a.kb_split : kb) * BK;
    tma_load_2d(sa, second ? a1 : a0, bar, kk, tl.row0);
    tma_load_3d(sb, second ? b1 : b0, bar, kk, tl.n0, tl.e);
  }
}

// TMA descriptors of the epilogue's outputs (kernel parameters): UP h1, h3, a;
// DOWN yp; DA dh1, dh3; DX dxp; WG dW1, dW3, dW2 ([E, M, N] each).
struct OutMaps {
  const CUtensorMap *o0, *o1, *o2;
};

// DA with quantised outputs: this lane's row of a 32-column chunk, packed in
// bf16 (o), as one MXFP8 block: 32 E4M3 codes to q, the E8M0 byte to *s.  The
// block is the stored bf16 values, so the codes equal a separate quantising
// pass over dh1 / dh3 (moe_mxfp8_quantize_rows).
__device__ __forceinline__ void quantize_chunk_row(const uint4 (&o)[4], uint8_t* q, uint8_t* s) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(o);
  float v[32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[2 * i] = bf16_lo(w[i]);
    v[2 * i + 1] = bf16_hi(w[i]);
    amax = fmaxf(amax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
  }
  const int e = mx::block_exponent(amax);
  const float inv = mx::inv_scale(e);
  uint4 c[2];
  uint32_t* cw = reinterpret_cast<uint32_t*>(c);
#pragma unroll
  for (int i = 0; i < 8; ++i) cw[i] = mx::e4m3x4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
  st_v4(q, c[0]);
  st_v4(q + 16, c[1]);
  *s = (uint8_t)(e + 127);
}

// Epilogue of one tile for the 32 rows of this warp's TMEM lane quarter and
// the half `half` of the tile's columns (two warps share a lane quarter).
// Accumulator rows arrive one per lane (tcgen05.ld 32x32b) and leave through
// the warp's staging buffer `stg`: a 32 x 32 chunk whose 32 rows all belong to
// the tile goes out as one TMA store; a slice cut short by the end of an
// expert's rows is written by coalesced stores of its own rows only.
template <int MODE>
__device__ __forceinline__ void epilogue_tile(const Tile& tl, uint32_t tacc, int lane_q, int half,
                                              int lane, uint8_t* stg, const GemmArgs& a,
                                              const OutMaps& om) {
  const uint32_t tbase = tacc + ((uint32_t)(lane_q * 32) << 16);
  if constexpr (MODE == kWG) {
    const int M = tl.which == 2 ? a.h : a.d;
    const int N = tl.which == 2 ? a.d : a.h;
    const int r0 = tl.m0 + lane_q * 32;               // first row of this warp's slice
    const int nrows = min(32, M - r0);
#pragma unroll 1
    for (int c = half * 4; c < half * 4 + 4; ++c) {
      float v[32];
      if (tl.nkb > 0) {
        uint32_t q[32];
        tmem_ld32(tbase + c * 32, q);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(q[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      const int col = tl.n0 + c * 32;
      if (col < N && nrows > 0)
        store_chunk_tma3(stg, v, lane, tl.which == 0 ? om.o0 : (tl.which == 1 ? om.o1 : om.o2),
                         col, r0, tl.e);
    }
  } else {
    const int nrows = min(32, tl.rows - lane_q * 32);  // rows of this slice in the segment
    const size_t r0 = (size_t)tl.row0 + (nrows > 0 ? lane_q * 32 : 0);
    const bool whole = nrows == 32;                     // TMA store of the whole slice
    if constexpr (MODE == kUp) {
#pragma unroll 1
      for (int c = half * 2; c < half * 2 + 2; ++c) {
        uint32_t q1[32], q3[32];
        tmem_ld32(tbase + c * 32, q1);
        tmem_ld32(tbase + 128 + c * 32, q3);
        tmem_ld_wait();
        const int col = tl.n0 + c * 32;
        if (col < a.h) {
          float h1[32], h3[32], av[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            h1[i] = __uint_as_float(q1[i]);
            h3[i] = __uint_as_float(q3[i]);
            av[i] = silu_f(h1[i]) * h3[i];
          }
          if (whole) {
            store_chunk_tma(stg, h1, lane, om.o0, col, (int)r0);
            store_chunk_tma(stg, h3, lane, om.o1, col, (int)r0);
            store_chunk_tma(stg, av, lane, om.o2, col, (int)r0);
          } else {
            stg_acquire(lane);
            store_chunk(stg, h1, lane, a.out0 + r0 * a.ldo + col, a.ldo, nrows);
            store_chunk(stg, h3, lane, a.out1 + r0 * a.ldo + col, a.ldo, nrows);
            store_chunk(stg, av, lane, a.out2 + r0 * a.ldo + col, a.ldo, nrows);
          }
        }
      }
    } else if constexpr (MODE == kDA) {
      // the h1/h3 chunk loads of chunk c+1 are in flight while chunk c is computed
      const int c0 = half * 4;
      uint4 p1[4], p3[4];
      {
        const int col = tl.n0 + c0 * 32;
        load_chunk(p1, a.in0 + r0 * a.ldo + col, a.ldo, lane, col < a.h ? nrows : 0);
        load_chunk(p3, a.in1 + r0 * a.ldo + col, a.ldo, lane, col < a.h ? nrows : 0);
      }
#pragma unroll 1
      for (int c = c0; c < c0 + 4; ++c) {
        uint32_t q[32];
        tmem_ld32(tbase + c * 32, q);
        const int col = tl.n0 + c * 32;
        uint32_t w1[16], w3[16];                 // h1, h3 of this row, bf16 pairs
        if (col < a.h) {
          chunk_to_row(p1, stg, lane, w1);
          chunk_to_row(p3, stg, lane, w3);
        }
        if (c + 1 < c0 + 4) {                  // prefetch buffers are free again
          const int ncol = col + 32;
          load_chunk(p1, a.in0 + r0 * a.ldo + ncol, a.ldo, lane, ncol < a.h ? nrows : 0);
          load_chunk(p3, a.in1 + r0 * a.ldo + ncol, a.ldo, lane, ncol < a.h ? nrows : 0);
        }
        tmem_ld_wait();
        if (col < a.h) {
          float g1[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float h1 = (i & 1) ? bf16_hi(w1[i >> 1]) : bf16_lo(w1[i >> 1]);
            const float h3 = (i & 1) ? bf16_hi(w3[i >> 1]) : bf16_lo(w3[i >> 1]);
            const float da = __uint_as_float(q[i]);
            const float sg = sigmoid_f(h1);
            g1[i] = da * h3 * sg * (1.f + h1 * (1.f - sg));
            q[i] = __float_as_uint(da * h1 * sg);                    // dh3 in place
          }
          // (plain coalesced stores: two TMA stores a chunk through the one
          // staging buffer made this epilogue slower)
          store_chunk(stg, g1, lane, a.out0 + r0 * a.ldo + col, a.ldo, nrows);
          store_chunk(stg, reinterpret_cast<const float*>(q), lane, a.out1 + r0 * a.ldo + col,
                      a.ldo, nrows);
          if (a.q0 != nullptr && lane < nrows) {
            uint4 o1[4], o3[4];
            pack_row32(g1, o1);
            pack_row32(reinterpret_cast<const float*>(q), o3);
            const size_t rq = (r0 + lane) * (size_t)a.h + col, rs = (r0 + lane) * (size_t)(a.h / 32) + col / 32;
            quantize_chunk_row(o1, a.q0 + rq, a.qs0 + rs);
            quantize_chunk_row(o3, a.q1 + rq, a.qs1 + rs);
          }
        }
      }
    } else {  // kDown, kDX: plain bf16 store of the accumulator
      const int N = a.d;
#pragma unroll 1
      for (int c = half * 4; c < half * 4 + 4; ++c) {
        uint32_t q[32];
        tmem_ld32(tbase + c * 32, q);
        tmem_ld_wait();
        const int col = tl.n0 + c * 32;
        if (col < N) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(q[i]);
          if (whole) {
            store_chunk_tma(stg, v, lane, om.o0, col, (int)r0);
          } else {
            stg_acquire(lane);
            store_chunk(stg, v, lane, a.out0 + r0 * a.ldo + col, a.ldo, nrows);
          }
        }
      }
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                    const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmO0,
                    const __grid_constant__ CUtensorMap tmO1, const __grid_constant__ CUtensorMap tmO2,
                    const GemmArgs args) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + SLOTS * A_STAGE;
  uint8_t* sStage = sB + SLOTS * B_STAGE;                    // kEpiWarps x kStageBytes
  Shared* sh = reinterpret_cast<Shared*>(sStage + kEpiWarps * kStageBytes);
  int* s_off = reinterpret_cast<int*>(sh + 1);
  int* s_ts = s_off + (args.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- set-up: tile table from the device offsets, barriers, TMEM
  for (int i = threadIdx.x; i <= args.E; i += blockDim.x) s_off[i] = __ldg(args.offsets + i);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
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
  if ((int)blockIdx.x >= total) return;      // uniform across the CTA; no TMEM taken yet

  if (warp == 1) {
    tmem_alloc(smem_u32(&sh->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA0); prefetch_tmap(&tmA1); prefetch_tmap(&tmB0);
    prefetch_tmap(&tmB1); prefetch_tmap(&tmB2);
    prefetch_tmap(&tmO0); prefetch_tmap(&tmO1); prefetch_tmap(&tmO2);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // the whole warp walks the schedule (converged); lane 0 issues the copies
    int stage = 0;
    uint32_t phase = 0, issued = 0, last_par = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = decode_tile<MODE>(t, args, s_off, s_ts);
      for (int kb0 = 0; kb0 < tl.nkb; kb0 += KPS1) {
        const int nk = min(KPS1, tl.nkb - kb0);
        if (!bounded_wait(smem_u32(&sh->empty[stage]), phase ^ 1u, &sh->abort_flag, args.status)) { ok = false; break; }
        if (lane == 0) {
          const uint32_t fb = smem_u32(&sh->full[stage]);
          mbar_arrive_expect_tx(fb, nk * (A_STAGE + B_STAGE));
          for (int j = 0; j < nk; ++j) {
            const int q = stage * KPS1 + j;
            issue_loads<MODE>(tl, kb0 + j, smem_u32(sA + q * A_STAGE), smem_u32(sB + q * B_STAGE),
                              fb, &tmA0, &tmA1, &tmB0, &tmB1, &tmB2, args);
          }
        }
        __syncwarp();
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      // let every copy this CTA started land before shared memory goes away
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) drain_wait(smem_u32(&sh->full[s]), (last_par >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    constexpr bool b_mn = (MODE == kUp || MODE == kDown);   // A (rows) is always K-major
    constexpr uint32_t idesc = idesc_bf16(BM, BN, false, b_mn);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true, issued_any = false;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = decode_tile<MODE>(t, args, s_off, s_ts);
      if (!bounded_wait(smem_u32(&sh->tempty[acc]), acc_phase ^ 1u, &sh->abort_flag, args.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t dt = tmem + (uint32_t)(acc * BN);
      if (tl.nkb == 0) {
        if (lane == 0) mbar_arrive(smem_u32(&sh->tfull[acc]));
      } else {
        for (int kb0 = 0; kb0 < tl.nkb; kb0 += KPS1) {
          constexpr int nkk = BK / 16;
          const int nk = min(KPS1, tl.nkb - kb0);
          if (!bounded_wait(smem_u32(&sh->full[stage]), phase, &sh->abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            for (int j = 0; j < nk; ++j) {
              const int kb = kb0 + j, q = stage * KPS1 + j;
              const uint32_t sa = smem_u32(sA + q * A_STAGE);
              const uint32_t sb = smem_u32(sB + q * B_STAGE);
              for (int kk = 0; kk < nkk; ++kk) {
                uint64_t bd;
                const uint64_t ad = sdesc_sw128(sa + kk * 32, 16, 1024);
                if constexpr (b_mn) bd = sdesc_sw128(sb + kk * 2048, SUB, 1024);
                else bd = sdesc_sw128(sb + kk * 32, 16, 1024);
                mma_f16(dt, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
              }
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
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (!ok && issued_any && lane == 0) {
      // wait for the tensor core to finish reading shared memory / writing TMEM
      mma_commit(smem_u32(&sh->drain));
      drain_wait(smem_u32(&sh->drain), 0);
    }
  } else {
    // --------------------------------------------------------------- epilogue
    const int lane_q = warp & 3;          // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;     // which half of the tile's columns
    const OutMaps om{&tmO0, &tmO1, &tmO2};
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode_tile<MODE>(t, args, s_off, s_ts);
      if (!bounded_wait(smem_u32(&sh->tfull[acc]), acc_phase, &sh->abort_flag, args.status)) break;
      tc_fence_after();
      epilogue_tile<MODE>(tl, tmem + (uint32_t)(acc * BN), lane_q, half, lane,
                          sStage + (warp - 2) * kStageBytes, args, om);
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

// ------------------------------------------------------------ CTA pairs
// The same GEMMs on pairs of CTAs (2-CTA clusters) with tcgen05 MMAs of
// M = 256, N = 256: CTA r of a pair stages rows [128r, 128r + 128) of the
// tile's A operand and columns [128r, 128r + 128) of its B operand for every
// 64-deep k-block, i.e. 32 KB per k-block for a 128 x 256 share of the output
// (48 KB on a single CTA).  Both CTAs' copies complete on the even CTA's
// `full` barrier; that CTA issues the MMAs and commits them to the `empty`
// and `tfull` barriers of both CTAs; every epilogue warp of the pair releases
// an accumulator on the even CTA's `tempty` barrier.
//   UP, DOWN, DX:      256-row tiles of an expert's rows; UP splits B into
//                      W1 columns (even CTA) and W3 columns (odd CTA), so the
//                      accumulator keeps the single-CTA column layout.
//   DA:                256-row tiles like DOWN, 5 stages; a ring loader warp
//                      brings the h1 / h3 the epilogue needs into shared
//                      memory by TMA ahead of time (see epilogue_da_ring); no
//                      staging buffers (its stores go out of the ring slots),
//                      and at most pair_max_experts<kDA>() experts (the tile
//                      table shares the 227 KB).
//   WG:                256 x 256 tiles of dW over the expert's rows; units
//                      from a device-built plan, and a warp that stores the
//                      empty experts' zero tiles.
constexpr int P_SLOTS = 6;                            // 32 KB k-block slots (DA: 5)
constexpr int P_HALF = 128 * BK * 2;                  // 16 KB: 128 rows x 64 deep
constexpr int P_TILE = 256;
// DA's epilogue ring: slot = one 32-column chunk of h1 and of h3 for the
// CTA's 128 rows (64-byte swizzled 32 x 128 boxes)
constexpr int kRingSlots = 4;
constexpr int kRingChunk = 128 * 32 * 2;              // 8 KB
constexpr int kRingSlotBytes = 2 * kRingChunk;
// A stage is one barrier wait and one commit on the MMA lane, each of which
// keeps the issuing thread off the tensor pipe for about a short MMA's time
// (measured on the GB300 with operands resident: a pair loop with one wait and
// two commits per 4-MMA k-block issues at 0.88 of the bf16 rate, with one of
// each per 8 MMAs at the full rate), so the pair GEMMs stage two k-blocks at
// a time: 3 stages of 2 k-block slots.  DA keeps 5 one-k-block stages next to
// its h1/h3 ring (2 stages of 2 slots there: 203 -> 234 us at T = 16384,
// E = 8).
template <int MODE> __host__ __device__ constexpr int pair_kps() { return MODE == kDA ? 1 : 2; }
template <int MODE> __host__ __device__ constexpr int pair_stages() { return MODE == kDA ? 5 : P_SLOTS / 2; }
template <int MODE> __host__ __device__ constexpr int pair_slots() { return pair_stages<MODE>() * pair_kps<MODE>(); }
template <int MODE> __host__ __device__ constexpr int pair_ring_bytes() { return MODE == kDA ? kRingSlots * kRingSlotBytes : 0; }
template <int MODE> __host__ __device__ constexpr int pair_stage_bytes() { return MODE == kDA ? 0 : kEpiWarps * kStageBytes; }
// WG: a 32 x 32 bf16 box of zeros, the source of every store of an empty expert's dW tiles
template <int MODE> __host__ __device__ constexpr int pair_zero_bytes() { return MODE == kWG ? 2048 : 0; }
template <int MODE> using PairSharedT = PipeShared<pair_stages<MODE>()>;
constexpr int kPairThreads = kThreads + 32;           // + DA's ring loader / WG's zero-tile warp

// WG: s_ts holds the plan's expert order (deepest first) and wg = {whole,
// split} its unit counts; the row-grouped modes ignore wg.
template <int MODE>
__device__ __forceinline__ Tile decode_pair_tile(int t, const GemmArgs& a, const int* s_off,
                                                 const int* s_ts, const int* wg = nullptr) {
  Tile tl{};
  tl.part = -1;
  if constexpr (MODE == kWG) {
    const int whole = wg[0], split = wg[1];
    int chunk = 0;
    if (split > 0 && t >= whole) {
      const int v = t - whole;
      tl.part = v;
      chunk = v % split;
      t = whole + v / split;
    }
    const int per = 2 * a.wg_t1 + a.wg_t2;
    const int rank = t / per;
    tl.e = s_ts[rank];
    int l = t - rank * per;
    int mt;
    if (l < a.wg_t1) { tl.which = 0; mt = a.wg_mt1; }
    else if (l < 2 * a.wg_t1) { tl.which = 1; l -= a.wg_t1; mt = a.wg_mt1; }
    else { tl.which = 2; l -= 2 * a.wg_t1; mt = a.wg_mt2; }
    tl.m0 = (l % mt) * P_TILE;
    tl.n0 = (l / mt) * P_TILE;
    int lo = s_off[tl.e], hi = s_off[tl.e + 1];
    lo = max(0, min(lo, a.R));
    hi = max(lo, min(hi, a.R));
    tl.krow0 = lo;
    tl.krows = hi - lo;
    tl.nkb = (tl.krows + BK - 1) / BK;
    if (tl.part >= 0) {
      // k-blocks [kb0, kb1) of the expert's rows
      const int kc = (tl.nkb + split - 1) / split;
      const int kb0 = min(tl.nkb, chunk * kc), kb1 = min(tl.nkb, kb0 + kc);
      tl.krow0 = lo + kb0 * BK;
      tl.krows = max(0, min(tl.krows - kb0 * BK, (kb1 - kb0) * BK));
      tl.nkb = kb1 - kb0;
    }
  } else {
    const RowTile r = decode_row_tile<P_TILE>(t, a.E, a.R, s_off, s_ts);
    tl.e = r.e;
    tl.row0 = r.row0;
    tl.rows = r.rows;
    tl.n0 = r.n_idx * (MODE == kUp ? BN / 2 : BN);
    tl.nkb = a.kb_total;
  }
  return tl;
}

// This CTA's share of k-block kb: 16 KB of A at sa, 16 KB of B at sb, both
// counted on the even CTA's barrier `fb`.
template <int MODE>
__device__ __forceinline__ void issue_loads_pair(const Tile& tl, int kb, uint32_t rank, uint32_t sa,
                                                 uint32_t sb, uint32_t fb, const CUtensorMap* a0,
                                                 const CUtensorMap* a1, const CUtensorMap* b0,
                                                 const CUtensorMap* b1, const GemmArgs& a) {
  const int r128 = 128 * (int)rank;
  if constexpr (MODE == kUp) {
    const CUtensorMap* bm = rank == 0 ? b0 : b1;           // W1 or W3 columns n0 .. n0+127
    tma_load_2d_pair(sa, a0, fb, kb * BK, tl.row0 + r128);
    tma_load_3d_pair(sb, bm, fb, tl.n0, kb * BK, tl.e);
    tma_load_3d_pair(sb + SUB, bm, fb, tl.n0 + 64, kb * BK, tl.e);
  } else if constexpr (MODE == kDown) {
    tma_load_2d_pair(sa, a0, fb, kb * BK, tl.row0 + r128);
    tma_load_3d_pair(sb, b0, fb, tl.n0 + r128, kb * BK, tl.e);
    tma_load_3d_pair(sb + SUB, b0, fb, tl.n0 + r128 + 64, kb * BK, tl.e);
  } else if constexpr (MODE == kDA) {
    (void)a1; (void)b1;
    tma_load_2d_pair(sa, a0, fb, kb * BK, tl.row0 + r128);
    tma_load_3d_pair(sb, b0, fb, kb * BK, tl.n0 + r128, tl.e);
  } else if constexpr (MODE == kDX) {
    const bool second = kb >= a.kb_split;
    const int kk = (second ? kb - a.kb_split : kb) * BK;
    tma_load_2d_pair(sa, second ? a1 : a0, fb, kk, tl.row0 + r128);
    tma_load_3d_pair(sb, second ? b1 : b0, fb, kk, tl.n0 + r128, tl.e);
  } else {  // kWG: the expert's own descriptors (rows past its end read as 0)
    const CUtensorMap* em = a.wg_maps + (size_t)tl.e * kWgradMaps;
    const CUtensorMap* am = em + (tl.which == 2 ? 1 : 0);
    const CUtensorMap* bm = em + 2 + tl.which;
    const int y = tl.krow0 + kb * BK;
    tma_load_2d_pair(sa, am, fb, tl.m0 + r128, y);
    tma_load_2d_pair(sa + SUB, am, fb, tl.m0 + r128 + 64, y);
    tma_load_2d_pair(sb, bm, fb, tl.n0 + r128, y);
    tma_load_2d_pair(sb + SUB, bm, fb, tl.n0 + r128 + 64, y);
  }
}

// DA epilogue on CTA pairs.  The ring loader warp streams, tile after tile,
// the 8 column chunks of the CTA's 128 rows of h1 and h3 into ring slots
// (slot g % kRingSlots for chunk g of the sequence); the warps of half h take
// chunks h, h + 2, h + 4, h + 6.  Each warp reads its 32 rows of the chunk
// (row r of a slot box at r * 64 bytes, 16-byte piece c at c ^ ((r >> 1) & 3)),
// forms dh1, dh3 with the accumulator, writes them back over its rows of the
// slot and stores them from there by TMA (a warp whose rows end inside the
// chunk writes its rows directly); the slot is released to the loader once
// the copy engine has read it.  rn = chunks of the sequence before this tile.
__device__ __forceinline__ bool epilogue_da_ring(const Tile& tl, uint32_t tacc, int lane_q, int half,
                                                 int lane, uint8_t* ring, uint64_t* rfull,
                                                 uint64_t* rempty, int* abort_flag, uint32_t rn,
                                                 const GemmArgs& a, const OutMaps& om) {
  const uint32_t tbase = tacc + ((uint32_t)(lane_q * 32) << 16);
  const int nrows = min(32, tl.rows - lane_q * 32);   // this warp's rows in the expert (may be <= 0)
  const int r0 = tl.row0 + lane_q * 32;
  const int x = (lane >> 1) & 3;
#pragma unroll 1
  for (int s = 0; s < 4; ++s) {
    const int c = 2 * s + half;
    const uint32_t g = rn + (uint32_t)c;
    const int slot = (int)(g % kRingSlots);
    if (!bounded_wait(smem_u32(&rfull[slot]), (g / kRingSlots) & 1u, abort_flag, a.status)) return false;
    uint8_t* p1 = ring + slot * kRingSlotBytes + lane_q * 2048 + lane * 64;
    uint8_t* p3 = p1 + kRingChunk;
    uint32_t w1[16], w3[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 t1 = *reinterpret_cast<const uint4*>(p1 + 16 * (i ^ x));
      const uint4 t3 = *reinterpret_cast<const uint4*>(p3 + 16 * (i ^ x));
      w1[4 * i] = t1.x; w1[4 * i + 1] = t1.y; w1[4 * i + 2] = t1.z; w1[4 * i + 3] = t1.w;
      w3[4 * i] = t3.x; w3[4 * i + 1] = t3.y; w3[4 * i + 2] = t3.z; w3[4 * i + 3] = t3.w;
    }
    uint32_t q[32];
    tmem_ld32(tbase + c * 32, q);
    tmem_ld_wait();
    float g1[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float h1 = (i & 1) ? bf16_hi(w1[i >> 1]) : bf16_lo(w1[i >> 1]);
      const float h3 = (i & 1) ? bf16_hi(w3[i >> 1]) : bf16_lo(w3[i >> 1]);
      const float da = __uint_as_float(q[i]);
      const float sg = sigmoid_f(h1);
      g1[i] = da * h3 * sg * (1.f + h1 * (1.f - sg));
      q[i] = __float_as_uint(da * h1 * sg);                      // dh3 in place
    }
    uint4 o1[4], o3[4];
    pack_row32(g1, o1);
    pack_row32(reinterpret_cast<const float*>(q), o3);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      *reinterpret_cast<uint4*>(p1 + 16 * (i ^ x)) = o1[i];
      *reinterpret_cast<uint4*>(p3 + 16 * (i ^ x)) = o3[i];
    }
    fence_proxy_async_smem();
    __syncwarp();
    const int col = tl.n0 + c * 32;
    if (col < a.h && nrows > 0) {
      if (nrows == 32) {
        if (lane == 0) {
          uint8_t* b1 = ring + slot * kRingSlotBytes + lane_q * 2048;
          tma_store_2d(om.o0, smem_u32(b1), col, r0);
          tma_store_2d(om.o1, smem_u32(b1 + kRingChunk), col, r0);
          bulk_commit();
        }
      } else if (lane < nrows) {
        uint16_t* d1 = a.out0 + (size_t)(r0 + lane) * a.ldo + col;
        uint16_t* d3 = a.out1 + (size_t)(r0 + lane) * a.ldo + col;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          st_v4(d1 + 8 * i, o1[i]);
          st_v4(d3 + 8 * i, o3[i]);
        }
      }
      if (a.q0 != nullptr && lane < nrows) {
        const size_t rq = (size_t)(r0 + lane) * a.h + col, rs = (size_t)(r0 + lane) * (a.h / 32) + col / 32;
        quantize_chunk_row(o1, a.q0 + rq, a.qs0 + rs);
        quantize_chunk_row(o3, a.q1 + rq, a.qs1 + rs);
      }
    }
    if (lane == 0) {
      bulk_wait_read_all();
      mbar_arrive(smem_u32(&rempty[slot]));
    }
    __syncwarp();
  }
  return true;
}

// Plain bf16 epilogue of a pair tile (WG, DOWN, DX) that frees the
// accumulator first: the warp's four 32-column chunks go to registers (128 a
// thread), the warp releases the accumulator to the MMA issuer, and only then
// stores the chunks, so the MMAs of the tile after next never wait for this
// tile's stores (T = 16384, d = 2048, h = 1024: DOWN 167 -> 162-165 us and DX
// 302-304 -> 300 us at E = 8, both about 4 us less at E = 128; the kernel
// then holds 163-168 registers a thread, one CTA an SM as before).
template <int MODE>
__device__ __forceinline__ void epilogue_tile_early(const Tile& tl, uint32_t tacc, int lane_q, int half,
                                                    int lane, uint8_t* stg, const GemmArgs& a,
                                                    const OutMaps& om, uint32_t tempty_leader) {
  const uint32_t tbase = tacc + ((uint32_t)(lane_q * 32) << 16);
  uint32_t q[4][32];
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld32(tbase + (half * 4 + c) * 32, q[c]);
  tmem_ld_wait();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive_cluster(tempty_leader);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int col = tl.n0 + (half * 4 + c) * 32;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(q[c][i]);
    if constexpr (MODE == kWG) {
      const int M = tl.which == 2 ? a.h : a.d;
      const int N = tl.which == 2 ? a.d : a.h;
      const int r0 = tl.m0 + lane_q * 32;
      const int nrows = min(32, M - r0);
      if (col < N && nrows > 0)
        store_chunk_tma3(stg, v, lane, tl.which == 0 ? om.o0 : (tl.which == 1 ? om.o1 : om.o2), col, r0, tl.e);
    } else {
      const int nrows = min(32, tl.rows - lane_q * 32);
      const size_t r0 = (size_t)tl.row0 + (nrows > 0 ? lane_q * 32 : 0);
      if (col < a.d) {
        if (nrows == 32) {
          store_chunk_tma(stg, v, lane, om.o0, col, (int)r0);
        } else {
          stg_acquire(lane);
          store_chunk(stg, v, lane, a.out0 + r0 * a.ldo + col, a.ldo, nrows);
        }
      }
    }
  }
}

// A whole dW tile of an expert with no rows: this warp's 32 rows x 4 chunks of
// 32 columns are TMA-stored from a shared box of zeros (no accumulator, no
// staging); lane 0 issues the stores as one bulk group.
__device__ __forceinline__ void epilogue_zero_tile(const Tile& tl, int lane_q, int half, int lane,
                                                   const uint8_t* zero, const GemmArgs& a,
                                                   const OutMaps& om) {
  const int M = tl.which == 2 ? a.h : a.d;
  const int N = tl.which == 2 ? a.d : a.h;
  const int r0 = tl.m0 + lane_q * 32;
  if (lane == 0 && r0 < M) {
    const CUtensorMap* map = tl.which == 0 ? om.o0 : (tl.which == 1 ? om.o1 : om.o2);
#pragma unroll 1
    for (int c = half * 4; c < half * 4 + 4; ++c) {
      const int col = tl.n0 + c * 32;
      if (col < N) tma_store_3d(map, smem_u32(zero), col, r0, tl.e);
    }
    bulk_commit();
  }
  __syncwarp();
}

// A K-chunk of a split wgrad tile: this CTA's 128 rows x 256 columns of the
// fp32 accumulator (zeros for an empty chunk) to partial slot tl.part; each
// lane writes its row's 32 values of a chunk as 128 contiguous bytes.
__device__ __forceinline__ void epilogue_partial(const Tile& tl, uint32_t tacc, int lane_q, int half,
                                                 int lane, uint32_t rank, const GemmArgs& a) {
  const uint32_t tbase = tacc + ((uint32_t)(lane_q * 32) << 16);
  const int row = 128 * (int)rank + lane_q * 32 + lane;
  float* dst = a.wg_part + (size_t)tl.part * (P_TILE * P_TILE) + (size_t)row * P_TILE;
#pragma unroll 1
  for (int c = half * 4; c < half * 4 + 4; ++c) {
    uint32_t q[32];
    if (tl.nkb > 0) {
      tmem_ld32(tbase + c * 32, q);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) q[i] = 0u;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      st_v4(dst + c * 32 + 4 * i, make_uint4(q[4 * i], q[4 * i + 1], q[4 * i + 2], q[4 * i + 3]));
  }
}

// Sum of the K-chunks of every split wgrad tile, in chunk order (so the
// result does not depend on timing), rounded once to bf16.  The plan says how
// many tiles were split (none: every block returns at once); block b takes
// row b of the split tiles (and b + gridDim.x, ..), thread = one column.
__global__ void __launch_bounds__(P_TILE) wgrad_fixup_kernel(const GemmArgs a) {
  pdl_enter();
  const int* plan = a.wg_plan;
  const int whole = plan[2], split = plan[3], units = plan[4];
  if (split <= 0 || a.wg_part == nullptr) return;
  const int L = (units - whole) / split;
  const int per = 2 * a.wg_t1 + a.wg_t2;
  const int col = threadIdx.x;
  for (int b = blockIdx.x; b < L * P_TILE; b += gridDim.x) {
    const int i = b / P_TILE, r = b % P_TILE;
    const int t = whole + i;
    const int e = plan[kWgradPlanHead + t / per];
    int l = t % per, which, mt;
    if (l < a.wg_t1) { which = 0; mt = a.wg_mt1; }
    else if (l < 2 * a.wg_t1) { which = 1; l -= a.wg_t1; mt = a.wg_mt1; }
    else { which = 2; l -= 2 * a.wg_t1; mt = a.wg_mt2; }
    const int m = (l % mt) * P_TILE + r, n = (l / mt) * P_TILE + col;
    const int M = which == 2 ? a.h : a.d, N = which == 2 ? a.d : a.h;
    if (m >= M || n >= N) continue;
    const float* src = a.wg_part + (size_t)i * split * (P_TILE * P_TILE) + (size_t)r * P_TILE + col;
    float acc = 0.f;
    for (int c = 0; c < split; ++c) acc += src[(size_t)c * (P_TILE * P_TILE)];
    uint16_t* out = which == 0 ? a.out0 : (which == 1 ? a.out1 : a.out2);
    out[((size_t)e * M + m) * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
  }
}

// The wgrad tile plan, from the offsets (one CTA of 1024 threads): the experts with rows in
// order of decreasing k-block count (ties: lower expert first), those without
// rows in expert order, and the units.  Thread e ranks expert e against all
// others (E <= 1024).  The last round of whole tiles holds the shallowest
// expert's tiles (2L <= npairs < tiles per expert); when it keeps at most
// half of the pairs busy, its L tiles are split along K into S chunks (L * S
// <= npairs, at most parts_max partial tiles, 4 or more of that expert's
// k-blocks a chunk).
__device__ __forceinline__ void wgrad_plan(const int32_t* __restrict__ offsets, int E, int R, int per,
                                           int npairs, int parts_max, int* __restrict__ plan) {
  __shared__ int s_kb[kMaxExperts];
  __shared__ int s_nc;
  if (threadIdx.x == 0) s_nc = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int lo = max(0, min(__ldg(offsets + e), R));
    const int hi = max(lo, min(__ldg(offsets + e + 1), R));
    s_kb[e] = (hi - lo + BK - 1) / BK;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int k = s_kb[e];
    int rank = 0;
    if (k > 0) {
      for (int j = 0; j < E; ++j) {
        const int kj = s_kb[j];
        rank += (kj > k) || (kj == k && j < e);
      }
      plan[kWgradPlanHead + rank] = e;
      atomicAdd(&s_nc, 1);
    } else {
      for (int j = 0; j < e; ++j) rank += s_kb[j] == 0;
      plan[kWgradPlanHead + E + rank] = e;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int nc = s_nc;
    const long long tiles = (long long)nc * per;
    const long long L = tiles % npairs;
    int whole = (int)tiles, split = 0, units = (int)tiles;
    if (L > 0 && 2 * L <= npairs && parts_max > 0 && nc > 0) {
      long long S = npairs / L;
      S = S < parts_max / L ? S : parts_max / L;
      const int kb_last = s_kb[plan[kWgradPlanHead + nc - 1]];
      S = S < kb_last / 4 ? S : kb_last / 4;
      if (S >= 2) {
        whole = (int)(tiles - L);
        split = (int)S;
        units = (int)(whole + L * S);
      }
    }
    plan[0] = nc;
    plan[1] = E - nc;
    plan[2] = whole;
    plan[3] = split;
    plan[4] = units;
    plan[5] = (E - nc) * per;
  }
}

template <int MODE>
__global__ void __launch_bounds__(kPairThreads, 1)
pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                 const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                 const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1,
                 const __grid_constant__ CUtensorMap tmO2, const GemmArgs args) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  constexpr int PS = pair_stages<MODE>(), KPS = pair_kps<MODE>();
  using PairShared = PairSharedT<MODE>;
  // PS * KPS k-block slots of A, then of B (slot q = stage * KPS + j)
  uint8_t* sB = smem + PS * KPS * P_HALF;
  uint8_t* ring = sB + PS * KPS * P_HALF;                    // DA only
  uint8_t* sStage = ring + pair_ring_bytes<MODE>();                 // not DA
  uint8_t* sZero = sStage + pair_stage_bytes<MODE>();               // WG only
  PairShared* sh = reinterpret_cast<PairShared*>(sZero + pair_zero_bytes<MODE>());
  int* s_off = reinterpret_cast<int*>(sh + 1);
  int* s_ts = s_off + (args.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  for (int i = threadIdx.x; i <= args.E; i += blockDim.x) s_off[i] = __ldg(args.offsets + i);
  if constexpr (MODE == kWG) {
    for (int i = threadIdx.x; i < pair_zero_bytes<MODE>() / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(sZero)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();              // the zeros are read by TMA stores
  }
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < PS; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&sh->tfull[s]), 1);
      mbar_init(smem_u32(&sh->tempty[s]), 2 * kEpiWarps);
    }
    for (int s = 0; s < kRingSlots; ++s) {
      mbar_init(smem_u32(&sh->rfull[s]), 1);
      mbar_init(smem_u32(&sh->rempty[s]), 4);              // the 4 warps of one half
    }
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if constexpr (MODE == kWG) {
    // the device-built plan: units, K-split, zero tiles; the expert order
    // goes where the row-grouped modes keep their tile table
    if (threadIdx.x == 0) {
      sh->total_tiles = args.wg_plan[4];
      sh->wg_whole = args.wg_plan[2];
      sh->wg_split = args.wg_plan[3];
      sh->wg_zero = args.wg_plan[5];
    }
    const int nc = min(args.wg_plan[0], args.E);
    for (int i = threadIdx.x; i < nc; i += blockDim.x) s_ts[i] = args.wg_plan[kWgradPlanHead + i];
  } else {
    if (warp == 0) {
      const int n = build_row_tile_table<P_TILE>(s_off, s_ts, args.E, args.R, args.n_tiles, lane);
      if (lane == 0) sh->total_tiles = n;
    }
  }
  // both CTAs' barriers exist before either CTA signals the other's; both
  // CTAs of a pair see the same offsets and so the same tile count
  cluster_sync();
  const int total = sh->total_tiles;
  // uniform across the pair; no TMEM taken.  (WG: a pair without compute
  // units stays for its share of the zero tiles when no pair has any.)
  if (pair >= (MODE == kWG ? max(total, 1) : total)) return;
  const int* wgp = &sh->wg_whole;                 // {whole, split} for decode_pair_tile<kWG>

  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&sh->tmem_base), kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    if (MODE != kWG) {
      prefetch_tmap(&tmA0); prefetch_tmap(&tmA1); prefetch_tmap(&tmB0); prefetch_tmap(&tmB1);
    }
    prefetch_tmap(&tmO0); prefetch_tmap(&tmO1); prefetch_tmap(&tmO2);
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0, issued = 0, last_par = 0;
    int wg_e = -1;                          // WG: expert of the descriptors acquired
    uint32_t wg_seen = 0;
    bool ok = true;
    for (int i = 0, t = pair_unit<MODE>(0, pair, npairs); t < total && ok; t = pair_unit<MODE>(++i, pair, npairs)) {
      const Tile tl = decode_pair_tile<MODE>(t, args, s_off, s_ts, wgp);
      if constexpr (MODE == kWG) {
        // the descriptors were written by an earlier kernel through the
        // generic proxy; make them visible to the tensormap proxy, once per
        // descriptor (a CTA meets the experts in increasing order)
        if (lane == 0 && tl.nkb > 0) {
          if (tl.e != wg_e) { wg_e = tl.e; wg_seen = 0; }
          const CUtensorMap* em = args.wg_maps + (size_t)tl.e * kWgradMaps;
          const int oa = tl.which == 2 ? 1 : 0, ob = 2 + tl.which;
          if (!(wg_seen & (1u << oa))) { tensormap_acquire(em + oa); wg_seen |= 1u << oa; }
          if (!(wg_seen & (1u << ob))) { tensormap_acquire(em + ob); wg_seen |= 1u << ob; }
        }
      }
      for (int kb0 = 0; kb0 < tl.nkb; kb0 += KPS) {
        const int nk = min(KPS, tl.nkb - kb0);
        if (!bounded_wait(smem_u32(&sh->empty[stage]), phase ^ 1u, &sh->abort_flag, args.status)) { ok = false; break; }
        if (lane == 0) {
          const uint32_t fb_local = smem_u32(&sh->full[stage]);
          if (leader) mbar_arrive_expect_tx(fb_local, nk * 4 * P_HALF);   // both CTAs' copies
          for (int j = 0; j < nk; ++j) {
            int kbr = kb0 + j;
            if constexpr (MODE == kWG) kbr = wg_kblock(tl, i, kbr);
            const int q = stage * KPS + j;
            issue_loads_pair<MODE>(tl, kbr, rank, smem_u32(sA + q * P_HALF), smem_u32(sB + q * P_HALF),
                                   mapa_shared(fb_local, 0), &tmA0, &tmA1, &tmB0, &tmB1, args);
          }
        }
        __syncwarp();
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        if (++stage == PS) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && leader && lane == 0) {
      // the even CTA's full barriers count both CTAs' copies
      for (int s = 0; s < PS; ++s)
        if (issued & (1u << s)) drain_wait(smem_u32(&sh->full[s]), (last_par >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------- MMA issuer (even CTA of the pair)
    if (leader) {
      constexpr bool a_mn = (MODE == kWG);
      constexpr bool b_mn = (MODE == kUp || MODE == kDown || MODE == kWG);
      constexpr uint32_t idesc = idesc_bf16(P_TILE, P_TILE, a_mn, b_mn);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true, issued_any = false;
      for (int i = 0, t = pair_unit<MODE>(0, pair, npairs); t < total && ok; t = pair_unit<MODE>(++i, pair, npairs)) {
        const Tile tl = decode_pair_tile<MODE>(t, args, s_off, s_ts, wgp);
        if constexpr (MODE == kWG) {
          if (tl.part < 0 && tl.nkb == 0) continue;     // empty expert: no accumulator (epilogue stores zeros)
        }
        if (!bounded_wait(smem_u32(&sh->tempty[acc]), acc_phase ^ 1u, &sh->abort_flag, args.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tf = smem_u32(&sh->tfull[acc]);
        if (tl.nkb == 0) {
          if (lane == 0) { mbar_arrive_cluster(mapa_shared(tf, 0)); mbar_arrive_cluster(mapa_shared(tf, 1)); }
        } else {
          const uint32_t dt = tmem + (uint32_t)(acc * P_TILE);
          for (int kb0 = 0; kb0 < tl.nkb; kb0 += KPS) {
            const int nk = min(KPS, tl.nkb - kb0);
            if (!bounded_wait(smem_u32(&sh->full[stage]), phase, &sh->abort_flag, args.status)) { ok = false; break; }
            tc_fence_after();
            if (lane == 0) {
              for (int j = 0; j < nk; ++j) {
                const int kb = kb0 + j, q = stage * KPS + j;
                int nkk = BK / 16;
                if constexpr (MODE == kWG) nkk = wg_groups(tl, wg_kblock(tl, i, kb));
                const uint32_t sa = smem_u32(sA + q * P_HALF), sb = smem_u32(sB + q * P_HALF);
                for (int kk = 0; kk < nkk; ++kk) {
                  uint64_t ad, bd;
                  if constexpr (a_mn) ad = sdesc_sw128(sa + kk * 2048, SUB, 1024);
                  else ad = sdesc_sw128(sa + kk * 32, 16, 1024);
                  if constexpr (b_mn) bd = sdesc_sw128(sb + kk * 2048, SUB, 1024);
                  else bd = sdesc_sw128(sb + kk * 32, 16, 1024);
                  mma_f16_pair(dt, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                }
              }
              mma_commit_pair_both(smem_u32(&sh->empty[stage]));
            }
            issued_any = true;
            __syncwarp();
            if (++stage == PS) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          if (lane == 0) mma_commit_pair_both(tf);
          __syncwarp();
        }
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok && issued_any && lane == 0) {
        mma_commit_pair(mapa_shared(smem_u32(&sh->drain), 0));
        drain_wait(smem_u32(&sh->drain), 0);
      }
    }
    // the odd CTA's MMA warp only holds its half of the TMEM allocation
  } else if (warp < 2 + kEpiWarps) {
    // --------------------------------------------------------------- epilogue
    const int lane_q = warp & 3;
    const int half = (warp - 2) >> 2;
    const OutMaps om{&tmO0, &tmO1, &tmO2};
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t rn = 0;                          // DA: ring chunks of the tiles before
    for (int i = 0, t = pair_unit<MODE>(0, pair, npairs); t < total; t = pair_unit<MODE>(++i, pair, npairs), rn += 8) {
      Tile tl = decode_pair_tile<MODE>(t, args, s_off, s_ts, wgp);
      // this CTA's rows of the output tile
      if constexpr (MODE == kWG) {
        tl.m0 += 128 * (int)rank;
        if (tl.part < 0 && tl.nkb == 0) {          // empty expert: dW tile of zeros, no accumulator
          epilogue_zero_tile(tl, lane_q, half, lane, sZero, args, om);
          continue;
        }
      } else {
        tl.row0 += 128 * (int)rank;
        tl.rows = max(0, min(128, tl.rows - 128 * (int)rank));
      }
      if (!bounded_wait(smem_u32(&sh->tfull[acc]), acc_phase, &sh->abort_flag, args.status)) break;
      tc_fence_after();
      bool whole = true;
      if constexpr (MODE == kWG) {
        if (tl.part >= 0) {
          epilogue_partial(tl, tmem + (uint32_t)(acc * P_TILE), lane_q, half, lane, rank, args);
          whole = false;
        }
      }
      if constexpr (MODE == kDA) {
        if (!epilogue_da_ring(tl, tmem + (uint32_t)(acc * P_TILE), lane_q, half, lane, ring, sh->rfull,
                              sh->rempty, &sh->abort_flag, rn, args, om))
          break;
      } else if (whole) {
        if constexpr (MODE == kWG || MODE == kDown || MODE == kDX) {
          epilogue_tile_early<MODE>(tl, tmem + (uint32_t)(acc * P_TILE), lane_q, half, lane,
                                    sStage + (warp - 2) * kStageBytes, args, om,
                                    mapa_shared(smem_u32(&sh->tempty[acc]), 0));
          if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
          continue;
        } else {
          epilogue_tile<MODE>(tl, tmem + (uint32_t)(acc * P_TILE), lane_q, half, lane,
                              sStage + (warp - 2) * kStageBytes, args, om);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&sh->tempty[acc]), 0));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    stg_finish(lane);
  } else if constexpr (MODE == kDA) {
    // ------------------------------------------------ DA: h1 / h3 ring loader
    // chunk c of every tile (this CTA's 128 rows, columns n0 + 32c ..) into
    // slot g % kRingSlots, g counting the chunks in order
    uint32_t g = 0, issued = 0, last_par = 0;
    bool ok = true;
    for (int i = 0, t = pair_unit<MODE>(0, pair, npairs); t < total && ok; t = pair_unit<MODE>(++i, pair, npairs)) {
      const Tile tl = decode_pair_tile<MODE>(t, args, s_off, s_ts, wgp);
      const int y = tl.row0 + 128 * (int)rank;
      for (int c = 0; c < 8; ++c, ++g) {
        const int slot = (int)(g % kRingSlots);
        const uint32_t par = (g / kRingSlots) & 1u;
        if (!bounded_wait(smem_u32(&sh->rempty[slot]), par ^ 1u, &sh->abort_flag, args.status)) { ok = false; break; }
        if (lane == 0) {
          const uint32_t fb = smem_u32(&sh->rfull[slot]);
          const uint32_t dst = smem_u32(ring + slot * kRingSlotBytes);
          mbar_arrive_expect_tx(fb, kRingSlotBytes);
          tma_load_2d(dst, &tmA1, fb, tl.n0 + 32 * c, y);                  // h1
          tma_load_2d(dst + kRingChunk, &tmB1, fb, tl.n0 + 32 * c, y);     // h3
        }
        __syncwarp();
        issued |= 1u << slot;
        last_par = (last_par & ~(1u << slot)) | (par << slot);
      }
    }
    if (!ok && lane == 0) {
      for (int s = 0; s < kRingSlots; ++s)
        if (issued & (1u << s)) drain_wait(smem_u32(&sh->rfull[s]), (last_par >> s) & 1u);
    }
    __syncwarp();
  } else if constexpr (MODE == kWG) {
    // ------------------------------------------- WG: the empty experts' dW
    // Experts without rows get dW = 0.  Their tiles are not work units: this
    // warp stores them from the shared box of zeros, round-robin over the
    // pairs that run, beside the MMAs and on its own bulk-store queue (so the
    // epilogue's waits for its staging buffers never wait for these stores),
    // with at most two tiles' stores in flight.
    const int per = 2 * args.wg_t1 + args.wg_t2;
    const int nz = sh->wg_zero;
    const int active = min(npairs, max(total, 1));
    if (lane == 0) {
      int n = 0;
      for (int z = pair; z < nz; z += active) {
        const int e = args.wg_plan[kWgradPlanHead + args.E + z / per];
        int l = z % per, which, mt;
        if (l < args.wg_t1) { which = 0; mt = args.wg_mt1; }
        else if (l < 2 * args.wg_t1) { which = 1; l -= args.wg_t1; mt = args.wg_mt1; }
        else { which = 2; l -= 2 * args.wg_t1; mt = args.wg_mt2; }
        const int M = which == 2 ? args.h : args.d, N = which == 2 ? args.d : args.h;
        const int m0 = (l % mt) * P_TILE + 128 * (int)rank, n0 = (l / mt) * P_TILE;
        const CUtensorMap* map = which == 0 ? &tmO0 : (which == 1 ? &tmO1 : &tmO2);
        for (int q = 0; q < 4 && m0 + 32 * q < M; ++q)
          for (int c = 0; c < 8 && n0 + 32 * c < N; ++c) tma_store_3d(map, smem_u32(sZero), n0 + 32 * c, m0 + 32 * q, e);
        bulk_commit();
        if (++n >= 2) bulk_wait_group<1>();
      }
      bulk_wait_all();
    }
    __syncwarp();
  }

  tc_fence_before();
  // no CTA leaves (or frees TMEM) while its peer may still signal it
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// wgrad descriptors: expert e gets copies of the five operand descriptors
// (xp, a, dh1, dh3, dyp) whose row extent is the expert's end row, so a tile
// that starts inside the expert reads zeros past its last row.  Thread i
// writes descriptor i of the [E][5] table.
struct WgradTemplates { CUtensorMap m[kWgradMaps]; };

// One launch prepares the wgrad: the last block writes the tile plan
// (wgrad_plan), the others the descriptors, thread i descriptor i.
__global__ void __launch_bounds__(1024)
wgrad_maps_kernel(const __grid_constant__ WgradTemplates tp, const int32_t* __restrict__ offsets,
                  int E, int R, CUtensorMap* __restrict__ maps, int per, int npairs, int parts_max,
                  int* __restrict__ plan) {
  pdl_enter();
  if (blockIdx.x == gridDim.x - 1) {
    wgrad_plan(offsets, E, R, per, npairs, parts_max, plan);
    return;
  }
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= E * kWgradMaps) return;
  const int e = i / kWgradMaps, op = i - e * kWgradMaps;
  const int lo = max(0, min(__ldg(offsets + e), R));
  const int hi = max(lo, min(__ldg(offsets + e + 1), R));
  const uint4* src = reinterpret_cast<const uint4*>(&tp.m[op]);
  uint4* dst = reinterpret_cast<uint4*>(maps + i);
#pragma unroll
  for (int j = 0; j < 8; ++j) dst[j] = src[j];
  // an empty expert's descriptor is never used; keep its extent legal
  tensormap_set_dim<1>(maps + i, max(hi, 1));
  tensormap_release();
}

// ------------------------------------------------------------------ host side

constexpr size_t smem_bytes(int E) {
  return 1024 + (size_t)SLOTS * (A_STAGE + B_STAGE) + (size_t)kEpiWarps * kStageBytes +
         sizeof(Shared) + 2 * (size_t)(E + 1) * 4;
}

// output descriptors of one GEMM launch (see OutMaps); unused slots repeat one
struct OutDescs {
  CUtensorMap m[3];
};

template <int MODE>
int launch(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
           const CUtensorMap& b1, const CUtensorMap& b2, const OutDescs& o, const GemmArgs& args,
           int grid, cudaStream_t s) {
  const size_t smem = smem_bytes(args.E);
  auto kern = grouped_gemm_kernel<MODE>;
  static bool attr_done[64] = {false};
  // set once per device for the largest size (E = 1024)
  if (ensure_smem_attr(kern, smem_bytes(kMaxExperts), attr_done) != MOE_OK) return MOE_ERR_CUDA;
  (void)launch_pdl(kern, grid, kThreads, smem, s, a0, a1, b0, b1, b2, o.m[0], o.m[1], o.m[2], args);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

template <int MODE>
constexpr size_t pair_smem_bytes(int E) {
  return 1024 + (size_t)pair_slots<MODE>() * 2 * P_HALF + pair_ring_bytes<MODE>() +
         (size_t)pair_stage_bytes<MODE>() + pair_zero_bytes<MODE>() + sizeof(PairSharedT<MODE>) +
         2 * (size_t)(E + 1) * 4;
}
// the largest expert count whose tile table still fits beside the pipeline
// in the 227 KB of shared memory a block may opt in to
constexpr size_t kSmemOptIn = 227 * 1024;
template <int MODE>
constexpr int pair_max_experts() {
  const long long room = (long long)kSmemOptIn - (long long)pair_smem_bytes<MODE>(0) + 8;
  const long long e = room / 8 - 1;
  return e < kMaxExperts ? (int)e : kMaxExperts;
}
static_assert(pair_max_experts<kUp>() == kMaxExperts && pair_max_experts<kWG>() == kMaxExperts,
              "the 3-stage (6-slot) pair GEMMs fit every expert count");
static_assert(pair_max_experts<kDA>() >= 128, "DA on pairs covers pools of 128 experts");

// at[] must hold two attributes: the 2-CTA cluster shape and programmatic
// stream serialisation (see launch_pdl)
inline cudaLaunchConfig_t pair_config(int npairs, size_t smem, cudaStream_t s, cudaLaunchAttribute* at) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * npairs);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2; at[0].val.clusterDim.y = 1; at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cfg;
}

// Co-resident 2-CTA clusters of pair_gemm_kernel<MODE>, queried once per
// device on the first call (outside any stream capture that follows).
template <int MODE>
int pair_limit(cudaStream_t s) {
  auto kern = pair_gemm_kernel<MODE>;
  static bool attr_done[64] = {false};
  static int limit[64] = {0};
  if (ensure_smem_attr(kern, pair_smem_bytes<MODE>(pair_max_experts<MODE>()), attr_done) != MOE_OK) return -1;
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return -1;
  if (limit[dev] == 0) {
    cudaLaunchAttribute at[2];
    cudaLaunchConfig_t q = pair_config(sm_count(), pair_smem_bytes<MODE>(pair_max_experts<MODE>()), s, at);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      return -1;
    }
    limit[dev] = n;
  }
  return limit[dev];
}

// Launches pair_gemm_kernel<MODE> on min(tiles_upper, co-resident pairs) clusters.
template <int MODE>
int launch_pair(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                const CUtensorMap& b1, const OutDescs& o, const GemmArgs& g, long long tiles_upper,
                cudaStream_t s) {
  auto kern = pair_gemm_kernel<MODE>;
  const int limit = pair_limit<MODE>(s);
  if (limit <= 0) return MOE_ERR_CUDA;
  cudaLaunchAttribute at[2];
  const long long ub = tiles_upper > 0 ? tiles_upper : 1;
  const int npairs = (int)(ub < limit ? ub : limit);
  cudaLaunchConfig_t cfg = pair_config(npairs, pair_smem_bytes<MODE>(g.E), s, at);
  if (cudaLaunchKernelEx(&cfg, kern, a0, a1, b0, b1, o.m[0], o.m[1], o.m[2], g) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

// UP, DOWN, DA and DX run on CTA pairs (256-row tiles) unless the experts are
// small on average: then the 128-row tiles of the single-CTA kernel waste
// less on each expert's last, partial tile.  DX (K = 2h, the longest
// mainloop per tile) gains least from the pairs; since the pair loop stages
// two k-blocks per barrier it is no slower there at 512 rows per expert
// (event-timed on the GB300, T = 16384, d = 2048, h = 1024, E = 128, top-4:
// 402-410 vs 406-410 us uniform, 326-330 vs 351-353 us Zipf-skewed), so it
// takes the same threshold.
constexpr long long kPairMinRowsPerExpert = 512;
constexpr long long kPairMinRowsPerExpertDX = 512;
inline bool rows_on_pairs(int R, int E, long long min_rows = kPairMinRowsPerExpert) {
  return (long long)R >= min_rows * E;
}

int check_common(const void* ws, size_t ws_bytes, int R, int E, int d, int h) {
  if (R < 0 || E < 1 || E > kMaxExperts || d <= 0 || h <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 64 != 0 || h % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (ws == nullptr || ws_bytes < kStatusBytes) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

namespace moe {
namespace {

// descriptors of up to three row-grouped [R, cols] bf16 outputs (row stride cols)
bool row_outs(OutDescs* o, int R, uint64_t cols, const void* p0, const void* p1 = nullptr,
              const void* p2 = nullptr) {
  const void* p[3] = {p0, p1 ? p1 : p0, p2 ? p2 : p0};
  for (int i = 0; i < 3; ++i)
    if (!map2d_out(&o->m[i], p[i], cols, (uint64_t)R, cols)) return false;
  return true;
}

GemmArgs base_args(const int32_t* offsets, int R, int E, int d, int h, void* ws) {
  GemmArgs g{};
  g.offsets = offsets; g.E = E; g.R = R; g.d = d; g.h = h; g.status = reinterpret_cast<int*>(ws);
  return g;
}

// [h1 | h3] = xp_e @ [W1[e] | W3[e]], a = silu(h1) * h3
int run_up(const moe_bf16_t* xp, const int32_t* offsets, int R, int E, int d, int h,
           const moe_bf16_t* W1, const moe_bf16_t* W3, moe_bf16_t* h1, moe_bf16_t* h3,
           moe_bf16_t* a, void* ws, cudaStream_t s) {
  MOE_CHECK_PTR(xp); MOE_CHECK_PTR(offsets); MOE_CHECK_PTR(W1); MOE_CHECK_PTR(W3);
  MOE_CHECK_PTR(h1); MOE_CHECK_PTR(h3); MOE_CHECK_PTR(a);
  CUtensorMap mx, mw1, mw3;
  if (!map2d(&mx, xp, d, R, 64, BM) || !map3d(&mw1, W1, h, d, E, 64, 64) ||
      !map3d(&mw3, W3, h, d, E, 64, 64))
    return MOE_ERR_CUDA;
  GemmArgs g = base_args(offsets, R, E, d, h, ws);
  g.n_tiles = (h + BN / 2 - 1) / (BN / 2);      // 128 h-columns of W1 and of W3 per tile
  g.kb_total = d / BK;
  g.out0 = h1; g.out1 = h3; g.out2 = a; g.ldo = h;
  OutDescs o;
  if (!row_outs(&o, R, h, h1, h3, a)) return MOE_ERR_CUDA;
  if (rows_on_pairs(R, E))
    return launch_pair<kUp>(mx, mx, mw1, mw3, o, g, row_tiles_upper(R, E, g.n_tiles, P_TILE), s);
  return launch<kUp>(mx, mx, mw1, mw3, mw3, o, g, row_grid_upper(R, E, g.n_tiles), s);
}

// yp = a_e @ W2[e]
int run_down(const moe_bf16_t* a, const int32_t* offsets, int R, int E, int d, int h,
             const moe_bf16_t* W2, moe_bf16_t* yp, void* ws, cudaStream_t s) {
  MOE_CHECK_PTR(a); MOE_CHECK_PTR(offsets); MOE_CHECK_PTR(W2); MOE_CHECK_PTR(yp);
  CUtensorMap ma, mw2;
  if (!map2d(&ma, a, h, R, 64, BM) || !map3d(&mw2, W2, d, h, E, 64, 64)) return MOE_ERR_CUDA;
  GemmArgs g = base_args(offsets, R, E, d, h, ws);
  g.n_tiles = (d + BN - 1) / BN;
  g.kb_total = h / BK;
  g.out0 = yp; g.ldo = d;
  OutDescs o;
  if (!row_outs(&o, R, d, yp)) return MOE_ERR_CUDA;
  if (rows_on_pairs(R, E))
    return launch_pair<kDown>(ma, ma, mw2, mw2, o, g, row_tiles_upper(R, E, g.n_tiles, P_TILE), s);
  return launch<kDown>(ma, ma, mw2, mw2, mw2, o, g, row_grid_upper(R, E, g.n_tiles), s);
}

// dA = dyp_e @ W2[e]^T with the SwiGLU backward epilogue -> dh1, dh3
int run_dact(const int32_t* offsets, int R, int E, int d, int h, const moe_bf16_t* W2,
             const moe_bf16_t* h1, const moe_bf16_t* h3, const moe_bf16_t* dyp, moe_bf16_t* dh1,
             moe_bf16_t* dh3, void* ws, cudaStream_t s, uint8_t* dh1q = nullptr,
             uint8_t* dh1s = nullptr, uint8_t* dh3q = nullptr, uint8_t* dh3s = nullptr) {
  MOE_CHECK_PTR(offsets); MOE_CHECK_PTR(W2); MOE_CHECK_PTR(h1); MOE_CHECK_PTR(h3);
  MOE_CHECK_PTR(dyp); MOE_CHECK_PTR(dh1); MOE_CHECK_PTR(dh3);
  if (dh1q != nullptr) {
    MOE_CHECK_PTR(dh1q); MOE_CHECK_PTR(dh3q);
    if (dh1s == nullptr || dh3s == nullptr) return MOE_ERR_INVALID_ARG;
  }
  const bool pairs = rows_on_pairs(R, E) && E <= pair_max_experts<kDA>();
  CUtensorMap m_dyp, m_w2k;
  if (!map2d(&m_dyp, dyp, d, R, 64, BM) || !map3d(&m_w2k, W2, d, h, E, 64, pairs ? BN / 2 : BN))
    return MOE_ERR_CUDA;
  GemmArgs g = base_args(offsets, R, E, d, h, ws);
  g.n_tiles = (h + BN - 1) / BN;
  g.kb_total = d / BK;
  g.out0 = dh1; g.out1 = dh3; g.in0 = h1; g.in1 = h3; g.ldo = h;
  g.q0 = dh1q; g.q1 = dh3q; g.qs0 = dh1s; g.qs1 = dh3s;
  OutDescs o;   // TMA stores on pairs; the single-CTA kernel stores without them
  if (!row_outs(&o, R, h, dh1, dh3)) return MOE_ERR_CUDA;
  if (pairs) {
    // the epilogue's h1 / h3 ring: 32-column x 128-row boxes
    CUtensorMap m_h1, m_h3;
    if (!map2d_out(&m_h1, h1, h, R, h, 128) || !map2d_out(&m_h3, h3, h, R, h, 128)) return MOE_ERR_CUDA;
    return launch_pair<kDA>(m_dyp, m_h1, m_w2k, m_h3, o, g, row_tiles_upper(R, E, g.n_tiles, P_TILE), s);
  }
  return launch<kDA>(m_dyp, m_dyp, m_w2k, m_w2k, m_w2k, o, g, row_grid_upper(R, E, g.n_tiles), s);
}

// dxp = dh1_e @ W1[e]^T + dh3_e @ W3[e]^T (one reduction over K = 2h)
int run_dx(const int32_t* offsets, int R, int E, int d, int h, const moe_bf16_t* W1,
           const moe_bf16_t* W3, const moe_bf16_t* dh1, const moe_bf16_t* dh3, moe_bf16_t* dxp,
           void* ws, cudaStream_t s) {
  MOE_CHECK_PTR(offsets); MOE_CHECK_PTR(W1); MOE_CHECK_PTR(W3); MOE_CHECK_PTR(dh1);
  MOE_CHECK_PTR(dh3); MOE_CHECK_PTR(dxp);
  const bool pairs = rows_on_pairs(R, E, kPairMinRowsPerExpertDX);
  const uint32_t bn = pairs ? BN / 2 : BN;
  CUtensorMap m_dh1, m_dh3, m_w1k, m_w3k;
  if (!map2d(&m_dh1, dh1, h, R, 64, BM) || !map2d(&m_dh3, dh3, h, R, 64, BM) ||
      !map3d(&m_w1k, W1, h, d, E, 64, bn) || !map3d(&m_w3k, W3, h, d, E, 64, bn))
    return MOE_ERR_CUDA;
  GemmArgs g = base_args(offsets, R, E, d, h, ws);
  g.n_tiles = (d + BN - 1) / BN;
  g.kb_total = 2 * (h / BK);
  g.kb_split = h / BK;
  g.out0 = dxp; g.ldo = d;
  OutDescs o;
  if (!row_outs(&o, R, d, dxp)) return MOE_ERR_CUDA;
  if (pairs)
    return launch_pair<kDX>(m_dh1, m_dh3, m_w1k, m_w3k, o, g, row_tiles_upper(R, E, g.n_tiles, P_TILE), s);
  return launch<kDX>(m_dh1, m_dh3, m_w1k, m_w3k, m_w3k, o, g, row_grid_upper(R, E, g.n_tiles), s);
}

// dW1[e] = xp_e^T dh1_e, dW3[e] = xp_e^T dh3_e, dW2[e] = a_e^T dyp_e (one launch)
int run_wgrad(const moe_bf16_t* xp, const int32_t* offsets, int R, int E, int d, int h,
              const moe_bf16_t* a, const moe_bf16_t* dyp, const moe_bf16_t* dh1,
              const moe_bf16_t* dh3, moe_bf16_t* dW1, moe_bf16_t* dW3, moe_bf16_t* dW2, void* ws,
              size_t ws_bytes, cudaStream_t s) {
  MOE_CHECK_PTR(dW1); MOE_CHECK_PTR(dW3); MOE_CHECK_PTR(dW2);
  if (R > 0) {
    if (ws_bytes < wgrad_plan_end(E)) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 127) != 0) return MOE_ERR_INVALID_ARG;
  }
  if (R == 0) {
    const size_t wb = (size_t)E * d * h * 2;
    if (cudaMemsetAsync(dW1, 0, wb, s) != cudaSuccess || cudaMemsetAsync(dW3, 0, wb, s) != cudaSuccess ||
        cudaMemsetAsync(dW2, 0, wb, s) != cudaSuccess) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }
  MOE_CHECK_PTR(xp); MOE_CHECK_PTR(offsets); MOE_CHECK_PTR(a); MOE_CHECK_PTR(dyp);
  MOE_CHECK_PTR(dh1); MOE_CHECK_PTR(dh3);
  WgradTemplates tp;
  // MN-major operands: 64 x 64 boxes along (feature, row)
  if (!map2d(&tp.m[0], xp, d, R, 64, 64) || !map2d(&tp.m[1], a, h, R, 64, 64) ||
      !map2d(&tp.m[2], dh1, h, R, 64, 64) || !map2d(&tp.m[3], dh3, h, R, 64, 64) ||
      !map2d(&tp.m[4], dyp, d, R, 64, 64))
    return MOE_ERR_CUDA;
  CUtensorMap* maps = reinterpret_cast<CUtensorMap*>(static_cast<uint8_t*>(ws) + kStatusBytes);
  GemmArgs g = base_args(offsets, R, E, d, h, ws);
  g.wg_maps = maps;
  g.out0 = dW1; g.out1 = dW3; g.out2 = dW2;
  // 256 x 256 output tiles, one per CTA pair
  g.wg_mt1 = (d + P_TILE - 1) / P_TILE;
  g.wg_mt2 = (h + P_TILE - 1) / P_TILE;
  g.wg_t1 = g.wg_mt1 * ((h + P_TILE - 1) / P_TILE);
  g.wg_t2 = g.wg_mt2 * ((d + P_TILE - 1) / P_TILE);
  const int per = 2 * g.wg_t1 + g.wg_t2;
  const long long tiles = (long long)E * per;
  // The work units are the tiles of the experts that have rows, deepest
  // expert first (the host never learns the row counts: a one-CTA kernel
  // writes the plan from the offsets); the pairs take them in snake order and
  // split the last round along K when it would keep at most half of them busy
  // (fp32 partials a second kernel adds in chunk order).  The empty experts'
  // zero tiles are stored beside the work units by one warp of each pair.
  const int P = pair_limit<kWG>(s);
  if (P <= 0) return MOE_ERR_CUDA;
  const int npairs = (int)(tiles < P ? tiles : P);
  const bool parts = ws_bytes >= wgrad_parts_end(E);
  int* plan = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + wgrad_plan_offset(E));
  (void)launch_pdl(wgrad_maps_kernel, (E * kWgradMaps + 1023) / 1024 + 1, 1024, 0, s, tp, offsets, E, R, maps,
                   per, npairs, parts ? kWgradParts : 0, plan);
  MOE_LAUNCH_CHECK(1);
  g.wg_plan = plan;
  g.wg_part = parts ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + wgrad_parts_offset(E)) : nullptr;
  OutDescs o;
  if (!map3d_out(&o.m[0], dW1, h, d, E) || !map3d_out(&o.m[1], dW3, h, d, E) ||
      !map3d_out(&o.m[2], dW2, d, h, E))
    return MOE_ERR_CUDA;
  const int st = launch_pair<kWG>(tp.m[0], tp.m[1], tp.m[2], tp.m[3], o, g, tiles, s);
  if (st != MOE_OK || !parts) return st;
  // up to npairs / 2 split tiles of 256 rows; 2048 blocks take them (one row
  // each at dense_e8's 8 split tiles) and return at once when nothing was split
  (void)launch_pdl(wgrad_fixup_kernel, 2048u, P_TILE, 0, s, g);
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

#define MOE_GEMM_PROLOGUE()                                   \
  int st = check_common(ws, ws_bytes, R, E, d, h);            \
  if (st != MOE_OK) return st;                                \
  cudaStream_t s = (cudaStream_t)stream;                      \
  (void)s

extern "C" {

int moe_grouped_swiglu_fwd(const moe_bf16_t* xp, const int32_t* offsets, int R, int E, int d, int h,
                           const moe_bf16_t* W1, const moe_bf16_t* W3, const moe_bf16_t* W2,
                           moe_bf16_t* h1, moe_bf16_t* h3, moe_bf16_t* a, moe_bf16_t* yp, void* ws,
                           size_t ws_bytes, moe_stream_t stream) {
  MOE_GEMM_PROLOGUE();
  if (R == 0) return MOE_OK;
  MOE_CHECK_PTR(W2); MOE_CHECK_PTR(yp);
  st = run_up(xp, offsets, R, E, d, h, W1, W3, h1, h3, a, ws, s);
  if (st != MOE_OK) return st;
  return run_down(a, offsets, R, E, d, h, W2, yp, ws, s);
}

int moe_grouped_swiglu_fwd_up(const moe_bf16_t* xp, const int32_t* offsets, int R, int E, int d,
                              int h, const moe_bf16_t* W1, const moe_bf16_t* W3, moe_bf16_t* h1,
                              moe_bf16_t* h3, moe_bf16_t* a, void* ws, size_t ws_bytes,
                              moe_stream_t stream) {
  MOE_GEMM_PROLOGUE();
  if (R == 0) return MOE_OK;
  return run_up(xp, offsets, R, E, d, h, W1, W3, h1, h3, a, ws, s);
}

int moe_grouped_swiglu_fwd_down(const moe_bf16_t* a, const int32_t* offsets, int R, int E, int d,
                                int h, const moe_bf16_t* W2, moe_bf16_t* yp, void* ws,
                                size_t ws_bytes, moe_stream_t stream) {
  MOE_GEMM_PROLOGUE();
  if (R == 0) return MOE_OK;
  return run_down(a, offsets, R, E, d, h, W2, yp, ws, s);
}

int moe_grouped_swiglu_bwd(const moe_bf16_t* xp, const int32_t* offsets, int R, int E, int d, int h,
                           const moe_bf16_t* W1, const moe_bf16_t* W3, const moe_bf16_t* W2,
                           const moe_bf16_t* h1, const moe_bf16_t* h3, const moe_bf16_t* a,
                           const moe_bf16_t* dyp, moe_bf16_t* dh1, moe_bf16_t* dh3, moe_bf16_t* dxp,
                           moe_bf16_t* dW1, moe_bf16_t* dW3, moe_bf16_t* dW2, void* ws,
                           size_t ws_bytes, moe_stream_t stream) {
  MOE_GEMM_PROLOGUE();
  if (R > 0) {
    st = run_dact(offsets, R, E, d, h, W2, h1, h3, dyp, dh1, dh3, ws, s);
    if (st != MOE_OK) return st;
    st = run_dx(offsets, R, E, d, h, W1, W3, dh1, dh3, dxp, ws, s);
    if (st != MOE_OK) return st;
  }
  return run_wgrad(xp, offsets, R, E, d, h, a, dyp, dh1, dh3, dW1, dW3, dW2, ws, ws_bytes, s);
}

int moe_grouped_swiglu_bwd_dact(const int32_t* offsets, int R, int E, int d, int h,
                                const moe_bf16_t* W2, const moe_bf16_t* h1, const moe_bf16_t* h3,
                                const moe_bf16_t* dyp, moe_bf16_t* dh1, moe_bf16_t* dh3, void* ws,
                                size_t ws_bytes, moe_stream_t stream) {
  MOE_GEMM_PROLOGUE();
  if (R == 0) return MOE_OK;
  return run_dact(offsets, R, E, d, h, W2, h1, h3, dyp, dh1, dh3, ws, s);
}

int moe_grouped_swiglu_bwd_dact_mxfp8(const int32_t* offsets, int R, int E, int d, int h,
                                      const moe_bf16_t* W2, const moe_bf16_t* h1, const moe_bf16_t* h3,
                                      const moe_bf16_t* dyp, moe_bf16_t* dh1, moe_bf16_t* dh3,
                                      uint8_t* dh1q, uint8_t* dh1s, uint8_t* dh3q, uint8_t* dh3s, void* ws,
                                      size_t ws_bytes, moe_stream_t stream) {
  MOE_GEMM_PROLOGUE();
  if (R == 0) return MOE_OK;
  if (dh1q == nullptr) return MOE_ERR_INVALID_ARG;
  return run_dact(offsets, R, E, d, h, W2, h1, h3, dyp, dh1, dh3, ws, s, dh1q, dh1s, dh3q, dh3s);
}

int moe_grouped_swiglu_bwd_dx(const int32_t* offsets, int R, int E, int d, int h,
                              const moe_bf16_t* W1, const moe_bf16_t* W3, const moe_bf16_t* dh1,
                              const moe_bf16_t* dh3, moe_bf16_t* dxp, void* ws, size_t ws_bytes,
                              moe_stream_t stream) {
  MOE_GEMM_PROLOGUE();
  if (R == 0) return MOE_OK;
  return run_dx(offsets, R, E, d, h, W1, W3, dh1, dh3, dxp, ws, s);
}

int moe_grouped_swiglu_bwd_wgrad(const moe_bf16_t* xp, const int32_t* offsets, int R, int E, int d,
                                 int h, const moe_bf16_t* a, const moe_bf16_t* dyp,
                                 const moe_bf16_t* dh1, const moe_bf16_t* dh3, moe_bf16_t* dW1,
                                 moe_bf16_t* dW3, moe_bf16_t* dW2, void* ws, size_t ws_bytes,
                                 moe_stream_t stream) {
  MOE_GEMM_PROLOGUE();
  return run_wgrad(xp, offsets, R, E, d, h, a, dyp, dh1, dh3, dW1, dW3, dW2, ws, ws_bytes, s);
}

}  // extern "C"
