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
// Tiles are 192 columns wide with BK = 128 fp8 a k-block (one 128-byte
// swizzled row per operand row).  Operands are K-major: activations
// [R][K], weights [E][N][K] (moe_mxfp8_quantize_weights transposes).
// Issue rates of block-scaled MMAs with their per-k-block scale copies,
// measured on the GB300 with operands resident in shared memory: N = 256 runs
// at the full fp8 rate, N = 192 at 93% and N = 128 at 65-68%.  Two 192-column
// fp32 accumulators (at TMEM columns 0 and 256) leave room for the scale
// factors, so the epilogue of one tile overlaps the next tile's mainloop
// (a 256-column tile would fit only one accumulator).
// Scale factors: the E8M0 scales come in 512-byte atoms, the layout in which
// tcgen05.cp .32x128b.warpx4 moves them to tensor memory (see mx_common.cuh:
// byte (r, 4j + q) of an atom is the scale of row or column 32j + r of a
// 128-row block for the q-th 32-block of a 128-deep k-block).  The atoms are
// kept in HBM in the order the tiles read them, so each stage's scales arrive
// by TMA on the same barrier as its operands: one atom for the A rows, two for
// the 192 B columns.  The MMA then reads row m's A scale at lane m, column
// base + m/32, and column n's B scale at lane n%32 of the issuing quarter,
// column base + n/32, byte = the MMA's scale-factor id (0..3).
//
// Two kernel forms.  Single CTA: 128 x 192 tiles, 4 stages of one k-block.
// CTA pairs (2-CTA clusters, cta_group::2): 256 x 192 tiles, 3 stages of two
// k-blocks; each CTA stages its own 128 A rows, half of the B columns (UP8:
// the even CTA the 96 W1 columns, the odd CTA the same 96 W3 columns) and the
// scale atoms its half of the MMA reads (its own A atom, both B atoms); all of
// a stage's copies, of both CTAs, complete on the even CTA's barrier, and the
// even CTA's scale-copy warp moves both CTAs' atoms into their tensor memory
// (tcgen05.cp.cta_group::2).  Per MMA a CTA then moves 7 KB through shared
// memory instead of 10 KB on one CTA.
#include "gemm_common.cuh"
#include "mx_common.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace gemm;

enum Mode8 : int { kUp8 = 0, kDown8 = 1, kDx8 = 2 };

constexpr int BN = 192, BK = 128;               // MMA N, k-block (fp8 bytes)
constexpr int A_STAGE = 128 * BK;               // 16 KB: one CTA's 128 A rows
constexpr int SF_STAGE = 3 * mx::kAtomBytes;    // a k-block's A atom + two B atoms
constexpr int kTmemCols = 512;
constexpr int kMaxExperts8 = 768;               // shared-memory tile table bound
constexpr int kThreads8 = kThreads + 32;        // + the scale-copy warp

// Per form: rows a tile covers, B rows a CTA stages, pipeline stages, k-blocks
// a stage holds (KPS), and the tensor-memory columns of the second
// accumulator and of stage s's scales (k-block j of the stage: A at
// sf_col(s) + 12j, B at sf_col(s) + 12j + 4; 12 columns a k-block).
// A stage costs the MMA lane its barrier waits and one commit.  Each of those
// takes the issuing thread off the tensor pipe for about a short MMA's time
// (measured on the GB300 with operands resident: a pair loop with two waits
// and two commits per 4-MMA k-block issues at 0.57 of the fp8 rate, with one
// wait and one commit per 8 MMAs at 0.92, two waits and one commit at 0.86),
// so the pair form stages two k-blocks at a time.
template <bool PAIR> struct Form;
template <> struct Form<false> {
  static constexpr int TM = 128, BROWS = 192, STAGES = 4, KPS = 1;
  __device__ static uint32_t acc_col(int acc) { return (uint32_t)acc * 256; }
  __device__ static uint32_t sf_col(int s) { return 448 + 12 * s; }
};
template <> struct Form<true> {
  static constexpr int TM = 256, BROWS = 96, STAGES = 3, KPS = 2;
  __device__ static uint32_t acc_col(int acc) { return (uint32_t)acc * 256; }
  // the 64 columns after each 192-column accumulator hold the three stages'
  // 24 scale columns (two after the first, one after the second)
  __device__ static uint32_t sf_col(int s) { return s == 0 ? 192u : s == 1 ? 216u : 448u; }
};
template <bool PAIR> constexpr int b_stage() { return Form<PAIR>::BROWS * BK; }
// one k-block's slot; a stage holds KPS consecutive slots of each operand
template <bool PAIR> constexpr int slot_bytes() { return A_STAGE + b_stage<PAIR>() + SF_STAGE; }
template <bool PAIR> constexpr int stage_bytes() { return Form<PAIR>::KPS * slot_bytes<PAIR>(); }

struct Args8 {
  const int32_t* offsets;
  int E, R, d, h;
  int n_tiles;                  // column tiles per expert
  int kb_total;                 // K / 128
  int kb_split;                 // DX8: k-blocks of (dh1, W1) before those of (dh3, W3)
  int N;                        // rows of one weight matrix (UP8: h, DOWN8 and DX8: d)
  uint16_t* out0;               // UP8: h1 / DOWN8: yp
  uint16_t* out1;               // UP8: h3
  uint16_t* out2;               // UP8: a
  uint8_t* aq;                  // UP8: quantised a [R][h]
  uint8_t* as;                  // UP8: scales of a [R][h/32], row-major
  int* status;
};

__device__ __forceinline__ void tmem_cp_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tmem_cp_warpx4_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
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
__device__ __forceinline__ void mma_mxf8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
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
  if (nrows <= 0) return;                         // warp-uniform: no rows of this quarter
  const size_t r0 = (size_t)rt.row0 + lane_q * 32;
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

// One persistent kernel per mode and form.  Warp 0 loads operands and scale
// atoms by TMA, warp 1 allocates tensor memory and one lane (of the even CTA,
// on pairs) issues the MMAs, warps 2-9 drain the other accumulator, warp 10
// (of the even CTA) copies each stage's scale atoms to tensor memory.
template <int MODE, bool PAIR>
__global__ void __launch_bounds__(kThreads8, 1)
grouped_mxfp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ CUtensorMap tmB0,
                     const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmSA,
                     const __grid_constant__ CUtensorMap tmSB, const __grid_constant__ CUtensorMap tmO0,
                     const __grid_constant__ CUtensorMap tmO1, const __grid_constant__ CUtensorMap tmO2,
                     const Args8 args) {
  using F = Form<PAIR>;
  constexpr int S = F::STAGES, TM = F::TM, KPS = F::KPS;
  constexpr int B_STAGE = b_stage<PAIR>();
  using Shared = PipeShared<S>;
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // S * KPS k-block slots of each: A (16 KB), B, scale atoms (1.5 KB)
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * KPS * A_STAGE;
  uint8_t* sSF = sB + S * KPS * B_STAGE;
  uint8_t* sStage = sSF + S * KPS * SF_STAGE;                // kEpiWarps x kStageBytes
  Shared* sh = reinterpret_cast<Shared*>(sStage + kEpiWarps * kStageBytes);
  uint64_t* sfull = reinterpret_cast<uint64_t*>(sh + 1);      // [S] scales in TMEM, [S] copy drain
  uint64_t* sfa = sfull + S + 1;                               // [S] a stage's scale atoms landed
  int* s_off = reinterpret_cast<int*>(sfull + 2 * S + 1);
  int* s_ts = s_off + (args.E + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;      // pair or CTA
  const int nunits = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  for (int i = threadIdx.x; i <= args.E; i += kThreads8) s_off[i] = __ldg(args.offsets + i);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
      mbar_init(smem_u32(&sh->empty[s]), 1);
      mbar_init(smem_u32(&sfull[s]), 1);
    }
    mbar_init(smem_u32(&sfull[S]), 1);
    for (int q = 0; q < S; ++q) mbar_init(smem_u32(&sfa[q]), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&sh->tfull[s]), 1);
      mbar_init(smem_u32(&sh->tempty[s]), (PAIR ? 2 : 1) * kEpiWarps);
    }
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    const int n = build_row_tile_table<TM>(s_off, s_ts, args.E, args.R, args.n_tiles, lane);
    if (lane == 0) sh->total_tiles = n;
  }
  if constexpr (PAIR) cluster_sync();      // both CTAs' barriers exist before either signals
  else __syncthreads();
  const int total = sh->total_tiles;
  if (unit >= total) return;               // uniform across a pair; no TMEM taken

  if (warp == 1) {
    if constexpr (PAIR) { tmem_alloc_pair(smem_u32(&sh->tmem_base), kTmemCols); tmem_relinquish_pair(); }
    else { tmem_alloc(smem_u32(&sh->tmem_base), kTmemCols); tmem_relinquish(); }
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA); prefetch_tmap(&tmA1); prefetch_tmap(&tmB0); prefetch_tmap(&tmB1);
    prefetch_tmap(&tmSA); prefetch_tmap(&tmSB);
    prefetch_tmap(&tmO0); prefetch_tmap(&tmO1); prefetch_tmap(&tmO2);
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  const int KB = args.kb_total;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0, issued = 0, last_par = 0;
    bool ok = true;
    for (int t = unit; t < total && ok; t += nunits) {
      const RowTile rt = decode_row_tile<TM>(t, args.E, args.R, s_off, s_ts);
      const int n0 = rt.n_idx * (MODE == kUp8 ? BN / 2 : BN);
      // this CTA's 128 rows start a 128-row block of the expert's scale rows
      const int e_off = max(0, min(s_off[rt.e], args.R));
      const int blk = mx::act_block0(e_off, rt.e) + (rt.row0 - e_off) / 128 + (int)rank;
      const int wat = (rt.e * args.n_tiles + rt.n_idx) * KB;
      for (int kb0 = 0; kb0 < KB; kb0 += KPS) {
        const int nk = min(KPS, KB - kb0);
        if (!bounded_wait(smem_u32(&sh->empty[stage]), phase ^ 1u, &sh->abort_flag, args.status)) { ok = false; break; }
        if (lane == 0) {
          const uint32_t fb_local = smem_u32(&sh->full[stage]);
          const int arow = rt.row0 + 128 * (int)rank;
          // the scale atoms of a stage's k-blocks are adjacent in HBM: one copy
          // of KPS A atoms and one of 2 * KPS B atoms (a copy past the end of a
          // tile's k-blocks reads atoms it does not use, zeros past the table),
          // counted on a barrier of their own so that their tensor-memory
          // copies need not wait for the stage's operands
          const uint32_t ssa = smem_u32(sSF + stage * KPS * SF_STAGE);
          const uint32_t ssb = ssa + KPS * mx::kAtomBytes;
          const uint32_t sb_local = smem_u32(&sfa[stage]);
          if constexpr (PAIR) {
            if (leader) { mbar_arrive_expect_tx(fb_local, 2 * nk * (A_STAGE + B_STAGE)); mbar_arrive_expect_tx(sb_local, 2 * KPS * SF_STAGE); }
            const uint32_t sbb = mapa_shared(sb_local, 0);
            tma_load_2d_pair(ssa, &tmSA, sbb, 0, blk * KB + kb0);
            tma_load_2d_pair(ssb, &tmSB, sbb, 0, (wat + kb0) * 2);
          } else {
            mbar_arrive_expect_tx(fb_local, nk * (A_STAGE + B_STAGE));
            mbar_arrive_expect_tx(sb_local, KPS * SF_STAGE);
            tma_load_2d(ssa, &tmSA, sb_local, 0, blk * KB + kb0);
            tma_load_2d(ssb, &tmSB, sb_local, 0, (wat + kb0) * 2);
          }
          for (int j = 0; j < nk; ++j) {
            const int kb = kb0 + j, q = stage * KPS + j;
            const uint32_t sa = smem_u32(sA + q * A_STAGE), sb = smem_u32(sB + q * B_STAGE);
            // DX8 reduces over [dh1 | dh3] x [W1 | W3]: the second pair of maps
            // from k-block kb_split on
            const bool second = MODE == kDx8 && kb >= args.kb_split;
            const int kx = (second ? kb - args.kb_split : kb) * BK;
            const CUtensorMap* ma = second ? &tmA1 : &tmA;
            const CUtensorMap* mb = second ? &tmB1 : &tmB0;
            if constexpr (PAIR) {
              const uint32_t fb = mapa_shared(fb_local, 0);
              tma_load_2d_pair(sa, ma, fb, kx, arow);
              if constexpr (MODE == kUp8) {
                // the even CTA stages the 96 W1 rows, the odd CTA the same W3 rows
                tma_load_3d_pair(sb, rank == 0 ? &tmB0 : &tmB1, fb, kx, n0, rt.e);
              } else {
                tma_load_3d_pair(sb, mb, fb, kx, n0 + 96 * (int)rank, rt.e);
              }
            } else {
              tma_load_2d(sa, ma, fb_local, kx, arow);
              if constexpr (MODE == kUp8) {
                // 96 rows of W1 then the same 96 rows of W3
                tma_load_3d(sb, &tmB0, fb_local, kx, n0, rt.e);
                tma_load_3d(sb + 96 * BK, &tmB1, fb_local, kx, n0, rt.e);
              } else {
                tma_load_3d(sb, mb, fb_local, kx, n0, rt.e);
              }
            }
          }
        }
        __syncwarp();
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && leader && lane == 0) {
      // the (even CTA's) full barriers count every copy of the stage
      for (int s = 0; s < S; ++s)
        if (issued & (1u << s)) { drain_wait(smem_u32(&sh->full[s]), (last_par >> s) & 1u); drain_wait(smem_u32(&sfa[s]), (last_par >> s) & 1u); }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (leader) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true, issued_any = false;
      for (int t = unit; t < total && ok; t += nunits) {
        if (!bounded_wait(smem_u32(&sh->tempty[acc]), acc_phase ^ 1u, &sh->abort_flag, args.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dt = tmem + F::acc_col(acc);
        for (int kb0 = 0; kb0 < KB; kb0 += KPS) {
          const int nk = min(KPS, KB - kb0);
          // the stage's scales are in tensor memory and its operands have landed
          // (two barriers: with the scale copies waiting for the atoms alone,
          // their latency hides under the operand copies, which costs the MMA
          // lane a second wait but took the train_e128 forward from 0.822 to
          // 0.796 ms against one wait on copies issued after the full barrier)
          if (!bounded_wait(smem_u32(&sfull[stage]), phase, &sh->abort_flag, args.status) ||
              !bounded_wait(smem_u32(&sh->full[stage]), phase, &sh->abort_flag, args.status)) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) {
            for (int j = 0; j < nk; ++j) {
              const int q = stage * KPS + j;
              const uint32_t sfa_t = tmem + F::sf_col(stage) + 12 * j, sfb_t = sfa_t + 4;
              const uint32_t sa = smem_u32(sA + q * A_STAGE), sb = smem_u32(sB + q * B_STAGE);
#pragma unroll
              for (int kk = 0; kk < BK / 32; ++kk) {
                const uint64_t ad = sdesc_sw128(sa + kk * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(sb + kk * 32, 16, 1024);
                const uint32_t accum = (kb0 + j > 0 || kk > 0) ? 1u : 0u;
                if constexpr (PAIR) mma_mxf8_pair(dt, ad, bd, idesc_mxf8(256, BN, kk), sfa_t, sfb_t, accum);
                else mma_mxf8(dt, ad, bd, idesc_mxf8(128, BN, kk), sfa_t, sfb_t, accum);
              }
            }
            const uint32_t eb = smem_u32(&sh->empty[stage]);
            if constexpr (PAIR) mma_commit_pair_both(eb);
            else mma_commit(eb);
          }
          issued_any = true;
          __syncwarp();
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (lane == 0) {
          const uint32_t tf = smem_u32(&sh->tfull[acc]);
          if constexpr (PAIR) mma_commit_pair_both(tf);
          else mma_commit(tf);
        }
        __syncwarp();
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok && issued_any && lane == 0) {
        if constexpr (PAIR) mma_commit_pair(mapa_shared(smem_u32(&sh->drain), 0));
        else mma_commit(smem_u32(&sh->drain));
        drain_wait(smem_u32(&sh->drain), 0);
      }
    }
    // the odd CTA's MMA warp only holds its half of the TMEM allocation
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int lane_q = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stg = sStage + (warp - 2) * kStageBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = unit; t < total; t += nunits) {
      RowTile rt = decode_row_tile<TM>(t, args.E, args.R, s_off, s_ts);
      const int n0 = rt.n_idx * (MODE == kUp8 ? BN / 2 : BN);
      if constexpr (PAIR) {                       // this CTA's 128 rows of the tile
        rt.row0 += 128 * (int)rank;
        rt.rows = max(0, min(128, rt.rows - 128 * (int)rank));
      }
      if (!bounded_wait(smem_u32(&sh->tfull[acc]), acc_phase, &sh->abort_flag, args.status)) break;
      tc_fence_after();
      epilogue8<MODE>(rt, n0, tmem + F::acc_col(acc), lane_q, half, lane, stg, args, &tmO0, &tmO1, &tmO2);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(smem_u32(&sh->tempty[acc]), 0));
        else mbar_arrive(smem_u32(&sh->tempty[acc]));
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    stg_finish(lane);
  } else if (leader) {
    // ------------------------------------------------ scale copies (even CTA)
    // A stage's atoms go to tensor memory from this warp, off the MMA lane:
    // tcgen05.cp of both CTAs' atoms (the pair form) once the stage's atoms
    // have landed, then a commit to sfull[stage] that the MMA lane waits on.
    // The stage's scale columns are rewritten only after the producer
    // refilled the stage, i.e. after the MMAs that read them completed.
    int stage = 0;
    uint32_t phase = 0;
    bool issued = false;
    for (int t = unit; t < total; t += nunits) {
      bool ok = true;
      for (int kb0 = 0; kb0 < KB; kb0 += KPS) {
        const int nk = min(KPS, KB - kb0);
        if (!bounded_wait(smem_u32(&sfa[stage]), phase, &sh->abort_flag, args.status)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          for (int j = 0; j < nk; ++j) {
            const uint32_t sfa_t = tmem + F::sf_col(stage) + 12 * j, sfb_t = sfa_t + 4;
            // the stage's A atoms, then its B atoms (two a k-block)
            const uint32_t ssa = smem_u32(sSF + stage * KPS * SF_STAGE) + j * mx::kAtomBytes;
            const uint32_t ssb = smem_u32(sSF + stage * KPS * SF_STAGE) + (KPS + 2 * j) * mx::kAtomBytes;
            if constexpr (PAIR) {
              tmem_cp_warpx4_pair(sfa_t, sdesc_atom(ssa));
              tmem_cp_warpx4_pair(sfb_t, sdesc_atom(ssb));             // B columns 0..127
              tmem_cp_warpx4_pair(sfb_t + 4, sdesc_atom(ssb + 512));   // B columns 128..191
            } else {
              tmem_cp_warpx4(sfa_t, sdesc_atom(ssa));
              tmem_cp_warpx4(sfb_t, sdesc_atom(ssb));
              tmem_cp_warpx4(sfb_t + 4, sdesc_atom(ssb + 512));
            }
          }
          const uint32_t sb = smem_u32(&sfull[stage]);
          if constexpr (PAIR) mma_commit_pair(mapa_shared(sb, 0));
          else mma_commit(sb);
        }
        issued = true;
        __syncwarp();
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
    if (issued && lane == 0) {            // every copy done before TMEM is freed
      if constexpr (PAIR) mma_commit_pair(mapa_shared(smem_u32(&sfull[S]), 0));
      else mma_commit(smem_u32(&sfull[S]));
      drain_wait(smem_u32(&sfull[S]), 0);
    }
    __syncwarp();
  }

  tc_fence_before();
  // no CTA leaves (or frees TMEM) while its peer may still signal it
  if constexpr (PAIR) cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, kTmemCols);
    else tmem_dealloc(tmem, kTmemCols);
  }
}

// Row-major activation scales [R][K/32] -> atoms (layout in mx_common.cuh).
// Thread per (row, k-block): the row's four scale bytes of the k-block, one
// 32-bit word of an atom.  Offsets are clamped to [0, R] as the GEMM reads
// them, so every word lands inside the (ceil(R/128) + E) K/128 atoms.
// kb_off / KB_total place a table that covers only part of the reduction
// (DX8's dh1 and dh3 halves of K = 2h) inside atoms of the whole K.
__global__ void __launch_bounds__(256)
act_atoms_kernel(const uint8_t* __restrict__ s, const int32_t* __restrict__ offsets, int E, int R, int K,
                 int kb_off, int KB_total, uint32_t* __restrict__ atoms) {
  pdl_enter();
  const int KB = K / 128;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)R * KB) return;
  const int row = (int)(i / KB), kb = (int)(i - (long long)row * KB);
  int lo = 0, hi = E;                 // the expert whose segment holds the row
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(offsets + mid) <= row) lo = mid; else hi = mid;
  }
  const int off = max(0, min(__ldg(offsets + lo), row));
  const int srow = row - off + 128 * mx::act_block0(off, lo);
  const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(s + (size_t)row * (K / 32)) + kb);
  atoms[((size_t)(srow >> 7) * KB_total + kb_off + kb) * 128 + (srow & 31) * 4 + ((srow >> 5) & 3)] = v;
}

// Row-major weight scales [E][N][Ksrc/32] -> the atoms of the GEMM's column
// tiles of `cols` columns over KB 128-deep k-blocks.  col_split = 96: tile
// columns 0-95 are rows of s0, 96-191 the same rows of s1 (the up-projection);
// kb_split < KB: k-blocks from kb_split on come from s1 (DX8's [W1 | W3]).
// Thread per (tile k-block, column 0..255); columns 192-255 and rows past N
// are zero.
__global__ void __launch_bounds__(256)
weight_atoms_kernel(const uint8_t* __restrict__ s0, const uint8_t* __restrict__ s1, int E, int N, int Ksrc,
                    int cols, int col_split, int NT, int KB, int kb_split, uint32_t* __restrict__ atoms) {
  pdl_enter();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)E * NT * KB * 256) return;
  const int c = (int)(i & 255);
  const long long p = i >> 8;                     // ((e * NT + nt) * KB + kb)
  const int kb = (int)(p % KB), nt = (int)((p / KB) % NT), e = (int)(p / ((long long)KB * NT));
  const uint8_t* tab = s0;
  int n = nt * cols + c, kk = kb;
  if (col_split > 0 && c >= col_split) { tab = s1; n -= col_split; }
  if (kb >= kb_split) { tab = s1; kk = kb - kb_split; }
  uint32_t v = 0;
  if (c < BN && n < N)
    v = __ldg(reinterpret_cast<const uint32_t*>(tab + ((size_t)e * N + n) * (Ksrc / 32)) + kk);
  atoms[(p * 2 + (c >> 7)) * 128 + (c & 31) * 4 + ((c >> 5) & 3)] = v;
}

// 2-D map over 512-byte atoms (32-bit elements, box = `count` whole atoms)
inline bool map_atoms(CUtensorMap* m, const void* ptr, uint64_t n_atoms, uint32_t count) {
  auto fn = encode_fn();
  if (!fn || n_atoms == 0) return false;
  cuuint64_t dims[2] = {128, n_atoms};
  cuuint64_t strides[1] = {mx::kAtomBytes};
  cuuint32_t box[2] = {128, count};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool PAIR>
constexpr size_t smem_bytes8(int E) {
  return 1024 + (size_t)Form<PAIR>::STAGES * stage_bytes<PAIR>() + (size_t)kEpiWarps * kStageBytes +
         sizeof(PipeShared<Form<PAIR>::STAGES>) + 8 * (2 * Form<PAIR>::STAGES + 1) + 2 * (size_t)(E + 1) * 4;
}
static_assert(smem_bytes8<true>(kMaxExperts8) <= 227 * 1024, "pair MXFP8 kernel fits in shared memory");
static_assert(smem_bytes8<false>(kMaxExperts8) <= 227 * 1024, "MXFP8 kernel fits in shared memory");

struct Maps8 { CUtensorMap a, a1, b0, b1, sa, sb, o0, o1, o2; };

template <int MODE, bool PAIR>
int launch8(const Maps8& m, const Args8& args, long long tiles_upper, cudaStream_t s) {
  auto kern = grouped_mxfp8_kernel<MODE, PAIR>;
  static bool attr_done[64] = {false};
  if (ensure_smem_attr(kern, smem_bytes8<PAIR>(kMaxExperts8), attr_done) != MOE_OK) return MOE_ERR_CUDA;
  const long long ub = tiles_upper > 0 ? tiles_upper : 1;
  if constexpr (PAIR) {
    const long long half_sms = sm_count() / 2;
    const long long npairs = ub < half_sms ? ub : half_sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * (npairs > 0 ? npairs : 1)));
    cfg.blockDim = dim3(kThreads8);
    cfg.dynamicSmemBytes = smem_bytes8<PAIR>(args.E);
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2; at[0].val.clusterDim.y = 1; at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, m.a, m.a1, m.b0, m.b1, m.sa, m.sb, m.o0, m.o1, m.o2, args) != cudaSuccess) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  } else {
    const long long g = ub < sm_count() ? ub : sm_count();
    (void)launch_pdl(kern, (unsigned)g, kThreads8, smem_bytes8<PAIR>(args.E), s, m.a, m.a1, m.b0, m.b1, m.sa, m.sb,
                     m.o0, m.o1, m.o2, args);
  }
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

// CTA pairs once the experts average at least this many rows (the 256-row
// tiles waste less than they gain); single CTAs below.
constexpr long long kPairMinRows8 = 512;

}  // namespace
}  // namespace moe

using namespace moe;
using namespace moe::gemm;

extern "C" size_t moe_mxfp8_weight_atom_bytes(int E, int d, int h) {
  if (E < 1 || d <= 0 || h <= 0 || d % 128 != 0 || h % 128 != 0) return 0;
  return (size_t)mx::weight_atom_bytes(E, d, h);
}

extern "C" int moe_mxfp8_weight_scale_atoms(const uint8_t* w1s, const uint8_t* w3s, const uint8_t* w2s,
                                            int E, int d, int h, uint8_t* atoms, moe_stream_t stream) {
  if (E < 1 || E > kMaxExperts || d <= 0 || h <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 128 != 0 || h % 128 != 0) return MOE_ERR_UNSUPPORTED;
  auto al4 = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!al4(w1s) || !al4(w3s) || !al4(w2s)) return MOE_ERR_INVALID_ARG;
  MOE_CHECK_PTR(atoms);
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* up = reinterpret_cast<uint32_t*>(atoms);
  uint32_t* dn = up + mx::up_atom_count(E, d, h) * 128;
  const int ntu = mx::up_tiles(h), ntd = mx::down_tiles(d);
  const long long nu = (long long)E * ntu * (d / 128) * 256, nd = (long long)E * ntd * (h / 128) * 256;
  (void)launch_pdl(weight_atoms_kernel, (unsigned)((nu + 255) / 256), 256, 0, s, w1s, w3s, E, h, d,
                   mx::kUpCols, mx::kUpCols, ntu, d / 128, d / 128, up);
  (void)launch_pdl(weight_atoms_kernel, (unsigned)((nd + 255) / 256), 256, 0, s, w2s, w2s, E, d, h,
                   mx::kDownCols, 0, ntd, h / 128, h / 128, dn);
  MOE_LAUNCH_CHECK(2);
  return MOE_OK;
}

extern "C" int moe_grouped_swiglu_fwd_mxfp8(
    const uint8_t* xq, const uint8_t* xs, const int32_t* offsets, int R, int E, int d, int h,
    const uint8_t* w1q, const uint8_t* w3q, const uint8_t* w2q, const uint8_t* w_atoms,
    moe_bf16_t* h1, moe_bf16_t* h3, moe_bf16_t* a, uint8_t* aq, uint8_t* as, moe_bf16_t* yp,
    void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (R < 0 || E < 1 || E > kMaxExperts || d <= 0 || h <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 128 != 0 || h % 128 != 0 || E > kMaxExperts8) return MOE_ERR_UNSUPPORTED;
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  const size_t need = mx_scratch_end(R, E, d, h);
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (R == 0) return MOE_OK;
  MOE_CHECK_PTR(xq); MOE_CHECK_PTR(offsets); MOE_CHECK_PTR(w1q); MOE_CHECK_PTR(w3q);
  MOE_CHECK_PTR(w2q); MOE_CHECK_PTR(w_atoms); MOE_CHECK_PTR(h1); MOE_CHECK_PTR(h3); MOE_CHECK_PTR(aq);
  MOE_CHECK_PTR(yp);
  if (a != nullptr && !aligned16(a)) return MOE_ERR_INVALID_ARG;      // a may be NULL
  // the row-major scale tables are read 4 bytes at a time
  auto al4 = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!al4(xs) || !al4(as)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  uint32_t* xatoms = reinterpret_cast<uint32_t*>(wsb + mx_scratch_x(R, E, d, h));
  uint32_t* aatoms = reinterpret_cast<uint32_t*>(wsb + mx_scratch_a(R, E, d, h));
  const long long nbx = mx::act_atom_blocks(R, E) * (d / 128), nba = mx::act_atom_blocks(R, E) * (h / 128);
  const uint8_t* up_atoms = w_atoms;
  const uint8_t* dn_atoms = w_atoms + mx::up_atom_count(E, d, h) * mx::kAtomBytes;
  const long long n_up_atoms = mx::up_atom_count(E, d, h);
  const long long n_dn_atoms = (long long)E * mx::down_tiles(d) * (h / 128) * 2;
  const bool pair = (long long)R >= kPairMinRows8 * E;
  const int TM = pair ? 256 : 128;
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint32_t brows = pair ? 96 : 192;
  const uint32_t kps = pair ? Form<true>::KPS : Form<false>::KPS;
  Maps8 mu{}, md{};
  if (!map2d(&mu.a, xq, d, R, BK, 128, U8, 1) || !map2d(&mu.a1, xq, d, R, BK, 128, U8, 1) ||
      !map3d(&mu.b0, w1q, d, h, E, BK, 96, U8, 1) ||
      !map3d(&mu.b1, w3q, d, h, E, BK, 96, U8, 1) || !map_atoms(&mu.sa, xatoms, nbx, kps) ||
      !map_atoms(&mu.sb, up_atoms, n_up_atoms, 2 * kps) ||
      !map2d(&md.a, aq, h, R, BK, 128, U8, 1) || !map3d(&md.b0, w2q, h, d, E, BK, brows, U8, 1) ||
      !map_atoms(&md.sa, aatoms, nba, kps) || !map_atoms(&md.sb, dn_atoms, n_dn_atoms, 2 * kps))
    return MOE_ERR_CUDA;
  md.b1 = md.b0; md.a1 = md.a;
  if (!map2d_out(&mu.o0, h1, h, R, h) || !map2d_out(&mu.o1, h3, h, R, h) ||
      !map2d_out(&mu.o2, a ? a : h1, h, R, h) || !map2d_out(&md.o0, yp, d, R, d))
    return MOE_ERR_CUDA;
  md.o1 = md.o0; md.o2 = md.o0;
  Args8 g{};
  g.offsets = offsets; g.E = E; g.R = R; g.d = d; g.h = h; g.status = reinterpret_cast<int*>(ws);
  // up-projection: K = d, 96 columns of W1 and of W3 per tile
  g.kb_total = d / BK; g.kb_split = g.kb_total; g.n_tiles = mx::up_tiles(h); g.N = h;
  g.out0 = h1; g.out1 = h3; g.out2 = a; g.aq = aq; g.as = as;
  const long long lx = (long long)R * (d / 128), la = (long long)R * (h / 128);
  (void)launch_pdl(act_atoms_kernel, (unsigned)((lx + 255) / 256), 256, 0, s, xs, offsets, E, R, d, 0,
                   d / 128, xatoms);
  MOE_LAUNCH_CHECK(1);
  int st = pair ? launch8<kUp8, true>(mu, g, row_tiles_upper(R, E, g.n_tiles, TM), s)
                : launch8<kUp8, false>(mu, g, row_tiles_upper(R, E, g.n_tiles, TM), s);
  if (st != MOE_OK) return st;
  // down-projection: K = h
  Args8 g2 = g;
  g2.kb_total = h / BK; g2.kb_split = g2.kb_total; g2.n_tiles = mx::down_tiles(d); g2.N = d;
  g2.out0 = yp; g2.out1 = nullptr; g2.out2 = nullptr; g2.aq = nullptr; g2.as = nullptr;
  (void)launch_pdl(act_atoms_kernel, (unsigned)((la + 255) / 256), 256, 0, s, as, offsets, E, R, h, 0,
                   h / 128, aatoms);
  MOE_LAUNCH_CHECK(1);
  return pair ? launch8<kDown8, true>(md, g2, row_tiles_upper(R, E, g2.n_tiles, TM), s)
              : launch8<kDown8, false>(md, g2, row_tiles_upper(R, E, g2.n_tiles, TM), s);
}

extern "C" size_t moe_mxfp8_dx_weight_atom_bytes(int E, int d, int h) {
  if (E < 1 || d <= 0 || h <= 0 || d % 128 != 0 || h % 128 != 0) return 0;
  return (size_t)E * mx::down_tiles(d) * (2 * h / 128) * 2 * mx::kAtomBytes;
}

extern "C" int moe_mxfp8_dx_weight_scale_atoms(const uint8_t* w1s_h, const uint8_t* w3s_h, int E, int d, int h,
                                               uint8_t* atoms, moe_stream_t stream) {
  if (E < 1 || E > kMaxExperts || d <= 0 || h <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 128 != 0 || h % 128 != 0) return MOE_ERR_UNSUPPORTED;
  auto al4 = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!al4(w1s_h) || !al4(w3s_h)) return MOE_ERR_INVALID_ARG;
  MOE_CHECK_PTR(atoms);
  const int nt = mx::down_tiles(d), KB = 2 * h / 128;
  const long long n = (long long)E * nt * KB * 256;
  (void)launch_pdl(weight_atoms_kernel, (unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream, w1s_h,
                   w3s_h, E, d, h, mx::kDownCols, 0, nt, KB, h / 128, reinterpret_cast<uint32_t*>(atoms));
  MOE_LAUNCH_CHECK(1);
  return MOE_OK;
}

extern "C" int moe_grouped_swiglu_bwd_dx_mxfp8(
    const uint8_t* dh1q, const uint8_t* dh1s, const uint8_t* dh3q, const uint8_t* dh3s,
    const int32_t* offsets, int R, int E, int d, int h, const uint8_t* w1q_h, const uint8_t* w3q_h,
    const uint8_t* dx_atoms, moe_bf16_t* dxp, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (R < 0 || E < 1 || E > kMaxExperts || d <= 0 || h <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 128 != 0 || h % 128 != 0 || E > kMaxExperts8) return MOE_ERR_UNSUPPORTED;
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < mx_scratch_end(R, E, d, h)) return MOE_ERR_WORKSPACE;
  if (R == 0) return MOE_OK;
  MOE_CHECK_PTR(dh1q); MOE_CHECK_PTR(dh3q); MOE_CHECK_PTR(offsets); MOE_CHECK_PTR(w1q_h);
  MOE_CHECK_PTR(w3q_h); MOE_CHECK_PTR(dx_atoms); MOE_CHECK_PTR(dxp);
  auto al4 = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!al4(dh1s) || !al4(dh3s)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* atoms = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + mx_scratch_x(R, E, d, h));
  const int KB = 2 * h / BK, KBh = h / BK;
  const long long nba = mx::act_atom_blocks(R, E) * KB;
  const long long n_w_atoms = (long long)E * mx::down_tiles(d) * KB * 2;
  const bool pair = (long long)R >= kPairMinRows8 * E;
  const int TM = pair ? 256 : 128;
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint32_t brows = pair ? 96 : 192;
  const uint32_t kps = pair ? Form<true>::KPS : Form<false>::KPS;
  Maps8 m{};
  if (!map2d(&m.a, dh1q, h, R, BK, 128, U8, 1) || !map2d(&m.a1, dh3q, h, R, BK, 128, U8, 1) ||
      !map3d(&m.b0, w1q_h, h, d, E, BK, brows, U8, 1) || !map3d(&m.b1, w3q_h, h, d, E, BK, brows, U8, 1) ||
      !map_atoms(&m.sa, atoms, nba, kps) || !map_atoms(&m.sb, dx_atoms, n_w_atoms, 2 * kps) ||
      !map2d_out(&m.o0, dxp, d, R, d))
    return MOE_ERR_CUDA;
  m.o1 = m.o0; m.o2 = m.o0;
  // the row-major scales of dh1 and dh3 become the two halves of K = 2h
  const long long l = (long long)R * KBh;
  (void)launch_pdl(act_atoms_kernel, (unsigned)((l + 255) / 256), 256, 0, s, dh1s, offsets, E, R, h, 0, KB,
                   atoms);
  (void)launch_pdl(act_atoms_kernel, (unsigned)((l + 255) / 256), 256, 0, s, dh3s, offsets, E, R, h, KBh, KB,
                   atoms);
  MOE_LAUNCH_CHECK(2);
  Args8 g{};
  g.offsets = offsets; g.E = E; g.R = R; g.d = d; g.h = h; g.status = reinterpret_cast<int*>(ws);
  g.kb_total = KB; g.kb_split = KBh; g.n_tiles = mx::down_tiles(d); g.N = d;
  g.out0 = dxp;
  return pair ? launch8<kDx8, true>(m, g, row_tiles_upper(R, E, g.n_tiles, TM), s)
              : launch8<kDx8, false>(m, g, row_tiles_upper(R, E, g.n_tiles, TM), s);
}
