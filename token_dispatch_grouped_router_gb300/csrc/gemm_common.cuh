// Pieces shared by the persistent tcgen05 grouped GEMMs (bf16 and MXFP8):
// bounded mbarrier waits, the epilogue's coalescing staging buffer, the
// SwiGLU activation, the row-grouped tile table built from the device
// offsets, and host-side TMA tensor-map encoding.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm103_ptx.cuh"

namespace moe {
namespace gemm {

using namespace ptx;

constexpr int kEpiWarps = 8;                    // two per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kEpiWarps;   // producer warp, MMA warp, epilogue
// per-epilogue-warp staging buffer: a 32-row x 32-column bf16 chunk with an
// 80-byte row pitch, so both the row-per-thread side and the coalesced side
// of the transpose are free of bank conflicts
constexpr int kStagePitch = 80;
constexpr int kStageBytes = 32 * kStagePitch;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s; a step takes milliseconds

// Pipeline barriers and CTA-wide flags of one persistent GEMM CTA.
template <int STAGES>
struct PipeShared {
  uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], drain;
  uint64_t rfull[4], rempty[4];   // CTA-pair DA: the epilogue's h1/h3 ring
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int wg_whole, wg_split, wg_zero;   // CTA-pair wgrad: the device-built tile plan
};

// Wait for the phase `parity` of an mbarrier; give up after kWaitLimitNs (or
// when another warp of the CTA has given up), recording MOE_DEV_WAIT_TIMEOUT.
// KIND 0: try_wait (the thread may be suspended until the phase completes);
// 1: the same with cluster-scope acquire; 2: polling with test_wait.
enum WaitKind : int { kWaitTry = 0, kWaitTryCluster = 1, kWaitPoll = 2 };
template <int KIND = kWaitTry>
__device__ __forceinline__ bool probe_phase(uint32_t bar, uint32_t parity) {
  if constexpr (KIND == kWaitTryCluster) return mbar_try_wait_cluster(bar, parity);
  else if constexpr (KIND == kWaitPoll) return mbar_test_wait(bar, parity);
  else return mbar_try_wait(bar, parity);
}
template <int KIND = kWaitTry>
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, int* abort_flag,
                                             int* status) {
  if (probe_phase<KIND>(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (probe_phase<KIND>(bar, parity)) return true;
    if ((n & 127u) == 0) {
      if (*(volatile int*)abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *(volatile int*)abort_flag = 1;
        set_status(status, MOE_DEV_WAIT_TIMEOUT);
        return false;
      }
    }
  }
}

// wait used only while draining after an abort: bounded, reports nothing
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

// ------------------------------------------------------------ activation
// sigmoid through the identity sigmoid(x) = (1 + tanh(x / 2)) / 2 on the
// hardware tanh approximation (one MUFU op instead of an exp and a divide);
// its error is far below the bf16 rounding of the stored results
__device__ __forceinline__ float tanh_hw(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigmoid_f(float x) { return fmaf(0.5f, tanh_hw(0.5f * x), 0.5f); }
__device__ __forceinline__ float silu_f(float x) { return x * sigmoid_f(x); }

// ---------------------------------------------------- epilogue staging
__device__ __forceinline__ void pack_row32(const float* v, uint4 (&o)[4]) {
  uint32_t* w = reinterpret_cast<uint32_t*>(o);
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
}

// The staging buffer may still be the source of this warp's last TMA store:
// lane 0 waits until the copy engine has read it, then the warp goes on.
// (store_chunk and chunk_to_row do not wait: a caller that mixes them with
// TMA stores calls this first.)
__device__ __forceinline__ void stg_acquire(int lane) {
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
}

// The warp's 32 rows (one per lane, 32 values each) -> global memory at
// g[row * ld + 0..31] for rows < nrows, through the staging buffer so that each
// store instruction writes 8 rows x 64 contiguous bytes.
__device__ __forceinline__ void store_chunk(uint8_t* stg, const float* v, int lane, uint16_t* g,
                                            size_t ld, int nrows) {
  uint4 o[4];
  pack_row32(v, o);
#pragma unroll
  for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(stg + lane * kStagePitch + 16 * i) = o[i];
  __syncwarp();
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int p = it * 32 + lane, row = p >> 2, c = p & 3;
    if (row < nrows)
      st_v4(g + (size_t)row * ld + 8 * c, *reinterpret_cast<const uint4*>(stg + row * kStagePitch + 16 * c));
  }
  __syncwarp();
}

// 32 bytes per lane-row (e.g. 32 fp8 codes) -> g[row * ld + 0..31] for rows <
// nrows; each store instruction writes 16 rows x 32 contiguous bytes.
__device__ __forceinline__ void store_chunk_bytes32(uint8_t* stg, const uint4 (&v)[2], int lane,
                                                    uint8_t* g, size_t ld, int nrows) {
  *reinterpret_cast<uint4*>(stg + lane * kStagePitch) = v[0];
  *reinterpret_cast<uint4*>(stg + lane * kStagePitch + 16) = v[1];
  __syncwarp();
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int p = it * 32 + lane, row = p >> 1, c = p & 1;
    if (row < nrows)
      st_v4(g + (size_t)row * ld + 16 * c, *reinterpret_cast<const uint4*>(stg + row * kStagePitch + 16 * c));
  }
  __syncwarp();
}

// Coalesced load of a 32-row x 32-column bf16 chunk (8 rows x 64 bytes per
// instruction); piece it*32+lane holds row (it*32+lane)/4, 16-byte column (..)%4.
__device__ __forceinline__ void load_chunk(uint4 (&q)[4], const uint16_t* g, size_t ld, int lane,
                                           int nrows) {
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int p = it * 32 + lane, row = p >> 2, c = p & 3;
    q[it] = row < nrows ? ld_nc_v4(g + (size_t)row * ld + 8 * c) : make_uint4(0, 0, 0, 0);
  }
}

// Pieces from load_chunk -> this lane's own row (32 bf16 values, packed in pairs).
__device__ __forceinline__ void chunk_to_row(const uint4 (&q)[4], uint8_t* stg, int lane,
                                             uint32_t (&w)[16]) {
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int p = it * 32 + lane, row = p >> 2, c = p & 3;
    *reinterpret_cast<uint4*>(stg + row * kStagePitch + 16 * c) = q[it];
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 t = *reinterpret_cast<const uint4*>(stg + lane * kStagePitch + 16 * i);
    w[4 * i + 0] = t.x; w[4 * i + 1] = t.y; w[4 * i + 2] = t.z; w[4 * i + 3] = t.w;
  }
  __syncwarp();
}

// The warp's 32 x 32 chunk (one row per lane) stored by TMA: the lanes write
// it to the staging buffer in the 64-byte swizzled layout of the output
// descriptor (CU_TENSOR_MAP_SWIZZLE_64B, 32 x 32 box; 16-byte piece c of row
// r at piece position c ^ ((r >> 1) & 3), buffer on a 512-byte boundary, so
// every 8 lanes cover all banks), then lane 0 issues one bulk store.  The
// descriptor clips rows and columns outside the tensor; rows inside it are
// all written, so callers use this only for slices whose 32 rows are theirs.
__device__ __forceinline__ void stage_chunk_sw64(uint8_t* stg, const float* v, int lane) {
  uint4 o[4];
  pack_row32(v, o);
  stg_acquire(lane);
  const int x = (lane >> 1) & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(stg + lane * 64 + 16 * (i ^ x)) = o[i];
  fence_proxy_async_smem();
  __syncwarp();
}
__device__ __forceinline__ void store_chunk_tma(uint8_t* stg, const float* v, int lane,
                                                const CUtensorMap* map, int col, int row) {
  stage_chunk_sw64(stg, v, lane);
  if (lane == 0) {
    tma_store_2d(map, smem_u32(stg), col, row);
    bulk_commit();
  }
}
__device__ __forceinline__ void store_chunk_tma3(uint8_t* stg, const float* v, int lane,
                                                 const CUtensorMap* map, int col, int row, int z) {
  stage_chunk_sw64(stg, v, lane);
  if (lane == 0) {
    tma_store_3d(map, smem_u32(stg), col, row, z);
    bulk_commit();
  }
}
// end of a warp's epilogue: its bulk stores have completed
__device__ __forceinline__ void stg_finish(int lane) {
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

// ------------------------------------------------- row-grouped tile table
// Expert e owns ceil(n_e / TM) row blocks x n_tiles column blocks; the
// tiles are numbered expert-major.  Warp 0 writes the expert offsets (clamped
// to [0, R]) into s_off[0..E] and the first tile of every expert into
// s_ts[0..E] (s_ts[E] = number of tiles).  s_off must already hold offsets.
template <int TM = 128>
__device__ __forceinline__ int build_row_tile_table(const int* s_off, int* s_ts, int E, int R,
                                                    int n_tiles, int lane) {
  int carry = 0;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    int cnt = 0;
    if (e < E) {
      const int lo = max(0, min(s_off[e], R));
      const int hi = max(lo, min(s_off[e + 1], R));
      cnt = ((hi - lo + TM - 1) / TM) * n_tiles;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (e < E) s_ts[e] = carry + incl - cnt;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) s_ts[E] = carry;
  return carry;
}

struct RowTile {
  int e, row0, rows, n_idx;
};

// Tile t -> expert, first row, valid rows (<= TM) and column-block index;
// within an expert the column block varies fastest, so the CTAs working at
// the same time on one row block read its rows from DRAM once (the expert's
// weights stay in L2 while its row blocks go by).
template <int TM = 128>
__device__ __forceinline__ RowTile decode_row_tile(int t, int E, int R, const int* s_off,
                                                   const int* s_ts) {
  int lo = 0, hi = E;                 // invariant: s_ts[lo] <= t < s_ts[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_ts[mid] <= t) lo = mid; else hi = mid;
  }
  RowTile r;
  r.e = lo;
  const int seg0 = max(0, min(s_off[lo], R));
  const int seg1 = max(seg0, min(s_off[lo + 1], R));
  const int mt = (seg1 - seg0 + TM - 1) / TM;
  const int l = t - s_ts[lo];
  const int nt = (s_ts[lo + 1] - s_ts[lo]) / mt;     // column blocks
  const int m_idx = l / nt;
  r.n_idx = l % nt;
  r.row0 = seg0 + m_idx * TM;
  r.rows = min(TM, seg1 - r.row0);
  return r;
}

// ------------------------------------------------------------ host side
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      (void)cudaGetLastError();
  }
  return fn;
}

// 2-D map over a row-major [outer, inner] tensor, box [box_outer, box_inner],
// 128-byte swizzle, zero fill out of bounds.
inline bool map2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                  uint32_t box_inner, uint32_t box_outer,
                  CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, uint32_t esize = 2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output descriptors for the TMA-stored epilogue: bf16 [rows, cols] with row
// stride ld (elements), or [outer, mid, inner]; 32-column boxes (32 rows, or
// box_rows) in the 64-byte swizzle.
inline bool map2d_out(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t ld,
                      uint32_t box_rows = 32) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
inline bool map3d_out(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t mid, uint64_t outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over a row-major [outer, mid, inner] tensor, box [1, box_mid, box_inner]
inline bool map3d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t mid, uint64_t outer,
                  uint32_t box_inner, uint32_t box_mid,
                  CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, uint32_t esize = 2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * esize, inner * mid * esize};
  cuuint32_t box[3] = {box_inner, box_mid, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Persistent grid for a row-grouped GEMM: at most one CTA per SM; the real
// tile count is only known on the device (<= (ceil(R/128) + E) * n_tiles) and
// CTAs without a tile exit at once.
inline long long row_tiles_upper(int R, int E, int n_tiles, int tm = 128) {
  return ((long long)(R + tm - 1) / tm + E) * n_tiles;
}
inline int row_grid_upper(int R, int E, int n_tiles) {
  long long ub = row_tiles_upper(R, E, n_tiles);
  long long g = sm_count();
  return (int)(ub < g ? (ub > 0 ? ub : 1) : g);
}

// Sets the kernel's dynamic shared memory limit once per device (so that no
// non-stream CUDA call happens on later, possibly graph-captured, calls).
template <typename K>
inline int ensure_smem_attr(K kern, size_t bytes, bool (&done)[64]) {
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (!done[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    done[dev] = true;
  }
  return MOE_OK;
}

}  // namespace gemm
}  // namespace moe
