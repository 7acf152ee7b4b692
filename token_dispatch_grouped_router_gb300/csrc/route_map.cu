// Device-resident route map: per-expert counts, offsets and the stable
// slot <-> row permutation, built with no host synchronisation.
//
// "OLMo-core 3：MoE 训练栈让专家池越大、吞吐不再越慢", section "另外两处税：主机同步
// 与 padding": the routing counts, each expert's row count (the grouped GEMM's
// M dimensions) and the per-expert permutation are all expressed by a route
// map generated on the device, which removes the two host syncs of the
// block all-to-all path.
//
// Three launches, all integer work, deterministic:
//  1. route_count: block b owns slots [b*1024, (b+1)*1024).  Each of its 8
//     warps walks 128 consecutive slots in order, ranking every slot among
//     the same-expert slots before it (match_any + popc) against a per-warp
//     shared histogram.  Warp histograms are then scanned per expert, giving
//     every slot its stable rank inside the block and the block's histogram.
//  2. route_scan: one block scans the block histograms per expert (column
//     scan over blocks -> block base per expert, counts[e]) and then scans
//     counts over experts -> offsets.
//  3. route_place: row = offsets[e] + block_base[b][e] + rank; writes
//     row_of_slot[s] and its inverse slot_of_row[row].
// Slots of one expert therefore land in ascending slot order (stable).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kRCThreads = 256;                     // 8 warps
constexpr int kRCWarps = kRCThreads / 32;
constexpr int kSlotsPerWarp = kRouteChunk / kRCWarps;   // 128
constexpr int kIters = kSlotsPerWarp / 32;              // 4

__global__ void __launch_bounds__(kRCThreads)
route_count_kernel(const int32_t* __restrict__ idx, int R, int E,
                   int32_t* __restrict__ chunk_counts, int32_t* __restrict__ local_rank,
                   int* __restrict__ status) {
  pdl_enter();
  extern __shared__ int32_t hist[];                 // [kRCWarps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kRCWarps * E; i += kRCThreads) hist[i] = 0;
  __syncthreads();
  int32_t* wh = hist + warp * E;
  const int base = blockIdx.x * kRouteChunk + warp * kSlotsPerWarp;
  int myE[kIters], myRank[kIters];
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    int s = base + it * 32 + lane;
    int e = -1;
    if (s < R) {
      e = __ldg(idx + s);
      if (e < 0 || e >= E) { set_status(status, MOE_DEV_BAD_EXPERT_ID); e = -1; }
    }
    unsigned peers = __match_any_sync(0xffffffffu, e);
    int r = -1;
    if (e >= 0) r = wh[e] + __popc(peers & lt_mask);
    __syncwarp();
    if (e >= 0 && (peers & lt_mask) == 0) wh[e] += __popc(peers);   // group leader
    __syncwarp();
    myE[it] = e;
    myRank[it] = r;
  }
  __syncthreads();
  // exclusive scan of the warp histograms per expert -> warp bases; totals
  int32_t* cc = chunk_counts + (size_t)blockIdx.x * E;
  for (int e = threadIdx.x; e < E; e += kRCThreads) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kRCWarps; ++w) {
      int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    cc[e] = run;
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    int s = base + it * 32 + lane;
    if (s < R && myE[it] >= 0) local_rank[s] = wh[myE[it]] + myRank[it];
  }
}

// Single block of 1024 threads.  The block histograms are scanned per expert
// over the chunks with coalesced accesses: lane = expert (32 consecutive
// experts per warp), the 32 warps split into G = ceil(E / 32) expert groups
// times S = 32 / G chunk ranges.  Pass 1: each warp sums its chunk range per
// expert; the S range sums of an expert are scanned in shared memory; pass 2:
// each warp rewrites its range with the running exclusive prefix.
constexpr int kScanWarps = 32;
__global__ void __launch_bounds__(1024)
route_scan_kernel(int32_t* __restrict__ chunk_counts, int nchunks, int E,
                  int32_t* __restrict__ counts, int32_t* __restrict__ offsets) {
  pdl_enter();
  __shared__ int32_t tot[kMaxExperts];
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t part[kScanWarps * 32];         // [warp] x [lane]: range sums, then bases
  {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = (E + 31) / 32, S = kScanWarps / G;
    const int g = warp / S, j = warp - g * S;
    const int e = 32 * g + lane;
    const int C = (nchunks + S - 1) / S;
    const int b0 = j * C, b1 = min(nchunks, b0 + C);
    const bool active = g < G && e < E;
    int sum = 0;
    if (active) {
#pragma unroll 8
      for (int b = b0; b < b1; ++b) sum += chunk_counts[(size_t)b * E + e];
    }
    part[warp * 32 + lane] = sum;
    __syncthreads();
    // per expert: exclusive scan of its S range sums (thread = expert)
    for (int ee = threadIdx.x; ee < E; ee += blockDim.x) {
      const int gg = ee / 32, l = ee - 32 * gg;
      int run = 0;
      for (int jj = 0; jj < S; ++jj) {
        int* p = &part[(gg * S + jj) * 32 + l];
        const int v = *p;
        *p = run;
        run += v;
      }
      tot[ee] = run;
      counts[ee] = run;
    }
    __syncthreads();
    if (active) {
      int run = part[warp * 32 + lane];
      for (int b = b0; b < b1; ++b) {
        const size_t at = (size_t)b * E + e;
        const int c = chunk_counts[at];
        chunk_counts[at] = run;
        run += c;
      }
    }
  }
  __syncthreads();
  // exclusive scan of tot[0..E) -> offsets (E <= 1024: one element per thread)
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  int v = t < E ? tot[t] : 0;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[w] = incl;
  __syncthreads();
  if (w == 0) {
    int ws = warp_sums[lane];
    int wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    warp_sums[lane] = wi - ws;     // exclusive prefix of warp totals
  }
  __syncthreads();
  int excl = warp_sums[w] + incl - v;
  if (t < E) offsets[t] = excl;
  if (t == E - 1) offsets[E] = excl + v;
}

__global__ void route_place_kernel(const int32_t* __restrict__ idx, int R, int E,
                                   const int32_t* __restrict__ chunk_base,
                                   const int32_t* __restrict__ local_rank,
                                   const int32_t* __restrict__ offsets,
                                   int32_t* __restrict__ row_of_slot,
                                   int32_t* __restrict__ slot_of_row) {
  pdl_enter();
  int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= R) return;
  int e = __ldg(idx + s);
  if (e < 0 || e >= E) {                       // reported by route_count
    row_of_slot[s] = -1;                       // the row kernels skip it
    return;
  }
  int b = s / kRouteChunk;
  int row = __ldg(offsets + e) + __ldg(chunk_base + (size_t)b * E + e) + __ldg(local_rank + s);
  row_of_slot[s] = row;
  slot_of_row[row] = s;
}

// Capacity-padded map: expert e owns rows [e*C, (e+1)*C); its first C routed
// slots in slot order keep their stable rank as the row inside that block,
// later ones are dropped (row -1).  Rows of a block past the expert's kept
// count hold no slot (slot_of_row -1).  One thread per index of the largest
// of the three ranges (slots, padded rows, experts).
__global__ void route_place_capacity_kernel(const int32_t* __restrict__ idx, int R, int E, int C,
                                            const int32_t* __restrict__ chunk_base,
                                            const int32_t* __restrict__ local_rank,
                                            const int32_t* __restrict__ routed_counts,
                                            int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                            int32_t* __restrict__ routed,
                                            int32_t* __restrict__ row_of_slot,
                                            int32_t* __restrict__ slot_of_row) {
  pdl_enter();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long EC = (long long)E * C;
  if (i < R) {
    const int s = (int)i;
    const int e = __ldg(idx + s);
    int row = -1;
    if (e >= 0 && e < E) {
      const int rank = __ldg(chunk_base + (size_t)(s / kRouteChunk) * E + e) + __ldg(local_rank + s);
      if (rank < C) row = e * C + rank;
    }
    row_of_slot[s] = row;
    if (row >= 0) slot_of_row[row] = s;
  }
  if (i < EC) {
    const int e = (int)(i / C), j = (int)(i - (long long)e * C);
    if (j >= __ldg(routed_counts + e)) slot_of_row[i] = -1;     // a zero row
  }
  if (i < E) {
    const int n = __ldg(routed_counts + i);
    counts[i] = min(n, C);
    offsets[i] = (int)i * C;
    if (routed) routed[i] = n;
  }
  if (i == 0) offsets[E] = (int)EC;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_expert_offsets(const int32_t* topk_idx, int T, int k, int E, int32_t* counts,
                                  int32_t* offsets, int32_t* row_of_slot, int32_t* slot_of_row,
                                  void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && k >= 1 && k <= kMaxTopK && E >= 1 && E <= kMaxExperts && k <= E);
  MOE_CHECK_ARG((long long)T * k <= 0x7fffffffLL);
  MOE_CHECK_PTR(counts); MOE_CHECK_PTR(offsets);
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  const long long R = (long long)T * k;
  if (R > 0) { MOE_CHECK_PTR(topk_idx); MOE_CHECK_PTR(row_of_slot); MOE_CHECK_PTR(slot_of_row); }
  RouteScratch L = route_scratch(R, E);
  if (ws_bytes < L.end) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  const int nchunks = (int)((R + kRouteChunk - 1) / kRouteChunk);
  char* wsb = reinterpret_cast<char*>(ws);
  int32_t* chunk_counts = reinterpret_cast<int32_t*>(wsb + L.chunk_counts);
  int32_t* local_rank = reinterpret_cast<int32_t*>(wsb + L.local_rank);
  int* status = reinterpret_cast<int*>(ws);
  if (R == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s) != cudaSuccess) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }
  size_t smem = sizeof(int32_t) * kRCWarps * E;
  (void)launch_pdl(route_count_kernel, nchunks, kRCThreads, smem, s, topk_idx, (int)R, E, chunk_counts,
                                                       local_rank, status);
  (void)launch_pdl(route_scan_kernel, 1, 1024, 0, s, chunk_counts, nchunks, E, counts, offsets);
  (void)launch_pdl(route_place_kernel, (int)((R + 255) / 256), 256, 0, s, topk_idx, (int)R, E, chunk_counts,
                                                             local_rank, offsets, row_of_slot,
                                                             slot_of_row);
  MOE_LAUNCH_CHECK(3);
  return MOE_OK;
}

extern "C" int moe_expert_offsets_capacity(const int32_t* topk_idx, int T, int k, int E, int C,
                                           int32_t* counts, int32_t* offsets, int32_t* row_of_slot,
                                           int32_t* slot_of_row, int32_t* routed, void* ws,
                                           size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && k >= 1 && k <= kMaxTopK && E >= 1 && E <= kMaxExperts && k <= E && C >= 1);
  MOE_CHECK_ARG((long long)T * k <= 0x7fffffffLL && (long long)E * C <= 0x7fffffffLL);
  MOE_CHECK_PTR(counts); MOE_CHECK_PTR(offsets); MOE_CHECK_PTR(slot_of_row);
  if (routed && !aligned16(routed)) return MOE_ERR_INVALID_ARG;
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  const long long R = (long long)T * k;
  if (R > 0) { MOE_CHECK_PTR(topk_idx); MOE_CHECK_PTR(row_of_slot); }
  const CapacityScratch L = capacity_scratch(R, E);
  if (ws_bytes < L.end) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  char* wsb = reinterpret_cast<char*>(ws);
  int32_t* chunk_counts = reinterpret_cast<int32_t*>(wsb + L.route.chunk_counts);
  int32_t* local_rank = reinterpret_cast<int32_t*>(wsb + L.route.local_rank);
  int32_t* rcounts = reinterpret_cast<int32_t*>(wsb + L.routed_counts);
  int32_t* roffsets = reinterpret_cast<int32_t*>(wsb + L.routed_offsets);
  int* status = reinterpret_cast<int*>(ws);
  const long long EC = (long long)E * C;
  int launches = 0;
  if (R > 0) {
    const int nchunks = (int)((R + kRouteChunk - 1) / kRouteChunk);
    (void)launch_pdl(route_count_kernel, nchunks, kRCThreads, sizeof(int32_t) * kRCWarps * E, s, topk_idx,
                     (int)R, E, chunk_counts, local_rank, status);
    (void)launch_pdl(route_scan_kernel, 1, 1024, 0, s, chunk_counts, nchunks, E, rcounts, roffsets);
    launches = 2;
  } else if (cudaMemsetAsync(rcounts, 0, sizeof(int32_t) * E, s) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  long long n = R > EC ? R : EC;
  if (n < E + 1) n = E + 1;
  (void)launch_pdl(route_place_capacity_kernel, (unsigned)((n + 255) / 256), 256, 0, s, topk_idx, (int)R, E, C,
                   chunk_counts, local_rank, rcounts, counts, offsets, routed, row_of_slot, slot_of_row);
  MOE_LAUNCH_CHECK(launches + 1);
  return MOE_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of moe_expert_offsets.
//
// For callers that cannot allocate device memory: code that runs while a
// stream is being captured into a CUDA graph (cudaMalloc/cudaFree are not
// allowed there and synchronise the device), engines that hand a plugin only
// the tensors they own from a pre-planned arena, and real-time loops that must
// never block on the allocator.  The route-map scratch (per-chunk expert
// histograms and in-chunk ranks) lives in this file-scope device array
// instead of a caller workspace.  Every GPU that loads the library keeps the
// array (2 MiB + 256 B) until the process exits.
#include <mutex>

namespace moe {
namespace {

constexpr int kNoAllocMaxSlots = 262144;                                // T * k
constexpr int kNoAllocChunkInts = (kNoAllocMaxSlots / kRouteChunk) * kMaxExperts;
constexpr int kNoAllocDummyInts = 64;                                   // status sink

static __device__ __align__(256) int32_t
    g_route_scratch[kNoAllocDummyInts + kNoAllocChunkInts + kNoAllocMaxSlots];

std::mutex g_noalloc_mu;
struct NoAllocSlot { unsigned long long ctx_id; int32_t* base; };
NoAllocSlot g_noalloc[64] = {};

// Unique id of the calling thread's current context (never reused within a
// process), through the driver entry points the runtime exposes; 0 if there
// is none yet or the driver lacks the query.
unsigned long long current_ctx_id() {
  using GetCurrent = int (*)(void**);
  using GetId = int (*)(void*, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static bool looked = false;
  if (!looked) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
    (void)cudaGetLastError();
    looked = true;
  }
  if (!get_current || !get_id) return 0;
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != 0 || ctx == nullptr || get_id(ctx, &id) != 0) return 0;
  return id;
}

// Device address of g_route_scratch in the current context (the host-side
// symbol itself is not a device address).  It is looked up on the first call
// on a device and again whenever that device's context has changed since
// (after a cudaDeviceReset the module, and with it the array, is loaded
// afresh at another address).
int32_t* noalloc_scratch(int dev) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocSlot& slot = g_noalloc[dev];
  const unsigned long long id = current_ctx_id();
  if (slot.base == nullptr || id == 0 || slot.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      slot.base = nullptr;
      return nullptr;
    }
    slot.base = static_cast<int32_t*>(p);
    slot.ctx_id = current_ctx_id();        // the lookup may have created the context
  }
  return slot.base;
}

}  // namespace
}  // namespace moe

extern "C" int moe_expert_offsets_noalloc(const int32_t* topk_idx, int T, int k, int E,
                                          int32_t* counts, int32_t* offsets,
                                          int32_t* row_of_slot, int32_t* slot_of_row,
                                          int32_t* status, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && k >= 1 && k <= kMaxTopK && E >= 1 && E <= kMaxExperts && k <= E);
  MOE_CHECK_ARG((long long)T * k <= 0x7fffffffLL);
  MOE_CHECK_PTR(counts); MOE_CHECK_PTR(offsets);
  if (status != nullptr && (reinterpret_cast<uintptr_t>(status) & 3u) != 0) return MOE_ERR_INVALID_ARG;
  const long long R = (long long)T * k;
  if (R > kNoAllocMaxSlots) return MOE_ERR_UNSUPPORTED;     // beyond the static scratch
  if (R > 0) { MOE_CHECK_PTR(topk_idx); MOE_CHECK_PTR(row_of_slot); MOE_CHECK_PTR(slot_of_row); }
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  int32_t* base = noalloc_scratch(dev);
  if (base == nullptr) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  if (R == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s) != cudaSuccess) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }
  // every scratch entry the kernels read is written earlier in the same call
  // (histograms for all chunks x E, ranks for every valid slot), so nothing
  // has to be cleared between calls
  int32_t* st = status ? status : base;                     // NULL: errors go to a sink
  int32_t* chunk_counts = base + kNoAllocDummyInts;
  int32_t* local_rank = chunk_counts + kNoAllocChunkInts;
  const int nchunks = (int)((R + kRouteChunk - 1) / kRouteChunk);
  size_t smem = sizeof(int32_t) * kRCWarps * E;
  (void)launch_pdl(route_count_kernel, nchunks, kRCThreads, smem, s, topk_idx, (int)R, E, chunk_counts,
                                                       local_rank, st);
  (void)launch_pdl(route_scan_kernel, 1, 1024, 0, s, chunk_counts, nchunks, E, counts, offsets);
  (void)launch_pdl(route_place_kernel, (int)((R + 255) / 256), 256, 0, s, topk_idx, (int)R, E, chunk_counts,
                                                             local_rank, offsets, row_of_slot,
                                                             slot_of_row);
  MOE_LAUNCH_CHECK(3);
  return MOE_OK;
}
