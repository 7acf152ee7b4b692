// Shared host/device helpers of libmoe: status handling, launch accounting,
// workspace layout and small device utilities.  sm_103a only.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/libmoe.h"

#include <utility>

namespace moe {

// ---------------------------------------------------------------- host side

// Counts every kernel this library enqueues (see moe_launch_count).
void note_launches(int n);

// Number of SMs of the current device (cached per device).
int sm_count();

// Current device ordinal.
int current_device();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define MOE_CHECK_ARG(cond) do { if (!(cond)) return MOE_ERR_INVALID_ARG; } while (0)
#define MOE_CHECK_PTR(p) do { if ((p) == nullptr || !::moe::aligned16(p)) return MOE_ERR_INVALID_ARG; } while (0)
#define MOE_LAUNCH_CHECK(n) do { ::moe::note_launches(n); \
    if (cudaPeekAtLastError() != cudaSuccess) { (void)cudaGetLastError(); return MOE_ERR_CUDA; } } while (0)

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 8;

// Workspace layout (bytes from the start of ws):
//   [0, 256)   status word (int32) + padding
//   [256, ..)  scratch shared by the calls that need it; each call uses it
//              only while its own kernels run, so the regions may overlap:
//              moe_expert_offsets: per-chunk histograms [chunks][E] int32,
//                                  then in-chunk stable ranks [R] int32;
//              moe_router_logits_bwd: dW_r split-K partials [splits][d][E] f32;
//              moe_grouped_swiglu_bwd(_wgrad): per-expert TMA descriptors
//                                  [E][5] x 128 B (needs a 128-byte aligned ws),
//                                  the tile plan (kWgradPlanHead int32 then
//                                  the [E] order of the experts with rows and
//                                  the [E] list of those without), then up to
//                                  kWgradParts fp32 256 x 256 partial tiles of
//                                  the K-split last round.
constexpr size_t kStatusBytes = 256;
constexpr int kRouteChunk = 1024;     // slots per route-map block
constexpr int kRouterSplits = 16;     // deterministic split-K for dW_r

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct RouteScratch { size_t chunk_counts, local_rank, end; };

inline RouteScratch route_scratch(long long R, int E) {
  long long chunks = (R + kRouteChunk - 1) / kRouteChunk;
  RouteScratch L;
  L.chunk_counts = kStatusBytes;
  L.local_rank = round_up(L.chunk_counts + (size_t)chunks * E * 4, 256);
  L.end = round_up(L.local_rank + (size_t)R * 4, 256);
  return L;
}

// moe_expert_offsets_capacity: the route-map scratch, then the routed
// (pre-capacity) counts and their offsets.
struct CapacityScratch { RouteScratch route; size_t routed_counts, routed_offsets, end; };

inline CapacityScratch capacity_scratch(long long R, int E) {
  CapacityScratch c;
  c.route = route_scratch(R, E);
  c.routed_counts = c.route.end;
  c.routed_offsets = round_up(c.routed_counts + (size_t)E * 4, 256);
  c.end = round_up(c.routed_offsets + (size_t)(E + 1) * 4, 256);
  return c;
}

// moe_grouped_swiglu_fwd_mxfp8: the E8M0 scale atoms of Xq (K = d), then of
// Aq (K = h): (ceil(R / 128) + E) 128-row blocks x K / 128 atoms of 512 bytes
// each (layout in mx_common.cuh); moe_grouped_swiglu_bwd_dx_mxfp8 puts those
// of [dh1 | dh3] (K = 2h) in the first region.
inline size_t mx_act_atom_bytes(long long R, int E, int K) {
  return (size_t)((R + 127) / 128 + E) * (size_t)(K / 128) * 512;
}
inline size_t mx_scratch_x(long long R, int E, int d, int h) { (void)R; (void)E; (void)d; (void)h; return kStatusBytes; }
inline size_t mx_scratch_a(long long R, int E, int d, int h) {
  // (the first region also holds the atoms of the MXFP8 dgrad's dh1 | dh3, K = 2h)
  const int K = d > 2 * h ? d : 2 * h;
  return round_up(mx_scratch_x(R, E, d, h) + mx_act_atom_bytes(R, E, K), 256);
}
inline size_t mx_scratch_end(long long R, int E, int d, int h) {
  return round_up(mx_scratch_a(R, E, d, h) + mx_act_atom_bytes(R, E, h), 256);
}

inline size_t router_scratch_end(int E, int d) {
  return round_up(kStatusBytes + (size_t)kRouterSplits * d * E * 4, 256);
}

constexpr int kWgradMaps = 5;          // xp, a, dh1, dh3, dyp
constexpr int kWgradParts = 80;        // fp32 256 x 256 partial tiles (20 MB)
inline size_t wgrad_maps_end(int E) { return kStatusBytes + (size_t)E * kWgradMaps * 128; }
// the wgrad tile plan, written on the device from the offsets: head words
// (non-empty experts, empty experts, whole units, K-split chunks, units,
// zero tiles), then the order of the non-empty experts and the empty ones
constexpr int kWgradPlanHead = 8;
inline size_t wgrad_plan_offset(int E) { return round_up(wgrad_maps_end(E), 256); }
inline size_t wgrad_plan_end(int E) { return wgrad_plan_offset(E) + (size_t)(kWgradPlanHead + 2 * E) * 4; }
inline size_t wgrad_parts_offset(int E) { return round_up(wgrad_plan_end(E), 256); }
inline size_t wgrad_parts_end(int E) {
  return wgrad_parts_offset(E) + (size_t)kWgradParts * 256 * 256 * 4;
}

inline size_t workspace_bytes(long long T, int E, int k, int d) {
  size_t a = capacity_scratch(T * (long long)k, E).end;
  size_t b = router_scratch_end(E, d);
  size_t c = wgrad_parts_end(E);
  a = a > b ? a : b;
  return a > c ? a : c;
}

// Programmatic dependent launch: every kernel of this library is launched
// with programmatic stream serialisation, lets the next launch on its stream
// be scheduled at once (griddepcontrol.launch_dependents) and waits for the
// kernel before it to complete and flush its memory (griddepcontrol.wait)
// before touching global memory, so stream order still holds while the next
// grid's launch overlaps the tail of the current one.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// -------------------------------------------------------------- device side

__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void set_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Two fp32 -> packed bf16x2 (round to nearest even), low half = a.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// A row index read from a route map is used only inside [0, R): slots whose
// expert id was out of range carry row -1 (and a caller-built map may hold
// anything), so the row kernels skip such rows instead of writing through them.
__device__ __forceinline__ bool row_ok(int row, int R) { return (unsigned)row < (unsigned)R; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace moe
