/*
 * libmoe — a GB300-native (sm_103a) single-GPU MoE expert layer behind a C ABI.
 *
 * The layer: router top-k -> device-resident route map (counts, offsets,
 * permutation) -> rowwise dispatch into expert-contiguous rows -> unpadded
 * grouped SwiGLU GEMM on tcgen05 tensor cores -> routing-weighted combine,
 * and the backward of every step.
 *
 * Sources.  "OLMo-core 3：MoE 训练栈让专家池越大、吞吐不再越慢" (bloombook.cn
 * tutorial), sections "rowwise EP：用 NVSHMEM 一端直写" (rows written straight
 * into the destination expert's input buffer by a route-table lookup; combine
 * brings them back) and "另外两处税：主机同步与 padding" (routing counts, expert
 * row counts and the per-expert permutation stay on the device, removing two
 * host syncs; one grouped-GEMM launch over all experts with their exact row
 * counts, no padding to a common capacity).  The Olmo-core MoE report's
 * speed-read summary (taotianhua.com), paragraph "GPU-resident metadata
 * removes recurring host waits", says the same of the report's Sections 8-9.
 * The pages define neither the router function nor the expert network; the
 * definitions below (softmax-then-top-k with renormalised gates, ties to the
 * lower expert id; SwiGLU experts W2(silu(x W1) * (x W3))) are the benchmark
 * specification's reading.
 *
 * Conventions shared by every entry point
 *  - Pointers are DEVICE pointers owned by the caller, except where a
 *    parameter says "host".  The library allocates no memory, never
 *    synchronises the host (moe_get_status excepted, on request) and enqueues
 *    all work on `stream` (NULL = the legacy default stream).
 *  - bf16 tensors are passed as moe_bf16_t* (uint16_t bit patterns), row-major.
 *  - Every device pointer must be 16-byte aligned.
 *  - Host-side argument errors return a negative moe_status_t and launch
 *    nothing.  A launch failure returns MOE_ERR_CUDA.  Data errors found on the
 *    device (an expert id outside [0, E), a wait that timed out) are written
 *    to the status word inside the workspace and leave the outputs
 *    unspecified; read it with moe_get_status.
 *  - T = 0 is a valid no-op (weight gradients are then written as zeros).
 *    Experts that receive no rows are valid.
 *  - Sizes: 1 <= k <= 8, k <= E <= 1024.  The grouped GEMMs need d and h to be
 *    multiples of 64 (MOE_ERR_UNSUPPORTED otherwise); the row kernels need d to
 *    be a multiple of 8.  T * k must fit in int32.
 *  - Calls are stateless apart from a per-device cache of the SM count and of
 *    kernel attributes; they are safe to call from several host threads on
 *    different streams with distinct workspaces.  One pairing may share a
 *    workspace: moe_grouped_swiglu_bwd_wgrad and moe_router_logits_bwd_topk
 *    use disjoint parts of it (the router backward's scratch lies past the
 *    weight-gradient GEMM's descriptors, plan and partial tiles), so they, and
 *    calls that take no workspace (moe_combine, moe_router_topk_bwd), may run
 *    at the same time on two streams; the status word is set atomically.
 */
#ifndef LIBMOE_H
#define LIBMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16_t;               /* bf16 bit pattern */
typedef struct CUstream_st* moe_stream_t;  /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,   /* null pointer, bad size, misaligned pointer */
  MOE_ERR_UNSUPPORTED = -2,   /* valid but outside what the kernels handle */
  MOE_ERR_WORKSPACE = -3,     /* workspace null or smaller than the query */
  MOE_ERR_CUDA = -4           /* a CUDA launch or runtime call failed */
} moe_status_t;

/* Device-side status codes written into the workspace status word. */
enum {
  MOE_DEV_OK = 0,
  MOE_DEV_BAD_EXPERT_ID = 1,  /* an expert id outside [0, E) was routed */
  MOE_DEV_WAIT_TIMEOUT = 2    /* a pipeline wait in a GEMM gave up */
};

/* Human-readable name of a moe_status_t. Never NULL. */
const char* moe_status_string(int status);

/* ABI version of this header (major * 100 + minor). */
int moe_version(void);

/* Number of kernels this library has enqueued since it was loaded (all
 * threads, all devices).  Host-side counter, for launch accounting. */
uint64_t moe_launch_count(void);

/* Bytes of workspace needed by moe_expert_offsets, moe_grouped_swiglu_fwd/bwd
 * and moe_router_logits_bwd for these sizes.  The first 256 bytes hold the
 * device status word; the rest is route-map and reduction scratch and the
 * weight-gradient phase's per-expert TMA descriptors.  The
 * workspace must be zeroed once (or reset with moe_reset_status) before its
 * status word is meaningful. */
size_t moe_workspace_size(int T, int E, int k, int d, int h);

/* Zero the device status word (async on `stream`). */
int moe_reset_status(void* ws, moe_stream_t stream);

/* Copy the device status word to *host_status (host pointer).  This call
 * synchronises `stream`; it is the only one that does. */
int moe_get_status(const void* ws, int32_t* host_status, moe_stream_t stream);

/* ---------------------------------------------------------------- router */

/* Router logits z[T,E] (fp32) = x[T,d] (bf16) @ W_r[d,E] (fp32) + b[E]
 * (b may be NULL).  fp32 accumulation. */
int moe_router_logits(const moe_bf16_t* x, const float* W_r, const float* b,
                      int T, int d, int E, float* logits, moe_stream_t stream);

/* The same logits on the tcgen05 tensor cores at fp32 accuracy.  W_r is split
 * exactly into three bf16 parts (W_r = W0 + W1 + W2, each the bf16 rounding of
 * what the earlier parts leave), written to the workspace scratch; the MMAs
 * form x W0 + x W1 + x W2 with exact bf16 products and fp32 accumulation.  The
 * router stays in high precision, as the page's DeepSeek-V3 paragraph asks
 * (OLMo-core 3 tutorial, section "一个低精度格式，同时压三个地方").
 * d % 8 == 0 (MOE_ERR_UNSUPPORTED otherwise); ws 16-byte aligned with at
 * least moe_workspace_size(...) bytes (the split needs 256 + 6 E
 * ceil(d/64)*64 bytes); a timed-out pipeline wait sets the status word. */
int moe_router_logits_tc(const moe_bf16_t* x, const float* W_r, const float* b,
                         int T, int d, int E, float* logits, void* ws, size_t ws_bytes,
                         moe_stream_t stream);

/* Top-k of each row of logits[T,E] (fp32): topk_idx[T,k] (int32) lists the k
 * largest logits in the total order (value descending, expert id ascending;
 * -0.0 == +0.0), and topk_gate[T,k] (fp32) = softmax over the k selected
 * logits (the full softmax renormalised over the selection).  NaN logits are
 * out of contract.  Requires k <= E <= 1024. */
int moe_router_topk(const float* logits, int T, int E, int k,
                    int32_t* topk_idx, float* topk_gate, moe_stream_t stream);

/* Gates for externally chosen experts: topk_gate[T,k] = softmax over each
 * row of sel_logits[T,k] (synthetic uniform routing). */
int moe_router_gates(const float* sel_logits, int T, int k, float* topk_gate,
                     moe_stream_t stream);

/* Backward of the renormalised top-k softmax: d_logits[T,E] (fp32, fully
 * written) is g_j * (dg_j - sum_l g_l dg_l) at column topk_idx[t,j] and zero
 * in every other column. */
int moe_router_topk_bwd(const float* topk_gate, const float* d_gate,
                        const int32_t* topk_idx, int T, int E, int k,
                        float* d_logits, moe_stream_t stream);

/* Backward of the router logits GEMM: dx[T,d] (bf16, read-modify-write)
 * += d_logits @ W_r^T; dW_r[d,E] = x^T @ d_logits; db[E] = column sums of
 * d_logits (db may be NULL).  Deterministic (fixed reduction order; uses the
 * workspace for split reductions). */
int moe_router_logits_bwd(const moe_bf16_t* x, const float* W_r,
                          const float* d_logits, int T, int d, int E,
                          moe_bf16_t* dx, float* dW_r, float* db,
                          void* ws, size_t ws_bytes, moe_stream_t stream);

/* The same backward when only the top-k logits carry gradient, as
 * moe_router_topk_bwd leaves d_logits (the gates are a softmax over the
 * selected logits, so every other entry is 0; this call reads only the
 * selected ones):
 *   dx[t] += sum_j d_logits[t, idx_tj] * W_r[:, idx_tj]   (bf16, one rounding)
 *   dW_r[:, e] = sum over the rows routed to e of d_logits[t, e] * x[t]
 *   db[e] = sum over the same rows of d_logits[t, e]         (db may be NULL)
 * The sums over rows follow the route map (offsets[E+1] and slot_of_row[T*k]
 * from moe_expert_offsets on topk_idx) in token order, in chunks of 256 rows
 * added in chunk order: deterministic.  Results equal moe_router_logits_bwd's
 * up to fp32 summation order.  d % 8 == 0 (MOE_ERR_UNSUPPORTED otherwise); ws
 * needs moe_workspace_size(T, E, k, d, h) bytes. */
int moe_router_logits_bwd_topk(const moe_bf16_t* x, const float* W_r, const float* d_logits,
                               const int32_t* topk_idx, const int32_t* offsets,
                               const int32_t* slot_of_row, int T, int d, int E, int k,
                               moe_bf16_t* dx, float* dW_r, float* db, void* ws, size_t ws_bytes,
                               moe_stream_t stream);

/* ------------------------------------------------------------- route map */

/* Device-resident route map from topk_idx[T,k] (flattened slot s = t*k + j):
 *   counts[E]       rows routed to each expert
 *   offsets[E+1]    exclusive prefix sum of counts (offsets[E] = T*k)
 *   row_of_slot[R]  row of the expert-sorted buffer that holds slot s:
 *                   offsets[e] + number of slots s' < s routed to e (stable)
 *   slot_of_row[R]  inverse permutation
 * No host synchronisation.  An expert id outside [0, E) sets
 * MOE_DEV_BAD_EXPERT_ID in the workspace status word; that slot gets
 * row_of_slot = -1 and takes no row (offsets[E] is then below T*k). */
int moe_expert_offsets(const int32_t* topk_idx, int T, int k, int E,
                       int32_t* counts, int32_t* offsets,
                       int32_t* row_of_slot, int32_t* slot_of_row,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* Allocation-free moe_expert_offsets (no counterpart on the pages).
 *
 * For callers that cannot allocate device memory: code running inside a CUDA
 * stream capture (cudaMalloc/cudaFree are illegal there and synchronise the
 * device), engines that give a plugin only the tensors from their own
 * pre-planned arena, and real-time loops that must not block on an allocator.
 * Same outputs as moe_expert_offsets, but the route-map scratch lives in a
 * static device array inside libmoe (2 MiB + 256 B, held on every GPU that
 * loads the library until the process exits) instead of a workspace.
 *  - Limit: T * k <= 262144; larger sizes return MOE_ERR_UNSUPPORTED and
 *    launch nothing.
 *  - status: optional device int32 (4-byte aligned) that receives
 *    MOE_DEV_BAD_EXPERT_ID like the workspace status word; NULL discards it.
 *    Clear it yourself before the call if you read it.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *    The address is looked up again when the device's context has changed
 *    since (after cudaDeviceReset the array lives at a new address), so the
 *    first call after a reset must also come before any capture.
 *  - All calls share the one array and no call clears it (every entry a call
 *    reads is written earlier in that call): calls that can overlap on the
 *    GPU (different streams, or concurrent host threads) race and must be
 *    serialised by the caller.
 *  - No cudaMalloc/cudaFree or allocating library call is made. */
int moe_expert_offsets_noalloc(const int32_t* topk_idx, int T, int k, int E,
                               int32_t* counts, int32_t* offsets,
                               int32_t* row_of_slot, int32_t* slot_of_row,
                               int32_t* status, moe_stream_t stream);

/* ------------------------------------------------------- dispatch/combine */

/* Rowwise dispatch: xp[row_of_slot[t*k+j], :] = x[t, :] for all t, j.
 * x[T,d] bf16 -> xp[T*k, d] bf16 (expert-contiguous).  Exact copy.
 * Here and in every call below that reads row_of_slot, an entry outside
 * [0, T*k) (the -1 of a slot with a bad expert id) is skipped: no row is
 * written through it, a combine adds nothing for it, and its dgate is 0. */
int moe_dispatch_rows(const moe_bf16_t* x, int T, int d, int k,
                      const int32_t* row_of_slot, moe_bf16_t* xp,
                      moe_stream_t stream);

/* Combine: out[t,:] = sum_j gate[t,j] * yp[row_of_slot[t*k+j], :] with an
 * fp32 sum in slot order, rounded once to bf16.  gate == NULL means all ones
 * (the unpermute-sum of the backward: dX = sum_j dXp[row(t,j)]). */
int moe_combine(const moe_bf16_t* yp, const int32_t* row_of_slot,
                const float* gate, int T, int k, int d, moe_bf16_t* out,
                moe_stream_t stream);

/* Combine backward: dyp[row(t,j), :] = bf16(gate[t,j] * dout[t, :]) and
 * dgate[t,j] = <dout[t,:], yp[row(t,j),:]> (fp32 accumulation). */
int moe_combine_bwd(const moe_bf16_t* dout, const moe_bf16_t* yp,
                    const int32_t* row_of_slot, const float* gate, int T,
                    int k, int d, moe_bf16_t* dyp, float* dgate,
                    moe_stream_t stream);

/* ------------------------------------------------------ grouped SwiGLU GEMM */

/* Forward of every expert's SwiGLU FFN on its rows of xp (expert e owns rows
 * [offsets[e], offsets[e+1]) of the R = T*k rows; offsets is device memory):
 *   h1 = xp_e @ W1[e],  h3 = xp_e @ W3[e],  a = silu(h1) * h3,  yp_e = a @ W2[e]
 * xp[R,d], W1/W3[E,d,h], W2[E,h,d], h1/h3/a[R,h], yp[R,d]: bf16; fp32
 * accumulation in tensor memory; a is computed from the fp32 accumulators.
 * Two persistent tcgen05 kernels whose tile scheduler reads offsets on the
 * device; no padding and no host synchronisation. */
int moe_grouped_swiglu_fwd(const moe_bf16_t* xp, const int32_t* offsets,
                           int R, int E, int d, int h,
                           const moe_bf16_t* W1, const moe_bf16_t* W3,
                           const moe_bf16_t* W2,
                           moe_bf16_t* h1, moe_bf16_t* h3, moe_bf16_t* a,
                           moe_bf16_t* yp, void* ws, size_t ws_bytes,
                           moe_stream_t stream);

/* Backward of moe_grouped_swiglu_fwd for the upstream gradient dyp[R,d]:
 *   dA  = dyp_e @ W2[e]^T
 *   dh1 = dA * h3 * silu'(h1)   (silu'(u) = s(u) (1 + u (1 - s(u))), s = sigmoid)
 *   dh3 = dA * silu(h1)
 *   dxp = dh1 @ W1[e]^T + dh3 @ W3[e]^T
 *   dW2[e] = a_e^T @ dyp_e,  dW1[e] = xp_e^T @ dh1_e,  dW3[e] = xp_e^T @ dh3_e
 * The weight gradients reduce over each expert's own row count (zero rows
 * give exactly zero).  dh1/dh3[R,h] are caller-provided intermediates (also
 * outputs).  dW1/dW3[E,d,h], dW2[E,h,d] bf16 from fp32 accumulators, no
 * atomics, deterministic.  The weight-gradient phase keeps five TMA
 * descriptors per expert in ws (bytes [256, 256 + 640 E)) and, after them, a
 * tile plan ((8 + 2E) int32: the experts with rows ordered by depth, the
 * empty ones, the unit counts), both written on the device from offsets; when
 * the last round of its 256 x 256 tiles would leave most SMs idle, it splits
 * those tiles along the rows into chunks whose fp32 partial sums (up to 80
 * tiles of 256 KB after the plan) are added in a fixed order.  For R > 0 ws
 * must be 128-byte aligned (MOE_ERR_INVALID_ARG) and hold at least the
 * descriptors and the plan (else MOE_ERR_WORKSPACE); moe_workspace_size(...)
 * also covers the partials. */
int moe_grouped_swiglu_bwd(const moe_bf16_t* xp, const int32_t* offsets,
                           int R, int E, int d, int h,
                           const moe_bf16_t* W1, const moe_bf16_t* W3,
                           const moe_bf16_t* W2,
                           const moe_bf16_t* h1, const moe_bf16_t* h3,
                           const moe_bf16_t* a, const moe_bf16_t* dyp,
                           moe_bf16_t* dh1, moe_bf16_t* dh3, moe_bf16_t* dxp,
                           moe_bf16_t* dW1, moe_bf16_t* dW3, moe_bf16_t* dW2,
                           void* ws, size_t ws_bytes, moe_stream_t stream);

/* The phases of the two calls above, one tcgen05 kernel each, for callers
 * that schedule or time them separately.  Same argument meanings; each phase
 * needs its inputs from the previous one in stream order:
 *   fwd_up    h1, h3, a  from xp          (a = silu(h1) * h3)
 *   fwd_down  yp         from a
 *   bwd_dact  dh1, dh3   from dyp, h1, h3 (dA = dyp W2^T, SwiGLU backward)
 *   bwd_dx    dxp        from dh1, dh3
 *   bwd_wgrad dW1, dW3, dW2 from xp, a, dh1, dh3, dyp (R = 0 writes zeros) */
int moe_grouped_swiglu_fwd_up(const moe_bf16_t* xp, const int32_t* offsets, int R,
                              int E, int d, int h, const moe_bf16_t* W1,
                              const moe_bf16_t* W3, moe_bf16_t* h1, moe_bf16_t* h3,
                              moe_bf16_t* a, void* ws, size_t ws_bytes,
                              moe_stream_t stream);
int moe_grouped_swiglu_fwd_down(const moe_bf16_t* a, const int32_t* offsets, int R,
                                int E, int d, int h, const moe_bf16_t* W2,
                                moe_bf16_t* yp, void* ws, size_t ws_bytes,
                                moe_stream_t stream);
int moe_grouped_swiglu_bwd_dact(const int32_t* offsets, int R, int E, int d, int h,
                                const moe_bf16_t* W2, const moe_bf16_t* h1,
                                const moe_bf16_t* h3, const moe_bf16_t* dyp,
                                moe_bf16_t* dh1, moe_bf16_t* dh3, void* ws,
                                size_t ws_bytes, moe_stream_t stream);
int moe_grouped_swiglu_bwd_dx(const int32_t* offsets, int R, int E, int d, int h,
                              const moe_bf16_t* W1, const moe_bf16_t* W3,
                              const moe_bf16_t* dh1, const moe_bf16_t* dh3,
                              moe_bf16_t* dxp, void* ws, size_t ws_bytes,
                              moe_stream_t stream);
int moe_grouped_swiglu_bwd_wgrad(const moe_bf16_t* xp, const int32_t* offsets, int R,
                                 int E, int d, int h, const moe_bf16_t* a,
                                 const moe_bf16_t* dyp, const moe_bf16_t* dh1,
                                 const moe_bf16_t* dh3, moe_bf16_t* dW1,
                                 moe_bf16_t* dW3, moe_bf16_t* dW2, void* ws,
                                 size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------ capacity-padded layer */
/* The alternative the unpadded layer replaces, built on the same kernels so
 * the two can be timed side by side ("OLMo-core 3：MoE 训练栈让专家池越大、吞吐
 * 不再越慢", section "另外两处税：主机同步与 padding": without the device route
 * map every expert batch is padded to one common capacity; the page gives no
 * capacity formula, so C is the caller's).  Every expert owns exactly C rows
 * of the expert-sorted buffers, rows [e*C, (e+1)*C): its first C routed slots
 * in token order (slot order) fill the front of that block, the remaining
 * rows are zero, and slots beyond the first C are dropped (they contribute
 * nothing to the output and the other gates are not renormalised).  The
 * grouped SwiGLU calls run on these buffers unchanged with R = E*C and
 * offsets[e] = e*C, so they multiply E*C rows however the tokens were
 * routed. */

/* Capacity-padded route map from topk_idx[T,k]:
 *   counts[E]        rows kept per expert, min(routed, C)
 *   offsets[E+1]     e*C (offsets[E] = E*C)
 *   row_of_slot[T*k] e*C + rank of the slot among expert e's slots in slot
 *                    order if that rank is below C, else -1 (dropped)
 *   slot_of_row[E*C] the slot a row holds, -1 for a zero row
 *   routed[E]        (optional, may be NULL) rows routed to e before the cut
 * C >= 1 and E*C must fit in int32; ws as for moe_expert_offsets (status
 * word, route-map scratch and 2 E int32).  A bad expert id sets
 * MOE_DEV_BAD_EXPERT_ID and its slot is dropped. */
int moe_expert_offsets_capacity(const int32_t* topk_idx, int T, int k, int E, int C,
                                int32_t* counts, int32_t* offsets,
                                int32_t* row_of_slot, int32_t* slot_of_row,
                                int32_t* routed, void* ws, size_t ws_bytes,
                                moe_stream_t stream);

/* Padded dispatch: xp[E*C, d] gets x[t] in row row_of_slot[t*k+j] for every
 * kept slot and zeros in every row e*C + j with j >= counts[e] (counts from
 * moe_expert_offsets_capacity).  Two launches (copy, zero rows). */
int moe_dispatch_rows_capacity(const moe_bf16_t* x, int T, int d, int k,
                               const int32_t* row_of_slot, const int32_t* counts,
                               int E, int C, moe_bf16_t* xp, moe_stream_t stream);

/* moe_combine over a padded yp[E*C, d]: out[t] = sum over the kept slots of
 * gate[t,j] * yp[row(t,j)] (gate == NULL: unit gates, the unpermute-sum). */
int moe_combine_capacity(const moe_bf16_t* yp, int E, int C, const int32_t* row_of_slot,
                         const float* gate, int T, int k, int d, moe_bf16_t* out,
                         moe_stream_t stream);

/* moe_combine_bwd over padded buffers: dyp[row(t,j)] = bf16(gate[t,j] dout[t])
 * for the kept slots, zeros in the zero rows (as moe_dispatch_rows_capacity),
 * dgate[t,j] = <dout[t], yp[row(t,j)]> for a kept slot and 0 for a dropped
 * one. */
int moe_combine_bwd_capacity(const moe_bf16_t* dout, const moe_bf16_t* yp, int E, int C,
                             const int32_t* row_of_slot, const int32_t* counts,
                             const float* gate, int T, int k, int d, moe_bf16_t* dyp,
                             float* dgate, moe_stream_t stream);

/* ----------------------------------------------------------------- MXFP8 */
/* MXFP8 = E4M3 codes (uint8) with one E8M0 scale byte (2^(byte-127)) per 32
 * consecutive elements along a GEMM's reduction dimension ("OLMo-core 3：MoE
 * 训练栈让专家池越大、吞吐不再越慢", section "一个低精度格式，同时压三个地方").  Scale
 * rule: e = smallest integer with max|block| <= 448 * 2^e (clamped to
 * [-127, 127], -127 for an all-zero block); codes = RNE_E4M3(v * 2^-e).  The
 * page's list of scale steps is garbled; this is the reading that its
 * surviving sentence (divide by 448, power of two, block max just fits)
 * supports.  Scale tables are row-major bytes, 4-byte aligned. */

/* src[rows][K] (bf16) -> q[rows][K] codes and scale[rows][K/32].  K % 32 == 0. */
int moe_mxfp8_quantize_rows(const moe_bf16_t* src, int rows, int K, uint8_t* q,
                            uint8_t* scale, moe_stream_t stream);

/* Expert weights W[E][K][N] (bf16, K = reduction dim) -> K-major codes
 * wq[E][N][K] and scales ws[E][N][K/32] (the transposed layout the
 * block-scaled GEMM reads).  K % 32 == 0, N % 128 == 0.  Call once per
 * optimizer step for W1, W3 (K = d, N = h) and W2 (K = h, N = d). */
int moe_mxfp8_quantize_weights(const moe_bf16_t* W, int E, int K, int N,
                               uint8_t* wq, uint8_t* ws, moe_stream_t stream);

/* The same from fp32 master weights W[E][K][N] (one rounding, fp32 -> E4M3).
 * The page keeps the FP32 master weights authoritative and re-makes the
 * low-precision copies after each optimizer step (same section).  Same layout,
 * limits and errors as moe_mxfp8_quantize_weights. */
int moe_mxfp8_quantize_weights_f32(const float* W, int E, int K, int N,
                                   uint8_t* wq, uint8_t* ws, moe_stream_t stream);

/* q[rows][K] codes with scale[rows][K/32] -> out[rows][K] bf16, each value
 * code * 2^(scale - 127) rounded to bf16 (RNE; exact for every value at or
 * above 2^-126).  For activations kept in MXFP8 between the forward and the
 * backward (the page also quantises saved activations, same section): the
 * bf16 backward reads them back through this call.  K % 32 == 0; q and out
 * 16-byte aligned; scale bytes of 255 (E8M0 NaN) are out of contract. */
int moe_mxfp8_dequantize_rows(const uint8_t* q, const uint8_t* scale, int rows, int K,
                              moe_bf16_t* out, moe_stream_t stream);

/* Rowwise dispatch of quantised rows: each token row is quantised once along d
 * and written to its k expert rows: xq[R][d] codes, xs[R][d/32] scales; the
 * bf16 row also goes to xp[R][d] when xp != NULL (the backward stays bf16).
 * d % 32 == 0. */
int moe_dispatch_rows_mxfp8(const moe_bf16_t* x, int T, int d, int k,
                            const int32_t* row_of_slot, uint8_t* xq, uint8_t* xs,
                            moe_bf16_t* xp, moe_stream_t stream);

/* Bytes of the scale atoms moe_mxfp8_weight_scale_atoms writes for E experts
 * (0 unless d and h are multiples of 128). */
size_t moe_mxfp8_weight_atom_bytes(int E, int d, int h);

/* The weight scales in the order the block-scaled GEMM's tiles read them.
 * The tensor cores take E8M0 scales from tensor memory, filled from 512-byte
 * shared-memory atoms (32 rows of 16 bytes; byte 4j + q of row r is the scale
 * of output column 32j + r of a 128-column group for the q-th 32-element block
 * of a 128-deep k-block); the GEMM fetches whole atoms by TMA.  From the
 * row-major tables of moe_mxfp8_quantize_weights (w1s/w3s [E][h][d/32], w2s
 * [E][d][h/32]) this writes, per expert, column tile and k-block, two atoms:
 * the up-projection's tiles are 96 rows of W1 followed by the same 96 rows of
 * W3 (ceil(h/96) tiles, K = d), then the down-projection's 192 rows of W2
 * (ceil(d/192) tiles, K = h); columns past the matrix hold 0.  Call it with
 * the weight quantisation, once per optimizer step.  d, h multiples of 128;
 * scale tables 4-byte aligned, atoms 16-byte aligned with
 * moe_mxfp8_weight_atom_bytes(E, d, h) bytes.  Two launches. */
int moe_mxfp8_weight_scale_atoms(const uint8_t* w1s, const uint8_t* w3s, const uint8_t* w2s,
                                 int E, int d, int h, uint8_t* atoms, moe_stream_t stream);

/* Forward of the grouped SwiGLU FFN with MXFP8 GEMM operands and fp32
 * accumulation (block-scaled tcgen05 MMA): h1 = Xq_e W1q[e], h3 = Xq_e W3q[e],
 * a = silu(h1) * h3 (bf16 h1, h3, a for the bf16 backward), a quantised along
 * h into aq[R][h] / as[R][h/32], yp = Aq_e W2q[e] (bf16).  a may be NULL:
 * then only its quantised form is written (a caller that keeps the saved
 * activation in MXFP8 and dequantises it for the backward).  Weights come from
 * moe_mxfp8_quantize_weights (w1q/w3q [E][h][d], w2q [E][d][h]) and their
 * scales from moe_mxfp8_weight_scale_atoms (w_atoms); xs and as are row-major
 * [R][K/32] tables, which the call lays out as atoms in the workspace
 * ((ceil(R/128) + E) (d + h) * 4 bytes after the status word; every expert's
 * rows start a fresh 128-row block there).  With at least 512 rows per expert
 * on average the GEMMs run on 2-CTA clusters (256 x 192 tiles), otherwise on
 * single CTAs (128 x 192).  d and h must be multiples of 128 and E <= 768
 * (MOE_ERR_UNSUPPORTED otherwise: the kernels keep an E-sized tile table
 * beside their operand stages in shared memory); ws needs
 * moe_workspace_size(T, E, k, d, h) bytes (MOE_ERR_WORKSPACE). */
int moe_grouped_swiglu_fwd_mxfp8(const uint8_t* xq, const uint8_t* xs,
                                 const int32_t* offsets, int R, int E, int d, int h,
                                 const uint8_t* w1q, const uint8_t* w3q, const uint8_t* w2q,
                                 const uint8_t* w_atoms,
                                 moe_bf16_t* h1, moe_bf16_t* h3, moe_bf16_t* a,
                                 uint8_t* aq, uint8_t* as, moe_bf16_t* yp,
                                 void* ws, size_t ws_bytes, moe_stream_t stream);

/* MXFP8 dgrad of the expert rows (the Dgrad GEMM the same page quantises with
 * the forward ones):
 *   dxp_e = Q(dh1_e) Q(W1[e])^T + Q(dh3_e) Q(W3[e])^T      (fp32 accumulate, bf16 out)
 * The reduction runs over h, so every operand is quantised along h: dh1q/dh3q
 * [R][h] codes with row-major scales dh1s/dh3s [R][h/32] (moe_mxfp8_quantize_rows
 * of dh1 and dh3), and the weights' rows along h, a second set of weight
 * copies beside the forward's: w1q_h/w3q_h [E][d][h] with scales [E][d][h/32]
 * (moe_mxfp8_quantize_rows of W1 and W3 viewed as [E*d][h]), whose scales
 * moe_mxfp8_dx_weight_scale_atoms lays out as the GEMM's atoms (per expert,
 * 192-column tile of d and 128-deep k-block of K = 2h: W1's k-blocks, then
 * W3's; two atoms each, columns past d zero).  CTA pairs from 512 rows per
 * expert on average.  d, h multiples of 128, E <= 768; ws as for
 * moe_grouped_swiglu_fwd_mxfp8 (the call lays out the scales of dh1 | dh3 as
 * atoms there). */
size_t moe_mxfp8_dx_weight_atom_bytes(int E, int d, int h);
/* moe_grouped_swiglu_bwd_dact that also writes dh1 / dh3 quantised along h
 * for the MXFP8 dgrad: dh1q/dh3q [R][h] codes, dh1s/dh3s [R][h/32] scales,
 * from the epilogue's own bf16 dh1 / dh3 (the same bytes as
 * moe_mxfp8_quantize_rows of them; the epilogue holds one row's 32-column
 * block per thread, so no separate pass over dh1 / dh3 is made).  Codes
 * 16-byte aligned. */
int moe_grouped_swiglu_bwd_dact_mxfp8(const int32_t* offsets, int R, int E, int d, int h,
                                      const moe_bf16_t* W2, const moe_bf16_t* h1,
                                      const moe_bf16_t* h3, const moe_bf16_t* dyp,
                                      moe_bf16_t* dh1, moe_bf16_t* dh3, uint8_t* dh1q,
                                      uint8_t* dh1s, uint8_t* dh3q, uint8_t* dh3s, void* ws,
                                      size_t ws_bytes, moe_stream_t stream);
int moe_mxfp8_dx_weight_scale_atoms(const uint8_t* w1s_h, const uint8_t* w3s_h, int E, int d, int h,
                                    uint8_t* atoms, moe_stream_t stream);
int moe_grouped_swiglu_bwd_dx_mxfp8(const uint8_t* dh1q, const uint8_t* dh1s,
                                    const uint8_t* dh3q, const uint8_t* dh3s,
                                    const int32_t* offsets, int R, int E, int d, int h,
                                    const uint8_t* w1q_h, const uint8_t* w3q_h,
                                    const uint8_t* dx_atoms, moe_bf16_t* dxp,
                                    void* ws, size_t ws_bytes, moe_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif /* LIBMOE_H */
