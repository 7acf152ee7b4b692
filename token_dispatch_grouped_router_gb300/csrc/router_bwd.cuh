// Workspace layout of moe_router_logits_bwd_topk (bytes from the start of ws,
// after the weight-gradient GEMM's part: its descriptors, tile plan and fp32
// partial tiles, so the two may run at once on two streams sharing one
// workspace): W_r transposed [E][d] fp32, the row-chunk
// table of the dW_r reduction (one entry per chunk of at most kRouterChunk
// rows of an expert's segment, plus per-expert first chunk and chunk count),
// the chunks' fp32 partial sums [chunks][d] and partial bias sums [chunks].
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kRouterChunk = 256;      // routed rows per dW_r partial

struct RouterTopkScratch { size_t wt, units, estart, ecount, total, part, pbias, end; long long max_units; };

inline RouterTopkScratch router_topk_scratch(long long R, int E, int d) {
  RouterTopkScratch s;
  s.max_units = (R + kRouterChunk - 1) / kRouterChunk + E;
  s.wt = round_up(wgrad_parts_end(E), 256);
  s.units = round_up(s.wt + (size_t)E * d * 4, 256);
  s.estart = round_up(s.units + (size_t)s.max_units * 16, 256);
  s.ecount = round_up(s.estart + (size_t)E * 4, 256);
  s.total = round_up(s.ecount + (size_t)E * 4, 256);
  s.part = round_up(s.total + 4, 256);
  s.pbias = round_up(s.part + (size_t)s.max_units * d * 4, 256);
  s.end = round_up(s.pbias + (size_t)s.max_units * 4, 256);
  return s;
}

}  // namespace moe
