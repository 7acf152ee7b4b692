/* A C program against include/libmoe.h alone: no Python, no GPU.  It links
 * libmoe.so, calls the entry points that do host work only (the status
 * strings, the version, the workspace and atom size queries) and the argument
 * checks that return before any CUDA call, and prints "ok" when every answer
 * is the documented one. */
#include <stdio.h>
#include <string.h>

#include "libmoe.h"

static int failures = 0;
#define EXPECT(cond)                                                  \
  do {                                                                \
    if (!(cond)) {                                                    \
      fprintf(stderr, "failed: %s (line %d)\n", #cond, __LINE__);     \
      ++failures;                                                     \
    }                                                                 \
  } while (0)

int main(void) {
  void* fake = (void*)0x1000;                  /* aligned, never dereferenced */
  EXPECT(moe_version() == 100);
  EXPECT(strncmp(moe_status_string(MOE_OK), "MOE_OK", 6) == 0);
  EXPECT(strstr(moe_status_string(MOE_ERR_WORKSPACE), "workspace") != NULL);
  EXPECT(moe_status_string(12345) != NULL);
  /* the workspace grows with the problem and covers the route-map scratch */
  size_t small = moe_workspace_size(512, 8, 2, 256, 512);
  size_t big = moe_workspace_size(32768, 128, 4, 2048, 1024);
  EXPECT(small >= 256 && big > small);
  EXPECT(moe_workspace_size(-1, 8, 2, 256, 512) == 0);
  EXPECT(moe_mxfp8_weight_atom_bytes(2, 256, 384) == (size_t)2 * (4 * 2 + 2 * 3) * 2 * 512);
  EXPECT(moe_mxfp8_dx_weight_atom_bytes(2, 128, 96) == 0);
  /* argument checks return before any CUDA call */
  EXPECT(moe_router_topk(fake, 4, 8, 9, fake, fake, NULL) == MOE_ERR_INVALID_ARG);     /* k > 8 */
  EXPECT(moe_dispatch_rows(fake, 4, 12, 2, fake, fake, NULL) == MOE_ERR_INVALID_ARG);  /* d % 8 */
  EXPECT(moe_expert_offsets(fake, 4, 2, 8, fake, fake, fake, fake, NULL, 0, NULL) == MOE_ERR_WORKSPACE);
  EXPECT(moe_expert_offsets_capacity(fake, 64, 2, 8, 0, fake, fake, fake, fake, NULL, fake, 1 << 20,
                                     NULL) == MOE_ERR_INVALID_ARG);                    /* C = 0 */
  EXPECT(moe_expert_offsets_noalloc(fake, 262145, 1, 8, fake, fake, fake, fake, NULL, NULL) ==
         MOE_ERR_UNSUPPORTED);                                                         /* past the scratch */
  EXPECT(moe_grouped_swiglu_fwd((const moe_bf16_t*)fake, fake, 8, 4, 96, 128, fake, fake, fake, fake, fake,
                                fake, fake, fake, 1 << 20, NULL) == MOE_ERR_UNSUPPORTED);  /* d % 64 */
  EXPECT(moe_get_status(NULL, NULL, NULL) == MOE_ERR_WORKSPACE);
  /* T = 0 is a no-op and launches nothing */
  uint64_t before = moe_launch_count();
  EXPECT(moe_combine(NULL, NULL, NULL, 0, 2, 256, NULL, NULL) == MOE_OK);
  EXPECT(moe_launch_count() == before);
  if (failures == 0) printf("ok\n");
  return failures == 0 ? 0 : 1;
}
