/* A plain C99 consumer of include/ssd.h: prints, as one JSON object, the
 * layout of the ABI's structs, the workspace sizes of two problems and the
 * status codes of calls that validation rejects before any CUDA call (so it
 * runs without a GPU).  Built and run by tests/test_c_abi.py. */
#include <stddef.h>
#include <stdio.h>

#include "ssd.h"

int main(void) {
  ssd_problem p = {2, 300, 8, 64, 128, 2, 128, SSD_BF16, 0};
  ssd_norm_problem np = {300, 4096, 512, 1e-5f, SSD_BF16, SSD_NORM_HAS_Z};
  char buf[64];
  void* fake = (void*)(buf + (16 - ((size_t)buf & 15)) % 16); /* aligned, never dereferenced */
  float* ffake = (float*)fake;
  ssd_problem bad = p;
  bad.ngroups = 3;
  printf("{\"sizeof_problem\": %zu, \"off_chunk\": %zu, \"off_dtype\": %zu, \"off_flags\": %zu,",
         sizeof(ssd_problem), offsetof(ssd_problem, chunk_size), offsetof(ssd_problem, dtype),
         offsetof(ssd_problem, flags));
  printf(" \"sizeof_norm\": %zu, \"off_eps\": %zu, \"off_ndtype\": %zu, \"off_nflags\": %zu,",
         sizeof(ssd_norm_problem), offsetof(ssd_norm_problem, eps),
         offsetof(ssd_norm_problem, dtype), offsetof(ssd_norm_problem, flags));
  printf(" \"fwd_ws\": %zu, \"bwd_ws\": %zu, \"bad_ws\": %zu, \"norm_ws\": %zu,",
         ssd_fwd_workspace_bytes(&p), ssd_bwd_workspace_bytes(&p), ssd_fwd_workspace_bytes(&bad),
         ssd_gated_rmsnorm_bwd_workspace_bytes(&np));
  printf(" \"fwd_null_x\": %d,",
         ssd_fwd(&p, NULL, fake, ffake, ffake, fake, fake, ffake, NULL, NULL, fake, ffake, fake,
                 (size_t)1 << 40, NULL));
  printf(" \"fwd_small_ws\": %d,",
         ssd_fwd(&p, fake, fake, ffake, ffake, fake, fake, ffake, NULL, NULL, fake, ffake, fake, 16,
                 NULL));
  printf(" \"norm_no_z\": %d,",
         ssd_gated_rmsnorm_fwd(&np, fake, NULL, ffake, fake, NULL, NULL));
  printf(" \"status_ok\": \"%s\", \"version\": \"%s\"}\n", ssd_status_string(SSD_OK),
         ssd_version());
  return 0;
}
