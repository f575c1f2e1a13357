/* The C ABI used from plain C (no Python, no torch): include the header, link
 * libssscan.so, and exercise the calls that need no GPU — workspace queries,
 * chunk counts, status strings and argument validation, which returns before
 * any launch.  Exits 0 when every check holds, else prints the failing one. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "ssscan.h"

static int failures = 0;
#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
      ++failures;                                                \
    }                                                            \
  } while (0)

int main(void) {
  /* fake, aligned device addresses: validation rejects the call before any use */
  void* p = (void*)(uintptr_t)0x100000;
  const float* pf = (const float*)(uintptr_t)0x200000;
  float* qf = (float*)(uintptr_t)0x300000;

  CHECK(ss_scan_num_chunks(2048, 8) == 256);
  CHECK(ss_scan_num_chunks(100, 64) == 2);
  CHECK(ss_scan_bwd_workspace_size(4, 2048, 4096, 16, 8, SS_BF16) > 0);
  CHECK(conv1d_causal_bwd_workspace_size(4, 2048, 4096, 4) > 0);
  CHECK(rmsnorm_bwd_workspace_size(8192, 2048) > 0);
  CHECK(ss_count_nonfinite_workspace_size() >= 4096);
  CHECK(strlen(ss_strerror(SS_OK)) > 0);
  CHECK(strcmp(ss_strerror(SS_ERR_NULL), ss_strerror(SS_ERR_DIM)) != 0);

  /* forward: NULL x, bad N, bad dims, unknown dtype */
  CHECK(ss_scan_fwd(NULL, p, pf, p, p, pf, p, NULL, p, qf, NULL, 2, 64, 16, 4, 64, SS_F32, NULL, 0, NULL, 0, NULL) ==
        SS_ERR_NULL);
  CHECK(ss_scan_fwd(p, p, pf, p, p, pf, p, NULL, p, qf, NULL, 2, 64, 16, 5, 64, SS_F32, NULL, 0, NULL, 0, NULL) ==
        SS_ERR_UNSUPPORTED);
  CHECK(ss_scan_fwd(p, p, pf, p, p, pf, p, NULL, p, qf, NULL, 0, 64, 16, 4, 64, SS_F32, NULL, 0, NULL, 0, NULL) ==
        SS_ERR_DIM);
  CHECK(ss_scan_fwd(p, p, pf, p, p, pf, p, NULL, p, qf, NULL, 2, 64, 16, 4, 64, 7, NULL, 0, NULL, 0, NULL) ==
        SS_ERR_UNSUPPORTED);
  /* conv backward: missing workspace */
  CHECK(conv1d_causal_bwd(pf, p, pf, qf, qf, qf, 2, 64, 16, 4, SS_F32, NULL, 0, NULL) == SS_ERR_WORKSPACE);
  /* RMSNorm backward: NULL dy */
  CHECK(rmsnorm_bwd(NULL, p, pf, pf, qf, qf, 4, 64, SS_F32, p, 1 << 20, NULL) == SS_ERR_NULL);
  /* non-finite count: unknown dtype */
  CHECK(ss_count_nonfinite(p, 16, 9, (unsigned long long*)p, p, 1 << 16, NULL) == SS_ERR_UNSUPPORTED);

  if (failures == 0) printf("abi_from_c: all checks passed\n");
  return failures == 0 ? 0 : 1;
}
