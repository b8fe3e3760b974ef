/*
 * A plain C99 user of libpkx: includes only pkx.h, links libpkx.so, and
 * makes the calls that need no GPU (version, workspace sizes, host-side
 * argument checks).  It shows that the boundary is usable without Python or
 * torch.  Exit status 0 when every check holds; the failing check otherwise.
 */
#include <stdio.h>
#include <string.h>

#include "pkx.h"

static int failures = 0;

#define CHECK(cond)                                               \
  do {                                                            \
    if (!(cond)) {                                                \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, \
              #cond);                                             \
      ++failures;                                                 \
    }                                                             \
  } while (0)

int main(void) {
  const char *ver = pkx_version();
  CHECK(ver != NULL && strstr(ver, "sm_103a") != NULL);

  /* Workspace sizes are pure host arithmetic. */
  {
    size_t ext = pkx_extend_workspace_size(16, 9000, 32, 8, 128, 128);
    size_t dec = pkx_decode_workspace_size(64, 32, 8, 128, 128);
    size_t dec_min = pkx_decode_workspace_min_size(64, 32, 8, 128, 128);
    CHECK(ext > 0);
    CHECK(dec > 0);
    CHECK(dec_min > 0 && dec_min <= dec);
  }

  /* merge_state with null pointers: rejected on the host, with a reason. */
  {
    int rc = pkx_merge_state(NULL, NULL, NULL, NULL, NULL, NULL, 4, 8, 128,
                             NULL);
    const char *why = pkx_last_error_string();
    CHECK(rc == PKX_EINVAL);
    CHECK(why != NULL && why[0] != '\0');
  }

  /* Unified index build with a negative batch: rejected on the host. */
  {
    int rc = pkx_build_unified_kv_indices(NULL, NULL, NULL, NULL, NULL, -1,
                                          NULL, NULL, NULL, NULL);
    CHECK(rc == PKX_EINVAL);
  }

  if (failures == 0) printf("ok %s\n", ver);
  return failures == 0 ? 0 : 1;
}
