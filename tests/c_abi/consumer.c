/* A plain C99 consumer of the C ABI declared in include/wtconv.h.
 *
 * It must compile as strict C99 (-std=c99 -pedantic -Wall -Wextra -Werror)
 * and link against libwtconv.so.  It calls only paths that the library
 * refuses during argument validation, before any device work, so it runs
 * without a GPU: status strings, bad descriptors, null and misaligned
 * pointers, workspace sizes and too-small workspaces.  The pointers are a
 * fixed address that is never dereferenced.  Exit status 0 when every check
 * holds. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "wtconv.h"

static int failures = 0;
#define EXPECT(cond)                                            \
  do {                                                          \
    if (!(cond)) {                                              \
      printf("failed: %s (line %d)\n", #cond, __LINE__);        \
      ++failures;                                               \
    }                                                           \
  } while (0)

int main(void) {
  const uintptr_t fake = 0x10000; /* never dereferenced: each call is refused first */
  float* const p = (float*)fake;
  wtconv_desc_t d;
  size_t need;

  EXPECT(strcmp(wtconv_status_string(WTCONV_OK), "WTCONV_OK") == 0);
  EXPECT(strcmp(wtconv_status_string(WTCONV_ERR_WORKSPACE), "WTCONV_ERR_WORKSPACE") == 0);

  /* a layer the library takes: x[2,4,56,56] float32, 3 levels, k = 5 */
  d.N = 2; d.C = 4; d.H = 56; d.W = 56; d.levels = 3; d.k = 5; d.dtype = WTCONV_F32;

  /* bad descriptors */
  d.k = 4;
  EXPECT(wtconv_fwd(&d, p, p, p, p, p, p, p, NULL, 0, NULL) == WTCONV_ERR_INVALID_ARG);
  EXPECT(strlen(wtconv_last_error()) > 0);
  d.k = 5;
  d.levels = 9;
  EXPECT(wtconv_bwd_data(&d, p, p, p, p, p, p, NULL, 0, NULL) == WTCONV_ERR_INVALID_ARG);
  d.levels = 3;
  EXPECT(wtconv_fwd(NULL, p, p, p, p, p, p, p, NULL, 0, NULL) == WTCONV_ERR_INVALID_ARG);

  /* null and misaligned pointers */
  EXPECT(wtconv_fwd(&d, NULL, p, p, p, p, p, p, NULL, 0, NULL) == WTCONV_ERR_INVALID_ARG);
  EXPECT(wtconv_fwd(&d, (void*)(fake + 2), p, p, p, p, p, p, NULL, 0, NULL) == WTCONV_ERR_MISALIGNED);

  /* workspaces */
  need = wtconv_workspace_size(&d, WTCONV_OP_BWD_WEIGHT);
  EXPECT(need > 0 && need % 256 == 0);
  EXPECT(wtconv_workspace_size(&d, WTCONV_OP_FWD) == 0);
  EXPECT(wtconv_bwd_weight(&d, p, p, p, p, p, p, p, p, p, p, p, p, NULL, need, NULL) == WTCONV_ERR_WORKSPACE);
  EXPECT(wtconv_bwd_weight(&d, p, p, p, p, p, p, p, p, p, p, p, p, p, need - 256, NULL) == WTCONV_ERR_WORKSPACE);
  need = wtconv_workspace_size(&d, WTCONV_OP_BWD);
  EXPECT(need > 0 && need % 256 == 0);
  EXPECT(wtconv_bwd(&d, p, p, p, p, p, p, p, p, p, p, p, p, p, NULL, need, NULL) == WTCONV_ERR_WORKSPACE);
  EXPECT(wtconv_bwd(&d, p, p, p, p, p, p, p, NULL, p, p, p, p, p, p, need, NULL) == WTCONV_ERR_INVALID_ARG);

  if (failures == 0) printf("ok\n");
  return failures != 0;
}
