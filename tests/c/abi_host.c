/* Plain C99 use of the library's C ABI without a GPU: a host-resident index
 * of the worked-example catalogue ("What problem does it solve": the items
 * 3-5-1 and 3-5-4 share the prefix 3-5), its statistics and its exported
 * step-3 table, and the error path of a bad argument. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "zerogr.h"

int main(void) {
  /* L = 3, V = 8: five items, the prefix 3-5 followed by 1 and 4 */
  const int32_t sids[5][3] = {{3, 5, 1}, {3, 5, 4}, {3, 2, 7}, {0, 1, 2}, {6, 6, 6}};
  zg_build_opts opts;
  memset(&opts, 0, sizeof opts);
  opts.residency = ZG_RESIDENT_HOST;
  zg_index* idx = NULL;
  if (zg_index_build(&sids[0][0], 5, 3, 8, &opts, NULL, &idx) != ZG_OK) {
    printf("build failed: %s\n", zg_last_error());
    return 1;
  }
  zg_index_info info;
  if (zg_index_info_get(idx, &info) != ZG_OK) return 2;
  zg_step_stats st;
  if (zg_index_stats(idx, 3, &st) != ZG_OK) return 3;
  size_t bytes = 0;
  if (zg_index_export(idx, 3, NULL, &bytes) != ZG_OK) return 4;
  unsigned char* buf = (unsigned char*)malloc(bytes);
  if (!buf || zg_index_export(idx, 3, buf, &bytes) != ZG_OK) return 5;
  printf("version %s\n", zg_version());
  printf("unique %lld rows3 %u nnz3 %u maxfan3 %u bytes3 %zu\n", (long long)info.n_unique, st.rows, st.nnz,
         st.max_fanout, bytes);
  free(buf);
  /* a token outside the codebook is an argument error with a message */
  const int32_t bad[1][3] = {{3, 5, 9}};
  zg_index* idx2 = NULL;
  const zg_status e = zg_index_build(&bad[0][0], 1, 3, 8, &opts, NULL, &idx2);
  printf("bad token status %d message %s\n", (int)e, zg_last_error()[0] ? "set" : "empty");
  zg_index_free(idx);
  return 0;
}
