/* A C caller of the library: compiles against include/sparse_engine.h alone
 * and exercises host-only paths (no GPU needed): status strings, argument
 * rejection before any launch, and the workspace size queries. Prints "ok"
 * and returns 0 when every check holds. */
#include <stdio.h>
#include <string.h>

#include "sparse_engine.h"

static int failures = 0;

static void check(int cond, const char* what) {
  if (!cond) {
    fprintf(stderr, "FAILED: %s\n", what);
    ++failures;
  }
}

int main(void) {
  check(strcmp(se_status_string(SE_OK), "SE_OK") == 0, "status string of SE_OK");
  check(strcmp(se_status_string(SE_ERR_WORKSPACE), "SE_ERR_WORKSPACE") == 0, "status string of SE_ERR_WORKSPACE");

  /* A NULL cache view is rejected on the host, before anything is launched. */
  se_status_t st = se_sparse_paged_decode(NULL, NULL, 32, NULL, 1, NULL, 1, NULL, NULL, 1, 1.0f, NULL, NULL, NULL,
                                          0, NULL);
  check(st == SE_ERR_INVALID_ARG, "NULL kv rejected with SE_ERR_INVALID_ARG");
  check(strstr(se_last_error_detail(), "kv") != NULL, "error detail names the argument");

  /* A page size other than 16 is rejected too. */
  se_paged_kv_t kv;
  memset(&kv, 0, sizeof(kv));
  kv.k = kv.v = (void*)(uintptr_t)0x1000;
  kv.num_pages = 4;
  kv.num_kv_heads = 1;
  kv.page_size = 32;
  kv.head_dim = kv.head_dim_v = 128;
  kv.row_stride_k = kv.row_stride_v = 128;
  st = se_sparse_paged_decode_noalloc(&kv, NULL, 4, NULL, 1, NULL, 0, NULL, NULL, 1, 1.0f, NULL, NULL, NULL);
  check(st == SE_ERR_INVALID_ARG, "page_size 32 rejected");

  /* Workspace sizes are host arithmetic. */
  check(se_sparse_decode_workspace_size(32, 32, 4, 128, 257) > 0, "decode workspace size");
  check(se_sparse_decode_workspace_size(-1, 32, 4, 128, 257) == 0, "negative batch gives size 0");
  check(se_snapkv_workspace_size(4, 8, 32, 32768) > 0, "SnapKV workspace size");

  if (failures == 0) printf("ok\n");
  return failures == 0 ? 0 : 1;
}
