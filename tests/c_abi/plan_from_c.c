/* A plain C99 caller of the library: plans the tiny decode batch (KV
 * lengths 1, 17, 64, 100 on 16-token pages; 8 query heads over 2 kv heads,
 * head_dim 64), plans it again with a left window through the documented
 * default options, and checks three host-side error paths. No kernel is
 * launched and no device memory is touched. Prints one line of results. */
#include <stdio.h>

#include "fi.h"

int main(void) {
  const int32_t page_indptr[5] = {0, 1, 3, 7, 14};
  const int32_t last_page_len[4] = {1, 1, 16, 4};
  fi_plan_t plan = NULL, windowed = NULL, unused = NULL;
  size_t ws = 0, ws_windowed = 0, ws_unused = 0;
  fi_plan_info info, info_w;
  fi_plan_options opt = FI_PLAN_OPTIONS_DEFAULT;
  fi_status st;

  st = fi_plan(FI_MODE_DECODE, 4, NULL, page_indptr, last_page_len, 8, 2, 64, 16, 0, NULL, 152,
               &plan, &ws);
  if (st != FI_OK) {
    printf("fi_plan: %s\n", fi_status_string(st));
    return 1;
  }
  if (fi_plan_get_info(plan, &info) != FI_OK) return 2;

  opt.window_left = 15; /* a decode row keeps its last 16 keys */
  st = fi_plan(FI_MODE_DECODE, 4, NULL, page_indptr, last_page_len, 8, 2, 64, 16, 0, &opt, 152,
               &windowed, &ws_windowed);
  if (st != FI_OK || fi_plan_get_info(windowed, &info_w) != FI_OK) return 3;

  /* head_dim 96 is valid but not built */
  st = fi_plan(FI_MODE_DECODE, 4, NULL, page_indptr, last_page_len, 8, 2, 96, 16, 0, NULL, 152,
               &unused, &ws_unused);
  if (st != FI_ERR_UNSUPPORTED || unused != NULL) return 4;
  /* a decreasing page_indptr */
  {
    const int32_t bad[5] = {0, 3, 1, 7, 14};
    st = fi_plan(FI_MODE_DECODE, 4, NULL, bad, last_page_len, 8, 2, 64, 16, 0, NULL, 152,
                 &unused, &ws_unused);
    if (st != FI_ERR_INVALID_ARG) return 5;
  }
  /* a run call with too small a workspace returns before touching anything */
  st = fi_batch_decode_paged(plan, (const void*)0x100000, (const void*)0x100000,
                             (const void*)0x100000, FI_LAYOUT_NHD, 0, 14,
                             (const int32_t*)0x100000, (const int32_t*)0x100000,
                             (const int32_t*)0x100000, 0.125f, 1.0f, 1.0f, NULL, NULL,
                             (void*)0x100000, NULL, (void*)0x100000, 16, NULL);
  if (st != FI_ERR_WORKSPACE_TOO_SMALL) return 6;

  printf("total_kv_tokens %lld items %d windowed_kv_tokens %lld windowed_items %d ws_ok %d\n",
         (long long)info.total_kv_tokens, info.num_items, (long long)info_w.total_kv_tokens,
         info_w.num_items, ws == (size_t)info.workspace_bytes);
  fi_plan_destroy(plan);
  fi_plan_destroy(windowed);
  fi_plan_destroy(NULL);
  return 0;
}
