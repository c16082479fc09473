/* A plain C11 client of the library's host-side calls, used by
 * tests/test_abi_c.py: it proves that include/hb.h compiles as C (not only
 * as C++) and that the calls work without Python.  It prints a text trace
 * that the test compares line by line with the same calls made through the
 * Python binding.  No GPU is touched: hb_plan runs without a workspace (host
 * plan only) and the batch's device pointers are never dereferenced. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "hb.h"

static int plan_trace(void) {
  /* rows (q_len, context_len): a decode row, a 5-token chunk, a 40-token
   * chunk after 60 cached tokens; 32 q / 8 kv heads, head_dim 128 */
  const int32_t q_len[3] = {1, 5, 40};
  const int32_t ctx[3] = {40, 9, 100};
  hb_batch b;
  memset(&b, 0, sizeof b);
  b.num_seqs = 3;
  b.total_q = 46;
  b.max_pages_per_seq = 7;
  b.num_pages = 12;
  b.num_q_heads = 32;
  b.num_kv_heads = 8;
  b.head_dim = 128;
  b.page_size = 16;
  b.cu_q_len = (const int32_t*)(uintptr_t)0x1000;     /* never dereferenced */
  b.context_len = (const int32_t*)(uintptr_t)0x1000;
  b.block_table = (const int32_t*)(uintptr_t)0x1000;
  size_t plan_bytes = 0, ws_bytes = 0;
  hb_status s = hb_plan(&b, q_len, ctx, 152, NULL, &plan_bytes, NULL, &ws_bytes, NULL);
  if (s != HB_OK) return 1;
  printf("sizes %zu %zu\n", plan_bytes, ws_bytes);
  unsigned char* plan = (unsigned char*)malloc(plan_bytes);
  if (!plan) return 1;
  s = hb_plan(&b, q_len, ctx, 152, plan, &plan_bytes, NULL, &ws_bytes, NULL);
  if (s != HB_OK) {
    free(plan);
    return 1;
  }
  printf("plan ");
  for (size_t i = 0; i < plan_bytes; ++i) printf("%02x", plan[i]);
  printf("\n");
  free(plan);
  /* a row breaking 1 <= q_len <= context_len */
  const int32_t bad_q[3] = {1, 10, 40};
  s = hb_plan(&b, bad_q, ctx, 152, NULL, &plan_bytes, NULL, &ws_bytes, NULL);
  printf("bad_row %s %d\n", hb_status_string(s), hb_last_error()[0] != '\0');
  s = hb_plan(NULL, q_len, ctx, 152, NULL, &plan_bytes, NULL, &ws_bytes, NULL);
  printf("null_batch %s %d\n", hb_status_string(s), hb_last_error()[0] != '\0');
  return 0;
}

static int builder_trace(void) {
  enum { kMaxRows = 8, kMaxPages = 4 };
  hb_builder* bld = NULL;
  if (hb_builder_create(24, 16, 10, kMaxPages, NULL, &bld) != HB_OK) return 1;
  /* id, prompt, max_new */
  const int64_t ids[3] = {7, 3, 9};
  const int32_t prompt[3] = {30, 5, 12};
  const int32_t max_new[3] = {2, 1, 3};
  for (int i = 0; i < 3; ++i)
    if (hb_builder_add_request(bld, ids[i], prompt[i], max_new[i]) != HB_OK) return 1;
  printf("duplicate %s\n", hb_status_string(hb_builder_add_request(bld, 7, 4, 1)));
  for (int it = 0; it < 16; ++it) {
    int32_t n = 0, over = 0;
    int32_t q[kMaxRows], c[kMaxRows], bt[kMaxRows * kMaxPages], kind[kMaxRows];
    int64_t rid[kMaxRows];
    if (hb_builder_step(bld, kMaxRows, &n, q, c, bt, rid, kind, &over) != HB_OK) return 1;
    if (n == 0) break;
    printf("step %d rows %d over %d\n", it, n, over);
    for (int r = 0; r < n; ++r) {
      printf("  row %lld kind %d q %d ctx %d pages", (long long)rid[r], kind[r], q[r], c[r]);
      for (int p = 0; p < kMaxPages; ++p) printf(" %d", bt[r * kMaxPages + p]);
      printf("\n");
    }
    int32_t nf = 0;
    int64_t fin[kMaxRows];
    if (hb_builder_complete(bld, kMaxRows, &nf, fin) != HB_OK) return 1;
    printf("  finished");
    for (int i = 0; i < nf; ++i) printf(" %lld", (long long)fin[i]);
    printf("\n");
  }
  int32_t w = 0, r = 0, f = 0;
  if (hb_builder_counts(bld, &w, &r, &f) != HB_OK) return 1;
  printf("counts %d %d %d\n", w, r, f);
  hb_builder_destroy(bld);
  return 0;
}

int main(void) {
  for (int s = HB_OK; s <= HB_ERR_OUT_OF_PAGES; ++s)
    printf("status %d %s\n", s, hb_status_string((hb_status)s));
  if (plan_trace() != 0) return 2;
  if (builder_trace() != 0) return 3;
  return 0;
}
