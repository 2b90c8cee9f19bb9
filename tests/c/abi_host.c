/* A plain C99 program against the C ABI: the header compiles as C, and the
 * host-only entry points (no GPU needed) link and behave.  Exit status 0 on
 * success; each failed check prints its line. */
#include <stddef.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "pagedattn.h"

static int failures = 0;
#define CHECK(c)                                                  \
  do {                                                            \
    if (!(c)) {                                                   \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
      ++failures;                                                 \
    }                                                             \
  } while (0)

int main(void) {
  CHECK(pa_status_string(PA_OK) != NULL);
  CHECK(pa_version() != NULL);

  /* a plan for two sequences, GQA-2, D = 64 */
  pa_shape_t s;
  memset(&s, 0, sizeof(s));
  s.batch = 2;
  s.num_q_heads = 4;
  s.num_kv_heads = 2;
  s.head_dim = 64;
  s.page_size = 16;
  s.max_pages_per_seq = 8;
  s.num_pages = 32;
  s.dtype = PA_DTYPE_F16;
  const int32_t lens[2] = {37, 100};
  pa_plan_t plan;
  CHECK(pa_plan(&s, lens, 152, 0, &plan) == PA_OK);
  CHECK(plan.num_work_items >= 2 * 2);
  CHECK(plan.workspace_bytes >= plan.blob_bytes && plan.blob_bytes > 0);
  CHECK(plan.host_blob != NULL && plan.owns_blob == 1);
  pa_plan_free(&plan);
  CHECK(plan.host_blob == NULL);

  /* shape errors are returned, not trapped */
  pa_shape_t bad = s;
  bad.head_dim = 96;
  CHECK(pa_plan(&bad, lens, 152, 0, &plan) != PA_OK);
  const int32_t too_long[2] = {37, 8 * 16 + 1};
  CHECK(pa_plan(&s, too_long, 152, 0, &plan) == PA_ERR_INVALID_ARG);

  /* the block allocator: all or nothing, validated frees */
  pa_block_allocator_t* a = NULL;
  CHECK(pa_block_allocator_create(8, &a) == PA_OK && a != NULL);
  int32_t blocks[8];
  CHECK(pa_block_alloc(a, 5, blocks) == PA_OK);
  CHECK(pa_block_num_free(a) == 3);
  CHECK(pa_block_alloc(a, 4, blocks + 5) == PA_ERR_NO_MEMORY);
  CHECK(pa_block_num_free(a) == 3);
  CHECK(pa_block_free(a, blocks, 5) == PA_OK);
  CHECK(pa_block_num_free(a) == 8);
  CHECK(pa_block_free(a, blocks, 1) != PA_OK); /* already free */
  pa_block_allocator_destroy(a);

  /* the multi-token plan covers every query row */
  const int32_t qls[2] = {37, 5};
  pa_prefill_plan_t pp;
  CHECK(pa_prefill_plan(&s, lens, qls, &pp) == PA_OK);
  CHECK(pp.total_q == 42 && pp.num_tiles > 0);
  pa_prefill_plan_free(&pp);

  /* the public structs' layout, for the ctypes binding to compare */
  printf("layout pa_shape_t %zu\n", sizeof(pa_shape_t));
  printf("layout pa_plan_t %zu merge %zu q8_stages %zu wait_limit_ns %zu early_kv %zu\n",
         sizeof(pa_plan_t), offsetof(pa_plan_t, merge), offsetof(pa_plan_t, q8_stages),
         offsetof(pa_plan_t, wait_limit_ns), offsetof(pa_plan_t, early_kv));
  printf("layout pa_plan_options_t %zu q8_stages %zu wait_limit_ns %zu early_kv %zu\n",
         sizeof(pa_plan_options_t), offsetof(pa_plan_options_t, q8_stages),
         offsetof(pa_plan_options_t, wait_limit_ns), offsetof(pa_plan_options_t, early_kv));
  printf("layout pa_prefill_plan_t %zu wait_limit_ns %zu\n", sizeof(pa_prefill_plan_t),
         offsetof(pa_prefill_plan_t, wait_limit_ns));
  printf("layout pa_prefill_options_t %zu wait_limit_ns %zu\n", sizeof(pa_prefill_options_t),
         offsetof(pa_prefill_options_t, wait_limit_ns));
  if (failures == 0) printf("abi ok\n");
  return failures == 0 ? 0 : 1;
}
