/* A plain C caller of libpageddecode: includes the public header, links the shared
 * library and exercises its host-only paths (no GPU needed): version, the split
 * planner, argument validation and the last-error string. */
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#include "pageddecode.h"

static pd_decode_desc desc(void) {
  pd_decode_desc d;
  memset(&d, 0, sizeof(d));
  d.B = 32;
  d.H_qo = 32;
  d.H_kv = 8;
  d.D = 128;
  d.page_size = 16;
  d.q_dtype = PD_BF16;
  d.kv_dtype = PD_BF16;
  d.out_dtype = PD_BF16;
  d.max_pages = 16384;
  d.nnz_pages = 4608;
  d.k_scale = 1.0f;
  d.v_scale = 1.0f;
  return d;
}

int main(void) {
  printf("version %d\n", (int)pd_version());
  pd_decode_desc d = desc();
  int32_t schedule = -1, grid = -1;
  size_t ws = 0;
  pd_status st = pd_plan(&d, 152, 2, &schedule, &grid, &ws);
  printf("plan %d schedule %d grid %d workspace %zu\n", (int)st, (int)schedule, (int)grid, ws);
  d.H_qo = 30; /* not a multiple of H_kv */
  st = pd_batch_decode_paged_kv(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 1.0f,
                                1e4f, 0.1f, &d, NULL);
  printf("bad heads %d %s\n", (int)st, pd_get_last_error_string());
  d = desc();
  d.flags = 4;
  st = pd_batch_decode_paged_kv(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 1.0f,
                                1e4f, 0.1f, &d, NULL);
  printf("bad flags %d\n", (int)st);
  st = pd_batch_decode_paged_kv_mq(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 0,
                                   1.0f, 1e4f, 0.1f, &d, NULL);
  printf("bad q_len %d\n", (int)st);
  /* host copies of the page table: one without the other, or a decreasing indptr */
  {
    int32_t ip[3] = {0, 2, 1}, li[2] = {5, 5};
    d = desc();
    d.B = 2;
    d.nnz_pages = 2;
    d.host_indptr = ip;
    st = pd_batch_decode_paged_kv((void*)16, (void*)16, (int32_t*)16, (int32_t*)16, (int32_t*)16, NULL,
                                  NULL, (void*)16, (float*)16, 0, 1.0f, 1e4f, 0.1f, &d, NULL);
    printf("host alone %d\n", (int)st);
    d.host_length_info = li;
    st = pd_batch_decode_paged_kv((void*)16, (void*)16, (int32_t*)16, (int32_t*)16, (int32_t*)16, NULL,
                                  NULL, (void*)16, (float*)16, 0, 1.0f, 1e4f, 0.1f, &d, NULL);
    printf("host decreasing %d\n", (int)st);
  }
  printf("desc %zu %zu %zu\n", sizeof(pd_decode_desc), offsetof(pd_decode_desc, host_indptr),
         offsetof(pd_decode_desc, host_length_info));
  return 0;
}
