/* The C ABI from plain C (C99, no CUDA headers): a host-only plan object
 * (no workspace) validates and plans; refusals come back as status codes
 * with a message. Exits non-zero on the first unexpected result. */
#include <stdio.h>
#include <string.h>

#include "fi.h"

static int expect(const char* what, fi_status got, fi_status want) {
  if (got != want) {
    printf("%s: got %s, want %s (%s)\n", what, fi_status_str(got), fi_status_str(want),
           fi_last_error());
    return 1;
  }
  return 0;
}

int main(void) {
  fi_plan_t p = NULL;
  int bad = 0;
  /* two decode requests: 40 and 17 keys in pages of 16 */
  const int32_t kv_indptr[3] = {0, 3, 5};
  const int32_t last_page_len[2] = {8, 1};
  bad |= expect("create", fi_plan_create(&p, NULL, 0, 0, 0, 0), FI_OK);
  bad |= expect("run before plan",
                fi_batch_decode_paged(p, NULL, NULL, NULL, NULL, 1.0f, NULL, NULL, NULL),
                FI_ERR_NOT_PLANNED);
  bad |= expect("decode plan", fi_plan(p, NULL, kv_indptr, last_page_len, 2, 16, 32, 8, 128, 0,
                                       -1, FI_BF16, 1, 0, NULL), FI_OK);
  bad |= expect("GQA 32/7", fi_plan(p, NULL, kv_indptr, last_page_len, 2, 16, 32, 7, 128, 0, -1,
                                    FI_BF16, 1, 0, NULL), FI_ERR_GQA_INDIVISIBLE);
  if (!bad && strstr(fi_last_error(), "num_kv_heads") == NULL) {
    printf("refusal message does not name the field: %s\n", fi_last_error());
    bad = 1;
  }
  bad |= expect("zero kv heads", fi_plan(p, NULL, kv_indptr, last_page_len, 2, 16, 32, 0, 128, 0,
                                         -1, FI_BF16, 1, 0, NULL), FI_ERR_GQA_INDIVISIBLE);
  {
    /* causal prefill of 20 rows over 17 keys: kv shorter than q */
    const int32_t qo_indptr[3] = {0, 4, 24};
    bad |= expect("kv < q", fi_plan(p, qo_indptr, kv_indptr, last_page_len, 2, 16, 32, 8, 128, 1,
                                    -1, FI_BF16, 0, 0, NULL), FI_ERR_KV_SHORTER_THAN_Q);
  }
  {
    fi_plan_info info;
    memset(&info, 0, sizeof info);
    /* the refused plans left the decode plan in place */
    bad |= expect("info", fi_plan_get_info(p, &info, NULL, 0, NULL, 0), FI_OK);
    if (!bad && (info.batch != 2 || info.total_rows != 2)) {
      printf("plan after refusals: batch %d rows %d\n", info.batch, info.total_rows);
      bad = 1;
    }
  }
  fi_plan_destroy(p);
  if (!bad) printf("c abi ok\n");
  return bad;
}
