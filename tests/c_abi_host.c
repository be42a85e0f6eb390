/* A C99 caller of librx's host-side calls: accounting, the radix cache, the contract checks and
 * plan building / introspection (no device is touched).  Built and run by test_c_abi.py; prints
 * "ok" and exits 0 when every check holds, else names the failing line. */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "rx.h"

#define CHECK(c)                                            \
  do {                                                      \
    if (!(c)) {                                             \
      printf("FAIL line %d: %s\n", __LINE__, #c);           \
      return 1;                                             \
    }                                                       \
  } while (0)

int main(void) {
  /* token accounting: the prefix-caching page's 1,000-token prefix at units 16 and 1 */
  CHECK(rx_saved_tokens(1000, 16) == 992);
  CHECK(rx_saved_tokens(1000, 1) == 1000);
  CHECK(fabs(rx_token_saving(1, 4) - 75.0) < 1e-12);
  CHECK(isnan(rx_token_saving(1, 0)));
  CHECK(fabs(rx_compute_reduction(2000, 100) - 2000.0 / 2100.0) < 1e-12);

  /* radix cache: insert, longest-prefix match (slots returned), match unit, stats */
  {
    rx_radix* t = NULL;
    int32_t a[6] = {1, 2, 3, 4, 5, 6}, sa[6] = {10, 11, 12, 13, 14, 15};
    int32_t b[5] = {1, 2, 3, 9, 9}, out[5];
    int64_t added = -1, saved = -1, ntok = -1, nodes = -1;
    CHECK(rx_radix_create(&t) == RX_OK && t != NULL);
    CHECK(rx_radix_insert(t, a, sa, 6, &added) == RX_OK && added == 6);
    CHECK(rx_radix_match(t, b, 5, 1, &saved, out) == RX_OK && saved == 3);
    CHECK(out[0] == 10 && out[1] == 11 && out[2] == 12);
    CHECK(rx_radix_match(t, b, 5, 2, &saved, NULL) == RX_OK && saved == 2);
    CHECK(rx_radix_stats(t, &ntok, &nodes) == RX_OK && ntok == 6 && nodes == 1);
    rx_radix_destroy(t);
  }

  /* contract checks */
  {
    int32_t slots[4] = {3, 1, 3, 0};
    int64_t bad = -2;
    CHECK(rx_check_slots(slots, 4, 8, &bad) == RX_ERR_INVALID && bad == 2);
    CHECK(strlen(rx_last_error()) > 0);
    CHECK(rx_check_slots(slots, 2, 8, &bad) == RX_OK && bad == -1);
  }

  /* a decode plan built on the host; the table pointer is recorded, never dereferenced here */
  {
    rx_kv_desc d;
    rx_plan* p = NULL;
    int32_t ri[2] = {0, 1}, sl[2] = {200, 150}, grp[2] = {0, 0}, gpl[1] = {100};
    size_t ws = 0;
    int32_t launches = -1;
    int64_t reads = -1;
    memset(&d, 0, sizeof d);
    d.num_q_heads = 8;
    d.num_kv_heads = 2;
    d.head_dim = 128;
    d.softmax_scale = 0.088f;
    d.pool_size = 4096;
    d.req_to_token = (const int32_t*)0x1000;
    d.req_to_token_rows = 4;
    d.req_to_token_stride = 256;
    CHECK(rx_plan_create(&p) == RX_OK);
    CHECK(rx_decode_plan(p, &d, 2, ri, sl, grp, 1, gpl) == RX_OK);
    CHECK(rx_plan_workspace_size(p, &ws) == RX_OK && ws > 256);
    /* 2 members x 4 query heads = 8 rows: mma.sync units and the merge */
    CHECK(rx_plan_launches(p, &launches) == RX_OK && launches == 2);
    /* the shared 100 keys once, then 100 and 50 own keys, for 2 KV heads */
    CHECK(rx_plan_key_reads(p, &reads) == RX_OK && reads == (100 + 100 + 50) * 2);
    d.head_dim = 64;
    CHECK(rx_decode_plan(p, &d, 2, ri, sl, grp, 1, gpl) == RX_ERR_UNSUPPORTED);
    rx_plan_destroy(p);
  }
  CHECK(strcmp(rx_status_string(RX_ERR_RANGE), "out of range") == 0);
  printf("ok\n");
  return 0;
}
