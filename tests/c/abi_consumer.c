/*
 * A plain C99 program that uses the library only through its header: it
 * checks that the header compiles as C, that the program links against
 * libmoe_gb300.so, and that the calls which need no GPU behave as declared.
 * Prints one "ok" line and exits 0, or names the first failed check and
 * exits 1.
 */
#include <stdio.h>
#include <string.h>

#include "moe_gb300.h"

#define CHECK(cond)                                         \
  do {                                                      \
    if (!(cond)) {                                          \
      fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
      return 1;                                             \
    }                                                       \
  } while (0)

int main(void) {
  moe_cache* cache = NULL;
  moe_expert_views v;
  moe_status st;

  CHECK(moe_version() >= 1);
  /* MXFP4 expert at H=4096, I=2048: three matrices of codes and E8M0 scales */
  CHECK(moe_fp4_expert_bytes(4096, 2048) == (size_t)13369344);
  CHECK(moe_fp4_expert_bytes(4096, 2047) == 0);

  /* argument checks return before any device work, with a message */
  st = moe_cache_create(0, 1, 8, 4096, NULL, NULL, &cache);
  CHECK(st == MOE_ERR_INVALID);
  CHECK(cache == NULL);
  CHECK(strlen(moe_last_error()) > 0);

  st = moe_mx_quantize(NULL, 2, 48, NULL, NULL, NULL);
  CHECK(st == MOE_ERR_INVALID);

  /* a successful host-only call clears the thread's message */
  st = moe_cache_destroy(NULL);
  CHECK(st == MOE_OK);
  CHECK(moe_last_error()[0] == '\0');

  /* workspace sizing is host arithmetic over the views */
  memset(&v, 0, sizeof v);
  v.H = 4096;
  v.I = 2048;
  v.fp4_num_slots = 64;
  CHECK(moe_expert_forward_workspace(&v, 64, 8) > 0);
  CHECK(moe_expert_forward_workspace(NULL, 64, 8) == 0);

  printf("ok\n");
  return 0;
}
