/* The C ABI used from plain C11 (no C++ and no CUDA headers in this file):
 * status strings, argument checks that refuse before touching a device, and
 * the host block manager end to end (admit, prefix hit, fork, copy-on-write,
 * swap out / in). Prints one line per check; exits non-zero on a failure.
 * Needs no GPU. */
#include <stdio.h>
#include <string.h>

#include "pagedattn.h"

static int failures = 0;

static void check(int ok, const char* what) {
  printf("%s %s\n", ok ? "ok" : "FAIL", what);
  if (!ok) ++failures;
}

int main(void) {
  check(strcmp(pa_status_string(PA_OK), "ok") == 0, "status string of PA_OK");
  check(pa_decode(NULL, NULL, NULL, NULL, 1, 4, 1, 1.0f, NULL, NULL, 0, 0, NULL) == PA_ERR_INVALID_ARG,
        "pa_decode refuses a null pool");
  check(pa_pool_block_bytes(NULL) == 0, "block bytes of a null pool");

  pa_block_manager* bm = NULL;
  check(pa_bm_create(8, 4, 1, &bm) == PA_OK && bm != NULL, "create a block manager");
  const int32_t prompt[6] = {10, 11, 12, 13, 14, 15}; /* one full block + 2 tokens */
  int32_t cached = -1;
  check(pa_bm_add_sequence(bm, 1, prompt, 6, &cached) == PA_OK && cached == 0, "admit sequence 1");
  check(pa_bm_add_sequence(bm, 2, prompt, 5, &cached) == PA_OK && cached == 4, "prefix hit of one block");
  check(pa_bm_fork(bm, 1, 3) == PA_OK, "fork sequence 1");
  int32_t src = -1, dst = -1, ncopy = -1;
  const int32_t tok = 16;
  check(pa_bm_append_tokens(bm, 3, &tok, 1, &src, &dst, 1, &ncopy) == PA_OK && ncopy == 1 && src != dst,
        "copy-on-write of the shared tail");
  int32_t table[4], nblocks = 0;
  int64_t len = 0;
  check(pa_bm_block_table(bm, 3, table, 4, &nblocks, &len) == PA_OK && nblocks == 2 && len == 7 &&
            table[1] == dst && table[2] == -1,
        "block table of the fork");
  check(pa_bm_set_cpu_blocks(bm, 4) == PA_OK, "host tier of 4 slots");
  int32_t g[4], c[4], n = -1;
  check(pa_bm_swap_out(bm, 3, g, c, 4, &n) == PA_OK && n == 2 && g[1] == dst, "swap out the fork");
  check(pa_bm_block_table(bm, 3, table, 4, &nblocks, &len) == PA_ERR_INVALID_ARG, "no table while swapped out");
  check(pa_bm_swap_in(bm, 3, c, g, 4, &n) == PA_OK && n == 2 && pa_bm_num_free_cpu_blocks(bm) == 4,
        "swap back in");
  check(pa_bm_free_sequence(bm, 1) == PA_OK && pa_bm_free_sequence(bm, 2) == PA_OK &&
            pa_bm_free_sequence(bm, 3) == PA_OK && pa_bm_num_free_blocks(bm) == 8,
        "every block free again");
  check(pa_bm_destroy(bm) == PA_OK, "destroy");
  printf("%d failure(s)\n", failures);
  return failures != 0;
}
