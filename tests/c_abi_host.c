/* A C program against the C ABI (include/ringattn.h, libringattn.so):
 * the host-side calls that need no GPU.  Built and run by
 * tests/test_abi_cpu.py; prints "ok" and exits 0 when every check holds.
 *
 * Checks: create validates its arguments; the causal striped plan of
 * N = 1024, P = 4 pairs step s with block (r - s) mod P and its shards do
 * equal work (the striped layout's point); the allowed pairs over all
 * shards are B*H*N*(N+1)/2; options are validated; the backward's
 * workspace grows by the accumulator buffers in the per-step schedule. */
#include <stdio.h>
#include <stdlib.h>

#include "ringattn.h"

#define CHECK(cond)                                                      \
  do {                                                                   \
    if (!(cond)) {                                                       \
      fprintf(stderr, "check failed at line %d: %s (%s)\n", __LINE__, #cond, \
              ring_attn_last_error());                                   \
      return 1;                                                          \
    }                                                                    \
  } while (0)

int main(void) {
  ring_attn_t h = NULL;
  /* N not a multiple of P, and d not 64 or 128, are rejected */
  CHECK(ring_attn_create(&h, 1, 2, 1000, 128, 3, 1, RING_LAYOUT_STRIPED) != RING_OK && h == NULL);
  CHECK(ring_attn_create(&h, 1, 2, 1024, 96, 4, 1, RING_LAYOUT_STRIPED) != RING_OK && h == NULL);

  const int B = 1, H = 2, P = 4;
  const long long N = 1024;
  CHECK(ring_attn_create(&h, B, H, N, 128, P, 1, RING_LAYOUT_STRIPED) == RING_OK && h != NULL);
  for (int s = 0; s < P; ++s)
    for (int r = 0; r < P; ++r) {
      int j = -1, cls = -1;
      long long delta = 0;
      CHECK(ring_attn_plan_block(h, r, s, &j, &cls, &delta) == RING_OK);
      CHECK(j == ((r - s) % P + P) % P);
    }
  long long pairs[4], tiles[4], total = 0;
  CHECK(ring_attn_shard_work(h, pairs, tiles) == RING_OK);
  for (int r = 0; r < P; ++r) total += pairs[r];
  CHECK(total == (long long)B * H * N * (N + 1) / 2);
  for (int r = 1; r < P; ++r) {
    long long diff = pairs[r] - pairs[0];
    if (diff < 0) diff = -diff;
    CHECK(diff * 100 <= pairs[0]); /* within 1 % of each other */
  }

  CHECK(ring_attn_set_option(h, RING_OPT_ROTATION, 3) == RING_ERR_INVALID_ARG);
  CHECK(ring_attn_set_option(h, RING_OPT_BWD_LAP, 1) == RING_OK);
  size_t lap = 0, per_step = 0, fwd = 0;
  CHECK(ring_attn_bwd_workspace_size(h, &lap) == RING_OK);
  CHECK(ring_attn_set_option(h, RING_OPT_BWD_LAP, 0) == RING_OK);
  CHECK(ring_attn_bwd_workspace_size(h, &per_step) == RING_OK);
  CHECK(per_step >= lap + 4 * (size_t)B * H * N * 128 * 4);
  CHECK(ring_attn_workspace_size(h, &fwd) == RING_OK && fwd > 0);

  CHECK(ring_attn_fwd_host(h, NULL, NULL, NULL, NULL, NULL, NULL) == RING_ERR_INVALID_ARG);
  CHECK(ring_attn_destroy(h) == RING_OK);
  CHECK(ring_attn_destroy(NULL) == RING_OK);
  printf("ok\n");
  return 0;
}
