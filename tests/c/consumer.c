/* A plain C99 consumer of the library's C ABI: it includes only
 * include/treeverify.h, links libtreeverify.so and exercises calls that need
 * no GPU (status strings, the version, the attention's split plan for an
 * explicit SM count, and argument checks that return before any launch).
 * Prints "ok" and exits 0 when every answer is the documented one. */
#include <stdio.h>
#include <string.h>

#include "treeverify.h"

static int failures = 0;

static void expect(int cond, const char* what) {
  if (!cond) {
    fprintf(stderr, "FAILED: %s\n", what);
    ++failures;
  }
}

int main(void) {
  int32_t row_groups = 0, splits = 0, kps = 0;
  size_t ws = 0;
  char fake_buf[64];
  void* fake = fake_buf + (16 - ((size_t)fake_buf & 15)) % 16; /* never dereferenced */

  expect(strcmp(tv_status_string(TV_OK), "ok") == 0, "status string of TV_OK");
  expect(strcmp(tv_status_string(99), "unknown status") == 0, "status string of 99");
  expect(tv_version() >= 100, "version");
  expect(tv_attn_uses_tensor_cores(TV_BF16) == 1, "bf16 runs on the tensor cores");

  /* the full verify step's layer on 152 SMs */
  expect(tv_attn_plan(64, 64, 8, 128, TV_BF16, 4096, 152, &row_groups, &splits, &kps, &ws) ==
             TV_OK, "plan status");
  expect(row_groups == 2 && splits == 9 && kps == 512, "plan of the full step");
  expect(ws == (size_t)9 * 4096 * 4 + (size_t)9 * 4096 * 128 * 2, "workspace of the full step");
  expect(tv_attn_plan(64, 64, 8, 96, TV_BF16, 4096, 152, &row_groups, &splits, &kps, &ws) ==
             TV_ERR_UNSUPPORTED, "d = 96 unsupported");

  /* host-side rejections, before anything reaches a device */
  expect(tv_tree_accept(NULL, 10, fake, fake, 3, 0, fake, fake, fake, fake, fake, fake, fake,
                        NULL, NULL) == TV_ERR_INVALID_ARG, "accept without logits");
  expect(tv_kv_compact(fake, fake, 2, 1 << 20, 2, 12, 64, TV_BF16, 10, 5, fake, NULL, NULL) ==
             TV_ERR_CAPACITY, "compaction past the capacity");
  {
    const int32_t off[3] = {0, 5, 140}, prefix[2] = {10, 20};
    expect(tv_tree_accept_batched(2, off, prefix, (const float*)fake, 100, fake, fake, fake,
                                  fake, fake, fake, fake, fake, fake, NULL, NULL) ==
               TV_ERR_INVALID_ARG, "batched accept with a 135-node request");
  }

  if (failures == 0) printf("ok\n");
  return failures == 0 ? 0 : 1;
}
