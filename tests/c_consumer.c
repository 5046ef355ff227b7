/*
 * A plain C program against include/pagedattn.h and libpagedattn.so: the
 * header needs no C++ and no CUDA include, and every entry point is callable
 * from C. Only host-side argument checks are exercised (no GPU needed): each
 * call below must be refused before any CUDA call. Prints "c consumer ok".
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "pagedattn.h"

#define FAKE ((void*)0x10000) /* aligned, never dereferenced */

static int fails = 0;

static void expect(int got, int want, const char* what) {
  if (got != want) {
    printf("%s: got %d, want %d\n", what, got, want);
    ++fails;
  }
}

int main(void) {
  if (strcmp(pa_status_str(PA_OK), "ok") != 0) ++fails;
  /* prefill: Hkv must divide Hq */
  expect(pa_attn_prefill(FAKE, FAKE, FAKE, FAKE, NULL, 1, 6, 4, 16, 64, NULL, 0, 1, 0, 0.f,
                         PA_BF16, NULL, NULL),
         PA_ERR_INVALID_ARG, "prefill Hkv");
  /* nothing to do: no launch */
  expect(pa_attn_prefill(FAKE, FAKE, FAKE, FAKE, NULL, 1, 4, 2, 0, 64, NULL, 0, 1, 0, 0.f,
                         PA_BF16, NULL, NULL),
         PA_OK, "prefill empty");
  /* decode: block size 16 only */
  expect(pa_attn_decode_paged(FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, NULL, 1, 4, 2, 64, 32, 8, 0,
                              0.f, 0, NULL, 0, PA_BF16, NULL, NULL),
         PA_ERR_UNSUPPORTED, "decode block size");
  /* backward: a workspace is required */
  expect(pa_attn_prefill_backward(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 2,
                                  16, 64, NULL, 0, 1, 0, 0.f, NULL, 0, PA_BF16, NULL, NULL),
         PA_ERR_WORKSPACE, "backward workspace");
  if (pa_attn_prefill_backward_workspace_bytes(16, 4, 64) == 0) ++fails;
  /* MLA: the scale is required */
  expect(pa_mla_decode_paged(FAKE, FAKE, FAKE, 8, FAKE, FAKE, NULL, 1, 16, 512, 64, 16, 8, 0.f, 0,
                             NULL, 0, PA_BF16, NULL, NULL),
         PA_ERR_INVALID_ARG, "mla scale");
  expect(pa_mla_append_paged(FAKE, FAKE, FAKE, 4, FAKE, NULL, 3, 2, 576, 16, 8, PA_BF16, NULL,
                             NULL),
         PA_ERR_INVALID_ARG, "mla append count");
  expect(pa_copy_blocks(FAKE, FAKE, FAKE, FAKE, 0, 16, 2, 64, 8, PA_BF16, NULL, NULL), PA_OK,
         "copy nothing");
  if (fails) return 1;
  printf("c consumer ok\n");
  return 0;
}
