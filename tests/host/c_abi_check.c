/* Plain C11 user of the library's C ABI: include/attn.h must compile as C, and every
 * entry point it declares must resolve from the shared library at link time.  Calls
 * only what needs no GPU: the version, status strings, workspace sizes and argument
 * checks that fail before any CUDA call. */
#include <stdio.h>
#include <string.h>

#include "attn.h"

typedef void (*any_fn)(void);

int main(void) {
  const any_fn entry_points[] = {
      (any_fn)attn_fwd, (any_fn)attn_fwd_bf16, (any_fn)attn_fwd_gqa, (any_fn)attn_fwd_gqa_bf16,
      (any_fn)attn_fwd_splitkv, (any_fn)attn_fwd_splitkv_bf16, (any_fn)attn_fwd_splitkv_noalloc,
      (any_fn)attn_splitkv_workspace_bytes, (any_fn)attn_splitkv_default_splits, (any_fn)attn_decode_paged,
      (any_fn)attn_decode_paged_bf16, (any_fn)attn_decode_workspace_bytes, (any_fn)attn_decode_default_splits,
      (any_fn)attn_paged_append, (any_fn)attn_row_softmax_f32, (any_fn)attn_device_status,
      (any_fn)attn_watchdog_selftest, (any_fn)attn_anatomy_read, (any_fn)attn_status_string,
      (any_fn)attn_version};
  const size_t n = sizeof(entry_points) / sizeof(entry_points[0]);
  for (size_t i = 0; i < n; ++i) {
    if (entry_points[i] == NULL) return 1;
  }
  const char* ok = attn_status_string(ATTN_OK);
  const char* bad = attn_status_string(ATTN_ERR_INVALID_ARG);
  if (ok == NULL || bad == NULL || strcmp(ok, bad) == 0) return 2;
  /* NULL tensors: rejected before anything touches a GPU. */
  if (attn_fwd(NULL, NULL, NULL, NULL, NULL, 1, 1, 128, 64, 1, 0.125f, NULL) != ATTN_ERR_INVALID_ARG) return 3;
  /* [splits, BH, N, D] fp32 partials + [splits, BH, N] fp32 lse, each rounded up to 256 bytes. */
  if (attn_splitkv_workspace_bytes(1, 2, 256, 64, 2) != (size_t)(2 * 2 * 256 * 64 * 4 + 2 * 2 * 256 * 4)) return 4;
  printf("entry points %zu, version %d, status 0 \"%s\"\n", n, attn_version(), ok);
  return 0;
}
