/*
 * A plain C99 caller of libh3attn: compiles against include/h3attn.h alone
 * and checks, without touching a GPU, the answers the host-side validation
 * gives before any launch.  Exit status 0 = every check held; otherwise the
 * failing line is printed.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "h3attn.h"

static int failures = 0;

#define EXPECT(call, want)                                                              \
  do {                                                                                  \
    h3attn_status_t got_ = (call);                                                      \
    if (got_ != (want)) {                                                               \
      printf("line %d: %s returned %d (%s), expected %d\n", __LINE__, #call, (int)got_, \
             h3attn_status_string(got_), (int)(want));                                  \
      ++failures;                                                                       \
    }                                                                                   \
  } while (0)

int main(void) {
  /* fake, 16-byte aligned device addresses: validation answers before any use */
  void* q = (void*)(uintptr_t)0x10000;
  void* k = (void*)(uintptr_t)0x20000;
  void* v = (void*)(uintptr_t)0x30000;
  void* o = (void*)(uintptr_t)0x40000;
  const float* w = (const float*)(uintptr_t)0x50000;
  const float* cs = (const float*)(uintptr_t)0x60000;
  h3attn_mask_t mask;
  h3attn_window_t win;

  if (h3attn_version() != 10000) {
    printf("version %d\n", h3attn_version());
    ++failures;
  }
  for (int s = 0; s <= 7; ++s) {
    const char* text = h3attn_status_string((h3attn_status_t)s);
    if (!text || !strcmp(text, "unknown status")) {
      printf("no text for status %d\n", s);
      ++failures;
    }
  }

  /* prefill: B, Sq, Sk, Hq, Hkv, D, scale, mask, causal */
  EXPECT(h3attn_prefill(q, k, v, o, 1, 256, 256, 4, 4, 96, 0.1f, NULL, 0, NULL), H3ATTN_ERR_UNSUPPORTED_HEAD_DIM);
  EXPECT(h3attn_prefill(q, k, v, o, 1, 256, 256, 4, 3, 128, 0.1f, NULL, 0, NULL), H3ATTN_ERR_INVALID_ARG);
  EXPECT(h3attn_prefill(q, k, v, o, 1, 256, 256, 4, 4, 128, 0.0f, NULL, 0, NULL), H3ATTN_ERR_INVALID_ARG);
  EXPECT(h3attn_prefill(q, k, v, o, 1, 256, 512, 4, 4, 128, 0.1f, NULL, 1, NULL), H3ATTN_ERR_INVALID_ARG);
  EXPECT(h3attn_prefill((char*)q + 8, k, v, o, 1, 256, 256, 4, 4, 128, 0.1f, NULL, 0, NULL), H3ATTN_ERR_MISALIGNED);
  EXPECT(h3attn_prefill(q, k, v, q, 1, 256, 256, 4, 4, 128, 0.1f, NULL, 0, NULL), H3ATTN_ERR_INVALID_ARG);
  EXPECT(h3attn_prefill(q, k, v, o, 0, 256, 256, 4, 4, 128, 0.1f, NULL, 0, NULL), H3ATTN_OK); /* empty batch */
  memset(&mask, 0, sizeof mask);
  mask.kv_len = (const int32_t*)((uintptr_t)0x70000 + 2);
  EXPECT(h3attn_prefill(q, k, v, o, 1, 256, 256, 4, 4, 128, 0.1f, &mask, 0, NULL), H3ATTN_ERR_MISALIGNED);

  /* norm/RoPE: B, S, Hq, Hkv, D, rotary_dim, eps */
  EXPECT(h3attn_qk_norm_rope(q, k, w, w, cs, cs, 1, 64, 4, 4, 128, 91, 1e-6f, NULL), H3ATTN_ERR_INVALID_ARG); /* odd */
  EXPECT(h3attn_qk_norm_rope(q, k, w, w, cs, cs, 1, 64, 4, 4, 100, 96, 1e-6f, NULL), H3ATTN_ERR_UNSUPPORTED_HEAD_DIM);
  EXPECT(h3attn_qk_norm_rope(q, k, w, w, NULL, NULL, 1, 64, 4, 4, 128, 96, 1e-6f, NULL), H3ATTN_ERR_INVALID_ARG);
  EXPECT(h3attn_qk_norm_rope(q, q, w, w, cs, cs, 1, 64, 4, 4, 128, 96, 1e-6f, NULL), H3ATTN_ERR_INVALID_ARG);
  EXPECT(h3attn_qk_norm_rope_out(q, k, o, v, w, w, cs, cs, 1, 64, 4, 4, 128, 96, -1.0f, NULL), H3ATTN_ERR_INVALID_ARG);

  /* window: frame_tokens, anchor_frames, chunk_frames, radius */
  EXPECT(h3attn_prefill_window(q, k, v, o, 1, 256, 4, 4, 128, 0.1f, NULL, NULL, NULL), H3ATTN_ERR_INVALID_ARG);
  win.frame_tokens = 16; win.anchor_frames = 1; win.chunk_frames = 5; win.radius = 1;
  EXPECT(h3attn_prefill_window(q, k, v, o, 1, 256, 4, 4, 256, 0.1f, &win, NULL, NULL), H3ATTN_ERR_UNSUPPORTED_HEAD_DIM);
  win.chunk_frames = 0;
  EXPECT(h3attn_prefill_window(q, k, v, o, 1, 256, 4, 4, 128, 0.1f, &win, NULL, NULL), H3ATTN_ERR_INVALID_ARG);

  /* AdaLN modulation: T, C, N, eps */
  EXPECT(h3attn_rmsnorm_modulate(q, o, NULL, k, v, NULL, 16, 100, 2, 1e-6f, NULL), H3ATTN_ERR_INVALID_ARG);
  EXPECT(h3attn_rmsnorm_modulate(q, o, NULL, k, v, NULL, 16, 16384, 2, 1e-6f, NULL), H3ATTN_ERR_INVALID_ARG);
  EXPECT(h3attn_rmsnorm_modulate(q, o, NULL, k, v, NULL, 0, 3072, 2, 1e-6f, NULL), H3ATTN_OK); /* no rows */

  if (failures == 0) printf("abi_check: ok\n");
  return failures == 0 ? 0 : 1;
}
