/*
 * A plain C99 caller of libsmla: the header compiles as C, the library links
 * from C, and the host-only entry points answer as the header documents
 * (layout fields, workspace sizing, argument errors, status names).  No device
 * work is enqueued.  Exit status 0 = every check passed; otherwise the number
 * of the first failed check.
 */
#include <stdio.h>
#include <string.h>

#include "smla.h"

#define CHECK(n, cond)                                   \
  do {                                                   \
    if (!(cond)) {                                       \
      fprintf(stderr, "check %d failed: %s\n", n, #cond); \
      return n;                                          \
    }                                                    \
  } while (0)

int main(void) {
  smla_layout_t lay;
  smla_params_t prm;
  memset(&lay, 0, sizeof lay);
  CHECK(1, smla_layout_init(&lay, 64, 1, 512, 64, 128, 128, 1000) == SMLA_OK);
  /* 512 E4M3 latent codes + 4 fp32 scales + 64 bf16 rope values = 656 bytes per token */
  CHECK(2, lay.rec_bytes == 656 && lay.rec_stride == 656 && lay.n_scales == 4);
  CHECK(3, lay.idx_key_off == 41984 && lay.idx_scale_off == 50176 && lay.block_stride == 50432);
  CHECK(4, smla_layout_init(&lay, 64, 1, 500, 64, 128, 128, 1000) == SMLA_ERR_INVALID_ARG);
  CHECK(5, smla_layout_init(&lay, 64, 1, 512, 64, 128, 128, 1000) == SMLA_OK);

  prm.n_heads = 64;
  prm.n_idx_heads = 64;
  prm.top_k = 2048;
  prm.softmax_scale = 1.0f / 24.0f;
  /* scores [4, 1000] fp32 and top-k indices [4, 2048] int32 at least */
  CHECK(6, smla_workspace_size(&lay, &prm, 4, 1000) >= (size_t)(4 * 1000 * 4 + 4 * 2048 * 4));
  CHECK(7, smla_workspace_size(&lay, &prm, 0, 1000) == 0);
  CHECK(8, smla_topk_workspace_size(&prm, 100000) == 0);

  /* argument errors come back before any device work */
  CHECK(9, kvpack_store(NULL, NULL, 0, NULL, NULL, NULL, NULL, NULL, 1, NULL) == SMLA_ERR_INVALID_ARG);
  CHECK(10, kvpack_store(&lay, NULL, 0, NULL, NULL, NULL, NULL, NULL, 0, NULL) == SMLA_OK);
  CHECK(11, smla_topk(&prm, NULL, 0, NULL, NULL, 1, 4, NULL, NULL, 0, NULL) == SMLA_ERR_INVALID_ARG);

  {
    /* The two fused entry points refuse the same malformed arguments with the same status,
     * before any device work.  The dummy pointers are never dereferenced on the host. */
    void* p = (void*)(uintptr_t)4096;
    const uint8_t* u8 = (const uint8_t*)p;
    const float* f32 = (const float*)p;
    const int32_t* i32 = (const int32_t*)p;
    const int64_t* i64 = (const int64_t*)p;
    smla_layout_t bad;
    smla_params_t bp;
    int c;
    for (c = 0; c < 6; ++c) {
      smla_status_t want = SMLA_ERR_INVALID_ARG;
      const void* q_pe = p;
      bad = lay;
      bp = prm;
      if (c == 0) bad.quant_tile = 0;        /* not a layout smla_layout_init makes */
      if (c == 1) bad.block_stride = 0;
      if (c == 2) bad.idx_key_off += 16;
      if (c == 3) q_pe = NULL;               /* d_rope > 0 needs q_pe */
      if (c == 4) bp.n_heads = 0;
      if (c == 5) {
        bp.n_idx_heads = 3;                  /* a shape the kernels do not build */
        want = SMLA_ERR_UNSUPPORTED;
      }
      CHECK(20 + c, smla_decode(&bad, &bp, p, 0, p, p, u8, f32, i64, p, q_pe, u8, f32, i32, 16, i32, i32, 1, 1, 1,
                                1000, p, (float*)p, NULL, p, (size_t)1 << 30, NULL) == want);
      CHECK(30 + c, smla_decode_static(&bad, &bp, p, 0, p, p, u8, f32, i64, p, q_pe, u8, f32, i32, 16, i32, i32, 1,
                                       1, 1, 1000, p, (float*)p, NULL, NULL) == want);
    }
  }

  /* FP4 (E2M1) indexer keys: 64 packed bytes per key instead of 128 */
  CHECK(40, smla_layout_init_keys(&lay, 64, 1, 512, 64, 128, 128, SMLA_KEY_E2M1, 1000) == SMLA_OK);
  CHECK(41, lay.idx_key_format == SMLA_KEY_E2M1 && lay.idx_scale_off == 46080 && lay.block_stride == 46336);
  CHECK(42, smla_layout_init_keys(&lay, 64, 1, 512, 64, 128, 128, 7, 1000) == SMLA_ERR_INVALID_ARG);
  CHECK(43, smla_layout_init(&lay, 64, 1, 512, 64, 128, 128, 1000) == SMLA_OK && lay.idx_key_format == SMLA_KEY_E4M3);

  CHECK(12, strcmp(smla_status_string(SMLA_ERR_BAD_INDEX), "SMLA_ERR_BAD_INDEX") == 0);
  CHECK(13, strcmp(smla_status_string(SMLA_ERR_SCRATCH_LIMIT), "SMLA_ERR_SCRATCH_LIMIT") == 0);
  CHECK(14, smla_version() >= 100);
  printf("abi host check ok\n");
  return 0;
}
