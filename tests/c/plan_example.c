/* A plain C99 caller of the library's host-only entry points: fills the
 * parameter block for B4 H16 S4096 d128 causal (device pointers are only
 * validated, never dereferenced, by these calls), asks for the launch plan
 * and the scheduler's work order, and checks the error reporting of an
 * unsupported head dimension. Exits 0 and prints "ok" on success. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "attn_fwd.h"

static int fail(const char *what) {
  fprintf(stderr, "FAILED: %s (%s)\n", what, attn_fwd_last_error());
  return 1;
}

int main(void) {
  attn_fwd_params p;
  attn_fwd_plan_info info;
  attn_work_tile tiles[16];
  int64_t n;
  const int64_t B = 4, S = 4096, H = 16, D = 128;

  if (attn_fwd_params_size() != sizeof(attn_fwd_params)) return fail("params layout");
  attn_fwd_params_init(&p);
  p.q = (const void *)(uintptr_t)0x100000;
  p.k = (const void *)(uintptr_t)0x200000;
  p.v = (const void *)(uintptr_t)0x300000;
  p.o = (void *)(uintptr_t)0x400000;
  p.workspace = (void *)(uintptr_t)0x500000;
  p.workspace_bytes = attn_fwd_workspace_bytes(&p);
  p.batch = (int32_t)B;
  p.seqlen_q = p.seqlen_k = (int32_t)S;
  p.num_heads_q = p.num_heads_kv = (int32_t)H;
  p.head_dim_qk = p.head_dim_v = (int32_t)D;
  p.causal = 1;
  p.softmax_scale = 0.08838834764831845f;
  p.q_stride[0] = p.k_stride[0] = p.v_stride[0] = p.o_stride[0] = S * H * D;
  p.q_stride[1] = p.k_stride[1] = p.v_stride[1] = p.o_stride[1] = H * D;
  p.q_stride[2] = p.k_stride[2] = p.v_stride[2] = p.o_stride[2] = D;
  p.workspace_bytes = attn_fwd_workspace_bytes(&p);
  if (p.workspace_bytes != ATTN_FWD_WORKSPACE_BYTES) return fail("workspace size");

  if (attn_fwd_plan(&p, &info) != ATTN_OK) return fail("plan");
  if (info.rows_per_tile != 256 || info.work_tiles != B * H * (S / 256) || info.num_splits != 1 ||
      info.block != 512 || info.tmem_columns != 512)
    return fail("plan contents");

  n = attn_fwd_schedule(&p, NULL, tiles, 16);
  if (n != B * H * (S / 256)) return fail("schedule length");
  if (tiles[0].batch != 0 || tiles[0].tile != S / 256 - 1 || tiles[0].split != 0)
    return fail("heaviest tile first");

  p.head_dim_qk = p.head_dim_v = 96;
  if (attn_fwd_plan(&p, &info) != ATTN_ERR_UNSUPPORTED) return fail("unsupported dims accepted");
  if (strlen(attn_fwd_last_error()) == 0) return fail("no error text");
  if (strcmp(attn_status_string(ATTN_ERR_UNSUPPORTED), "unsupported configuration") != 0)
    return fail("status string");

  printf("ok\n");
  return 0;
}
