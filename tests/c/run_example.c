/* A plain C99 program that runs the attention forward on the GPU through the
 * C ABI, with the CUDA runtime for device memory. With Q = 0 every visible
 * score is 0, so each weight is exactly 1: O_i = mean of V_0..V_i (causal)
 * and LSE_i = ln(i + 1), which the program checks for a ragged length.
 * Exits 0 and prints "ok" on success. */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "attn_fwd.h"

enum { B = 1, S = 300, H = 2, D = 128 };

static uint16_t to_bf16(float x) { /* exact for the small integers used here */
  uint32_t u;
  memcpy(&u, &x, sizeof(u));
  return (uint16_t)(u >> 16);
}
static float from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float x;
  memcpy(&x, &u, sizeof(x));
  return x;
}
static float vval(int j, int d) { return (float)((j * 5 + d) % 7 - 3); }

#define CK(x)                                                          \
  do {                                                                 \
    cudaError_t e_ = (x);                                              \
    if (e_ != cudaSuccess) {                                           \
      fprintf(stderr, "CUDA error %s at %s\n", cudaGetErrorString(e_), #x); \
      return 1;                                                        \
    }                                                                  \
  } while (0)

int main(void) {
  const size_t n = (size_t)B * S * H * D;
  uint16_t *hq = calloc(n, 2), *hk = malloc(n * 2), *hv = malloc(n * 2), *ho = malloc(n * 2);
  float *hl = malloc(sizeof(float) * B * H * S);
  void *dq, *dk, *dv, *dout, *ws;
  float *dl;
  attn_fwd_params p;
  int t, h, d, j;
  double worst_o = 0.0, worst_l = 0.0;

  for (t = 0; t < S; ++t)
    for (h = 0; h < H; ++h)
      for (d = 0; d < D; ++d) {
        hk[((size_t)t * H + h) * D + d] = to_bf16((float)((t + 3 * d + h) % 5 - 2));
        hv[((size_t)t * H + h) * D + d] = to_bf16(vval(t, d) + (float)h);
      }
  CK(cudaMalloc(&dq, n * 2));
  CK(cudaMalloc(&dk, n * 2));
  CK(cudaMalloc(&dv, n * 2));
  CK(cudaMalloc(&dout, n * 2));
  CK(cudaMalloc((void **)&dl, sizeof(float) * B * H * S));
  CK(cudaMemcpy(dq, hq, n * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dk, hk, n * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dv, hv, n * 2, cudaMemcpyHostToDevice));

  attn_fwd_params_init(&p);
  p.q = dq; p.k = dk; p.v = dv; p.o = dout; p.lse = dl;
  p.batch = B; p.seqlen_q = p.seqlen_k = S; p.num_heads_q = p.num_heads_kv = H;
  p.head_dim_qk = p.head_dim_v = D; p.causal = 1; p.softmax_scale = 0.125f;
  p.q_stride[0] = p.k_stride[0] = p.v_stride[0] = p.o_stride[0] = (int64_t)S * H * D;
  p.q_stride[1] = p.k_stride[1] = p.v_stride[1] = p.o_stride[1] = (int64_t)H * D;
  p.q_stride[2] = p.k_stride[2] = p.v_stride[2] = p.o_stride[2] = D;
  p.workspace_bytes = attn_fwd_workspace_bytes(&p);
  CK(cudaMalloc(&ws, p.workspace_bytes));
  CK(cudaMemset(ws, 0, p.workspace_bytes));
  p.workspace = ws;

  if (attn_fwd(&p, NULL) != ATTN_OK) {
    fprintf(stderr, "attn_fwd: %s\n", attn_fwd_last_error());
    return 1;
  }
  if (attn_fwd_check(ws, NULL) != ATTN_OK) {
    fprintf(stderr, "attn_fwd_check: %s\n", attn_fwd_last_error());
    return 1;
  }
  CK(cudaMemcpy(ho, dout, n * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(hl, dl, sizeof(float) * B * H * S, cudaMemcpyDeviceToHost));

  for (h = 0; h < H; ++h)
    for (t = 0; t < S; ++t) {
      const double lse_ref = log((double)(t + 1));
      const double el = fabs((double)hl[(size_t)h * S + t] - lse_ref);
      if (el > worst_l) worst_l = el;
      for (d = 0; d < D; ++d) {
        double mean = 0.0;
        for (j = 0; j <= t; ++j) mean += vval(j, d) + (double)h;
        mean /= (double)(t + 1);
        {
          const double eo = fabs((double)from_bf16(ho[((size_t)t * H + h) * D + d]) - mean);
          if (eo > worst_o) worst_o = eo;
        }
      }
    }
  printf("O max-abs %.3e, LSE max-abs %.3e\n", worst_o, worst_l);
  if (worst_o > 2e-2 || worst_l > 1e-4) return 1;
  cudaFree(dq); cudaFree(dk); cudaFree(dv); cudaFree(dout); cudaFree(dl); cudaFree(ws);
  free(hq); free(hk); free(hv); free(ho); free(hl);
  printf("ok\n");
  return 0;
}
