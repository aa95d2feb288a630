/* Host cost of one attn_fwd call through the C ABI, for the 128-token
 * workload shape (B1 H2 S128 d64, no mask): the time the calling thread
 * spends inside attn_fwd (validation, tensor-map encoding or reuse, launch),
 * and the time per call of back-to-back calls (the larger of that host time
 * and the kernel time), both averaged over many calls. Prints one line:
 *   enqueue_us <t> back_to_back_us <t> ok
 * Inputs are zero (the numbers do not depend on values). */
#define _POSIX_C_SOURCE 199309L
#include <cuda_runtime.h>
#include <stdio.h>
#include <time.h>

#include "attn_fwd.h"

enum { B = 1, S = 128, H = 2, D = 64, CALLS = 2000, BATCH = 50 };

static double now_us(void) {
  struct timespec ts;
  clock_gettime(CLOCK_MONOTONIC, &ts);
  return (double)ts.tv_sec * 1e6 + (double)ts.tv_nsec * 1e-3;
}

#define CK(x)                                                                  \
  do {                                                                         \
    cudaError_t e_ = (x);                                                      \
    if (e_ != cudaSuccess) {                                                   \
      fprintf(stderr, "CUDA error %s at %s\n", cudaGetErrorString(e_), #x);    \
      return 1;                                                                \
    }                                                                          \
  } while (0)

int main(void) {
  const size_t n = (size_t)B * S * H * D;
  void *dq, *dk, *dv, *dout, *ws;
  float *dl;
  attn_fwd_params p;
  cudaStream_t st;
  double inside = 0.0, t0, t1;
  int i, j;

  CK(cudaStreamCreate(&st));
  CK(cudaMalloc(&dq, n * 2));
  CK(cudaMalloc(&dk, n * 2));
  CK(cudaMalloc(&dv, n * 2));
  CK(cudaMalloc(&dout, n * 2));
  CK(cudaMalloc((void **)&dl, sizeof(float) * B * H * S));
  CK(cudaMemset(dq, 0, n * 2));
  CK(cudaMemset(dk, 0, n * 2));
  CK(cudaMemset(dv, 0, n * 2));

  attn_fwd_params_init(&p);
  p.q = dq; p.k = dk; p.v = dv; p.o = dout; p.lse = dl;
  p.batch = B; p.seqlen_q = p.seqlen_k = S; p.num_heads_q = p.num_heads_kv = H;
  p.head_dim_qk = p.head_dim_v = D; p.causal = 0; p.softmax_scale = 0.125f;
  p.q_stride[0] = p.k_stride[0] = p.v_stride[0] = p.o_stride[0] = (int64_t)S * H * D;
  p.q_stride[1] = p.k_stride[1] = p.v_stride[1] = p.o_stride[1] = (int64_t)H * D;
  p.q_stride[2] = p.k_stride[2] = p.v_stride[2] = p.o_stride[2] = D;
  p.workspace_bytes = attn_fwd_workspace_bytes(&p);
  CK(cudaMalloc(&ws, p.workspace_bytes));
  CK(cudaMemset(ws, 0, p.workspace_bytes));
  p.workspace = ws;

  /* warm-up: first-call set-up (tensor maps, kernel attributes, module load) */
  for (i = 0; i < 20; ++i)
    if (attn_fwd(&p, st) != ATTN_OK) {
      fprintf(stderr, "attn_fwd: %s\n", attn_fwd_last_error());
      return 1;
    }
  if (attn_fwd_check(ws, st) != ATTN_OK) {
    fprintf(stderr, "attn_fwd_check: %s\n", attn_fwd_last_error());
    return 1;
  }

  /* time inside attn_fwd; the stream drains between batches, untimed */
  for (i = 0; i < CALLS / BATCH; ++i) {
    for (j = 0; j < BATCH; ++j) {
      t0 = now_us();
      if (attn_fwd(&p, st) != ATTN_OK) return 1;
      t1 = now_us();
      inside += t1 - t0;
    }
    CK(cudaStreamSynchronize(st));
  }

  /* back-to-back calls */
  CK(cudaStreamSynchronize(st));
  t0 = now_us();
  for (i = 0; i < CALLS; ++i)
    if (attn_fwd(&p, st) != ATTN_OK) return 1;
  CK(cudaStreamSynchronize(st));
  t1 = now_us();
  if (attn_fwd_check(ws, st) != ATTN_OK) return 1;
  printf("enqueue_us %.3f back_to_back_us %.3f ok\n", inside / CALLS, (t1 - t0) / CALLS);
  return 0;
}
