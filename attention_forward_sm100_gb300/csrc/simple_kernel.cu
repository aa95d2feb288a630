// Plain fp32 CUDA-core attention forward, used only to cross-check the
// tcgen05 kernel and the host-side argument handling (strides, packed
// sequences, GQA, rope, FP8 scales, depth-major FP8 V, LSE layout). One warp owns one query row;
// each lane scores one key of a 32-key chunk, the chunk's softmax update is a
// warp reduction, and each lane accumulates Dv/32 output columns.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "internal.h"

namespace af {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxD = 256;   // Dqk + R and Dv bound of this kernel

__device__ __forceinline__ float load_qk(const void* base, int64_t idx, int fp8) {
  if (fp8) {
    __nv_fp8_e4m3 x;
    x.__x = static_cast<const __nv_fp8_storage_t*>(base)[idx];
    return static_cast<float>(x);
  }
  return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
}

__global__ void __launch_bounds__(kWarps * 32) simple_attn_kernel(const attn_fwd_params p) {
  __shared__ float q_sh[kWarps][kMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, h = blockIdx.y;
  const int i = blockIdx.x * kWarps + warp;     // query row within the sequence
  const bool packed = p.cu_seqlens_q != nullptr;
  int64_t q_base_tok = 0, k_base_tok = 0;
  int lq = p.seqlen_q, lk = p.seqlen_k;
  if (packed) {
    q_base_tok = p.cu_seqlens_q[b];
    lq = p.cu_seqlens_q[b + 1] - p.cu_seqlens_q[b];
    k_base_tok = p.cu_seqlens_k[b];
    lk = p.cu_seqlens_k[b + 1] - p.cu_seqlens_k[b];
    // offsets outside q/k/v/o: leave the sequence alone (cross-check kernel only)
    if (q_base_tok < 0 || lq < 0 || q_base_tok + lq > p.total_q || k_base_tok < 0 || lk < 0 ||
        k_base_tok + lk > p.total_k)
      return;
  }
  if (i >= lq) return;
  const int hk = h / (p.num_heads_q / p.num_heads_kv);
  const int dq = p.head_dim_qk, dr = p.rope_depth, dv = p.head_dim_v;
  const int fp8 = p.qk_dtype == ATTN_DTYPE_FP8_E4M3;
  const bool v_fp8 = p.v_dtype == ATTN_DTYPE_FP8_E4M3;   // weights stay fp32 here (no P rounding)
  const int64_t bq = packed ? 0 : b, tq = q_base_tok + i;

  // Q row (nope then rope) into shared memory, as fp32.
  for (int d = lane; d < dq; d += 32)
    q_sh[warp][d] = load_qk(p.q, bq * p.q_stride[0] + tq * p.q_stride[1] + h * p.q_stride[2] + d, fp8);
  for (int d = lane; d < dr; d += 32)
    q_sh[warp][dq + d] = __bfloat162float(static_cast<const __nv_bfloat16*>(p.q_rope)[
        bq * p.q_rope_stride[0] + tq * p.q_rope_stride[1] + h * p.q_rope_stride[2] + d]);
  __syncwarp();

  float qs = 1.f;
  if (fp8) qs = packed ? p.q_scale[(int64_t)h * p.total_q + tq]
                       : p.q_scale[((int64_t)b * p.num_heads_q + h) * p.seqlen_q + i];
  const float scale = p.softmax_scale * qs;

  const int kv_end = p.causal ? min(lk, i + 1) : lk;
  float m = -INFINITY, l = 0.f;
  float acc[kMaxD / 32];
#pragma unroll
  for (int c = 0; c < kMaxD / 32; ++c) acc[c] = 0.f;

  for (int j0 = 0; j0 < kv_end; j0 += 32) {
    const int j = j0 + lane;
    float s = -INFINITY;
    if (j < kv_end) {
      const int64_t tk = k_base_tok + j;
      const int64_t kb = (packed ? 0 : (int64_t)b) * p.k_stride[0] + tk * p.k_stride[1] + (int64_t)hk * p.k_stride[2];
      float dot = 0.f;
      for (int d = 0; d < dq; ++d) dot = fmaf(q_sh[warp][d], load_qk(p.k, kb + d, fp8), dot);
      if (dr) {
        const int64_t rb = (packed ? 0 : (int64_t)b) * p.k_rope_stride[0] + tk * p.k_rope_stride[1];
        const __nv_bfloat16* kr = static_cast<const __nv_bfloat16*>(p.k_rope);
        for (int d = 0; d < dr; ++d) dot = fmaf(q_sh[warp][dq + d], __bfloat162float(kr[rb + d]), dot);
      }
      float ks = 1.f;
      if (fp8) ks = packed ? p.k_scale[(int64_t)hk * p.total_k + tk]
                           : p.k_scale[((int64_t)b * p.num_heads_kv + hk) * p.seqlen_k + j];
      s = dot * scale * ks;
    }
    float cmax = s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
    const float m_new = fmaxf(m, cmax);
    const float alpha = expf(m - m_new);          // 0 on the first chunk (m = -inf)
    const float pj = (j < kv_end) ? expf(s - m_new) : 0.f;
    float psum = pj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
    l = l * alpha + psum;
#pragma unroll
    for (int c = 0; c < kMaxD / 32; ++c) acc[c] *= alpha;
    const int nj = min(32, kv_end - j0);
    for (int jj = 0; jj < nj; ++jj) {
      const float w = __shfl_sync(0xffffffffu, pj, jj);
      const int64_t tk = k_base_tok + j0 + jj;
      if (v_fp8) {
        // depth-major e4m3 V: [B, Hkv, Dv, Sk], keys contiguous
        const int64_t vb = (int64_t)b * p.v_stride[0] + (int64_t)hk * p.v_stride[2] + tk;
#pragma unroll
        for (int c = 0; c < kMaxD / 32; ++c) {
          const int d = c * 32 + lane;
          if (d < dv) acc[c] = fmaf(w, load_qk(p.v, vb + (int64_t)d * p.v_stride[1], 1), acc[c]);
        }
      } else {
        const int64_t vb =
            (packed ? 0 : (int64_t)b) * p.v_stride[0] + tk * p.v_stride[1] + (int64_t)hk * p.v_stride[2];
        const __nv_bfloat16* vv = static_cast<const __nv_bfloat16*>(p.v);
#pragma unroll
        for (int c = 0; c < kMaxD / 32; ++c) {
          const int d = c * 32 + lane;
          if (d < dv) acc[c] = fmaf(w, __bfloat162float(vv[vb + d]), acc[c]);
        }
      }
    }
    m = m_new;
  }

  const float inv_l = l > 0.f ? 1.f / l : 0.f;
  const int64_t ob = (packed ? 0 : (int64_t)b) * p.o_stride[0] + tq * p.o_stride[1] + (int64_t)h * p.o_stride[2];
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o);
#pragma unroll
  for (int c = 0; c < kMaxD / 32; ++c) {
    const int d = c * 32 + lane;
    if (d < dv) o[ob + d] = __float2bfloat16_rn(acc[c] * inv_l);
  }
  if (p.lse != nullptr && lane == 0) {
    const float lse = l > 0.f ? m + logf(l) : -INFINITY;
    if (packed) p.lse[(int64_t)h * p.total_q + tq] = lse;
    else p.lse[((int64_t)b * p.num_heads_q + h) * p.seqlen_q + i] = lse;
  }
}

}  // namespace

cudaError_t simple_launch(const attn_fwd_params& p, cudaStream_t stream) {
  if (p.head_dim_qk + p.rope_depth > kMaxD || p.head_dim_v > kMaxD) return cudaErrorInvalidValue;
  dim3 grid((p.seqlen_q + kWarps - 1) / kWarps, p.num_heads_q, p.batch);
  if (grid.x == 0 || grid.z == 0) return cudaSuccess;
  simple_attn_kernel<<<grid, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace af
