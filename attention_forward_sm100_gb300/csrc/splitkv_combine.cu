// Merge of split-KV partial results (the LSE-combine pass that the
// "splitk_partitions" field of the SM100AttentionSMem page's configuration
// calls for).
//
// With the keys of one query tile cut into S ranges, range s leaves for each
// (row, head) its softmax-normalised partial output O_s and the natural-log
// sum of exponentials L_s of its own scores. The exact result over all keys
// follows from the identity
//     L = log sum_s exp(L_s),    O = sum_s exp(L_s - L) * O_s,
// which this kernel evaluates with the maximum of the L_s subtracted first
// so that no exponential overflows. One warp merges one (row, head): lane k
// holds the weights of ranges k and k + 32, and each lane accumulates
// Dv / 32 consecutive output columns, so every partial row is read once,
// coalesced (streaming loads: nothing reads it again), and O is rounded to
// bf16 once.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace af {
namespace {

constexpr int kCombineWarps = 8;

// kBatch: partial rows each lane loads before accumulating (4 for up to four
// ranges, so that fewer registers leave room for more warps; 8 otherwise)
template <int DV, int kBatch>
__global__ void __launch_bounds__(kCombineWarps * 32) splitkv_combine_kernel(const SplitCombineParams p) {
  constexpr int C = DV / 32;   // output columns per lane
  // Launched as a programmatic dependent of the attention kernel: wait until
  // that grid has completed and its partial results are visible.
  ptx::grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  // (query row, head) pairs, head fastest; query rows are (b, i) or packed t
  const int64_t row = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  const int64_t qrows = p.packed ? (int64_t)p.total_q : (int64_t)p.batch * p.seqlen_q;
  const int64_t rows = qrows * p.heads_q;
  if (row >= rows) return;
  const int h = (int)(row % p.heads_q);
  const int64_t t = row / p.heads_q;
  // Partial LSE: S copies of the LSE layout ([B][Hq][Sq] or [Hq][Tq]);
  // partial O: [S][rows][Hq][Dv].
  int64_t lse_row, o_off;
  if (p.packed) {
    lse_row = (int64_t)h * p.total_q + t;
    o_off = t * p.o_stride_t + (int64_t)h * p.o_stride_h;
  } else {
    const int i = (int)(t % p.seqlen_q);
    const int b = (int)(t / p.seqlen_q);
    lse_row = ((int64_t)b * p.heads_q + h) * p.seqlen_q + i;
    o_off = (int64_t)b * p.o_stride_b + (int64_t)i * p.o_stride_t + (int64_t)h * p.o_stride_h;
  }
  const int64_t lse_split = qrows * p.heads_q;
  const int64_t o_split = rows * DV;
  const float* src = p.o_part + row * DV + C * lane;
  // Ranges in batches of kBatch: a batch's loads are all issued before any
  // is used, and the first batch is issued before the weights are worked
  // out (the partial rows do not depend on them), so each warp keeps its
  // row reads in flight across the LSE reduction.
  float v[kBatch][C];
  auto load_batch = [&](int s0) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (s0 + u < p.splits) {
        const float* x = src + (int64_t)(s0 + u) * o_split;
        if constexpr (C == 4) {
          const float4 t4 = __ldcs(reinterpret_cast<const float4*>(x));
          v[u][0] = t4.x; v[u][1] = t4.y; v[u][2] = t4.z; v[u][3] = t4.w;
        } else {
          const float2 t2 = __ldcs(reinterpret_cast<const float2*>(x));
          v[u][0] = t2.x; v[u][1] = t2.y;
        }
      }
    }
  };
  load_batch(0);
  float l0 = -INFINITY, l1 = -INFINITY;
  if (lane < p.splits) l0 = p.lse_part[lane * lse_split + lse_row];
  if (lane + 32 < p.splits) l1 = p.lse_part[(lane + 32) * lse_split + lse_row];
  float mx = fmaxf(l0, l1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + o_off;
  if (mx == -INFINITY) {   // no key reached this row in any range
    for (int c = 0; c < C; ++c) orow[C * lane + c] = __float2bfloat16(0.f);
    if (p.lse != nullptr && lane == 0) p.lse[lse_row] = -INFINITY;
    return;
  }
  float w0 = expf(l0 - mx), w1 = expf(l1 - mx);
  float sum = w0 + w1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = 1.f / sum;
  w0 *= inv;
  w1 *= inv;
  float acc[C];
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = 0.f;
  for (int s0 = 0; s0 < p.splits; s0 += kBatch) {
    if (s0 > 0) load_batch(s0);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int s = s0 + u;
      const float w = __shfl_sync(0xffffffffu, s < 32 ? w0 : w1, s & 31);
      if (s < p.splits) {
#pragma unroll
        for (int c = 0; c < C; ++c) acc[c] = fmaf(w, v[u][c], acc[c]);
      }
    }
  }
  if constexpr (C == 4) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0], acc[1]), hi = __floats2bfloat162_rn(acc[2], acc[3]);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(orow + C * lane) = pk;
  } else {
    *reinterpret_cast<__nv_bfloat162*>(orow + C * lane) = __floats2bfloat162_rn(acc[0], acc[1]);
  }
  if (p.lse != nullptr && lane == 0) p.lse[lse_row] = mx + logf(sum);
}

}  // namespace

cudaError_t splitkv_combine_launch(const SplitCombineParams& p, int head_dim_v, cudaStream_t stream) {
  const int64_t rows = (p.packed ? (int64_t)p.total_q : (int64_t)p.batch * p.seqlen_q) * p.heads_q;
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + kCombineWarps - 1) / kCombineWarps;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  const bool few = p.splits <= 4;
  void (*kern)(const SplitCombineParams) = nullptr;
  if (head_dim_v == 128)
    kern = few ? splitkv_combine_kernel<128, 4> : splitkv_combine_kernel<128, 8>;
  else if (head_dim_v == 64)
    kern = few ? splitkv_combine_kernel<64, 4> : splitkv_combine_kernel<64, 8>;
  else
    return cudaErrorInvalidValue;
  // Programmatic dependent launch: the merge's blocks may start while the
  // attention kernel's last CTAs finish (each waits at griddepcontrol.wait).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kCombineWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace af
