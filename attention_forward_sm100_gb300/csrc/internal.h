// Declarations shared by the host API and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/attn_fwd.h"

namespace af {

constexpr int kRowsPerTile = 256;   // query rows per work tile of the tcgen05 kernel (one CTA)
constexpr int kRowsPerTilePair = 512;   // the same for a CTA pair (two M = 256 MMA tiles)
constexpr int kBlockM = 128;        // query rows per MMA tile (one TMEM lane per row)
constexpr int kBlockN = 128;        // keys per K/V tile
constexpr int64_t kL2ChunkBudget = 48ll << 20;   // K/V bytes one scheduling chunk may keep in L2
constexpr int64_t kL2ChunkBudgetFp8 = 24ll << 20;   // the same for fp8 Q/K (measured best)
constexpr int kMaxSplits = 64;      // split-KV ranges per query tile (the merge kernel holds 2 per lane)

// Workspace words (uint32 each).
enum WorkspaceWord : int {
  kWsTileCounter = 0,   // next dynamic work index minus gridDim.x
  kWsDoneCounter = 1,   // CTAs finished (the last one resets both counters)
  kWsErrorCode = 2,     // 0 or a device error code
  kWsErrorInfo = 3,     // block, role and barrier of the first error
  kWsWords = 4
};

// Device error codes recorded in kWsErrorCode.
enum DeviceError : uint32_t {
  kDevErrNone = 0,
  kDevErrTimeout = 1,
  kDevErrBadSeqlens = 3,   // packed offsets out of order or past total_q / total_k (info: sequence)
};

// Everything the tcgen05 kernel needs, passed as one __grid_constant__ struct.
struct Tc05Params {
  CUtensorMap tm_q;        // Q (nope part): box {64 or 128 elements, 1, 128, 1}
  CUtensorMap tm_k;        // K (nope part)
  CUtensorMap tm_v;        // V: box {64, 1, 128, 1}
  CUtensorMap tm_qr;       // Q rope part (rope only)
  CUtensorMap tm_kr;       // K rope part (rope only): box {64, 1, 128, 1}
  const float* q_scale;    // fp8 only
  const float* k_scale;
  const int32_t* cu_q;     // packed only
  const int32_t* cu_k;
  const int32_t* cu_v;     // packed e4m3 V only: key starts of the sequences along V's key dimension
  int32_t total_v;         // packed e4m3 V: length of V's key dimension
  uint16_t* o;             // output rows (bf16 bits)
  float* lse;
  uint32_t* ws;            // workspace words
  int64_t o_stride_b, o_stride_t, o_stride_h;  // elements
  int32_t o_store32;       // 1: o and every row stride are 32-byte aligned (256-bit row stores)
  int32_t batch, seqlen_q, seqlen_k, heads_q, heads_kv, group;
  int32_t tiles_per_seq;   // fixed length: ceil(Sq / rows_per_tile)
  int32_t rows_per_tile;   // query rows per work tile (kRowsPerTile, or kRowsPerTilePair for CTA pairs)
  int32_t kv_chunk;        // KV heads per scheduling chunk
  int64_t total_work;      // fixed length: exact number of work tiles
  int32_t packed;
  int32_t total_q;         // packed: rows of q (LSE and q_scale layout [Hq, Tq])
  int32_t total_k;         // packed: rows of k (k_scale layout [Hkv, Tk])
  float scale_log2;        // softmax_scale * log2(e)
  uint64_t timeout_ns;     // limit of every device wait
  int32_t withhold_v;      // testing: block 0 skips its first V tile load
  int32_t schedule;        // attn_schedule: how the producer advances to its next work index
  int32_t dependent_launch; // host only: launch as a programmatic dependent of the previous kernel
  int32_t num_splits;      // key ranges per query tile (1: no split-KV)
  int32_t kv_tiles;        // split-KV: ceil(seqlen_k / kBlockN)
  float* lse_part;         // split-KV: partial LSE [splits][B][Hq][Sq] / [splits][Hq][Tq]
  float* o_part;           // split-KV: partial O (normalised, fp32) [splits][rows][Hq][Dv]
};

// Arguments of the split-KV merge kernel.
struct SplitCombineParams {
  const float* lse_part;   // [splits][B][Hq][Sq], packed [splits][Hq][Tq]
  const float* o_part;     // [splits][rows][Hq][Dv], rows = B*Sq or Tq
  uint16_t* o;             // bf16 output rows
  float* lse;              // [B][Hq][Sq] / [Hq][Tq], or NULL
  int32_t splits, batch, seqlen_q, heads_q;
  int32_t packed, total_q;
  int64_t o_stride_b, o_stride_t, o_stride_h;   // elements
};

// Kernel variants of the tcgen05 path.
enum Tc05Variant : int {
  kVarD64 = 0,        // bf16, Dqk = Dv = 64
  kVarD128 = 1,       // bf16, Dqk = Dv = 128
  kVarD128Rope64 = 2, // bf16, Dqk = 128 + rope 64, Dv = 128
  kVarFp8D128 = 3,    // fp8 e4m3 Q/K, Dqk = Dv = 128
  kVarFp8QkvD128 = 4, // fp8 e4m3 Q/K/V (depth-major V, P rounded to e4m3), Dqk = Dv = 128
  kVarD128Pair = 5,   // kVarD128 on CTA pairs (M = 256 MMAs over two CTAs)
  kVarD128Rope64Pair = 6, // kVarD128Rope64 on CTA pairs
  kVarCount = 7
};

struct Tc05Config {
  int smem_bytes;
  int k_stages;
  int v_stages;
  int threads;
  int tmem_cols;
};

// Records the calling thread's last-error text (attn_fwd_last_error) and
// returns `st`.
attn_status report_error(attn_status st, const char* fmt, ...);

// Static configuration of a variant (host).
Tc05Config tc05_config(int variant);
// Flavours of the tcgen05 kernel, two bits: causal mask (1) and split-KV
// (2), so that a kernel carries only the code its calls run (the split
// partial stores, for one, are compiled out of the unsplit flavours). Pair
// variants have no causal split flavour.
enum Tc05Mask : int { kMaskNone = 0, kMaskCausal = 1, kMaskNoneSplit = 2, kMaskCausalSplit = 3 };
// Launch of one variant (defined in the per-variant translation units); a
// pair variant's grid counts CTAs and must be even.
cudaError_t tc05_launch(int variant, int mask, const Tc05Params& prm, int grid, cudaStream_t stream);
// Pair variants: clusters of two CTAs that fit on the current device at once
// (0 when unknown).
int tc05_max_clusters(int variant);
inline bool tc05_is_pair(int variant) { return variant == kVarD128Pair || variant == kVarD128Rope64Pair; }
// Launch of the split-KV merge kernel (head_dim_v 64 or 128).
cudaError_t splitkv_combine_launch(const SplitCombineParams& p, int head_dim_v, cudaStream_t stream);
// Launch of the plain CUDA-core kernel.
cudaError_t simple_launch(const attn_fwd_params& p, cudaStream_t stream);

}  // namespace af
