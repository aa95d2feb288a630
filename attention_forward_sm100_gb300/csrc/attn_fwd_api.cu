// Host side of the C ABI declared in include/attn_fwd.h: argument validation,
// launch planning (grid, split-KV count, workspace layout), TMA descriptor
// encoding and kernel dispatch (the attention kernel, then the split-KV
// merge when the keys are split).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "schedule.cuh"

namespace {

thread_local char g_last_error[512] = {0};

attn_status fail(attn_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() { g_last_error[0] = 0; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int qk_elem_bytes(const attn_fwd_params* p) { return p->qk_dtype == ATTN_DTYPE_FP8_E4M3 ? 1 : 2; }

// ---------------------------------------------------------------- validation
attn_status validate(const attn_fwd_params* p) {
  if (p == nullptr) return fail(ATTN_ERR_INVALID_ARG, "params is NULL");
  if (p->qk_dtype != ATTN_DTYPE_BF16 && p->qk_dtype != ATTN_DTYPE_FP8_E4M3)
    return fail(ATTN_ERR_INVALID_ARG, "unknown qk_dtype %d", p->qk_dtype);
  if (p->v_dtype != ATTN_DTYPE_BF16 && p->v_dtype != ATTN_DTYPE_FP8_E4M3)
    return fail(ATTN_ERR_INVALID_ARG, "unknown v_dtype %d", p->v_dtype);
  if (p->backend != ATTN_BACKEND_TCGEN05 && p->backend != ATTN_BACKEND_SIMPLE)
    return fail(ATTN_ERR_INVALID_ARG, "unknown backend %d", p->backend);
  if (p->fault_injection != 0 && p->fault_injection != 1)
    return fail(ATTN_ERR_INVALID_ARG, "unknown fault_injection %d", p->fault_injection);
  if (p->schedule != ATTN_SCHEDULE_DYNAMIC && p->schedule != ATTN_SCHEDULE_STATIC &&
      p->schedule != ATTN_SCHEDULE_GRID)
    return fail(ATTN_ERR_INVALID_ARG, "unknown schedule %d", p->schedule);
  if (p->pair_cta != ATTN_PAIR_AUTO && p->pair_cta != ATTN_PAIR_OFF && p->pair_cta != ATTN_PAIR_ON)
    return fail(ATTN_ERR_INVALID_ARG, "unknown pair_cta %d", p->pair_cta);
  if (p->pair_cta == ATTN_PAIR_ON) {
    if (p->backend != ATTN_BACKEND_TCGEN05) return fail(ATTN_ERR_UNSUPPORTED, "CTA pairs run on the tcgen05 backend only");
    if (p->qk_dtype != ATTN_DTYPE_BF16 || p->v_dtype != ATTN_DTYPE_BF16 || p->head_dim_qk != 128 ||
        p->head_dim_v != 128 || (p->rope_depth != 0 && p->rope_depth != 64))
      return fail(ATTN_ERR_UNSUPPORTED, "CTA pairs support bf16 Q/K/V with Dqk = Dv = 128 and rope 0 or 64");
    if (p->fault_injection != 0) return fail(ATTN_ERR_UNSUPPORTED, "fault injection is not available with CTA pairs");
  }
  if (p->num_splits < 0 || p->num_splits > af::kMaxSplits)
    return fail(ATTN_ERR_INVALID_ARG, "num_splits %d outside [0, %d]", p->num_splits, af::kMaxSplits);
  if (p->num_splits >= 2) {
    if (p->backend != ATTN_BACKEND_TCGEN05)
      return fail(ATTN_ERR_UNSUPPORTED, "split-KV runs on the tcgen05 backend only");
    if (p->causal && p->pair_cta == ATTN_PAIR_ON)
      return fail(ATTN_ERR_UNSUPPORTED, "causal split-KV is not supported with CTA pairs");
  }
  if (p->batch < 0 || p->seqlen_q < 0 || p->seqlen_k < 0 || p->total_q < 0 || p->total_k < 0)
    return fail(ATTN_ERR_INVALID_ARG, "negative size");
  if (p->num_heads_q <= 0 || p->num_heads_kv <= 0)
    return fail(ATTN_ERR_INVALID_ARG, "head counts must be positive");
  if (p->num_heads_q % p->num_heads_kv != 0)
    return fail(ATTN_ERR_INVALID_ARG, "num_heads_q %d is not a multiple of num_heads_kv %d",
                p->num_heads_q, p->num_heads_kv);
  if (p->head_dim_qk <= 0 || p->head_dim_v <= 0 || p->rope_depth < 0)
    return fail(ATTN_ERR_INVALID_ARG, "head dims must be positive");
  if (!(p->softmax_scale > 0.f) || p->softmax_scale != p->softmax_scale)
    return fail(ATTN_ERR_INVALID_ARG, "softmax_scale must be a positive number");
  const bool packed = p->cu_seqlens_q != nullptr;
  // K, V and the K rope part may be NULL only when there are no keys at all
  // (an empty tensor has no storage); O is then 0 and LSE -inf.
  const bool no_keys = packed ? p->total_k == 0 : p->seqlen_k == 0;
  // Likewise Q and O without query rows (nothing is launched).
  const bool no_queries = p->batch == 0 || (packed ? p->total_q == 0 : p->seqlen_q == 0);
  if (packed != (p->cu_seqlens_k != nullptr))
    return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k must both be set or both NULL");
  if (packed && ((reinterpret_cast<uintptr_t>(p->cu_seqlens_q) | reinterpret_cast<uintptr_t>(p->cu_seqlens_k)) & 3))
    return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens must be 4-byte aligned");
  if (packed && (p->total_q <= 0 && p->batch > 0 && p->seqlen_q > 0))
    return fail(ATTN_ERR_INVALID_ARG, "packed layout needs total_q");
  if ((!no_queries && (p->q == nullptr || p->o == nullptr)) ||
      (!no_keys && !no_queries && (p->k == nullptr || p->v == nullptr)))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
  if (p->rope_depth > 0 && !no_queries && (p->q_rope == nullptr || (!no_keys && p->k_rope == nullptr)))
    return fail(ATTN_ERR_INVALID_ARG, "rope_depth > 0 needs q_rope and k_rope");
  if (p->qk_dtype == ATTN_DTYPE_FP8_E4M3) {
    if ((!no_queries && p->q_scale == nullptr) || (!no_keys && !no_queries && p->k_scale == nullptr))
      return fail(ATTN_ERR_INVALID_ARG, "fp8 Q/K need q_scale and k_scale");
    if (p->rope_depth > 0) return fail(ATTN_ERR_UNSUPPORTED, "fp8 Q/K with a rope part");
  }
  if (p->v_dtype == ATTN_DTYPE_FP8_E4M3) {
    if (p->qk_dtype != ATTN_DTYPE_FP8_E4M3) return fail(ATTN_ERR_UNSUPPORTED, "fp8 V needs fp8 Q/K");
    if (packed && !no_keys && !no_queries &&
        (p->cu_seqlens_v == nullptr || (reinterpret_cast<uintptr_t>(p->cu_seqlens_v) & 3) || p->total_v <= 0))
      return fail(ATTN_ERR_INVALID_ARG, "packed fp8 V needs cu_seqlens_v (4-byte aligned) and total_v");
    if (p->head_dim_qk != 128 || p->head_dim_v != 128)
      return fail(ATTN_ERR_UNSUPPORTED, "fp8 V supports Dqk = Dv = 128 only");
    if (p->v_stride[1] % 16)
      return fail(ATTN_ERR_INVALID_ARG, "fp8 V: the depth-row stride must be a multiple of 16 bytes");
  }
  for (int i = 0; i < 3; ++i) {
    if (p->q_stride[i] < 0 || p->k_stride[i] < 0 || p->v_stride[i] < 0 || p->o_stride[i] < 0 ||
        p->q_rope_stride[i] < 0 || (i < 2 && p->k_rope_stride[i] < 0))
      return fail(ATTN_ERR_INVALID_ARG, "negative stride");
  }
  if (p->backend == ATTN_BACKEND_TCGEN05) {
    const size_t need = attn_fwd_workspace_bytes(p);
    if (p->workspace == nullptr || p->workspace_bytes < need)
      return fail(ATTN_ERR_INVALID_ARG, "workspace of at least %zu bytes is required", need);
    if (reinterpret_cast<uintptr_t>(p->workspace) & 255u)
      return fail(ATTN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    // TMA: 16-byte aligned bases and strides that are multiples of 16 bytes.
    const int es = qk_elem_bytes(p);
    if (!aligned16(p->q) || !aligned16(p->k) || !aligned16(p->v))
      return fail(ATTN_ERR_INVALID_ARG, "q, k, v must be 16-byte aligned");
    const int ves = p->v_dtype == ATTN_DTYPE_FP8_E4M3 ? 1 : 2;
    for (int i = packed ? 1 : 0; i < 3; ++i) {
      if ((p->q_stride[i] * es) % 16 || (p->k_stride[i] * es) % 16 || (p->v_stride[i] * ves) % 16)
        return fail(ATTN_ERR_INVALID_ARG, "q/k/v strides must be multiples of 16 bytes");
    }
    if (p->rope_depth > 0) {
      if (!aligned16(p->q_rope) || !aligned16(p->k_rope))
        return fail(ATTN_ERR_INVALID_ARG, "q_rope, k_rope must be 16-byte aligned");
      for (int i = packed ? 1 : 0; i < 3; ++i)
        if ((p->q_rope_stride[i] * 2) % 16) return fail(ATTN_ERR_INVALID_ARG, "q_rope strides must be multiples of 16 bytes");
      for (int i = packed ? 1 : 0; i < 2; ++i)
        if ((p->k_rope_stride[i] * 2) % 16) return fail(ATTN_ERR_INVALID_ARG, "k_rope strides must be multiples of 16 bytes");
    }
    // The epilogue stores whole rows in 16-byte pieces, so every stride that
    // moves between rows (batch too, unless packed) must keep that alignment.
    if ((p->o_stride[2] * 2) % 16 || (p->o_stride[1] * 2) % 16 || (!packed && (p->o_stride[0] * 2) % 16) ||
        !aligned16(p->o))
      return fail(ATTN_ERR_INVALID_ARG, "o must be 16-byte aligned with 16-byte multiple strides");
    const bool ok_bf16 = p->qk_dtype == ATTN_DTYPE_BF16 &&
        ((p->head_dim_qk == 64 && p->head_dim_v == 64 && p->rope_depth == 0) ||
         (p->head_dim_qk == 128 && p->head_dim_v == 128 && (p->rope_depth == 0 || p->rope_depth == 64)));
    const bool ok_fp8 = p->qk_dtype == ATTN_DTYPE_FP8_E4M3 && p->head_dim_qk == 128 &&
                        p->head_dim_v == 128 && p->rope_depth == 0;
    if (!ok_bf16 && !ok_fp8)
      return fail(ATTN_ERR_UNSUPPORTED, "tcgen05 kernel supports (Dqk,Dv,R) = (64,64,0), (128,128,0), "
                  "(128,128,64) for bf16 and (128,128,0) for fp8; got (%d,%d,%d)",
                  p->head_dim_qk, p->head_dim_v, p->rope_depth);
  } else {
    if (p->head_dim_qk + p->rope_depth > 256 || p->head_dim_v > 256)
      return fail(ATTN_ERR_UNSUPPORTED, "simple kernel supports Dqk + R <= 256 and Dv <= 256");
  }
  return ATTN_OK;
}

// CTA pairs for this call (pair_cta after validation; the automatic choice
// keeps one CTA per MMA tile).
bool use_pair(const attn_fwd_params* p) { return p->pair_cta == ATTN_PAIR_ON; }

int tc05_variant(const attn_fwd_params* p) {
  if (p->qk_dtype == ATTN_DTYPE_FP8_E4M3)
    return p->v_dtype == ATTN_DTYPE_FP8_E4M3 ? af::kVarFp8QkvD128 : af::kVarFp8D128;
  if (p->head_dim_qk == 64) return af::kVarD64;
  if (use_pair(p)) return p->rope_depth ? af::kVarD128Rope64Pair : af::kVarD128Pair;
  return p->rope_depth ? af::kVarD128Rope64 : af::kVarD128;
}

// Query rows of one work tile.
int32_t rows_for(const attn_fwd_params* p) { return use_pair(p) ? af::kRowsPerTilePair : af::kRowsPerTile; }

int sm_count_cached() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 148;
  }
  if (dev < 0 || dev >= 64) return 148;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
    cudaGetLastError();
    return 148;
  }
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

// Clusters of two CTAs resident at once for a pair variant (cached per
// device; half the SMs when the query is not possible).
int max_clusters_cached(int variant) {
  static std::atomic<int> cache[64][2];
  const int slot = variant == af::kVarD128Rope64Pair ? 1 : 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return sm_count_cached() / 2;
  }
  if (dev < 0 || dev >= 64) return sm_count_cached() / 2;
  int v = cache[dev][slot].load(std::memory_order_relaxed);
  if (v > 0) return v;
  v = af::tc05_max_clusters(variant);
  if (v <= 0) return sm_count_cached() / 2;
  cache[dev][slot].store(v, std::memory_order_relaxed);
  return v;
}

// Persistent work units of the launch: CTAs, or clusters for CTA pairs.
int persistent_units(const attn_fwd_params* p) {
  return use_pair(p) ? max_clusters_cached(tc05_variant(p)) : sm_count_cached();
}

int32_t kv_chunk_for(const attn_fwd_params* p) {
  const int64_t row = (int64_t)(p->head_dim_qk * qk_elem_bytes(p)) + 2ll * p->rope_depth +
                      (p->v_dtype == ATTN_DTYPE_FP8_E4M3 ? 1ll : 2ll) * p->head_dim_v;
  // Measured on GB300: 48 MB suits bf16 (MLA loses ~2 % at 24 or 96 MB),
  // 24 MB suits fp8 Q/K (~1 % over 48 MB).
  const int64_t budget = p->qk_dtype == ATTN_DTYPE_FP8_E4M3 ? af::kL2ChunkBudgetFp8 : af::kL2ChunkBudget;
  return af::choose_kv_chunk(p->seqlen_k, row, p->num_heads_kv, budget);
}

int64_t work_tiles_bound(const attn_fwd_params* p) {
  const int64_t T = af::tiles_for(p->seqlen_q, rows_for(p));
  return (int64_t)p->batch * p->num_heads_q * T;
}

// Key ranges per query tile for `p` (1 = no split-KV). Explicit counts are
// capped at the number of key tiles (of the longest sequence when packed);
// 0 asks for the scheduler's choice (for packed sequences from the longest
// lengths and the upper bound of the query tiles, B * ceil(max_len / rows)).
// Causal problems on CTA pairs do not split.
int32_t resolve_splits(const attn_fwd_params* p) {
  if (p == nullptr || p->num_splits == 1 || p->num_splits < 0 || p->num_splits > af::kMaxSplits ||
      p->backend != ATTN_BACKEND_TCGEN05 || (p->causal && use_pair(p)) || p->batch <= 0 || p->seqlen_q <= 0 ||
      p->seqlen_k <= 0 || p->num_heads_q <= 0 || (p->cu_seqlens_q != nullptr && p->total_q <= 0))
    return 1;
  const int32_t kv_tiles = af::tiles_for(p->seqlen_k, af::kBlockN);
  if (p->num_splits >= 2) return p->num_splits < kv_tiles ? p->num_splits : kv_tiles;
  if (p->causal)
    return af::choose_splits_causal((int64_t)p->batch * p->num_heads_q, p->seqlen_q, p->seqlen_k, rows_for(p),
                                    af::kBlockM, af::kBlockN, p->head_dim_v, persistent_units(p), af::kMaxSplits);
  return af::choose_splits(work_tiles_bound(p), kv_tiles, persistent_units(p), af::kMaxSplits);
}

size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }

// CTAs launched for `work` work tiles: one per SM for the persistent
// schedules, one per work tile otherwise; CTA pairs launch two CTAs per
// cluster and one cluster per resident cluster slot (or per work tile).
int64_t grid_for(const attn_fwd_params* p, int64_t work) {
  const int64_t per_unit = use_pair(p) ? 2 : 1;
  if (p->schedule == ATTN_SCHEDULE_GRID) return per_unit * work;
  const int64_t units = persistent_units(p);
  return per_unit * (work < units ? work : units);
}

// Split-KV partial results in the workspace, after the 256 bytes of counters:
// per range one copy of the LSE layout and one fp32 O row per query row.
size_t partial_query_rows(const attn_fwd_params* p) {
  return p->cu_seqlens_q != nullptr ? (size_t)p->total_q : (size_t)p->batch * p->seqlen_q;
}
size_t lse_part_bytes(const attn_fwd_params* p, int32_t splits) {
  return round256((size_t)splits * partial_query_rows(p) * p->num_heads_q * sizeof(float));
}
size_t o_part_bytes(const attn_fwd_params* p, int32_t splits) {
  return (size_t)splits * partial_query_rows(p) * p->num_heads_q * p->head_dim_v * sizeof(float);
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

// Encoded 4-D maps of the calling thread's recent calls, so a call that
// repeats another one's tensors (a serving loop, a benchmark) skips the
// driver's encoder. The key holds every encoder argument; a map depends on
// nothing else, so a hit is exact.
struct MapKey {
  const void* base;
  int dt;
  cuuint64_t dims[4];
  cuuint64_t strides[3];
  cuuint32_t box[4];
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool used;
};
constexpr int kMapCacheEntries = 16;
thread_local MapEntry g_map_cache[kMapCacheEntries];
thread_local int g_map_cache_next = 0;

CUresult encode_4d_cached(EncodeTiledFn fn, CUtensorMap* map, CUtensorMapDataType dt, const void* base,
                          const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
  MapKey key;
  memset(&key, 0, sizeof(key));
  key.base = base;
  key.dt = (int)dt;
  memcpy(key.dims, dims, sizeof(key.dims));
  memcpy(key.strides, strides, sizeof(key.strides));
  memcpy(key.box, box, sizeof(key.box));
  for (int i = 0; i < kMapCacheEntries; ++i) {
    if (g_map_cache[i].used && memcmp(&g_map_cache[i].key, &key, sizeof(key)) == 0) {
      *map = g_map_cache[i].map;
      return CUDA_SUCCESS;
    }
  }
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = fn(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) {
    MapEntry& e = g_map_cache[g_map_cache_next];
    g_map_cache_next = (g_map_cache_next + 1) % kMapCacheEntries;
    e.key = key;
    e.map = *map;
    e.used = true;
  }
  return r;
}

// 4-D map over (depth, head, token, batch); box {box_d, 1, box_rows, 1}, 128-byte swizzle.
attn_status make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int es, int64_t depth,
                     int64_t heads, int64_t tokens, int64_t batches, int64_t sh, int64_t st, int64_t sb,
                     int box_d, int box_rows = af::kBlockN) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  if (heads <= 1) sh = st > 0 ? st : depth;   // a size-1 dimension: any legal stride
  if (batches <= 1) sb = st * (tokens > 0 ? tokens : 1);
  if (tokens < 1) tokens = 1;
  cuuint64_t dims[4] = {(cuuint64_t)depth, (cuuint64_t)heads, (cuuint64_t)tokens, (cuuint64_t)batches};
  cuuint64_t strides[3] = {(cuuint64_t)(sh * es), (cuuint64_t)(st * es), (cuuint64_t)(sb * es)};
  cuuint32_t box[4] = {(cuuint32_t)box_d, 1u, (cuuint32_t)box_rows, 1u};
  CUresult r = encode_4d_cached(fn, map, dt, base, dims, strides, box);
  if (r != CUDA_SUCCESS)
    return fail(ATTN_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d) for a %lldx%lldx%lldx%lld tensor", (int)r,
                (long long)depth, (long long)heads, (long long)tokens, (long long)batches);
  return ATTN_OK;
}

// Depth-major fp8 V, [B][Hkv][Dv][Sk] (packed: [Hkv][Dv][Tv]) with the keys
// contiguous: 4-D map over (key, depth, head, batch); box {128 keys, Dv rows,
// 1, 1}, 128-byte swizzle, so one box is the K-major B operand of the P.V
// product.
attn_status make_map_vt(CUtensorMap* map, const attn_fwd_params* p, const void* base) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  const bool packed = p->cu_seqlens_q != nullptr;
  const int64_t nb = packed ? 1 : p->batch;
  const int64_t keys = packed ? p->total_v : p->seqlen_k;
  const int64_t sk = keys > 0 ? keys : 1;
  const int64_t sd = p->v_stride[1];
  const int64_t sh = p->num_heads_kv > 1 ? p->v_stride[2] : sd * p->head_dim_v;
  const int64_t sb = nb > 1 ? p->v_stride[0] : sh * p->num_heads_kv;
  cuuint64_t dims[4] = {(cuuint64_t)sk, (cuuint64_t)p->head_dim_v, (cuuint64_t)p->num_heads_kv,
                        (cuuint64_t)nb};
  cuuint64_t strides[3] = {(cuuint64_t)sd, (cuuint64_t)sh, (cuuint64_t)sb};
  cuuint32_t box[4] = {(cuuint32_t)af::kBlockN, (cuuint32_t)p->head_dim_v, 1u, 1u};
  CUresult r = encode_4d_cached(fn, map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, dims, strides, box);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d) for fp8 V", (int)r);
  return ATTN_OK;
}

attn_status launch_tc05(const attn_fwd_params* p, cudaStream_t stream) {
  const bool packed = p->cu_seqlens_q != nullptr;
  const int variant = tc05_variant(p);
  af::Tc05Params prm;
  memset(&prm, 0, sizeof(prm));
  const bool fp8 = p->qk_dtype == ATTN_DTYPE_FP8_E4M3;
  const CUtensorMapDataType qk_t = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int es = fp8 ? 1 : 2;
  const int box_qk = fp8 ? 128 : 64;
  const int64_t tq = packed ? p->total_q : p->seqlen_q, tk = packed ? p->total_k : p->seqlen_k;
  const int64_t nb = packed ? 1 : p->batch;
  // A CTA pair loads half of each K tile per CTA: 64-row K boxes.
  const int k_rows = use_pair(p) ? af::kBlockN / 2 : af::kBlockN;
  attn_status st;
  if ((st = make_map(&prm.tm_q, p->q, qk_t, es, p->head_dim_qk, p->num_heads_q, tq, nb, p->q_stride[2],
                     p->q_stride[1], p->q_stride[0], box_qk)) != ATTN_OK)
    return st;
  // Without keys K and V are never read; their maps then point at Q.
  const void* k_base = p->k != nullptr ? p->k : p->q;
  const void* v_base = p->v != nullptr ? p->v : p->q;
  const void* kr_base = p->k_rope != nullptr ? p->k_rope : p->q_rope;
  if ((st = make_map(&prm.tm_k, k_base, qk_t, es, p->head_dim_qk, p->num_heads_kv, tk, nb, p->k_stride[2],
                     p->k_stride[1], p->k_stride[0], box_qk, k_rows)) != ATTN_OK)
    return st;
  if (p->v_dtype == ATTN_DTYPE_FP8_E4M3) {
    if ((st = make_map_vt(&prm.tm_v, p, v_base)) != ATTN_OK) return st;
  } else if ((st = make_map(&prm.tm_v, v_base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->head_dim_v, p->num_heads_kv,
                            tk, nb, p->v_stride[2], p->v_stride[1], p->v_stride[0], 64)) != ATTN_OK) {
    return st;
  }
  if (p->rope_depth > 0) {
    if ((st = make_map(&prm.tm_qr, p->q_rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->rope_depth, p->num_heads_q,
                       tq, nb, p->q_rope_stride[2], p->q_rope_stride[1], p->q_rope_stride[0], 64)) != ATTN_OK)
      return st;
    if ((st = make_map(&prm.tm_kr, kr_base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->rope_depth, 1, tk, nb,
                       p->k_rope_stride[1], p->k_rope_stride[1], p->k_rope_stride[0], 64, k_rows)) != ATTN_OK)
      return st;
  }
  prm.q_scale = p->q_scale;
  prm.k_scale = p->k_scale;
  prm.cu_q = p->cu_seqlens_q;
  prm.cu_k = p->cu_seqlens_k;
  prm.cu_v = (packed && p->v_dtype == ATTN_DTYPE_FP8_E4M3) ? p->cu_seqlens_v : nullptr;
  prm.total_v = prm.cu_v != nullptr ? p->total_v : 0;
  prm.o = static_cast<uint16_t*>(p->o);
  prm.lse = p->lse;
  prm.ws = static_cast<uint32_t*>(p->workspace);
  prm.o_stride_b = packed ? 0 : p->o_stride[0];
  prm.o_stride_t = p->o_stride[1];
  prm.o_stride_h = p->o_stride[2];
  prm.o_store32 = (reinterpret_cast<uintptr_t>(p->o) & 31u) == 0 && (p->o_stride[2] * 2) % 32 == 0 &&
                  (p->o_stride[1] * 2) % 32 == 0 && (packed || (p->o_stride[0] * 2) % 32 == 0);
  prm.batch = p->batch;
  prm.seqlen_q = p->seqlen_q;
  prm.seqlen_k = p->seqlen_k;
  prm.heads_q = p->num_heads_q;
  prm.heads_kv = p->num_heads_kv;
  prm.group = p->num_heads_q / p->num_heads_kv;
  prm.rows_per_tile = rows_for(p);
  prm.tiles_per_seq = af::tiles_for(p->seqlen_q, prm.rows_per_tile);
  prm.kv_chunk = kv_chunk_for(p);
  prm.total_work = packed ? 0 : work_tiles_bound(p);
  prm.packed = packed ? 1 : 0;
  prm.total_q = packed ? p->total_q : 0;
  prm.total_k = packed ? p->total_k : 0;
  prm.scale_log2 = p->softmax_scale * 1.4426950408889634f;
  prm.withhold_v = p->fault_injection == 1 ? 1 : 0;
  prm.timeout_ns = prm.withhold_v ? 200000000ull : 2000000000ull;
  const int32_t splits = resolve_splits(p);
  prm.num_splits = splits;
  prm.kv_tiles = af::tiles_for(p->seqlen_k, af::kBlockN);
  if (splits > 1) {
    uint8_t* ws = static_cast<uint8_t*>(p->workspace);
    prm.lse_part = reinterpret_cast<float*>(ws + ATTN_FWD_WORKSPACE_BYTES);
    prm.o_part = reinterpret_cast<float*>(ws + ATTN_FWD_WORKSPACE_BYTES + lse_part_bytes(p, splits));
    prm.total_work *= splits;
  }
  const int64_t bound = work_tiles_bound(p) * splits;
  if (bound <= 0) return ATTN_OK;
  if (grid_for(p, bound) > 0x7fffffffll) return fail(ATTN_ERR_UNSUPPORTED, "too many work tiles for one grid");
  const int grid = (int)grid_for(p, bound);
  prm.schedule = p->schedule;
  // Calls with fewer CTAs than SMs are dominated by launch latency: their
  // set-up overlaps the previous kernel (programmatic dependent launch; bf16
  // variants, which wait for that kernel before any global access). A full
  // grid gains nothing from it.
  prm.dependent_launch = (p->qk_dtype == ATTN_DTYPE_BF16 && grid < sm_count_cached()) ? 1 : 0;
  const int mask = (p->causal != 0 ? af::kMaskCausal : 0) | (splits > 1 ? af::kMaskNoneSplit : 0);
  cudaError_t e = af::tc05_launch(variant, mask, prm, grid, stream);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "tcgen05 kernel launch failed: %s", cudaGetErrorString(e));
  if (splits > 1) {
    af::SplitCombineParams cp;
    cp.lse_part = prm.lse_part;
    cp.o_part = prm.o_part;
    cp.o = prm.o;
    cp.lse = p->lse;
    cp.splits = splits;
    cp.batch = p->batch;
    cp.seqlen_q = p->seqlen_q;
    cp.heads_q = p->num_heads_q;
    cp.packed = packed ? 1 : 0;
    cp.total_q = packed ? p->total_q : 0;
    cp.o_stride_b = packed ? 0 : p->o_stride[0];
    cp.o_stride_t = p->o_stride[1];
    cp.o_stride_h = p->o_stride[2];
    e = af::splitkv_combine_launch(cp, p->head_dim_v, stream);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "split-KV merge launch failed: %s", cudaGetErrorString(e));
  }
  return ATTN_OK;
}

}  // namespace

attn_status af::report_error(attn_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

extern "C" {

void attn_fwd_params_init(attn_fwd_params* p) {
  if (p == nullptr) return;
  memset(p, 0, sizeof(*p));
  p->qk_dtype = ATTN_DTYPE_BF16;
  p->backend = ATTN_BACKEND_TCGEN05;
  p->softmax_scale = 1.f;
}

size_t attn_fwd_workspace_bytes(const attn_fwd_params* p) {
  const int32_t splits = resolve_splits(p);
  if (splits <= 1) return ATTN_FWD_WORKSPACE_BYTES;
  return ATTN_FWD_WORKSPACE_BYTES + lse_part_bytes(p, splits) + o_part_bytes(p, splits);
}

size_t attn_fwd_params_size(void) { return sizeof(attn_fwd_params); }

attn_status attn_fwd(const attn_fwd_params* p, attn_stream_t stream) {
  clear_error();
  attn_status st = validate(p);
  if (st != ATTN_OK) return st;
  if (p->batch == 0 || p->seqlen_q == 0) return ATTN_OK;
  if (p->cu_seqlens_q != nullptr && p->total_q == 0) return ATTN_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->backend == ATTN_BACKEND_SIMPLE) {
    cudaError_t e = af::simple_launch(*p, s);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "simple kernel launch failed: %s", cudaGetErrorString(e));
    return ATTN_OK;
  }
  return launch_tc05(p, s);
}

attn_status attn_fwd_check(void* workspace, attn_stream_t stream) {
  clear_error();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "stream error: %s", cudaGetErrorString(e));
  if (workspace == nullptr) return ATTN_OK;
  uint32_t w[af::kWsWords];
  e = cudaMemcpy(w, workspace, sizeof(w), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "reading the workspace failed: %s", cudaGetErrorString(e));
  if (w[af::kWsErrorCode] != af::kDevErrNone) {
    const uint32_t info = w[af::kWsErrorInfo];
    cudaMemset(static_cast<uint32_t*>(workspace) + af::kWsErrorCode, 0, 2 * sizeof(uint32_t));
    cudaDeviceSynchronize();
    if (w[af::kWsErrorCode] == af::kDevErrBadSeqlens)
      return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens of sequence %u are decreasing or exceed total_q / total_k "
                  "(nothing of that call's output can be trusted)", info);
    return fail(ATTN_ERR_DEVICE_TIMEOUT, "device wait timed out (code %u, block %u, role %u, barrier %u)",
                w[af::kWsErrorCode], info >> 16, (info >> 8) & 0xffu, info & 0xffu);
  }
  return ATTN_OK;
}

attn_status attn_fwd_plan(const attn_fwd_params* p, attn_fwd_plan_info* out) {
  clear_error();
  if (out == nullptr) return fail(ATTN_ERR_INVALID_ARG, "out is NULL");
  attn_status st = validate(p);
  if (st != ATTN_OK) return st;
  memset(out, 0, sizeof(*out));
  out->backend = p->backend;
  if (p->backend == ATTN_BACKEND_SIMPLE) {
    out->rows_per_tile = 4;
    out->work_tiles = (int64_t)((p->seqlen_q + 3) / 4) * p->num_heads_q * p->batch;
    out->grid = (int32_t)out->work_tiles;
    out->block = 128;
    out->num_splits = 1;
    out->pair_cta = ATTN_PAIR_OFF;
    return ATTN_OK;
  }
  const af::Tc05Config c = af::tc05_config(tc05_variant(p));
  out->rows_per_tile = rows_for(p);
  out->pair_cta = use_pair(p) ? ATTN_PAIR_ON : ATTN_PAIR_OFF;
  out->num_splits = resolve_splits(p);
  out->work_tiles = work_tiles_bound(p) * out->num_splits;
  const int64_t grid = grid_for(p, out->work_tiles);
  if (grid > 0x7fffffffll) return fail(ATTN_ERR_UNSUPPORTED, "too many work tiles for one grid");
  out->grid = (int32_t)grid;
  out->block = c.threads;
  out->smem_bytes = c.smem_bytes;
  out->k_stages = c.k_stages;
  out->v_stages = c.v_stages;
  out->tmem_columns = c.tmem_cols;
  return ATTN_OK;
}

int64_t attn_fwd_schedule(const attn_fwd_params* p, const int32_t* host_cu_seqlens_q, attn_work_tile* out,
                          int64_t cap) {
  clear_error();
  if (p == nullptr || p->num_heads_kv <= 0 || p->num_heads_q % p->num_heads_kv) return -1;
  const int group = p->num_heads_q / p->num_heads_kv;
  const int32_t chunk = kv_chunk_for(p);
  int64_t n = 0;
  auto emit = [&](const af::WorkTile& w) {
    if (n < cap && out != nullptr) {
      out[n].batch = w.b;
      out[n].head = w.h;
      out[n].tile = w.t;
      out[n].split = w.split;
    }
    ++n;
  };
  if (host_cu_seqlens_q == nullptr) {
    const int32_t T = af::tiles_for(p->seqlen_q, rows_for(p));
    const int32_t splits = resolve_splits(p);
    const int64_t total = (int64_t)p->batch * p->num_heads_q * T * splits;
    for (int64_t w = 0; w < total; ++w) emit(af::decode_fixed(w, T, splits, p->num_heads_q, group, chunk));
    return n;
  }
  const int32_t splits = resolve_splits(p);
  for (int b = 0; b < p->batch; ++b) {
    const int32_t len = host_cu_seqlens_q[b + 1] - host_cu_seqlens_q[b];
    const int32_t T = af::tiles_for(len, rows_for(p));
    for (int64_t wl = 0; wl < (int64_t)T * splits * p->num_heads_q; ++wl) {
      af::WorkTile w = af::decode_in_sequence(wl, b, T * splits, group, p->num_heads_kv, chunk);
      w.split = w.t % splits;
      w.t /= splits;
      emit(w);
    }
  }
  return n;
}

attn_status attn_fwd_key_range(const attn_fwd_params* p, int32_t tile, int32_t split, int32_t seqlen_k,
                               int32_t* key_begin, int32_t* key_end) {
  clear_error();
  if (p == nullptr || key_begin == nullptr || key_end == nullptr)
    return fail(ATTN_ERR_INVALID_ARG, "NULL argument");
  if (tile < 0 || seqlen_k < 0) return fail(ATTN_ERR_INVALID_ARG, "tile %d / seqlen_k %d negative", tile, seqlen_k);
  const int32_t splits = resolve_splits(p);
  if (split < 0 || split >= splits) return fail(ATTN_ERR_INVALID_ARG, "split %d outside [0, %d)", split, splits);
  if (splits == 1) {
    *key_begin = 0;
    *key_end = seqlen_k;
    return ATTN_OK;
  }
  const int32_t rows = rows_for(p);
  if ((int64_t)tile * rows > 0x7fffffffll - rows) return fail(ATTN_ERR_INVALID_ARG, "tile %d too large", tile);
  int32_t j0 = 0, j1 = 0;
  if (p->causal)
    af::causal_split_range(split, splits, tile * rows, af::kBlockM, rows, seqlen_k, af::kBlockN, &j0, &j1);
  else
    af::split_range(split, splits, af::tiles_for(seqlen_k, af::kBlockN), &j0, &j1);
  const int64_t b = (int64_t)j0 * af::kBlockN, e = (int64_t)j1 * af::kBlockN;
  *key_begin = (int32_t)(b < seqlen_k ? b : seqlen_k);
  *key_end = (int32_t)(e < seqlen_k ? e : seqlen_k);
  return ATTN_OK;
}

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* attn_fwd_last_error(void) { return g_last_error; }

}  // extern "C"
