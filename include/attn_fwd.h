/*
 * attn_fwd.h - C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * Operation (the forward pass of the flash-attention kernel whose shared-memory
 * layout the "SM100AttentionSMem" page documents; the rope sub-depth and the
 * per-token Q/K scale are the optional parts of that page's Parameters
 * section; the persistent work loop follows the "MHATileScheduler" page and
 * the staged K/V loads the "TMAProducerPipeline" page):
 *
 *   for each sequence b, query head h, query row i:
 *     hk    = h / (Hq / Hkv)                        consecutive query heads share a KV head
 *     J_i   = { j < Sk_b : !causal || j <= i }      causal mask is top-left aligned
 *     s_ij  = scale * (q_i . k_j + q_rope_i . k_rope_j)            bf16 Q/K (rope optional)
 *     s_ij  = scale * q_scale_i * k_scale_j * (Q8_i . K8_j)         fp8 e4m3 Q/K
 *     LSE_i = ln sum_{j in J_i} exp(s_ij)                           natural log
 *     O_i   = sum_{j in J_i} exp(s_ij - LSE_i) * v_j                bf16, rounded once
 *   With fp8 e4m3 V (v_dtype; Q/K fp8 too: the page's single qkv_dtype) the
 *   weights exp(s_ij - m) are rounded to e4m3 before the P.V product (O_i is
 *   then exact up to that rounding, at most 2^-4 relative per weight, plus
 *   2^-10 absolute per weight relative to the row maximum); LSE_i is not.
 *   Rows with an empty J_i get O_i = 0 and LSE_i = -inf.
 *
 * Conventions
 *   - Every pointer in attn_fwd_params is a DEVICE pointer owned by the caller.
 *     The library allocates no memory. Its only process-wide state is
 *     read-mostly caches (the SM count per device, the driver's tensor-map
 *     encoder entry point) and the fixed scratch array of attn_fwd_noalloc;
 *     calls on different workspaces and streams are independent.
 *   - attn_fwd() validates, encodes TMA descriptors on the host and enqueues
 *     one kernel on `stream` (two with split-KV: the partial ranges, then
 *     their merge); it returns without synchronising. Invalid
 *     arguments are reported before anything is enqueued and no memory is
 *     touched. No C++ exception crosses this boundary.
 *   - Kernel-side failures (a bounded wait that ran out) are recorded in the
 *     workspace and reported by attn_fwd_check().
 */
#ifndef ATTN_FWD_H
#define ATTN_FWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *attn_stream_t;

typedef enum attn_dtype {
  ATTN_DTYPE_BF16 = 0,      /* Q and K bf16 */
  ATTN_DTYPE_FP8_E4M3 = 1   /* Q and K float8_e4m3fn with per-token fp32 scales */
} attn_dtype;

typedef enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,     /* malformed arguments (null, misaligned, inconsistent sizes) */
  ATTN_ERR_UNSUPPORTED = 2,     /* well-formed but not handled (head dims, dtype mix) */
  ATTN_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed */
  ATTN_ERR_DEVICE_TIMEOUT = 4   /* a kernel wait ran out of time (see attn_fwd_check) */
} attn_status;

typedef enum attn_backend {
  ATTN_BACKEND_TCGEN05 = 0,     /* persistent warp-specialised tcgen05/TMA kernel */
  ATTN_BACKEND_SIMPLE = 1       /* plain fp32 CUDA-core kernel, for cross-checking only */
} attn_backend;

/* Work distribution of the tcgen05 kernel (the "mha_schedule" and
 * "may_advance" members of the MHATileScheduler page). Every mode visits
 * the same work tiles in the same heaviest-first order (attn_fwd_schedule)
 * and gives bit-identical results; they differ only in how tiles reach CTAs. */
typedef enum attn_schedule {
  ATTN_SCHEDULE_DYNAMIC = 0,    /* persistent, one CTA per SM; each CTA takes the next work index
                                   from an atomic counter when it finishes a tile (default) */
  ATTN_SCHEDULE_STATIC = 1,     /* persistent, one CTA per SM; CTA c takes indices c, c + grid, ... */
  ATTN_SCHEDULE_GRID = 2        /* one CTA per work tile, no advance; the hardware launches CTAs
                                   in index order as SMs free up */
} attn_schedule;

/* CTA pairs (the "pair_cta" option of the SM100AttentionSMem page's barrier
 * set, FA4MiscMBars): two CTAs of a cluster on neighbouring SMs share every
 * tensor-core instruction (M = 256 rows, tcgen05 cta_group::2). Each CTA
 * holds 128 of the rows of an instruction, half of every K tile (64 keys) and
 * half of every V tile (64 depth columns), so each SM reads and stages half
 * the K/V bytes; a work tile is 512 query rows. Results are those of the
 * one-CTA kernel (same arithmetic per row). */
typedef enum attn_pair_cta {
  ATTN_PAIR_AUTO = 0,           /* the library chooses */
  ATTN_PAIR_OFF = 1,            /* one CTA per MMA tile */
  ATTN_PAIR_ON = 2              /* CTA pairs: bf16 Q/K/V, Dqk = Dv = 128, rope 0 or 64; tcgen05 backend */
} attn_pair_cta;

/* Bytes of workspace attn_fwd needs without split-KV; the workspace holds the
 * persistent scheduler's work counter and the device error record (and, with
 * split-KV, the partial results: see attn_fwd_workspace_bytes). */
#define ATTN_FWD_WORKSPACE_BYTES 256

/* Size of the scratch array that attn_fwd_noalloc keeps inside the library
 * (one copy per GPU that loads the library). */
#define ATTN_FWD_STATIC_WORKSPACE_BYTES 256

typedef struct attn_fwd_params {
  /* ---- tensors (device pointers, caller-owned) ------------------------- */
  const void *q;        /* fixed [B,Sq,Hq,Dqk] / packed [Tq,Hq,Dqk]; bf16 or fp8 (qk_dtype) */
  const void *k;        /* fixed [B,Sk,Hkv,Dqk] / packed [Tk,Hkv,Dqk]; same type as q */
  const void *v;        /* bf16 (v_dtype BF16): fixed [B,Sk,Hkv,Dv] / packed [Tk,Hkv,Dv];
                           fp8 e4m3 (v_dtype FP8_E4M3): depth-major with the keys contiguous,
                           fixed [B,Hkv,Dv,Sk] / packed [Hkv,Dv,Tv] (sequence b at keys
                           cu_seqlens_v[b] ...; v_stride: see below) */
  const void *q_rope;   /* rope_depth > 0 only: [B,Sq,Hq,R] / [Tq,Hq,R]; bf16 */
  const void *k_rope;   /* rope_depth > 0 only: [B,Sk,R] / [Tk,R]; bf16, shared by all heads */
  const float *q_scale; /* fp8 only: [B,Hq,Sq] / [Hq,Tq], contiguous fp32 */
  const float *k_scale; /* fp8 only: [B,Hkv,Sk] / [Hkv,Tk], contiguous fp32 */
  const int32_t *cu_seqlens_q; /* packed only: [B+1] prefix offsets of the query rows */
  const int32_t *cu_seqlens_k; /* packed only: [B+1] prefix offsets of the key rows */
  void *o;              /* fixed [B,Sq,Hq,Dv] / packed [Tq,Hq,Dv]; bf16, written */
  float *lse;           /* [B,Hq,Sq] / [Hq,Tq] contiguous fp32, written; may be NULL */
  void *workspace;      /* >= attn_fwd_workspace_bytes(p) device bytes, 256-byte aligned,
                           zero-filled once before its first use; every call leaves it
                           zeroed again. Calls that share a workspace must not overlap. */
  size_t workspace_bytes;

  /* ---- sizes ------------------------------------------------------------ */
  int32_t batch;        /* B, number of sequences */
  int32_t seqlen_q;     /* fixed: Sq; packed: an upper bound of every query length */
  int32_t seqlen_k;     /* fixed: Sk; packed: an upper bound of every key length */
  int32_t total_q;      /* packed only: Tq (rows of q and o) */
  int32_t total_k;      /* packed only: Tk (rows of k and v) */
  int32_t num_heads_q;  /* Hq */
  int32_t num_heads_kv; /* Hkv, divides Hq */
  int32_t head_dim_qk;  /* Dqk, depth of q and k without the rope part */
  int32_t head_dim_v;   /* Dv */
  int32_t rope_depth;   /* R, 0 or 64 */
  int32_t causal;       /* non-zero: query i sees keys 0..i of its sequence */
  float softmax_scale;  /* scale of the scores; > 0 */
  int32_t qk_dtype;     /* attn_dtype */
  int32_t v_dtype;      /* attn_dtype of v: BF16, or FP8_E4M3 (needs fp8 q/k, Dqk = Dv = 128,
                           no rope; no scale: V's e4m3 values are used as is) */
  int32_t backend;      /* attn_backend */

  /* ---- element strides: [0] batch (unused when packed), [1] token, [2] head.
   *      The innermost dimension is contiguous. For depth-major fp8 v,
   *      v_stride is [0] batch, [1] depth row, [2] head (keys contiguous;
   *      the depth-row stride must be a multiple of 16 bytes). ------------- */
  int64_t q_stride[3];
  int64_t k_stride[3];
  int64_t v_stride[3];
  int64_t o_stride[3];
  int64_t q_rope_stride[3];
  int64_t k_rope_stride[2]; /* [0] batch, [1] token */

  /* Testing only; leave 0. 1: the first CTA withholds its first V tile, so a
   * bounded device wait runs out (limit 200 ms instead of 2 s), the kernel
   * aborts cleanly and attn_fwd_check reports ATTN_ERR_DEVICE_TIMEOUT. */
  int32_t fault_injection;

  /* Split-KV: number of key ranges each query tile is split into (the
   * "splitk_partitions" of the SM100AttentionSMem page's configuration).
   * 0 = chosen by the library (splits problems whose query tiles cannot
   * fill the GPU: unmasked problems with too few query tiles, causal
   * problems whose heaviest query tile outlasts the rest of the work),
   * 1 = off, n >= 2 = n ranges (at most 64, capped at the key tiles of the
   * longest sequence; a sequence or, under the causal mask, a query tile
   * with fewer key tiles leaves some of its ranges empty; attn_fwd_key_range
   * gives each range's keys). Each range writes a normalised partial O and
   * its LSE into the workspace (attn_fwd_workspace_bytes grows accordingly)
   * and a second small kernel merges them. Causal split-KV with CTA pairs is
   * UNSUPPORTED (n >= 2); the automatic choice does not split there. */
  int32_t num_splits;

  /* attn_schedule; ignored by the simple backend. */
  int32_t schedule;

  /* attn_pair_cta. ATTN_PAIR_ON outside its supported configurations (see
   * attn_pair_cta) is UNSUPPORTED; with it fault_injection must be 0. */
  int32_t pair_cta;

  /* Packed e4m3 V only (NULL otherwise): [B+1] device int32, the key index
   * along V's contiguous key dimension where sequence b's Lk_b keys start;
   * every start must be a multiple of 16 (a TMA copy starts on a 16-byte
   * boundary) and start + Lk_b <= total_v. The kernel checks this and
   * reports a violation through attn_fwd_check as INVALID_ARG. */
  const int32_t *cu_seqlens_v;
  int32_t total_v;          /* packed e4m3 V: Tv, the length of V's key dimension */
} attn_fwd_params;

/* Query results of attn_fwd_plan (host only; no GPU needed). */
typedef struct attn_fwd_plan_info {
  int32_t backend;          /* kernel that attn_fwd would launch */
  int32_t rows_per_tile;    /* query rows per work tile (256; 512 with CTA pairs) */
  int64_t work_tiles;       /* fixed: exact count; packed: upper bound B*Hq*ceil(Sq/rows) */
  int32_t grid;             /* CTAs launched (persistent: min(SMs, work_tiles); CTA pairs:
                               2 * min(resident clusters, work_tiles)) */
  int32_t block;            /* threads per CTA */
  int32_t smem_bytes;       /* dynamic shared memory per CTA */
  int32_t k_stages;         /* depth of the K ring */
  int32_t v_stages;         /* depth of the V ring */
  int32_t tmem_columns;     /* tensor-memory columns allocated per CTA */
  int32_t num_splits;       /* key ranges per query tile (1 = no split-KV) */
  int32_t pair_cta;         /* 1 = one CTA per MMA tile, 2 = CTA pairs */
} attn_fwd_plan_info;

/* One work tile as the persistent scheduler hands it out. */
typedef struct attn_work_tile {
  int32_t batch;            /* sequence b */
  int32_t head;             /* query head h */
  int32_t tile;             /* query tile t: rows [t*rows_per_tile, (t+1)*rows_per_tile) */
  int32_t split;            /* split-KV key range (0 without split-KV) */
} attn_work_tile;

/* Fills `p` with zeros and the defaults (bf16, tcgen05 backend). */
void attn_fwd_params_init(attn_fwd_params *p);

/* sizeof(attn_fwd_params) as compiled into the library (binding check). */
size_t attn_fwd_params_size(void);

/* Workspace bytes needed for `p`: ATTN_FWD_WORKSPACE_BYTES, plus with
 * split-KV (n ranges) the partial LSE, n*R*Hq floats rounded up to 256
 * bytes, and the partial O, n*R*Hq*Dv floats (R = B*Sq, or Tq when packed). The automatic split count
 * (num_splits = 0) depends on the SM count of the current device: call this
 * with the device current that attn_fwd will run on. Never fails (an invalid
 * `p` or NULL gives ATTN_FWD_WORKSPACE_BYTES). */
size_t attn_fwd_workspace_bytes(const attn_fwd_params *p);

/* Validates `p` and enqueues the forward on `stream`. Asynchronous. Errors:
 * INVALID_ARG / UNSUPPORTED before launch; CUDA if the launch failed. */
attn_status attn_fwd(const attn_fwd_params *p, attn_stream_t stream);

/* attn_fwd for callers that cannot allocate device memory: it takes no
 * workspace (p->workspace is ignored) and uses a fixed scratch array of
 * ATTN_FWD_STATIC_WORKSPACE_BYTES inside the library instead. The paper has
 * no counterpart of this call; it exists for code that only receives tensors
 * and a stream from a host framework that owns all device memory, or that
 * must not allocate once it is running. It allocates nothing and calls no
 * allocating routine. The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current), so make it
 * before any stream capture; calls outside a capture look it up again (no
 * allocation), so the address stays valid across a cudaDeviceReset. Every
 * call clears and reuses the same array: calls that overlap on the GPU
 * (concurrent streams, or other threads) race on it and must be serialised
 * by the caller. Device-side wait timeouts of this variant are not reported
 * (there is no caller-visible error record): if a bounded wait inside the
 * kernel ran out, which only a defect can cause, that call's O and LSE are
 * undefined and nothing says so.
 * num_splits = 0 means "no split" here; an explicit split count needs more
 * scratch than the array holds. Returns UNSUPPORTED if a call would need more
 * scratch than the array holds, otherwise as attn_fwd. */
attn_status attn_fwd_noalloc(const attn_fwd_params *p, attn_stream_t stream);

/* Synchronises `stream`, reads and clears the device error record of
 * `workspace`. Returns DEVICE_TIMEOUT if a kernel wait ran out, INVALID_ARG
 * if the kernel found packed offsets (cu_seqlens) decreasing or past
 * total_q / total_k (it then skipped that work and wrote nothing outside
 * the tensors; the call's output cannot be trusted), CUDA for a pending CUDA
 * error, else OK. */
attn_status attn_fwd_check(void *workspace, attn_stream_t stream);

/* Validates `p` and reports the launch plan without touching the GPU,
 * except for reading the SM count of the current device when one exists
 * (148 SMs are assumed otherwise). */
attn_status attn_fwd_plan(const attn_fwd_params *p, attn_fwd_plan_info *out);

/* Host copy of the persistent scheduler's order: writes up to `cap` work
 * tiles in the order the kernel hands them out and returns how many there
 * are in total. `host_cu_seqlens_q` is a HOST array of B+1 offsets, or NULL
 * for fixed length. Used to test the schedule on a CPU. */
int64_t attn_fwd_schedule(const attn_fwd_params *p, const int32_t *host_cu_seqlens_q,
                          attn_work_tile *out, int64_t cap);

/* Keys [*key_begin, *key_end) of one sequence (seqlen_k keys) that range
 * `split` of query tile `tile` covers, as the kernel computes them (split-KV,
 * the "splitk_partitions" of the SM100AttentionSMem page's configuration).
 * Without split-KV the range is the whole sequence. Unmasked, the ranges cut
 * the sequence's key tiles into num_splits contiguous parts. Under the
 * causal mask they cut the key tiles the query tile's first 128 rows see, and
 * the last range also takes the tiles only its later rows see: every range
 * that holds keys starts at or before the tile's first row, and the ranges
 * end where the tile's last row stops seeing keys (the mask applies within a
 * range as without split-KV). A range may be empty (*key_begin == *key_end)
 * when the tile sees fewer key tiles than there are ranges. Host only: the
 * split count is resolved as attn_fwd_plan reports it. Returns INVALID_ARG
 * for a NULL pointer, tile < 0, seqlen_k < 0 or split outside
 * [0, num_splits). */
attn_status attn_fwd_key_range(const attn_fwd_params *p, int32_t tile, int32_t split, int32_t seqlen_k,
                               int32_t *key_begin, int32_t *key_end);

/* Static description of a status code. */
const char *attn_status_string(attn_status s);

/* Detail of the last error returned to the calling thread (empty if none). */
const char *attn_fwd_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_H */
