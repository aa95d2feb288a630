// Persistent, warp-specialised attention forward for sm_103a (tcgen05 + TMA).
//
// Design (prior art: the SM100 flash-attention pages "SM100AttentionSMem",
// "TMAProducerPipeline" and "MHATileScheduler"; rebuilt here for one GB300
// CTA per SM):
//   * a work tile is 256 query rows of one (sequence, head), split into two
//     128-row Q tiles that ping-pong between two softmax warpgroups so the
//     tensor core always has one Q tile's MMAs to run while the other tile's
//     softmax runs (with split-KV, a work tile also names one range of the
//     keys);
//   * warp 14 is the scheduler and the Q/K producer: it takes work indices
//     from an atomic counter (or a static stride, or none: one CTA per work
//     tile), publishes each decoded work tile through a two-slot
//     shared-memory ring (the shared work index of the scheduler page,
//     initial_state / advance) and streams K tiles into a staged ring with
//     TMA and transaction-count mbarriers (acquire / expect-bytes / commit of
//     the producer-pipeline page); warp 15 streams V tiles into their own
//     ring. K is stored k-major and V mn-major (k-major when V is e4m3 and
//     depth-major in memory), all with the 128-byte swizzle, exactly as the
//     MMAs read them;
//   * warps 12 and 13 each issue the tcgen05.mma of one Q tile from one
//     thread: per K/V step one group, O_i += P_i V (P_i read from tensor
//     memory where the softmax left it, over the S_i columns) then
//     S_i = Q_i K^T into tensor memory (fp32); the two issuers' groups
//     strictly alternate through a turn token (the forced-ordering barriers
//     of the layout page);
//   * warpgroups 0 and 1 own Q tiles 0 and 1: thread r owns row r (TMEM lane
//     r), loads S, applies the causal / sequence-end mask, keeps the running
//     max m and sum l in log2 units and writes P = 2^(s*c - m) (bf16, or
//     e4m3 for an e4m3 V) back to tensor memory in two halves. The running
//     max only moves when it grows by more than 2^8, so most tiles need no
//     rescale; when it moves, the softmax warp rescales its own rows of O_i
//     in tensor memory before publishing P. O and l share the max, so O/l is
//     exact;
//   * warpgroup 2 is the epilogue: after the last P V it normalises O by 1/l
//     (handed over through shared memory, the correction region of the
//     layout page), rounds once to bf16 and stores it, or stores the fp32
//     partial row of a split-KV range.
//   * CTA pairs (the pair_cta option of the layout page's barrier set;
//     Tc05Traits<..., PAIR = true>): two CTAs of a cluster on neighbouring
//     SMs share every MMA. A work tile is then 512 rows; each of its two MMA
//     tiles is 256 rows, 128 in each CTA, issued as one M = 256
//     tcgen05.mma.cta_group::2 by the first CTA's issuers. Each CTA loads its
//     own Q rows, half of each K tile (64 keys) and half of each V tile (64
//     depth columns); all copies complete on the first CTA's barriers, the
//     MMA commits arrive in both CTAs (multicast), and the softmax and
//     epilogue warps of the second CTA report to the first CTA's barriers
//     through the cluster window. Work indices are fetched by the first CTA
//     and forwarded to the second through its shared memory.
// Every wait is bounded: on timeout the CTA records an error in the
// workspace, raises a shared abort flag that all waits poll (and, in a pair,
// the peer's flag), drains its outstanding copies and MMAs, frees tensor
// memory and exits.
#pragma once
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"
#include "schedule.cuh"

namespace af {

constexpr uint32_t kFull = 0xffffffffu;
constexpr uint64_t kDrainTimeoutNs = 100000000ull;

enum Role : int { kRoleSoftmax0 = 0, kRoleSoftmax1 = 1, kRoleCorrection = 2, kRoleMma = 3, kRoleLoadQK = 4,
                  kRoleLoadV = 5 };

enum BarId : int {
  BAR_Q_FULL = 0,        // +i, TMA transaction barrier of Q tile i
  BAR_Q_EMPTY = 2,       // last S MMA of Q tile 0 done: its Q region is free (tile 1: BAR_Q_EMPTY1)
  BAR_S_FULL = 3,        // +i, S_i = Q_i K^T complete
  BAR_P_LO = 5,          // +i, first half of P_i (keys 0..63) in tensor memory (128 arrivals)
  BAR_STATS = 7,         // +i, final 1/l of Q tile i in shared memory (128 arrivals)
  BAR_P_HI = 9,          // +i, second half of P_i (keys 64..127) in tensor memory (128)
  BAR_O_FINAL = 11,      // +i, last P_i V of a work tile complete
  BAR_O_FREE = 13,       // +i, epilogue finished reading O_i (128)
  BAR_STATS_FREE = 15,   // +i, correction read the 1/l of Q tile i (128)
  BAR_KS = 17,           // +i, fp8 k-scale tile written by the softmax warpgroup (128)
  BAR_SCHED_FULL = 19,   // +slot
  BAR_SCHED_EMPTY = 21,  // +slot
  BAR_DRAIN = 23,        // final commit of the MMA threads
  BAR_ORDER = 24,        // +i, issue turn of MMA issuer i (forced ordering of the two Q tiles)
  BAR_Q_EMPTY1 = 26,     // last S MMA of Q tile 1 done
  BAR_WORK_FULL = 27,    // +slot, CTA pairs: work index written into the second CTA by the first
  BAR_WORK_EMPTY = 29,   // +slot, CTA pairs: the second CTA read that work index
  BAR_SM_TURN = 31,      // +i, softmax turn of warpgroup i (128 arrivals of the other warpgroup)
  BAR_FIXED = 33         // then K_FULL[NK], K_EMPTY[NK], V_FULL[NV], V_EMPTY[NV]
};

constexpr int kSlotBytes = 48;   // shared-memory bytes of one SchedSlot entry

// Consumers of a scheduler slot: the two MMA lanes, 2 softmax warpgroups, the
// correction warpgroup and the V producer lane.
constexpr uint32_t kSchedConsumers = 2 + 128 + 128 + 128 + 1;

template <int DQK_, int DR_, int DV_, bool FP8_, bool V8_ = false, bool PAIR_ = false>
struct Tc05Traits {
  static constexpr int DQK = DQK_, DR = DR_, DV = DV_;
  static constexpr bool FP8 = FP8_;
  // e4m3 V, depth-major in global memory: a V stage is Dv rows of 128 keys
  // (K-major B operand of P.V) and P is rounded to e4m3 for kind::f8f6f4.
  static constexpr bool V8 = V8_;
  static_assert(!V8 || (FP8 && DV == 128), "e4m3 V needs e4m3 Q/K and Dv = 128");
  // CTA pair: M = 256 MMAs over two CTAs; this CTA holds 128 of the rows,
  // 64 keys of each K tile and 64 depth columns of each V tile.
  static constexpr bool PAIR = PAIR_;
  static_assert(!PAIR || (!FP8 && DQK == 128 && DV == 128), "CTA pairs: bf16 with Dqk = Dv = 128");
  static constexpr int BM = kBlockM, BN = kBlockN, NQ = 2;
  static constexpr int MMA_M = PAIR ? 2 * kBlockM : kBlockM;   // rows of one MMA tile (both CTAs)
  static constexpr int ROWS_PER_WORK = NQ * MMA_M;              // rows of one work tile
  static constexpr int QK_CHUNK_ELEMS = FP8 ? 128 : 64;   // elements of one 128-byte swizzle row
  static constexpr int QK_CHUNKS = DQK / QK_CHUNK_ELEMS;
  static constexpr int R_CHUNKS = DR / 64;
  static constexpr int V_CHUNKS = V8 ? 1 : (PAIR ? 1 : DV / 64);   // TMA boxes per V stage (this CTA)
  static constexpr int CHUNK_BYTES = 128 * 128;           // 128 rows x 128 bytes
  static constexpr int K_ROWS = PAIR ? kBlockN / 2 : kBlockN;   // keys of a K stage held by this CTA
  static constexpr int K_CHUNK_BYTES = K_ROWS * 128;
  static constexpr int Q_TILE_BYTES = (QK_CHUNKS + R_CHUNKS) * CHUNK_BYTES;
  static constexpr int K_STAGE_BYTES = (QK_CHUNKS + R_CHUNKS) * K_CHUNK_BYTES;
  static constexpr int V_STAGE_BYTES = V8 ? DV * 128 : V_CHUNKS * CHUNK_BYTES;
  static constexpr int NK = PAIR ? (DR > 0 ? 3 : 5) : (DR > 0 ? 2 : (FP8 ? 4 : (DQK == 64 ? 4 : 3)));
  static constexpr int NV = PAIR ? (DR > 0 ? 3 : 4) : (DR > 0 ? 1 : (V8 ? 4 : (FP8 ? 3 : (DQK == 64 ? 4 : 2))));
  // Bytes one phase of a Q / K / V full barrier waits for (a pair's first CTA
  // counts both CTAs' copies).
  static constexpr uint32_t Q_TX = (PAIR ? 2 : 1) * Q_TILE_BYTES;
  static constexpr uint32_t K_TX = (PAIR ? 2 : 1) * K_STAGE_BYTES;
  static constexpr uint32_t V_TX = (PAIR ? 2 : 1) * V_STAGE_BYTES;

  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = NQ * Q_TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NK * K_STAGE_BYTES;
  static constexpr int OFF_RCPL = OFF_V + NV * V_STAGE_BYTES;       // float [NQ][BM]
  static constexpr int OFF_KS = OFF_RCPL + NQ * BM * 4;             // float [NQ][2][BN] (fp8)
  static constexpr int KS_BYTES = FP8 ? NQ * 2 * BN * 4 : 0;
  static constexpr int OFF_SCHED = OFF_KS + KS_BYTES;               // 2 slots x kSlotBytes
  static constexpr int OFF_WORK = OFF_SCHED + 2 * kSlotBytes;       // CTA pairs: 2 x int64 work index
  static constexpr int OFF_BAR = OFF_WORK + 16;
  static constexpr int NUM_BARS = BAR_FIXED + 2 * NK + 2 * NV;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 12;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA exceeded");
  static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0, "swizzled tiles need 1024-byte alignment");

  static constexpr int BAR_K_FULL = BAR_FIXED;
  static constexpr int BAR_K_EMPTY = BAR_FIXED + NK;
  static constexpr int BAR_V_FULL = BAR_FIXED + 2 * NK;
  static constexpr int BAR_V_EMPTY = BAR_FIXED + 2 * NK + NV;

  static constexpr uint32_t TMEM_COLS = 512;
  // Tensor-memory columns: S_0, S_1 (P_i overwrites the first 64 columns of
  // S_i as packed bf16 pairs), O_0, O_1.
  __host__ __device__ static constexpr uint32_t tm_s(int i) { return i ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t tm_o(int i) { return i ? 384u : 256u; }

  static constexpr uint32_t IDESC_S =
      FP8 ? ptx::idesc_f32acc(0, 0, false, false, 128, 128) : ptx::idesc_f32acc(1, 1, false, false, MMA_M, 128);
  static constexpr uint32_t IDESC_PV =
      V8 ? ptx::idesc_f32acc(0, 0, false, false, 128, DV) : ptx::idesc_f32acc(1, 1, false, true, MMA_M, DV);
  // P.V instructions per half tile of 64 keys (K = 16 per bf16 instruction, 32 per e4m3).
  static constexpr int PV_INSTR_HALF = V8 ? 2 : 4;
  // TMEM columns of one half of P (64 keys as bf16 pairs or e4m3 quads).
  static constexpr int P_COLS_HALF = V8 ? 16 : 32;
  // MMA instructions of one S = Q K^T (K = 16 per bf16 instruction, 32 per fp8).
  static constexpr int S_INSTR = FP8 ? DQK / 32 : (DQK + DR) / 16;
  // S instructions issued after handing the turn to the other issuer: enough
  // tensor work (~4 x 73 cycles) to cover the other issuer's wake-up.
  static constexpr int S_AFTER_HANDOFF = S_INSTR < 4 ? S_INSTR : 4;

  // Register split (setmaxnreg) of a 512-thread CTA launched with 128 registers per thread.
  // The FP8 softmax (k-scale multiply, e4m3 packing) takes 192 registers; its
  // epilogue warpgroup then fits in 64 (measured: +1-3 % on the FP8
  // workloads, no change for bf16).
  static constexpr int REG_SOFTMAX = FP8 ? 192 : 184, REG_CORR = FP8 ? 64 : 80, REG_MISC = 64;
  // Softmax turn: 0 = the two softmax warpgroups run freely; 1 / 2 = they
  // take turns, handing over after the first half of P / after the tile.
  // With FP8 Q/K a tile's MMAs take less time than a softmax, and two
  // softmaxes that overlap each take twice as long: taking turns keeps them
  // apart.
  static constexpr int SM_TURN = FP8 ? 1 : 0;
  static_assert(2 * 128 * REG_SOFTMAX + 128 * REG_CORR + 128 * REG_MISC <= 512 * 128,
                "register split exceeds the launch allocation");
};

// One decoded work tile as published to every role. With split-KV, k_start
// and lk already describe the tile's own key range.
struct SchedSlot {
  int32_t valid, b, h, t, q_start, lq, k_start, lk, split;
  int32_t v_start;   // first key of the tile's range along V's key dimension (packed e4m3 V: own offsets)
  int32_t koff;      // first key of the range within its sequence (0 without split-KV): the causal mask
};

struct Ctx {
  uint8_t* smem;
  uint32_t sbase;
  uint32_t tmem;
  volatile int* abort_flag;
  uint32_t* ws;
  uint64_t timeout_ns;
  int bar_off;
  uint32_t rank;         // CTA pairs: this CTA's rank in the cluster (0 issues the MMAs); else 0
  uint32_t peer_abort;   // CTA pairs: cluster-window address of the peer's abort flag; else 0
  __device__ __forceinline__ uint32_t bar(int i) const { return sbase + bar_off + 8u * (uint32_t)i; }
  // Cluster-window address of barrier i in the pair's first CTA.
  __device__ __forceinline__ uint32_t bar_lead(int i) const { return ptx::mapa(bar(i), 0); }
  __device__ __forceinline__ static int q_empty_id(int i) { return i == 0 ? BAR_Q_EMPTY : BAR_Q_EMPTY1; }
};

__device__ __forceinline__ void raise_error(const Ctx& c, int role, int id) {
  if (atomicCAS(&c.ws[kWsErrorCode], 0u, (uint32_t)kDevErrTimeout) == 0u)
    atomicExch(&c.ws[kWsErrorInfo], ((uint32_t)blockIdx.x << 16) | ((uint32_t)role << 8) | (uint32_t)id);
  *c.abort_flag = 1;
  if (c.peer_abort != 0u) ptx::st_cluster_u32(c.peer_abort, 1u);
}

// Warp-uniform bounded wait: every lane polls, the result is the same in all
// lanes. CLUSTER: the phase completes through arrivals of the peer CTA of a
// pair, whose writes it must see (cluster-scope acquire).
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_warp(const Ctx& c, int id, uint32_t parity, int role) {
  const uint32_t bar = c.bar(id);
  if (__all_sync(kFull, CLUSTER ? ptx::mbar_test_wait_cluster(bar, parity) : ptx::mbar_test_wait(bar, parity)))
    return true;
  const uint64_t t0 = __shfl_sync(kFull, ptx::globaltimer(), 0);
  for (uint32_t it = 1;; ++it) {
    if (__all_sync(kFull, CLUSTER ? ptx::mbar_test_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity)))
      return true;
    if ((it & 63u) == 0u) {
      if (__any_sync(kFull, *c.abort_flag != 0)) return false;
      const uint64_t now = __shfl_sync(kFull, ptx::globaltimer(), 0);
      if (now - t0 > c.timeout_ns) {
        if ((threadIdx.x & 31) == 0) raise_error(c, role, id);
        __syncwarp();
        return false;
      }
    }
  }
}

// Bounded wait of a single thread (the MMA issuers). It polls without ever
// suspending: a thread suspended in mbarrier.try_wait was seen to resume
// hundreds of cycles after the phase completed, and every cycle an issuer
// loses leaves the tensor core idle.
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_one(const Ctx& c, int id, uint32_t parity, int role) {
  const uint32_t bar = c.bar(id);
  auto test = [&]() { return CLUSTER ? ptx::mbar_test_wait_cluster(bar, parity) : ptx::mbar_test_wait(bar, parity); };
  if (test()) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (test()) return true;
    if ((it & 255u) == 0u) {
      if (*c.abort_flag != 0) return false;
      if (ptx::globaltimer() - t0 > c.timeout_ns) {
        raise_error(c, role, id);
        return false;
      }
    }
  }
}

// Bounded wait of one thread that ignores the abort flag (drain paths).
__device__ __forceinline__ bool wait_drain(const Ctx& c, int id, uint32_t parity) {
  const uint32_t bar = c.bar(id);
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kDrainTimeoutNs) return false;
  }
  return true;
}

// CTA pairs: arrival on barrier `id` of the pair's first CTA (a local arrive
// there, a release at cluster scope through the cluster window from the
// second CTA).
__device__ __forceinline__ void arrive_lead(const Ctx& c, int id) {
  if (c.rank == 0) ptx::mbar_arrive(c.bar(id));
  else ptx::mbar_arrive_cluster(c.bar_lead(id));
}

// Ring position: stage index and phase parity.
template <int N>
struct Ring {
  uint32_t idx = 0, phase = 0;
  __device__ __forceinline__ void next() {
    if (++idx == (uint32_t)N) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

struct Geo {
  int q0;       // first row (within its sequence) of the work tile
  int row[2];   // first row of this CTA's 128 rows of MMA tile i
  int n[2];     // K/V tiles MMA tile i visits
};

template <class T, int CAUSAL>
__device__ __forceinline__ Geo tile_geo(const SchedSlot& s, uint32_t rank) {
  Geo g;
  g.q0 = s.t * T::ROWS_PER_WORK;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    g.row[i] = g.q0 + T::MMA_M * i + kBlockM * (int)rank;
    // causal: keys up to the tile's last row, counted from the range's first key
    const int kv_end = (CAUSAL & kMaskCausal) ? min(s.lk, g.q0 + T::MMA_M * (i + 1) - s.koff) : s.lk;
    g.n[i] = kv_end > 0 ? (kv_end + kBlockN - 1) / kBlockN : 0;
  }
  return g;
}

// Whether this kernel flavour runs split-KV ranges (fixed at compile time;
// the host launches the split flavours exactly when num_splits > 1).
template <int CAUSAL>
__device__ __forceinline__ constexpr bool splits_keys(const Tc05Params&) {
  return (CAUSAL & kMaskNoneSplit) != 0;
}

// The range's key offset travels only in the causal split flavour (its only user).
template <int CAUSAL>
__device__ __forceinline__ SchedSlot read_slot(const Ctx& c, int slot, int off_sched) {
  const volatile int32_t* p = reinterpret_cast<const volatile int32_t*>(c.smem + off_sched + kSlotBytes * slot);
  SchedSlot s;
  s.valid = p[0]; s.b = p[1]; s.h = p[2]; s.t = p[3];
  s.q_start = p[4]; s.lq = p[5]; s.k_start = p[6]; s.lk = p[7]; s.split = p[8]; s.v_start = p[9];
  s.koff = CAUSAL == kMaskCausalSplit ? p[10] : 0;
  return s;
}

// ---------------------------------------------------------------------------------------------
// Scheduler decode (warp 13, all lanes): work index -> work tile.
struct Cursor {
  int b = 0;
  int64_t base = 0;
};

template <int CAUSAL>
__device__ __forceinline__ SchedSlot decode_work(const Tc05Params& P, int64_t w, Cursor& cur) {
  SchedSlot s;
  s.valid = 0;
  s.b = s.h = s.t = s.q_start = s.k_start = s.split = s.v_start = s.koff = 0;
  s.lq = P.seqlen_q;
  s.lk = P.seqlen_k;
  if (!P.packed) {
    if (w < P.total_work) {
      const WorkTile wt = decode_fixed(w, P.tiles_per_seq, P.num_splits, P.heads_q, P.group, P.kv_chunk);
      s.valid = 1; s.b = wt.b; s.h = wt.h; s.t = wt.t; s.split = wt.split;
      if (splits_keys<CAUSAL>(P)) {
        int32_t j0, j1;
        if (CAUSAL & kMaskCausal)
          causal_split_range(wt.split, P.num_splits, wt.t * P.rows_per_tile, kBlockM, P.rows_per_tile, P.seqlen_k,
                             kBlockN, &j0, &j1);
        else
          split_range(wt.split, P.num_splits, P.kv_tiles, &j0, &j1);
        s.k_start = j0 * kBlockN;
        s.lk = min(P.seqlen_k, j1 * kBlockN) - s.k_start;
        if (CAUSAL == kMaskCausalSplit) s.koff = s.k_start;
      }
      s.v_start = s.k_start;
    }
    return s;
  }
  const int lane = threadIdx.x & 31;
  while (true) {
    const int bb = cur.b + lane;
    int64_t u = 0;
    bool bad = false;
    if (bb < P.batch) {
      // Offsets that would index outside q/k/v/o are refused here, before
      // any use: every sequence passes through this scan in some CTA (the
      // one whose work index runs past the batch scans to its end).
      const int qs = P.cu_q[bb], qe = P.cu_q[bb + 1], ks = P.cu_k[bb], ke = P.cu_k[bb + 1];
      bad = qs < 0 || qe < qs || qe > P.total_q || ks < 0 || ke < ks || ke > P.total_k;
      if (P.cu_v != nullptr) {
        // packed e4m3 V: each sequence's keys start on a 16-key boundary of V
        const int vs = P.cu_v[bb];
        bad = bad || vs < 0 || (vs & 15) != 0 || (int64_t)vs + (ke - ks) > (int64_t)P.total_v;
      }
      if (!bad) u = (int64_t)tiles_for(qe - qs, P.rows_per_tile) * P.heads_q * P.num_splits;
    }
    const unsigned bad_lanes = __ballot_sync(kFull, bad);
    if (bad_lanes) {
      // record it and end this CTA's work (its roles see an invalid slot)
      if (lane == 0 && atomicCAS(&P.ws[kWsErrorCode], 0u, (uint32_t)kDevErrBadSeqlens) == 0u)
        atomicExch(&P.ws[kWsErrorInfo], (uint32_t)(cur.b + __ffs(bad_lanes) - 1));
      return s;
    }
    int64_t incl = u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t n = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += n;
    }
    const unsigned hit = __ballot_sync(kFull, bb < P.batch && w < cur.base + incl);
    if (hit) {
      const int L = __ffs(hit) - 1;
      cur.base += __shfl_sync(kFull, incl - u, L);
      cur.b += L;
      const int b = cur.b;
      const int qs = P.cu_q[b], qe = P.cu_q[b + 1], ks = P.cu_k[b], ke = P.cu_k[b + 1];
      const WorkTile wt = decode_in_sequence(w - cur.base, b, tiles_for(qe - qs, P.rows_per_tile) * P.num_splits,
                                             P.group, P.heads_kv, P.kv_chunk);
      s.valid = 1; s.b = b; s.h = wt.h; s.t = wt.t;
      s.q_start = qs; s.lq = qe - qs; s.k_start = ks; s.lk = ke - ks;
      if (splits_keys<CAUSAL>(P)) {
        // this sequence's own key tiles, cut like the fixed-length case (a
        // range can be empty when the sequence has fewer key tiles than ranges)
        s.split = wt.t % P.num_splits;
        s.t = wt.t / P.num_splits;
        int32_t j0, j1;
        if (CAUSAL & kMaskCausal)
          causal_split_range(s.split, P.num_splits, s.t * P.rows_per_tile, kBlockM, P.rows_per_tile, ke - ks,
                             kBlockN, &j0, &j1);
        else
          split_range(s.split, P.num_splits, tiles_for(ke - ks, kBlockN), &j0, &j1);
        s.k_start = ks + j0 * kBlockN;
        s.lk = min(ke - ks, j1 * kBlockN) - j0 * kBlockN;
        if (CAUSAL == kMaskCausalSplit) s.koff = j0 * kBlockN;
      }
      s.v_start = P.cu_v != nullptr ? P.cu_v[b] + (s.k_start - ks) : s.k_start;
      return s;
    }
    if (cur.b + 32 >= P.batch) return s;
    cur.base += __shfl_sync(kFull, incl, 31);
    cur.b += 32;
  }
}

// ---------------------------------------------------------------------------------------------
// TMA load of one box into this CTA's shared memory, completing on barrier
// `bar` (in a pair: on that barrier of the pair's first CTA).
template <class T>
__device__ __forceinline__ void load_box(const Ctx& c, uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                         int c1, int c2, int c3) {
  if constexpr (T::PAIR) ptx::tma_load_4d_pair(dst, map, ptx::mapa(bar, 0), c0, c1, c2, c3);
  else ptx::tma_load_4d(dst, map, bar, c0, c1, c2, c3);
}

// Waits out this CTA's copies in flight after an abort. A pair's second CTA
// cannot watch its copies (they complete on the first CTA's barriers): it
// waits a fixed 200 us, far longer than any copy takes.
__device__ __forceinline__ void pair_copy_grace() {
  const uint64_t t0 = ptx::globaltimer();
  while (ptx::globaltimer() - t0 < 200000ull) {
  }
}

template <class T, int CAUSAL>
__device__ void role_load_qk(const Tc05Params& P, const Ctx& c) {
  const int lane = threadIdx.x & 31;
  const bool lead = c.rank == 0;
  Ring<2> sched;
  Ring<2> fwd;   // CTA pairs: work-index hand-over slots
  Ring<T::NK> kr;
  uint32_t q_empty_phase = 0;
  uint32_t k_fill_parity[T::NK];
  bool k_used[T::NK];
  bool q_loaded[2] = {false, false};
  uint32_t q_fill_parity = 0;
#pragma unroll
  for (int s = 0; s < T::NK; ++s) { k_fill_parity[s] = 0; k_used[s] = false; }
  Cursor cur;
  // The first work index is this CTA's own (a pair's: the cluster's).
  int64_t w = T::PAIR ? (int64_t)ptx::cluster_id_x() : (int64_t)blockIdx.x;
  const int64_t units = T::PAIR ? (int64_t)ptx::nclusters_x() : (int64_t)gridDim.x;
  bool aborted = false;
  while (true) {
    const SchedSlot s = decode_work<CAUSAL>(P, w, cur);
    if (!wait_warp(c, BAR_SCHED_EMPTY + sched.idx, sched.phase ^ 1u, kRoleLoadQK)) { aborted = true; break; }
    if (lane == 0) {
      volatile int32_t* p = reinterpret_cast<volatile int32_t*>(c.smem + T::OFF_SCHED + kSlotBytes * sched.idx);
      p[0] = s.valid; p[1] = s.b; p[2] = s.h; p[3] = s.t;
      p[4] = s.q_start; p[5] = s.lq; p[6] = s.k_start; p[7] = s.lk; p[8] = s.split; p[9] = s.v_start;
      if (CAUSAL == kMaskCausalSplit) p[10] = s.koff;
      ptx::mbar_arrive(c.bar(BAR_SCHED_FULL + sched.idx));
    }
    __syncwarp();
    sched.next();
    if (!s.valid) break;
    const Geo g = tile_geo<T, CAUSAL>(s, c.rank);
    const int n1 = g.n[1];
    if (n1 > 0) {
      const int hk = s.h / P.group;
      const int qb = P.packed ? 0 : s.b;
      auto load_q = [&](int i) {
        const uint32_t bar = c.bar(BAR_Q_FULL + i);
        const uint32_t dst = c.sbase + T::OFF_Q + i * T::Q_TILE_BYTES;
        const int row = s.q_start + g.row[i];
        if (lead) ptx::mbar_expect_tx(bar, T::Q_TX);
#pragma unroll
        for (int ch = 0; ch < T::QK_CHUNKS; ++ch)
          load_box<T>(c, dst + ch * T::CHUNK_BYTES, &P.tm_q, bar, ch * T::QK_CHUNK_ELEMS, s.h, row, qb);
        if (T::DR > 0) load_box<T>(c, dst + T::QK_CHUNKS * T::CHUNK_BYTES, &P.tm_qr, bar, 0, s.h, row, qb);
      };
      // Q tile 0, K_0, then Q tile 1: each Q region is refilled as soon as
      // its own last S MMA of the previous work tile is done.
      if (!wait_warp(c, BAR_Q_EMPTY, q_empty_phase ^ 1u, kRoleLoadQK)) { aborted = true; break; }
      if (lane == 0) load_q(0);
      q_fill_parity = q_empty_phase;   // parity of the Q_FULL phases these loads complete
      q_loaded[0] = true;
      q_loaded[1] = false;
      for (int j = 0; j < n1; ++j) {
        if (!wait_warp(c, T::BAR_K_EMPTY + kr.idx, kr.phase ^ 1u, kRoleLoadQK)) { aborted = true; break; }
        if (lane == 0) {
          const uint32_t bar = c.bar(T::BAR_K_FULL + kr.idx);
          const uint32_t dst = c.sbase + T::OFF_K + kr.idx * T::K_STAGE_BYTES;
          // a pair's CTA r holds keys [64 r, 64 r + 64) of the tile
          const int row = s.k_start + kBlockN * j + (T::PAIR ? T::K_ROWS * (int)c.rank : 0);
          if (lead) ptx::mbar_expect_tx(bar, T::K_TX);
#pragma unroll
          for (int ch = 0; ch < T::QK_CHUNKS; ++ch)
            load_box<T>(c, dst + ch * T::K_CHUNK_BYTES, &P.tm_k, bar, ch * T::QK_CHUNK_ELEMS, hk, row, qb);
          if (T::DR > 0) load_box<T>(c, dst + T::QK_CHUNKS * T::K_CHUNK_BYTES, &P.tm_kr, bar, 0, 0, row, qb);
        }
        k_fill_parity[kr.idx] = kr.phase;
        k_used[kr.idx] = true;
        kr.next();
        if (j == 0) {
          if (!wait_warp(c, BAR_Q_EMPTY1, q_empty_phase ^ 1u, kRoleLoadQK)) { aborted = true; break; }
          if (lane == 0) load_q(1);
          q_loaded[1] = true;
          q_empty_phase ^= 1u;
        }
      }
      if (aborted) break;
    }
    // Next work index: from the shared counter (dynamic), one grid stride on
    // (static), or none (one CTA per work tile). A pair's first CTA takes it
    // from the counter and writes it into the second CTA's shared memory.
    if (P.schedule == ATTN_SCHEDULE_DYNAMIC) {
      if (!T::PAIR || lead) {
        int64_t nw = 0;
        if (lane == 0) nw = units + (int64_t)atomicAdd(&c.ws[kWsTileCounter], 1u);
        w = __shfl_sync(kFull, nw, 0);
      }
      if constexpr (T::PAIR) {
        const uint32_t slot = c.sbase + T::OFF_WORK + 8u * fwd.idx;
        if (lead) {
          if (!wait_warp<true>(c, BAR_WORK_EMPTY + fwd.idx, fwd.phase ^ 1u, kRoleLoadQK)) { aborted = true; break; }
          if (lane == 0) {
            ptx::st_cluster_u32(ptx::mapa(slot, 1), (uint32_t)(uint64_t)w);
            ptx::st_cluster_u32(ptx::mapa(slot + 4u, 1), (uint32_t)((uint64_t)w >> 32));
            ptx::mbar_arrive_cluster(ptx::mapa(c.bar(BAR_WORK_FULL + fwd.idx), 1));
          }
        } else {
          if (!wait_warp<true>(c, BAR_WORK_FULL + fwd.idx, fwd.phase, kRoleLoadQK)) { aborted = true; break; }
          const volatile uint32_t* ws = reinterpret_cast<const volatile uint32_t*>(c.smem + T::OFF_WORK + 8 * fwd.idx);
          w = (int64_t)(((uint64_t)ws[1] << 32) | (uint64_t)ws[0]);
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive_cluster(c.bar_lead(BAR_WORK_EMPTY + fwd.idx));
        }
        __syncwarp();
        fwd.next();
      }
    } else if (P.schedule == ATTN_SCHEDULE_STATIC) {
      w += units;
    } else {
      w = INT64_MAX;
    }
  }
  if (aborted && lane == 0) {
    if (lead) {
      // Let every copy this warp issued land before the CTA exits.
#pragma unroll
      for (int s = 0; s < T::NK; ++s)
        if (k_used[s]) wait_drain(c, T::BAR_K_FULL + s, k_fill_parity[s]);
#pragma unroll
      for (int i = 0; i < 2; ++i)
        if (q_loaded[i]) wait_drain(c, BAR_Q_FULL + i, q_fill_parity);
    } else {
      pair_copy_grace();
    }
  }
  __syncwarp();
}

template <class T, int CAUSAL>
__device__ void role_load_v(const Tc05Params& P, const Ctx& c) {
  const int lane = threadIdx.x & 31;
  const bool lead = c.rank == 0;
  Ring<2> sched;
  Ring<T::NV> vr;
  uint32_t v_fill_parity[T::NV];
  bool v_used[T::NV];
#pragma unroll
  for (int s = 0; s < T::NV; ++s) { v_fill_parity[s] = 0; v_used[s] = false; }
  bool first_v = true;
  bool aborted = false;
  while (true) {
    if (!wait_warp(c, BAR_SCHED_FULL + sched.idx, sched.phase, kRoleLoadV)) { aborted = true; break; }
    const SchedSlot s = read_slot<CAUSAL>(c, sched.idx, T::OFF_SCHED);
    if (lane == 0) ptx::mbar_arrive(c.bar(BAR_SCHED_EMPTY + sched.idx));
    sched.next();
    if (!s.valid) break;
    const Geo g = tile_geo<T, CAUSAL>(s, c.rank);
    const int hk = s.h / P.group;
    const int vb = P.packed ? 0 : s.b;
    for (int j = 0; j < g.n[1]; ++j) {
      if (!wait_warp(c, T::BAR_V_EMPTY + vr.idx, vr.phase ^ 1u, kRoleLoadV)) { aborted = true; break; }
      // Fault injection (testing only): block 0 never loads its first V tile,
      // so the MMA issuer's bounded wait for it runs out.
      const bool withhold = P.withhold_v && blockIdx.x == 0 && first_v;
      first_v = false;
      if (lane == 0 && !withhold) {
        const uint32_t bar = c.bar(T::BAR_V_FULL + vr.idx);
        const uint32_t dst = c.sbase + T::OFF_V + vr.idx * T::V_STAGE_BYTES;
        const int row = s.k_start + kBlockN * j;
        if (lead) ptx::mbar_expect_tx(bar, T::V_TX);
        if (T::V8) {
          // depth-major e4m3 V: coordinates (key, depth row, head, batch); the
          // key coordinate is a multiple of 16 (a multiple of 128 for fixed
          // length; packed sequences start on 16-key boundaries of V)
          ptx::tma_load_4d(dst, &P.tm_v, bar, s.v_start + kBlockN * j, 0, hk, vb);
        } else if (T::PAIR) {
          // a pair's CTA r holds depth columns [64 r, 64 r + 64) of the tile
          load_box<T>(c, dst, &P.tm_v, bar, 64 * (int)c.rank, hk, row, vb);
        } else {
#pragma unroll
          for (int ch = 0; ch < T::V_CHUNKS; ++ch)
            ptx::tma_load_4d(dst + ch * T::CHUNK_BYTES, &P.tm_v, bar, ch * 64, hk, row, vb);
        }
      }
      v_fill_parity[vr.idx] = vr.phase;
      v_used[vr.idx] = v_used[vr.idx] || !withhold;
      vr.next();
    }
    if (aborted) break;
  }
  if (aborted && lane == 0) {
    if (lead) {
#pragma unroll
      for (int s = 0; s < T::NV; ++s)
        if (v_used[s]) wait_drain(c, T::BAR_V_FULL + s, v_fill_parity[s]);
    } else {
      pair_copy_grace();
    }
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------------------------
// S_i = Q_i K^T, MMA instructions [B, E) of the K loop (nope part first,
// then the shared rope part).
template <class T, int B, int E>
__device__ __forceinline__ void issue_s(const Ctx& c, int i, uint32_t kstage) {
  constexpr uint32_t HI = ptx::sdesc_hi_sw128(1024);
  const uint32_t d = c.tmem + T::tm_s(i);
  const uint32_t qa = ptx::sdesc_lo(ptx::opaque(c.sbase + T::OFF_Q + i * T::Q_TILE_BYTES), 16);
  const uint32_t ka = ptx::sdesc_lo(ptx::opaque(c.sbase + T::OFF_K + kstage * T::K_STAGE_BYTES), 16);
#pragma unroll
  for (int kk = B; kk < E; ++kk) {
    if (T::FP8) {
      ptx::mma_fp8_ss_lo<HI, HI, T::IDESC_S>(d, qa + kk * 2, ka + kk * 2, kk > 0);
    } else {
      // Q chunks are 128 rows, K chunks K_ROWS rows (64 in a pair)
      const bool rope = kk >= T::DQK / 16;
      const uint32_t qo = (rope ? (T::QK_CHUNKS * T::CHUNK_BYTES + (kk - T::DQK / 16) * 32)
                                : ((kk >> 2) * T::CHUNK_BYTES + (kk & 3) * 32)) >> 4;
      const uint32_t ko = (rope ? (T::QK_CHUNKS * T::K_CHUNK_BYTES + (kk - T::DQK / 16) * 32)
                                : ((kk >> 2) * T::K_CHUNK_BYTES + (kk & 3) * 32)) >> 4;
      if constexpr (T::PAIR) ptx::mma_bf16_ss_lo_pair<HI, HI, T::IDESC_S>(d, qa + qo, ka + ko, kk > 0);
      else ptx::mma_bf16_ss_lo<HI, HI, T::IDESC_S>(d, qa + qo, ka + ko, kk > 0);
    }
  }
}

// O_i += P_i V for keys [64*HALF, 64*HALF + 64) of the tile.
template <class T, int HALF>
__device__ __forceinline__ void issue_pv(const Ctx& c, int i, uint32_t vstage, bool accumulate) {
  constexpr uint32_t HI = ptx::sdesc_hi_sw128(1024);
  const uint32_t d = c.tmem + T::tm_o(i);
  const uint32_t a = c.tmem + T::tm_s(i);   // P: 8 TMEM columns per instruction (16 bf16 / 32 e4m3 keys)
  if (T::V8) {
    // K-major V stage (Dv rows x 128 keys): 32 keys = 32 bytes per instruction
    const uint32_t va = ptx::sdesc_lo(ptx::opaque(c.sbase + T::OFF_V + vstage * T::V_STAGE_BYTES), 16);
#pragma unroll
    for (int kk = 2 * HALF; kk < 2 * HALF + 2; ++kk)
      ptx::mma_fp8_ts_lo<HI, T::IDESC_PV>(d, a + kk * 8, va + kk * 2, (accumulate || kk > 0) ? 1u : 0u);
  } else {
    // MN-major V stage (128 keys x Dv): 16 keys = 2048 bytes per instruction
    const uint32_t va =
        ptx::sdesc_lo(ptx::opaque(c.sbase + T::OFF_V + vstage * T::V_STAGE_BYTES), T::CHUNK_BYTES);
#pragma unroll
    for (int kk = 4 * HALF; kk < 4 * HALF + 4; ++kk) {
      if constexpr (T::PAIR)
        ptx::mma_bf16_ts_lo_pair<HI, T::IDESC_PV>(d, a + kk * 8, va + kk * (2048 >> 4), (accumulate || kk > 0) ? 1u : 0u);
      else
        ptx::mma_bf16_ts_lo<HI, T::IDESC_PV>(d, a + kk * 8, va + kk * (2048 >> 4), (accumulate || kk > 0) ? 1u : 0u);
    }
  }
}

// One MMA-issuing warp per Q tile (warp 12 for tile 0, warp 13 for tile 1).
// Per K/V step g each issues one group, O_i += P_i V_{g-1} then S_i = Q_i K_g^T
// (P_i V first: S_i overwrites the columns holding P_i). The groups of the
// two issuers strictly alternate through a turn token (the forced-ordering
// barriers of the layout page): the tensor core runs tile 0's group while
// tile 1's softmax runs and the other way round. Tile 0, which visits at most
// as many K/V tiles as tile 1, pads with empty groups so that the
// alternation never has to wait for the next work tile. K, V and Q stages are
// released by one commit from each issuer.
// Commit of the issuing thread's MMAs to barrier `id`: in a pair, to that
// barrier in both CTAs (ALL) or in the first CTA only.
template <class T, bool ALL = true>
__device__ __forceinline__ void commit(const Ctx& c, int id) {
  if constexpr (T::PAIR) ptx::mma_commit_pair(c.bar(id), ALL ? (uint16_t)3 : (uint16_t)1);
  else ptx::mma_commit(c.bar(id));
}

template <class T, int CAUSAL>
__device__ void role_mma(const Tc05Params& P, const Ctx& c, const int i) {
  // Runs on lane 0 of warp 12 + i only (in a pair: of the first CTA): one
  // thread issues, waits and commits.
  const int role = kRoleMma;
  Ring<2> sched;
  Ring<T::NK> kr;   // stage of the next K tile
  Ring<T::NV> vr;   // stage of the next V tile
  uint32_t q_full_phase = 0, p_phase = 0, ofree_phase = 0, order_phase = 0;
  // Issuer 0 takes the first turn: its first wait passes on the fresh barrier.
  const uint32_t order_flip = i == 0 ? 1u : 0u;
  bool aborted = false;
#define AF_WAIT(id, par)                   \
  if (!wait_one(c, (id), (par), role)) {   \
    aborted = true;                        \
    break;                                 \
  }
  // barriers that the peer CTA of a pair arrives on
#define AF_WAIT_CL(id, par)                         \
  if (!wait_one<T::PAIR>(c, (id), (par), role)) {   \
    aborted = true;                                 \
    break;                                          \
  }
  while (true) {
    if (!wait_one(c, BAR_SCHED_FULL + sched.idx, sched.phase, role)) { aborted = true; break; }
    const SchedSlot s = read_slot<CAUSAL>(c, sched.idx, T::OFF_SCHED);
    ptx::mbar_arrive(c.bar(BAR_SCHED_EMPTY + sched.idx));
    sched.next();
    if (!s.valid) break;
    const Geo g = tile_geo<T, CAUSAL>(s, c.rank);
    const int n = g.n[i], n1 = g.n[1];
    if (n1 == 0) {
      // No keys: keep the per-tile O-free handshake in step with the epilogue.
      AF_WAIT_CL(BAR_O_FREE + i, ofree_phase ^ 1u);
      ofree_phase ^= 1u;
      continue;
    }
    AF_WAIT(BAR_Q_FULL + i, q_full_phase);
    q_full_phase ^= 1u;
    for (int grp = 0; grp <= n1; ++grp) {
      const bool has_pv = grp >= 1 && grp <= n;
      const bool has_s = grp < n;
      // Operands that are usually ready first, then the turn, the softmax's
      // first half of P last: once it lands the issuer goes straight to
      // issuing (each barrier check costs this thread ~100-200 cycles while
      // the softmax warps keep tensor and shared memory busy).
      if (has_pv) {
        if (grp == 1) {
          AF_WAIT_CL(BAR_O_FREE + i, ofree_phase ^ 1u);
          ofree_phase ^= 1u;
        }
        AF_WAIT(T::BAR_V_FULL + vr.idx, vr.phase);
      }
      if (has_s) AF_WAIT(T::BAR_K_FULL + kr.idx, kr.phase);
      if (!wait_one(c, BAR_ORDER + i, order_phase ^ order_flip, role)) { aborted = true; break; }
      order_phase ^= 1u;
      if (has_pv) AF_WAIT_CL(BAR_P_LO + i, p_phase);
      ptx::tc_fence_after();
      if (has_pv) {
        issue_pv<T, 0>(c, i, vr.idx, grp > 1);
        AF_WAIT_CL(BAR_P_HI + i, p_phase);
        p_phase ^= 1u;
        ptx::tc_fence_after();
        issue_pv<T, 1>(c, i, vr.idx, true);
        commit<T>(c, T::BAR_V_EMPTY + vr.idx);
        if (grp == n) commit<T>(c, BAR_O_FINAL + i);
        vr.next();
      }
      if (has_s) {
        // Hand the turn over before the last S_AFTER_HANDOFF instructions, so
        // the other issuer's wake-up overlaps their execution.
        issue_s<T, 0, T::S_INSTR - T::S_AFTER_HANDOFF>(c, i, kr.idx);
        ptx::mbar_arrive(c.bar(BAR_ORDER + (i ^ 1)));
        issue_s<T, T::S_INSTR - T::S_AFTER_HANDOFF, T::S_INSTR>(c, i, kr.idx);
        commit<T>(c, BAR_S_FULL + i);
        commit<T>(c, T::BAR_K_EMPTY + kr.idx);
        if (grp == n - 1) commit<T>(c, Ctx::q_empty_id(i));
        kr.next();
      } else {
        ptx::mbar_arrive(c.bar(BAR_ORDER + (i ^ 1)));   // the other issuer's turn
      }
      if (!has_pv && !has_s) {
        // A K/V tile only the other Q tile visits: release this issuer's share.
        AF_WAIT(T::BAR_K_FULL + kr.idx, kr.phase);
        commit<T>(c, T::BAR_K_EMPTY + kr.idx);
        kr.next();
        AF_WAIT(T::BAR_V_FULL + vr.idx, vr.phase);
        commit<T>(c, T::BAR_V_EMPTY + vr.idx);
        vr.next();
      }
    }
    if (aborted) break;
  }
#undef AF_WAIT
#undef AF_WAIT_CL
  // Drain: the arrive of this commit follows every MMA and commit this thread
  // issued (both issuers commit; the phase completes after both).
  commit<T, false>(c, BAR_DRAIN);
  wait_drain(c, BAR_DRAIN, 0);
  (void)aborted;
}

// ---------------------------------------------------------------------------------------------
template <class T, int CAUSAL>
__device__ void role_softmax(const Tc05Params& P, const Ctx& c, const int i) {
  const int tid = threadIdx.x - 128 * i;          // row of the Q tile == TMEM lane
  const uint32_t lane_base = (uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16;
  const uint32_t tS = c.tmem + lane_base + T::tm_s(i);
  const uint32_t tO = c.tmem + lane_base + T::tm_o(i);
  float* rcpl_sm = reinterpret_cast<float*>(c.smem + T::OFF_RCPL) + i * kBlockM;
  float* ks_sm = reinterpret_cast<float*>(c.smem + T::OFF_KS) + i * 2 * kBlockN;
  const int role = i == 0 ? kRoleSoftmax0 : kRoleSoftmax1;
  Ring<2> sched;
  uint32_t s_phase = 0, ks_phase = 0, stats_phase = 0, turn_phase = 0;
  const uint32_t turn_flip = i == 0 ? 1u : 0u;   // warpgroup 0 takes the first turn
  while (true) {
    if (!wait_warp(c, BAR_SCHED_FULL + sched.idx, sched.phase, role)) return;
    const SchedSlot s = read_slot<CAUSAL>(c, sched.idx, T::OFF_SCHED);
    ptx::mbar_arrive(c.bar(BAR_SCHED_EMPTY + sched.idx));
    sched.next();
    if (!s.valid) return;
    const Geo g = tile_geo<T, CAUSAL>(s, c.rank);
    const int n = g.n[i];
    const int qi = g.row[i] + tid;               // row within the sequence
    const bool row_valid = qi < s.lq;
    // keys of the range visible to this row (causal: keys 0..qi of the
    // sequence, the range starting at key koff of it)
    const int lim = (CAUSAL & kMaskCausal) ? min(s.lk, qi + 1 - s.koff) : s.lk;
    const int first_row = g.row[i];
    // LSE element: [B][Hq][Sq] (or [Hq][Tq] packed); a split-KV range writes
    // its partial LSE to copy `split` of that layout, [split][B][Hq][Sq] (or
    // [split][Hq][Tq]).
    const bool split_kv = splits_keys<CAUSAL>(P);
    const int sp = split_kv ? s.split : 0;
    const int64_t lse_idx = P.packed ? ((int64_t)sp * P.heads_q + s.h) * P.total_q + s.q_start + qi
                                     : (((int64_t)sp * P.batch + s.b) * P.heads_q + s.h) * P.seqlen_q + qi;
    float c_row = P.scale_log2;
    int64_t ks_base = 0;
    if (T::FP8) {
      const int hk = s.h / P.group;
      float qs = 1.f;
      if (row_valid)
        qs = P.packed ? P.q_scale[(int64_t)s.h * P.total_q + s.q_start + qi]
                      : P.q_scale[((int64_t)s.b * P.heads_q + s.h) * P.seqlen_q + qi];
      c_row *= qs;
      ks_base = P.packed ? (int64_t)hk * P.total_k + s.k_start
                         : ((int64_t)s.b * P.heads_kv + hk) * P.seqlen_k + s.k_start;
    }
    float ks_next = 0.f;
    if (T::FP8 && n > 0) ks_next = tid < s.lk ? __ldg(P.k_scale + ks_base + tid) : 0.f;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < n; ++j) {
      const int kb = kBlockN * j;
      if (T::FP8) {
        ks_sm[(j & 1) * kBlockN + tid] = ks_next;
        ptx::mbar_arrive(c.bar(BAR_KS + i));
        if (!wait_warp(c, BAR_KS + i, ks_phase, role)) return;
        ks_phase ^= 1u;
        if (j + 1 < n) ks_next = (kb + kBlockN + tid < s.lk) ? __ldg(P.k_scale + ks_base + kb + kBlockN + tid) : 0.f;
      }
      if (!wait_warp(c, BAR_S_FULL + i, s_phase, role)) return;
      s_phase ^= 1u;
      if (T::SM_TURN) {
        if (!wait_warp(c, BAR_SM_TURN + i, turn_phase ^ turn_flip, role)) return;
        turn_phase ^= 1u;
      }
      ptx::tc_fence_after();
      float sv[128];
      {
        uint32_t r[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) ptx::tmem_ld32(tS + 32 * q, r[q]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int e = 0; e < 32; ++e) sv[32 * q + e] = __uint_as_float(r[q][e]);
      }
      if (T::FP8) {
        const float2* k2 = reinterpret_cast<const float2*>(ks_sm + (j & 1) * kBlockN);
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const float2 kv = k2[e];
          float a0, a1;
          ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(sv[2 * e], sv[2 * e + 1]), ptx::f2_pack(kv.x, kv.y)), a0, a1);
          sv[2 * e] = a0;
          sv[2 * e + 1] = a1;
        }
      }
      const bool need_mask = (kb + kBlockN > s.lk) || ((CAUSAL & kMaskCausal) && s.koff + kb + kBlockN - 1 > first_row);
      if (need_mask) {
        const int vis = lim - kb;
        if constexpr (T::V8) {
          // one compare per key (measured 5 % faster here than the per-chunk
          // bit pattern below, which is ~1 % faster in the other variants)
#pragma unroll
          for (int e = 0; e < 128; ++e)
            if (e >= vis) sv[e] = -INFINITY;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int vq = min(max(vis - 32 * q, 0), 32);
            const uint32_t bits = vq >= 32 ? 0xffffffffu : ((1u << vq) - 1u);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (!((bits >> e) & 1u)) sv[32 * q + e] = -INFINITY;
          }
        }
      }
      float mx0 = ptx::max3(sv[0], sv[1], sv[2]), mx1 = ptx::max3(sv[3], sv[4], sv[5]);
      float mx2 = ptx::max3(sv[6], sv[7], sv[8]), mx3 = ptx::max3(sv[9], sv[10], sv[11]);
#pragma unroll
      for (int e = 12; e < 124; e += 8) {
        mx0 = ptx::max3(mx0, sv[e], sv[e + 1]);
        mx1 = ptx::max3(mx1, sv[e + 2], sv[e + 3]);
        mx2 = ptx::max3(mx2, sv[e + 4], sv[e + 5]);
        mx3 = ptx::max3(mx3, sv[e + 6], sv[e + 7]);
      }
      mx0 = ptx::max3(mx0, sv[124], sv[125]);
      mx1 = ptx::max3(mx1, sv[126], sv[127]);
      const float mx = ptx::max3(mx0, mx1, fmaxf(mx2, mx3)) * c_row;
      const float m_new = fmaxf(m, mx);
      float m_use = m, alpha = 1.f;
      if (j == 0) {
        m_use = m_new;
      } else if (m_new > m + 8.f) {
        m_use = m_new;
        alpha = ptx::ex2(m - m_new);
      }
      const uint64_t c2 = ptx::f2_pack(c_row, c_row);
      const uint64_t n2 = ptx::f2_pack(-m_use, -m_use);
      uint64_t acc0 = 0, acc1 = 0;   // (+0.0f, +0.0f) pairs
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // P for keys [64*half, 64*half + 64) -> 32 packed bf16 pairs (or 16
        // e4m3 quads).
        uint32_t pk[T::P_COLS_HALF];
        [[maybe_unused]] float q0 = 0.f, q1 = 0.f;   // e4m3: the previous pair of the quad
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int el = 64 * half + 2 * e;
          float x0, x1;
          ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(sv[el], sv[el + 1]), c2, n2), x0, x1);
          const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
          if (e & 1) acc1 = ptx::f2_add(acc1, ptx::f2_pack(p0, p1));
          else acc0 = ptx::f2_add(acc0, ptx::f2_pack(p0, p1));
          if constexpr (T::V8) {
            if (e & 1) pk[e >> 1] = ptx::pack_e4m3x4(q0, q1, p0, p1);
            q0 = p0;
            q1 = p1;
          } else {
            pk[e] = ptx::pack_bf16(p0, p1);
          }
        }
        if constexpr (T::V8) ptx::tmem_st16(tS + T::P_COLS_HALF * half, pk);
        else ptx::tmem_st32(tS + T::P_COLS_HALF * half, pk);
        if (half == 0 && __any_sync(kFull, alpha != 1.f)) {
          // Correction: the running max moved (rare with the 2^8 headroom), so
          // rescale this warp's rows of O_i before the next P V accumulates
          // into it. P_i(j-1) V was complete when S_i(j) arrived (same issuer,
          // in order).
#pragma unroll 1
          for (int q = 0; q < T::DV / 32; ++q) {
            uint32_t r[32];
            ptx::tmem_ld32(tO + 32 * q, r);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            ptx::tmem_st32(tO + 32 * q, r);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        if constexpr (T::PAIR) {
          // one arrival per warp on the first CTA's barrier
          __syncwarp();
          if ((threadIdx.x & 31) == 0) arrive_lead(c, (half == 0 ? BAR_P_LO : BAR_P_HI) + i);
        } else {
          ptx::mbar_arrive(c.bar((half == 0 ? BAR_P_LO : BAR_P_HI) + i));
        }
        if (T::SM_TURN == half + 1) ptx::mbar_arrive(c.bar(BAR_SM_TURN + (i ^ 1)));   // the other warpgroup's turn
      }
      float s0, s1, s2, s3;
      ptx::f2_unpack(acc0, s0, s1);
      ptx::f2_unpack(acc1, s2, s3);
      l = l * alpha + ((s0 + s1) + (s2 + s3));
      m = m_use;
    }
    if (T::SM_TURN) {
      // K/V tiles only the other Q tile visits: pass the turn on.
      for (int j = n; j < g.n[1]; ++j) {
        if (!wait_warp(c, BAR_SM_TURN + i, turn_phase ^ turn_flip, role)) return;
        turn_phase ^= 1u;
        ptx::mbar_arrive(c.bar(BAR_SM_TURN + (i ^ 1)));
      }
    }
    // Row statistics: LSE (natural log) here, 1/l to the epilogue. A split-KV
    // range writes the LSE of its own keys for the merge.
    float* const lse_dst = splits_keys<CAUSAL>(P) ? P.lse_part : P.lse;
    if (row_valid && lse_dst != nullptr) {
      const float lse = l > 0.f ? (m + ptx::lg2(l)) * 0.69314718055994531f : -INFINITY;
      lse_dst[lse_idx] = lse;
    }
    if (!wait_warp(c, BAR_STATS_FREE + i, stats_phase ^ 1u, role)) return;
    stats_phase ^= 1u;
    rcpl_sm[tid] = l > 0.f ? 1.f / l : 0.f;
    ptx::mbar_arrive(c.bar(BAR_STATS + i));
  }
}

// ---------------------------------------------------------------------------------------------
// 32 columns of one O row (64 bytes) as bf16: two 32-byte stores when O is
// 32-byte aligned (whole sectors per instruction), else four 16-byte ones.
template <class T>
__device__ __forceinline__ void store_row_chunk(uint16_t* dst, const uint32_t (&r)[32], float scale, bool wide) {
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e)
    pk[e] = ptx::pack_bf16(__uint_as_float(r[2 * e]) * scale, __uint_as_float(r[2 * e + 1]) * scale);
  if (wide) {
    ptx::st_global_v8(dst, pk);
    ptx::st_global_v8(dst + 16, pk + 8);
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int e = 0; e < 4; ++e) d[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
  }
}

// Split-KV: row of the partial O array [split][rows][Hq] (rows = B*Sq, or Tq
// when packed) of query row qi of work tile s.
__device__ __forceinline__ int64_t partial_row(const Tc05Params& P, const SchedSlot& s, int qi) {
  const int64_t rows = P.packed ? (int64_t)P.total_q : (int64_t)P.batch * P.seqlen_q;
  const int64_t row = P.packed ? (int64_t)s.q_start + qi : (int64_t)s.b * P.seqlen_q + qi;
  return ((int64_t)s.split * rows + row) * P.heads_q + s.h;
}

// Split-KV: one 32-column chunk of a row of normalised partial O, in fp32,
// as four 32-byte stores (partial rows are 32-byte aligned in the workspace).
__device__ __forceinline__ void store_row_chunk_f32(float* dst, const uint32_t (&r)[32], float scale) {
  uint32_t v[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(r[e]) * scale);
#pragma unroll
  for (int e = 0; e < 4; ++e) ptx::st_global_v8(dst + 8 * e, v + 8 * e);
}

template <class T, int CAUSAL>
__device__ void role_correction(const Tc05Params& P, const Ctx& c) {
  const int tid = threadIdx.x - 256;
  const uint32_t lane_base = (uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16;
  const float* rcpl_sm = reinterpret_cast<const float*>(c.smem + T::OFF_RCPL);
  Ring<2> sched;
  uint32_t stats_phase[2] = {0, 0}, ofinal_phase[2] = {0, 0};
  while (true) {
    if (!wait_warp(c, BAR_SCHED_FULL + sched.idx, sched.phase, kRoleCorrection)) return;
    const SchedSlot s = read_slot<CAUSAL>(c, sched.idx, T::OFF_SCHED);
    ptx::mbar_arrive(c.bar(BAR_SCHED_EMPTY + sched.idx));
    sched.next();
    if (!s.valid) return;
    const Geo g = tile_geo<T, CAUSAL>(s, c.rank);
#pragma unroll 1
    for (int i = 0; i < 2; ++i) {
      // Epilogue of Q tile i: O = O / l, rounded once to bf16, stored row by row.
      if (!wait_warp(c, BAR_STATS + i, stats_phase[i], kRoleCorrection)) return;
      stats_phase[i] ^= 1u;
      const float rl = rcpl_sm[i * kBlockM + tid];
      ptx::mbar_arrive(c.bar(BAR_STATS_FREE + i));
      const int qi = g.row[i] + tid;
      const bool row_valid = qi < s.lq;
      uint16_t* orow = P.o + (int64_t)s.b * P.o_stride_b + (int64_t)(s.q_start + qi) * P.o_stride_t +
                       (int64_t)s.h * P.o_stride_h;
      if (g.n[i] > 0) {
        if (!wait_warp(c, BAR_O_FINAL + i, ofinal_phase[i], kRoleCorrection)) return;
        ofinal_phase[i] ^= 1u;
        ptx::tc_fence_after();
        const uint32_t tO = c.tmem + lane_base + T::tm_o(i);
        if (splits_keys<CAUSAL>(P)) {
          // Split-KV range: normalised partial O in fp32 for the merge.
          float* prow = P.o_part + partial_row(P, s, qi) * T::DV;
#pragma unroll 1
          for (int q = 0; q < T::DV / 32; ++q) {
            uint32_t r[32];
            ptx::tmem_ld32(tO + 32 * q, r);
            ptx::tmem_wait_ld();
            if (row_valid) store_row_chunk_f32(prow + 32 * q, r, rl);
          }
        } else {
#pragma unroll
          for (int q = 0; q < T::DV / 32; ++q) {
            uint32_t r[32];
            ptx::tmem_ld32(tO + 32 * q, r);
            ptx::tmem_wait_ld();
            if (row_valid) store_row_chunk<T>(orow + 32 * q, r, rl, P.o_store32 != 0);
          }
        }
      } else if (row_valid && splits_keys<CAUSAL>(P)) {
        // An empty key range (a short packed sequence, or under the causal
        // mask a range this tile's rows do not reach): a zero partial row
        // (its LSE is -inf, so the merge gives it no weight).
        float4* d = reinterpret_cast<float4*>(P.o_part + partial_row(P, s, qi) * T::DV);
#pragma unroll 1
        for (int e = 0; e < T::DV / 4; ++e) d[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else if (row_valid) {
        uint4* d = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int e = 0; e < T::DV / 8; ++e) d[e] = make_uint4(0u, 0u, 0u, 0u);
      }
      ptx::tc_fence_before();
      if constexpr (T::PAIR) {
        // one arrival per warp on the first CTA's barrier (its MMAs write both CTAs' O)
        __syncwarp();
        if ((threadIdx.x & 31) == 0) arrive_lead(c, BAR_O_FREE + i);
      } else {
        ptx::mbar_arrive(c.bar(BAR_O_FREE + i));
      }
    }
  }
}

// ---------------------------------------------------------------------------------------------
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <class T, int CAUSAL>
__global__ void __launch_bounds__(512, 1) fa_tc05_kernel(const __grid_constant__ Tc05Params P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctx c;
  c.smem = smem;
  c.sbase = ptx::smem_u32(smem);
  c.ws = P.ws;
  c.abort_flag = reinterpret_cast<volatile int*>(smem + T::OFF_ABORT);
  c.bar_off = T::OFF_BAR;
  c.timeout_ns = P.timeout_ns;
  c.rank = T::PAIR ? ptx::cluster_ctarank() : 0u;
  c.peer_abort = 0u;
  if (c.sbase & 1023u) {  // the swizzled tiles need a 1024-byte aligned base (same in both CTAs of a pair)
    if constexpr (!T::FP8) ptx::grid_dependency_wait();
    if (threadIdx.x == 0) atomicCAS(&P.ws[kWsErrorCode], 0u, 2u);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Barriers that the second CTA of a pair reports to per warp (4 warps per CTA).
  const uint32_t warp_count = T::PAIR ? 8u : 128u;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(c.bar(BAR_Q_FULL + i), 1);
      ptx::mbar_init(c.bar(BAR_S_FULL + i), 1);
      ptx::mbar_init(c.bar(BAR_P_LO + i), warp_count);
      ptx::mbar_init(c.bar(BAR_STATS + i), 128);
      ptx::mbar_init(c.bar(BAR_P_HI + i), warp_count);
      ptx::mbar_init(c.bar(BAR_ORDER + i), 1);
      ptx::mbar_init(c.bar(BAR_O_FINAL + i), 1);
      ptx::mbar_init(c.bar(BAR_O_FREE + i), warp_count);
      ptx::mbar_init(c.bar(BAR_STATS_FREE + i), 128);
      ptx::mbar_init(c.bar(BAR_KS + i), 128);
      ptx::mbar_init(c.bar(BAR_SCHED_FULL + i), 1);
      // a pair's second CTA runs no MMA issuers
      ptx::mbar_init(c.bar(BAR_SCHED_EMPTY + i), kSchedConsumers - (c.rank != 0 ? 2u : 0u));
      ptx::mbar_init(c.bar(BAR_WORK_FULL + i), 1);
      ptx::mbar_init(c.bar(BAR_WORK_EMPTY + i), 1);
      ptx::mbar_init(c.bar(BAR_SM_TURN + i), 128);
    }
    ptx::mbar_init(c.bar(BAR_Q_EMPTY), 1);
    ptx::mbar_init(c.bar(BAR_Q_EMPTY1), 1);
    ptx::mbar_init(c.bar(BAR_DRAIN), 2);
#pragma unroll
    for (int s = 0; s < T::NK; ++s) {
      ptx::mbar_init(c.bar(T::BAR_K_FULL + s), 1);
      ptx::mbar_init(c.bar(T::BAR_K_EMPTY + s), 2);
    }
#pragma unroll
    for (int s = 0; s < T::NV; ++s) {
      ptx::mbar_init(c.bar(T::BAR_V_FULL + s), 1);
      ptx::mbar_init(c.bar(T::BAR_V_EMPTY + s), 2);
    }
    *c.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 12) {
    if constexpr (T::PAIR) {
      ptx::tmem_alloc_pair(c.sbase + T::OFF_TMEM_SLOT, T::TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(c.sbase + T::OFF_TMEM_SLOT, T::TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  if (warp == 14 && lane == 0) {
    ptx::prefetch_tmap(&P.tm_q);
    ptx::prefetch_tmap(&P.tm_k);
    ptx::prefetch_tmap(&P.tm_v);
    if (T::DR > 0) {
      ptx::prefetch_tmap(&P.tm_qr);
      ptx::prefetch_tmap(&P.tm_kr);
    }
  }
  ptx::tc_fence_before();
  // A pair's barriers must be initialised in both CTAs before either CTA
  // copies into, or arrives on, the other's.
  __syncwarp();
  if constexpr (T::PAIR) ptx::cluster_sync();
  else __syncthreads();
  ptx::tc_fence_after();
  c.tmem = *reinterpret_cast<volatile uint32_t*>(smem + T::OFF_TMEM_SLOT);
  if constexpr (T::PAIR) c.peer_abort = ptx::mapa(c.sbase + T::OFF_ABORT, c.rank ^ 1u);
  // The set-up above touches no global memory, so it may overlap the
  // previous kernel on the stream (programmatic dependent launch); from here
  // on the kernel reads inputs and writes outputs and the workspace, so it
  // waits until that kernel has completed and its writes are visible. (The
  // FP8 variants are never launched that way: any added code in them
  // measured ~1 % slower, their softmax being at its register ceiling.)
  if constexpr (!T::FP8) ptx::grid_dependency_wait();   // returns at once without a dependency

  const int wg = warp >> 2;
  if (wg < 2) {
    setmaxnreg_inc<T::REG_SOFTMAX>();
    role_softmax<T, CAUSAL>(P, c, wg);
  } else if (wg == 2) {
    setmaxnreg_dec<T::REG_CORR>();
    role_correction<T, CAUSAL>(P, c);
  } else {
    setmaxnreg_dec<T::REG_MISC>();
    if (warp == 12 || warp == 13) {
      if (lane == 0 && c.rank == 0) role_mma<T, CAUSAL>(P, c, warp - 12);
      __syncwarp();
    }
    else if (warp == 14) role_load_qk<T, CAUSAL>(P, c);
    else role_load_v<T, CAUSAL>(P, c);
  }

  ptx::tc_fence_before();
  // Both CTAs of a pair are done with the MMAs (which use both CTAs' tensor
  // and shared memory) before either frees its tensor memory or exits.
  __syncwarp();
  if constexpr (T::PAIR) ptx::cluster_sync();
  else __syncthreads();
  if (warp == 12) {
    ptx::tc_fence_after();
    if constexpr (T::PAIR) ptx::tmem_dealloc_pair(c.tmem, T::TMEM_COLS);
    else ptx::tmem_dealloc(c.tmem, T::TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&P.ws[kWsDoneCounter], 1u) == gridDim.x - 1) {
      atomicExch(&P.ws[kWsTileCounter], 0u);
      atomicExch(&P.ws[kWsDoneCounter], 0u);
      __threadfence();
    }
  }
}

// Launch configuration of a pair variant: clusters of two CTAs.
template <class T>
cudaLaunchConfig_t pair_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(512, 1, 1);
  cfg.dynamicSmemBytes = T::SMEM_BYTES;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Raises a kernel's dynamic shared-memory limit once per device (the
// attribute stays set for the life of the context); `force` sets it again
// (after a context was torn down and recreated).
template <auto KERN>
cudaError_t set_smem_once(int bytes, bool force = false) {
  static std::atomic<uint64_t> done{0};   // one per kernel
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (!force && bit != 0ull && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0ull) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launches `launch()`; if that fails, sets the kernel's shared-memory limit
// again and retries once.
template <auto KERN, class F>
cudaError_t launch_with_smem(int bytes, F launch) {
  cudaError_t e = set_smem_once<KERN>(bytes);
  if (e != cudaSuccess) return e;
  e = launch();
  if (e == cudaSuccess) return e;
  if ((e = set_smem_once<KERN>(bytes, true)) != cudaSuccess) return e;
  return launch();
}

template <class T, int CAUSAL>
cudaError_t tc05_launch_tc(const Tc05Params& prm, int grid, cudaStream_t stream) {
  constexpr auto kern = fa_tc05_kernel<T, CAUSAL>;
  return launch_with_smem<kern>(T::SMEM_BYTES, [&]() -> cudaError_t {
    if constexpr (T::PAIR) {
      if (grid % 2 != 0) return cudaErrorInvalidValue;
      cudaLaunchAttribute attr[1];
      const cudaLaunchConfig_t cfg = pair_config<T>(grid, stream, attr);
      const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, prm);
      if (e != cudaSuccess) return e;
    } else if (T::FP8 || !prm.dependent_launch) {
      kern<<<grid, 512, T::SMEM_BYTES, stream>>>(prm);
    } else {
      // programmatic dependent launch: set-up overlaps the previous kernel's
      // last CTAs (the kernel waits before its first global access)
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)grid);
      cfg.blockDim = dim3(512);
      cfg.dynamicSmemBytes = T::SMEM_BYTES;
      cfg.stream = stream;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, prm);
      if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
  });
}

template <class T>
cudaError_t tc05_launch_t(int mask, const Tc05Params& prm, int grid, cudaStream_t stream) {
  if (mask == kMaskNone) return tc05_launch_tc<T, kMaskNone>(prm, grid, stream);
  if (mask == kMaskCausal) return tc05_launch_tc<T, kMaskCausal>(prm, grid, stream);
  if (mask == kMaskNoneSplit) return tc05_launch_tc<T, kMaskNoneSplit>(prm, grid, stream);
  if constexpr (!T::PAIR) {
    if (mask == kMaskCausalSplit) return tc05_launch_tc<T, kMaskCausalSplit>(prm, grid, stream);
  }
  return cudaErrorInvalidValue;
}

// Clusters of a pair variant that can be resident at once on the current
// device (0 if the query fails or the variant is not a pair variant).
template <class T>
int tc05_max_clusters_t() {
  if constexpr (!T::PAIR) {
    return 0;
  } else {
    auto kern = fa_tc05_kernel<T, kMaskCausal>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pair_config<T>(2, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n;
  }
}

template <class T>
Tc05Config tc05_config_t() {
  Tc05Config c;
  c.smem_bytes = T::SMEM_BYTES;
  c.k_stages = T::NK;
  c.v_stages = T::NV;
  c.threads = 512;
  c.tmem_cols = (int)T::TMEM_COLS;
  return c;
}

using TraitsD64 = Tc05Traits<64, 0, 64, false>;
using TraitsD128 = Tc05Traits<128, 0, 128, false>;
using TraitsD128R64 = Tc05Traits<128, 64, 128, false>;
using TraitsFp8D128 = Tc05Traits<128, 0, 128, true>;
using TraitsFp8QkvD128 = Tc05Traits<128, 0, 128, true, true>;
using TraitsD128Pair = Tc05Traits<128, 0, 128, false, false, true>;
using TraitsD128R64Pair = Tc05Traits<128, 64, 128, false, false, true>;

cudaError_t tc05_launch_d64(int mask, const Tc05Params& prm, int grid, cudaStream_t stream);
cudaError_t tc05_launch_d128(int mask, const Tc05Params& prm, int grid, cudaStream_t stream);
cudaError_t tc05_launch_d128r64(int mask, const Tc05Params& prm, int grid, cudaStream_t stream);
cudaError_t tc05_launch_fp8d128(int mask, const Tc05Params& prm, int grid, cudaStream_t stream);
cudaError_t tc05_launch_fp8qkvd128(int mask, const Tc05Params& prm, int grid, cudaStream_t stream);
cudaError_t tc05_launch_d128pair(int mask, const Tc05Params& prm, int grid, cudaStream_t stream);
cudaError_t tc05_launch_d128r64pair(int mask, const Tc05Params& prm, int grid, cudaStream_t stream);
int tc05_max_clusters_d128pair();
int tc05_max_clusters_d128r64pair();

}  // namespace af
