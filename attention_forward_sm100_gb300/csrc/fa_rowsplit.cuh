// Row-split attention forward for e4m3 Q/K on sm_103a (tcgen05 + TMA).
//
// With FP8 Q/K a K/V step's MMAs take less time than the softmax of one
// 128 x 128 score tile, so the two-Q-tile ping-pong of fa_tc05.cuh leaves the
// tensor core waiting on the softmax. This kernel rebuilds the pipeline
// around that:
//   * a work tile is one 128-row Q tile (M = 128 MMAs);
//   * S is double-buffered in tensor memory (columns [0,128) and [128,256),
//     O in [256,384)): the MMA issuer computes S(j+1) while the softmax works
//     on S(j), and issues O += P(j) V(j) as soon as P(j) is published; P(j)
//     overwrites S(j)'s buffer (bf16 pairs, or e4m3 quads for e4m3 V);
//   * the softmax of every row is split over two warpgroups: warpgroup g
//     owns the keys [64 g, 64 g + 64) of each tile for all 128 rows, so each
//     thread handles 64 scores. The two halves of a row exchange their
//     maxima through shared memory once per tile (one mbarrier per 32-row
//     quarter) and their sums once per work tile, so both use the same
//     running maximum and the lazy 2^8 rescale of O stays exact; a rescale is
//     split by columns of O and waits for the previous P V to complete;
//   * the Q/K producer also delivers each K tile's 128 per-token k-scales
//     into a shared-memory slot beside the K stage (4-byte cp.async copies
//     that complete on the slot's mbarrier), released by the softmax warps.
// Roles: warps 0-3 / 4-7 softmax halves, 8-11 epilogue (O / l -> bf16, or
// the fp32 split-KV partial), warp 12 lane 0 the MMA issuer (warp 12 also
// owns tensor memory), warp 14 scheduler + Q/K/k-scale producer, warp 15 V
// producer. Scheduling, split-KV ranges, bounded waits and the abort path
// are those of fa_tc05.cuh.
#pragma once
#include "fa_tc05.cuh"

namespace af {

enum RsBar : int {
  RB_Q_FULL = 0,        // +slot (2), Q tile landed
  RB_Q_EMPTY = 2,       // +slot, last S MMA of that Q tile done
  RB_S_FULL = 4,        // +buffer (2), S in that tensor-memory buffer
  // P barriers come in one pair per S buffer: the rows of one 32-row quarter
  // can start step j + 1 (its S is already computed) before another quarter
  // has published P of step j, and those arrivals must not count for step j.
  RB_P_LO = 6,          // +buffer, keys 0..63 of P stored (warpgroup 0) and warpgroup 1's part of any O rescale done (256)
  RB_P_HI = 8,          // +buffer, keys 64..127 of P stored (warpgroup 1, 128)
  RB_O_READY = 10,      // one phase per P V instruction group
  RB_O_FINAL = 11,      // last P V of a work tile
  RB_O_FREE = 12,       // epilogue read O (128)
  RB_STATS = 13,        // 1/l of the work tile in shared memory (128)
  RB_STATS_FREE = 14,   // epilogue read 1/l (128)
  RB_XCH = 15,          // +quarter (4), exchange between the two halves of rows [32q, 32q + 32) (64)
  RB_SCHED_FULL = 19,   // +slot
  RB_SCHED_EMPTY = 21,  // +slot
  RB_DRAIN = 23,        // final commit of the MMA thread
  RB_FIXED = 24         // then K_FULL[NK], K_EMPTY[NK], KS_FULL[NK], KS_EMPTY[NK], V_FULL[NV], V_EMPTY[NV]
};

// Consumers of a scheduler slot: the MMA lane, both softmax halves, the
// epilogue warpgroup and the V producer lane.
constexpr uint32_t kRsSchedConsumers = 1 + 128 + 128 + 128 + 1;

template <bool V8_>
struct RsTraits {
  static constexpr bool V8 = V8_;   // e4m3 V (depth-major), P rounded to e4m3
  static constexpr int DQK = 128, DV = 128;
  static constexpr int ROWS = kBlockM;                 // rows of one work tile
  static constexpr int CHUNK_BYTES = 128 * 128;
  static constexpr int Q_BYTES = CHUNK_BYTES;          // 128 rows x 128 e4m3
  static constexpr int K_STAGE_BYTES = CHUNK_BYTES;    // 128 keys x 128 e4m3
  static constexpr int V_STAGE_BYTES = V8 ? CHUNK_BYTES : 2 * CHUNK_BYTES;
  static constexpr int NK = 4, NV = V8 ? 5 : 3;
  static constexpr int OFF_Q = 0;                                       // 2 slots
  static constexpr int OFF_K = 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NK * K_STAGE_BYTES;
  static constexpr int OFF_KS = OFF_V + NV * V_STAGE_BYTES;             // float [NK][128]
  static constexpr int OFF_XM = OFF_KS + NK * kBlockN * 4;              // float [2 buffers][2 halves][128]
  static constexpr int OFF_XL = OFF_XM + 2 * 2 * kBlockM * 4;           // float [2 halves][128]
  static constexpr int OFF_RCPL = OFF_XL + 2 * kBlockM * 4;             // float [128]
  static constexpr int OFF_SCHED = OFF_RCPL + kBlockM * 4;
  static constexpr int OFF_BAR = OFF_SCHED + 2 * kSlotBytes;
  static constexpr int NUM_BARS = RB_FIXED + 4 * NK + 2 * NV;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 12;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA exceeded");
  static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0, "swizzled tiles need 1024-byte alignment");

  static constexpr int BAR_K_FULL = RB_FIXED;
  static constexpr int BAR_K_EMPTY = RB_FIXED + NK;
  static constexpr int BAR_KS_FULL = RB_FIXED + 2 * NK;
  static constexpr int BAR_KS_EMPTY = RB_FIXED + 3 * NK;
  static constexpr int BAR_V_FULL = RB_FIXED + 4 * NK;
  static constexpr int BAR_V_EMPTY = RB_FIXED + 4 * NK + NV;

  static constexpr uint32_t TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t tm_s(uint32_t buf) { return buf ? 128u : 0u; }
  static constexpr uint32_t TM_O = 256;

  static constexpr uint32_t IDESC_S = ptx::idesc_f32acc(0, 0, false, false, 128, 128);
  static constexpr uint32_t IDESC_PV =
      V8 ? ptx::idesc_f32acc(0, 0, false, false, 128, DV) : ptx::idesc_f32acc(1, 1, false, true, 128, DV);
  static constexpr int P_COLS_HALF = V8 ? 16 : 32;   // tensor-memory columns of 64 keys of P

  // Register split of the 512-thread CTA launched with 128 registers a thread.
  static constexpr int REG_SOFTMAX = 152, REG_CORR = 104, REG_MISC = 96;
  static_assert(2 * 128 * REG_SOFTMAX + 128 * REG_CORR + 128 * REG_MISC <= 512 * 128,
                "register split exceeds the launch allocation");
};

// K/V tiles a work tile visits.
template <bool CAUSAL>
__device__ __forceinline__ int rs_tiles(const SchedSlot& s) {
  const int q0 = s.t * kBlockM;
  const int kv_end = CAUSAL ? min(s.lk, q0 + kBlockM) : s.lk;
  return kv_end > 0 ? (kv_end + kBlockN - 1) / kBlockN : 0;
}

// ---------------------------------------------------------------------------------------------
template <class T, bool CAUSAL>
__device__ void rs_load_qk(const Tc05Params& P, const Ctx& c) {
  const int lane = threadIdx.x & 31;
  Ring<2> sched, qr;
  Ring<T::NK> kr;
  uint32_t k_fill_parity[T::NK], q_fill_parity[2];
  bool k_used[T::NK], q_used[2] = {false, false};
#pragma unroll
  for (int s = 0; s < T::NK; ++s) { k_fill_parity[s] = 0; k_used[s] = false; }
  q_fill_parity[0] = q_fill_parity[1] = 0;
  Cursor cur;
  int64_t w = blockIdx.x;
  bool aborted = false;
  while (true) {
    const SchedSlot s = decode_work(P, w, cur);
    if (!wait_warp(c, RB_SCHED_EMPTY + sched.idx, sched.phase ^ 1u, kRoleLoadQK)) { aborted = true; break; }
    if (lane == 0) {
      volatile int32_t* p = reinterpret_cast<volatile int32_t*>(c.smem + T::OFF_SCHED + kSlotBytes * sched.idx);
      p[0] = s.valid; p[1] = s.b; p[2] = s.h; p[3] = s.t;
      p[4] = s.q_start; p[5] = s.lq; p[6] = s.k_start; p[7] = s.lk; p[8] = s.split;
      ptx::mbar_arrive(c.bar(RB_SCHED_FULL + sched.idx));
    }
    __syncwarp();
    sched.next();
    if (!s.valid) break;
    const int n = rs_tiles<CAUSAL>(s);
    if (n > 0) {
      const int hk = s.h / P.group;
      const int qb = P.packed ? 0 : s.b;
      if (!wait_warp(c, RB_Q_EMPTY + qr.idx, qr.phase ^ 1u, kRoleLoadQK)) { aborted = true; break; }
      if (lane == 0) {
        const uint32_t bar = c.bar(RB_Q_FULL + qr.idx);
        ptx::mbar_expect_tx(bar, T::Q_BYTES);
        ptx::tma_load_4d(c.sbase + T::OFF_Q + qr.idx * T::Q_BYTES, &P.tm_q, bar, 0, s.h, s.q_start + s.t * kBlockM,
                         qb);
      }
      q_fill_parity[qr.idx] = qr.phase;
      q_used[qr.idx] = true;
      qr.next();
      // k-scales of this (sequence, KV head) from the range's first key: [B][Hkv][Sk] or [Hkv][Tk]
      const float* ks_row = P.k_scale + (P.packed ? (int64_t)hk * P.total_k + s.k_start
                                                  : ((int64_t)s.b * P.heads_kv + hk) * P.seqlen_k + s.k_start);
      for (int j = 0; j < n; ++j) {
        if (!wait_warp(c, T::BAR_K_EMPTY + kr.idx, kr.phase ^ 1u, kRoleLoadQK)) { aborted = true; break; }
        if (!wait_warp(c, T::BAR_KS_EMPTY + kr.idx, kr.phase ^ 1u, kRoleLoadQK)) { aborted = true; break; }
        if (lane == 0) {
          const uint32_t bar = c.bar(T::BAR_K_FULL + kr.idx);
          ptx::mbar_expect_tx(bar, T::K_STAGE_BYTES);
          ptx::tma_load_4d(c.sbase + T::OFF_K + kr.idx * T::K_STAGE_BYTES, &P.tm_k, bar, 0, hk,
                           s.k_start + kBlockN * j, qb);
        }
        // 128 k-scales, 4 per lane; keys past the range read nothing and give 0
        const uint32_t ks_dst = c.sbase + T::OFF_KS + kr.idx * (kBlockN * 4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = lane + 32 * e;
          const int kk = kBlockN * j + key;
          const bool in = kk < s.lk;
          ptx::cp_async_4(ks_dst + 4u * key, ks_row + (in ? kk : 0), in ? 4u : 0u);
        }
        ptx::cp_async_mbar_arrive_noinc(c.bar(T::BAR_KS_FULL + kr.idx));
        k_fill_parity[kr.idx] = kr.phase;
        k_used[kr.idx] = true;
        kr.next();
      }
      if (aborted) break;
    }
    if (P.schedule == ATTN_SCHEDULE_DYNAMIC) {
      int64_t nw = 0;
      if (lane == 0) nw = (int64_t)gridDim.x + (int64_t)atomicAdd(&c.ws[kWsTileCounter], 1u);
      w = __shfl_sync(kFull, nw, 0);
    } else if (P.schedule == ATTN_SCHEDULE_STATIC) {
      w += gridDim.x;
    } else {
      w = INT64_MAX;
    }
  }
  // every lane's k-scale copies land before the CTA goes on
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (aborted && lane == 0) {
#pragma unroll
    for (int s = 0; s < T::NK; ++s)
      if (k_used[s]) wait_drain(c, T::BAR_K_FULL + s, k_fill_parity[s]);
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (q_used[i]) wait_drain(c, RB_Q_FULL + i, q_fill_parity[i]);
  }
  __syncwarp();
}

template <class T, bool CAUSAL>
__device__ void rs_load_v(const Tc05Params& P, const Ctx& c) {
  const int lane = threadIdx.x & 31;
  Ring<2> sched;
  Ring<T::NV> vr;
  uint32_t v_fill_parity[T::NV];
  bool v_used[T::NV];
#pragma unroll
  for (int s = 0; s < T::NV; ++s) { v_fill_parity[s] = 0; v_used[s] = false; }
  bool first_v = true, aborted = false;
  while (true) {
    if (!wait_warp(c, RB_SCHED_FULL + sched.idx, sched.phase, kRoleLoadV)) { aborted = true; break; }
    const SchedSlot s = read_slot(c, sched.idx, T::OFF_SCHED);
    if (lane == 0) ptx::mbar_arrive(c.bar(RB_SCHED_EMPTY + sched.idx));
    sched.next();
    if (!s.valid) break;
    const int n = rs_tiles<CAUSAL>(s);
    const int hk = s.h / P.group;
    const int vb = P.packed ? 0 : s.b;
    for (int j = 0; j < n; ++j) {
      if (!wait_warp(c, T::BAR_V_EMPTY + vr.idx, vr.phase ^ 1u, kRoleLoadV)) { aborted = true; break; }
      // Fault injection (testing only): block 0 never loads its first V tile.
      const bool withhold = P.withhold_v && blockIdx.x == 0 && first_v;
      first_v = false;
      if (lane == 0 && !withhold) {
        const uint32_t bar = c.bar(T::BAR_V_FULL + vr.idx);
        const uint32_t dst = c.sbase + T::OFF_V + vr.idx * T::V_STAGE_BYTES;
        const int row = s.k_start + kBlockN * j;
        ptx::mbar_expect_tx(bar, T::V_STAGE_BYTES);
        if (T::V8) {
          ptx::tma_load_4d(dst, &P.tm_v, bar, row, 0, hk, vb);   // (key, depth row, head, batch)
        } else {
          ptx::tma_load_4d(dst, &P.tm_v, bar, 0, hk, row, vb);
          ptx::tma_load_4d(dst + T::CHUNK_BYTES, &P.tm_v, bar, 64, hk, row, vb);
        }
      }
      v_fill_parity[vr.idx] = vr.phase;
      v_used[vr.idx] = v_used[vr.idx] || !withhold;
      vr.next();
    }
    if (aborted) break;
  }
  if (aborted && lane == 0) {
#pragma unroll
    for (int s = 0; s < T::NV; ++s)
      if (v_used[s]) wait_drain(c, T::BAR_V_FULL + s, v_fill_parity[s]);
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------------------------
// One thread issues every MMA: S(0), S(1), then per K/V step j
// O += P(j) V(j) followed by S(j + 2) into the buffer P(j) occupied.
template <class T, bool CAUSAL>
__device__ void rs_mma(const Tc05Params& P, const Ctx& c) {
  const int role = kRoleMma;
  constexpr uint32_t HI = ptx::sdesc_hi_sw128(1024);
  Ring<2> sched, qr;
  Ring<T::NK> kr;
  Ring<T::NV> vr;
  uint32_t t = 0;   // global K/V step of this CTA: S buffer t & 1, its use (t >> 1)
  uint32_t ofree_phase = 0;
  bool aborted = false;
#define RS_WAIT(id, par)                   \
  if (!wait_one(c, (id), (par), role)) {   \
    aborted = true;                        \
    break;                                 \
  }
  while (true) {
    if (!wait_one(c, RB_SCHED_FULL + sched.idx, sched.phase, role)) { aborted = true; break; }
    const SchedSlot s = read_slot(c, sched.idx, T::OFF_SCHED);
    ptx::mbar_arrive(c.bar(RB_SCHED_EMPTY + sched.idx));
    sched.next();
    if (!s.valid) break;
    const int n = rs_tiles<CAUSAL>(s);
    if (n == 0) {
      RS_WAIT(RB_O_FREE, ofree_phase ^ 1u);
      ofree_phase ^= 1u;
      continue;
    }
    RS_WAIT(RB_Q_FULL + qr.idx, qr.phase);
    const uint32_t qa = ptx::sdesc_lo(ptx::opaque(c.sbase + T::OFF_Q + qr.idx * T::Q_BYTES), 16);
    // S(j) = Q K(j)^T into buffer (t + j) & 1: 4 e4m3 instructions of K = 32.
    auto issue_s = [&](int j) -> bool {
      if (!wait_one(c, T::BAR_K_FULL + kr.idx, kr.phase, role)) return false;
      ptx::tc_fence_after();
      const uint32_t buf = (t + (uint32_t)j) & 1u;
      const uint32_t ka = ptx::sdesc_lo(ptx::opaque(c.sbase + T::OFF_K + kr.idx * T::K_STAGE_BYTES), 16);
#pragma unroll
      for (int kk = 0; kk < T::DQK / 32; ++kk)
        ptx::mma_fp8_ss_lo<HI, HI, T::IDESC_S>(c.tmem + T::tm_s(buf), qa + kk * 2, ka + kk * 2, kk > 0);
      ptx::mma_commit(c.bar(RB_S_FULL + buf));
      ptx::mma_commit(c.bar(T::BAR_K_EMPTY + kr.idx));
      kr.next();
      if (j == n - 1) ptx::mma_commit(c.bar(RB_Q_EMPTY + qr.idx));   // the Q tile's last S
      return true;
    };
    if (!issue_s(0)) { aborted = true; break; }
    if (n > 1 && !issue_s(1)) { aborted = true; break; }
    for (int j = 0; j < n; ++j) {
      const uint32_t buf = (t + (uint32_t)j) & 1u;
      if (j == 0) {
        RS_WAIT(RB_O_FREE, ofree_phase ^ 1u);   // the epilogue read the previous work tile's O
        ofree_phase ^= 1u;
      }
      const uint32_t p_phase = ((t + (uint32_t)j) >> 1) & 1u;
      RS_WAIT(T::BAR_V_FULL + vr.idx, vr.phase);
      RS_WAIT(RB_P_LO + buf, p_phase);
      ptx::tc_fence_after();
      const uint32_t a = c.tmem + T::tm_s(buf);
      const uint32_t d = c.tmem + T::TM_O;
      if (T::V8) {
        // K-major e4m3 V stage (Dv rows x 128 keys): 32 keys per instruction
        const uint32_t va = ptx::sdesc_lo(ptx::opaque(c.sbase + T::OFF_V + vr.idx * T::V_STAGE_BYTES), 16);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) ptx::mma_fp8_ts_lo<HI, T::IDESC_PV>(d, a + kk * 8, va + kk * 2, (j > 0 || kk > 0) ? 1u : 0u);
        RS_WAIT(RB_P_HI + buf, p_phase);
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 2; kk < 4; ++kk) ptx::mma_fp8_ts_lo<HI, T::IDESC_PV>(d, a + kk * 8, va + kk * 2, 1u);
      } else {
        // MN-major bf16 V stage (128 keys x Dv): 16 keys per instruction
        const uint32_t va =
            ptx::sdesc_lo(ptx::opaque(c.sbase + T::OFF_V + vr.idx * T::V_STAGE_BYTES), T::CHUNK_BYTES);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_bf16_ts_lo<HI, T::IDESC_PV>(d, a + kk * 8, va + kk * (2048 >> 4), (j > 0 || kk > 0) ? 1u : 0u);
        RS_WAIT(RB_P_HI + buf, p_phase);
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 4; kk < 8; ++kk) ptx::mma_bf16_ts_lo<HI, T::IDESC_PV>(d, a + kk * 8, va + kk * (2048 >> 4), 1u);
      }
      ptx::mma_commit(c.bar(T::BAR_V_EMPTY + vr.idx));
      ptx::mma_commit(c.bar(RB_O_READY));
      if (j == n - 1) ptx::mma_commit(c.bar(RB_O_FINAL));
      vr.next();
      // S(j + 2) overwrites P(j): issued after the P V that reads it
      if (j + 2 < n && !issue_s(j + 2)) { aborted = true; break; }
    }
    if (aborted) break;
    qr.next();
    t += (uint32_t)n;
  }
#undef RS_WAIT
  ptx::mma_commit(c.bar(RB_DRAIN));
  wait_drain(c, RB_DRAIN, 0);
  (void)aborted;
}

// ---------------------------------------------------------------------------------------------
// Softmax half `g` (warpgroup g): keys [64 g, 64 g + 64) of every tile, one
// row per thread.
template <class T, bool CAUSAL>
__device__ void rs_softmax(const Tc05Params& P, const Ctx& c, const int g) {
  const int tid = threadIdx.x - 128 * g;   // row of the Q tile == TMEM lane
  const int quarter = tid >> 5;
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  float* xm = reinterpret_cast<float*>(c.smem + T::OFF_XM);     // [buf][half][row]
  float* xl = reinterpret_cast<float*>(c.smem + T::OFF_XL);     // [half][row]
  float* rcpl_sm = reinterpret_cast<float*>(c.smem + T::OFF_RCPL);
  const int role = g == 0 ? kRoleSoftmax0 : kRoleSoftmax1;
  Ring<2> sched;
  Ring<T::NK> kr;
  uint32_t t = 0, xch_phase = 0, stats_phase = 0;
  while (true) {
    if (!wait_warp(c, RB_SCHED_FULL + sched.idx, sched.phase, role)) return;
    const SchedSlot s = read_slot(c, sched.idx, T::OFF_SCHED);
    ptx::mbar_arrive(c.bar(RB_SCHED_EMPTY + sched.idx));
    sched.next();
    if (!s.valid) return;
    const int n = rs_tiles<CAUSAL>(s);
    const int first_row = s.t * kBlockM;
    const int qi = first_row + tid;
    const bool row_valid = qi < s.lq;
    const int lim = CAUSAL ? min(s.lk, qi + 1) : s.lk;
    const bool split_kv = !CAUSAL && P.num_splits > 1;
    const int sp = split_kv ? s.split : 0;
    const int64_t lse_idx = P.packed ? ((int64_t)sp * P.heads_q + s.h) * P.total_q + s.q_start + qi
                                     : (((int64_t)sp * P.batch + s.b) * P.heads_q + s.h) * P.seqlen_q + qi;
    float qs = 1.f;
    if (row_valid)
      qs = P.packed ? P.q_scale[(int64_t)s.h * P.total_q + s.q_start + qi]
                    : P.q_scale[((int64_t)s.b * P.heads_q + s.h) * P.seqlen_q + qi];
    const float c_row = P.scale_log2 * qs;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < n; ++j) {
      const uint32_t gstep = t + (uint32_t)j;
      const uint32_t buf = gstep & 1u;
      const int kb = kBlockN * j;
      if (!wait_warp(c, RB_S_FULL + buf, (gstep >> 1) & 1u, role)) return;
      ptx::tc_fence_after();
      float sv[64];
      {
        uint32_t r[2][32];
#pragma unroll
        for (int q = 0; q < 2; ++q) ptx::tmem_ld32(c.tmem + lane_base + T::tm_s(buf) + 64 * g + 32 * q, r[q]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int e = 0; e < 32; ++e) sv[32 * q + e] = __uint_as_float(r[q][e]);
      }
      // per-key scales of this half of the tile
      if (!wait_warp(c, T::BAR_KS_FULL + kr.idx, kr.phase, role)) return;
      {
        const float4* k4 = reinterpret_cast<const float4*>(c.smem + T::OFF_KS + kr.idx * (kBlockN * 4)) + 16 * g;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float4 kv = k4[e];
          float a0, a1, a2, a3;
          ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(sv[4 * e], sv[4 * e + 1]), ptx::f2_pack(kv.x, kv.y)), a0, a1);
          ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(sv[4 * e + 2], sv[4 * e + 3]), ptx::f2_pack(kv.z, kv.w)), a2, a3);
          sv[4 * e] = a0; sv[4 * e + 1] = a1; sv[4 * e + 2] = a2; sv[4 * e + 3] = a3;
        }
      }
      __syncwarp();
      if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(c.bar(T::BAR_KS_EMPTY + kr.idx));
      kr.next();
      const bool need_mask = (kb + kBlockN > s.lk) || (CAUSAL && kb + kBlockN - 1 > first_row);
      if (need_mask) {
        const int vis = lim - kb - 64 * g;   // keys of this half visible to the row
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (e >= vis) sv[e] = -INFINITY;
      }
      float mx0 = ptx::max3(sv[0], sv[1], sv[2]), mx1 = ptx::max3(sv[3], sv[4], sv[5]);
#pragma unroll
      for (int e = 6; e < 62; e += 4) {
        mx0 = ptx::max3(mx0, sv[e], sv[e + 1]);
        mx1 = ptx::max3(mx1, sv[e + 2], sv[e + 3]);
      }
      mx0 = ptx::max3(mx0, sv[62], sv[63]);
      float mx = fmaxf(mx0, mx1);
      // Both halves of the row agree on the maximum. The exchange also
      // orders this half's tensor-memory loads of S before the other half's
      // stores of P into the same buffer (P of keys 64..127 lands on S
      // columns of keys 32..63).
      xm[(buf * 2 + g) * kBlockM + tid] = mx;
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.bar(RB_XCH + quarter));
      if (!wait_warp(c, RB_XCH + quarter, xch_phase, role)) return;
      xch_phase ^= 1u;
      ptx::tc_fence_after();
      mx = fmaxf(mx, xm[(buf * 2 + (g ^ 1)) * kBlockM + tid]) * c_row;
      const float m_new = fmaxf(m, mx);
      float m_use = m, alpha = 1.f;
      if (j == 0) {
        m_use = m_new;
      } else if (m_new > m + 8.f) {
        m_use = m_new;
        alpha = ptx::ex2(m - m_new);
      }
      if (__any_sync(kFull, alpha != 1.f)) {
        // Rescale this half's columns of O: the previous P V must be done.
        if (!wait_warp(c, RB_O_READY, (gstep - 1u) & 1u, role)) return;
        ptx::tc_fence_after();
        const uint32_t tO = c.tmem + lane_base + T::TM_O + 64 * g;
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
          uint32_t r[32];
          ptx::tmem_ld32(tO + 32 * q, r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          ptx::tmem_st32(tO + 32 * q, r);
        }
        ptx::tmem_wait_st();
      }
      if (g == 1) {
        // the first half of P V may start once this half's O columns are rescaled
        ptx::tc_fence_before();
        ptx::mbar_arrive(c.bar(RB_P_LO + buf));
      }
      const uint64_t c2 = ptx::f2_pack(c_row, c_row);
      const uint64_t n2 = ptx::f2_pack(-m_use, -m_use);
      uint64_t acc0 = 0, acc1 = 0;
      uint32_t pk[T::P_COLS_HALF];
      [[maybe_unused]] float q0 = 0.f, q1 = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        float x0, x1;
        ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(sv[2 * e], sv[2 * e + 1]), c2, n2), x0, x1);
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
      const uint32_t tP = c.tmem + lane_base + T::tm_s(buf) + T::P_COLS_HALF * g;
      if constexpr (T::V8) ptx::tmem_st16(tP, pk);
      else ptx::tmem_st32(tP, pk);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.bar((g == 0 ? RB_P_LO : RB_P_HI) + buf));
      float s0, s1, s2, s3;
      ptx::f2_unpack(acc0, s0, s1);
      ptx::f2_unpack(acc1, s2, s3);
      l = l * alpha + ((s0 + s1) + (s2 + s3));
      m = m_use;
    }
    t += (uint32_t)n;
    if (n > 0) {
      // the row sum of both halves
      xl[g * kBlockM + tid] = l;
      ptx::mbar_arrive(c.bar(RB_XCH + quarter));
      if (!wait_warp(c, RB_XCH + quarter, xch_phase, role)) return;
      xch_phase ^= 1u;
      l += xl[(g ^ 1) * kBlockM + tid];
    }
    if (g == 0) {
      // row statistics: LSE (natural log) here, 1/l to the epilogue
      float* const lse_dst = split_kv ? P.lse_part : P.lse;
      if (row_valid && lse_dst != nullptr)
        lse_dst[lse_idx] = l > 0.f ? (m + ptx::lg2(l)) * 0.69314718055994531f : -INFINITY;
      if (!wait_warp(c, RB_STATS_FREE, stats_phase ^ 1u, role)) return;
      stats_phase ^= 1u;
      rcpl_sm[tid] = l > 0.f ? 1.f / l : 0.f;
      ptx::mbar_arrive(c.bar(RB_STATS));
    }
  }
}

// ---------------------------------------------------------------------------------------------
template <class T, bool CAUSAL>
__device__ void rs_epilogue(const Tc05Params& P, const Ctx& c) {
  const int tid = threadIdx.x - 256;
  const uint32_t lane_base = (uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16;
  const float* rcpl_sm = reinterpret_cast<const float*>(c.smem + T::OFF_RCPL);
  Ring<2> sched;
  uint32_t stats_phase = 0, ofinal_phase = 0;
  while (true) {
    if (!wait_warp(c, RB_SCHED_FULL + sched.idx, sched.phase, kRoleCorrection)) return;
    const SchedSlot s = read_slot(c, sched.idx, T::OFF_SCHED);
    ptx::mbar_arrive(c.bar(RB_SCHED_EMPTY + sched.idx));
    sched.next();
    if (!s.valid) return;
    const int n = rs_tiles<CAUSAL>(s);
    if (!wait_warp(c, RB_STATS, stats_phase, kRoleCorrection)) return;
    stats_phase ^= 1u;
    const float rl = rcpl_sm[tid];
    ptx::mbar_arrive(c.bar(RB_STATS_FREE));
    const int qi = s.t * kBlockM + tid;
    const bool row_valid = qi < s.lq;
    const bool split_kv = !CAUSAL && P.num_splits > 1;
    uint16_t* orow = P.o + (int64_t)s.b * P.o_stride_b + (int64_t)(s.q_start + qi) * P.o_stride_t +
                     (int64_t)s.h * P.o_stride_h;
    if (n > 0) {
      if (!wait_warp(c, RB_O_FINAL, ofinal_phase, kRoleCorrection)) return;
      ofinal_phase ^= 1u;
      ptx::tc_fence_after();
      const uint32_t tO = c.tmem + lane_base + T::TM_O;
      if (split_kv) {
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
          if (row_valid) store_row_chunk<T>(orow + 32 * q, r, rl);
        }
      }
    } else if (row_valid && split_kv) {
      float4* d = reinterpret_cast<float4*>(P.o_part + partial_row(P, s, qi) * T::DV);
#pragma unroll 1
      for (int e = 0; e < T::DV / 4; ++e) d[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else if (row_valid) {
      uint4* d = reinterpret_cast<uint4*>(orow);
#pragma unroll
      for (int e = 0; e < T::DV / 8; ++e) d[e] = make_uint4(0u, 0u, 0u, 0u);
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(c.bar(RB_O_FREE));
  }
}

// ---------------------------------------------------------------------------------------------
template <class T, bool CAUSAL>
__global__ void __launch_bounds__(512, 1) fa_rowsplit_kernel(const __grid_constant__ Tc05Params P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctx c;
  c.smem = smem;
  c.sbase = ptx::smem_u32(smem);
  c.ws = P.ws;
  c.abort_flag = reinterpret_cast<volatile int*>(smem + T::OFF_ABORT);
  c.bar_off = T::OFF_BAR;
  c.timeout_ns = P.timeout_ns;
  c.rank = 0u;
  c.peer_abort = 0u;
  if (c.sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(&P.ws[kWsErrorCode], 0u, 2u);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(c.bar(RB_Q_FULL + i), 1);
      ptx::mbar_init(c.bar(RB_Q_EMPTY + i), 1);
      ptx::mbar_init(c.bar(RB_S_FULL + i), 1);
      ptx::mbar_init(c.bar(RB_SCHED_FULL + i), 1);
      ptx::mbar_init(c.bar(RB_SCHED_EMPTY + i), kRsSchedConsumers);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(c.bar(RB_P_LO + b), 256);
      ptx::mbar_init(c.bar(RB_P_HI + b), 128);
    }
    ptx::mbar_init(c.bar(RB_O_READY), 1);
    ptx::mbar_init(c.bar(RB_O_FINAL), 1);
    ptx::mbar_init(c.bar(RB_O_FREE), 128);
    ptx::mbar_init(c.bar(RB_STATS), 128);
    ptx::mbar_init(c.bar(RB_STATS_FREE), 128);
#pragma unroll
    for (int q = 0; q < 4; ++q) ptx::mbar_init(c.bar(RB_XCH + q), 64);
    ptx::mbar_init(c.bar(RB_DRAIN), 1);
#pragma unroll
    for (int s = 0; s < T::NK; ++s) {
      ptx::mbar_init(c.bar(T::BAR_K_FULL + s), 1);
      ptx::mbar_init(c.bar(T::BAR_K_EMPTY + s), 1);
      ptx::mbar_init(c.bar(T::BAR_KS_FULL + s), 32);   // one cp.async arrival per producer lane
      ptx::mbar_init(c.bar(T::BAR_KS_EMPTY + s), 8);   // one arrival per softmax warp
    }
#pragma unroll
    for (int s = 0; s < T::NV; ++s) {
      ptx::mbar_init(c.bar(T::BAR_V_FULL + s), 1);
      ptx::mbar_init(c.bar(T::BAR_V_EMPTY + s), 1);
    }
    *c.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 12) {
    ptx::tmem_alloc(c.sbase + T::OFF_TMEM_SLOT, T::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (warp == 14 && lane == 0) {
    ptx::prefetch_tmap(&P.tm_q);
    ptx::prefetch_tmap(&P.tm_k);
    ptx::prefetch_tmap(&P.tm_v);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  c.tmem = *reinterpret_cast<volatile uint32_t*>(smem + T::OFF_TMEM_SLOT);

  const int wg = warp >> 2;
  if (wg < 2) {
    setmaxnreg_inc<T::REG_SOFTMAX>();
    rs_softmax<T, CAUSAL>(P, c, wg);
  } else if (wg == 2) {
    setmaxnreg_dec<T::REG_CORR>();
    rs_epilogue<T, CAUSAL>(P, c);
  } else {
    setmaxnreg_dec<T::REG_MISC>();
    if (warp == 12) {
      if (lane == 0) rs_mma<T, CAUSAL>(P, c);
      __syncwarp();
    } else if (warp == 14) {
      rs_load_qk<T, CAUSAL>(P, c);
    } else if (warp == 15) {
      rs_load_v<T, CAUSAL>(P, c);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(c.tmem, T::TMEM_COLS);
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

template <class T, bool CAUSAL>
cudaError_t rs_launch_tc(const Tc05Params& prm, int grid, cudaStream_t stream) {
  constexpr auto kern = fa_rowsplit_kernel<T, CAUSAL>;
  return launch_with_smem<kern>(T::SMEM_BYTES, [&]() -> cudaError_t {
    kern<<<grid, 512, T::SMEM_BYTES, stream>>>(prm);
    return cudaGetLastError();
  });
}

template <class T>
cudaError_t rs_launch_t(bool causal, const Tc05Params& prm, int grid, cudaStream_t stream) {
  return causal ? rs_launch_tc<T, true>(prm, grid, stream) : rs_launch_tc<T, false>(prm, grid, stream);
}

template <class T>
Tc05Config rs_config_t() {
  Tc05Config c;
  c.smem_bytes = T::SMEM_BYTES;
  c.k_stages = T::NK;
  c.v_stages = T::NV;
  c.threads = 512;
  c.tmem_cols = (int)T::TMEM_COLS;
  return c;
}

using RsTraitsFp8 = RsTraits<false>;
using RsTraitsFp8Qkv = RsTraits<true>;

cudaError_t rs_launch_fp8(bool causal, const Tc05Params& prm, int grid, cudaStream_t stream);
cudaError_t rs_launch_fp8qkv(bool causal, const Tc05Params& prm, int grid, cudaStream_t stream);

}  // namespace af
