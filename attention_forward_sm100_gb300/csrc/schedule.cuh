// Work decomposition of the persistent kernel (host and device).
//
// The "MHATileScheduler" page (trait description, grid_dim and advance)
// describes a persistent schedule that maps work tiles over (sequence, head,
// query tile) to CTAs and walks each CTA through the grid. Here a work tile is
// ROWS_PER_TILE query rows of one (sequence b, query head h). Work indices are
// handed out by an atomic counter; index w decodes as follows:
//   * sequences in order (packed inputs: b-major with a cursor over cu_seqlens);
//   * inside a sequence, KV heads in chunks of kv_chunk heads, sized so the
//     K/V of one chunk stays in L2 while its tiles are processed;
//   * inside a chunk, query tiles from the last (most keys under a causal
//     mask) to the first, and for each tile index every query head of the
//     chunk, the heads that share one KV head next to each other: the
//     heaviest tiles are taken first and the light ones fill the tail.
// With split-KV (the "splitk_partitions" of the SM100AttentionSMem page's
// configuration) each query tile is cut into `splits` key ranges and every
// (tile, range) pair is a work tile of its own: the decode runs over
// T * splits virtual tiles, tile t range r being virtual tile t * splits + r.
// Without a mask the ranges cut the sequence's key tiles; under the causal
// mask they cut the key tiles the query tile sees (causal_split_range).
#pragma once
#include <stdint.h>

#ifndef __CUDACC__
#define AF_HD
#else
#define AF_HD __host__ __device__
#endif

namespace af {

struct WorkTile {
  int32_t b;
  int32_t h;
  int32_t t;
  int32_t split;   // key range (0 without split-KV)
};

AF_HD inline int32_t tiles_for(int32_t len, int32_t rows) { return (len + rows - 1) / rows; }

// Work index local to one sequence (0 <= wl < T * Hq) -> (h, t).
AF_HD inline WorkTile decode_in_sequence(int64_t wl, int32_t b, int32_t T, int32_t group, int32_t heads_kv,
                                         int32_t kv_chunk) {
  const int64_t chunk_units = (int64_t)T * kv_chunk * group;
  const int32_t c = (int32_t)(wl / chunk_units);
  const int32_t r = (int32_t)(wl - (int64_t)c * chunk_units);
  const int32_t kv_lo = c * kv_chunk;
  const int32_t kv_n = heads_kv - kv_lo < kv_chunk ? heads_kv - kv_lo : kv_chunk;
  const int32_t per_t = kv_n * group;
  WorkTile w;
  w.b = b;
  w.t = T - 1 - r / per_t;
  w.h = kv_lo * group + r % per_t;
  w.split = 0;
  return w;
}

// Fixed-length decode: every sequence has T query tiles per head, each cut
// into `splits` key ranges.
AF_HD inline WorkTile decode_fixed(int64_t w, int32_t T, int32_t splits, int32_t heads_q, int32_t group,
                                   int32_t kv_chunk) {
  const int64_t per_seq = (int64_t)T * splits * heads_q;
  const int32_t b = (int32_t)(w / per_seq);
  WorkTile u = decode_in_sequence(w - (int64_t)b * per_seq, b, T * splits, group, heads_q / group, kv_chunk);
  u.split = u.t % splits;
  u.t /= splits;
  return u;
}

// Key tiles [*j0, *j1) of range `split` out of `splits` over kv_tiles key
// tiles: contiguous, sizes differing by at most one, none empty while
// splits <= kv_tiles.
AF_HD inline void split_range(int32_t split, int32_t splits, int32_t kv_tiles, int32_t* j0, int32_t* j1) {
  *j0 = (int32_t)((int64_t)split * kv_tiles / splits);
  *j1 = (int32_t)((int64_t)(split + 1) * kv_tiles / splits);
}

// Causal split-KV: key tiles [*j0, *j1) of range `split` out of `splits` for
// the work tile whose rows start at q0 (rows of them, the first first_rows
// forming its first MMA tile) over lk keys of tile kv_tile. The ranges cut the
// key tiles that the first MMA tile sees (top-left mask: keys up to its last
// row) and the last range also takes the tiles only the rest of the work tile
// sees. So every non-empty range starts at or before row q0: each of the work
// tile's rows sees the first key of every range it visits, and the first MMA
// tile visits every non-empty range. Empty ranges (fewer tiles than ranges)
// start inside the keys (*j0 < tiles) and hold no key.
AF_HD inline void causal_split_range(int32_t split, int32_t splits, int32_t q0, int32_t first_rows, int32_t rows,
                                     int32_t lk, int32_t kv_tile, int32_t* j0, int32_t* j1) {
  const int32_t seen_first = q0 + first_rows < lk ? q0 + first_rows : lk;
  const int32_t seen_all = q0 + rows < lk ? q0 + rows : lk;
  split_range(split, splits, tiles_for(seen_first, kv_tile), j0, j1);
  if (split == splits - 1) *j1 = tiles_for(seen_all, kv_tile);
}

// Split count for `work` equal query tiles of kv_tiles key tiles each on
// `ctas` persistent CTAs. The time of a split count s is modelled as
// waves(s) * (ceil(kv_tiles / s) + 2): the CTAs run the work * s pieces in
// ceil(work * s / ctas) waves, and each piece costs its key tiles plus about
// two tiles' worth of fixed cost (its Q load, pipeline fill and the partial
// result write). The smallest s of least modelled time in
// [1, min(kv_tiles, max_splits)] is chosen.
AF_HD inline int32_t choose_splits(int64_t work, int32_t kv_tiles, int32_t ctas, int32_t max_splits) {
  if (work <= 0 || kv_tiles <= 1 || ctas <= 0) return 1;
  const int32_t hi = kv_tiles < max_splits ? kv_tiles : max_splits;
  int32_t best = 1;
  int64_t best_cost = -1;
  for (int32_t s = 1; s <= hi; ++s) {
    const int64_t waves = (work * s + ctas - 1) / ctas;
    const int64_t cost = waves * ((kv_tiles + s - 1) / s + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// Split count for a causal problem of `heads` (B * Hq) x ceil(lq / rows)
// query tiles over lk keys (the longest lengths when packed) on `ctas`
// persistent CTAs, in units of one MMA tile's step over one key tile. Query
// tile t (rows from q0 = t * rows; the first first_rows form its first MMA
// tile) costs n0 + n1 units, n_i being the key tiles its MMA tile i sees. With
// s ranges (causal_split_range) its heaviest piece is 2 * ceil(n0 / s) + 1
// units, every piece adds kPieceUnits of fixed cost (Q load, pipeline fill,
// partial write), and the merge costs kMergeUnits plus its traffic (the fp32
// partial O written and read back, s * heads * lq * dv * 8 bytes, at
// kMergeBytesPerUnit). The modelled time of s is
//   max(heaviest piece, ceil(total units / ctas)) + merge(s),
// and the smallest s of least modelled time in [1, min(key tiles, max_splits)]
// is chosen: long sequences with few heads split, full grids do not.
// One unit (a 128 x 128 x (Dqk + Dv) step) is ~0.6 us of tensor-core time on
// GB300; the merge launch and its dependent start ~5 us; its traffic moves at
// ~6 TB/s.
constexpr int64_t kPieceUnits = 4;
constexpr int64_t kMergeUnits = 8;
constexpr int64_t kMergeBytesPerUnit = 3600000;
AF_HD inline int32_t choose_splits_causal(int64_t heads, int32_t lq, int32_t lk, int32_t rows, int32_t first_rows,
                                          int32_t kv_tile, int32_t dv, int32_t ctas, int32_t max_splits) {
  if (heads <= 0 || lq <= 0 || lk <= 0 || rows <= 0 || ctas <= 0) return 1;
  const int32_t T = tiles_for(lq, rows);
  int64_t units = 0;   // sum over one head's query tiles of n0 + n1
  for (int32_t t = 0; t < T; ++t) {
    const int64_t q0 = (int64_t)t * rows;
    units += tiles_for((int32_t)(q0 + first_rows < lk ? q0 + first_rows : lk), kv_tile) +
             tiles_for((int32_t)(q0 + rows < lk ? q0 + rows : lk), kv_tile);
  }
  const int64_t q_last = (int64_t)(T - 1) * rows;
  const int32_t n0_max = tiles_for((int32_t)(q_last + first_rows < lk ? q_last + first_rows : lk), kv_tile);
  const int32_t kv_tiles = tiles_for(lk, kv_tile);
  const int32_t hi = kv_tiles < max_splits ? kv_tiles : max_splits;
  int32_t best = 1;
  int64_t best_cost = -1;
  for (int32_t s = 1; s <= hi; ++s) {
    const int64_t piece = 2 * (int64_t)((n0_max + s - 1) / s) + 1 + kPieceUnits;
    const int64_t total = heads * (units + (int64_t)T * s * kPieceUnits);
    const int64_t spread = (total + ctas - 1) / ctas;
    const int64_t merge = s > 1 ? kMergeUnits + (int64_t)s * heads * lq * dv * 8 / kMergeBytesPerUnit : 0;
    const int64_t cost = (piece > spread ? piece : spread) + merge;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// KV heads per chunk: as many as keep the chunk's K/V (seqlen_k rows of
// k_row_bytes + v_row_bytes per head) within l2_budget bytes.
AF_HD inline int32_t choose_kv_chunk(int64_t seqlen_k, int64_t kv_row_bytes, int32_t heads_kv, int64_t l2_budget) {
  const int64_t per_head = seqlen_k * kv_row_bytes;
  int64_t c = per_head > 0 ? l2_budget / per_head : heads_kv;
  if (c < 1) c = 1;
  if (c > heads_kv) c = heads_kv;
  return (int32_t)c;
}

}  // namespace af
