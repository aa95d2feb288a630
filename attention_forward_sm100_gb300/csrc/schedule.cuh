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
// configuration; fixed-length, unmasked problems only) each query tile is
// cut into `splits` key ranges and every (tile, range) pair is a work tile of
// its own: the decode runs over T * splits virtual tiles, tile t range r
// being virtual tile t * splits + r.
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
