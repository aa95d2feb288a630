// Work decomposition of the persistent kernel (host and device).
//
// The "MHATileScheduler" page (trait description, grid_dim and advance)
// describes a persistent schedule that maps work tiles over (sequence, head,
// query tile) to CTAs and walks each CTA through the grid. Here a work tile is
// ROWS_PER_TILE query rows of one (sequence b, query head h). Work indices are
// handed out by an atomic counter; index w decodes as follows:
//   * sequences in order (packed inputs: b-major with a cursor over cu_seqlens);
//   * inside a sequence, groups of query heads that share one KV head, so the
//     heads reading the same K/V tiles run at the same time and share L2;
//   * inside a group, query tiles from the last (most keys under a causal
//     mask) to the first, heads of the group interleaved: the heaviest tiles
//     are taken first and the light ones fill the tail.
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
};

AF_HD inline int32_t tiles_for(int32_t len, int32_t rows) { return (len + rows - 1) / rows; }

// Work index local to one sequence (0 <= wl < T * Hq) -> (h, t).
AF_HD inline WorkTile decode_in_sequence(int64_t wl, int32_t b, int32_t T, int32_t group) {
  const int64_t per_group = (int64_t)T * group;
  const int32_t grp = (int32_t)(wl / per_group);
  const int32_t rem = (int32_t)(wl - (int64_t)grp * per_group);
  WorkTile w;
  w.b = b;
  w.h = grp * group + rem % group;
  w.t = T - 1 - rem / group;
  return w;
}

// Fixed-length decode: every sequence has T tiles per head.
AF_HD inline WorkTile decode_fixed(int64_t w, int32_t T, int32_t heads_q, int32_t group) {
  const int64_t per_seq = (int64_t)T * heads_q;
  const int32_t b = (int32_t)(w / per_seq);
  return decode_in_sequence(w - (int64_t)b * per_seq, b, T, group);
}

}  // namespace af
