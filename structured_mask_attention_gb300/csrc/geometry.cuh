// geometry.cuh -- tile geometry of the two-stream BDLM block mask, shared by
// the host work-list builder and the device kernels.
//
// Mask ("Block Parallelism For Efficient Distributed Long-Context Diffusion
// Language Model Training", arxiv.science abstract: autoregressive across
// blocks, parallel inside a block; evolve.pub review FAQ on CSBP: corrupted
// blocks read the shared clean prefix and keep their own keys), with
// blk(i) = i / B:
//   clean row i     -> clean key j      iff blk(j) <= blk(i)
//   corrupted row i -> clean key j      iff blk(j) <  blk(i)
//   corrupted row i -> corrupted key j  iff blk(j) == blk(i)
// A call may restrict the clean keys to one shard [kv_begin, kv_end) and drop
// the corrupted own-block keys (include_local = 0): the per-shard view of CSBP.
//
// For one query row every visible key set is a half-open interval per key
// stream, so masking a partially visible tile is an interval test, and the
// visible key tiles of a query tile are two contiguous tile ranges.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define BDLM_HD __host__ __device__ __forceinline__
#else
#define BDLM_HD inline
#endif

namespace bdlm {

struct Geom {
  int64_t L, B;
  int Hq, Hkv;
  int64_t kv_begin, kv_end;  // clean key range of this call
  int include_local;         // corrupted rows also read their own block
  int naive_order = 0;       // 1: items in natural order, round-robin over the grid
  int round_items = 152;     // CTAs of the persistent grid (the device's SM count): items per block and KV head
};

// Query rows a call computes, per stream (0 clean, 1 corrupted): [lo, hi).
// The defaults cover every row.  A rank of a multi-rank CSBP deployment
// computes only the rows it owns; rows outside are neither computed into
// other rows' results nor written.  (Kept apart from Geom: the kernels that
// do not restrict rows keep their parameter blocks, and registers, as is.)
//
// The same calls describe where the tensors' rows live.  The row-indexed
// tensors of stream s (its Q, dO, O, LSE, D, dQ; for the corrupted stream
// also its K, V, dK, dV, since a rank owns whole corrupted blocks) hold rows
// [base[s], base[s] + len[s]), row i at local index i - base[s]; the clean K,
// V, dK, dV hold keys [kbase, kbase + klen).  Full-length tensors: base 0,
// len = klen = L.  Rank-local tensors: base = lo, len = hi - lo, and the
// clean keys the call reads.  The kernels' tensor maps cover only the held
// rows, so a tile that reaches past them reads zeros there.
struct RowRange {
  int32_t lo[2] = {0, 0};
  int32_t hi[2] = {0x7fffffff, 0x7fffffff};
  int32_t base[2] = {0, 0};
  int32_t len[2] = {0, 0};
  int32_t kbase = 0, klen = 0;
};

BDLM_HD int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
BDLM_HD int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }
BDLM_HD int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Visible clean-key interval [lo, hi) of query row i of `stream` (0 clean,
// 1 corrupted); empty when hi <= lo.
BDLM_HD void clean_interval(const Geom& g, int stream, int64_t i, int64_t& lo, int64_t& hi) {
  const int64_t b = i / g.B;
  const int64_t lim = stream == 0 ? (b + 1) * g.B : b * g.B;
  lo = g.kv_begin;
  hi = imin64(g.kv_end, lim);
}

// Visible corrupted-key interval of query row i (only corrupted rows, only
// with include_local).
BDLM_HD void noisy_interval(const Geom& g, int stream, int64_t i, int64_t& lo, int64_t& hi) {
  if (stream == 1 && g.include_local) {
    const int64_t b = i / g.B;
    lo = b * g.B;
    hi = (b + 1) * g.B;
  } else {
    lo = 0;
    hi = 0;
  }
}

// A row range's bounds for `stream` (selected, not indexed, so that a local
// copy stays in registers).
BDLM_HD int64_t range_lo(const RowRange& r, int stream) { return stream ? r.lo[1] : r.lo[0]; }
BDLM_HD int64_t range_hi(const RowRange& r, int stream) { return stream ? r.hi[1] : r.hi[0]; }

// Local index of row i of `stream` in that stream's row-indexed tensors, the
// row stride of its [H, rows] statistics, and the local index of key j of
// key stream ks.
BDLM_HD int64_t local_row(const RowRange& r, int stream, int64_t i) { return i - (stream ? r.base[1] : r.base[0]); }
BDLM_HD int64_t held_rows(const RowRange& r, int stream) { return stream ? r.len[1] : r.len[0]; }
BDLM_HD int64_t local_key(const RowRange& r, int ks, int64_t j) { return j - (ks ? r.base[1] : r.kbase); }

// True when key j of key stream ks is held by the call's K / V tensors.
BDLM_HD bool key_held(const RowRange& r, int ks, int64_t j) {
  const int64_t k = local_key(r, ks, j);
  return k >= 0 && k < (ks ? r.len[1] : r.klen);
}

// True when query row i of `stream` is in the range.
BDLM_HD bool row_in(const RowRange& r, int stream, int64_t i) {
  return i >= range_lo(r, stream) && i < range_hi(r, stream);
}

// True when some row of the query tile [r0, r1) of `stream` is in the range.
// (The forward and dQ visit the key tiles of a tile's rows and write only
// the range's rows; a tile without any is skipped.)
BDLM_HD bool tile_in(const RowRange& r, int stream, int64_t r0, int64_t r1) {
  return r1 > range_lo(r, stream) && r0 < range_hi(r, stream);
}

// The query rows of each stream that read a key tile (kv_tile_rows),
// restricted to the range.
BDLM_HD void clamp_rows(const RowRange& r, int64_t& c_lo, int64_t& c_hi, int64_t& n_lo, int64_t& n_hi) {
  c_lo = imax64(c_lo, r.lo[0]); c_hi = imin64(c_hi, r.hi[0]);
  n_lo = imax64(n_lo, r.lo[1]); n_hi = imin64(n_hi, r.hi[1]);
  if (c_hi <= c_lo) c_lo = c_hi = 0;
  if (n_hi <= n_lo) n_lo = n_hi = 0;
}

BDLM_HD bool visible(const Geom& g, int stream, int64_t i, int key_stream, int64_t j) {
  int64_t lo, hi;
  if (key_stream == 0) clean_interval(g, stream, i, lo, hi);
  else noisy_interval(g, stream, i, lo, hi);
  return j >= lo && j < hi;
}

// Key-tile ranges [c0, c1) (clean) and [n0, n1) (corrupted) in units of tk
// keys that the query rows [r0, r1) of `stream` can see, and for each range
// the key interval every row of the tile sees (to tell full tiles from
// partial ones).
struct QTileRanges {
  int64_t c0, c1, n0, n1;          // tile ranges
  int64_t c_all_lo, c_all_hi;      // clean keys seen by every row
  int64_t n_all_lo, n_all_hi;      // corrupted keys seen by every row
};

BDLM_HD QTileRanges qtile_ranges(const Geom& g, int stream, int64_t r0, int64_t r1, int tk) {
  QTileRanges q;
  int64_t lo_first, hi_first, lo_last, hi_last;
  clean_interval(g, stream, r0, lo_first, hi_first);
  clean_interval(g, stream, r1 - 1, lo_last, hi_last);
  // union over rows: [kv_begin, hi of the last row); intersection: [kv_begin, hi of the first row)
  if (hi_last > lo_last) {
    q.c0 = lo_last / tk;
    q.c1 = cdiv64(hi_last, tk);
  } else {
    q.c0 = q.c1 = 0;
  }
  q.c_all_lo = lo_first;
  q.c_all_hi = hi_first;
  int64_t nlo_first, nhi_first, nlo_last, nhi_last;
  noisy_interval(g, stream, r0, nlo_first, nhi_first);
  noisy_interval(g, stream, r1 - 1, nlo_last, nhi_last);
  if (nhi_last > nlo_first) {
    q.n0 = nlo_first / tk;
    q.n1 = cdiv64(nhi_last, tk);
  } else {
    q.n0 = q.n1 = 0;
  }
  q.n_all_lo = nlo_last;   // largest lower bound
  q.n_all_hi = nhi_first;  // smallest upper bound
  return q;
}

// True when every (row, key) pair of the key tile [j0, j0 + tk) is visible to
// every row of the query tile and the tile lies inside the sequence.
BDLM_HD bool tile_full(int64_t j0, int tk, int64_t all_lo, int64_t all_hi, int64_t L) {
  return j0 >= all_lo && j0 + tk <= all_hi && j0 + tk <= L;
}

// Forward / dQ work items: (query tile, head, stream), longest first.  For a
// fixed shard the visible key count of a query tile never decreases with its
// position, so query tiles are taken from the last to the first.  With many
// query tiles (at least kBlockedMinQBlocks blocks) they go in blocks of
// q_block() tiles, and inside a block the items of one KV head (its query
// heads, both streams) come together, one KV head after the other: such a
// block is about one round of the persistent grid (g.round_items CTAs, one
// per SM), whose key sweeps
// then read one head's K and V, which fit in L2, instead of every head's.
// Otherwise, inside one query-tile index the two streams of one head are
// adjacent, then the heads.  (The kernels also start each item's clean-key
// sweep at a different tile, so that the items of a round do not all read
// the same tile at once.)
struct QItem {
  int stream, head;
  int64_t qtile;
};

constexpr int64_t kBlockedMinQBlocks = 6;

BDLM_HD int64_t q_items(const Geom& g, int tq) { return cdiv64(g.L, tq) * g.Hq * 2; }

BDLM_HD int64_t q_block(const Geom& g) {
  const int64_t per_kv = (int64_t)(g.Hq / g.Hkv) * 2;  // items per query tile and KV head
  const int64_t qb = g.round_items / per_kv;
  return qb > 0 ? qb : 1;
}

BDLM_HD QItem q_item(const Geom& g, int tq, int64_t idx) {
  const int64_t nqt = cdiv64(g.L, tq);
  const int64_t qb = q_block(g);
  QItem it;
  if (g.naive_order) {  // natural order: first query tile first
    const int64_t per = (int64_t)g.Hq * 2;
    it.qtile = idx / per;
    const int64_t rem = idx % per;
    it.stream = (int)(rem % 2);
    it.head = (int)(rem / 2);
    return it;
  }
  if (nqt < kBlockedMinQBlocks * qb) {
    const int64_t per = (int64_t)g.Hq * 2;
    it.qtile = nqt - 1 - idx / per;
    const int64_t rem = idx % per;
    it.stream = (int)(rem % 2);
    it.head = (int)(rem / 2);
    return it;
  }
  const int grp = g.Hq / g.Hkv;
  const int64_t per_kv = (int64_t)grp * 2;
  const int64_t per_block = qb * g.Hq * 2;  // items of a full block
  const int64_t bi = idx / per_block;
  const int64_t hi = nqt - 1 - bi * qb;      // first (largest) query tile of the block
  const int64_t lo = imax64(0, hi - qb + 1);
  const int64_t nb = hi - lo + 1;            // query tiles in this block
  const int64_t r = idx - bi * per_block;
  const int64_t kv = r / (nb * per_kv);
  const int64_t r2 = r - kv * (nb * per_kv);
  const int64_t combo = r2 % per_kv;
  it.qtile = hi - r2 / per_kv;
  it.stream = (int)(combo % 2);
  it.head = (int)(kv * grp + combo / 2);
  return it;
}

// Work items of a row-restricted call (one rank's rows of a multi-rank
// deployment): only the query tiles that hold rows of the call's range, so
// that the persistent grid's rounds stay full.  Per stream those tiles are
// one range [t0, t1); the two ranges are merged by tile index, largest
// first (the clean tile before the corrupted one of the same index: a
// query tile's visible key count grows with its index in either stream),
// and the merged list takes the place of the query tiles in the blocked,
// longest-first order above, one stream per entry.
BDLM_HD void range_tiles(const Geom& g, const RowRange& r, int stream, int tq, int64_t& t0, int64_t& t1) {
  const int64_t lo = range_lo(r, stream), hi = imin64(range_hi(r, stream), g.L);
  if (hi <= lo) {
    t0 = t1 = 0;
    return;
  }
  t0 = lo / tq;
  t1 = cdiv64(hi, tq);
}

// Tiles of [t0, t1) at index t or above.
BDLM_HD int64_t tiles_at_least(int64_t t0, int64_t t1, int64_t t) {
  const int64_t lo = imax64(t0, t);
  return t1 > lo ? t1 - lo : 0;
}

struct RowTiles {
  int64_t a0, a1, b0, b1;  // clean and corrupted tile ranges
  BDLM_HD int64_t at_least(int64_t t) const { return tiles_at_least(a0, a1, t) + tiles_at_least(b0, b1, t); }
  BDLM_HD int64_t count() const { return at_least(0); }
};

BDLM_HD RowTiles row_tiles(const Geom& g, const RowRange& r, int tq) {
  RowTiles rt;
  range_tiles(g, r, 0, tq, rt.a0, rt.a1);
  range_tiles(g, r, 1, tq, rt.b0, rt.b1);
  return rt;
}

// Entry v (0 <= v < count) of the merged list: its tile and stream.  The
// tile is the largest t with more than v entries at index t or above
// (binary search: that count falls as t grows).
BDLM_HD void row_tile_at(const RowTiles& rt, int64_t v, int64_t& tile, int& stream) {
  int64_t lo = 0, hi = imax64(rt.a1, rt.b1);  // at_least(lo) > v >= at_least(hi) = 0
  while (hi - lo > 1) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (rt.at_least(mid) > v) lo = mid;
    else hi = mid;
  }
  tile = lo;
  const bool in_a = lo >= rt.a0 && lo < rt.a1;
  const int64_t first = rt.at_least(lo + 1);  // entries of larger tiles come first
  stream = (in_a && v == first) ? 0 : 1;
}

BDLM_HD int64_t q_items_rows(const Geom& g, const RowRange& r, int tq) { return row_tiles(g, r, tq).count() * g.Hq; }

// Entry and head of item idx of a segment of ne merged entries: blocks of qb
// entries, one KV head after the other inside a block (or the heads of one
// entry together when the segment is short).
BDLM_HD void segment_item(int64_t ne, int64_t qb, int grp, int Hq, int64_t idx, int64_t& e, int& head) {
  if (ne < kBlockedMinQBlocks * qb) {
    e = idx / Hq;
    head = (int)(idx % Hq);
    return;
  }
  const int64_t per_block = qb * Hq;
  const int64_t bi = idx / per_block;
  const int64_t e0 = bi * qb;
  const int64_t nb = imin64(qb, ne - e0);
  const int64_t rr = idx - bi * per_block;
  const int64_t kv = rr / (nb * grp);
  const int64_t r2 = rr - kv * (nb * grp);
  e = e0 + r2 / grp;
  head = (int)(kv * grp + r2 % grp);
}

// When the two tile ranges do not overlap the merged list is the upper range
// followed by the lower one, and each is blocked on its own, so that no
// block (about one grid round) mixes the long items of one with the short
// items of the other.
BDLM_HD QItem q_item_rows(const Geom& g, const RowRange& r, int tq, int64_t idx) {
  const RowTiles rt = row_tiles(g, r, tq);
  const int64_t n = rt.count();
  const int grp = g.Hq / g.Hkv;
  const int64_t qb = imax64(g.round_items / grp, 1);  // entries per block: about one grid round
  const bool disjoint = rt.a1 <= rt.b0 || rt.b1 <= rt.a0;
  const int64_t n0 = disjoint ? (rt.a0 >= rt.b1 ? rt.a1 - rt.a0 : rt.b1 - rt.b0) : n;  // first segment
  int64_t e;
  QItem it;
  if (idx < n0 * g.Hq) {
    segment_item(n0, qb, grp, g.Hq, idx, e, it.head);
  } else {
    segment_item(n - n0, qb, grp, g.Hq, idx - n0 * g.Hq, e, it.head);
    e += n0;
  }
  row_tile_at(rt, e, it.qtile, it.stream);
  return it;
}

// First clean key tile of an item's sweep, relative to its clean range of nc
// tiles: items that run together start at different tiles.
// (32-bit arithmetic: item indices stay far below 2^32.)
BDLM_HD int sweep_rotation(int64_t idx, int nc) {
  return nc > 0 ? (int)((uint32_t)idx % (uint32_t)nc) : 0;
}

// Below this many key tiles per key stream (six grid rounds) the dK/dV list
// stays tile-major: blocks would then cover tiles of very different lengths,
// and the long items of a late block can end after everything else.
BDLM_HD int64_t kv_blocked_min_tiles(const Geom& g) { return 6 * (int64_t)g.round_items; }

// The geometry of one sequence of a packed batch: rows [off, off + L) of the
// packed tensors, all of its clean keys, its own corrupted block included.
BDLM_HD Geom seq_geom(const Geom& all, int64_t L) {
  Geom g = all;
  g.L = L;
  g.kv_begin = 0;
  g.kv_end = L;
  g.include_local = 1;
  return g;
}

// dK/dV work items: (key stream, key/value head, key tile).  Clean key tiles
// first in increasing position (a clean key is read by every later row, so
// earlier tiles carry more work), then corrupted key tiles (each read only by
// its own block's rows).  A long range (at least kv_blocked_min_tiles) goes
// in blocks of g.round_items tiles (one grid round) with one KV head after
// the other inside a block, so the items running together read one head's Q
// and dO; a short range goes tile by tile with the KV heads inside.  Only
// tiles that intersect this call's keys count.
struct KVItem {
  int key_stream, kv_head;
  int64_t ktile;
};

BDLM_HD void kv_tile_span(const Geom& g, int tk, int64_t& c_first, int64_t& c_count, int64_t& n_count) {
  if (g.kv_end > g.kv_begin) {
    c_first = g.kv_begin / tk;
    c_count = cdiv64(g.kv_end, tk) - c_first;
  } else {
    c_first = 0;
    c_count = 0;
  }
  n_count = g.include_local ? cdiv64(g.L, tk) : 0;
}

BDLM_HD int64_t kv_items(const Geom& g, int tk) {
  int64_t cf, cc, nc;
  kv_tile_span(g, tk, cf, cc, nc);
  return (cc + nc) * g.Hkv;
}

BDLM_HD KVItem kv_item(const Geom& g, int tk, int64_t idx) {
  int64_t cf, cc, nc;
  kv_tile_span(g, tk, cf, cc, nc);
  KVItem it;
  int64_t i = idx, base = cf, count = cc;
  it.key_stream = 0;
  if (idx >= cc * g.Hkv) {
    i = idx - cc * g.Hkv;
    base = 0;
    count = nc;
    it.key_stream = 1;
  }
  if (count < kv_blocked_min_tiles(g) || g.naive_order) {
    // short range: tile-major, KV head minor (rounds of similar lengths)
    it.kv_head = (int)(i % g.Hkv);
    it.ktile = base + i / g.Hkv;
    return it;
  }
  // long range: blocks of g.round_items tiles, one KV head after the other
  // inside a block; a block of one head is about one grid round
  const int64_t R = g.round_items;
  const int64_t bi = i / (R * g.Hkv);
  const int64_t t0 = bi * R;
  const int64_t nb = imin64(R, count - t0);
  const int64_t r = i - t0 * g.Hkv;
  it.kv_head = (int)(r / nb);
  it.ktile = base + t0 + r % nb;
  return it;
}

// Query rows that can see some key of the key tile [j0, j1) of `key_stream`:
// [c_lo, L) of clean rows and [n_lo, n_hi) of corrupted rows (empty if
// hi <= lo).  A clean key of block b is read by clean rows of blocks >= b and
// corrupted rows of blocks > b; a corrupted key only by its own block's
// corrupted rows.  Keys outside this call's key set see no rows.
BDLM_HD void kv_tile_rows(const Geom& g, int key_stream, int64_t j0, int64_t j1,
                          int64_t& c_lo, int64_t& c_hi, int64_t& n_lo, int64_t& n_hi) {
  if (key_stream == 0) {
    const int64_t a = imax64(j0, g.kv_begin), z = imin64(j1, g.kv_end);
    if (z <= a) { c_lo = c_hi = n_lo = n_hi = 0; return; }
    const int64_t b = a / g.B;
    c_lo = b * g.B; c_hi = g.L;
    n_lo = (b + 1) * g.B; n_hi = g.L;
  } else {
    c_lo = c_hi = 0;
    if (!g.include_local) { n_lo = n_hi = 0; return; }
    n_lo = (j0 / g.B) * g.B;
    n_hi = imin64(g.L, ((j1 - 1) / g.B + 1) * g.B);
  }
}

}  // namespace bdlm
