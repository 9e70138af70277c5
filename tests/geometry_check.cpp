// Host check of the work orders in geometry.cuh (compiled with g++ by
// tests/test_geometry_host.py): every enumeration the kernels walk must visit
// each work item exactly once, for blocked and unblocked lists, sharded key
// ranges and the natural (ablation) order.  Prints one line per failure and
// exits non-zero if any.
#include <cstdio>
#include <cstdlib>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "geometry.cuh"

using namespace bdlm;

static int failures = 0;
#define CHECK(cond, ...)                     \
  do {                                       \
    if (!(cond)) {                           \
      ++failures;                            \
      if (failures < 20) {                   \
        std::printf("FAIL %s: ", #cond);     \
        std::printf(__VA_ARGS__);            \
        std::printf("\n");                   \
      }                                      \
    }                                        \
  } while (0)

// (stream, head, query tile) items of the forward / dQ lists.
static void check_q(const Geom& g, int tq) {
  const int64_t nqt = cdiv64(g.L, tq);
  const int64_t n = q_items(g, tq);
  CHECK(n == nqt * g.Hq * 2, "L=%lld tq=%d", (long long)g.L, tq);
  std::vector<unsigned char> seen((size_t)n, 0);
  for (int64_t i = 0; i < n; ++i) {
    const QItem it = q_item(g, tq, i);
    const bool ok = it.stream >= 0 && it.stream < 2 && it.head >= 0 && it.head < g.Hq && it.qtile >= 0 &&
                    it.qtile < nqt;
    CHECK(ok, "q item %lld out of range (L=%lld Hq=%d Hkv=%d tq=%d)", (long long)i, (long long)g.L, g.Hq, g.Hkv,
          tq);
    if (!ok) continue;
    const int64_t key = (it.qtile * g.Hq + it.head) * 2 + it.stream;
    CHECK(!seen[(size_t)key], "q item repeated (L=%lld tq=%d idx=%lld)", (long long)g.L, tq, (long long)i);
    seen[(size_t)key] = 1;
  }
  // rotation of the clean-key sweep stays inside the range
  for (int64_t i = 0; i < n; i += 97)
    for (int nc = 1; nc < 600; nc += 37) {
      const int r = sweep_rotation(i, nc);
      CHECK(r >= 0 && r < nc, "rotation %d of %d", r, nc);
    }
}

// Items of a row-restricted call: exactly the (stream, head, query tile)
// whose tile holds rows of the range, each once; the merged tile list runs
// from the largest tile down, and inside each stream tiles never increase
// along the list in the unblocked order.
static void check_q_rows(const Geom& g, const RowRange& r, int tq) {
  const int64_t nqt = cdiv64(g.L, tq);
  std::vector<unsigned char> want((size_t)(nqt * g.Hq * 2), 0);
  int64_t n_want = 0;
  for (int s = 0; s < 2; ++s)
    for (int64_t t = 0; t < nqt; ++t) {
      const int64_t r0 = t * tq, r1 = imin64(r0 + tq, g.L);
      if (!tile_in(r, s, r0, r1)) continue;
      for (int h = 0; h < g.Hq; ++h) {
        want[(size_t)((t * g.Hq + h) * 2 + s)] = 1;
        ++n_want;
      }
    }
  const int64_t n = q_items_rows(g, r, tq);
  CHECK(n == n_want, "rows item count %lld vs %lld (L=%lld tq=%d)", (long long)n, (long long)n_want,
        (long long)g.L, tq);
  const RowTiles rt = row_tiles(g, r, tq);
  int64_t prev = 1LL << 62;
  for (int64_t v = 0; v < rt.count(); ++v) {  // merged list: largest tile first, each (tile, stream) once
    int64_t t;
    int s;
    row_tile_at(rt, v, t, s);
    const bool in = s == 0 ? (t >= rt.a0 && t < rt.a1) : (t >= rt.b0 && t < rt.b1);
    CHECK(in && t <= prev, "merged entry %lld -> tile %lld stream %d", (long long)v, (long long)t, s);
    if (v > 0 && t == prev) {
      int64_t tp;
      int sp;
      row_tile_at(rt, v - 1, tp, sp);
      CHECK(sp == 0 && s == 1, "equal tiles: clean first (entry %lld)", (long long)v);
    }
    prev = t;
  }
  std::vector<unsigned char> seen(want.size(), 0);
  for (int64_t i = 0; i < n; ++i) {
    const QItem it = q_item_rows(g, r, tq, i);
    const bool ok = it.stream >= 0 && it.stream < 2 && it.head >= 0 && it.head < g.Hq && it.qtile >= 0 &&
                    it.qtile < nqt;
    CHECK(ok, "rows item %lld out of range (L=%lld tq=%d)", (long long)i, (long long)g.L, tq);
    if (!ok) continue;
    const size_t key = (size_t)((it.qtile * g.Hq + it.head) * 2 + it.stream);
    CHECK(want[key], "rows item %lld outside the range (tile %lld stream %d)", (long long)i, (long long)it.qtile,
          it.stream);
    CHECK(!seen[key], "rows item %lld repeated", (long long)i);
    seen[key] = 1;
  }
}

// (key stream, KV head, key tile) items of the dK/dV list.// (key stream, KV head, key tile) items of the dK/dV list.
static void check_kv(const Geom& g, int tk) {
  int64_t cf, cc, nn;
  kv_tile_span(g, tk, cf, cc, nn);
  const int64_t n = kv_items(g, tk);
  CHECK(n == (cc + nn) * g.Hkv, "kv count L=%lld", (long long)g.L);
  const int64_t ntile = cdiv64(g.L, tk);
  std::vector<unsigned char> seen((size_t)(2 * g.Hkv * ntile), 0);
  for (int64_t i = 0; i < n; ++i) {
    const KVItem it = kv_item(g, tk, i);
    const bool in_span = it.key_stream == 0 ? (it.ktile >= cf && it.ktile < cf + cc) : (it.ktile >= 0 && it.ktile < nn);
    const bool ok = (it.key_stream == 0 || it.key_stream == 1) && it.kv_head >= 0 && it.kv_head < g.Hkv && in_span;
    CHECK(ok, "kv item %lld out of range (L=%lld kv=[%lld,%lld) local=%d)", (long long)i, (long long)g.L,
          (long long)g.kv_begin, (long long)g.kv_end, g.include_local);
    if (!ok) continue;
    const int64_t key = ((int64_t)it.key_stream * g.Hkv + it.kv_head) * ntile + it.ktile;
    CHECK(!seen[(size_t)key], "kv item repeated (L=%lld idx=%lld)", (long long)g.L, (long long)i);
    seen[(size_t)key] = 1;
  }
}

// Per-CTA totals when the persistent CTAs claim a list's items in order,
// each item going to the CTA that becomes free first (the kernels' dynamic
// claiming, every CTA equally fast, ties to the lowest index).  With this
// greedy rule no CTA ends more than one item's cost after another.
static std::vector<double> claim_totals(const std::vector<double>& costs, int grid) {
  typedef std::pair<double, int> Slot;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
  for (int c = 0; c < grid; ++c) free_at.push(Slot(0.0, c));
  std::vector<double> tot((size_t)grid, 0.0);
  for (double cost : costs) {
    const Slot s = free_at.top();
    free_at.pop();
    tot[(size_t)s.second] = s.first + cost;
    free_at.push(Slot(tot[(size_t)s.second], s.second));
  }
  return tot;
}

// Brute-force visibility (the mask, with the call's key restriction and,
// for the key-tile row ranges, the call's row range).
static RowRange g_rows;  // the row range under test (default: every row)
static bool sees(const Geom& g, int s, int64_t i, int ks, int64_t j) {
  const int64_t bi = i / g.B, bj = j / g.B;
  if (i < g_rows.lo[s] || i >= g_rows.hi[s]) return false;
  if (ks == 0) {
    if (j < g.kv_begin || j >= g.kv_end) return false;
    return s == 0 ? bj <= bi : bj < bi;
  }
  return g.include_local && s == 1 && bj == bi;
}

// kv_tile_rows (the rows a key tile is read by) and qtile_ranges (the key
// tiles a query tile reads, and the keys all its rows see) against the mask.
static void check_ranges(const Geom& g, int t) {
  const int64_t nt = cdiv64(g.L, t);
  for (int ks = 0; ks < 2; ++ks)
    for (int64_t kt = 0; kt < nt; ++kt) {
      const int64_t j0 = kt * t, j1 = imin64(j0 + t, g.L);
      int64_t r[4];
      kv_tile_rows(g, ks, j0, j1, r[0], r[1], r[2], r[3]);
      clamp_rows(g_rows, r[0], r[1], r[2], r[3]);
      for (int s = 0; s < 2; ++s) {
        const int64_t lo = r[2 * s], hi = r[2 * s + 1];
        for (int64_t i = 0; i < g.L; ++i) {
          bool any = false;
          for (int64_t j = j0; j < j1 && !any; ++j) any = sees(g, s, i, ks, j);
          CHECK(any == (i >= lo && i < hi), "kv_tile_rows ks=%d tile=%lld s=%d row=%lld (L=%lld B=%lld)", ks,
                (long long)kt, s, (long long)i, (long long)g.L, (long long)g.B);
        }
      }
    }
  // (qtile_ranges covers every row of a tile: the forward and dQ skip
  // tiles without any of the call's rows and write only the call's rows)
  if (g_rows.lo[0] != 0 || g_rows.lo[1] != 0 || g_rows.hi[0] < g.L || g_rows.hi[1] < g.L) return;
  for (int s = 0; s < 2; ++s)
    for (int64_t qt = 0; qt < nt; ++qt) {
      const int64_t r0 = qt * t, r1 = imin64(r0 + t, g.L);
      const QTileRanges q = qtile_ranges(g, s, r0, r1, t);
      for (int ks = 0; ks < 2; ++ks)
        for (int64_t kt = 0; kt < nt; ++kt) {
          const int64_t j0 = kt * t, j1 = imin64(j0 + t, g.L);
          bool any = false;
          for (int64_t i = r0; i < r1 && !any; ++i)
            for (int64_t j = j0; j < j1 && !any; ++j) any = sees(g, s, i, ks, j);
          const bool listed = ks == 0 ? (kt >= q.c0 && kt < q.c1) : (kt >= q.n0 && kt < q.n1);
          CHECK(any == listed, "qtile_ranges s=%d qtile=%lld ks=%d ktile=%lld (L=%lld B=%lld)", s, (long long)qt,
                ks, (long long)kt, (long long)g.L, (long long)g.B);
        }
      // keys every row of the tile sees: exactly the stated intervals
      for (int64_t j = 0; j < g.L; ++j) {
        bool all_c = true, all_n = true;
        for (int64_t i = r0; i < r1; ++i) {
          all_c = all_c && sees(g, s, i, 0, j);
          all_n = all_n && sees(g, s, i, 1, j);
        }
        CHECK(all_c == (j >= q.c_all_lo && j < q.c_all_hi), "c_all s=%d qtile=%lld key=%lld", s, (long long)qt,
              (long long)j);
        CHECK(all_n == (j >= q.n_all_lo && j < q.n_all_hi), "n_all s=%d qtile=%lld key=%lld", s, (long long)qt,
              (long long)j);
      }
    }
}

// Per-CTA totals of the dynamic claiming over a work list, with the list's
// own costs (visible key tiles of a query item; query rows reading a key
// tile): over a longest-first (or blocked) list every CTA ends within
// max_over_mean of the mean, and within one item of every other CTA.
static void check_balance(const Geom& g, int grid, bool kv, double max_over_mean) {
  const int tq = 256, tk = 128;
  const int64_t n = kv ? kv_items(g, tk) : q_items(g, tq);
  std::vector<double> costs;
  double cmax = 0.0, sum = 0.0;
  for (int64_t idx = 0; idx < n; ++idx) {
      double cost;
      if (kv) {
        const KVItem it = kv_item(g, tk, idx);
        int64_t cl, ch, nl, nh;
        kv_tile_rows(g, it.key_stream, it.ktile * tk, imin64(it.ktile * tk + tk, g.L), cl, ch, nl, nh);
        cost = (double)(imax64(0, ch - cl) + imax64(0, nh - nl));
      } else {
        const QItem it = q_item(g, tq, idx);
        const int64_t r0 = it.qtile * tq;
        const QTileRanges q = qtile_ranges(g, it.stream, r0, imin64(r0 + tq, g.L), tk);
        cost = (double)((q.c1 - q.c0) + (q.n1 - q.n0));
      }
      costs.push_back(cost);
      cmax = cost > cmax ? cost : cmax;
      sum += cost;
  }
  const std::vector<double> tot = claim_totals(costs, grid);
  double mx = 0.0, mn = 1e300;
  for (double t : tot) { mx = t > mx ? t : mx; mn = t < mn ? t : mn; }
  const double mean = sum / grid;
  CHECK(mx <= mean * max_over_mean, "balance %s grid=%d L=%lld: max %.0f mean %.0f (ratio %.4f)", kv ? "kv" : "q",
        grid, (long long)g.L, mx, mean, mx / mean);
  CHECK(mx - mn <= cmax, "spread %s grid=%d L=%lld: max %.0f min %.0f item %.0f", kv ? "kv" : "q", grid,
        (long long)g.L, mx, mn, cmax);
}

// The same per-CTA balance over a row-restricted list (one rank's rows):
// no CTA more than two items' cost above the mean.
static void check_balance_rows(const Geom& g, const RowRange& rows, int grid, int tq) {
  const int tk = 128;
  const int64_t n = q_items_rows(g, rows, tq);
  std::vector<double> costs;
  double sum = 0.0, cmax = 0.0;
  for (int64_t idx = 0; idx < n; ++idx) {
    const QItem it = q_item_rows(g, rows, tq, idx);
    const int64_t r0 = it.qtile * tq;
    const QTileRanges q = qtile_ranges(g, it.stream, r0, imin64(r0 + tq, g.L), tk);
    const double cost = (double)((q.c1 - q.c0) + (q.n1 - q.n0));
    costs.push_back(cost);
    sum += cost;
    cmax = cost > cmax ? cost : cmax;
  }
  const std::vector<double> tot = claim_totals(costs, grid);
  double mx = 0.0;
  for (double t : tot) mx = t > mx ? t : mx;
  CHECK(mx <= sum / grid + 2 * cmax, "rows balance grid=%d L=%lld tq=%d rows c[%d,%d) n[%d,%d): max %.0f mean %.0f item %.0f",
        grid, (long long)g.L, tq, rows.lo[0], rows.hi[0], rows.lo[1], rows.hi[1], mx, sum / grid, cmax);
}

int main() {
  const int64_t Ls[] = {96, 256, 1024, 8192, 16384, 32768, 131072, 262144};
  const int64_t Bs[] = {32, 128, 512};
  const int heads[][2] = {{2, 2}, {16, 8}, {32, 8}, {40, 8}, {8, 4}, {5, 1}};
  for (int naive = 0; naive < 2; ++naive)
    for (int64_t L : Ls)
      for (int64_t B : Bs) {
        if (L % B) continue;
        for (const auto& h : heads) {
          Geom g{L, B, h[0], h[1], 0, L, 1};
          g.naive_order = naive;
          for (int tq : {128, 256}) check_q(g, tq);
          check_kv(g, 128);
          // clean-key shards (CSBP), with and without the local block
          const int P = 8;
          if (L % P == 0)
            for (int s = 0; s < P; s += 3) {
              Geom gs = g;
              gs.kv_begin = s * (L / P);
              gs.kv_end = (s + 1) * (L / P);
              gs.include_local = 0;
              check_kv(gs, 128);
              for (int tq : {128, 256}) check_q(gs, tq);
            }
          Geom gl = g;
          gl.kv_begin = gl.kv_end = 0;  // the local partial alone
          check_kv(gl, 128);
          // one sequence of a packed batch
          const Geom gp = seq_geom(g, L / 2 - (L / 2) % B > 0 ? L / 2 - (L / 2) % B : B);
          check_kv(gp, 128);
          check_q(gp, 128);
        }
        Geom g{L, B, 16, 8, 0, L, 1};
        g.naive_order = naive;
      }
  // the work-order blocking follows the grid: one round of the persistent
  // grid per block, for devices of 132, 148 and 152 SMs
  for (int grid : {132, 148, 152})
    for (int64_t L : {16384, 32768, 131072, 262144})
      for (const auto& h : heads) {
        const int64_t B = 512;
        Geom g{L, B, h[0], h[1], 0, L, 1};
        g.round_items = grid;
        for (int tq : {128, 256}) check_q(g, tq);
        check_kv(g, 128);
        Geom gs = g;
        gs.kv_begin = L / 8;
        gs.kv_end = L / 4;
        gs.include_local = 0;
        check_kv(gs, 128);
        check_q(gs, 128);
        if (L >= 131072) {
          check_balance(g, grid, false, 1.02);
          check_balance(g, grid, true, 1.05);
        }
      }
  // one rank's rows at full size: the mirror and the by-position
  // assignments of an R-rank plan, and rows not aligned to tiles
  for (int64_t L : {16384, 131072, 262144})
    for (const auto& h : heads)
      for (int R : {2, 4, 8}) {
        Geom g{L, 512, h[0], h[1], 0, L, 1};
        const int64_t sl = L / R;
        for (int r = 0; r < R; ++r)
          for (int mirror = 0; mirror < 2; ++mirror) {
            RowRange rows;
            rows.lo[0] = (int32_t)(r * sl);
            rows.hi[0] = (int32_t)((r + 1) * sl);
            const int64_t m = mirror ? R - 1 - r : r;
            rows.lo[1] = (int32_t)(m * sl + (mirror ? 0 : 77));
            rows.hi[1] = (int32_t)((m + 1) * sl - (mirror ? 0 : 13));
            for (int tq : {128, 256}) check_q_rows(g, rows, tq);
            if (L >= 131072)
              for (int tq : {128, 256}) check_balance_rows(g, rows, 152, tq);
          }
      }
  // tile ranges against the mask on small shapes: tiles smaller than,
  // equal to and larger than the blocks, ragged tails, shards, no local block
  for (int64_t L : {48, 96, 160, 256})
    for (int64_t B : {1, 8, 16, 32, 48})
      for (int t : {16, 32, 64}) {
        if (L % B) continue;
        for (int v = 0; v < 6; ++v) {
          Geom g{L, B, 2, 1, 0, L, 1};
          if (v == 1) { g.kv_begin = L / 4; g.kv_end = L / 2; }
          if (v == 2) { g.kv_begin = L / 3; g.kv_end = L; g.include_local = 0; }
          if (v == 3) { g.kv_begin = g.kv_end = 0; }
          g_rows = RowRange();
          if (v == 4) {  // one rank's rows: a clean slice and another corrupted slice
            g_rows.lo[0] = (int32_t)(L / 4); g_rows.hi[0] = (int32_t)(L / 2);
            g_rows.lo[1] = (int32_t)(L / 2); g_rows.hi[1] = (int32_t)(3 * L / 4);
          }
          if (v == 5) {  // rows not aligned to tiles, with a key shard
            g_rows.lo[0] = 5; g_rows.hi[0] = (int32_t)(L - 7);
            g_rows.lo[1] = (int32_t)(L / 3); g_rows.hi[1] = (int32_t)(L / 3 + 9);
            g.kv_begin = L / 8; g.kv_end = L / 2;
          }
          check_ranges(g, t);
          if (v >= 4) check_q_rows(g, g_rows, t);
          g_rows = RowRange();
        }
      }
  if (failures) {
    std::printf("%d failures\n", failures);
    return 1;
  }
  std::printf("ok\n");
  return 0;
}
