// bwd_dkv.cu -- dK/dV pass of the two-stream BDLM attention backward (sm_103a).
//
// dV = sum_group P^T dO and dK = scale sum_group dS^T Q over each key row's
// visible query rows (see bwd_common.cuh for the gradient definitions and
// their source).
//
// Item = (128-row key tile, KV head, key stream).  K and V of the item stay in
// shared memory; 128-row Q/dO tiles of every query head of the GQA group
// (clean rows, then corrupted rows, only those that see some key of the
// tile) stream through a 2-stage TMA ring together with their LSE and D.
// TMEM holds dK (columns 0..), dV (128..), S^T (256..383) and dP^T
// (384..511), the last two single-buffered.  Per step k, MMA warp:
//   S^T(k)  = K Q^T                              -> S^T columns
//   dK     += dS^T(k-1) Q(k-1)                   (dS^T packed over dP^T)
//   dP^T(k) = V dO^T                             -> dP^T columns
//   dV     += P^T(k) dO(k)                       (P^T packed over S^T)
// The elementwise warps (thread = key row, 64 query rows per warpgroup) first
// turn S^T into P (kept in registers) and P^T (bf16, written back), which
// releases dV(k) and, behind it in the tensor pipe, S^T(k+1); then they form
// dS^T from dP^T, which releases dK(k) and dP^T(k+1).  With every MMA at
// N = 128 the pipe stays busy while either half of the elementwise work runs.
#include "bwd_common.cuh"
#include "sched.cuh"

namespace bdlm {
namespace {

using namespace bwd;

constexpr int KBM = 128;  // keys per item
constexpr int KBN = 128;  // query rows per step
constexpr int QNS = 2;    // Q/dO stages

enum { KV_KF = 0, KV_KE = 1, KV_QF = 2, KV_QE = 4, KV_SF = 6, KV_DPF = 7, KV_PF = 8, KV_DSF = 9, KV_ACCDONE = 10,
       KV_ACCE = 11,
       KV_IF = 12, KV_IE = 12 + kRingSlots, KV_NBAR = 12 + 2 * kRingSlots };
// The 256 bytes after the tiles: barriers, the TMEM address, the abort flag,
// the work-item ring's slots.
static_assert(8 * KV_NBAR + 8 + 8 * kRingSlots <= 256, "barrier area overflows");

template <int HD>
struct DkvLayout {
  static constexpr int kTile = 128 * HD * 2;  // 128 rows x HD bf16
  static constexpr int kPanel = 128 * 128;    // 128 rows x 64 bf16
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;
  static constexpr int kdO = kQ + QNS * kTile;
  static constexpr int kStat = kdO + QNS * kTile;  // per stage: LSE[128] then D[128], fp32
  static constexpr int kBar = kStat + QNS * 2 * KBN * 4;
  static constexpr int kGeo = kBar + 256;  // the work-item ring's geometry slots
  static constexpr int kBytes = kGeo + 512;
  static constexpr int kAlloc = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
};

struct DkvGeo {
  int ks, kvh;
  int64_t j0;
  int64_t rlo0, rhi0, rlo1, rhi1;  // query rows of each stream that can see some key of the tile
  int64_t t00, t01;                // first query tile of each stream
  int nt0, nt1;                    // query tiles of each stream
  int per_head, n;                 // steps per head, total steps
  int64_t off, L;                  // first row of the item's sequence in the packed tensors, its length
};
static_assert(kRingSlots * sizeof(DkvGeo) <= 512, "geometry slots overflow");

// VL: packed variable-length batch; ROWS: the call computes a row range
// (separate instantiations).
template <bool VL, bool ROWS>
__device__ __forceinline__ DkvGeo dkv_geo(const BwdParams& p, const VarlenTabs& vt, int64_t idx) {
  DkvGeo t;
  Geom g = p.g;
  t.off = 0;
  if (VL) {  // packed batch: the item and its sequence from the tables
    const int4 e = vt.kv_items[idx];
    t.ks = e.y & 1;
    t.kvh = e.y >> 1;
    t.j0 = (int64_t)e.z * KBM;
    t.off = vt.seq_off[e.x];
    g = seq_geom(p.g, vt.seq_off[e.x + 1] - t.off);
  } else {
    const KVItem it = kv_item(p.g, KBM, idx);
    t.ks = it.key_stream;
    t.kvh = it.kv_head;
    t.j0 = it.ktile * KBM;
  }
  t.L = g.L;
  const int64_t j1 = imin64(t.j0 + KBM, g.L);
  kv_tile_rows(g, t.ks, t.j0, j1, t.rlo0, t.rhi0, t.rlo1, t.rhi1);
  if (ROWS) clamp_rows(p.rows, t.rlo0, t.rhi0, t.rlo1, t.rhi1);  // only the call's rows
  if (t.rhi0 > t.rlo0) {
    t.t00 = t.rlo0 / KBN;
    t.nt0 = (int)(cdiv64(t.rhi0, KBN) - t.t00);
  } else {
    t.t00 = 0;
    t.nt0 = 0;
  }
  if (t.rhi1 > t.rlo1) {
    t.t01 = t.rlo1 / KBN;
    t.nt1 = (int)(cdiv64(t.rhi1, KBN) - t.t01);
  } else {
    t.t01 = 0;
    t.nt1 = 0;
  }
  t.per_head = t.nt0 + t.nt1;
  t.n = t.per_head * (p.g.Hq / p.g.Hkv);
  return t;
}

// Walks the steps of an item in order: query heads of the GQA group, and for
// each head the query tiles of the clean rows, then of the corrupted rows.
struct DkvCursor {
  int hh, r;  // head within the group, tile index within the head's steps
  __device__ __forceinline__ void reset() { hh = 0; r = 0; }
  __device__ __forceinline__ void advance(const DkvGeo& t) {
    if (++r == t.per_head) { r = 0; ++hh; }
  }
  __device__ __forceinline__ void get(const BwdParams& p, const DkvGeo& t, int& head, int& s, int64_t& q0) const {
    head = t.kvh * (p.g.Hq / p.g.Hkv) + hh;
    s = r < t.nt0 ? 0 : 1;
    q0 = (s == 0 ? t.t00 + r : t.t01 + (r - t.nt0)) * KBN;
  }
};

// Query-row interval [lo, hi) of stream s that sees key j of key stream ks
// (empty if the key is not in this call's key set or j >= L), within the
// call's row range when ROWS.
template <bool ROWS>
__device__ __forceinline__ void key_rows(const Geom& g, const RowRange& rows, int ks, int64_t j, int s, int64_t& lo,
                                         int64_t& hi) {
  lo = 0;
  hi = 0;
  if (j >= g.L) return;
  const int64_t b = j / g.B;
  if (ks == 0) {
    if (j < g.kv_begin || j >= g.kv_end) return;
    lo = s == 0 ? b * g.B : (b + 1) * g.B;
    hi = g.L;
  } else {
    if (!g.include_local || s == 0) return;
    lo = b * g.B;
    hi = (b + 1) * g.B;
  }
  if (ROWS) {  // only this call's rows
    lo = imax64(lo, range_lo(rows, s));
    hi = imin64(hi, range_hi(rows, s));
    if (hi <= lo) lo = hi = 0;
  }
}

// P = exp2(s sl2 - LSE log2 e) for 32 query rows (columns of S^T) of one key
// row: scores us, their rows' LSE in lse[0..32), key offsets c0 + [0, 32)
// outside [lo, hi) give 0 unless FULL.  fp32 P into pf, packed bf16 into pk.
// The masked variant is a separate instantiation so that the common, fully
// visible case is one straight-line block the compiler can schedule.
template <bool FULL>
__device__ __forceinline__ void p_cols32(const uint32_t (&us)[32], const float* lse, uint64_t sl2x2,
                                         uint64_t nlog2e, int c0, int lo, int hi, float (&pf)[32],
                                         uint32_t (&pk)[16]) {
#pragma unroll
  for (int c4 = 0; c4 < 8; ++c4) {
    const float4 l4 = *reinterpret_cast<const float4*>(lse + 4 * c4);
    const uint64_t nlA = f2_mul(f2(l4.x, l4.y), nlog2e), nlB = f2_mul(f2(l4.z, l4.w), nlog2e);
    float x0, x1, x2, x3;
    f2_split(f2_fma(f2(__uint_as_float(us[4 * c4]), __uint_as_float(us[4 * c4 + 1])), sl2x2, nlA), x0, x1);
    f2_split(f2_fma(f2(__uint_as_float(us[4 * c4 + 2]), __uint_as_float(us[4 * c4 + 3])), sl2x2, nlB), x2, x3);
    float pe[4] = {ex2_approx(x0), ex2_approx(x1), ex2_approx(x2), ex2_approx(x3)};
    if (!FULL) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = c0 + 4 * c4 + e;
        pe[e] = (c >= lo && c < hi) ? pe[e] : 0.f;
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) pf[4 * c4 + e] = pe[e];
    pk[2 * c4] = pack_bf16x2(pe[0], pe[1]);
    pk[2 * c4 + 1] = pack_bf16x2(pe[2], pe[3]);
  }
}

template <int HD, bool VL, bool ROWS>
__global__ void __launch_bounds__(kThreads, 1)
    bdlm_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tQc, const __grid_constant__ CUtensorMap tQn,
                           const __grid_constant__ CUtensorMap tdOc, const __grid_constant__ CUtensorMap tdOn,
                           const __grid_constant__ CUtensorMap tKc, const __grid_constant__ CUtensorMap tKn,
                           const __grid_constant__ CUtensorMap tVc, const __grid_constant__ CUtensorMap tVn,
                           const BwdParams p, const VarlenTabs vt, const int64_t n_items, uint32_t* status,
                           const uint64_t limit_ns) {
  using LY = DkvLayout<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  const uint32_t sK = base + LY::kK, sV = base + LY::kV, sQ = base + LY::kQ, sdO = base + LY::kdO,
                 sStat = base + LY::kStat;
  const float* stat_ptr = reinterpret_cast<const float*>(base_ptr + LY::kStat);
  const uint32_t bars = base + LY::kBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + LY::kBar + 8 * KV_NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + LY::kBar + 8 * KV_NBAR + 4);
  auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  const ItemRing ring{BAR(KV_IF), BAR(KV_IE),
                      reinterpret_cast<volatile int64_t*>(base_ptr + LY::kBar + 8 * KV_NBAR + 8)};
  // each ring slot also carries its item's geometry, computed once by the producer
  DkvGeo* geo_slot = reinterpret_cast<DkvGeo*>(base_ptr + LY::kGeo);
  const Role R = role();

  if (threadIdx.x == 0) {
    mbar_init(BAR(KV_KF), 1);
    mbar_init(BAR(KV_KE), 1);
    for (int s = 0; s < QNS; ++s) {
      mbar_init(BAR(KV_QF + s), 1 + 32);  // expect_tx arrival + one cp.async arrival per producer lane
      mbar_init(BAR(KV_QE + s), 1);
    }
    mbar_init(BAR(KV_SF), 1);
    mbar_init(BAR(KV_DPF), 1);
    mbar_init(BAR(KV_PF), kEwThreads);
    mbar_init(BAR(KV_DSF), kEwThreads);
    mbar_init(BAR(KV_ACCDONE), 1);
    mbar_init(BAR(KV_ACCE), kEwThreads);
    for (int s = 0; s < kRingSlots; ++s) {
      mbar_init(BAR(KV_IF + s), 1);
      mbar_init(BAR(KV_IE + s), 1 + kEwThreads);  // the MMA thread and every elementwise thread
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (R.warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Watchdog wd{status, limit_ns, abort_flag};
  const int grid = gridDim.x, cta = blockIdx.x;
  constexpr uint32_t kColDK = 0, kColDV = 128, kColS = 256, kColDP = 384;

  if (R.warp == 0) {
    // ---------------------------------------------------------- producer (whole warp)
    uint32_t itn = 0, qc = 0;
    bool ok = true;
    for (int64_t rnd = 0; ok; ++rnd) {
      // lane 0 claims and publishes the item; the warp takes it from lane 0
      int64_t idx = 0;
      if (R.lane == 0) {
        idx = claim_item(p.g, status + kSchedWordDkv, rnd, cta, grid);
        ok = ring_acquire(ring, rnd, wd, 93);
        if (ok) {
          if (idx < n_items) geo_slot[rnd & (kRingSlots - 1)] = dkv_geo<VL, ROWS>(p, vt, idx);
          ring_publish(ring, rnd, idx);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      if (!ok) break;
      if (idx >= n_items) break;
      // (lane 0 wrote the slot; the slot is not reused before this warp
      // acquires it again, kRingSlots rounds on)
      __syncwarp();
      const DkvGeo t = geo_slot[rnd & (kRingSlots - 1)];
      if (t.n == 0) continue;
      if (itn > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(BAR(KV_KE), (itn - 1) & 1, wd, 41));
        if (!ok) break;
      }
      if (R.lane == 0) {
        mbar_arrive_expect_tx(BAR(KV_KF), 2 * LY::kTile);
        const CUtensorMap* mk = t.ks ? &tKn : &tKc;
        const CUtensorMap* mv = t.ks ? &tVn : &tVc;
#pragma unroll
        for (int pn = 0; pn < HD / 64; ++pn) {
          // (a row-restricted call's K / V hold only its keys: local index)
          const int kj = (int)((VL ? t.off : 0) + (ROWS ? local_key(p.rows, t.ks, t.j0) : t.j0));
          tma_load_3d(sK + pn * LY::kPanel, mk, BAR(KV_KF), pn * 64, t.kvh, kj);
          tma_load_3d(sV + pn * LY::kPanel, mv, BAR(KV_KF), pn * 64, t.kvh, kj);
        }
      }
      DkvCursor cur;
      cur.reset();
      for (int k = 0; k < t.n; ++k, ++qc, cur.advance(t)) {
        const int st = qc & 1;
        if (qc >= QNS) {
          ok = __all_sync(0xffffffffu, mbar_wait(BAR(KV_QE + st), ((qc >> 1) - 1) & 1, wd, 42));
          if (!ok) break;
        }
        int head, s;
        int64_t q0;
        cur.get(p, t, head, s, q0);
        if (R.lane == 0) {
          mbar_arrive_expect_tx(BAR(KV_QF + st), 2 * LY::kTile);
          const CUtensorMap* mq = s ? &tQn : &tQc;
          const CUtensorMap* mo = s ? &tdOn : &tdOc;
#pragma unroll
          for (int pn = 0; pn < HD / 64; ++pn) {
            tma_load_3d(sQ + st * LY::kTile + pn * LY::kPanel, mq, BAR(KV_QF + st), pn * 64, head,
                        (int)((VL ? t.off : 0) + (ROWS ? local_row(p.rows, s, q0) : q0)));
            tma_load_3d(sdO + st * LY::kTile + pn * LY::kPanel, mo, BAR(KV_QF + st), pn * 64, head,
                        (int)((VL ? t.off : 0) + (ROWS ? local_row(p.rows, s, q0) : q0)));
          }
        }
        // LSE and D of the tile's 128 rows, asynchronously (rows >= L, and rows
        // a row-restricted call's statistics do not hold, read as 0)
        const int64_t lstride = ROWS ? held_rows(p.rows, s) : p.g.L;
        const float* LSE = (s ? p.LSEn : p.LSEc) + (int64_t)head * lstride + (VL ? t.off : 0);
        const float* Dr = (s ? p.Dn : p.Dc) + (int64_t)head * lstride + (VL ? t.off : 0);
        const uint32_t stat = sStat + st * 2 * KBN * 4;
#pragma unroll
        for (int c = R.lane; c < KBN; c += 32) {
          const int64_t r = q0 + c;
          const int64_t lr = ROWS ? local_row(p.rows, s, r) : r;
          const bool v = ROWS ? (r < p.g.L && lr >= 0 && lr < lstride) : r < (VL ? t.L : p.g.L);
          cp_async4(stat + c * 4, LSE + (v ? lr : 0), v);
          cp_async4(stat + (KBN + c) * 4, Dr + (v ? lr : 0), v);
        }
        cp_async_mbar_arrive(BAR(KV_QF + st));
      }
      if (!ok) break;
      ++itn;
    }
  } else if (R.warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (R.lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(KBM, KBN, false, false);
      constexpr uint32_t kIdA = idesc_bf16(KBM, HD, false, true);
      const uint64_t dK0 = sdesc_sw128(sK, 16, 1024), dV0 = sdesc_sw128(sV, 16, 1024);
      uint32_t itn = 0, qc = 0;
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        int64_t idx;
        if (!ring_wait(ring, rnd, idx, wd, 94)) { ok = false; break; }
        if (idx >= n_items) break;
        const DkvGeo t = geo_slot[rnd & (kRingSlots - 1)];
        ring_release(ring, rnd);
        if (t.n == 0) continue;
        if (!mbar_wait(BAR(KV_KF), itn & 1, wd, 43)) { ok = false; break; }
        const uint32_t q_base = qc;
        // dK += dS^T(kk) Q(kk): A = dS^T packed over the dP^T columns
        auto do_dk = [&](int kk) -> bool {
          const uint32_t qq = q_base + kk;
          const int st = qq & 1;
          if (!mbar_wait(BAR(KV_DSF), qq & 1, wd, 44)) return false;
          tc_fence_after();
          const uint64_t bq0 = sdesc_sw128(sQ + st * LY::kTile, LY::kPanel, 1024);
#pragma unroll
          for (int k4 = 0; k4 < KBN / 16; ++k4)
            tc_mma_ts(tmem + kColDK, tmem + kColDP + packed_col128(k4), desc_add(bq0, k4 * 2048), kIdA,
                      (kk > 0 || k4 > 0) ? 1u : 0u);
          // Q and dO of this stage are no longer read: dV(kk) was issued earlier
          tc_commit(BAR(KV_QE + st));
          return true;
        };
        for (int k = 0; k < t.n && ok; ++k, ++qc) {
          const int st = qc & 1;
          if (!mbar_wait(BAR(KV_QF + st), (qc >> 1) & 1, wd, 46)) { ok = false; break; }
          tc_fence_after();
          // S^T(k) over P^T(k-1): dV(k-1), its reader, was issued before this point
          const uint64_t dq0 = sdesc_sw128(sQ + st * LY::kTile, 16, 1024);
          const uint64_t do0 = sdesc_sw128(sdO + st * LY::kTile, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * LY::kPanel + (kk & 3) * 32;
            tc_mma_ss(tmem + kColS, desc_add(dK0, off), desc_add(dq0, off), kIdS, kk > 0 ? 1u : 0u);
          }
          tc_commit(BAR(KV_SF));
          if (k >= 1 && !do_dk(k - 1)) { ok = false; break; }
          // dP^T(k) over dS^T(k-1): dK(k-1), its reader, was just issued
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * LY::kPanel + (kk & 3) * 32;
            tc_mma_ss(tmem + kColDP, desc_add(dV0, off), desc_add(do0, off), kIdS, kk > 0 ? 1u : 0u);
          }
          tc_commit(BAR(KV_DPF));
          // dV += P^T(k) dO(k)
          if (!mbar_wait(BAR(KV_PF), qc & 1, wd, 47)) { ok = false; break; }
          if (k == 0 && itn > 0 && !mbar_wait(BAR(KV_ACCE), (itn - 1) & 1, wd, 45)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bo0 = sdesc_sw128(sdO + st * LY::kTile, LY::kPanel, 1024);
#pragma unroll
          for (int k4 = 0; k4 < KBN / 16; ++k4)
            tc_mma_ts(tmem + kColDV, tmem + kColS + packed_col128(k4), desc_add(bo0, k4 * 2048), kIdA,
                      (k > 0 || k4 > 0) ? 1u : 0u);
        }
        if (!ok) break;
        if (!do_dk(t.n - 1)) { ok = false; break; }
        tc_commit(BAR(KV_ACCDONE));
        tc_commit(BAR(KV_KE));
        ++itn;
      }
    }
  } else {
    // ---------------------------------------------------------- elementwise (thread = key row)
    // warpgroup `half` = query rows [64 half, 64 half + 64) of a step
    const int row = R.row, half = R.half;
    uint32_t itn = 0, qc = 0;
    bool ok = true;
    const uint64_t sl2x2 = f2(p.scale_log2, p.scale_log2), nlog2e = f2(-kLog2e, -kLog2e);
    for (int64_t rnd = 0; ok; ++rnd) {
      int64_t idx;
      if (!ring_wait(ring, rnd, idx, wd, 95)) { ok = false; break; }
      if (idx >= n_items) break;
      const DkvGeo t = geo_slot[rnd & (kRingSlots - 1)];
      ring_release(ring, rnd);
      if (t.n == 0) continue;
      const int64_t j = t.j0 + row;
      // query-row bounds as 32-bit values (rows are TMA coordinates, < 2^31):
      // rows of each stream this key sees, and rows every key of the tile sees
      int kl[2], kh[2], al[2], ah[2];
      {
        const Geom gm = VL ? seq_geom(p.g, t.L) : p.g;
        const int64_t jl = imin64(t.j0 + KBM, gm.L) - 1;
        bool all_in = t.j0 + KBM <= gm.L;
        if (t.ks == 0) all_in = all_in && t.j0 >= gm.kv_begin && t.j0 + KBM <= gm.kv_end;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          int64_t lo, hi, a0, b0, a1, b1;
          key_rows<ROWS>(gm, p.rows, t.ks, j, s, lo, hi);
          key_rows<ROWS>(gm, p.rows, t.ks, t.j0, s, a0, b0);
          key_rows<ROWS>(gm, p.rows, t.ks, jl, s, a1, b1);
          kl[s] = (int)lo;
          kh[s] = (int)hi;
          al[s] = (int)imax64(a0, a1);
          ah[s] = all_in ? (int)imin64(b0, b1) : al[s];
        }
      }
      DkvCursor cur;
      cur.reset();
      for (int k = 0; k < t.n; ++k, ++qc, cur.advance(t)) {
        int head, s;
        int64_t q0;
        cur.get(p, t, head, s, q0);
        (void)head;
        const int st = qc & 1;
        ok = mbar_wait(BAR(KV_SF), qc & 1, wd, 48);
        if (ok) ok = mbar_wait(BAR(KV_QF + st), (qc >> 1) & 1, wd, 49);  // LSE/D landed
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float* stl = stat_ptr + st * 2 * KBN + half * 64;  // LSE of this half's 64 rows; D at +KBN
        const int q0i = (int)q0;
        const int a_lo = s ? al[1] : al[0], a_hi = s ? ah[1] : ah[0];
        const int k_lo = s ? kl[1] : kl[0], k_hi = s ? kh[1] : kh[0];
        const bool full = q0i >= a_lo && q0i + KBN <= a_hi;
        const int base_row = q0i + half * 64;
        const int lo = full ? -1 : max(min(k_lo - base_row, 65), -1);
        const int hi = full ? 65 : max(min(k_hi - base_row, 65), -1);
        // P = exp(scale S - LSE) on this half's 64 query rows, kept in fp32
        float pf[2][32];
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          uint32_t us[32];
          tmem_ld32(tmem + R.tl + kColS + half * 64 + sub * 32, us);
          uint32_t pk[16];
          if (full) p_cols32<true>(us, stl + sub * 32, sl2x2, nlog2e, sub * 32, lo, hi, pf[sub], pk);
          else p_cols32<false>(us, stl + sub * 32, sl2x2, nlog2e, sub * 32, lo, hi, pf[sub], pk);
          // P^T (bf16) over S^T columns this warpgroup has already read
          tmem_st16(tmem + R.tl + kColS + half * 64 + sub * 16, pk);
        }
        tc_fence_before();
        mbar_arrive(BAR(KV_PF));
        // dS = P o (dP - D)
        ok = __all_sync(0xffffffffu, mbar_wait(BAR(KV_DPF), qc & 1, wd, 50));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          uint32_t ud[32];
          tmem_ld32(tmem + R.tl + kColDP + half * 64 + sub * 32, ud);
          uint32_t dk[16];
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 d4 = *reinterpret_cast<const float4*>(stl + KBN + sub * 32 + 4 * c4);
            const uint64_t tA = f2_sub(f2(__uint_as_float(ud[4 * c4]), __uint_as_float(ud[4 * c4 + 1])), f2(d4.x, d4.y));
            const uint64_t tB =
                f2_sub(f2(__uint_as_float(ud[4 * c4 + 2]), __uint_as_float(ud[4 * c4 + 3])), f2(d4.z, d4.w));
            float s0, s1, s2, s3;
            f2_split(f2_mul(f2(pf[sub][4 * c4], pf[sub][4 * c4 + 1]), tA), s0, s1);
            f2_split(f2_mul(f2(pf[sub][4 * c4 + 2], pf[sub][4 * c4 + 3]), tB), s2, s3);
            dk[2 * c4] = pack_bf16x2(s0, s1);
            dk[2 * c4 + 1] = pack_bf16x2(s2, s3);
          }
          // dS^T (bf16) over dP^T columns this warpgroup has already read
          tmem_st16(tmem + R.tl + kColDP + half * 64 + sub * 16, dk);
        }
        tc_fence_before();
        mbar_arrive(BAR(KV_DSF));
      }
      if (!ok) break;
      ok = mbar_wait(BAR(KV_ACCDONE), itn & 1, wd, 51);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // the key set of this call: clean keys in [kv_begin, kv_end), corrupted keys all
      // (and, in a row-restricted call, the keys its dK / dV hold)
      const bool wr = VL ? j < t.L
                         : j < p.g.L && (t.ks == 1 || (j >= p.g.kv_begin && j < p.g.kv_end)) &&
                               (!ROWS || key_held(p.rows, t.ks, j));
      void* dKo = t.ks ? p.dKn : p.dKc;
      void* dVo = t.ks ? p.dVn : p.dVc;
      const int64_t oofs =
          (((VL ? t.off : 0) + (ROWS ? local_key(p.rows, t.ks, j) : j)) * p.g.Hkv + t.kvh) * HD + half * (HD / 2);
#pragma unroll
      for (int c4 = 0; c4 < HD / 64; ++c4) {
        uint32_t uk[32], uv[32];
        tmem_ld32x2(tmem + R.tl + kColDK + half * (HD / 2) + c4 * 32,
                    tmem + R.tl + kColDV + half * (HD / 2) + c4 * 32, uk, uv);
        if (wr) {
          store_row32(dKo, oofs + c4 * 32, uk, p.scale, p.g_f32, ROWS ? p.dkv_accumulate : 0);
          store_row32(dVo, oofs + c4 * 32, uv, 1.f, p.g_f32, ROWS ? p.dkv_accumulate : 0);
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(KV_ACCE));
      ++itn;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) sched_release(status + kSchedWordDkv, grid);
  if (*abort_flag) drain_after_abort(200);
  if (R.warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int HD, bool VL, bool ROWS = false>
cudaError_t launch_dkv_t(const BwdMaps& m, const BwdParams& p, const VarlenTabs& vt, int64_t n, int grid,
                         uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  auto k = bdlm_bwd_dkv_tc_kernel<HD, VL, ROWS>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, DkvLayout<HD>::kAlloc);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, DkvLayout<HD>::kAlloc, stream>>>(m.Qc, m.Qn, m.dOc, m.dOn, m.Kc, m.Kn, m.Vc, m.Vn, p, vt, n,
                                                        status, limit_ns);
  return cudaSuccess;
}

cudaError_t launch_bwd_dkv_tc(const BwdMaps& m, const BwdParams& p, const VarlenTabs* vt, int num_sms,
                              uint32_t* status, uint64_t limit_ns, cudaStream_t stream, int* launches) {
  const int64_t n = vt ? vt->n_kv : kv_items(p.g, KBM);
  if (n == 0) return cudaSuccess;
  const int grid = (int)(n < num_sms ? n : num_sms);
  const VarlenTabs none{nullptr, nullptr, nullptr, 0, 0};
  const VarlenTabs& t = vt ? *vt : none;
  // a row range, or accumulation across calls: the rows instantiation (one sequence)
  const bool rows = p.rows_call != 0;
  if (rows && vt) return cudaErrorInvalidValue;
  cudaError_t e;
  if (rows)
    e = p.d == 128 ? launch_dkv_t<128, false, true>(m, p, t, n, grid, status, limit_ns, stream)
                   : launch_dkv_t<64, false, true>(m, p, t, n, grid, status, limit_ns, stream);
  else
    e = p.d == 128 ? (vt ? launch_dkv_t<128, true>(m, p, t, n, grid, status, limit_ns, stream)
                         : launch_dkv_t<128, false>(m, p, t, n, grid, status, limit_ns, stream))
                   : (vt ? launch_dkv_t<64, true>(m, p, t, n, grid, status, limit_ns, stream)
                         : launch_dkv_t<64, false>(m, p, t, n, grid, status, limit_ns, stream));
  if (e != cudaSuccess) return e;
  if (launches) ++*launches;
  return cudaGetLastError();
}

}  // namespace bdlm
