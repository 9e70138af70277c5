// bwd_dq.cu -- dQ pass of the two-stream BDLM attention backward (sm_103a).
//
// dQ = scale dS K with dS = P o (dP - D), P = exp(scale Q K^T - LSE),
// dP = dO V^T, over each query row's visible keys (see bwd_common.cuh for
// the gradient definitions and their source).
//
// Item = (128-row query tile, head, stream) in the forward's longest-first
// order.  Q and dO of the item stay in shared memory; 128-key K tiles stream
// through a 3-stage TMA ring (a K tile is read by S(j) and by dQ(j), one
// step later) and V tiles through a 2-stage ring.  Per step j (128 keys),
// MMA warp:
//   S(j)  = Q K^T   into S buffer j & 1      (TMEM, 128 columns)
//   dP(j) = dO V^T  into the dP buffer       (TMEM, 128 columns), issued once
//                   the elementwise warps have read dP(j-1)
//   dQ   += dS(j-1) K(j-1)                   (dS as packed bf16 in TMEM over
//                   S buffer (j-1) & 1, K read as an MN-major operand)
// The elementwise warps (thread = query row, 64 keys per warpgroup) form dS
// and write it back over the S columns they have just read.  The S MMA that
// next reuses a buffer is issued after the dQ MMA reading its dS (the tensor
// pipe runs in issue order).  Every output row is written once.
#include "bwd_common.cuh"
#include "sched.cuh"

namespace bdlm {
namespace {

using namespace bwd;

constexpr int QBM = 128;  // query rows per item
constexpr int QBN = 128;  // keys per step
constexpr int KNS = 3;    // K stages
constexpr int VNS = 2;    // V stages

enum { DQ_QF = 0, DQ_QE = 1, DQ_KF = 2, DQ_KE = 5, DQ_VF = 8, DQ_VE = 10, DQ_DPF = 12, DQ_DPFREE = 13,
       DQ_DSF = 14, DQ_DONE = 16, DQ_OE = 17, DQ_IF = 18, DQ_IE = 18 + kRingSlots, DQ_NBAR = 18 + 2 * kRingSlots };
// The 256 bytes after the tiles: barriers, the TMEM address, the abort flag,
// the work-item ring's slots.
static_assert(8 * DQ_NBAR + 8 + 8 * kRingSlots <= 256, "barrier area overflows");

template <int HD>
struct DqLayout {
  static constexpr int kTile = 128 * HD * 2;  // 128 rows x HD bf16 (Q, dO, K, V tiles alike)
  static constexpr int kPanel = 128 * 128;    // 128 rows x 64 bf16
  static constexpr int kQ = 0;
  static constexpr int kdO = kQ + kTile;
  static constexpr int kK = kdO + kTile;
  static constexpr int kV = kK + KNS * kTile;
  static constexpr int kBar = kV + VNS * kTile;
  static constexpr int kGeo = kBar + 256;  // the work-item ring's geometry slots
  static constexpr int kBytes = kGeo + 512;
  static constexpr int kAlloc = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
};

struct DqGeo {
  int stream, head, kvh;
  int64_t r0;
  QTileRanges q;
  int nc, n;
  int rot;         // the clean-key sweep starts at clean tile c0 + rot
  int64_t off, L;  // first row of the item's sequence in the packed tensors, its length
};
static_assert(kRingSlots * sizeof(DqGeo) <= 512, "geometry slots overflow");

// VL: packed variable-length batch (a separate instantiation).
template <bool VL, bool ROWS>
__device__ __forceinline__ DqGeo dq_geo(const BwdParams& p, const VarlenTabs& vt, int64_t idx) {
  DqGeo t;
  Geom g = p.g;
  int64_t qtile;
  t.off = 0;
  if (VL) {  // packed batch: the item and its sequence from the tables
    const int4 e = vt.q_items[idx];
    t.stream = e.y & 1;
    t.head = e.y >> 1;
    qtile = e.z;
    t.off = vt.seq_off[e.x];
    g = seq_geom(p.g, vt.seq_off[e.x + 1] - t.off);
  } else {
    const QItem it = ROWS ? q_item_rows(p.g, p.rows, QBM, idx) : q_item(p.g, QBM, idx);
    t.stream = it.stream;
    t.head = it.head;
    qtile = it.qtile;
  }
  t.L = g.L;
  t.kvh = t.head / (p.g.Hq / p.g.Hkv);
  t.r0 = qtile * QBM;
  const int64_t r1 = imin64(t.r0 + QBM, g.L);
  t.q = qtile_ranges(g, t.stream, t.r0, r1, QBN);
  t.nc = (int)(t.q.c1 - t.q.c0);
  t.n = t.nc + (int)(t.q.n1 - t.q.n0);
  if (ROWS && !tile_in(p.rows, t.stream, t.r0, r1)) t.nc = t.n = 0;  // none of the call's rows (not listed)
  t.rot = sweep_rotation(idx, t.nc);
  return t;
}

// First key of step j: clean tiles from c0 + rot round to c0 + rot - 1, then
// the corrupted tiles (dQ sums over keys in any order).
__device__ __forceinline__ int dq_key0(const DqGeo& t, int j) {
  int c = j + t.rot;
  if (c >= t.nc) c -= t.nc;
  return (int)((j < t.nc ? t.q.c0 + c : t.q.n0 + (j - t.nc)) * QBN);
}

template <int HD, bool VL, bool ROWS>
__global__ void __launch_bounds__(kThreads, 1)
    bdlm_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tQc, const __grid_constant__ CUtensorMap tQn,
                          const __grid_constant__ CUtensorMap tdOc, const __grid_constant__ CUtensorMap tdOn,
                          const __grid_constant__ CUtensorMap tKc, const __grid_constant__ CUtensorMap tKn,
                          const __grid_constant__ CUtensorMap tVc, const __grid_constant__ CUtensorMap tVn,
                          const BwdParams p, const VarlenTabs vt, const int64_t n_items, uint32_t* status,
                          const uint64_t limit_ns) {
  using LY = DqLayout<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  const uint32_t sQ = base + LY::kQ, sdO = base + LY::kdO, sK = base + LY::kK, sV = base + LY::kV;
  const uint32_t bars = base + LY::kBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + LY::kBar + 8 * DQ_NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + LY::kBar + 8 * DQ_NBAR + 4);
  auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  const ItemRing ring{BAR(DQ_IF), BAR(DQ_IE),
                      reinterpret_cast<volatile int64_t*>(base_ptr + LY::kBar + 8 * DQ_NBAR + 8)};
  // each ring slot also carries its item's geometry, computed once by the producer
  DqGeo* geo_slot = reinterpret_cast<DqGeo*>(base_ptr + LY::kGeo);
  const Role R = role();

  if (threadIdx.x == 0) {
    mbar_init(BAR(DQ_QF), 1);
    mbar_init(BAR(DQ_QE), 1);
    for (int s = 0; s < KNS; ++s) {
      mbar_init(BAR(DQ_KF + s), 1);
      mbar_init(BAR(DQ_KE + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(BAR(DQ_VF + s), 1);
      mbar_init(BAR(DQ_VE + s), 1);
      mbar_init(BAR(DQ_DSF + s), kEwThreads);
    }
    mbar_init(BAR(DQ_DPF), 1);
    mbar_init(BAR(DQ_DPFREE), kEwThreads);
    mbar_init(BAR(DQ_DONE), 1);
    mbar_init(BAR(DQ_OE), kEwThreads);
    for (int s = 0; s < kRingSlots; ++s) {
      mbar_init(BAR(DQ_IF + s), 1);
      mbar_init(BAR(DQ_IE + s), 1 + kEwThreads);  // the MMA thread and every elementwise thread
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
  // TMEM columns: S buffers at 0 and 128 (dS over them), dP at 256, dQ at 384
  constexpr uint32_t kColDP = 256, kColDQ = 384;

  if (R.warp == 0) {
    // ------------------------------------------------------------ producer
    if (R.lane == 0) {
      uint32_t itn = 0, g = 0;  // items with work, global step count
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        const int64_t idx = claim_item(p.g, status + kSchedWordDq, rnd, cta, grid);
        if (!ring_acquire(ring, rnd, wd, 96)) { ok = false; break; }
        DqGeo t;
        if (idx < n_items) {
          t = dq_geo<VL, ROWS>(p, vt, idx);
          geo_slot[rnd & (kRingSlots - 1)] = t;
        }
        ring_publish(ring, rnd, idx);
        if (idx >= n_items) break;
        if (t.n == 0) continue;
        if (itn > 0 && !mbar_wait(BAR(DQ_QE), (itn - 1) & 1, wd, 21)) { ok = false; break; }
        mbar_arrive_expect_tx(BAR(DQ_QF), 2 * LY::kTile);
        const CUtensorMap* mq = t.stream ? &tQn : &tQc;
        const CUtensorMap* mo = t.stream ? &tdOn : &tdOc;
#pragma unroll
        for (int pn = 0; pn < HD / 64; ++pn) {
          tma_load_3d(sQ + pn * LY::kPanel, mq, BAR(DQ_QF), pn * 64, t.head, (int)((VL ? t.off : 0) + (ROWS ? local_row(p.rows, t.stream, t.r0) : t.r0)));
          tma_load_3d(sdO + pn * LY::kPanel, mo, BAR(DQ_QF), pn * 64, t.head, (int)((VL ? t.off : 0) + (ROWS ? local_row(p.rows, t.stream, t.r0) : t.r0)));
        }
        ++itn;
        for (int j = 0; j < t.n; ++j, ++g) {
          const bool cs = j < t.nc;
          // packed-tensor row, or the key's index in a row-restricted call's K / V
          const int key0 =
              (int)((VL ? t.off : 0) + (ROWS ? local_key(p.rows, cs ? 0 : 1, dq_key0(t, j)) : dq_key0(t, j)));
          const int ks = g % KNS, vs = g & 1;
          if (g >= KNS && !mbar_wait(BAR(DQ_KE + ks), ((g / KNS) - 1) & 1, wd, 22)) { ok = false; break; }
          mbar_arrive_expect_tx(BAR(DQ_KF + ks), LY::kTile);
#pragma unroll
          for (int pn = 0; pn < HD / 64; ++pn)
            tma_load_3d(sK + ks * LY::kTile + pn * LY::kPanel, cs ? &tKc : &tKn, BAR(DQ_KF + ks), pn * 64, t.kvh,
                        key0);
          if (g >= VNS && !mbar_wait(BAR(DQ_VE + vs), ((g >> 1) - 1) & 1, wd, 23)) { ok = false; break; }
          mbar_arrive_expect_tx(BAR(DQ_VF + vs), LY::kTile);
#pragma unroll
          for (int pn = 0; pn < HD / 64; ++pn)
            tma_load_3d(sV + vs * LY::kTile + pn * LY::kPanel, cs ? &tVc : &tVn, BAR(DQ_VF + vs), pn * 64, t.kvh,
                        key0);
        }
      }
    }
  } else if (R.warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (R.lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(QBM, QBN, false, false);
      constexpr uint32_t kIdQ = idesc_bf16(QBM, HD, false, true);
      const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024), do0 = sdesc_sw128(sdO, 16, 1024);
      uint32_t itn = 0, g = 0;
      uint32_t ks = 0, kph = 0;  // K stage of step g and its phase parity
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        int64_t idx;
        if (!ring_wait(ring, rnd, idx, wd, 97)) { ok = false; break; }
        if (idx >= n_items) break;
        const DqGeo t = geo_slot[rnd & (kRingSlots - 1)];
        ring_release(ring, rnd);
        if (t.n == 0) continue;
        if (!mbar_wait(BAR(DQ_QF), itn & 1, wd, 24)) { ok = false; break; }
        // stage of the previous step (read by its dQ MMA)
        uint32_t pks = 0;
        // dQ += dS(g-1) K(g-1), dS packed over S buffer (g-1) & 1
        auto do_dq = [&](uint32_t gg, uint32_t kst, bool first) -> bool {
          const uint32_t b = gg & 1;
          if (!mbar_wait(BAR(DQ_DSF + b), (gg >> 1) & 1, wd, 25)) return false;
          if (first && itn > 0 && !mbar_wait(BAR(DQ_OE), (itn - 1) & 1, wd, 26)) return false;
          tc_fence_after();
          const uint64_t bk0 = sdesc_sw128(sK + kst * LY::kTile, LY::kPanel, 1024);
          const uint32_t a0 = tmem + b * 128;
#pragma unroll
          for (int kk = 0; kk < QBN / 16; ++kk)
            tc_mma_ts(tmem + kColDQ, a0 + packed_col128(kk), desc_add(bk0, kk * 2048), kIdQ,
                      (kk > 0 || !first) ? 1u : 0u);
          tc_commit(BAR(DQ_KE + kst));
          return true;
        };
        for (int j = 0; j < t.n && ok; ++j, ++g) {
          const uint32_t b = g & 1, vs = g & 1;
          // S(j) into buffer b: the dS last held there (step g-2) was read by
          // the dQ MMA issued one iteration earlier
          if (!mbar_wait(BAR(DQ_KF + ks), kph, wd, 27)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dk0 = sdesc_sw128(sK + ks * LY::kTile, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * LY::kPanel + (kk & 3) * 32;
            tc_mma_ss(tmem + b * 128, desc_add(dq0, off), desc_add(dk0, off), kIdS, kk > 0 ? 1u : 0u);
          }
          // dP(j) once the elementwise warps have read dP(j-1); its commit
          // also tells them that S(j) is complete
          if (g >= 1 && !mbar_wait(BAR(DQ_DPFREE), (g - 1) & 1, wd, 28)) { ok = false; break; }
          if (!mbar_wait(BAR(DQ_VF + vs), (g >> 1) & 1, wd, 29)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dv0 = sdesc_sw128(sV + vs * LY::kTile, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * LY::kPanel + (kk & 3) * 32;
            tc_mma_ss(tmem + kColDP, desc_add(do0, off), desc_add(dv0, off), kIdS, kk > 0 ? 1u : 0u);
          }
          tc_commit(BAR(DQ_DPF));
          tc_commit(BAR(DQ_VE + vs));
          if (j == t.n - 1) tc_commit(BAR(DQ_QE));
          if (j >= 1 && !do_dq(g - 1, pks, j == 1)) { ok = false; break; }
          pks = ks;
          if (++ks == KNS) { ks = 0; kph ^= 1; }
        }
        if (!ok) break;
        if (!do_dq(g - 1, pks, t.n == 1)) { ok = false; break; }
        tc_commit(BAR(DQ_DONE));
        ++itn;
      }
    }
  } else {
    // ------------------------------------------------------------ elementwise
    // thread = query row; warpgroup `half` = keys [64 half, 64 half + 64) of a
    // step, taken in two 32-key sub-steps
    const int row = R.row, half = R.half;
    uint32_t itn = 0, g = 0;
    bool ok = true;
    for (int64_t rnd = 0; ok; ++rnd) {
      int64_t idx;
      if (!ring_wait(ring, rnd, idx, wd, 98)) { ok = false; break; }
      if (idx >= n_items) break;
      const DqGeo t = geo_slot[rnd & (kRingSlots - 1)];
      ring_release(ring, rnd);
      // (one sequence: its length and offset come from the parameters)
      const int64_t seqL = VL ? t.L : p.g.L, seq0 = VL ? t.off : 0;
      const int64_t r = t.r0 + row;  // row within the item's sequence
      const bool valid = r < seqL && (!ROWS || row_in(p.rows, t.stream, r));
      void* dqbase = t.stream ? p.dQn : p.dQc;
      // the row's index in its stream's tensors (packed row in a batch, local
      // row in a row-restricted call) and the [H, rows] statistics' stride
      const int64_t lrow = VL ? seq0 + r : (ROWS ? local_row(p.rows, t.stream, r) : r);
      const int64_t lstride = ROWS ? held_rows(p.rows, t.stream) : p.g.L;
      const int64_t oofs = (lrow * p.g.Hq + t.head) * HD + half * (HD / 2);
      if (t.n == 0) {
        // no visible key for the whole tile: dQ rows are zero
        if (valid && !p.dq_accumulate) {
          if (p.g_f32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(dqbase) + oofs);
#pragma unroll
            for (int c = 0; c < HD / 8; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dqbase) + oofs);
#pragma unroll
            for (int c = 0; c < HD / 16; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
      const int64_t rr = r < seqL ? r : seqL - 1;
      const Geom gm = VL ? seq_geom(p.g, t.L) : p.g;
      int64_t clo, chi, nlo, nhi;
      clean_interval(gm, t.stream, rr, clo, chi);
      noisy_interval(gm, t.stream, rr, nlo, nhi);
      const int64_t srow = (int64_t)t.head * lstride + lrow;  // [H, rows] statistics
      const float nlse2 = valid ? -(t.stream ? p.LSEn : p.LSEc)[srow] * kLog2e : 0.f;
      const float Dv = valid ? (t.stream ? p.Dn : p.Dc)[srow] : 0.f;
      const uint64_t sl2x2 = f2(p.scale_log2, p.scale_log2), nl2 = f2(nlse2, nlse2), nD2 = f2(-Dv, -Dv);
      for (int j = 0; j < t.n; ++j, ++g) {
        const bool cs = j < t.nc;
        const int64_t key0 = dq_key0(t, j);
        const bool full = cs ? tile_full(key0, QBN, t.q.c_all_lo, t.q.c_all_hi, seqL)
                             : tile_full(key0, QBN, t.q.n_all_lo, t.q.n_all_hi, seqL);
        const int b = g & 1;
        // dP(j) complete (its commit follows S(j)'s MMAs)
        ok = mbar_wait(BAR(DQ_DPF), g & 1, wd, 31);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const uint32_t col = half * 64 + s * 32;
          uint32_t us[32], ud[32];
          tmem_ld32x2(tmem + R.tl + b * 128 + col, tmem + R.tl + kColDP + col, us, ud);
          if (s == 1) {
            // both dP halves of this warpgroup read: the next dP may land
            tc_fence_before();
            mbar_arrive(BAR(DQ_DPFREE));
          }
          uint32_t pk[16];
          int lo = -1, hi = 33;
          if (!full) {
            const int64_t k0 = key0 + col;
            lo = (int)imax64(imin64((cs ? clo : nlo) - k0, 33), -1);
            hi = (int)imax64(imin64((cs ? chi : nhi) - k0, 33), -1);
          }
          if (full) ds_row32<true>(us, ud, sl2x2, nl2, nD2, lo, hi, pk);
          else ds_row32<false>(us, ud, sl2x2, nl2, nD2, lo, hi, pk);
          // 32 keys of dS as 16 packed columns over S columns this warpgroup
          // has already read (layout of packed_col128)
          tmem_st16(tmem + R.tl + b * 128 + half * 64 + s * 16, pk);
        }
        tc_fence_before();
        mbar_arrive(BAR(DQ_DSF + b));
      }
      if (!ok) break;
      ok = mbar_wait(BAR(DQ_DONE), itn & 1, wd, 32);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c4 = 0; c4 < HD / 64; ++c4) {
        uint32_t u[32];
        tmem_ld32(tmem + R.tl + kColDQ + half * (HD / 2) + c4 * 32, u);
        if (valid) store_row32(dqbase, oofs + c4 * 32, u, p.scale, p.g_f32, p.dq_accumulate);
      }
      tc_fence_before();
      mbar_arrive(BAR(DQ_OE));
      ++itn;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) sched_release(status + kSchedWordDq, grid);
  if (*abort_flag) drain_after_abort(200);
  if (R.warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int HD, bool VL, bool ROWS = false>
cudaError_t launch_dq_t(const BwdMaps& m, const BwdParams& p, const VarlenTabs& vt, int64_t n, int grid,
                        uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  auto k = bdlm_bwd_dq_tc_kernel<HD, VL, ROWS>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, DqLayout<HD>::kAlloc);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, DqLayout<HD>::kAlloc, stream>>>(m.Qc, m.Qn, m.dOc, m.dOn, m.Kc, m.Kn, m.Vc, m.Vn, p, vt, n,
                                                       status, limit_ns);
  return cudaSuccess;
}

cudaError_t launch_bwd_dq_tc(const BwdMaps& m, const BwdParams& p, const VarlenTabs* vt, int num_sms,
                             uint32_t* status, uint64_t limit_ns, cudaStream_t stream, int* launches) {
  // a row-restricted call lists only the query tiles that hold its rows (one sequence)
  const bool rows = p.rows_call != 0;
  if (rows && vt) return cudaErrorInvalidValue;
  const int64_t n = vt ? vt->n_q : rows ? q_items_rows(p.g, p.rows, QBM) : q_items(p.g, QBM);
  if (n == 0) return cudaSuccess;
  const int grid = (int)(n < num_sms ? n : num_sms);
  const VarlenTabs none{nullptr, nullptr, nullptr, 0, 0};
  const VarlenTabs& t = vt ? *vt : none;
  cudaError_t e;
  if (rows)
    e = p.d == 128 ? launch_dq_t<128, false, true>(m, p, t, n, grid, status, limit_ns, stream)
                   : launch_dq_t<64, false, true>(m, p, t, n, grid, status, limit_ns, stream);
  else
    e = p.d == 128 ? (vt ? launch_dq_t<128, true>(m, p, t, n, grid, status, limit_ns, stream)
                         : launch_dq_t<128, false>(m, p, t, n, grid, status, limit_ns, stream))
                   : (vt ? launch_dq_t<64, true>(m, p, t, n, grid, status, limit_ns, stream)
                         : launch_dq_t<64, false>(m, p, t, n, grid, status, limit_ns, stream));
  if (e != cudaSuccess) return e;
  if (launches) ++*launches;
  return cudaGetLastError();
}

}  // namespace bdlm
