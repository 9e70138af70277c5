// bwd_tc.cu -- two-stream BDLM attention backward on the sm_103a tensor cores.
//
// Gradients of softmax attention under the two-stream block mask, no gradient
// through LSE ("Block Parallelism For Efficient Distributed Long-Context
// Diffusion Language Model Training": training gradients, evolve.pub review
// "Key claims" / Proposition 1; only clean K/V gradients cross context shards,
// evolve.pub FAQ on CSBP):
//   P = exp(scale Q K^T - LSE), dP = dO V^T, dS = P o (dP - D),
//   dV = sum_group P^T dO, dK = scale sum_group dS^T Q, dQ = scale dS K.
// Two deterministic passes; every output element is written once:
//
// dQ pass (bdlm_bwd_dq_tc): persistent, one item per (128-row query tile,
//   head, stream) in the forward's longest-first order.  Q and dO stay in
//   shared memory; 64-key K/V tiles stream through a 3-stage TMA ring.
//   MMA warp: S = Q K^T and dP = dO V^T into one of two TMEM buffer pairs,
//   then dQ += dS K (K read as an MN-major operand from the same tile).
//   Elementwise warpgroup (thread = query row): P = exp2(S c - LSE2),
//   dS = P (dP - D) -> bf16 swizzled shared tile (double-buffered).
//
// dK/dV pass (bdlm_bwd_dkv_tc): persistent, one item per (key stream, KV
//   head, 128-key tile): clean tiles first (they are read by every later
//   row), then corrupted tiles.  K and V stay in shared memory; 64-row Q/dO
//   tiles of every query head of the GQA group and both streams that can see
//   the keys stream through a 2-stage ring (with their LSE and D slices).
//   MMA warp: S^T = K Q^T, dP^T = V dO^T, then dV += P^T dO and
//   dK += dS^T Q with Q/dO read as MN-major operands.  Elementwise warpgroup
//   (thread = key row) forms P^T and dS^T.  dK and dV accumulate in TMEM
//   across the whole group and are written once.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;

// ====================================================================== dQ
constexpr int QBM = 128;  // query rows per item
constexpr int QBN = 64;   // keys per step
constexpr int QNS = 3;    // K/V stages

enum { DQ_QFULL = 0, DQ_QEMPTY = 1, DQ_KVFULL = 2, DQ_KVEMPTY = 5, DQ_SFULL = 8, DQ_SEMPTY = 10, DQ_DSFULL = 12,
       DQ_DSEMPTY = 14, DQ_DONE = 16, DQ_OEMPTY = 17, DQ_NBAR = 18 };

template <int HD>
struct DqLayout {
  static constexpr int kQTile = QBM * HD * 2;    // 128 rows
  static constexpr int kKTile = QBN * HD * 2;    // 64 rows
  static constexpr int kQPanel = QBM * 128;      // 16 KB
  static constexpr int kKPanel = QBN * 128;      // 8 KB
  static constexpr int kDsTile = QBM * QBN * 2;  // 16 KB
  static constexpr int kQ = 0;
  static constexpr int kdO = kQ + kQTile;
  static constexpr int kK = kdO + kQTile;
  static constexpr int kV = kK + QNS * kKTile;
  static constexpr int kDs = kV + QNS * kKTile;
  static constexpr int kBar = kDs + 2 * kDsTile;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
};

struct DqGeo {
  int stream, head, kvh;
  int64_t r0;
  QTileRanges q;
  int nc, n;
};

__device__ __forceinline__ DqGeo dq_geo(const BwdParams& p, int64_t idx) {
  DqGeo t;
  const QItem it = q_item(p.g, QBM, idx);
  t.stream = it.stream;
  t.head = it.head;
  t.kvh = it.head / (p.g.Hq / p.g.Hkv);
  t.r0 = it.qtile * QBM;
  const int64_t r1 = imin64(t.r0 + QBM, p.g.L);
  t.q = qtile_ranges(p.g, t.stream, t.r0, r1, QBN);
  t.nc = (int)(t.q.c1 - t.q.c0);
  t.n = t.nc + (int)(t.q.n1 - t.q.n0);
  return t;
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    bdlm_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tQc, const __grid_constant__ CUtensorMap tQn,
                          const __grid_constant__ CUtensorMap tdOc, const __grid_constant__ CUtensorMap tdOn,
                          const __grid_constant__ CUtensorMap tKc, const __grid_constant__ CUtensorMap tKn,
                          const __grid_constant__ CUtensorMap tVc, const __grid_constant__ CUtensorMap tVn,
                          const BwdParams p, const int64_t n_items, uint32_t* status, const uint64_t limit_ns) {
  using LY = DqLayout<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  const uint32_t sQ = base + LY::kQ, sdO = base + LY::kdO, sK = base + LY::kK, sV = base + LY::kV,
                 sDs = base + LY::kDs;
  const uint32_t bars = base + LY::kBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + LY::kBar + 8 * DQ_NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + LY::kBar + 8 * DQ_NBAR + 4);
  auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(BAR(DQ_QFULL), 1);
    mbar_init(BAR(DQ_QEMPTY), 1);
    for (int s = 0; s < QNS; ++s) {
      mbar_init(BAR(DQ_KVFULL + s), 1);
      mbar_init(BAR(DQ_KVEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(BAR(DQ_SFULL + s), 1);
      mbar_init(BAR(DQ_SEMPTY + s), 128);
      mbar_init(BAR(DQ_DSFULL + s), 128);
      mbar_init(BAR(DQ_DSEMPTY + s), 1);
    }
    mbar_init(BAR(DQ_DONE), 1);
    mbar_init(BAR(DQ_OEMPTY), 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Watchdog wd{status, limit_ns, abort_flag};
  const int grid = gridDim.x, cta = blockIdx.x;
  // TMEM columns: S[2] at 0/64, dP[2] at 128/192, dQ at 256
  if (warp == 0) {
    if (lane == 0) {
      uint32_t itn = 0, kvc = 0;
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        const int64_t idx = snake_item(rnd, cta, grid);
        if (idx >= n_items) break;
        const DqGeo t = dq_geo(p, idx);
        if (t.n == 0) continue;
        if (itn > 0 && !mbar_wait(BAR(DQ_QEMPTY), (itn - 1) & 1, wd, 21)) { ok = false; break; }
        mbar_arrive_expect_tx(BAR(DQ_QFULL), 2 * LY::kQTile);
        const CUtensorMap* mq = t.stream ? &tQn : &tQc;
        const CUtensorMap* mo = t.stream ? &tdOn : &tdOc;
#pragma unroll
        for (int pn = 0; pn < HD / 64; ++pn) {
          tma_load_3d(sQ + pn * LY::kQPanel, mq, BAR(DQ_QFULL), pn * 64, t.head, (int)t.r0);
          tma_load_3d(sdO + pn * LY::kQPanel, mo, BAR(DQ_QFULL), pn * 64, t.head, (int)t.r0);
        }
        for (int j = 0; j < t.n; ++j, ++kvc) {
          const int st = kvc % QNS;
          if (kvc >= QNS && !mbar_wait(BAR(DQ_KVEMPTY + st), ((kvc / QNS) - 1) & 1, wd, 22)) { ok = false; break; }
          const bool cs = j < t.nc;
          const int key0 = (int)((cs ? t.q.c0 + j : t.q.n0 + (j - t.nc)) * QBN);
          const CUtensorMap* mk = cs ? &tKc : &tKn;
          const CUtensorMap* mv = cs ? &tVc : &tVn;
          mbar_arrive_expect_tx(BAR(DQ_KVFULL + st), 2 * LY::kKTile);
#pragma unroll
          for (int pn = 0; pn < HD / 64; ++pn) {
            tma_load_3d(sK + st * LY::kKTile + pn * LY::kKPanel, mk, BAR(DQ_KVFULL + st), pn * 64, t.kvh, key0);
            tma_load_3d(sV + st * LY::kKTile + pn * LY::kKPanel, mv, BAR(DQ_KVFULL + st), pn * 64, t.kvh, key0);
          }
        }
        ++itn;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(QBM, QBN, false, false);
      constexpr uint32_t kIdQ = idesc_bf16(QBM, HD, false, true);
      uint32_t itn = 0, kvc = 0, sc = 0, dc = 0;
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        const int64_t idx = snake_item(rnd, cta, grid);
        if (idx >= n_items) break;
        const DqGeo t = dq_geo(p, idx);
        if (t.n == 0) continue;
        if (!mbar_wait(BAR(DQ_QFULL), itn & 1, wd, 23)) { ok = false; break; }
        const uint32_t kv_base = kvc;
        auto do_dq = [&](int jj) -> bool {
          const uint32_t kv = kv_base + jj;
          const int st = kv % QNS;
          const int db = dc & 1;
          if (!mbar_wait(BAR(DQ_DSFULL + db), (dc >> 1) & 1, wd, 24)) return false;
          if (jj == 0 && itn > 0 && !mbar_wait(BAR(DQ_OEMPTY), (itn - 1) & 1, wd, 25)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < QBN / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(sDs + db * LY::kDsTile + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sK + st * LY::kKTile + kk * 2048, LY::kKPanel, 1024);
            tc_mma_ss(tmem + 256, ad, bd, kIdQ, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(BAR(DQ_KVEMPTY + st));
          tc_commit(BAR(DQ_DSEMPTY + db));
          ++dc;
          return true;
        };
        for (int j = 0; j < t.n && ok; ++j, ++kvc, ++sc) {
          const int st = kvc % QNS;
          const int sb = sc & 1;
          if (!mbar_wait(BAR(DQ_KVFULL + st), (kvc / QNS) & 1, wd, 26)) { ok = false; break; }
          if (sc >= 2 && !mbar_wait(BAR(DQ_SEMPTY + sb), ((sc >> 1) - 1) & 1, wd, 27)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t qo = (kk >> 2) * LY::kQPanel + (kk & 3) * 32;
            const uint32_t ko = st * LY::kKTile + (kk >> 2) * LY::kKPanel + (kk & 3) * 32;
            tc_mma_ss(tmem + sb * QBN, sdesc_sw128(sQ + qo, 16, 1024), sdesc_sw128(sK + ko, 16, 1024), kIdS,
                      kk > 0 ? 1u : 0u);
            tc_mma_ss(tmem + 128 + sb * QBN, sdesc_sw128(sdO + qo, 16, 1024), sdesc_sw128(sV + ko, 16, 1024),
                      kIdS, kk > 0 ? 1u : 0u);
          }
          tc_commit(BAR(DQ_SFULL + sb));
          if (j == t.n - 1) tc_commit(BAR(DQ_QEMPTY));
          if (j >= 1 && !do_dq(j - 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!do_dq(t.n - 1)) { ok = false; break; }
        tc_commit(BAR(DQ_DONE));
        ++itn;
      }
    }
  } else {
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t tl = (uint32_t)(quarter * 32) << 16;
    uint32_t itn = 0, sc = 0, dc = 0;
    bool ok = true;
    for (int64_t rnd = 0; ok; ++rnd) {
      const int64_t idx = snake_item(rnd, cta, grid);
      if (idx >= n_items) break;
      const DqGeo t = dq_geo(p, idx);
      const int64_t r = t.r0 + row;
      const bool valid = r < p.g.L;
      void* dqbase = t.stream ? p.dQn : p.dQc;
      const int64_t oofs = (r * p.g.Hq + t.head) * HD;
      if (t.n == 0) {
        if (valid && !p.dq_accumulate) {
          if (p.g_f32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(dqbase) + oofs);
#pragma unroll
            for (int c = 0; c < HD / 4; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dqbase) + oofs);
#pragma unroll
            for (int c = 0; c < HD / 8; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
      const int64_t rr = valid ? r : p.g.L - 1;
      int64_t clo, chi, nlo, nhi;
      clean_interval(p.g, t.stream, rr, clo, chi);
      noisy_interval(p.g, t.stream, rr, nlo, nhi);
      const float lse2 = valid ? (t.stream ? p.LSEn : p.LSEc)[(int64_t)t.head * p.g.L + r] * kLog2e : 0.f;
      const float Dv = valid ? (t.stream ? p.Dn : p.Dc)[(int64_t)t.head * p.g.L + r] : 0.f;
      for (int j = 0; j < t.n; ++j, ++sc) {
        const bool cs = j < t.nc;
        const int64_t key0 = (cs ? t.q.c0 + j : t.q.n0 + (j - t.nc)) * QBN;
        const bool full = cs ? tile_full(key0, QBN, t.q.c_all_lo, t.q.c_all_hi, p.g.L)
                             : tile_full(key0, QBN, t.q.n_all_lo, t.q.n_all_hi, p.g.L);
        const int sb = sc & 1;
        ok = mbar_wait(BAR(DQ_SFULL + sb), (sc >> 1) & 1, wd, 28);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float s[QBN], dp[QBN];
#pragma unroll
        for (int c4 = 0; c4 < QBN / 32; ++c4) {
          uint32_t u[32];
          tmem_ld32(tmem + tl + sb * QBN + c4 * 32, u);
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c4 * 32 + c] = __uint_as_float(u[c]);
          tmem_ld32(tmem + tl + 128 + sb * QBN + c4 * 32, u);
#pragma unroll
          for (int c = 0; c < 32; ++c) dp[c4 * 32 + c] = __uint_as_float(u[c]);
        }
        tc_fence_before();
        mbar_arrive(BAR(DQ_SEMPTY + sb));
        const int64_t lo = (cs ? clo : nlo) - key0, hi = (cs ? chi : nhi) - key0;
        uint32_t pk[QBN / 2];
#pragma unroll
        for (int c = 0; c < QBN; c += 2) {
          float d0 = 0.f, d1 = 0.f;
          if (full || (c >= lo && c < hi)) d0 = ex2_approx(fmaf(s[c], p.scale_log2, -lse2)) * (dp[c] - Dv);
          if (full || (c + 1 >= lo && c + 1 < hi))
            d1 = ex2_approx(fmaf(s[c + 1], p.scale_log2, -lse2)) * (dp[c + 1] - Dv);
          pk[c / 2] = pack_bf16x2(d0, d1);
        }
        const int db = dc & 1;
        if (dc >= 2) {
          ok = mbar_wait(BAR(DQ_DSEMPTY + db), ((dc >> 1) - 1) & 1, wd, 29);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
#pragma unroll
        for (int ch = 0; ch < QBN / 8; ++ch) {
          const uint32_t addr = sDs + db * LY::kDsTile + row * 128 + ((ch ^ (row & 7)) << 4);
          st_shared_v4(addr, pk[ch * 4 + 0], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(BAR(DQ_DSFULL + db));
        ++dc;
      }
      if (!ok) break;
      ok = mbar_wait(BAR(DQ_DONE), itn & 1, wd, 30);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c4 = 0; c4 < HD / 32; ++c4) {
        uint32_t u[32];
        tmem_ld32(tmem + tl + 256 + c4 * 32, u);
        if (valid) {
          if (p.g_f32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(dqbase) + oofs + c4 * 32);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              float4 v = make_float4(__uint_as_float(u[4 * c]) * p.scale, __uint_as_float(u[4 * c + 1]) * p.scale,
                                     __uint_as_float(u[4 * c + 2]) * p.scale,
                                     __uint_as_float(u[4 * c + 3]) * p.scale);
              if (p.dq_accumulate) {
                const float4 old = o[c];
                v.x += old.x; v.y += old.y; v.z += old.z; v.w += old.w;
              }
              o[c] = v;
            }
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dqbase) + oofs + c4 * 32);
            const float sc2 = p.scale;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              o[c] = make_uint4(pack_bf16x2(__uint_as_float(u[8 * c + 0]) * sc2, __uint_as_float(u[8 * c + 1]) * sc2),
                                pack_bf16x2(__uint_as_float(u[8 * c + 2]) * sc2, __uint_as_float(u[8 * c + 3]) * sc2),
                                pack_bf16x2(__uint_as_float(u[8 * c + 4]) * sc2, __uint_as_float(u[8 * c + 5]) * sc2),
                                pack_bf16x2(__uint_as_float(u[8 * c + 6]) * sc2, __uint_as_float(u[8 * c + 7]) * sc2));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(DQ_OEMPTY));
      ++itn;
    }
  }
  __syncthreads();
  if (*abort_flag) drain_after_abort(200);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// =================================================================== dK / dV
constexpr int KBM = 128;  // keys per item
constexpr int KBN = 64;   // query rows per step
constexpr int KNS = 2;    // Q/dO stages

enum { KV_KFULL = 0, KV_KEMPTY = 1, KV_QFULL = 2, KV_QEMPTY = 4, KV_SFULL = 6, KV_SEMPTY = 8, KV_PFULL = 10,
       KV_PEMPTY = 12, KV_ACCDONE = 14, KV_ACCEMPTY = 15, KV_NBAR = 16 };

template <int HD>
struct DkvLayout {
  static constexpr int kKTile = KBM * HD * 2;    // 128 key rows
  static constexpr int kQTile = KBN * HD * 2;    // 64 query rows
  static constexpr int kKPanel = KBM * 128;      // 16 KB
  static constexpr int kQPanel = KBN * 128;      // 8 KB
  static constexpr int kPTile = KBM * KBN * 2;   // 16 KB
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKTile;
  static constexpr int kQ = kV + kKTile;
  static constexpr int kdO = kQ + KNS * kQTile;
  static constexpr int kPt = kdO + KNS * kQTile;
  static constexpr int kdSt = kPt + 2 * kPTile;
  static constexpr int kStat = kdSt + 2 * kPTile;  // LSE2 and D per stage: KNS x 2 x 64 floats
  static constexpr int kBar = kStat + KNS * 2 * KBN * 4;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
};

struct DkvGeo {
  int ks, kvh;
  int64_t j0;
  int64_t rlo[2], rhi[2];  // query rows of each stream that can see some key of the tile
  int64_t t0[2];           // first query tile index of each stream
  int nt[2];               // query tiles of each stream
  int per_head, n;         // steps per head, total steps
};

__device__ __forceinline__ DkvGeo dkv_geo(const BwdParams& p, int64_t idx) {
  DkvGeo t;
  const KVItem it = kv_item(p.g, KBM, idx);
  t.ks = it.key_stream;
  t.kvh = it.kv_head;
  t.j0 = it.ktile * KBM;
  const int64_t j1 = imin64(t.j0 + KBM, p.g.L);
  kv_tile_rows(p.g, t.ks, t.j0, j1, t.rlo[0], t.rhi[0], t.rlo[1], t.rhi[1]);
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    if (t.rhi[s] > t.rlo[s]) {
      t.t0[s] = t.rlo[s] / KBN;
      t.nt[s] = (int)(cdiv64(t.rhi[s], KBN) - t.t0[s]);
    } else {
      t.t0[s] = 0;
      t.nt[s] = 0;
    }
  }
  t.per_head = t.nt[0] + t.nt[1];
  t.n = t.per_head * (p.g.Hq / p.g.Hkv);
  return t;
}

// step k of an item -> (query head, stream, first query row)
__device__ __forceinline__ void dkv_step(const BwdParams& p, const DkvGeo& t, int k, int& head, int& s,
                                         int64_t& q0) {
  const int G = p.g.Hq / p.g.Hkv;
  (void)G;
  const int hh = k / t.per_head;
  const int r = k % t.per_head;
  head = t.kvh * (p.g.Hq / p.g.Hkv) + hh;
  s = r < t.nt[0] ? 0 : 1;
  q0 = (s == 0 ? t.t0[0] + r : t.t0[1] + (r - t.nt[0])) * KBN;
}

// Query-row interval [lo, hi) of stream s that sees key j of key stream ks
// (empty if the key is not in this call's key set or j >= L).
__device__ __forceinline__ void key_rows(const Geom& g, int ks, int64_t j, int s, int64_t& lo, int64_t& hi) {
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
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    bdlm_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tQc, const __grid_constant__ CUtensorMap tQn,
                           const __grid_constant__ CUtensorMap tdOc, const __grid_constant__ CUtensorMap tdOn,
                           const __grid_constant__ CUtensorMap tKc, const __grid_constant__ CUtensorMap tKn,
                           const __grid_constant__ CUtensorMap tVc, const __grid_constant__ CUtensorMap tVn,
                           const BwdParams p, const int64_t n_items, uint32_t* status, const uint64_t limit_ns) {
  using LY = DkvLayout<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  const uint32_t sK = base + LY::kK, sV = base + LY::kV, sQ = base + LY::kQ, sdO = base + LY::kdO,
                 sPt = base + LY::kPt, sdSt = base + LY::kdSt;
  float* sStat = reinterpret_cast<float*>(base_ptr + LY::kStat);  // [stage][lse2 | D][64]
  const uint32_t bars = base + LY::kBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + LY::kBar + 8 * KV_NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + LY::kBar + 8 * KV_NBAR + 4);
  auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(BAR(KV_KFULL), 1);
    mbar_init(BAR(KV_KEMPTY), 1);
    for (int s = 0; s < KNS; ++s) {
      mbar_init(BAR(KV_QFULL + s), 1 + 32);  // expect_tx arrival + the warp's LSE/D stores
      mbar_init(BAR(KV_QEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(BAR(KV_SFULL + s), 1);
      mbar_init(BAR(KV_SEMPTY + s), 128);
      mbar_init(BAR(KV_PFULL + s), 128);
      mbar_init(BAR(KV_PEMPTY + s), 1);
    }
    mbar_init(BAR(KV_ACCDONE), 1);
    mbar_init(BAR(KV_ACCEMPTY), 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Watchdog wd{status, limit_ns, abort_flag};
  const int grid = gridDim.x, cta = blockIdx.x;
  // TMEM columns: dK at 0, dV at 128, S^T[2] at 256/320, dP^T[2] at 384/448
  if (warp == 0) {
    // ---------------------------------------------------------- producer (whole warp)
    uint32_t itn = 0, qc = 0;
    bool ok = true;
    for (int64_t rnd = 0; ok; ++rnd) {
      const int64_t idx = snake_item(rnd, cta, grid);
      if (idx >= n_items) break;
      const DkvGeo t = dkv_geo(p, idx);
      if (t.n == 0) continue;
      if (itn > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(BAR(KV_KEMPTY), (itn - 1) & 1, wd, 41));
        if (!ok) break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(BAR(KV_KFULL), 2 * LY::kKTile);
        const CUtensorMap* mk = t.ks ? &tKn : &tKc;
        const CUtensorMap* mv = t.ks ? &tVn : &tVc;
#pragma unroll
        for (int pn = 0; pn < HD / 64; ++pn) {
          tma_load_3d(sK + pn * LY::kKPanel, mk, BAR(KV_KFULL), pn * 64, t.kvh, (int)t.j0);
          tma_load_3d(sV + pn * LY::kKPanel, mv, BAR(KV_KFULL), pn * 64, t.kvh, (int)t.j0);
        }
      }
      for (int k = 0; k < t.n; ++k, ++qc) {
        const int st = qc % KNS;
        if (qc >= KNS) {
          ok = __all_sync(0xffffffffu, mbar_wait(BAR(KV_QEMPTY + st), ((qc / KNS) - 1) & 1, wd, 42));
          if (!ok) break;
        }
        int head, s;
        int64_t q0;
        dkv_step(p, t, k, head, s, q0);
        if (lane == 0) {
          mbar_arrive_expect_tx(BAR(KV_QFULL + st), 2 * LY::kQTile);
          const CUtensorMap* mq = s ? &tQn : &tQc;
          const CUtensorMap* mo = s ? &tdOn : &tdOc;
#pragma unroll
          for (int pn = 0; pn < HD / 64; ++pn) {
            tma_load_3d(sQ + st * LY::kQTile + pn * LY::kQPanel, mq, BAR(KV_QFULL + st), pn * 64, head, (int)q0);
            tma_load_3d(sdO + st * LY::kQTile + pn * LY::kQPanel, mo, BAR(KV_QFULL + st), pn * 64, head, (int)q0);
          }
        }
        const float* LSE = (s ? p.LSEn : p.LSEc) + (int64_t)head * p.g.L;
        const float* Dr = (s ? p.Dn : p.Dc) + (int64_t)head * p.g.L;
        float* stat = sStat + st * 2 * KBN;
#pragma unroll
        for (int c = lane; c < KBN; c += 32) {
          const int64_t r = q0 + c;
          const bool v = r < p.g.L;
          stat[c] = v ? LSE[r] * kLog2e : 0.f;
          stat[KBN + c] = v ? Dr[r] : 0.f;
        }
        mbar_arrive(BAR(KV_QFULL + st));
      }
      if (!ok) break;
      ++itn;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(KBM, KBN, false, false);
      constexpr uint32_t kIdA = idesc_bf16(KBM, HD, false, true);
      uint32_t itn = 0, qc = 0, sc = 0, pc = 0;
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        const int64_t idx = snake_item(rnd, cta, grid);
        if (idx >= n_items) break;
        const DkvGeo t = dkv_geo(p, idx);
        if (t.n == 0) continue;
        if (!mbar_wait(BAR(KV_KFULL), itn & 1, wd, 43)) { ok = false; break; }
        const uint32_t q_base = qc;
        auto do_acc = [&](int kk) -> bool {
          const uint32_t qq = q_base + kk;
          const int st = qq % KNS;
          const int pb = pc & 1;
          if (!mbar_wait(BAR(KV_PFULL + pb), (pc >> 1) & 1, wd, 44)) return false;
          if (kk == 0 && itn > 0 && !mbar_wait(BAR(KV_ACCEMPTY), (itn - 1) & 1, wd, 45)) return false;
          tc_fence_after();
#pragma unroll
          for (int k4 = 0; k4 < KBN / 16; ++k4) {
            const uint32_t acc = (kk > 0 || k4 > 0) ? 1u : 0u;
            const uint64_t bo = sdesc_sw128(sdO + st * LY::kQTile + k4 * 2048, LY::kQPanel, 1024);
            const uint64_t bq = sdesc_sw128(sQ + st * LY::kQTile + k4 * 2048, LY::kQPanel, 1024);
            tc_mma_ss(tmem + 128, sdesc_sw128(sPt + pb * LY::kPTile + k4 * 32, 16, 1024), bo, kIdA, acc);
            tc_mma_ss(tmem + 0, sdesc_sw128(sdSt + pb * LY::kPTile + k4 * 32, 16, 1024), bq, kIdA, acc);
          }
          tc_commit(BAR(KV_QEMPTY + st));
          tc_commit(BAR(KV_PEMPTY + pb));
          ++pc;
          return true;
        };
        for (int k = 0; k < t.n && ok; ++k, ++qc, ++sc) {
          const int st = qc % KNS;
          const int sb = sc & 1;
          if (!mbar_wait(BAR(KV_QFULL + st), (qc / KNS) & 1, wd, 46)) { ok = false; break; }
          if (sc >= 2 && !mbar_wait(BAR(KV_SEMPTY + sb), ((sc >> 1) - 1) & 1, wd, 47)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t ko = (kk >> 2) * LY::kKPanel + (kk & 3) * 32;
            const uint32_t qo = st * LY::kQTile + (kk >> 2) * LY::kQPanel + (kk & 3) * 32;
            tc_mma_ss(tmem + 256 + sb * KBN, sdesc_sw128(sK + ko, 16, 1024), sdesc_sw128(sQ + qo, 16, 1024), kIdS,
                      kk > 0 ? 1u : 0u);
            tc_mma_ss(tmem + 384 + sb * KBN, sdesc_sw128(sV + ko, 16, 1024), sdesc_sw128(sdO + qo, 16, 1024),
                      kIdS, kk > 0 ? 1u : 0u);
          }
          tc_commit(BAR(KV_SFULL + sb));
          if (k >= 1 && !do_acc(k - 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!do_acc(t.n - 1)) { ok = false; break; }
        tc_commit(BAR(KV_ACCDONE));
        tc_commit(BAR(KV_KEMPTY));
        ++itn;
      }
    }
  } else {
    // ---------------------------------------------------------- elementwise (thread = key row)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t tl = (uint32_t)(quarter * 32) << 16;
    uint32_t itn = 0, qc = 0, sc = 0, pc = 0;
    bool ok = true;
    for (int64_t rnd = 0; ok; ++rnd) {
      const int64_t idx = snake_item(rnd, cta, grid);
      if (idx >= n_items) break;
      const DkvGeo t = dkv_geo(p, idx);
      if (t.n == 0) continue;
      const int64_t j = t.j0 + row;
      int64_t klo[2], khi[2];
      key_rows(p.g, t.ks, j, 0, klo[0], khi[0]);
      key_rows(p.g, t.ks, j, 1, klo[1], khi[1]);
      // rows every key of the tile sees (for the full-tile test)
      int64_t alo[2], ahi[2];
      {
        const int64_t jl = imin64(t.j0 + KBM, p.g.L) - 1;
        bool all_in = t.j0 + KBM <= p.g.L;
        if (t.ks == 0) all_in = all_in && t.j0 >= p.g.kv_begin && t.j0 + KBM <= p.g.kv_end;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          int64_t a0, b0, a1, b1;
          key_rows(p.g, t.ks, t.j0, s, a0, b0);
          key_rows(p.g, t.ks, jl, s, a1, b1);
          alo[s] = imax64(a0, a1);
          ahi[s] = all_in ? imin64(b0, b1) : alo[s];
        }
      }
      for (int k = 0; k < t.n; ++k, ++qc, ++sc) {
        int head, s;
        int64_t q0;
        dkv_step(p, t, k, head, s, q0);
        const int st = qc % KNS;
        const int sb = sc & 1;
        ok = mbar_wait(BAR(KV_SFULL + sb), (sc >> 1) & 1, wd, 48);
        if (ok) ok = mbar_wait(BAR(KV_QFULL + st), (qc / KNS) & 1, wd, 49);  // LSE/D visibility
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float sv[KBN], dpv[KBN];
#pragma unroll
        for (int c4 = 0; c4 < KBN / 32; ++c4) {
          uint32_t u[32];
          tmem_ld32(tmem + tl + 256 + sb * KBN + c4 * 32, u);
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[c4 * 32 + c] = __uint_as_float(u[c]);
          tmem_ld32(tmem + tl + 384 + sb * KBN + c4 * 32, u);
#pragma unroll
          for (int c = 0; c < 32; ++c) dpv[c4 * 32 + c] = __uint_as_float(u[c]);
        }
        tc_fence_before();
        mbar_arrive(BAR(KV_SEMPTY + sb));
        const float* stat = sStat + st * 2 * KBN;
        const bool full = q0 >= alo[s] && q0 + KBN <= ahi[s];
        const int64_t lo = klo[s] - q0, hi = khi[s] - q0;
        uint32_t pp[KBN / 2], dd[KBN / 2];
#pragma unroll
        for (int c = 0; c < KBN; c += 2) {
          float p0 = 0.f, p1 = 0.f;
          if (full || (c >= lo && c < hi)) p0 = ex2_approx(fmaf(sv[c], p.scale_log2, -stat[c]));
          if (full || (c + 1 >= lo && c + 1 < hi)) p1 = ex2_approx(fmaf(sv[c + 1], p.scale_log2, -stat[c + 1]));
          pp[c / 2] = pack_bf16x2(p0, p1);
          dd[c / 2] = pack_bf16x2(p0 * (dpv[c] - stat[KBN + c]), p1 * (dpv[c + 1] - stat[KBN + c + 1]));
        }
        const int pb = pc & 1;
        if (pc >= 2) {
          ok = mbar_wait(BAR(KV_PEMPTY + pb), ((pc >> 1) - 1) & 1, wd, 50);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
#pragma unroll
        for (int ch = 0; ch < KBN / 8; ++ch) {
          const uint32_t off = row * 128 + ((ch ^ (row & 7)) << 4);
          st_shared_v4(sPt + pb * LY::kPTile + off, pp[ch * 4 + 0], pp[ch * 4 + 1], pp[ch * 4 + 2], pp[ch * 4 + 3]);
          st_shared_v4(sdSt + pb * LY::kPTile + off, dd[ch * 4 + 0], dd[ch * 4 + 1], dd[ch * 4 + 2], dd[ch * 4 + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(BAR(KV_PFULL + pb));
        ++pc;
      }
      if (!ok) break;
      ok = mbar_wait(BAR(KV_ACCDONE), itn & 1, wd, 51);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // the key set of this call: clean keys in [kv_begin, kv_end), corrupted keys all
      const bool wr = j < p.g.L && (t.ks == 1 || (j >= p.g.kv_begin && j < p.g.kv_end));
      void* dKo = t.ks ? p.dKn : p.dKc;
      void* dVo = t.ks ? p.dVn : p.dVc;
      const int64_t oofs = (j * p.g.Hkv + t.kvh) * HD;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        void* obase = which == 0 ? dKo : dVo;
        const float mul = which == 0 ? p.scale : 1.f;
#pragma unroll
        for (int c4 = 0; c4 < HD / 32; ++c4) {
          uint32_t u[32];
          tmem_ld32(tmem + tl + which * 128 + c4 * 32, u);
          if (wr) {
            if (p.g_f32) {
              float4* o = reinterpret_cast<float4*>(static_cast<float*>(obase) + oofs + c4 * 32);
#pragma unroll
              for (int c = 0; c < 8; ++c)
                o[c] = make_float4(__uint_as_float(u[4 * c]) * mul, __uint_as_float(u[4 * c + 1]) * mul,
                                   __uint_as_float(u[4 * c + 2]) * mul, __uint_as_float(u[4 * c + 3]) * mul);
            } else {
              uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(obase) + oofs + c4 * 32);
#pragma unroll
              for (int c = 0; c < 4; ++c)
                o[c] = make_uint4(pack_bf16x2(__uint_as_float(u[8 * c + 0]) * mul, __uint_as_float(u[8 * c + 1]) * mul),
                                  pack_bf16x2(__uint_as_float(u[8 * c + 2]) * mul, __uint_as_float(u[8 * c + 3]) * mul),
                                  pack_bf16x2(__uint_as_float(u[8 * c + 4]) * mul, __uint_as_float(u[8 * c + 5]) * mul),
                                  pack_bf16x2(__uint_as_float(u[8 * c + 6]) * mul, __uint_as_float(u[8 * c + 7]) * mul));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(KV_ACCEMPTY));
      ++itn;
    }
  }
  __syncthreads();
  if (*abort_flag) drain_after_abort(200);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_bwd_dq_tc(const BwdMaps& m, const BwdParams& p, int num_sms, uint32_t* status,
                             uint64_t limit_ns, cudaStream_t stream, int* launches) {
  const int64_t n = q_items(p.g, QBM);
  if (n == 0) return cudaSuccess;
  const int grid = (int)(n < num_sms ? n : num_sms);
  cudaError_t e;
  if (p.d == 128) {
    e = cudaFuncSetAttribute(bdlm_bwd_dq_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DqLayout<128>::kAlloc);
    if (e != cudaSuccess) return e;
    bdlm_bwd_dq_tc_kernel<128><<<grid, kThreads, DqLayout<128>::kAlloc, stream>>>(
        m.Qc128, m.Qn128, m.dOc128, m.dOn128, m.Kc64, m.Kn64, m.Vc64, m.Vn64, p, n, status, limit_ns);
  } else {
    e = cudaFuncSetAttribute(bdlm_bwd_dq_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DqLayout<64>::kAlloc);
    if (e != cudaSuccess) return e;
    bdlm_bwd_dq_tc_kernel<64><<<grid, kThreads, DqLayout<64>::kAlloc, stream>>>(
        m.Qc128, m.Qn128, m.dOc128, m.dOn128, m.Kc64, m.Kn64, m.Vc64, m.Vn64, p, n, status, limit_ns);
  }
  if (launches) ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkv_tc(const BwdMaps& m, const BwdParams& p, int num_sms, uint32_t* status,
                              uint64_t limit_ns, cudaStream_t stream, int* launches) {
  const int64_t n = kv_items(p.g, KBM);
  if (n == 0) return cudaSuccess;
  const int grid = (int)(n < num_sms ? n : num_sms);
  cudaError_t e;
  if (p.d == 128) {
    e = cudaFuncSetAttribute(bdlm_bwd_dkv_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DkvLayout<128>::kAlloc);
    if (e != cudaSuccess) return e;
    bdlm_bwd_dkv_tc_kernel<128><<<grid, kThreads, DkvLayout<128>::kAlloc, stream>>>(
        m.Qc64, m.Qn64, m.dOc64, m.dOn64, m.Kc128, m.Kn128, m.Vc128, m.Vn128, p, n, status, limit_ns);
  } else {
    e = cudaFuncSetAttribute(bdlm_bwd_dkv_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DkvLayout<64>::kAlloc);
    if (e != cudaSuccess) return e;
    bdlm_bwd_dkv_tc_kernel<64><<<grid, kThreads, DkvLayout<64>::kAlloc, stream>>>(
        m.Qc64, m.Qn64, m.dOc64, m.dOn64, m.Kc128, m.Kn128, m.Vc128, m.Vn128, p, n, status, limit_ns);
  }
  if (launches) ++*launches;
  return cudaGetLastError();
}

}  // namespace bdlm
