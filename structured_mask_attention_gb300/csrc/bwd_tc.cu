// bwd_tc.cu -- two-stream BDLM attention backward on the sm_103a tensor cores.
//
// Gradients of softmax attention under the two-stream block mask, no gradient
// through LSE ("Block Parallelism For Efficient Distributed Long-Context
// Diffusion Language Model Training": training gradients, evolve.pub review
// "Key claims" / Proposition 1; only clean K/V gradients cross context shards,
// evolve.pub FAQ on CSBP):
//   P = exp(scale Q K^T - LSE), dP = dO V^T, dS = P o (dP - D),
//   dV = sum_group P^T dO, dK = scale sum_group dS^T Q, dQ = scale dS K.
// Two deterministic passes; every output element is written once.
//
// Both kernels are persistent (one CTA per SM) with 10 warps:
//   warp 0     producer: TMA tiles into shared-memory rings (and, for dK/dV,
//              the LSE/D slices of each query tile through cp.async);
//   warp 1     owns TMEM; one lane issues tcgen05.mma;
//   warps 2-9  two elementwise warpgroups.  A thread owns one TMEM lane (a
//              query row for dQ, a key row for dK/dV); the two warpgroups
//              split the 64 columns of each step, 32 each, so every SM
//              sub-partition runs two of these warps.  Tiles that every row
//              sees completely take a branch-free path.  Each warpgroup
//              writes its bf16 results (dS, or P^T and dS^T) back into the
//              TMEM columns it has just read, where the next MMA takes them
//              as its A operand; the MMA warp issues the MMA that overwrites
//              those columns only after the one that reads them (the tensor
//              pipe runs in issue order).
//
// dQ pass (bdlm_bwd_dq_tc): item = (128-row query tile, head, stream), in the
//   forward's longest-first order.  Q and dO of the item are copied into TMEM
//   by the elementwise threads (one row each) and stay there; 64-key K/V
//   tiles stream through a 4-stage TMA ring.  MMA: S = Q K^T and dP = dO V^T
//   (A operands in TMEM) into one of two TMEM buffer pairs, then
//   dQ += dS K (dS in TMEM, K read as an MN-major operand of the same tile).
//
// dK/dV pass (bdlm_bwd_dkv_tc): item = (key stream, KV head, 128-key tile):
//   clean tiles first (read by every later row), then corrupted tiles.  K and
//   V stay in shared memory; 64-row Q/dO tiles of every query head of the GQA
//   group and both streams that see the keys stream through a 4-stage ring.
//   MMA: S^T = K Q^T, dP^T = V dO^T, then dV += P^T dO and dK += dS^T Q with
//   P^T and dS^T in TMEM and Q/dO read as MN-major operands.  dK and dV
//   accumulate in TMEM across the whole group and are written once.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

constexpr int kThreads = 320;
constexpr int kEwThreads = 256;  // elementwise threads (barrier arrival counts)
constexpr float kLog2e = 1.4426950408889634f;

// thread roles
struct Role {
  int warp, lane, quarter, half, row;
  uint32_t tl;  // TMEM lane offset of this warp
};
__device__ __forceinline__ Role role() {
  Role r;
  r.warp = threadIdx.x >> 5;
  r.lane = threadIdx.x & 31;
  r.quarter = r.warp & 3;
  r.half = (r.warp - 2) >> 2;  // valid for warps 2..9
  r.row = r.quarter * 32 + r.lane;
  r.tl = (uint32_t)(r.quarter * 32) << 16;
  return r;
}

__device__ __forceinline__ void store_row32(void* base, int64_t off, const uint32_t (&u)[32], float mul, int f32,
                                            int accumulate) {
  if (f32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float4 v = make_float4(__uint_as_float(u[4 * c]) * mul, __uint_as_float(u[4 * c + 1]) * mul,
                             __uint_as_float(u[4 * c + 2]) * mul, __uint_as_float(u[4 * c + 3]) * mul);
      if (accumulate) {
        const float4 old = o[c];
        v.x += old.x; v.y += old.y; v.z += old.z; v.w += old.w;
      }
      o[c] = v;
    }
  } else {
    uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      o[c] = make_uint4(pack_bf16x2(__uint_as_float(u[8 * c + 0]) * mul, __uint_as_float(u[8 * c + 1]) * mul),
                        pack_bf16x2(__uint_as_float(u[8 * c + 2]) * mul, __uint_as_float(u[8 * c + 3]) * mul),
                        pack_bf16x2(__uint_as_float(u[8 * c + 4]) * mul, __uint_as_float(u[8 * c + 5]) * mul),
                        pack_bf16x2(__uint_as_float(u[8 * c + 6]) * mul, __uint_as_float(u[8 * c + 7]) * mul));
  }
}

// TMEM column of the packed bf16 A operand for 16-row (or 16-key) K-step kk
// of a 64-wide step whose two 32-wide halves were written, 16 packed columns
// each, at the start of the 32-column region the half had read.
__device__ __forceinline__ uint32_t packed_col(int kk) { return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8); }

// ====================================================================== dQ
constexpr int QBM = 128;  // query rows per item
constexpr int QBN = 64;   // keys per step
constexpr int QNS = 4;    // K/V stages

enum { DQ_QL = 0, DQ_KVFULL = 1, DQ_KVEMPTY = 5, DQ_SFULL = 9, DQ_DSFULL = 11, DQ_DONE = 13, DQ_OEMPTY = 14,
       DQ_NBAR = 15 };

template <int HD>
struct DqLayout {
  static constexpr int kKTile = QBN * HD * 2;  // 64 rows
  static constexpr int kKPanel = QBN * 128;    // 8 KB
  static constexpr int kK = 0;
  static constexpr int kV = kK + QNS * kKTile;
  static constexpr int kBar = kV + QNS * kKTile;
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

// One row's half of a [L, H, HD] bf16 tensor row (HD/2 elements = HD/4
// packed columns) -> TMEM, packed two bf16 per 32-bit column in memory order.
template <int HD>
__device__ __forceinline__ void row_half_to_tmem(uint32_t taddr, const __nv_bfloat16* src, bool valid) {
  constexpr int NC = HD / 4;  // packed columns per half: 32 (HD=128) or 16 (HD=64)
  uint32_t u[NC];
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < NC / 4; ++i) {
    const uint4 v = valid ? s4[i] : make_uint4(0u, 0u, 0u, 0u);
    u[4 * i + 0] = v.x;
    u[4 * i + 1] = v.y;
    u[4 * i + 2] = v.z;
    u[4 * i + 3] = v.w;
  }
  if constexpr (NC == 32) {
    tmem_st32(taddr, u);
  } else {
    tmem_st16(taddr, u);
  }
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    bdlm_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tKc, const __grid_constant__ CUtensorMap tKn,
                          const __grid_constant__ CUtensorMap tVc, const __grid_constant__ CUtensorMap tVn,
                          const BwdParams p, const int64_t n_items, uint32_t* status, const uint64_t limit_ns) {
  using LY = DqLayout<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  const uint32_t sK = base + LY::kK, sV = base + LY::kV;
  const uint32_t bars = base + LY::kBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + LY::kBar + 8 * DQ_NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + LY::kBar + 8 * DQ_NBAR + 4);
  auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  const Role R = role();

  if (threadIdx.x == 0) {
    mbar_init(BAR(DQ_QL), kEwThreads);
    for (int s = 0; s < QNS; ++s) {
      mbar_init(BAR(DQ_KVFULL + s), 1);
      mbar_init(BAR(DQ_KVEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(BAR(DQ_SFULL + s), 1);
      mbar_init(BAR(DQ_DSFULL + s), kEwThreads);
    }
    mbar_init(BAR(DQ_DONE), 1);
    mbar_init(BAR(DQ_OEMPTY), kEwThreads);
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
  // TMEM columns: S[2] at 0/64 (dS over them), dP[2] at 128/192, dQ at 256,
  // Q at 384, dO at 384 + HD/2 (packed bf16)
  constexpr uint32_t kColQ = 384, kColdO = 384 + HD / 2;
  if (R.warp == 0) {
    if (R.lane == 0) {
      uint32_t kvc = 0;
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        const int64_t idx = snake_item(rnd, cta, grid);
        if (idx >= n_items) break;
        const DqGeo t = dq_geo(p, idx);
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
      }
    }
  } else if (R.warp == 1) {
    if (R.lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(QBM, QBN, false, false);
      constexpr uint32_t kIdQ = idesc_bf16(QBM, HD, false, true);
      uint32_t itn = 0, kvc = 0, sc = 0, dc = 0;
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        const int64_t idx = snake_item(rnd, cta, grid);
        if (idx >= n_items) break;
        const DqGeo t = dq_geo(p, idx);
        if (t.n == 0) continue;
        if (!mbar_wait(BAR(DQ_QL), itn & 1, wd, 23)) { ok = false; break; }  // Q, dO in TMEM
        const uint32_t kv_base = kvc;
        auto do_dq = [&](int jj) -> bool {
          const uint32_t kv = kv_base + jj;
          const int st = kv % QNS;
          const int db = dc & 1;
          if (!mbar_wait(BAR(DQ_DSFULL + db), (dc >> 1) & 1, wd, 24)) return false;
          if (jj == 0 && itn > 0 && !mbar_wait(BAR(DQ_OEMPTY), (itn - 1) & 1, wd, 25)) return false;
          tc_fence_after();
          const uint64_t bk0 = sdesc_sw128(sK + st * LY::kKTile, LY::kKPanel, 1024);
          const uint32_t acc0 = jj > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < QBN / 16; ++kk)
            tc_mma_ts(tmem + 256, tmem + db * QBN + packed_col(kk), desc_add(bk0, kk * 2048), kIdQ,
                      kk > 0 ? 1u : acc0);
          tc_commit(BAR(DQ_KVEMPTY + st));
          ++dc;
          return true;
        };
        for (int j = 0; j < t.n && ok; ++j, ++kvc, ++sc) {
          const int st = kvc % QNS;
          const int sb = sc & 1;
          if (!mbar_wait(BAR(DQ_KVFULL + st), (kvc / QNS) & 1, wd, 26)) { ok = false; break; }
          tc_fence_after();
          // buffer sb was last read by dQ(j-2), issued before this point
          const uint64_t dk0 = sdesc_sw128(sK + st * LY::kKTile, 16, 1024);
          const uint64_t dv0 = sdesc_sw128(sV + st * LY::kKTile, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t ko = (kk >> 2) * LY::kKPanel + (kk & 3) * 32;
            tc_mma_ts(tmem + sb * QBN, tmem + kColQ + kk * 8, desc_add(dk0, ko), kIdS, kk > 0 ? 1u : 0u);
            tc_mma_ts(tmem + 128 + sb * QBN, tmem + kColdO + kk * 8, desc_add(dv0, ko), kIdS, kk > 0 ? 1u : 0u);
          }
          tc_commit(BAR(DQ_SFULL + sb));
          if (j >= 1 && !do_dq(j - 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!do_dq(t.n - 1)) { ok = false; break; }
        tc_commit(BAR(DQ_DONE));
        ++itn;
      }
    }
  } else {
    // elementwise: thread = query row, warpgroup `half` = key columns [32 half, 32 half + 32)
    const int row = R.row, half = R.half;
    uint32_t itn = 0, sc = 0;
    bool ok = true;
    for (int64_t rnd = 0; ok; ++rnd) {
      const int64_t idx = snake_item(rnd, cta, grid);
      if (idx >= n_items) break;
      const DqGeo t = dq_geo(p, idx);
      const int64_t r = t.r0 + row;
      const bool valid = r < p.g.L;
      void* dqbase = t.stream ? p.dQn : p.dQc;
      const int64_t oofs = (r * p.g.Hq + t.head) * HD + half * (HD / 2);
      if (t.n == 0) {
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
      // Q and dO rows of this item into TMEM (the previous item's MMAs that
      // read them are complete: its epilogue waited for DQ_DONE)
      {
        const int64_t rs = valid ? r : 0;
        const __nv_bfloat16* qsrc = static_cast<const __nv_bfloat16*>(t.stream ? p.Qn : p.Qc) +
                                    (rs * p.g.Hq + t.head) * HD + half * (HD / 2);
        const __nv_bfloat16* osrc = static_cast<const __nv_bfloat16*>(t.stream ? p.dOn : p.dOc) +
                                    (rs * p.g.Hq + t.head) * HD + half * (HD / 2);
        row_half_to_tmem<HD>(tmem + R.tl + kColQ + half * (HD / 4), qsrc, valid);
        row_half_to_tmem<HD>(tmem + R.tl + kColdO + half * (HD / 4), osrc, valid);
        tc_fence_before();
        mbar_arrive(BAR(DQ_QL));
      }
      const int64_t rr = valid ? r : p.g.L - 1;
      int64_t clo, chi, nlo, nhi;
      clean_interval(p.g, t.stream, rr, clo, chi);
      noisy_interval(p.g, t.stream, rr, nlo, nhi);
      const float nlse2 = valid ? -(t.stream ? p.LSEn : p.LSEc)[(int64_t)t.head * p.g.L + r] * kLog2e : 0.f;
      const float Dv = valid ? (t.stream ? p.Dn : p.Dc)[(int64_t)t.head * p.g.L + r] : 0.f;
      const float sl2 = p.scale_log2;
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
        uint32_t us[32], ud[32];
        const uint32_t tS = tmem + R.tl + sb * QBN + half * 32;
        tmem_ld32x2(tS, tmem + R.tl + 128 + sb * QBN + half * 32, us, ud);
        uint32_t pk[16];
        if (full) {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float d0 = ex2_approx(fmaf(__uint_as_float(us[c]), sl2, nlse2)) * (__uint_as_float(ud[c]) - Dv);
            const float d1 =
                ex2_approx(fmaf(__uint_as_float(us[c + 1]), sl2, nlse2)) * (__uint_as_float(ud[c + 1]) - Dv);
            pk[c / 2] = pack_bf16x2(d0, d1);
          }
        } else {
          const int lo = (int)imax64(imin64((cs ? clo : nlo) - key0 - half * 32, 33), -1);
          const int hi = (int)imax64(imin64((cs ? chi : nhi) - key0 - half * 32, 33), -1);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float d0 = ex2_approx(fmaf(__uint_as_float(us[c]), sl2, nlse2)) * (__uint_as_float(ud[c]) - Dv);
            float d1 = ex2_approx(fmaf(__uint_as_float(us[c + 1]), sl2, nlse2)) * (__uint_as_float(ud[c + 1]) - Dv);
            d0 = (c >= lo && c < hi) ? d0 : 0.f;
            d1 = (c + 1 >= lo && c + 1 < hi) ? d1 : 0.f;
            pk[c / 2] = pack_bf16x2(d0, d1);
          }
        }
        // dS (bf16) over the first 16 columns of the S columns this half read
        tmem_st16(tS, pk);
        tc_fence_before();
        mbar_arrive(BAR(DQ_DSFULL + sb));
      }
      if (!ok) break;
      ok = mbar_wait(BAR(DQ_DONE), itn & 1, wd, 30);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c4 = 0; c4 < HD / 64; ++c4) {
        uint32_t u[32];
        tmem_ld32(tmem + R.tl + 256 + half * (HD / 2) + c4 * 32, u);
        if (valid) store_row32(dqbase, oofs + c4 * 32, u, p.scale, p.g_f32, p.dq_accumulate);
      }
      tc_fence_before();
      mbar_arrive(BAR(DQ_OEMPTY));
      ++itn;
    }
  }
  __syncthreads();
  if (*abort_flag) drain_after_abort(200);
  if (R.warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// =================================================================== dK / dV
constexpr int KBM = 128;  // keys per item
constexpr int KBN = 64;   // query rows per step
constexpr int KNS = 4;    // Q/dO stages

enum { KV_KFULL = 0, KV_KEMPTY = 1, KV_QFULL = 2, KV_QEMPTY = 6, KV_SFULL = 10, KV_PFULL = 12, KV_ACCDONE = 14,
       KV_ACCEMPTY = 15, KV_NBAR = 16 };

template <int HD>
struct DkvLayout {
  static constexpr int kKTile = KBM * HD * 2;  // 128 key rows
  static constexpr int kQTile = KBN * HD * 2;  // 64 query rows
  static constexpr int kKPanel = KBM * 128;    // 16 KB
  static constexpr int kQPanel = KBN * 128;    // 8 KB
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKTile;
  static constexpr int kQ = kV + kKTile;
  static constexpr int kdO = kQ + KNS * kQTile;
  static constexpr int kStat = kdO + KNS * kQTile;  // per stage: LSE[64] then D[64], fp32
  static constexpr int kBar = kStat + KNS * 2 * KBN * 4;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
};

struct DkvGeo {
  int ks, kvh;
  int64_t j0;
  int64_t rlo0, rhi0, rlo1, rhi1;  // query rows of each stream that can see some key of the tile
  int64_t t00, t01;                // first query tile of each stream
  int nt0, nt1;                    // query tiles of each stream
  int per_head, n;                 // steps per head, total steps
};

__device__ __forceinline__ DkvGeo dkv_geo(const BwdParams& p, int64_t idx) {
  DkvGeo t;
  const KVItem it = kv_item(p.g, KBM, idx);
  t.ks = it.key_stream;
  t.kvh = it.kv_head;
  t.j0 = it.ktile * KBM;
  const int64_t j1 = imin64(t.j0 + KBM, p.g.L);
  kv_tile_rows(p.g, t.ks, t.j0, j1, t.rlo0, t.rhi0, t.rlo1, t.rhi1);
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
                 sStat = base + LY::kStat;
  const float* stat_ptr = reinterpret_cast<const float*>(base_ptr + LY::kStat);
  const uint32_t bars = base + LY::kBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + LY::kBar + 8 * KV_NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + LY::kBar + 8 * KV_NBAR + 4);
  auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  const Role R = role();

  if (threadIdx.x == 0) {
    mbar_init(BAR(KV_KFULL), 1);
    mbar_init(BAR(KV_KEMPTY), 1);
    for (int s = 0; s < KNS; ++s) {
      mbar_init(BAR(KV_QFULL + s), 1 + 32);  // expect_tx arrival + one cp.async arrival per producer lane
      mbar_init(BAR(KV_QEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(BAR(KV_SFULL + s), 1);
      mbar_init(BAR(KV_PFULL + s), kEwThreads);
    }
    mbar_init(BAR(KV_ACCDONE), 1);
    mbar_init(BAR(KV_ACCEMPTY), kEwThreads);
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
  // TMEM columns: dK at 0, dV at 128, S^T[2] at 256/320 (P^T over them),
  // dP^T[2] at 384/448 (dS^T over them)
  if (R.warp == 0) {
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
      if (R.lane == 0) {
        mbar_arrive_expect_tx(BAR(KV_KFULL), 2 * LY::kKTile);
        const CUtensorMap* mk = t.ks ? &tKn : &tKc;
        const CUtensorMap* mv = t.ks ? &tVn : &tVc;
#pragma unroll
        for (int pn = 0; pn < HD / 64; ++pn) {
          tma_load_3d(sK + pn * LY::kKPanel, mk, BAR(KV_KFULL), pn * 64, t.kvh, (int)t.j0);
          tma_load_3d(sV + pn * LY::kKPanel, mv, BAR(KV_KFULL), pn * 64, t.kvh, (int)t.j0);
        }
      }
      DkvCursor cur;
      cur.reset();
      for (int k = 0; k < t.n; ++k, ++qc, cur.advance(t)) {
        const int st = qc % KNS;
        if (qc >= KNS) {
          ok = __all_sync(0xffffffffu, mbar_wait(BAR(KV_QEMPTY + st), ((qc / KNS) - 1) & 1, wd, 42));
          if (!ok) break;
        }
        int head, s;
        int64_t q0;
        cur.get(p, t, head, s, q0);
        if (R.lane == 0) {
          mbar_arrive_expect_tx(BAR(KV_QFULL + st), 2 * LY::kQTile);
          const CUtensorMap* mq = s ? &tQn : &tQc;
          const CUtensorMap* mo = s ? &tdOn : &tdOc;
#pragma unroll
          for (int pn = 0; pn < HD / 64; ++pn) {
            tma_load_3d(sQ + st * LY::kQTile + pn * LY::kQPanel, mq, BAR(KV_QFULL + st), pn * 64, head, (int)q0);
            tma_load_3d(sdO + st * LY::kQTile + pn * LY::kQPanel, mo, BAR(KV_QFULL + st), pn * 64, head, (int)q0);
          }
        }
        // LSE and D of the tile's 64 rows, asynchronously (rows >= L read as 0)
        const float* LSE = (s ? p.LSEn : p.LSEc) + (int64_t)head * p.g.L;
        const float* Dr = (s ? p.Dn : p.Dc) + (int64_t)head * p.g.L;
        const uint32_t stat = sStat + st * 2 * KBN * 4;
#pragma unroll
        for (int c = R.lane; c < KBN; c += 32) {
          const int64_t r = q0 + c;
          const bool v = r < p.g.L;
          cp_async4(stat + c * 4, LSE + (v ? r : 0), v);
          cp_async4(stat + (KBN + c) * 4, Dr + (v ? r : 0), v);
        }
        cp_async_mbar_arrive(BAR(KV_QFULL + st));
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
          const uint64_t bo0 = sdesc_sw128(sdO + st * LY::kQTile, LY::kQPanel, 1024);
          const uint64_t bq0 = sdesc_sw128(sQ + st * LY::kQTile, LY::kQPanel, 1024);
          const uint32_t acc0 = kk > 0 ? 1u : 0u;
#pragma unroll
          for (int k4 = 0; k4 < KBN / 16; ++k4) {
            const uint32_t acc = k4 > 0 ? 1u : acc0;
            tc_mma_ts(tmem + 128, tmem + 256 + pb * KBN + packed_col(k4), desc_add(bo0, k4 * 2048), kIdA, acc);
            tc_mma_ts(tmem + 0, tmem + 384 + pb * KBN + packed_col(k4), desc_add(bq0, k4 * 2048), kIdA, acc);
          }
          tc_commit(BAR(KV_QEMPTY + st));
          ++pc;
          return true;
        };
        for (int k = 0; k < t.n && ok; ++k, ++qc, ++sc) {
          const int st = qc % KNS;
          const int sb = sc & 1;
          if (!mbar_wait(BAR(KV_QFULL + st), (qc / KNS) & 1, wd, 46)) { ok = false; break; }
          tc_fence_after();
          // buffer sb was last read by the dV/dK MMAs of step k-2, issued before this point
          const uint64_t dq0 = sdesc_sw128(sQ + st * LY::kQTile, 16, 1024);
          const uint64_t do0 = sdesc_sw128(sdO + st * LY::kQTile, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t ko = (kk >> 2) * LY::kKPanel + (kk & 3) * 32;
            const uint32_t qo = (kk >> 2) * LY::kQPanel + (kk & 3) * 32;
            tc_mma_ss(tmem + 256 + sb * KBN, desc_add(dK0, ko), desc_add(dq0, qo), kIdS, kk > 0 ? 1u : 0u);
            tc_mma_ss(tmem + 384 + sb * KBN, desc_add(dV0, ko), desc_add(do0, qo), kIdS, kk > 0 ? 1u : 0u);
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
    const int row = R.row, half = R.half;
    uint32_t itn = 0, qc = 0, sc = 0;
    bool ok = true;
    const float sl2 = p.scale_log2;
    for (int64_t rnd = 0; ok; ++rnd) {
      const int64_t idx = snake_item(rnd, cta, grid);
      if (idx >= n_items) break;
      const DkvGeo t = dkv_geo(p, idx);
      if (t.n == 0) continue;
      const int64_t j = t.j0 + row;
      int64_t klo0, khi0, klo1, khi1;
      key_rows(p.g, t.ks, j, 0, klo0, khi0);
      key_rows(p.g, t.ks, j, 1, klo1, khi1);
      // rows every key of the tile sees (for the full-tile test)
      int64_t alo0, ahi0, alo1, ahi1;
      {
        const int64_t jl = imin64(t.j0 + KBM, p.g.L) - 1;
        bool all_in = t.j0 + KBM <= p.g.L;
        if (t.ks == 0) all_in = all_in && t.j0 >= p.g.kv_begin && t.j0 + KBM <= p.g.kv_end;
        int64_t a0, b0, a1, b1;
        key_rows(p.g, t.ks, t.j0, 0, a0, b0);
        key_rows(p.g, t.ks, jl, 0, a1, b1);
        alo0 = imax64(a0, a1);
        ahi0 = all_in ? imin64(b0, b1) : alo0;
        key_rows(p.g, t.ks, t.j0, 1, a0, b0);
        key_rows(p.g, t.ks, jl, 1, a1, b1);
        alo1 = imax64(a0, a1);
        ahi1 = all_in ? imin64(b0, b1) : alo1;
      }
      DkvCursor cur;
      cur.reset();
      for (int k = 0; k < t.n; ++k, ++qc, ++sc, cur.advance(t)) {
        int head, s;
        int64_t q0;
        cur.get(p, t, head, s, q0);
        (void)head;
        const int st = qc % KNS;
        const int sb = sc & 1;
        ok = mbar_wait(BAR(KV_SFULL + sb), (sc >> 1) & 1, wd, 48);
        if (ok) ok = mbar_wait(BAR(KV_QFULL + st), (qc / KNS) & 1, wd, 49);  // LSE/D landed
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t us[32], ud[32];
        const uint32_t tS = tmem + R.tl + 256 + sb * KBN + half * 32;
        const uint32_t tD = tmem + R.tl + 384 + sb * KBN + half * 32;
        tmem_ld32x2(tS, tD, us, ud);
        const float* stl = stat_ptr + st * 2 * KBN + half * 32;  // LSE of this half's 32 rows; D at +KBN
        const bool full = s == 0 ? (q0 >= alo0 && q0 + KBN <= ahi0) : (q0 >= alo1 && q0 + KBN <= ahi1);
        const int64_t base_row = q0 + half * 32;
        const int lo = full ? -1 : (int)imax64(imin64((s == 0 ? klo0 : klo1) - base_row, 33), -1);
        const int hi = full ? 33 : (int)imax64(imin64((s == 0 ? khi0 : khi1) - base_row, 33), -1);
        uint32_t pp[16], dd[16];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 l4 = *reinterpret_cast<const float4*>(stl + 4 * c4);
          const float4 d4 = *reinterpret_cast<const float4*>(stl + KBN + 4 * c4);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
          float pv[4], sv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 4 * c4 + e;
            float pe = ex2_approx(fmaf(__uint_as_float(us[c]), sl2, -lv[e] * kLog2e));
            if (!full) pe = (c >= lo && c < hi) ? pe : 0.f;
            pv[e] = pe;
            sv[e] = pe * (__uint_as_float(ud[c]) - dv[e]);
          }
          pp[2 * c4] = pack_bf16x2(pv[0], pv[1]);
          pp[2 * c4 + 1] = pack_bf16x2(pv[2], pv[3]);
          dd[2 * c4] = pack_bf16x2(sv[0], sv[1]);
          dd[2 * c4 + 1] = pack_bf16x2(sv[2], sv[3]);
        }
        // P^T and dS^T (bf16) over the first 16 columns of what this half read
        tmem_st16(tS, pp);
        tmem_st16(tD, dd);
        tc_fence_before();
        mbar_arrive(BAR(KV_PFULL + sb));
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
      const int64_t oofs = (j * p.g.Hkv + t.kvh) * HD + half * (HD / 2);
#pragma unroll
      for (int c4 = 0; c4 < HD / 64; ++c4) {
        uint32_t uk[32], uv[32];
        tmem_ld32x2(tmem + R.tl + half * (HD / 2) + c4 * 32, tmem + R.tl + 128 + half * (HD / 2) + c4 * 32, uk, uv);
        if (wr) {
          store_row32(dKo, oofs + c4 * 32, uk, p.scale, p.g_f32, 0);
          store_row32(dVo, oofs + c4 * 32, uv, 1.f, p.g_f32, 0);
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(KV_ACCEMPTY));
      ++itn;
    }
  }
  __syncthreads();
  if (*abort_flag) drain_after_abort(200);
  if (R.warp == 1) {
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
        m.Kc64, m.Kn64, m.Vc64, m.Vn64, p, n, status, limit_ns);
  } else {
    e = cudaFuncSetAttribute(bdlm_bwd_dq_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DqLayout<64>::kAlloc);
    if (e != cudaSuccess) return e;
    bdlm_bwd_dq_tc_kernel<64><<<grid, kThreads, DqLayout<64>::kAlloc, stream>>>(
        m.Kc64, m.Kn64, m.Vc64, m.Vn64, p, n, status, limit_ns);
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
