// fwd_tc.cu -- two-stream BDLM attention forward on the sm_103a tensor cores.
//
// Computes, for every query row of both streams, O = softmax(scale Q K^T) V
// over the row's visible keys and LSE = ln sum exp(scale q.k) ("Block
// Parallelism For Efficient Distributed Long-Context Diffusion Language Model
// Training": the clean-plus-corrupted sequence and its block mask, arxiv.science
// abstract; per-target-block separation, evolve.pub review "Scope & Claims",
// Eq. 3 / Eq. 6).  The same kernel computes one context shard's partial
// (clean keys restricted to [kv_begin, kv_end), corrupted own block optional:
// CSBP, evolve.pub FAQ), writing O = 0, LSE = -inf for rows with no key.
//
// Design (one CTA per SM, persistent; 10 warps).  A CTA works on a PAIR of
// 128-row query tiles at once: the clean and the corrupted tile of the same
// head and position (equal work: both see (b+1)B keys per row).  Keys come in
// steps of 64.  Each tile has its own Q slot, two K and two V slots in shared
// memory, and in TMEM two 64-column S buffers and its O accumulator:
//   warp 0      TMA producer (K of a step as soon as the S MMA two steps
//               back released its slot, V likewise after the PV MMA);
//   warp 1      owns TMEM (512 columns); one lane issues tcgen05.mma: per
//               step, S(j) = Q K^T(j) of both tiles into the free S buffers,
//               then PV(j-1) of both tiles, so every tile's softmax of step j
//               overlaps its own S(j+1) and the other tile's MMAs;
//   warps 2-5   softmax warpgroup of tile 0, warps 6-9 of tile 1: one query
//               row per thread, online softmax in the log2 domain with a lazy
//               rescale (the reference max moves only when the row max grows
//               by more than 8), P written back over the S buffer in TMEM as
//               packed bf16 and consumed from there by the PV MMA (A operand
//               in TMEM).  The S MMA that next reuses a buffer is issued after
//               the PV MMA that reads its P (the tensor pipe runs in issue
//               order).
// Only key tiles some row of the query tile can see are visited; a per-row
// interval test masks the tiles that are not fully visible.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

constexpr int BM = kFwdTileQ;   // query rows per tile
constexpr int BN = kFwdTileK;   // keys per step (64)
constexpr int kThreads = 320;
constexpr int kQPanel = BM * 128;  // 128 rows x 128 bytes (64 bf16)
constexpr int kKPanel = BN * 128;  // 64 rows x 128 bytes
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// barrier slots per tile (tile t adds t * B_PER_TILE)
enum { B_QF = 0, B_QE = 1, B_KF = 2, B_KE = 4, B_VF = 6, B_VE = 8, B_SF = 10, B_PF = 12, B_PVD = 13, B_OE = 14,
       B_PER_TILE = 15, B_COUNT = 30 };

template <int HD>
struct Layout {
  static constexpr int kQBytes = BM * HD * 2;  // 128 rows x HD bf16
  static constexpr int kKBytes = BN * HD * 2;  // 64 rows x HD bf16
  // per tile t at t * kTile: Q, K[2], V[2]
  static constexpr int kTile = kQBytes + 4 * kKBytes;
  static constexpr int kBar = 2 * kTile;
  static constexpr int kBytes = kBar + 512;
  // 1024 bytes of slack for alignment; never below 120 KB so that a second
  // CTA cannot share the SM (each CTA holds all 512 TMEM columns).
  static constexpr int kAlloc = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
};

struct ItemGeo {
  int stream, head, kvh;
  int64_t r0;
  QTileRanges q;
  int nc, n;  // clean tiles, total tiles
};

__device__ __forceinline__ ItemGeo item_geo(const FwdParams& p, int64_t idx) {
  ItemGeo t;
  const QItem it = q_item(p.g, BM, idx);
  t.stream = it.stream;
  t.head = it.head;
  t.kvh = it.head / (p.g.Hq / p.g.Hkv);
  t.r0 = it.qtile * BM;
  const int64_t r1 = imin64(t.r0 + BM, p.g.L);
  t.q = qtile_ranges(p.g, t.stream, t.r0, r1, BN);
  t.nc = (int)(t.q.c1 - t.q.c0);
  t.n = t.nc + (int)(t.q.n1 - t.q.n0);
  return t;
}

__device__ __forceinline__ int64_t tile_key0(const ItemGeo& t, int j) {
  return (j < t.nc ? t.q.c0 + j : t.q.n0 + (j - t.nc)) * BN;
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    bdlm_fwd_tc_kernel(const __grid_constant__ CUtensorMap tQc, const __grid_constant__ CUtensorMap tQn,
                       const __grid_constant__ CUtensorMap tKc, const __grid_constant__ CUtensorMap tKn,
                       const __grid_constant__ CUtensorMap tVc, const __grid_constant__ CUtensorMap tVn,
                       const FwdParams p) {
  using LY = Layout<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  auto sQ = [&](int t) -> uint32_t { return base + t * LY::kTile; };
  auto sK = [&](int t, int st) -> uint32_t { return base + t * LY::kTile + LY::kQBytes + st * LY::kKBytes; };
  auto sV = [&](int t, int st) -> uint32_t {
    return base + t * LY::kTile + LY::kQBytes + (2 + st) * LY::kKBytes;
  };
  const uint32_t bars = base + LY::kBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + LY::kBar + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + LY::kBar + 8 * B_COUNT + 4);
  auto BAR = [&](int i, int t) -> uint32_t { return bars + 8u * (uint32_t)(i + t * B_PER_TILE); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR(B_QF, t), 1);
      mbar_init(BAR(B_QE, t), 1);
      for (int st = 0; st < 2; ++st) {
        mbar_init(BAR(B_KF + st, t), 1);
        mbar_init(BAR(B_KE + st, t), 1);
        mbar_init(BAR(B_VF + st, t), 1);
        mbar_init(BAR(B_VE + st, t), 1);
        mbar_init(BAR(B_SF + st, t), 1);
      }
      mbar_init(BAR(B_PF, t), 128);
      mbar_init(BAR(B_PVD, t), 1);
      mbar_init(BAR(B_OE, t), 128);
    }
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
  const Watchdog wd{p.status, p.limit_ns, abort_flag};
  const int grid = gridDim.x, cta = blockIdx.x;
  const int64_t n_pairs = p.n_items / 2;  // items 2i, 2i+1: clean and corrupted tile of one head/position
  // TMEM columns: S buffers of tile t at 128 t + {0, 64} (P over their first
  // 32 columns), O of tile t at 256 + 128 t

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tQc); tma_prefetch_desc(&tQn); tma_prefetch_desc(&tKc);
      tma_prefetch_desc(&tKn); tma_prefetch_desc(&tVc); tma_prefetch_desc(&tVn);
      uint32_t qc[2] = {0, 0}, kc[2] = {0, 0}, vc[2] = {0, 0};
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        const int64_t pi = snake_item(rnd, cta, grid);
        if (pi >= n_pairs) break;
        const ItemGeo g0 = item_geo(p, 2 * pi), g1 = item_geo(p, 2 * pi + 1);
        const int nmax = g0.n > g1.n ? g0.n : g1.n;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const ItemGeo& g = t ? g1 : g0;
          if (g.n == 0 || !ok) continue;
          if (qc[t] > 0 && !mbar_wait(BAR(B_QE, t), (qc[t] - 1) & 1, wd, 1)) { ok = false; continue; }
          mbar_arrive_expect_tx(BAR(B_QF, t), LY::kQBytes);
          const CUtensorMap* mq = g.stream ? &tQn : &tQc;
#pragma unroll
          for (int pn = 0; pn < HD / 64; ++pn)
            tma_load_3d(sQ(t) + pn * kQPanel, mq, BAR(B_QF, t), pn * 64, g.head, (int)g.r0);
          ++qc[t];
        }
        for (int j = 0; j < nmax && ok; ++j) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const ItemGeo& g = t ? g1 : g0;
            if (j >= g.n || !ok) continue;
            const uint32_t k = kc[t];
            const int st = k & 1;
            if (k >= 2 && !mbar_wait(BAR(B_KE + st, t), ((k >> 1) - 1) & 1, wd, 2)) { ok = false; continue; }
            const CUtensorMap* mk = j < g.nc ? &tKc : &tKn;
            mbar_arrive_expect_tx(BAR(B_KF + st, t), LY::kKBytes);
#pragma unroll
            for (int pn = 0; pn < HD / 64; ++pn)
              tma_load_3d(sK(t, st) + pn * kKPanel, mk, BAR(B_KF + st, t), pn * 64, g.kvh, (int)tile_key0(g, j));
            ++kc[t];
          }
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const ItemGeo& g = t ? g1 : g0;
            if (j >= g.n || !ok) continue;
            const uint32_t v = vc[t];
            const int st = v & 1;
            if (v >= 2 && !mbar_wait(BAR(B_VE + st, t), ((v >> 1) - 1) & 1, wd, 3)) { ok = false; continue; }
            const CUtensorMap* mv = j < g.nc ? &tVc : &tVn;
            mbar_arrive_expect_tx(BAR(B_VF + st, t), LY::kKBytes);
#pragma unroll
            for (int pn = 0; pn < HD / 64; ++pn)
              tma_load_3d(sV(t, st) + pn * kKPanel, mv, BAR(B_VF + st, t), pn * 64, g.kvh, (int)tile_key0(g, j));
            ++vc[t];
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16(BM, BN, false, false);
      constexpr uint32_t kIdescO = idesc_bf16(BM, HD, false, true);
      uint32_t qc[2] = {0, 0}, kc[2] = {0, 0}, vc[2] = {0, 0}, oc[2] = {0, 0};
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        const int64_t pi = snake_item(rnd, cta, grid);
        if (pi >= n_pairs) break;
        const ItemGeo g0 = item_geo(p, 2 * pi), g1 = item_geo(p, 2 * pi + 1);
        const int nmax = g0.n > g1.n ? g0.n : g1.n;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const ItemGeo& g = t ? g1 : g0;
          if (g.n == 0 || !ok) continue;
          if (!mbar_wait(BAR(B_QF, t), qc[t] & 1, wd, 4)) { ok = false; continue; }
          ++qc[t];
        }
        for (int j = 0; j <= nmax && ok; ++j) {
          // S(j) of both tiles: buffer (S count & 1); its previous P was read
          // by the PV MMA issued one iteration earlier
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const ItemGeo& g = t ? g1 : g0;
            if (j >= g.n || !ok) continue;
            const uint32_t k = kc[t];
            const int st = k & 1;
            if (!mbar_wait(BAR(B_KF + st, t), (k >> 1) & 1, wd, 8)) { ok = false; continue; }
            tc_fence_after();
            const uint32_t tS = tmem + t * 128 + st * BN;
            const uint64_t dq0 = sdesc_sw128(sQ(t), 16, 1024), dk0 = sdesc_sw128(sK(t, st), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
              const uint32_t qo = (kk >> 2) * kQPanel + (kk & 3) * 32;
              const uint32_t ko = (kk >> 2) * kKPanel + (kk & 3) * 32;
              tc_mma_ss(tS, desc_add(dq0, qo), desc_add(dk0, ko), kIdescS, kk > 0 ? 1u : 0u);
            }
            tc_commit(BAR(B_SF + st, t));
            tc_commit(BAR(B_KE + st, t));
            if (j == g.n - 1) tc_commit(BAR(B_QE, t));
            ++kc[t];
          }
          // PV(j-1) of both tiles: O += P V, P (bf16) in TMEM over its S buffer
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const ItemGeo& g = t ? g1 : g0;
            if (j < 1 || j > g.n || !ok) continue;
            const uint32_t v = vc[t];
            const int st = v & 1;
            if (!mbar_wait(BAR(B_PF, t), v & 1, wd, 5)) { ok = false; continue; }
            if (j == 1 && oc[t] > 0 && !mbar_wait(BAR(B_OE, t), (oc[t] - 1) & 1, wd, 6)) { ok = false; continue; }
            if (!mbar_wait(BAR(B_VF + st, t), (v >> 1) & 1, wd, 7)) { ok = false; continue; }
            tc_fence_after();
            const uint32_t tP = tmem + t * 128 + st * BN, tO = tmem + 256 + t * 128;
            const uint64_t dv0 = sdesc_sw128(sV(t, st), kKPanel, 1024);
            const uint32_t acc0 = j > 1 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              tc_mma_ts(tO, tP + kk * 8, desc_add(dv0, kk * 2048), kIdescO, kk > 0 ? 1u : acc0);
            tc_commit(BAR(B_VE + st, t));
            tc_commit(BAR(B_PVD, t));
            ++vc[t];
            if (j == g.n) ++oc[t];
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax (thread = row of tile t)
    const int t = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t tl = (uint32_t)(quarter * 32) << 16;
    const uint32_t tO = tmem + tl + 256 + t * 128;
    uint32_t sc = 0;
    bool ok = true;
    for (int64_t rnd = 0; ok; ++rnd) {
      const int64_t pi = snake_item(rnd, cta, grid);
      if (pi >= n_pairs) break;
      const ItemGeo g = item_geo(p, 2 * pi + t);
      const int64_t r = g.r0 + row;
      const bool valid = r < p.g.L;
      float* lse_out = (g.stream ? p.LSEn : p.LSEc) + (int64_t)g.head * p.g.L;
      void* obase = g.stream ? p.On : p.Oc;
      const int64_t oofs = (r * p.g.Hq + g.head) * HD;
      if (g.n == 0) {
        if (valid) {
          if (p.o_f32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(obase) + oofs);
#pragma unroll
            for (int c = 0; c < HD / 4; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(obase) + oofs);
#pragma unroll
            for (int c = 0; c < HD / 8; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
          }
          lse_out[r] = -INFINITY;
        }
        continue;
      }
      const int64_t rr = valid ? r : p.g.L - 1;
      int64_t clo, chi, nlo, nhi;
      clean_interval(p.g, g.stream, rr, clo, chi);
      noisy_interval(p.g, g.stream, rr, nlo, nhi);
      const float sl2 = p.scale_log2;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < g.n; ++j, ++sc) {
        const bool cs = j < g.nc;
        const int64_t key0 = tile_key0(g, j);
        const bool full = cs ? tile_full(key0, BN, g.q.c_all_lo, g.q.c_all_hi, p.g.L)
                             : tile_full(key0, BN, g.q.n_all_lo, g.q.n_all_hi, p.g.L);
        const int sb = sc & 1;
        ok = mbar_wait(BAR(B_SF + sb, t), (sc >> 1) & 1, wd, 9);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tmem + tl + t * 128 + sb * BN;
        uint32_t a[32], b[32];
        tmem_ld32x2(tS, tS + 32, a, b);
        float mx = -INFINITY;
        if (full) {
#pragma unroll
          for (int c = 0; c < 32; ++c) mx = fmaxf(mx, fmaxf(__uint_as_float(a[c]), __uint_as_float(b[c])));
        } else {
          const int lo = (int)imax64(imin64((cs ? clo : nlo) - key0, BN + 1), -1);
          const int hi = (int)imax64(imin64((cs ? chi : nhi) - key0, BN + 1), -1);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c < lo || c >= hi) a[c] = __float_as_uint(-INFINITY);
            if (c + 32 < lo || c + 32 >= hi) b[c] = __float_as_uint(-INFINITY);
            mx = fmaxf(mx, fmaxf(__uint_as_float(a[c]), __uint_as_float(b[c])));
          }
        }
        const float mx2 = mx * sl2;
        bool rescale = false;
        float alpha = 1.f, m_use = m_ref;
        if (m_ref == -INFINITY) {
          m_use = mx2;  // first visible keys of this row (O holds zeros so far)
        } else if (mx2 > m_ref + kRescaleThreshold) {
          m_use = mx2;
          alpha = ex2_approx(m_ref - m_use);
          rescale = true;
        }
        const float nm = (m_use == -INFINITY) ? 0.f : -m_use;
        // P = exp2(s c - m) (masked entries are -inf -> 0), row sum, and P as
        // packed bf16 over the first 32 columns of this S buffer
        float rs0 = 0.f, rs1 = 0.f;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(a[c]), sl2, nm));
          const float p1 = ex2_approx(fmaf(__uint_as_float(a[c + 1]), sl2, nm));
          const float q0 = ex2_approx(fmaf(__uint_as_float(b[c]), sl2, nm));
          const float q1 = ex2_approx(fmaf(__uint_as_float(b[c + 1]), sl2, nm));
          rs0 += p0 + p1;
          rs1 += q0 + q1;
          pk[c / 2] = pack_bf16x2(p0, p1);
          pk[16 + c / 2] = pack_bf16x2(q0, q1);
        }
        tmem_st32(tS, pk);
        l = l * alpha + (rs0 + rs1);
        m_ref = m_use;
        if (j > 0) {
          // PV(j-1) must be complete before O is rescaled
          ok = mbar_wait(BAR(B_PVD, t), (sc - 1) & 1, wd, 10);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int c4 = 0; c4 < HD / 32; ++c4) {
              uint32_t o[32];
              tmem_ld32(tO + c4 * 32, o);
#pragma unroll
              for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
              tmem_st32(tO + c4 * 32, o);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(BAR(B_PF, t));
      }
      if (!ok) break;
      ok = mbar_wait(BAR(B_PVD, t), (sc - 1) & 1, wd, 11);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c4 = 0; c4 < HD / 64; ++c4) {
        uint32_t a[32], b[32];
        tmem_ld32x2(tO + c4 * 64, tO + c4 * 64 + 32, a, b);
        if (valid) {
          if (p.o_f32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(obase) + oofs + c4 * 64);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              o[c] = make_float4(__uint_as_float(a[4 * c]) * inv, __uint_as_float(a[4 * c + 1]) * inv,
                                 __uint_as_float(a[4 * c + 2]) * inv, __uint_as_float(a[4 * c + 3]) * inv);
              o[8 + c] = make_float4(__uint_as_float(b[4 * c]) * inv, __uint_as_float(b[4 * c + 1]) * inv,
                                     __uint_as_float(b[4 * c + 2]) * inv, __uint_as_float(b[4 * c + 3]) * inv);
            }
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(obase) + oofs + c4 * 64);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              o[c] = make_uint4(pack_bf16x2(__uint_as_float(a[8 * c + 0]) * inv, __uint_as_float(a[8 * c + 1]) * inv),
                                pack_bf16x2(__uint_as_float(a[8 * c + 2]) * inv, __uint_as_float(a[8 * c + 3]) * inv),
                                pack_bf16x2(__uint_as_float(a[8 * c + 4]) * inv, __uint_as_float(a[8 * c + 5]) * inv),
                                pack_bf16x2(__uint_as_float(a[8 * c + 6]) * inv, __uint_as_float(a[8 * c + 7]) * inv));
              o[4 + c] =
                  make_uint4(pack_bf16x2(__uint_as_float(b[8 * c + 0]) * inv, __uint_as_float(b[8 * c + 1]) * inv),
                             pack_bf16x2(__uint_as_float(b[8 * c + 2]) * inv, __uint_as_float(b[8 * c + 3]) * inv),
                             pack_bf16x2(__uint_as_float(b[8 * c + 4]) * inv, __uint_as_float(b[8 * c + 5]) * inv),
                             pack_bf16x2(__uint_as_float(b[8 * c + 6]) * inv, __uint_as_float(b[8 * c + 7]) * inv));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(B_OE, t));
      if (valid) lse_out[r] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
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

cudaError_t launch_fwd(const FwdMaps& maps, const FwdParams& p, int d, int num_sms, cudaStream_t stream,
                       int* launches) {
  const int64_t n_pairs = p.n_items / 2;
  const int64_t grid64 = n_pairs < num_sms ? n_pairs : num_sms;
  const int grid = (int)(grid64 > 0 ? grid64 : 1);
  cudaError_t e;
  if (d == 128) {
    e = cudaFuncSetAttribute(bdlm_fwd_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Layout<128>::kAlloc);
    if (e != cudaSuccess) return e;
    bdlm_fwd_tc_kernel<128><<<grid, kThreads, Layout<128>::kAlloc, stream>>>(maps.Qc, maps.Qn, maps.Kc, maps.Kn,
                                                                          maps.Vc, maps.Vn, p);
  } else {
    e = cudaFuncSetAttribute(bdlm_fwd_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Layout<64>::kAlloc);
    if (e != cudaSuccess) return e;
    bdlm_fwd_tc_kernel<64><<<grid, kThreads, Layout<64>::kAlloc, stream>>>(maps.Qc, maps.Qn, maps.Kc, maps.Kn,
                                                                        maps.Vc, maps.Vn, p);
  }
  if (launches) ++*launches;
  return cudaGetLastError();
}

}  // namespace bdlm
