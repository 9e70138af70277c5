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
// Design (one CTA per SM, persistent; 6 warps):
//   warp 0      TMA producer: Q tile once per item, K and V tiles into a
//               two-stage ring (128-byte swizzle, 64-column panels).
//   warp 1      owns TMEM (512 columns); one lane issues tcgen05.mma:
//               S = Q K^T into one of two TMEM S buffers, O += P V into TMEM.
//   warps 2-5   softmax warpgroup, one query row per thread (TMEM lane):
//               online softmax in the log2 domain with a lazy rescale (the
//               running reference max only moves when the row max grows by
//               more than 8, so O rarely needs a TMEM round trip), writes P as
//               bf16 into a swizzled shared-memory tile, and runs the
//               epilogue (O / l, LSE).
// Only key tiles some row of the query tile can see are visited; a per-row
// interval test masks the tiles that are not fully visible.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

constexpr int BM = kFwdTileQ;   // query rows per tile
constexpr int BN = kFwdTileK;   // keys per tile
constexpr int NS = 2;           // K/V pipeline stages
constexpr int kThreads = 192;
constexpr int kPanelBytes = 128 * 128;  // 128 rows x 128 bytes (64 bf16)
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// barrier slots
enum { B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_VFULL = 4, B_KVEMPTY = 6, B_SFULL = 8, B_SEMPTY = 10,
       B_PFULL = 12, B_PVDONE = 13, B_OEMPTY = 14, B_COUNT = 15 };

template <int HD>
struct Layout {
  static constexpr int kTileBytes = 128 * HD * 2;  // 128 rows x HD bf16
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + NS * kTileBytes;
  static constexpr int kP = kV + NS * kTileBytes;
  static constexpr int kBar = kP + BM * BN * 2;
  static constexpr int kBytes = kBar + 256;
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
  const uint32_t sQ = base + LY::kQ, sK = base + LY::kK, sV = base + LY::kV, sP = base + LY::kP;
  const uint32_t bars = base + LY::kBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + LY::kBar + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + LY::kBar + 8 * B_COUNT + 4);
  auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(BAR(B_QFULL), 1);
    mbar_init(BAR(B_QEMPTY), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(BAR(B_KFULL + s), 1);
      mbar_init(BAR(B_VFULL + s), 1);
      mbar_init(BAR(B_KVEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(BAR(B_SFULL + s), 1);
      mbar_init(BAR(B_SEMPTY + s), 128);
    }
    mbar_init(BAR(B_PFULL), 128);
    mbar_init(BAR(B_PVDONE), 1);
    mbar_init(BAR(B_OEMPTY), 128);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tQc); tma_prefetch_desc(&tQn); tma_prefetch_desc(&tKc);
      tma_prefetch_desc(&tKn); tma_prefetch_desc(&tVc); tma_prefetch_desc(&tVn);
      uint32_t itn = 0, kvc = 0;
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        const int64_t idx = snake_item(rnd, cta, grid);
        if (idx >= p.n_items) break;
        const ItemGeo t = item_geo(p, idx);
        if (t.n == 0) continue;
        if (itn > 0 && !mbar_wait(BAR(B_QEMPTY), (itn - 1) & 1, wd, 1)) { ok = false; break; }
        mbar_arrive_expect_tx(BAR(B_QFULL), LY::kTileBytes);
        const CUtensorMap* mq = t.stream ? &tQn : &tQc;
#pragma unroll
        for (int pn = 0; pn < HD / 64; ++pn)
          tma_load_3d(sQ + pn * kPanelBytes, mq, BAR(B_QFULL), pn * 64, t.head, (int)t.r0);
        for (int j = 0; j < t.n; ++j, ++kvc) {
          const int st = kvc % NS;
          if (kvc >= NS && !mbar_wait(BAR(B_KVEMPTY + st), ((kvc / NS) - 1) & 1, wd, 2)) { ok = false; break; }
          const bool cs = j < t.nc;
          const int key0 = (int)tile_key0(t, j);
          const CUtensorMap* mk = cs ? &tKc : &tKn;
          const CUtensorMap* mv = cs ? &tVc : &tVn;
          mbar_arrive_expect_tx(BAR(B_KFULL + st), LY::kTileBytes);
#pragma unroll
          for (int pn = 0; pn < HD / 64; ++pn)
            tma_load_3d(sK + st * LY::kTileBytes + pn * kPanelBytes, mk, BAR(B_KFULL + st), pn * 64, t.kvh, key0);
          mbar_arrive_expect_tx(BAR(B_VFULL + st), LY::kTileBytes);
#pragma unroll
          for (int pn = 0; pn < HD / 64; ++pn)
            tma_load_3d(sV + st * LY::kTileBytes + pn * kPanelBytes, mv, BAR(B_VFULL + st), pn * 64, t.kvh, key0);
        }
        ++itn;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16(BM, BN, false, false);
      constexpr uint32_t kIdescO = idesc_bf16(BM, HD, false, true);
      const uint32_t tS = tmem, tO = tmem + 256;
      uint32_t itn = 0, kvc = 0, sc = 0, pc = 0;
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        const int64_t idx = snake_item(rnd, cta, grid);
        if (idx >= p.n_items) break;
        const ItemGeo t = item_geo(p, idx);
        if (t.n == 0) continue;
        if (!mbar_wait(BAR(B_QFULL), itn & 1, wd, 3)) { ok = false; break; }
        const uint32_t kv_base = kvc;
        auto do_pv = [&](int jj) -> bool {
          const uint32_t kv = kv_base + jj;
          const int st = kv % NS;
          if (!mbar_wait(BAR(B_PFULL), pc & 1, wd, 4)) return false;
          if (jj == 0 && itn > 0 && !mbar_wait(BAR(B_OEMPTY), (itn - 1) & 1, wd, 5)) return false;
          if (!mbar_wait(BAR(B_VFULL + st), (kv / NS) & 1, wd, 6)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(sP + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sV + st * LY::kTileBytes + kk * 2048, kPanelBytes, 1024);
            tc_mma_ss(tO, ad, bd, kIdescO, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(BAR(B_KVEMPTY + st));
          tc_commit(BAR(B_PVDONE));
          ++pc;
          return true;
        };
        for (int j = 0; j < t.n && ok; ++j, ++kvc, ++sc) {
          const int st = kvc % NS;
          const int sb = sc & 1;
          if (!mbar_wait(BAR(B_KFULL + st), (kvc / NS) & 1, wd, 7)) { ok = false; break; }
          if (sc >= 2 && !mbar_wait(BAR(B_SEMPTY + sb), ((sc >> 1) - 1) & 1, wd, 8)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(sQ + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sK + st * LY::kTileBytes + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
            tc_mma_ss(tS + sb * BN, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
          }
          tc_commit(BAR(B_SFULL + sb));
          if (j == t.n - 1) tc_commit(BAR(B_QEMPTY));
          if (j >= 1 && !do_pv(j - 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!do_pv(t.n - 1)) { ok = false; break; }
        ++itn;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t tl = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + tl, tO = tmem + tl + 256;
    uint32_t sc = 0, pc = 0;
    bool ok = true;
    for (int64_t rnd = 0; ok; ++rnd) {
      const int64_t idx = snake_item(rnd, cta, grid);
      if (idx >= p.n_items) break;
      const ItemGeo t = item_geo(p, idx);
      const int64_t r = t.r0 + row;
      const bool valid = r < p.g.L;
      float* lse_out = (t.stream ? p.LSEn : p.LSEc) + (int64_t)t.head * p.g.L;
      void* obase = t.stream ? p.On : p.Oc;
      const int64_t oofs = (r * p.g.Hq + t.head) * HD;
      if (t.n == 0) {
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
      clean_interval(p.g, t.stream, rr, clo, chi);
      noisy_interval(p.g, t.stream, rr, nlo, nhi);
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < t.n; ++j, ++sc) {
        const bool cs = j < t.nc;
        const int64_t key0 = tile_key0(t, j);
        const bool full = cs ? tile_full(key0, BN, t.q.c_all_lo, t.q.c_all_hi, p.g.L)
                             : tile_full(key0, BN, t.q.n_all_lo, t.q.n_all_hi, p.g.L);
        const int sb = sc & 1;
        ok = mbar_wait(BAR(B_SFULL + sb), (sc >> 1) & 1, wd, 9);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float s[BN];
#pragma unroll
        for (int c4 = 0; c4 < BN / 32; ++c4) {
          uint32_t u[32];
          tmem_ld32(tS + sb * BN + c4 * 32, u);
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c4 * 32 + c] = __uint_as_float(u[c]);
        }
        tc_fence_before();
        mbar_arrive(BAR(B_SEMPTY + sb));
        if (!full) {
          const int64_t lo = (cs ? clo : nlo) - key0, hi = (cs ? chi : nhi) - key0;
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c < lo || c >= hi) s[c] = -INFINITY;
        }
        float mx = s[0];
#pragma unroll
        for (int c = 1; c < BN; ++c) mx = fmaxf(mx, s[c]);
        const float mx2 = mx * p.scale_log2;
        bool rescale = false;
        float alpha = 1.f, m_use = m_ref;
        if (m_ref == -INFINITY) {
          m_use = mx2;  // first visible keys of this row (O holds zeros so far)
        } else if (mx2 > m_ref + kRescaleThreshold) {
          m_use = mx2;
          alpha = ex2_approx(m_ref - m_use);
          rescale = true;
        }
        const float msub = (m_use == -INFINITY) ? 0.f : m_use;
        uint32_t pk[BN / 2];
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < BN; c += 2) {
          const float p0 = ex2_approx(fmaf(s[c], p.scale_log2, -msub));
          const float p1 = ex2_approx(fmaf(s[c + 1], p.scale_log2, -msub));
          rs += p0 + p1;
          pk[c / 2] = pack_bf16x2(p0, p1);
        }
        l = l * alpha + rs;
        m_ref = m_use;
        if (j > 0) {
          ok = mbar_wait(BAR(B_PVDONE), (pc - 1) & 1, wd, 10);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int c4 = 0; c4 < HD / 32; ++c4) {
              uint32_t u[32];
              tmem_ld32(tO + c4 * 32, u);
#pragma unroll
              for (int c = 0; c < 32; ++c) u[c] = __float_as_uint(__uint_as_float(u[c]) * alpha);
              tmem_st32(tO + c4 * 32, u);
            }
          }
        }
        // P row -> swizzled K-major tile (two 64-key panels)
#pragma unroll
        for (int ch = 0; ch < BN / 8; ++ch) {
          const int pn = ch >> 3, cw = ch & 7;
          const uint32_t addr = sP + pn * kPanelBytes + row * 128 + ((cw ^ (row & 7)) << 4);
          st_shared_v4(addr, pk[ch * 4 + 0], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(BAR(B_PFULL));
        ++pc;
      }
      if (!ok) break;
      ok = mbar_wait(BAR(B_PVDONE), (pc - 1) & 1, wd, 11);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c4 = 0; c4 < HD / 32; ++c4) {
        uint32_t u[32];
        tmem_ld32(tO + c4 * 32, u);
        if (valid) {
          if (p.o_f32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(obase) + oofs + c4 * 32);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              o[c] = make_float4(__uint_as_float(u[4 * c]) * inv, __uint_as_float(u[4 * c + 1]) * inv,
                                 __uint_as_float(u[4 * c + 2]) * inv, __uint_as_float(u[4 * c + 3]) * inv);
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(obase) + oofs + c4 * 32);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              o[c] = make_uint4(pack_bf16x2(__uint_as_float(u[8 * c + 0]) * inv, __uint_as_float(u[8 * c + 1]) * inv),
                                pack_bf16x2(__uint_as_float(u[8 * c + 2]) * inv, __uint_as_float(u[8 * c + 3]) * inv),
                                pack_bf16x2(__uint_as_float(u[8 * c + 4]) * inv, __uint_as_float(u[8 * c + 5]) * inv),
                                pack_bf16x2(__uint_as_float(u[8 * c + 6]) * inv, __uint_as_float(u[8 * c + 7]) * inv));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(B_OEMPTY));
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
  const int64_t grid64 = p.n_items < num_sms ? p.n_items : num_sms;
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
