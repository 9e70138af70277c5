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
// Design (one CTA per SM, persistent; 12 warps in three warpgroups).  An
// item is 256 consecutive query rows of one stream and head, split into two
// 128-row sub-tiles that share every key tile (rows of one block see the
// same keys), so each 128-key K/V tile is loaded once for both:
//   warp 0      TMA producer: Q of both sub-tiles, then K and V tiles through
//               two 2-stage rings;
//   warp 1      owns TMEM (512 columns: S of sub-tile t at 128 t, O of
//               sub-tile t at 256 + 128 t); one lane issues tcgen05.mma in the
//               order S0(j), S1(j), PV0(j), S0(j+1), PV1(j), S1(j+1), ... so
//               the tensor pipe works on one sub-tile while the other one's
//               softmax runs;
//   warps 2-3   no role: they complete the first warpgroup, which gives its
//               registers to the softmax warpgroups (setmaxnreg), so that a
//               softmax thread holds its row's 128 scores without spilling;
//   warps 4-7   softmax of sub-tile 0, warps 8-11 of sub-tile 1: one query row
//               per thread, online softmax in the log2 domain with a lazy
//               rescale (the reference max moves only when the row max grows
//               by more than 8), P written back over S in TMEM as packed bf16
//               and read from there by the PV MMA (A operand in TMEM).  The S
//               MMA that next overwrites a sub-tile's S is issued after the PV
//               MMA that reads its P (the tensor pipe runs in issue order), and
//               its completion implies that PV's, so the softmax may rescale O
//               right after S lands.
// Every MMA is M = 128, N = 128 (N = d for PV).  Only key tiles some row of
// the item can see are visited; a per-row interval test masks the tiles that
// are not fully visible.
//
// A separate instantiation (FIXREF) serves verification: each row takes a
// fixed reference M_ref from the caller in place of its running maximum, so
// P = exp(scale q.k - M_ref) needs no rescaling and is rounded to bf16 the
// same way in every call that sees the same key tile for that row (the
// sharded and unsharded paths then differ only by fp32 summation order).
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace bdlm {
namespace {

constexpr int BM = kFwdTileQ;      // query rows per sub-tile (128)
constexpr int BI = kFwdItemRows;   // query rows per item (256)
constexpr int BN = kFwdTileK;      // keys per step (128)
constexpr int kThreads = 384;      // three warpgroups (see the register split below)
// Register split: the block launches with kThreads x kLaunchRegs registers
// (the kernel's register count under __launch_bounds__(kThreads, 1)); the
// first warpgroup (TMA producer, MMA issuer, two idle warps) keeps
// kRegsControl per thread and gives the rest to the two softmax warpgroups.
constexpr int kLaunchRegs = 168;
constexpr int kRegsControl = 104, kRegsSoftmax = 200;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * kLaunchRegs, "register split exceeds the block");
constexpr int kPanel = 128 * 128;  // 128 rows x 128 bytes (64 bf16)
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum { B_QF = 0, B_QE = 1, B_KF = 2, B_KE = 4, B_VF = 6, B_VE = 8, B_SF = 10, B_PF = 12, B_OD = 14, B_OE = 16,
       B_IF = 18, B_IE = 18 + kRingSlots, B_COUNT = 18 + 2 * kRingSlots };
// The 256 bytes after the tiles: barriers, the TMEM address, the abort flag,
// the work-item ring's slots.
static_assert(8 * B_COUNT + 8 + 8 * kRingSlots <= 256, "barrier area overflows");

constexpr int kGeoBytes = 512;  // kRingSlots ItemGeo

template <int HD>
struct Layout {
  static constexpr int kTile = 128 * HD * 2;  // 128 rows x HD bf16 (Q sub-tile, K, V alike)
  static constexpr int kQ = 0;                // Q of sub-tiles 0, 1
  static constexpr int kK = 2 * kTile;        // K stages 0, 1
  static constexpr int kV = 4 * kTile;        // V stages 0, 1
  static constexpr int kBar = 6 * kTile;
  static constexpr int kGeo = kBar + 256;  // the work-item ring's geometry slots
  static constexpr int kBytes = kGeo + kGeoBytes;
  // 1024 bytes of slack for alignment; never below 120 KB so that a second
  // CTA cannot share the SM (each CTA holds all 512 TMEM columns).
  static constexpr int kAlloc = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
};

struct ItemGeo {
  int stream, head, kvh;
  int64_t r0;
  QTileRanges q;
  int nc, n;  // clean key tiles, all key tiles
  int rot;    // the clean-key sweep starts at clean tile c0 + rot
  int64_t off, L;  // first row of the item's sequence in the packed tensors, its length
};
static_assert(kRingSlots * sizeof(ItemGeo) <= kGeoBytes, "geometry slots overflow");

// VL: packed variable-length batch (a separate instantiation, so that the
// one-sequence kernel keeps its register budget).
template <bool VL, bool ROWS = false>
__device__ __forceinline__ ItemGeo item_geo(const FwdParams& p, const VarlenTabs& vt, const RowRange& rows,
                                            int64_t idx) {
  ItemGeo t;
  Geom gs;  // the item's sequence (packed batch only)
  int64_t qtile;
  t.off = 0;
  if (VL) {  // packed batch: the item and its sequence from the tables
    const int4 e = vt.q_items[idx];
    t.stream = e.y & 1;
    t.head = e.y >> 1;
    qtile = e.z;
    t.off = vt.seq_off[e.x];
    gs = seq_geom(p.g, vt.seq_off[e.x + 1] - t.off);
  } else {
    const QItem it = ROWS ? q_item_rows(p.g, rows, BI, idx) : q_item(p.g, BI, idx);
    t.stream = it.stream;
    t.head = it.head;
    qtile = it.qtile;
  }
  const Geom& g = VL ? gs : p.g;
  t.L = g.L;
  t.kvh = t.head / (p.g.Hq / p.g.Hkv);
  t.r0 = qtile * BI;
  const int64_t r1 = imin64(t.r0 + BI, g.L);
  t.q = qtile_ranges(g, t.stream, t.r0, r1, BN);
  t.nc = (int)(t.q.c1 - t.q.c0);
  t.n = t.nc + (int)(t.q.n1 - t.q.n0);
  if (ROWS && !tile_in(rows, t.stream, t.r0, r1)) t.nc = t.n = 0;  // none of the call's rows (not listed)
  t.rot = sweep_rotation(idx, t.nc);
  return t;
}

// The geometry the item's rows are masked with (its sequence's, in a batch).
template <bool VL>
__device__ __forceinline__ Geom item_mask_geom(const FwdParams& p, const ItemGeo& t) {
  return VL ? seq_geom(p.g, t.L) : p.g;
}

// First key of step j: the clean tiles from c0 + rot round to c0 + rot - 1,
// then the corrupted tiles (the online softmax is order-independent).
__device__ __forceinline__ int clean_step(int j, int rot, int nc) {
  const int x = j + rot;
  return x < nc ? x : x - nc;
}
__device__ __forceinline__ int64_t tile_key0(const ItemGeo& t, int j) {
  return (j < t.nc ? t.q.c0 + clean_step(j, t.rot, t.nc) : t.q.n0 + (j - t.nc)) * BN;
}

// P is stored as packed bf16 over the S columns it replaces: keys [64, 128)
// (held in registers since the row-max pass) at columns [64, 96), keys
// [0, 64) (loaded again) at columns [0, 32).  The 16 keys of PV K-step kk
// start at column
__device__ __forceinline__ uint32_t p_col(int kk) { return (uint32_t)(kk * 8 + (kk >= 4 ? 32 : 0)); }

// max of 64 scores: a tree of 3-input maxima (32 instructions)
__device__ __forceinline__ float max64(const uint32_t (&a)[32], const uint32_t (&b)[32]) {
  float u[16];
#pragma unroll
  for (int c = 0; c < 16; ++c)
    u[c] = fmax3(__uint_as_float(a[2 * c]), __uint_as_float(a[2 * c + 1]), __uint_as_float(b[c]));
#pragma unroll
  for (int c = 0; c < 8; ++c) u[c] = fmax3(u[2 * c], u[2 * c + 1], __uint_as_float(b[16 + c]));
#pragma unroll
  for (int c = 0; c < 4; ++c) u[c] = fmax3(u[2 * c], u[2 * c + 1], __uint_as_float(b[24 + c]));
#pragma unroll
  for (int c = 0; c < 2; ++c) u[c] = fmax3(u[2 * c], u[2 * c + 1], __uint_as_float(b[28 + c]));
  return fmax3(u[0], u[1], fmaxf(__uint_as_float(b[30]), __uint_as_float(b[31])));
}

// Scores outside [lo, hi) (key offsets within the step) become -inf.
__device__ __forceinline__ void mask64(uint32_t (&a)[32], uint32_t (&b)[32], int off, int lo, int hi) {
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    if (off + c < lo || off + c >= hi) a[c] = __float_as_uint(-INFINITY);
    if (off + 32 + c < lo || off + 32 + c >= hi) b[c] = __float_as_uint(-INFINITY);
  }
}

// P = exp2(s sl2 - m) of 32 scores (masked -inf -> 0), stored as 16 packed
// bf16 columns at taddr; returns the partial row sums of even and odd keys.
// The fma runs on packed fp32 pairs (half the issue slots of scalar code).
__device__ __forceinline__ uint64_t exp_store32(const uint32_t (&a)[32], uint64_t sl2x2, uint64_t nm2,
                                                uint32_t taddr) {
  uint32_t pk[16];
  float r0 = 0.f, r1 = 0.f;
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    float x0, x1;
    f2_split(f2_fma(f2(__uint_as_float(a[c]), __uint_as_float(a[c + 1])), sl2x2, nm2), x0, x1);
    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    r0 += p0; r1 += p1;
    pk[c / 2] = pack_bf16x2(p0, p1);
  }
  tmem_st16(taddr, pk);
  return f2(r0, r1);
}
// The same for 64 scores (two 32-key halves).
__device__ __forceinline__ uint64_t exp_store64(const uint32_t (&a)[32], const uint32_t (&b)[32], uint64_t sl2x2,
                                                uint64_t nm2, uint32_t taddr) {
  const uint64_t r = exp_store32(a, sl2x2, nm2, taddr);
  return f2_add(r, exp_store32(b, sl2x2, nm2, taddr + 16));
}

template <int HD, bool VL, bool FIXREF, bool ROWS>
__global__ void __launch_bounds__(kThreads, 1)
    bdlm_fwd_tc_kernel(const __grid_constant__ CUtensorMap tQc, const __grid_constant__ CUtensorMap tQn,
                       const __grid_constant__ CUtensorMap tKc, const __grid_constant__ CUtensorMap tKn,
                       const __grid_constant__ CUtensorMap tVc, const __grid_constant__ CUtensorMap tVn,
                       const FwdParams p, const VarlenTabs vt, const FwdRef ref, const RowRange rows) {
  using LY = Layout<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  const uint32_t sQ = base + LY::kQ, sK = base + LY::kK, sV = base + LY::kV;
  const uint32_t bars = base + LY::kBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + LY::kBar + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + LY::kBar + 8 * B_COUNT + 4);
  auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  const ItemRing ring{BAR(B_IF), BAR(B_IE),
                      reinterpret_cast<volatile int64_t*>(base_ptr + LY::kBar + 8 * B_COUNT + 8)};
  // each ring slot also carries its item's geometry, computed once by the
  // producer; the softmax warps keep their slot until the item's epilogue
  ItemGeo* geo_slot = reinterpret_cast<ItemGeo*>(base_ptr + LY::kGeo);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(BAR(B_QF), 1);
    mbar_init(BAR(B_QE), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(BAR(B_KF + s), 1);
      mbar_init(BAR(B_KE + s), 1);
      mbar_init(BAR(B_VF + s), 1);
      mbar_init(BAR(B_VE + s), 1);
      mbar_init(BAR(B_SF + s), 1);
      mbar_init(BAR(B_PF + s), 128);
      mbar_init(BAR(B_OD + s), 1);
      mbar_init(BAR(B_OE + s), 128);
    }
    for (int s = 0; s < kRingSlots; ++s) {
      mbar_init(BAR(B_IF + s), 1);
      mbar_init(BAR(B_IE + s), 1 + 256);  // the MMA thread and every softmax thread
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
  const int64_t n_items = p.n_items;

  // (each role sets its warpgroup's register budget first, inside its own
  // branch, so that every role's code is compiled with its own budget)
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    setmaxnreg_dec<kRegsControl>();
    if (lane == 0) {
      tma_prefetch_desc(&tQc); tma_prefetch_desc(&tQn); tma_prefetch_desc(&tKc);
      tma_prefetch_desc(&tKn); tma_prefetch_desc(&tVc); tma_prefetch_desc(&tVn);
      uint32_t itn = 0, kc = 0;
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        const int64_t idx = claim_item(p.g, p.status + kSchedWordFwd, rnd, cta, grid);
        if (!ring_acquire(ring, rnd, wd, 90)) { ok = false; break; }
        ItemGeo g;
        if (idx < n_items) {
          g = item_geo<VL, ROWS>(p, vt, rows, idx);
          geo_slot[rnd & (kRingSlots - 1)] = g;
        }
        ring_publish(ring, rnd, idx);
        if (idx >= n_items) break;
        if (g.n == 0) continue;
        if (itn > 0 && !mbar_wait(BAR(B_QE), (itn - 1) & 1, wd, 1)) { ok = false; break; }
        mbar_arrive_expect_tx(BAR(B_QF), 2 * LY::kTile);
        const CUtensorMap* mq = g.stream ? &tQn : &tQc;
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int pn = 0; pn < HD / 64; ++pn)
            tma_load_3d(sQ + t * LY::kTile + pn * kPanel, mq, BAR(B_QF), pn * 64, g.head,
                        (int)(g.off + (ROWS ? local_row(rows, g.stream, g.r0 + t * BM) : g.r0 + t * BM)));
        ++itn;
        for (int j = 0; j < g.n; ++j, ++kc) {
          const int st = kc & 1;
          const bool cs = j < g.nc;
          // packed-tensor row, or the key's index in a row-restricted call's K / V
          const int key0 = (int)(g.off + (ROWS ? local_key(rows, cs ? 0 : 1, tile_key0(g, j)) : tile_key0(g, j)));
          if (kc >= 2 && !mbar_wait(BAR(B_KE + st), ((kc >> 1) - 1) & 1, wd, 2)) { ok = false; break; }
          mbar_arrive_expect_tx(BAR(B_KF + st), LY::kTile);
#pragma unroll
          for (int pn = 0; pn < HD / 64; ++pn)
            tma_load_3d(sK + st * LY::kTile + pn * kPanel, cs ? &tKc : &tKn, BAR(B_KF + st), pn * 64, g.kvh, key0);
          if (kc >= 2 && !mbar_wait(BAR(B_VE + st), ((kc >> 1) - 1) & 1, wd, 3)) { ok = false; break; }
          mbar_arrive_expect_tx(BAR(B_VF + st), LY::kTile);
#pragma unroll
          for (int pn = 0; pn < HD / 64; ++pn)
            tma_load_3d(sV + st * LY::kTile + pn * kPanel, cs ? &tVc : &tVn, BAR(B_VF + st), pn * 64, g.kvh, key0);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    setmaxnreg_dec<kRegsControl>();
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(BM, BN, false, false);
      constexpr uint32_t kIdO = idesc_bf16(BM, HD, false, true);
      const uint64_t dq[2] = {sdesc_sw128(sQ, 16, 1024), sdesc_sw128(sQ + LY::kTile, 16, 1024)};
      // S_t(k) = Q_t K(k)^T into the S columns of sub-tile t
      auto issue_s = [&](int t, uint32_t k) {
        const uint64_t dk0 = sdesc_sw128(sK + (k & 1) * LY::kTile, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          tc_mma_ss(tmem + t * 128, desc_add(dq[t], off), desc_add(dk0, off), kIdS, kk > 0 ? 1u : 0u);
        }
        tc_commit(BAR(B_SF + t));
      };
      // O_t += P_t(k) V(k), P_t packed bf16 over the S columns
      auto issue_pv = [&](int t, uint32_t k, bool first) {
        const uint64_t dv0 = sdesc_sw128(sV + (k & 1) * LY::kTile, kPanel, 1024);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          tc_mma_ts(tmem + 256 + t * 128, tmem + t * 128 + p_col(kk), desc_add(dv0, kk * 2048), kIdO,
                    (kk > 0 || !first) ? 1u : 0u);
      };
      uint32_t itn = 0, kc = 0;
      bool ok = true;
      for (int64_t rnd = 0; ok; ++rnd) {
        int64_t idx;
        if (!ring_wait(ring, rnd, idx, wd, 91)) { ok = false; break; }
        if (idx >= n_items) break;
        const ItemGeo g = geo_slot[rnd & (kRingSlots - 1)];
        ring_release(ring, rnd);
        if (g.n == 0) continue;
        if (!mbar_wait(BAR(B_QF), itn & 1, wd, 4)) { ok = false; break; }
        if (!mbar_wait(BAR(B_KF + (kc & 1)), (kc >> 1) & 1, wd, 5)) { ok = false; break; }
        tc_fence_after();
        issue_s(0, kc);
        issue_s(1, kc);
        tc_commit(BAR(B_KE + (kc & 1)));
        if (g.n == 1) tc_commit(BAR(B_QE));
        for (int j = 0; j < g.n; ++j) {
          const uint32_t k = kc + j;
          const bool last = j == g.n - 1;
          // PV0(j), then S0(j+1) over P0(j)
          if (!mbar_wait(BAR(B_PF + 0), k & 1, wd, 6)) { ok = false; break; }
          if (j == 0 && itn > 0 && !mbar_wait(BAR(B_OE + 0), (itn - 1) & 1, wd, 7)) { ok = false; break; }
          if (!mbar_wait(BAR(B_VF + (k & 1)), (k >> 1) & 1, wd, 8)) { ok = false; break; }
          tc_fence_after();
          issue_pv(0, k, j == 0);
          if (last) tc_commit(BAR(B_OD + 0));
          if (!last) {
            if (!mbar_wait(BAR(B_KF + ((k + 1) & 1)), ((k + 1) >> 1) & 1, wd, 9)) { ok = false; break; }
            tc_fence_after();
            issue_s(0, k + 1);
          }
          // PV1(j), then S1(j+1) over P1(j)
          if (!mbar_wait(BAR(B_PF + 1), k & 1, wd, 10)) { ok = false; break; }
          if (j == 0 && itn > 0 && !mbar_wait(BAR(B_OE + 1), (itn - 1) & 1, wd, 11)) { ok = false; break; }
          tc_fence_after();
          issue_pv(1, k, j == 0);
          tc_commit(BAR(B_VE + (k & 1)));
          if (last) tc_commit(BAR(B_OD + 1));
          if (!last) {
            issue_s(1, k + 1);
            tc_commit(BAR(B_KE + ((k + 1) & 1)));
            if (j + 1 == g.n - 1) tc_commit(BAR(B_QE));
          }
        }
        kc += g.n;
        ++itn;
      }
    }
  } else if (warp < 4) {
    setmaxnreg_dec<kRegsControl>();  // warps 2 and 3: no role
  } else {
    // ------------------------------------------------------------ softmax (thread = row of sub-tile t)
    setmaxnreg_inc<kRegsSoftmax>();
    const int t = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t tl = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + tl + t * 128, tO = tmem + tl + 256 + t * 128;
    uint32_t sc = 0, itn = 0;
    bool ok = true;
    for (int64_t rnd = 0; ok; ++rnd) {
      int64_t idx;
      if (!ring_wait(ring, rnd, idx, wd, 92)) { ok = false; break; }
      if (idx >= n_items) break;
      const ItemGeo g = geo_slot[rnd & (kRingSlots - 1)];  // the slot stays ours until the epilogue
      // (one sequence: its length and offset come from the parameters, so
      // that they occupy no registers across the loop)
      const int64_t seqL = VL ? g.L : p.g.L, seq0 = VL ? g.off : 0;
      const int64_t r = g.r0 + t * BM + row;  // row within the item's sequence
      const bool valid = r < seqL;
      // the row's index in its stream's O and LSE (the packed row in a batch,
      // the local row in a row-restricted call) and the LSE row stride
      const int64_t lrow = VL ? seq0 + r : (ROWS ? local_row(rows, g.stream, r) : r);
      const int64_t lstride = ROWS ? held_rows(rows, g.stream) : p.g.L;
      float* lse_out = (g.stream ? p.LSEn : p.LSEc) + (int64_t)g.head * lstride;
      void* obase = g.stream ? p.On : p.Oc;
      const int64_t oofs = (lrow * p.g.Hq + g.head) * HD;
      if (g.n == 0) {
        if (valid && (!ROWS || row_in(rows, g.stream, r))) {
          if (p.o_f32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(obase) + oofs);
#pragma unroll
            for (int c = 0; c < HD / 4; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(obase) + oofs);
#pragma unroll
            for (int c = 0; c < HD / 8; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
          }
          lse_out[lrow] = -INFINITY;
        }
        ring_release(ring, rnd);
        continue;
      }
      // loop state in 32-bit (rows and keys are TMA coordinates, < 2^31):
      // key tile ranges, keys every row of the item sees (clipped to L), and
      // this row's visible key intervals
      int lo_c, hi_c, lo_n, hi_n;
      {
        const int64_t rr = valid ? r : seqL - 1;
        const Geom gm = item_mask_geom<VL>(p, g);
        int64_t a0, a1, b0, b1;
        clean_interval(gm, g.stream, rr, a0, a1);
        noisy_interval(gm, g.stream, rr, b0, b1);
        lo_c = (int)a0; hi_c = (int)a1; lo_n = (int)b0; hi_n = (int)b1;
      }
      const int nc = g.nc, n = g.n, c0 = (int)g.q.c0, n0 = (int)g.q.n0, rot = g.rot;
      const int call_lo = (int)g.q.c_all_lo, call_hi = (int)imin64(g.q.c_all_hi, seqL);
      const int nall_lo = (int)g.q.n_all_lo, nall_hi = (int)imin64(g.q.n_all_hi, seqL);
      const float sl2 = p.scale_log2;
      float m_ref = -INFINITY, l = 0.f;
      if (FIXREF) {
        // the caller's reference, natural log -> the kernel's log2 units
        const float* rp = g.stream ? ref.n : ref.c;
        const float mr = valid ? rp[(int64_t)g.head * p.g.L + r] * kLog2e : 0.f;
        m_ref = fabsf(mr) < INFINITY ? mr : 0.f;
      }
      for (int j = 0; j < n; ++j, ++sc) {
        const bool cs = j < nc;
        const int key0 = (cs ? c0 + clean_step(j, rot, nc) : n0 + (j - nc)) * BN;
        const bool full = cs ? (key0 >= call_lo && key0 + BN <= call_hi) : (key0 >= nall_lo && key0 + BN <= nall_hi);
        ok = mbar_wait(BAR(B_SF + t), sc & 1, wd, 12);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // pass 1, the row max; S of keys [64, 128) stays in registers
        int lo = -1, hi = BN + 1;
        if (!full) {
          lo = max(min((cs ? lo_c : lo_n) - key0, BN + 1), -1);
          hi = max(min((cs ? hi_c : hi_n) - key0, BN + 1), -1);
        }
        uint32_t a0[32], a1[32], h0[32], h1[32];
        tmem_ld32x4(tS, tS + 32, tS + 64, tS + 96, a0, a1, h0, h1);  // the row's 128 scores, one wait
        if (!full) {
          mask64(a0, a1, 0, lo, hi);
          mask64(h0, h1, 64, lo, hi);
        }
        const float mx = fmaxf(max64(a0, a1), max64(h0, h1));
        const float mx2 = mx * sl2;
        bool rescale = false;
        float alpha = 1.f, m_use = m_ref;
        if (FIXREF) {
          // fixed reference: no rescaling
        } else if (m_ref == -INFINITY) {
          m_use = mx2;  // first visible keys of this row (O holds zeros so far)
        } else if (mx2 > m_ref + kRescaleThreshold) {
          m_use = mx2;
          alpha = ex2_approx(m_ref - m_use);
          rescale = true;
        }
        const float nm = (m_use == -INFINITY) ? 0.f : -m_use;
        // P and its row sum: keys [64, 128) from registers, then keys [0, 64)
        // loaded again (layout of p_col)
        const uint64_t sl2x2 = f2(sl2, sl2), nm2 = f2(nm, nm);
        uint64_t rs = exp_store64(h0, h1, sl2x2, nm2, tS + 64);
        rs = f2_add(rs, exp_store64(a0, a1, sl2x2, nm2, tS));  // keys [0, 64), masked in pass 1
        float r0, r1;
        f2_split(rs, r0, r1);
        l = l * alpha + (r0 + r1);
        m_ref = m_use;
        // O is complete up to step j-1 (S_t(j) was issued after PV_t(j-1))
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
        tc_fence_before();
        mbar_arrive(BAR(B_PF + t));
      }
      if (!ok) break;
      ok = mbar_wait(BAR(B_OD + t), itn & 1, wd, 13);
      const ItemGeo ge = geo_slot[rnd & (kRingSlots - 1)];
      const int64_t seqL_e = VL ? ge.L : p.g.L, seq0_e = VL ? ge.off : 0;
      const int64_t re = ge.r0 + t * BM + row;
      const bool ve = re < seqL_e && (!ROWS || row_in(rows, ge.stream, re));
      const int64_t lrow_e = VL ? seq0_e + re : (ROWS ? local_row(rows, ge.stream, re) : re);
      const int64_t lstride_e = ROWS ? held_rows(rows, ge.stream) : p.g.L;
      float* lse_e = (ge.stream ? p.LSEn : p.LSEc) + (int64_t)ge.head * lstride_e;
      void* obase_e = ge.stream ? p.On : p.Oc;
      const int64_t oofs_e = (lrow_e * p.g.Hq + ge.head) * HD;
      ring_release(ring, rnd);  // the item's geometry is in registers now
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c4 = 0; c4 < HD / 64; ++c4) {
        uint32_t a[32], b[32];
        tmem_ld32x2(tO + c4 * 64, tO + c4 * 64 + 32, a, b);
        if (ve) {
          if (p.o_f32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(obase_e) + oofs_e + c4 * 64);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              o[c] = make_float4(__uint_as_float(a[4 * c]) * inv, __uint_as_float(a[4 * c + 1]) * inv,
                                 __uint_as_float(a[4 * c + 2]) * inv, __uint_as_float(a[4 * c + 3]) * inv);
              o[8 + c] = make_float4(__uint_as_float(b[4 * c]) * inv, __uint_as_float(b[4 * c + 1]) * inv,
                                     __uint_as_float(b[4 * c + 2]) * inv, __uint_as_float(b[4 * c + 3]) * inv);
            }
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(obase_e) + oofs_e + c4 * 64);
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
      mbar_arrive(BAR(B_OE + t));
      if (ve) lse_e[lrow_e] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      ++itn;
    }
  }

  __syncthreads();
  if (threadIdx.x == 0) sched_release(p.status + kSchedWordFwd, grid);
  if (*abort_flag) drain_after_abort(200);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int HD, bool VL, bool FIXREF, bool ROWS = false>
cudaError_t launch_fwd_t(const FwdMaps& maps, const FwdParams& p, const VarlenTabs& vt, const FwdRef& ref,
                         const RowRange& rows, int grid, cudaStream_t stream) {
  auto k = bdlm_fwd_tc_kernel<HD, VL, FIXREF, ROWS>;
  // the register split needs the block's full allotment: refuse to launch otherwise
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, k);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * kThreads < 128 * kRegsControl + 256 * kRegsSoftmax) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<HD>::kAlloc);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, Layout<HD>::kAlloc, stream>>>(maps.Qc, maps.Qn, maps.Kc, maps.Kn, maps.Vc, maps.Vn, p, vt,
                                                    ref, rows);
  return cudaSuccess;
}

cudaError_t launch_fwd(const FwdMaps& maps, const FwdParams& p, const VarlenTabs* vt, const FwdRef* ref,
                       const RowRange* rows, int d, int num_sms, cudaStream_t stream, int* launches) {
  const int64_t grid64 = p.n_items < num_sms ? p.n_items : num_sms;
  const int grid = (int)(grid64 > 0 ? grid64 : 1);
  const VarlenTabs none{nullptr, nullptr, nullptr, 0, 0};
  const VarlenTabs& t = vt ? *vt : none;
  const FwdRef noref{nullptr, nullptr};
  const RowRange all;
  cudaError_t e;
  if (ref) {  // verification mode: one sequence only, all rows
    if (vt || rows) return cudaErrorInvalidValue;
    e = d == 128 ? launch_fwd_t<128, false, true>(maps, p, t, *ref, all, grid, stream)
                 : launch_fwd_t<64, false, true>(maps, p, t, *ref, all, grid, stream);
  } else if (rows) {  // one rank's rows: one sequence only
    if (vt) return cudaErrorInvalidValue;
    e = d == 128 ? launch_fwd_t<128, false, false, true>(maps, p, t, noref, *rows, grid, stream)
                 : launch_fwd_t<64, false, false, true>(maps, p, t, noref, *rows, grid, stream);
  } else {
    e = d == 128 ? (vt ? launch_fwd_t<128, true, false>(maps, p, t, noref, all, grid, stream)
                       : launch_fwd_t<128, false, false>(maps, p, t, noref, all, grid, stream))
                 : (vt ? launch_fwd_t<64, true, false>(maps, p, t, noref, all, grid, stream)
                       : launch_fwd_t<64, false, false>(maps, p, t, noref, all, grid, stream));
  }
  if (e != cudaSuccess) return e;
  if (launches) ++*launches;
  return cudaGetLastError();
}

}  // namespace bdlm
