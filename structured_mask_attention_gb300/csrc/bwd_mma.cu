// bwd_mma.cu -- two-stream BDLM attention backward, deterministic, on
// warp-level bf16 MMA (mma.sync m16n8k16, fp32 accumulate).
//
// Gradients of softmax attention under the two-stream block mask with no
// gradient through LSE ("Block Parallelism For Efficient Distributed
// Long-Context Diffusion Language Model Training": the training objective's
// gradients, evolve.pub review "Key claims" / Proposition 1; only clean K/V
// gradients cross context shards, evolve.pub FAQ on CSBP):
//   P = exp(scale Q K^T - LSE), dP = dO V^T, dS = P o (dP - D),
//   dV = sum_group P^T dO, dK = scale sum_group dS^T Q, dQ = scale dS K.
// Two passes, each writing every output element exactly once:
//   dK/dV pass: one CTA per (key stream, KV head, 64-key tile); it walks every
//               query row of every head of the GQA group that sees the tile,
//               32 rows at a time, accumulating dK and dV in registers.
//   dQ pass:    one CTA per (query tile of 64 rows, head, stream); it walks the
//               visible key tiles 32 keys at a time.
// Both recompute P from Q, K and the forward LSE.  Blocks are launched in
// longest-first order.  Shared-memory tiles use a 16-byte XOR swizzle so
// ldmatrix reads are free of bank conflicts.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(pred ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Byte offset of element (row, col) in a [rows x HD] bf16 tile whose 16-byte
// chunks are XOR-swizzled by (row & 7).
template <int HD>
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return (uint32_t)(row * (HD * 2) + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1));
}

// rows [r0, r0 + R) of head h of a [L, H, HD] bf16 tensor -> swizzled tile;
// rows outside [0, L) are zero-filled.
template <int HD, int R>
__device__ __forceinline__ void load_tile(uint32_t sbase, const __nv_bfloat16* X, int64_t r0, int64_t L, int H,
                                          int h) {
  constexpr int CH = HD / 8;
  for (int i = threadIdx.x; i < R * CH; i += kThreads) {
    const int row = i / CH, ch = i % CH;
    const int64_t r = r0 + row;
    const bool ok = r >= 0 && r < L;
    const __nv_bfloat16* src = X + ((ok ? r : 0) * H + h) * HD + ch * 8;
    cp_async16(sbase + (uint32_t)(row * HD * 2 + ((ch ^ (row & 7)) << 4)), src, ok);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) { return pack_bf16x2(lo, hi); }

__device__ __forceinline__ void store_pair(void* base, int64_t off, float v0, float v1, int f32, int acc) {
  if (f32) {
    float2* p = reinterpret_cast<float2*>(static_cast<float*>(base) + off);
    if (acc) {
      const float2 o = *p;
      v0 += o.x;
      v1 += o.y;
    }
    *p = make_float2(v0, v1);
  } else {
    *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(base) + off) = pack2(v0, v1);
  }
}

// True when query row i (of `stream`) sees every key of [j0, j0 + n) of key_stream.
__device__ __forceinline__ bool row_sees_all(const Geom& g, int stream, int64_t i, int key_stream, int64_t j0,
                                             int n) {
  int64_t lo, hi;
  if (key_stream == 0) clean_interval(g, stream, i, lo, hi);
  else noisy_interval(g, stream, i, lo, hi);
  return j0 >= lo && j0 + n <= hi;
}

// ----------------------------------------------------------------- dK / dV
template <int HD>
__global__ void __launch_bounds__(kThreads) bdlm_bwd_dkv_kernel(const BwdParams p) {
  constexpr int BK = kDkvTileK, BQ = kDkvTileQ;
  constexpr int TB = HD * 2;  // bytes per tile row
  extern __shared__ __align__(128) uint8_t sm[];
  const uint32_t sK = smem_u32(sm), sV = sK + BK * TB, sQ = sV + BK * TB, sdO = sQ + BQ * TB;
  float* sLse = reinterpret_cast<float*>(sm + 2 * BK * TB + 2 * BQ * TB);
  float* sD = sLse + BQ;

  const Geom& g = p.g;
  const KVItem it = kv_item(g, BK, blockIdx.x);
  const int ks = it.key_stream, kvh = it.kv_head;
  const int64_t j0 = it.ktile * BK, j1 = imin64(j0 + BK, g.L);
  const int64_t klo = ks == 0 ? imax64(j0, g.kv_begin) : j0;
  const int64_t khi = ks == 0 ? imin64(j1, g.kv_end) : j1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  const int G = g.Hq / g.Hkv;

  load_tile<HD, BK>(sK, static_cast<const __nv_bfloat16*>(ks ? p.Kn : p.Kc), j0, g.L, g.Hkv, kvh);
  load_tile<HD, BK>(sV, static_cast<const __nv_bfloat16*>(ks ? p.Vn : p.Vc), j0, g.L, g.Hkv, kvh);

  int64_t c_lo, c_hi, n_lo, n_hi;
  kv_tile_rows(g, ks, j0, j1, c_lo, c_hi, n_lo, n_hi);

  float dk[HD / 8][4], dv[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;

  const int64_t keyA = j0 + 16 * warp + gq;  // this thread's key rows: keyA, keyA + 8

  for (int hh = 0; hh < G; ++hh) {
    const int h = kvh * G + hh;
    for (int s = 0; s < 2; ++s) {
      const int64_t lo = s == 0 ? c_lo : n_lo, hi = s == 0 ? c_hi : n_hi;
      if (hi <= lo) continue;
      const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(s ? p.Qn : p.Qc);
      const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(s ? p.dOn : p.dOc);
      const float* LSE = (s ? p.LSEn : p.LSEc) + (int64_t)h * g.L;
      const float* Dr = (s ? p.Dn : p.Dc) + (int64_t)h * g.L;
      for (int64_t q0 = lo; q0 < hi; q0 += BQ) {
        __syncthreads();
        load_tile<HD, BQ>(sQ, Q, q0, g.L, g.Hq, h);
        load_tile<HD, BQ>(sdO, dO, q0, g.L, g.Hq, h);
        if (threadIdx.x < BQ) {
          const int64_t r = q0 + threadIdx.x;
          const bool ok = r < g.L;
          sLse[threadIdx.x] = ok ? LSE[r] * kLog2e : 0.f;
          sD[threadIdx.x] = ok ? Dr[r] : 0.f;
        }
        cp_async_wait_all();
        __syncthreads();
        const bool full = (q0 + BQ <= g.L) && (j0 + BK <= g.L) && row_sees_all(g, s, q0, ks, j0, BK) &&
                          row_sees_all(g, s, q0 + BQ - 1, ks, j0, BK);

        // S^T = K_w Q^T and dP^T = V_w dO^T, [16 keys x 32 rows] per warp
        float st[4][4], dpt[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) st[i][e] = dpt[i][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          uint32_t ak[4], av[4];
          const int arow = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8, acol = 16 * kk + (lane >> 4) * 8;
          ldsm_x4(sK + swz<HD>(arow, acol), ak);
          ldsm_x4(sV + swz<HD>(arow, acol), av);
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            uint32_t bq[4], bo[4];
            const int brow = 16 * np + (lane & 7) + (lane >> 4) * 8, bcol = 16 * kk + ((lane >> 3) & 1) * 8;
            ldsm_x4(sQ + swz<HD>(brow, bcol), bq);
            ldsm_x4(sdO + swz<HD>(brow, bcol), bo);
            mma16816(st[2 * np], ak, bq[0], bq[1]);
            mma16816(st[2 * np + 1], ak, bq[2], bq[3]);
            mma16816(dpt[2 * np], av, bo[0], bo[1]);
            mma16816(dpt[2 * np + 1], av, bo[2], bo[3]);
          }
        }
        // P^T and dS^T
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int qi = 8 * nt + 2 * tq + (e & 1);
            const int64_t key = keyA + ((e >> 1) << 3);
            bool vis = full;
            if (!vis) vis = (q0 + qi < g.L) && visible(g, s, q0 + qi, ks, key);
            const float pv = vis ? ex2_approx(fmaf(st[nt][e], p.scale_log2, -sLse[qi])) : 0.f;
            st[nt][e] = pv;
            dpt[nt][e] = pv * (dpt[nt][e] - sD[qi]);
          }
        // dV += P^T dO, dK += dS^T Q
#pragma unroll
        for (int kq = 0; kq < 2; ++kq) {
          uint32_t ap[4], as[4];
          ap[0] = pack2(st[2 * kq][0], st[2 * kq][1]);
          ap[1] = pack2(st[2 * kq][2], st[2 * kq][3]);
          ap[2] = pack2(st[2 * kq + 1][0], st[2 * kq + 1][1]);
          ap[3] = pack2(st[2 * kq + 1][2], st[2 * kq + 1][3]);
          as[0] = pack2(dpt[2 * kq][0], dpt[2 * kq][1]);
          as[1] = pack2(dpt[2 * kq][2], dpt[2 * kq][3]);
          as[2] = pack2(dpt[2 * kq + 1][0], dpt[2 * kq + 1][1]);
          as[3] = pack2(dpt[2 * kq + 1][2], dpt[2 * kq + 1][3]);
#pragma unroll
          for (int dn = 0; dn < HD / 16; ++dn) {
            uint32_t bo[4], bq[4];
            const int brow = 16 * kq + (lane & 7) + ((lane >> 3) & 1) * 8, bcol = 16 * dn + (lane >> 4) * 8;
            ldsm_x4_t(sdO + swz<HD>(brow, bcol), bo);
            ldsm_x4_t(sQ + swz<HD>(brow, bcol), bq);
            mma16816(dv[2 * dn], ap, bo[0], bo[1]);
            mma16816(dv[2 * dn + 1], ap, bo[2], bo[3]);
            mma16816(dk[2 * dn], as, bq[0], bq[1]);
            mma16816(dk[2 * dn + 1], as, bq[2], bq[3]);
          }
        }
      }
    }
  }

  void* dKo = ks ? p.dKn : p.dKc;
  void* dVo = ks ? p.dVn : p.dVc;
#pragma unroll
  for (int nt = 0; nt < HD / 8; ++nt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int64_t key = keyA + 8 * hf;
      if (key < klo || key >= khi) continue;
      const int64_t off = (key * g.Hkv + kvh) * HD + 8 * nt + 2 * tq;
      store_pair(dKo, off, dk[nt][2 * hf] * p.scale, dk[nt][2 * hf + 1] * p.scale, p.g_f32, 0);
      store_pair(dVo, off, dv[nt][2 * hf], dv[nt][2 * hf + 1], p.g_f32, 0);
    }
}

// ----------------------------------------------------------------- dQ
template <int HD>
__global__ void __launch_bounds__(kThreads) bdlm_bwd_dq_kernel(const BwdParams p) {
  constexpr int BQ = kDqTileQ, BK = kDqTileK;
  constexpr int TB = HD * 2;
  extern __shared__ __align__(128) uint8_t sm[];
  const uint32_t sQ = smem_u32(sm), sdO = sQ + BQ * TB, sK = sdO + BQ * TB, sV = sK + BK * TB;

  const Geom& g = p.g;
  const QItem it = q_item(g, BQ, blockIdx.x);
  const int s = it.stream, h = it.head, kvh = h / (g.Hq / g.Hkv);
  const int64_t r0 = it.qtile * BQ, r1 = imin64(r0 + BQ, g.L);
  const QTileRanges q = qtile_ranges(g, s, r0, r1, BK);
  const int nc = (int)(q.c1 - q.c0), n = nc + (int)(q.n1 - q.n0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;

  load_tile<HD, BQ>(sQ, static_cast<const __nv_bfloat16*>(s ? p.Qn : p.Qc), r0, g.L, g.Hq, h);
  load_tile<HD, BQ>(sdO, static_cast<const __nv_bfloat16*>(s ? p.dOn : p.dOc), r0, g.L, g.Hq, h);
  cp_async_wait_all();
  __syncthreads();

  uint32_t qa[HD / 16][4], oa[HD / 16][4];
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const int arow = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8, acol = 16 * kk + (lane >> 4) * 8;
    ldsm_x4(sQ + swz<HD>(arow, acol), qa[kk]);
    ldsm_x4(sdO + swz<HD>(arow, acol), oa[kk]);
  }
  // this thread's rows: ra = r0 + 16 warp + gq and ra + 8
  int64_t rows[2], clo[2], chi[2], nlo[2], nhi[2];
  float lse2[2], Dv[2];
  bool rvalid[2];
  const float* LSE = (s ? p.LSEn : p.LSEc) + (int64_t)h * g.L;
  const float* Dr = (s ? p.Dn : p.Dc) + (int64_t)h * g.L;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    rows[hf] = r0 + 16 * warp + gq + 8 * hf;
    rvalid[hf] = rows[hf] < g.L;
    const int64_t rr = rvalid[hf] ? rows[hf] : g.L - 1;
    clean_interval(g, s, rr, clo[hf], chi[hf]);
    noisy_interval(g, s, rr, nlo[hf], nhi[hf]);
    lse2[hf] = rvalid[hf] ? LSE[rows[hf]] * kLog2e : 0.f;
    Dv[hf] = rvalid[hf] ? Dr[rows[hf]] : 0.f;
  }

  float dq[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dq[i][e] = 0.f;

  for (int j = 0; j < n; ++j) {
    const bool cs = j < nc;
    const int64_t key0 = (cs ? q.c0 + j : q.n0 + (j - nc)) * BK;
    __syncthreads();
    load_tile<HD, BK>(sK, static_cast<const __nv_bfloat16*>(cs ? p.Kc : p.Kn), key0, g.L, g.Hkv, kvh);
    load_tile<HD, BK>(sV, static_cast<const __nv_bfloat16*>(cs ? p.Vc : p.Vn), key0, g.L, g.Hkv, kvh);
    cp_async_wait_all();
    __syncthreads();
    const bool full = cs ? tile_full(key0, BK, q.c_all_lo, q.c_all_hi, g.L)
                         : tile_full(key0, BK, q.n_all_lo, q.n_all_hi, g.L);

    float sc[4][4], dp[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[i][e] = dp[i][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk)
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t bk[4], bv[4];
        const int brow = 16 * np + (lane & 7) + (lane >> 4) * 8, bcol = 16 * kk + ((lane >> 3) & 1) * 8;
        ldsm_x4(sK + swz<HD>(brow, bcol), bk);
        ldsm_x4(sV + swz<HD>(brow, bcol), bv);
        mma16816(sc[2 * np], qa[kk], bk[0], bk[1]);
        mma16816(sc[2 * np + 1], qa[kk], bk[2], bk[3]);
        mma16816(dp[2 * np], oa[kk], bv[0], bv[1]);
        mma16816(dp[2 * np + 1], oa[kk], bv[2], bv[3]);
      }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hf = e >> 1;
        const int64_t key = key0 + 8 * nt + 2 * tq + (e & 1);
        bool vis = full;
        if (!vis) vis = cs ? (key >= clo[hf] && key < chi[hf]) : (key >= nlo[hf] && key < nhi[hf]);
        const float pv = vis ? ex2_approx(fmaf(sc[nt][e], p.scale_log2, -lse2[hf])) : 0.f;
        dp[nt][e] = pv * (dp[nt][e] - Dv[hf]);
      }
#pragma unroll
    for (int kq = 0; kq < 2; ++kq) {
      uint32_t as[4];
      as[0] = pack2(dp[2 * kq][0], dp[2 * kq][1]);
      as[1] = pack2(dp[2 * kq][2], dp[2 * kq][3]);
      as[2] = pack2(dp[2 * kq + 1][0], dp[2 * kq + 1][1]);
      as[3] = pack2(dp[2 * kq + 1][2], dp[2 * kq + 1][3]);
#pragma unroll
      for (int dn = 0; dn < HD / 16; ++dn) {
        uint32_t bk[4];
        const int brow = 16 * kq + (lane & 7) + ((lane >> 3) & 1) * 8, bcol = 16 * dn + (lane >> 4) * 8;
        ldsm_x4_t(sK + swz<HD>(brow, bcol), bk);
        mma16816(dq[2 * dn], as, bk[0], bk[1]);
        mma16816(dq[2 * dn + 1], as, bk[2], bk[3]);
      }
    }
  }

  void* dQo = s ? p.dQn : p.dQc;
#pragma unroll
  for (int nt = 0; nt < HD / 8; ++nt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      if (!rvalid[hf]) continue;
      const int64_t off = (rows[hf] * g.Hq + h) * HD + 8 * nt + 2 * tq;
      store_pair(dQo, off, dq[nt][2 * hf] * p.scale, dq[nt][2 * hf + 1] * p.scale, p.g_f32, p.dq_accumulate);
    }
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

cudaError_t launch_bwd_dkv(const BwdParams& p, cudaStream_t stream, int* launches) {
  const int64_t n = kv_items(p.g, kDkvTileK);
  if (n == 0) return cudaSuccess;
  const int bytes = (2 * kDkvTileK + 2 * kDkvTileQ) * p.d * 2 + 2 * kDkvTileQ * 4;
  cudaError_t e;
  if (p.d == 128) {
    if ((e = set_smem(bdlm_bwd_dkv_kernel<128>, bytes)) != cudaSuccess) return e;
    bdlm_bwd_dkv_kernel<128><<<(unsigned)n, kThreads, bytes, stream>>>(p);
  } else {
    if ((e = set_smem(bdlm_bwd_dkv_kernel<64>, bytes)) != cudaSuccess) return e;
    bdlm_bwd_dkv_kernel<64><<<(unsigned)n, kThreads, bytes, stream>>>(p);
  }
  if (launches) ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdParams& p, cudaStream_t stream, int* launches) {
  const int64_t n = q_items(p.g, kDqTileQ);
  if (n == 0) return cudaSuccess;
  const int bytes = (2 * kDqTileQ + 2 * kDqTileK) * p.d * 2;
  cudaError_t e;
  if (p.d == 128) {
    if ((e = set_smem(bdlm_bwd_dq_kernel<128>, bytes)) != cudaSuccess) return e;
    bdlm_bwd_dq_kernel<128><<<(unsigned)n, kThreads, bytes, stream>>>(p);
  } else {
    if ((e = set_smem(bdlm_bwd_dq_kernel<64>, bytes)) != cudaSuccess) return e;
    bdlm_bwd_dq_kernel<64><<<(unsigned)n, kThreads, bytes, stream>>>(p);
  }
  if (launches) ++*launches;
  return cudaGetLastError();
}

}  // namespace bdlm
