// small_kernels.cu -- HBM-bound kernels: the exact LSE merge of partial
// attention results, the backward row statistic D; the work-list expansion
// of a packed batch; the watchdog self-test.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace {

// Merge of partial softmax-attention results over disjoint key sets (CSBP's
// per-shard partials; Proposition 1, evolve.pub FAQ "Does CSBP change
// training results?": equal to the unsharded result up to reduction order):
//   M = max_p LSE_p, LSE = M + ln sum_p exp(LSE_p - M),
//   O = sum_p exp(LSE_p - LSE) O_p, skipping LSE_p = -inf.
// One warp per (head, row): lane p reads LSE_p; the warp then streams the
// non-empty partials' O rows (HD fp32, 16 bytes per lane) in partial order.
template <int HD>
__global__ void __launch_bounds__(256) bdlm_merge_kernel(const MergeParams p) {
  const int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= p.rows * p.H) return;
  const int h = (int)(wid / p.rows);
  const int64_t r = wid % p.rows;
  const float lp = lane < p.n ? p.LSE[lane][(int64_t)h * p.rows + r] : -INFINITY;
  float M = lp;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const bool any = M != -INFINITY;
  const float w = (any && lp != -INFINITY) ? __expf(lp - M) : 0.f;
  float tot = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const float inv = any ? 1.f / tot : 0.f;
  constexpr int PER = HD / 32;  // floats per lane
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  const int64_t off = (r * p.H + h) * HD + lane * PER;
  for (int q = 0; q < p.n; ++q) {
    const float c = __shfl_sync(0xffffffffu, w, q) * inv;
    if (c == 0.f) continue;
    if (PER == 4) {
      const float4 v = *reinterpret_cast<const float4*>(p.O[q] + off);
      acc[0] = fmaf(c, v.x, acc[0]);
      acc[1] = fmaf(c, v.y, acc[1]);
      acc[2] = fmaf(c, v.z, acc[2]);
      acc[3] = fmaf(c, v.w, acc[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(p.O[q] + off);
      acc[0] = fmaf(c, v.x, acc[0]);
      acc[1] = fmaf(c, v.y, acc[1]);
    }
  }
  if (p.out_f32) {
    float* o = static_cast<float*>(p.out) + off;
    if (PER == 4) *reinterpret_cast<float4*>(o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    else *reinterpret_cast<float2*>(o) = make_float2(acc[0], acc[1]);
  } else {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + off;
    if (PER == 4) *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
    else *reinterpret_cast<uint32_t*>(o) = pack_bf16x2(acc[0], acc[1]);
  }
  if (p.lse_out && lane == 0) p.lse_out[(int64_t)h * p.rows + r] = any ? M + __logf(tot) : -INFINITY;
}

// D_i = sum_d dO_i * O_i, [H, rows] fp32 (the row statistic of the
// softmax-attention backward).  O and dO are [rows, H, HD]: one (row, head)
// pair is HD contiguous elements, and consecutive pairs are contiguous, so
// the pairs are read as one stream of 16-byte chunks.  A pair's HD / 8 chunks
// go to HD / 8 consecutive lanes (two pairs per warp at HD = 128, four at 64),
// each warp takes kUnroll groups of pairs per pass with all their loads
// issued before the first use, and the lanes of a pair reduce by shuffles.
template <int HD, bool OF32>
__global__ void __launch_bounds__(256) bdlm_preprocess_kernel(const void* __restrict__ O,
                                                              const __nv_bfloat16* __restrict__ dO, int64_t rows,
                                                              int H, float* __restrict__ D) {
  constexpr int kCh = HD / 8;            // 16-byte chunks of bf16 per pair
  constexpr int kPairs = 32 / kCh;       // pairs per warp per group
  constexpr int kUnroll = 4;             // groups per warp per pass
  const int lane = threadIdx.x & 31;
  const int64_t npairs = rows * H;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int sub = lane / kCh, ch = lane % kCh;
  for (int64_t g0 = warp0 * kUnroll; g0 * kPairs < npairs; g0 += nwarps * kUnroll) {
    uint4 o[kUnroll][OF32 ? 2 : 1], g[kUnroll];
    int64_t pr[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      pr[u] = (g0 + u) * kPairs + sub;
      const bool v = pr[u] < npairs;
      const int64_t e = (v ? pr[u] : 0) * HD + ch * 8;  // first element of this lane's chunk
      g[u] = v ? __ldg(reinterpret_cast<const uint4*>(dO + e)) : make_uint4(0u, 0u, 0u, 0u);
      if (OF32) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const float*>(O) + e);
        o[u][0] = v ? __ldg(src) : make_uint4(0u, 0u, 0u, 0u);
        o[u][OF32 ? 1 : 0] = v ? __ldg(src + 1) : make_uint4(0u, 0u, 0u, 0u);
      } else {
        o[u][0] = v ? __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(O) + e))
                    : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const __nv_bfloat162* gp = reinterpret_cast<const __nv_bfloat162*>(&g[u]);
      float acc = 0.f;
      if (OF32) {
        const float* of = reinterpret_cast<const float*>(&o[u][0]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 gf = __bfloat1622float2(gp[k]);
          acc = fmaf(of[2 * k], gf.x, acc);
          acc = fmaf(of[2 * k + 1], gf.y, acc);
        }
      } else {
        const __nv_bfloat162* op = reinterpret_cast<const __nv_bfloat162*>(&o[u][0]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 of = __bfloat1622float2(op[k]), gf = __bfloat1622float2(gp[k]);
          acc = fmaf(of.x, gf.x, acc);
          acc = fmaf(of.y, gf.y, acc);
        }
      }
#pragma unroll
      for (int k = kCh / 2; k > 0; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
      if (ch == 0 && pr[u] < npairs) {
        const int64_t r = pr[u] / H;
        const int h = (int)(pr[u] - r * H);
        D[(int64_t)h * rows + r] = acc;
      }
    }
  }
}

// Waits on an mbarrier that nobody arrives on, through the same bounded wait
// the attention kernels use; no asynchronous copy or MMA is in flight.
__global__ void bdlm_watchdog_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Watchdog wd{status, limit_ns, &abort_flag};
  (void)mbar_wait(smem_u32(&bar), 0, wd, 0x7f);
}

// Item table of a packed batch in sequence-major order: the sequences in the
// order given by `order`, each sequence's items in its one-sequence order.
// beg[k] is the first item of the k-th sequence of that order (beg[n] = total).
// kind 0: query items {sequence, stream + 2 * head, query tile, visible key
// tiles} with tiles of tq rows and tk keys; kind 1: key items {sequence, key
// stream + 2 * KV head, key tile, query rows that see it}, tiles of tk keys.
__global__ void __launch_bounds__(256) bdlm_varlen_items_kernel(const Geom all, const int64_t* off,
                                                                 const int64_t* order, const int64_t* beg, int n,
                                                                 int kind, int tq, int tk, int4* out) {
  const int64_t total = beg[n];
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    int lo = 0, hi = n - 1;  // last k with beg[k] <= idx
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (beg[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    const int s = (int)order[lo];
    const int64_t local = idx - beg[lo];
    const Geom g = seq_geom(all, off[s + 1] - off[s]);
    if (kind == 0) {
      const QItem it = q_item(g, tq, local);
      const int64_t r0 = it.qtile * tq, r1 = imin64(r0 + tq, g.L);
      const QTileRanges q = qtile_ranges(g, it.stream, r0, r1, tk);
      out[idx] = make_int4(s, it.stream + 2 * it.head, (int)it.qtile, (int)((q.c1 - q.c0) + (q.n1 - q.n0)));
    } else {
      const KVItem it = kv_item(g, tk, local);
      int64_t cl, ch, nl, nh;
      kv_tile_rows(g, it.key_stream, it.ktile * tk, imin64(it.ktile * tk + tk, g.L), cl, ch, nl, nh);
      out[idx] = make_int4(s, it.key_stream + 2 * it.kv_head, (int)it.ktile,
                           (int)(imax64(0, ch - cl) + imax64(0, nh - nl)));
    }
  }
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream, int* launches) {
  const int64_t warps = p.rows * p.H;
  if (warps == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  if (p.d == 128) bdlm_merge_kernel<128><<<blocks, 256, 0, stream>>>(p);
  else bdlm_merge_kernel<64><<<blocks, 256, 0, stream>>>(p);
  if (launches) ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_preprocess(const void* O, int o_f32, const void* dO, int64_t rows, int H, int d, float* D,
                              cudaStream_t stream, int* launches, int num_sms) {
  const int64_t pairs = rows * H;
  if (pairs == 0) return cudaSuccess;
  // 8 warps per block, each taking 4 groups of 32 / (d / 8) pairs per pass;
  // at most 8 resident blocks per SM, grid-stride beyond that
  const int64_t per_block = 8 * 4 * (32 / (d / 8));
  int64_t blocks = (pairs + per_block - 1) / per_block;
  const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 152) * 8;
  if (blocks > cap) blocks = cap;
  const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(dO);
  const unsigned nb = (unsigned)blocks;
  if (d == 128) {
    if (o_f32) bdlm_preprocess_kernel<128, true><<<nb, 256, 0, stream>>>(O, g, rows, H, D);
    else bdlm_preprocess_kernel<128, false><<<nb, 256, 0, stream>>>(O, g, rows, H, D);
  } else {
    if (o_f32) bdlm_preprocess_kernel<64, true><<<nb, 256, 0, stream>>>(O, g, rows, H, D);
    else bdlm_preprocess_kernel<64, false><<<nb, 256, 0, stream>>>(O, g, rows, H, D);
  }
  if (launches) ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_varlen_items(const Geom& all, const int64_t* off, const int64_t* order, const int64_t* beg, int n,
                                int64_t total, int kind, int tq, int tk, int4* out, cudaStream_t stream,
                                int* launches) {
  if (total == 0) return cudaSuccess;
  const int64_t blocks = (total + 255) / 256;
  bdlm_varlen_items_kernel<<<(int)(blocks < 1024 ? blocks : 1024), 256, 0, stream>>>(all, off, order, beg, n, kind,
                                                                                     tq, tk, out);
  if (launches) ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_watchdog(uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  bdlm_watchdog_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace bdlm
