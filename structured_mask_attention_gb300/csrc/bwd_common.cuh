// bwd_common.cuh -- pieces shared by the two backward passes (bwd_dq.cu,
// bwd_dkv.cu): thread roles, row stores and the packed-operand column map.
//
// Gradients of softmax attention under the two-stream block mask, no gradient
// through LSE ("Block Parallelism For Efficient Distributed Long-Context
// Diffusion Language Model Training": training gradients, evolve.pub review
// "Key claims" / Proposition 1; only clean K/V gradients cross context shards,
// evolve.pub FAQ on CSBP):
//   P = exp(scale Q K^T - LSE), dP = dO V^T, dS = P o (dP - D),
//   dV = sum_group P^T dO, dK = scale sum_group dS^T Q, dQ = scale dS K.
//
// Both passes are persistent (one CTA per SM) with 10 warps: warp 0 feeds
// shared memory with TMA, warp 1 owns TMEM and one of its lanes issues
// tcgen05.mma, warps 2-9 form two elementwise warpgroups.  A thread owns one
// TMEM lane (a query row for dQ, a key row for dK/dV); the two warpgroups
// split the 128 columns of each step, 64 each.  Every MMA has N >= 128: at
// M = 128, K = 16 an N = 64 MMA takes ~50 cycles for half the work of an
// N = 128 one (~65 cycles) on this part.
#pragma once
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bdlm {
namespace bwd {

constexpr int kThreads = 320;
constexpr int kEwThreads = 256;  // elementwise threads (barrier arrival counts)
constexpr float kLog2e = 1.4426950408889634f;

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

// 32 fp32 values of one row (times mul) -> global, fp32 (optionally added
// to what is there) or bf16.
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

// dS = exp2(s sl2 + nl) (dP - D) for 32 keys of one query row (nl = -LSE
// log2 e, nD = -D, both broadcast in packed pairs); keys outside [lo, hi)
// (offsets within the 32) give 0 unless FULL.  Packed bf16 pairs into pk.
// fma, add and mul run on packed fp32 pairs.
template <bool FULL>
__device__ __forceinline__ void ds_row32(const uint32_t (&us)[32], const uint32_t (&ud)[32], uint64_t sl2x2,
                                         uint64_t nl2, uint64_t nD2, int lo, int hi, uint32_t (&pk)[16]) {
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    float x0, x1, d0, d1;
    f2_split(f2_fma(f2(__uint_as_float(us[c]), __uint_as_float(us[c + 1])), sl2x2, nl2), x0, x1);
    const uint64_t t = f2_add(f2(__uint_as_float(ud[c]), __uint_as_float(ud[c + 1])), nD2);
    f2_split(f2_mul(f2(ex2_approx(x0), ex2_approx(x1)), t), d0, d1);
    if (!FULL) {
      d0 = (c >= lo && c < hi) ? d0 : 0.f;
      d1 = (c + 1 >= lo && c + 1 < hi) ? d1 : 0.f;
    }
    pk[c / 2] = pack_bf16x2(d0, d1);
  }
}

// A 128-wide step is read and rewritten in four 32-column quarters: quarter q
// (warpgroup q / 2, sub-step q % 2) reads fp32 columns [32 q, 32 q + 32) and
// writes its 16 packed bf16 columns at 32 (q / 2) * 2 + 16 (q % 2), i.e. over
// columns its own warpgroup has already read.  K-step kk (16 elements) of the
// packed A operand therefore sits at this column:
__device__ __forceinline__ uint32_t packed_col128(int kk) {
  return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8);
}

}  // namespace bwd
}  // namespace bdlm
