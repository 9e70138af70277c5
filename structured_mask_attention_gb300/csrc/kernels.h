// kernels.h -- launch interfaces of the device kernels (host side).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "geometry.cuh"

namespace bdlm {

// ------------------------------------------------------------- forward
struct FwdParams {
  Geom g;
  float scale_log2;  // softmax scale * log2(e)
  void* Oc;
  void* On;
  int o_f32;  // outputs fp32 (else bf16)
  float* LSEc;
  float* LSEn;
  int64_t n_items;
  uint32_t* status;
  uint64_t limit_ns;
};

// Work-item tables of a packed variable-length batch, passed to the batch
// instantiations of the kernels as a separate argument (so the one-sequence
// kernels keep their parameter block, and their register allocation, as is).
// Query items {sequence, stream + 2 * head, query tile, cost}, key items
// {sequence, key stream + 2 * KV head, key tile, cost}, both in launch order,
// and the n_seqs + 1 row offsets of the sequences.  With a batch, g.L in the
// parameters is the total row count (the LSE / D row stride) and each item's
// own geometry comes from its sequence.
struct VarlenTabs {
  const int4* q_items;
  const int4* kv_items;
  const int64_t* seq_off;
  int64_t n_q, n_kv;
};

struct FwdMaps {
  CUtensorMap Qc, Qn, Kc, Kn, Vc, Vn;
};

// Per-row reference of the fixed-reference verification mode: [Hq, L] fp32,
// natural-log units, one array per stream.  When given, every row forms its
// probabilities as exp(scale q.k - M_ref) against this fixed value instead of
// its running maximum (no rescaling), so two calls that see the same key tile
// for the same row round the same probabilities to bf16.  Null: production.
struct FwdRef {
  const float* c;
  const float* n;
};

// Words (uint32) of the workspace header that the kernels use: word 0 is the
// status word; from kSchedWordFwd / Dkv / Dq on, each attention kernel's work
// item counter and its count of finished CTAs (two words each; sched.cuh).
// The host zeroes the first kHeaderClearBytes of the header before each call.
constexpr int kSchedWordFwd = 8, kSchedWordDkv = 10, kSchedWordDq = 12;
constexpr int kHeaderClearBytes = 64;

// Tile sizes of the tensor-core forward: items of 256 query rows (two
// 128-row sub-tiles sharing their key tiles), 128 keys per step.
constexpr int kFwdTileQ = 128;
constexpr int kFwdItemRows = 256;
constexpr int kFwdTileK = 128;

// vt: null for one sequence.  ref: null for the production kernel (see FwdRef).
// rows: null for every row (else one sequence, no ref).
cudaError_t launch_fwd(const FwdMaps& maps, const FwdParams& p, const VarlenTabs* vt, const FwdRef* ref,
                       const RowRange* rows, int d, int num_sms, cudaStream_t stream, int* launches);

// ------------------------------------------------------------- backward
struct BwdParams {
  Geom g;
  int d;
  float scale;       // softmax scale (for dQ, dK)
  float scale_log2;  // scale * log2(e)
  const void *Qc, *Kc, *Vc, *Qn, *Kn, *Vn, *dOc, *dOn;  // bf16
  const float *LSEc, *LSEn, *Dc, *Dn;                  // [Hq, L]
  void *dQc, *dQn, *dKc, *dVc, *dKn, *dVn;
  int g_f32;         // gradient outputs fp32 (else bf16)
  int dq_accumulate; // dQ += contribution (fp32 only)
  int dkv_accumulate;  // dK, dV += contribution (fp32 only)
  int rows_call;       // row-restricted call: the kernels' rows instantiations
  RowRange rows;       // query rows of the call and where its tensors' rows live
};

// Tensor maps of the tensor-core backward passes: [L, H, d] bf16 viewed 3-D,
// 64-column (128-byte) x 128-row boxes, 128-byte swizzle.
constexpr int kBwdTile = 128;
struct BwdMaps {
  CUtensorMap Qc, Qn, dOc, dOn, Kc, Kn, Vc, Vn;
};
cudaError_t launch_bwd_dq_tc(const BwdMaps& m, const BwdParams& p, const VarlenTabs* vt, int num_sms,
                             uint32_t* status, uint64_t limit_ns, cudaStream_t stream, int* launches);
cudaError_t launch_bwd_dkv_tc(const BwdMaps& m, const BwdParams& p, const VarlenTabs* vt, int num_sms,
                              uint32_t* status, uint64_t limit_ns, cudaStream_t stream, int* launches);

// ------------------------------------------------------------- small kernels
constexpr int kMaxParts = 32;
struct MergeParams {
  const float* O[kMaxParts];
  const float* LSE[kMaxParts];
  int n;
  int64_t rows;
  int H, d;
  void* out;
  int out_f32;
  float* lse_out;
};

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream, int* launches);
cudaError_t launch_preprocess(const void* O, int o_f32, const void* dO, int64_t rows, int H, int d, float* D,
                              cudaStream_t stream, int* launches, int num_sms);
cudaError_t launch_watchdog(uint32_t* status, uint64_t limit_ns, cudaStream_t stream);
// Packed-batch item table, sequence-major (kind 0: query items, 1: key items).
cudaError_t launch_varlen_items(const Geom& all, const int64_t* off, const int64_t* order, const int64_t* beg, int n,
                                int64_t total, int kind, int tq, int tk, int4* out, cudaStream_t stream,
                                int* launches);

// Records the message bdlm_last_error() returns on this thread.
void set_last_error(const std::string& msg);

}  // namespace bdlm
