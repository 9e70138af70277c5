/*
 * bdlm_attn.h -- C ABI of the two-stream block-diffusion (BDLM) attention
 * library for NVIDIA GB300 (sm_103a).
 *
 * The operation.  A block diffusion language model reads a clean sequence of
 * length L together with a corrupted copy of it, both split into N = L / B
 * blocks of B tokens ("Block Parallelism For Efficient Distributed
 * Long-Context Diffusion Language Model Training", arxiv.science abstract:
 * autoregressive dependencies across blocks, parallel denoising inside a
 * block).  Attention over the combined 2L sequence uses the two-stream block
 * mask, blk(i) = floor(i / B):
 *   clean row i     reads clean key j      iff blk(j) <= blk(i)
 *   corrupted row i reads clean key j      iff blk(j) <  blk(i)
 *   corrupted row i reads corrupted key j  iff blk(j) == blk(i)
 *   clean rows never read corrupted keys.
 * Per query head h (key/value head floor(h / (Hq/Hkv))):
 *   s_ij = scale * q_i . k_j,  LSE_i = ln sum_j exp(s_ij),
 *   O_i = sum_j exp(s_ij - LSE_i) v_j.
 * The mask is never materialised: kernels visit only the key tiles a query
 * tile can see (the per-target-block separation of the evolve.pub review,
 * "Scope & Claims", Eq. 3 / Eq. 6).
 *
 * Context sharding (CSBP: evolve.pub review FAQ "What is context-sharded block
 * parallelism?"; Sec. 4 / Fig. 3): the clean keys can be split into contiguous
 * shards; attention against each shard gives a partial (O_p, LSE_p), and the
 * exact log-sum-exp merge of the partials equals the unsharded result up to
 * floating-point reduction order (Proposition 1, evolve.pub FAQ "Does CSBP
 * change training results?").
 *
 * Conventions for every call:
 *  - Layout.  Q, K, V, O, dO and gradients are token-major [L, H, d] arrays,
 *    contiguous, one per stream (clean "c", corrupted "n").  LSE and D are
 *    [H, L] fp32.  Batch is 1.  d is 64 or 128.  Q/K/V/dO are bf16.
 *  - Memory.  Every pointer is a device pointer owned by the caller, who also
 *    owns the workspace (size from bdlm_workspace_size).  The library
 *    allocates and frees nothing.  Device pointers must be 16-byte aligned.
 *    A workspace serves one call at a time: calls that may overlap on the
 *    GPU (different streams, no ordering) need workspaces of their own.
 *  - Execution.  Calls enqueue work on `stream` and return without waiting.
 *  - Validation.  Arguments are checked on the host before anything is
 *    enqueued; a failing check returns a non-OK status, enqueues nothing and
 *    records a message for bdlm_last_error().  No C++ exception crosses this
 *    boundary.
 *  - Watchdog.  Every device-side wait in the kernels is bounded in time; on
 *    expiry the kernel records an error in the workspace's status word and
 *    returns.  bdlm_sync_status() reports it as BDLM_ERR_TIMEOUT.
 */
#ifndef BDLM_ATTN_H
#define BDLM_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BDLM_OK = 0,
  BDLM_ERR_INVALID_ARG = 1, /* null pointer, bad enum, bad scale */
  BDLM_ERR_SHAPE = 2,       /* L % B, Hq % Hkv, d not in {64,128}, L % P, bad range */
  BDLM_ERR_ALIGN = 3,       /* a pointer not 16-byte aligned */
  BDLM_ERR_WORKSPACE = 4,   /* workspace missing or smaller than bdlm_workspace_size */
  BDLM_ERR_CUDA = 5,        /* a CUDA runtime/driver call or launch failed */
  BDLM_ERR_UNSUPPORTED = 6, /* device is not sm_103; or a packed-batch call inside CUDA-graph capture */
  BDLM_ERR_TIMEOUT = 7      /* a device-side bounded wait expired */
} bdlm_status;

typedef enum { BDLM_BF16 = 0, BDLM_F32 = 1 } bdlm_dtype;

typedef enum {
  BDLM_OP_FWD = 0,
  BDLM_OP_FWD_SHARD = 1,
  BDLM_OP_BWD = 2,
  BDLM_OP_BWD_SHARD = 3
} bdlm_op;

/* Opaque CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef void* bdlm_stream;

/* Workspace bytes a call of kind `op` needs at this shape (P is ignored by
 * every op today and kept for shard-count dependent variants).  The
 * workspace holds a 256-byte header (the status word in its first 4 bytes,
 * then the counters from which the kernels' persistent CTAs claim work
 * items; every call zeroes what it uses before its first kernel) and, for
 * BDLM_OP_BWD, the row statistic D of both streams.  Returns 0 for an
 * invalid shape. */
size_t bdlm_workspace_size(int op, int64_t L, int64_t B, int Hq, int Hkv, int d, int P);

/* Two-stream forward (arxiv.science abstract; the mask above).
 * In:  Qc, Qn [L,Hq,d] bf16; Kc, Vc, Kn, Vn [L,Hkv,d] bf16.
 * Out: Oc, On [L,Hq,d] in o_dtype; LSEc, LSEn [Hq,L] fp32, natural log.
 * scale > 0 (usually 1/sqrt(d)).  Requires L % B == 0, Hq % Hkv == 0. */
bdlm_status bdlm_attn_fwd(const void* Qc, const void* Kc, const void* Vc,
                          const void* Qn, const void* Kn, const void* Vn,
                          int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                          void* Oc, void* On, bdlm_dtype o_dtype,
                          float* LSEc, float* LSEn,
                          void* workspace, size_t ws_bytes, bdlm_stream stream);

/* Partial forward of one context shard (CSBP, evolve.pub FAQ on CSBP):
 * both streams' rows attend only to clean keys in [kv_begin, kv_end) and, if
 * include_local != 0, the corrupted rows also to their own corrupted block.
 * Rows with no visible key in this partial get O = 0 and LSE = -inf.
 * Out: Op_c, Op_n [L,Hq,d] fp32; LSEp_c, LSEp_n [Hq,L] fp32.
 * 0 <= kv_begin <= kv_end <= L; any boundaries (need not align to B). */
bdlm_status bdlm_attn_fwd_shard(const void* Qc, const void* Kc, const void* Vc,
                                const void* Qn, const void* Kn, const void* Vn,
                                int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                                int64_t kv_begin, int64_t kv_end, int include_local,
                                float* Op_c, float* Op_n, float* LSEp_c, float* LSEp_n,
                                void* workspace, size_t ws_bytes, bdlm_stream stream);

/* Verification mode of the partial forward, for checking that
 * shard-and-merge reproduces the unsharded result up to floating-point
 * reduction order (Proposition 1; evolve.pub FAQ "Does CSBP change training
 * results?").  The production kernels round the probabilities P to bf16
 * before the P.V product relative to each row's running maximum, which
 * differs between a shard and the whole key range, so their fp32 outputs
 * also differ by that rounding.  This call is bdlm_attn_fwd_shard with one
 * change: every row forms P = exp(scale q.k - Mref) against a fixed reference
 * Mref supplied by the caller, with no rescaling.  Called for the whole key
 * range (kv_begin = 0, kv_end = L, include_local = 1) it gives the unsharded
 * result; called per shard with the same Mref, every (row, key) probability
 * is rounded identically in both, and only fp32 summation order differs.
 * Mref_c, Mref_n: [Hq, L] fp32, natural log, finite, and at least the row's
 * largest scaled score over the keys of the call (the LSE of the unsharded
 * forward qualifies); a smaller value can overflow P.  Same outputs, layout
 * and errors as bdlm_attn_fwd_shard; same speed class (one extra load per
 * row).  Not for training: use the production calls. */
bdlm_status bdlm_attn_fwd_shard_refmax(const void* Qc, const void* Kc, const void* Vc,
                                       const void* Qn, const void* Kn, const void* Vn,
                                       int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                                       int64_t kv_begin, int64_t kv_end, int include_local,
                                       const float* Mref_c, const float* Mref_n,
                                       float* Op_c, float* Op_n, float* LSEp_c, float* LSEp_n,
                                       void* workspace, size_t ws_bytes, bdlm_stream stream);

/* Exact merge of partial attention results over disjoint key sets
 * (Proposition 1 / evolve.pub FAQ "Does CSBP change training results?"):
 *   M = max_p LSE_p,  LSE = M + ln sum_p exp(LSE_p - M),
 *   O = sum_p exp(LSE_p - LSE) O_p,   partials with LSE_p = -inf skipped;
 *   a row whose partials are all -inf gets O = 0, LSE = -inf.
 * O_parts / LSE_parts: HOST arrays of n_parts DEVICE pointers (1 <= n_parts
 * <= 32) to O_p [rows,H,d] fp32 and LSE_p [H,rows] fp32.  Summation order is
 * the partial order (deterministic).  Out: O [rows,H,d] in o_dtype, LSE
 * [H,rows] fp32.  LSE may be NULL to skip writing it. */
bdlm_status bdlm_lse_merge(int n_parts, const float* const* O_parts, const float* const* LSE_parts,
                           int64_t rows, int H, int d, void* O, bdlm_dtype o_dtype, float* LSE,
                           bdlm_stream stream);

/* Backward row statistic D_i = sum_d dO_i * O_i (softmax-attention backward;
 * the gradients Proposition 1 covers).  O and dO [rows,H,d] bf16 (or O fp32
 * when o_dtype = BDLM_F32); D [H,rows] fp32. */
bdlm_status bdlm_bwd_preprocess(const void* O, bdlm_dtype o_dtype, const void* dO,
                                int64_t rows, int H, int d, float* D, bdlm_stream stream);

/* Two-stream backward, no gradient through LSE:
 *   D_i = dO_i.O_i, dS_ij = p_ij (dO_i.v_j - D_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_{h in group} sum_i dS_ij q_i,
 *   dV_j = sum_{h in group} sum_i p_ij dO_i.
 * In: the forward's inputs, Oc/On and dOc/dOn [L,Hq,d] bf16, LSEc/LSEn from
 * bdlm_attn_fwd.  Out: dQc, dQn [L,Hq,d]; dKc, dVc, dKn, dVn [L,Hkv,d], all
 * in g_dtype.  Deterministic: every gradient element is written once, by one
 * thread, after a fixed-order reduction. */
bdlm_status bdlm_attn_bwd(const void* Qc, const void* Kc, const void* Vc,
                          const void* Qn, const void* Kn, const void* Vn,
                          const void* Oc, const void* On, const void* dOc, const void* dOn,
                          const float* LSEc, const float* LSEn,
                          int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                          void* dQc, void* dKc, void* dVc, void* dQn, void* dKn, void* dVn,
                          bdlm_dtype g_dtype, void* workspace, size_t ws_bytes, bdlm_stream stream);

/* bdlm_attn_bwd for callers that cannot allocate device memory.  (The paper
 * has no counterpart: this is a deployment variant of the backward.)
 * Plugin hosts that hand a library only its input and output buffers,
 * runtimes that reserve all device memory up front, and latency-critical
 * code that avoids cudaMalloc (it may synchronize the device) cannot supply
 * a workspace.  This call takes the same arguments as bdlm_attn_bwd minus
 * the workspace and runs the same kernels with their workspace placed in a
 * fixed 32 MiB array of device global memory declared by the library.
 *  - Limit: the workspace (256 + 8 * Hq * L bytes) must fit the array, i.e.
 *    Hq * L <= 4194272; larger shapes return BDLM_ERR_WORKSPACE, enqueue
 *    nothing, and bdlm_last_error() names the limit.
 *  - The array is created when the library's module is loaded on a device
 *    and every GPU that loads it holds it until the process exits.  The first
 *    call on a device looks up the array's device address with that device
 *    current (and looks it up again after the device's context was
 *    re-created, e.g. by cudaDeviceReset); that lookup may load the
 *    library's device code, so make the first call before any stream
 *    capture.
 *  - Every call shares the one array per device and leaves its contents
 *    behind; each call clears the status word and the work counters and
 *    rewrites D before use.
 *    Calls that overlap on the GPU (different streams, no ordering) race on
 *    the array and must not be issued.
 *  - No cudaMalloc, cudaFree or allocating library routine is called.  With
 *    per-kernel timing enabled (bdlm_timing_enable), launches also record
 *    CUDA events from a pool the library creates on first use: keep timing
 *    off when no allocation at all is allowed.
 * Kernel status (a device wait that ran out of time) goes to the array's
 * status word, not to this call's return value, which reports argument and
 * launch errors: read it with bdlm_sync_status_noalloc. */
bdlm_status bdlm_attn_bwd_noalloc(const void* Qc, const void* Kc, const void* Vc,
                                  const void* Qn, const void* Kn, const void* Vn,
                                  const void* Oc, const void* On, const void* dOc, const void* dOn,
                                  const float* LSEc, const float* LSEn,
                                  int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                                  void* dQc, void* dKc, void* dVc, void* dQn, void* dKn, void* dVn,
                                  bdlm_dtype g_dtype, bdlm_stream stream);

/* bdlm_sync_status for the array of bdlm_attn_bwd_noalloc on the current
 * device: waits for `stream`, reads and clears the array's status word, and
 * returns BDLM_ERR_TIMEOUT if a kernel of an earlier allocation-free call
 * gave up on a device wait, BDLM_ERR_CUDA on a stream error, else BDLM_OK.
 * Allocates nothing. */
bdlm_status bdlm_sync_status_noalloc(bdlm_stream stream);

/* bdlm_watchdog_selftest run on the status word of the allocation-free
 * array (see bdlm_watchdog_selftest below): a wait nobody ends runs out after
 * limit_us microseconds and the call returns BDLM_ERR_TIMEOUT, read back
 * through bdlm_sync_status_noalloc.  Allocates nothing. */
bdlm_status bdlm_watchdog_selftest_noalloc(uint32_t limit_us, bdlm_stream stream);

/* Gradient contribution of one context shard, given the MERGED forward
 * statistics LSEc/LSEn and D (from bdlm_bwd_preprocess on the merged O):
 * keys are clean [kv_begin, kv_end) plus, if include_local, the corrupted own
 * blocks.  dK/dV of disjoint shards are independent: this call writes
 * dKc/dVc rows [kv_begin, kv_end) and, if include_local, all rows of dKn/dVn
 * (fp32); other rows are left untouched.  dQ is accumulated:
 * dQc_acc += contribution, dQn_acc += contribution (fp32, [L,Hq,d]); the
 * caller zeroes them before the first shard.  Calls on one stream in a fixed
 * shard order give a deterministic dQ. */
bdlm_status bdlm_attn_bwd_shard(const void* Qc, const void* Kc, const void* Vc,
                                const void* Qn, const void* Kn, const void* Vn,
                                const void* dOc, const void* dOn,
                                const float* LSEc, const float* LSEn, const float* Dc, const float* Dn,
                                int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                                int64_t kv_begin, int64_t kv_end, int include_local,
                                float* dQc_acc, float* dQn_acc,
                                float* dKc, float* dVc, float* dKn, float* dVn,
                                void* workspace, size_t ws_bytes, bdlm_stream stream);

/* ---- One rank's rows (multi-rank CSBP) -----------------------------------
 * A rank of a context-sharded deployment (evolve.pub FAQ on CSBP: ranks own
 * complete corrupted blocks and a shard of the clean context; only clean K/V
 * and their gradients cross ranks) computes its own query rows only.  These
 * two calls are bdlm_attn_fwd_shard and bdlm_attn_bwd_shard restricted to
 * the clean rows [rows_c_begin, rows_c_end) and the corrupted rows
 * [rows_n_begin, rows_n_end) (0 <= begin <= end <= L; any boundaries, most
 * naturally whole blocks).  Other rows are neither computed into the
 * results nor written.
 *  - bdlm_attn_fwd_shard_rows writes Op/LSEp of those rows only (rows with no
 *    visible key: O = 0, LSE = -inf), against clean keys [kv_begin, kv_end)
 *    and, with include_local, the rows' own corrupted blocks.
 *  - bdlm_attn_bwd_shard_rows ADDS the contributions of those rows: dQ of
 *    the rows into dQc_acc / dQn_acc, and dK, dV of the call's keys (clean
 *    [kv_begin, kv_end), plus every corrupted key with include_local) into
 *    dKc_acc, dVc_acc, dKn_acc, dVn_acc (all fp32, zeroed by the caller
 *    before the first call).  LSE and D are the merged, full-row statistics.
 *    Contributions of disjoint row sets to the same keys add up to the
 *    gradient of all rows; on one stream in a fixed order the sums are
 *    deterministic. */
bdlm_status bdlm_attn_fwd_shard_rows(const void* Qc, const void* Kc, const void* Vc,
                                     const void* Qn, const void* Kn, const void* Vn,
                                     int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                                     int64_t kv_begin, int64_t kv_end, int include_local,
                                     int64_t rows_c_begin, int64_t rows_c_end,
                                     int64_t rows_n_begin, int64_t rows_n_end,
                                     float* Op_c, float* Op_n, float* LSEp_c, float* LSEp_n,
                                     void* workspace, size_t ws_bytes, bdlm_stream stream);

bdlm_status bdlm_attn_bwd_shard_rows(const void* Qc, const void* Kc, const void* Vc,
                                     const void* Qn, const void* Kn, const void* Vn,
                                     const void* dOc, const void* dOn,
                                     const float* LSEc, const float* LSEn, const float* Dc, const float* Dn,
                                     int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                                     int64_t kv_begin, int64_t kv_end, int include_local,
                                     int64_t rows_c_begin, int64_t rows_c_end,
                                     int64_t rows_n_begin, int64_t rows_n_end,
                                     float* dQc_acc, float* dQn_acc,
                                     float* dKc_acc, float* dVc_acc, float* dKn_acc, float* dVn_acc,
                                     void* workspace, size_t ws_bytes, bdlm_stream stream);

/* ---- One rank's rows with rank-local tensors (multi-rank CSBP) -----------
 * The same computation as bdlm_attn_fwd_shard_rows / bdlm_attn_bwd_shard_rows,
 * with every tensor holding only what the rank holds (so that no rank stores
 * the whole sequence: evolve.pub FAQ on CSBP, memory):
 *  - clean-stream row tensors hold rows [rows_c_begin, rows_c_end) only:
 *    Qc, dOc, Op_c, dQc_acc as [rows_c_end - rows_c_begin, H, d], LSEp_c,
 *    LSEc, Dc as [Hq, rows_c_end - rows_c_begin];
 *  - corrupted-stream tensors hold rows [rows_n_begin, rows_n_end) only: Qn,
 *    Kn, Vn, dOn, Op_n, LSEp_n, LSEn, Dn, dQn_acc, dKn_acc, dVn_acc (with the
 *    local partial, include_local, this range must be whole blocks of B, or
 *    end at L: a corrupted row reads its whole block's keys);
 *  - Kc, Vc, dKc_acc, dVc_acc hold the clean keys [kv_begin, kv_end) only
 *    (one shard as received, or the whole gathered clean sequence).
 * L is the full sequence length; row and key indices are global.  A tensor
 * of a stream with no rows may be any valid 16-byte-aligned device buffer
 * (it is not read).  Errors as for the full-length calls, plus
 * BDLM_ERR_SHAPE for a corrupted range that is not whole blocks. */
bdlm_status bdlm_attn_fwd_rank(const void* Qc, const void* Kc, const void* Vc,
                               const void* Qn, const void* Kn, const void* Vn,
                               int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                               int64_t kv_begin, int64_t kv_end, int include_local,
                               int64_t rows_c_begin, int64_t rows_c_end,
                               int64_t rows_n_begin, int64_t rows_n_end,
                               float* Op_c, float* Op_n, float* LSEp_c, float* LSEp_n,
                               void* workspace, size_t ws_bytes, bdlm_stream stream);

bdlm_status bdlm_attn_bwd_rank(const void* Qc, const void* Kc, const void* Vc,
                               const void* Qn, const void* Kn, const void* Vn,
                               const void* dOc, const void* dOn,
                               const float* LSEc, const float* LSEn, const float* Dc, const float* Dn,
                               int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                               int64_t kv_begin, int64_t kv_end, int include_local,
                               int64_t rows_c_begin, int64_t rows_c_end,
                               int64_t rows_n_begin, int64_t rows_n_end,
                               float* dQc_acc, float* dQn_acc,
                               float* dKc_acc, float* dVc_acc, float* dKn_acc, float* dVn_acc,
                               void* workspace, size_t ws_bytes, bdlm_stream stream);

/* ---- Packed variable-length batch (batch > 1) ---------------------------
 * Several independent two-stream problems in one call, for batches of
 * sequences (the pages tune the batch size alongside the parallelism:
 * "Block Parallelism ...", nips.cc abstract).  n_seqs sequences are stored
 * back to back along the token dimension: sequence s owns rows
 * [seq_offsets[s], seq_offsets[s+1]) of both streams of Q/K/V/O/dO and of the
 * gradients ([T, H, d], T = seq_offsets[n_seqs]) and the same columns of LSE
 * ([Hq, T], natural log).  seq_offsets is a host array of n_seqs + 1 int64,
 * seq_offsets[0] = 0, every sequence length a positive multiple of B; a row
 * attends only within its own sequence, with the mask of the one-sequence
 * calls.  All sequences run in one launch per kernel over one work list:
 * the sequences one after the other, longest first, each in its
 * one-sequence order.  The offsets are read before the call returns (the
 * host array may be freed then); the library's own copy reaches the
 * workspace on the stream, and a small kernel expands it into the work list.
 * These calls cannot be captured into a CUDA graph (BDLM_ERR_UNSUPPORTED):
 * they copy host data that differs from call to call.
 * BDLM_VARLEN_ORDER=lpt instead orders all items longest first over the
 * whole batch, built on the host (a scheduling ablation).  Same conventions,
 * dtypes and error behaviour as bdlm_attn_fwd / bdlm_attn_bwd (the backward
 * takes the forward's O and LSE of the same packed batch).
 *
 * bdlm_workspace_size_varlen: bytes of workspace for op BDLM_OP_FWD or
 * BDLM_OP_BWD (0 for another op or a bad shape). */
size_t bdlm_workspace_size_varlen(int op, const int64_t* seq_offsets, int n_seqs, int Hq, int Hkv, int d);

bdlm_status bdlm_attn_fwd_varlen(const void* Qc, const void* Kc, const void* Vc,
                                 const void* Qn, const void* Kn, const void* Vn,
                                 const int64_t* seq_offsets, int n_seqs, int64_t B,
                                 int Hq, int Hkv, int d, float scale,
                                 void* Oc, void* On, bdlm_dtype o_dtype,
                                 float* LSEc, float* LSEn,
                                 void* workspace, size_t ws_bytes, bdlm_stream stream);

bdlm_status bdlm_attn_bwd_varlen(const void* Qc, const void* Kc, const void* Vc,
                                 const void* Qn, const void* Kn, const void* Vn,
                                 const void* Oc, const void* On, const void* dOc, const void* dOn,
                                 const float* LSEc, const float* LSEn,
                                 const int64_t* seq_offsets, int n_seqs, int64_t B,
                                 int Hq, int Hkv, int d, float scale,
                                 void* dQc, void* dKc, void* dVc, void* dQn, void* dKn, void* dVn,
                                 bdlm_dtype g_dtype, void* workspace, size_t ws_bytes,
                                 bdlm_stream stream);

/* Host-only: the forward work list in the order the persistent CTAs claim
 * its items, for inspection and tests.
 * One item per (query tile of tile_q rows, query head, stream), longest
 * first: query tiles from the last to the first.  With at least
 * 6 * G / (2 Hq / Hkv) query tiles they go in blocks of G / (2 Hq / Hkv)
 * tiles (G = 152 here, a GB300's SM count; the kernels use the grid they
 * run on), and inside a block the items of one KV head (its query heads, both
 * streams) come together, one KV head after the other, so that the items a
 * persistent grid runs at the same time read the same keys; otherwise the two
 * streams of one head are adjacent, then the heads.  Along the list the
 * number of visible key tiles never exceeds the largest seen so far (plus one
 * tile for the corrupted stream, whose own-block range can straddle one more
 * tile).
 * Each item is 8 int32:
 *   {stream (0 clean, 1 corrupted), head, q_tile, clean_tile_begin,
 *    clean_tile_end, corrupted_tile_begin, corrupted_tile_end, n_tiles}
 * in units of tile_k keys.  Writes min(count, cap) items to `out` (may be
 * NULL when cap == 0) and returns the total count, or -1 on a bad shape. */
int64_t bdlm_worklist(int64_t L, int64_t B, int Hq, int Hkv, int tile_q, int tile_k,
                      int64_t kv_begin, int64_t kv_end, int include_local,
                      int32_t* out, int64_t cap);

/* Waits for `stream`, then reads and clears the workspace's status word.
 * Returns BDLM_ERR_TIMEOUT if a kernel's bounded wait expired, BDLM_ERR_CUDA
 * if the stream reported an error, else BDLM_OK. */
bdlm_status bdlm_sync_status(void* workspace, bdlm_stream stream);

/* Exercises the device watchdog: launches a one-warp kernel that waits on an
 * mbarrier nobody arrives on, with a limit of `limit_us` microseconds (no
 * asynchronous copy or tensor-core work is in flight).  The kernel gives up,
 * records the timeout in the workspace status word and returns; the call then
 * behaves like bdlm_sync_status and returns BDLM_ERR_TIMEOUT when the
 * watchdog works. */
bdlm_status bdlm_watchdog_selftest(void* workspace, size_t ws_bytes, uint32_t limit_us,
                                   bdlm_stream stream);

/* Per-kernel timing.  When enabled, every kernel launch is bracketed by two
 * CUDA events recorded on the launching stream (event objects come from a
 * host-side pool that the library owns; no device memory is allocated).
 * bdlm_timing_report() waits for the recorded events, accumulates each
 * kernel kind's launch count and total milliseconds, and writes lines
 * "<kernel> <launches> <total_ms>\n" into buf (NUL-terminated, truncated to
 * cap bytes); it returns the number of bytes the full report needs (without
 * the NUL), or -1 on a CUDA error.  reset != 0 clears the totals after the
 * report.  Off by default; enabling it adds two event records per launch. */
bdlm_status bdlm_timing_enable(int on);
int64_t bdlm_timing_report(char* buf, int64_t cap, int reset);

/* Number of kernels this library has launched in this process (all calls,
 * all devices); callers diff it around a region to count launches. */
uint64_t bdlm_kernel_launches(void);

/* Thread-local message describing the last non-OK status on this thread. */
const char* bdlm_last_error(void);

/* Library version string. */
const char* bdlm_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BDLM_ATTN_H */
