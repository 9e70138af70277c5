// abi.cu -- the C ABI declared in include/bdlm_attn.h: argument validation,
// TMA tensor-map encoding, work-list export and kernel launches.
//
// Every entry point validates on the host before enqueuing anything, catches
// every C++ exception, and reports failures as bdlm_status plus a
// thread-local message.  The library allocates no device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <initializer_list>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/bdlm_attn.h"
#include "geometry.cuh"
#include "kernels.h"

using namespace bdlm;

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};

// ---------------------------------------------------------------- timing
enum KernelKind { K_FWD = 0, K_DKV, K_DQ, K_PREP, K_MERGE, K_WATCHDOG, K_COUNT };
const char* const kKindNames[K_COUNT] = {"bdlm_fwd_tc", "bdlm_bwd_dkv", "bdlm_bwd_dq",
                                         "bdlm_preprocess", "bdlm_merge", "bdlm_watchdog"};

struct Timing {
  std::mutex mu;
  std::atomic<bool> on{false};
  std::vector<cudaEvent_t> pool;
  struct Pending {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<Pending> pending;
  double total_ms[K_COUNT] = {};
  uint64_t count[K_COUNT] = {};
};
Timing& timing() {
  static Timing* t = new Timing();  // never destroyed: events may outlive static teardown order
  return *t;
}

cudaEvent_t take_event(Timing& t) {
  if (!t.pool.empty()) {
    cudaEvent_t e = t.pool.back();
    t.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Brackets one kernel launch with events on its stream when timing is on.
struct ScopedKernelTimer {
  int kind;
  cudaStream_t st;
  cudaEvent_t a = nullptr, b = nullptr;
  ScopedKernelTimer(int k, cudaStream_t s) : kind(k), st(s) {
    Timing& t = timing();
    if (!t.on.load()) return;
    std::lock_guard<std::mutex> lock(t.mu);
    a = take_event(t);
    b = take_event(t);
    if (a && b) cudaEventRecord(a, st);
  }
  void stop() {
    if (!a || !b) return;
    Timing& t = timing();
    cudaEventRecord(b, st);
    std::lock_guard<std::mutex> lock(t.mu);
    t.pending.push_back({kind, a, b});
    a = b = nullptr;
  }
  ~ScopedKernelTimer() { stop(); }
};

bdlm_status fail(bdlm_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
bdlm_status fail(bdlm_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

bdlm_status cuda_fail(cudaError_t e, const char* what) {
  return fail(BDLM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr size_t kWsHeader = 256;  // status word, the kernels' work counters, padding
static_assert(kHeaderClearBytes <= (int)kWsHeader, "header words outside the header");

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bdlm_status check_shape(int64_t L, int64_t B, int Hq, int Hkv, int d) {
  if (L <= 0 || B <= 0) return fail(BDLM_ERR_SHAPE, "L=%lld and B=%lld must be positive", (long long)L, (long long)B);
  if (L % B) return fail(BDLM_ERR_SHAPE, "L=%lld is not a multiple of B=%lld", (long long)L, (long long)B);
  if (L > (int64_t)1 << 30) return fail(BDLM_ERR_SHAPE, "L=%lld exceeds 2^30", (long long)L);
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv)
    return fail(BDLM_ERR_SHAPE, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  if (Hq > 4096) return fail(BDLM_ERR_SHAPE, "Hq=%d exceeds 4096", Hq);
  if (d != 64 && d != 128) return fail(BDLM_ERR_SHAPE, "head dim d=%d must be 64 or 128", d);
  return BDLM_OK;
}

bdlm_status check_scale(float scale) {
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(BDLM_ERR_INVALID_ARG, "scale=%g must be finite and > 0", scale);
  return BDLM_OK;
}

#define BDLM_CHECK(expr)            \
  do {                              \
    bdlm_status _s = (expr);        \
    if (_s != BDLM_OK) return _s;   \
  } while (0)

bdlm_status check_ptrs(const char* names, std::initializer_list<const void*> ptrs) {
  int i = 0;
  for (const void* p : ptrs) {
    if (!p) return fail(BDLM_ERR_INVALID_ARG, "null pointer (argument %d of %s)", i, names);
    if (!aligned16(p)) return fail(BDLM_ERR_ALIGN, "pointer not 16-byte aligned (argument %d of %s)", i, names);
    ++i;
  }
  return BDLM_OK;
}

bdlm_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return fail(BDLM_ERR_WORKSPACE, "workspace is null (need %zu bytes)", need);
  if (!aligned16(ws)) return fail(BDLM_ERR_ALIGN, "workspace not 16-byte aligned");
  if (ws_bytes < need) return fail(BDLM_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return BDLM_OK;
}

struct DeviceInfo {
  int sms = 0;
  int major = 0, minor = 0;
};

bdlm_status device_info(DeviceInfo& info) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(BDLM_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    cache[dev].sms = prop.multiProcessorCount;
    cache[dev].major = prop.major;
    cache[dev].minor = prop.minor;
    have[dev] = true;
  }
  info = cache[dev];
  if (info.major != 10 || info.minor != 3)
    return fail(BDLM_ERR_UNSUPPORTED, "device is sm_%d%d; this library is built for sm_103a", info.major, info.minor);
  return BDLM_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bdlm_status get_encoder(EncodeTiledFn& fn) {
  static std::once_flag once;
  static EncodeTiledFn cached = nullptr;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) cached = reinterpret_cast<EncodeTiledFn>(f);
  });
  if (!cached) return fail(BDLM_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
  fn = cached;
  return BDLM_OK;
}

// [L, H, d] bf16 tensor as a 3-D TMA map (d innermost), box 64 x 1 x box_rows,
// 128-byte swizzle; out-of-range rows read as zero.
// box_rows must equal the row count of the shared-memory slot the kernel
// loads the box into (the kernel's expected transaction bytes assume it).
bdlm_status encode_lhd(EncodeTiledFn fn, CUtensorMap* m, const void* ptr, int64_t L, int H, int d,
                       int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)L};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(BDLM_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return BDLM_OK;
}

uint64_t wait_limit_ns() {
  static uint64_t v = [] {
    const char* s = std::getenv("BDLM_WAIT_LIMIT_MS");
    long ms = s ? std::strtol(s, nullptr, 10) : 2000;
    if (ms <= 0) ms = 2000;
    return (uint64_t)ms * 1000000ull;
  }();
  return v;
}

// BDLM_SCHED=naive: work items in natural order, round robin over the grid
// (the load-balancing ablation); otherwise longest first, claimed in list order.
// Read on every call, so one process can time both.
int naive_schedule() {
  const char* s = std::getenv("BDLM_SCHED");
  return (s && std::strcmp(s, "naive") == 0) ? 1 : 0;
}

bdlm_status clear_status(void* ws, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeaderClearBytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status)");
  return BDLM_OK;
}

bdlm_status finish(cudaError_t e, int launches, const char* what) {
  g_launches.fetch_add((uint64_t)launches);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return BDLM_OK;
}

// Query-row ranges of a call: rows[0..1] the clean rows, rows[2..3] the
// corrupted rows, [begin, end) each (validated by the caller).  local: the
// call's tensors hold only its rows (and the clean K / V only the keys
// [kv_begin, kv_end)); else they are full length.
RowRange row_range(const int64_t* rows, int64_t L, bool local, int64_t kv_begin, int64_t kv_end) {
  RowRange r;
  for (int s = 0; s < 2; ++s) {
    r.lo[s] = (int32_t)rows[2 * s];
    r.hi[s] = (int32_t)rows[2 * s + 1];
    r.base[s] = local ? (int32_t)rows[2 * s] : 0;
    r.len[s] = (int32_t)(local ? rows[2 * s + 1] - rows[2 * s] : L);
  }
  r.kbase = local ? (int32_t)kv_begin : 0;
  r.klen = (int32_t)(local ? kv_end - kv_begin : L);
  return r;
}

// Rows a tensor map covers: the held rows (at least one, so that a map over
// a stream with no rows, which no kernel reads, still encodes).
int64_t map_rows(int64_t held) { return held > 0 ? held : 1; }

bdlm_status check_rows(const int64_t* rows, int64_t L) {
  for (int s = 0; s < 2; ++s)
    if (rows[2 * s] < 0 || rows[2 * s + 1] < rows[2 * s] || rows[2 * s + 1] > L)
      return fail(BDLM_ERR_SHAPE, "%s row range [%lld, %lld) is not inside [0, %lld)", s ? "corrupted" : "clean",
                  (long long)rows[2 * s], (long long)rows[2 * s + 1], (long long)L);
  return BDLM_OK;
}

bdlm_status fwd_common(const void* Qc, const void* Kc, const void* Vc, const void* Qn, const void* Kn,
                       const void* Vn, int64_t L, int64_t B, int Hq, int Hkv, int d, float scale, int64_t kv_begin,
                       int64_t kv_end, int include_local, void* Oc, void* On, int o_f32, float* LSEc, float* LSEn,
                       void* ws, size_t ws_bytes, cudaStream_t st, const VarlenTabs* vt = nullptr,
                       const FwdRef* ref = nullptr, const RowRange* rows = nullptr) {
  DeviceInfo info;
  BDLM_CHECK(device_info(info));
  EncodeTiledFn enc;
  BDLM_CHECK(get_encoder(enc));
  FwdMaps maps;
  // rows held by each tensor (a row-restricted call may hold only its own)
  const int64_t hc = rows ? map_rows(rows->len[0]) : L, hn = rows ? map_rows(rows->len[1]) : L;
  const int64_t hk = rows ? map_rows(rows->klen) : L;
  BDLM_CHECK(encode_lhd(enc, &maps.Qc, Qc, hc, Hq, d, kFwdTileQ));
  BDLM_CHECK(encode_lhd(enc, &maps.Qn, Qn, hn, Hq, d, kFwdTileQ));
  BDLM_CHECK(encode_lhd(enc, &maps.Kc, Kc, hk, Hkv, d, kFwdTileK));
  BDLM_CHECK(encode_lhd(enc, &maps.Kn, Kn, hn, Hkv, d, kFwdTileK));
  BDLM_CHECK(encode_lhd(enc, &maps.Vc, Vc, hk, Hkv, d, kFwdTileK));
  BDLM_CHECK(encode_lhd(enc, &maps.Vn, Vn, hn, Hkv, d, kFwdTileK));
  FwdParams p;
  p.g = Geom{L, B, Hq, Hkv, kv_begin, kv_end, include_local ? 1 : 0};
  p.g.naive_order = naive_schedule();
  p.g.round_items = info.sms;  // the persistent grid: one CTA per SM
  p.scale_log2 = scale * 1.4426950408889634f;
  p.Oc = Oc;
  p.On = On;
  p.o_f32 = o_f32;
  p.LSEc = LSEc;
  p.LSEn = LSEn;
  // a row-restricted call lists only the query tiles that hold its rows
  p.n_items = vt ? vt->n_q : rows ? q_items_rows(p.g, *rows, kFwdItemRows) : q_items(p.g, kFwdItemRows);
  p.status = static_cast<uint32_t*>(ws);
  p.limit_ns = wait_limit_ns();
  BDLM_CHECK(clear_status(ws, st));
  int launches = 0;
  ScopedKernelTimer tm(K_FWD, st);
  cudaError_t e = launch_fwd(maps, p, vt, ref, rows, d, info.sms, st, &launches);
  tm.stop();
  return finish(e, launches, "forward launch");
}

BwdParams bwd_params(const void* Qc, const void* Kc, const void* Vc, const void* Qn, const void* Kn, const void* Vn,
                     const void* dOc, const void* dOn, const float* LSEc, const float* LSEn, const float* Dc,
                     const float* Dn, int64_t L, int64_t B, int Hq, int Hkv, int d, float scale, int64_t kv_begin,
                     int64_t kv_end, int include_local, int num_sms) {
  BwdParams p;
  p.g = Geom{L, B, Hq, Hkv, kv_begin, kv_end, include_local ? 1 : 0};
  p.g.naive_order = naive_schedule();
  p.g.round_items = num_sms;  // the persistent grid: one CTA per SM
  p.d = d;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.Qc = Qc; p.Kc = Kc; p.Vc = Vc; p.Qn = Qn; p.Kn = Kn; p.Vn = Vn;
  p.dOc = dOc; p.dOn = dOn;
  p.LSEc = LSEc; p.LSEn = LSEn; p.Dc = Dc; p.Dn = Dn;
  p.dQc = p.dQn = p.dKc = p.dVc = p.dKn = p.dVn = nullptr;
  p.g_f32 = 0;
  p.dq_accumulate = 0;
  p.dkv_accumulate = 0;
  p.rows_call = 0;
  return p;
}

// Launches the dK/dV pass then the dQ pass for the key set of p (vt: item tables of a packed batch, or null).
cudaError_t launch_backward_passes(const BwdParams& p, const DeviceInfo& info, void* ws, cudaStream_t st,
                                   int* launches, bdlm_status* vstatus, const VarlenTabs* vt = nullptr) {
  *vstatus = BDLM_OK;
  EncodeTiledFn enc;
  if ((*vstatus = get_encoder(enc)) != BDLM_OK) return cudaSuccess;
  BwdMaps m;
  const int64_t L = p.g.L;
  const int Hq = p.g.Hq, Hkv = p.g.Hkv, d = p.d;
  // rows held by each tensor (a row-restricted call may hold only its own)
  const bool rc = p.rows_call != 0;
  const int64_t hc = rc ? map_rows(p.rows.len[0]) : L, hn = rc ? map_rows(p.rows.len[1]) : L;
  const int64_t hk = rc ? map_rows(p.rows.klen) : L;
  struct E { CUtensorMap* map; const void* ptr; int H; int64_t rows; };
  const E list[8] = {{&m.Qc, p.Qc, Hq, hc},   {&m.Qn, p.Qn, Hq, hn},   {&m.dOc, p.dOc, Hq, hc},
                     {&m.dOn, p.dOn, Hq, hn}, {&m.Kc, p.Kc, Hkv, hk},  {&m.Kn, p.Kn, Hkv, hn},
                     {&m.Vc, p.Vc, Hkv, hk},  {&m.Vn, p.Vn, Hkv, hn}};
  for (const E& x : list)
    if ((*vstatus = encode_lhd(enc, x.map, x.ptr, x.rows, x.H, d, kBwdTile)) != BDLM_OK) return cudaSuccess;
  uint32_t* status = static_cast<uint32_t*>(ws);
  cudaError_t e;
  {
    ScopedKernelTimer tm(K_DKV, st);
    e = launch_bwd_dkv_tc(m, p, vt, info.sms, status, wait_limit_ns(), st, launches);
  }
  if (e == cudaSuccess) {
    ScopedKernelTimer tm(K_DQ, st);
    e = launch_bwd_dq_tc(m, p, vt, info.sms, status, wait_limit_ns(), st, launches);
  }
  return e;
}

template <typename F>
bdlm_status guarded(F&& f) {
  try {
    return f();
  } catch (const std::exception& ex) {
    return fail(BDLM_ERR_INVALID_ARG, "internal exception: %s", ex.what());
  } catch (...) {
    return fail(BDLM_ERR_INVALID_ARG, "internal exception");
  }
}


// ------------------------------------------------------------ packed batch
// Sequence s owns rows [off[s], off[s+1]) of the packed tensors; the kernels
// read their items from tables in the workspace (see varlen_tables below).
constexpr int64_t kMaxSeqs = 1 << 20;

bdlm_status check_varlen(const int64_t* off, int n, int64_t B, int Hq, int Hkv, int d, int64_t* T) {
  if (!off) return fail(BDLM_ERR_INVALID_ARG, "seq_offsets is null");
  if (n <= 0 || n > kMaxSeqs) return fail(BDLM_ERR_SHAPE, "n_seqs=%d must be in [1, 2^20]", n);
  if (off[0] != 0) return fail(BDLM_ERR_SHAPE, "seq_offsets[0]=%lld must be 0", (long long)off[0]);
  for (int s = 0; s < n; ++s) {
    const int64_t len = off[s + 1] - off[s];
    if (len <= 0 || (B > 0 && len % B))
      return fail(BDLM_ERR_SHAPE, "sequence %d has length %lld: must be a positive multiple of B=%lld", s,
                  (long long)len, (long long)B);
  }
  *T = off[n];
  return check_shape(*T, B > 0 ? B : *T, Hq, Hkv, d);
}

int64_t varlen_q_count(const int64_t* off, int n, int Hq, int tq) {
  int64_t c = 0;
  for (int s = 0; s < n; ++s) c += cdiv64(off[s + 1] - off[s], tq) * Hq * 2;
  return c;
}

int64_t varlen_kv_count(const int64_t* off, int n, int Hkv, int tk) {
  int64_t c = 0;
  for (int s = 0; s < n; ++s) c += cdiv64(off[s + 1] - off[s], tk) * 2 * Hkv;
  return c;
}

// Order of a packed batch's items.  Default: one sequence after the other,
// longest sequence first, each in its one-sequence order (the items running
// together then read one sequence's keys), expanded on the device from a
// per-sequence directory.  BDLM_VARLEN_ORDER=lpt (ablation): longest item
// first over all sequences, tables built on the host.
bool varlen_lpt_order() {
  const char* s = std::getenv("BDLM_VARLEN_ORDER");
  return s && std::strcmp(s, "lpt") == 0;
}

// {sequence, stream + 2 * head, query tile, visible key tiles}, longest first
std::vector<int4> varlen_q_table(const Geom& all, const int64_t* off, int n, int tq, int tk) {
  std::vector<int4> v;
  v.reserve((size_t)varlen_q_count(off, n, all.Hq, tq));
  for (int s = 0; s < n; ++s) {
    const Geom g = seq_geom(all, off[s + 1] - off[s]);
    const int64_t nqt = cdiv64(g.L, tq);
    for (int64_t qt = 0; qt < nqt; ++qt)
      for (int h = 0; h < g.Hq; ++h)
        for (int st = 0; st < 2; ++st) {
          const int64_t r0 = qt * tq, r1 = imin64(r0 + tq, g.L);
          const QTileRanges q = qtile_ranges(g, st, r0, r1, tk);
          v.push_back(make_int4(s, st + 2 * h, (int)qt, (int)((q.c1 - q.c0) + (q.n1 - q.n0))));
        }
  }
  std::stable_sort(v.begin(), v.end(), [](const int4& a, const int4& b) { return a.w > b.w; });
  return v;
}

// {sequence, key stream + 2 * KV head, key tile, query rows that see it}, longest first
std::vector<int4> varlen_kv_table(const Geom& all, const int64_t* off, int n, int tk) {
  std::vector<int4> v;
  v.reserve((size_t)varlen_kv_count(off, n, all.Hkv, tk));
  for (int s = 0; s < n; ++s) {
    const Geom g = seq_geom(all, off[s + 1] - off[s]);
    const int64_t nt = cdiv64(g.L, tk);
    for (int ks = 0; ks < 2; ++ks)
      for (int h = 0; h < g.Hkv; ++h)
        for (int64_t kt = 0; kt < nt; ++kt) {
          int64_t cl, ch, nl, nh;
          kv_tile_rows(g, ks, kt * tk, imin64(kt * tk + tk, g.L), cl, ch, nl, nh);
          const int64_t rows = imax64(0, ch - cl) + imax64(0, nh - nl);
          v.push_back(make_int4(s, ks + 2 * h, (int)kt, (int)rows));
        }
  }
  std::stable_sort(v.begin(), v.end(), [](const int4& a, const int4& b) { return a.w > b.w; });
  return v;
}

// Directory of a packed batch, uploaded as one int64 array:
//   [0, n]        sequence offsets (as given)
//   [n+1, 2n+1]   first query item of each sequence in directory order (+ total)
//   [2n+2, 3n+2]  first key item of each sequence in directory order (+ total)
//   [3n+3, 4n+2]  sequence ids, longest first (ties: lower id first)
std::vector<int64_t> varlen_directory(const Geom& all, const int64_t* off, int n, int tq, int tk) {
  std::vector<int64_t> v((size_t)(4 * n + 3));
  int64_t* o = v.data();
  int64_t* qb = o + n + 1;
  int64_t* kb = qb + n + 1;
  int64_t* ord = kb + n + 1;
  for (int s = 0; s <= n; ++s) o[s] = off[s];
  std::vector<int> idx(n);
  for (int s = 0; s < n; ++s) idx[s] = s;
  std::stable_sort(idx.begin(), idx.end(),
                   [off](int a, int b) { return off[a + 1] - off[a] > off[b + 1] - off[b]; });
  qb[0] = kb[0] = 0;
  for (int k = 0; k < n; ++k) {
    const int s = idx[k];
    const Geom g = seq_geom(all, off[s + 1] - off[s]);
    ord[k] = s;
    qb[k + 1] = qb[k] + q_items(g, tq);
    kb[k + 1] = kb[k] + kv_items(g, tk);
  }
  return v;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of a packed-batch call: header, [D of both streams], directory, item tables.
struct VarlenLayout {
  size_t d_bytes, dir_at, q_at, kv_at, total;
};
VarlenLayout varlen_layout(int op, const int64_t* off, int n, int Hq, int Hkv, int64_t T) {
  VarlenLayout l;
  l.d_bytes = op == BDLM_OP_BWD ? round256(2 * (size_t)Hq * (size_t)T * sizeof(float)) : 0;
  l.dir_at = kWsHeader + l.d_bytes;
  l.q_at = l.dir_at + round256((size_t)(4 * n + 3) * sizeof(int64_t));
  const int64_t nq = op == BDLM_OP_BWD ? varlen_q_count(off, n, Hq, kBwdTile) : varlen_q_count(off, n, Hq, kFwdItemRows);
  l.kv_at = l.q_at + round256((size_t)nq * sizeof(int4));
  const int64_t nkv = op == BDLM_OP_BWD ? varlen_kv_count(off, n, Hkv, kBwdTile) : 0;
  l.total = l.kv_at + round256((size_t)nkv * sizeof(int4));
  return l;
}

// Host -> device copy on the stream; the caller keeps `src` alive until the
// copy has run.
bdlm_status upload(void* dst, const void* src, size_t bytes, cudaStream_t st) {
  if (!bytes) return BDLM_OK;
  cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(work list)");
  return BDLM_OK;
}

// Uploads the directory of a packed batch and fills its item tables (query
// items with tiles of tq rows; key items too when with_kv), on the stream.
// Host arrays of a packed-batch call, kept alive until their copies to the
// device have run: a copy from pageable memory may still read its source
// after cudaMemcpyAsync returns, so a host function enqueued behind the
// copies frees them.
struct VarlenHostArrays {
  std::vector<int64_t> dir;
  std::vector<int4> q, kv;
};
void CUDART_CB free_varlen_host_arrays(void* p) { delete static_cast<VarlenHostArrays*>(p); }

bdlm_status varlen_tables(const Geom& all, const int64_t* off, int n, int tq, bool with_kv, const VarlenLayout& lay,
                          char* w, cudaStream_t st, int* launches, VarlenTabs* vt) {
  const int tk = kBwdTile;  // key tiles: 128 keys in every pass
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone)
    return fail(BDLM_ERR_UNSUPPORTED, "packed-batch calls copy host arrays and cannot be captured into a graph");
  VarlenHostArrays* h = new VarlenHostArrays;
  h->dir = varlen_directory(all, off, n, tq, tk);
  const int64_t* d_dir = reinterpret_cast<const int64_t*>(w + lay.dir_at);
  int4* q_tab = reinterpret_cast<int4*>(w + lay.q_at);
  int4* kv_tab = reinterpret_cast<int4*>(w + lay.kv_at);
  const int64_t nq = h->dir[2 * (size_t)n + 1], nkv = with_kv ? h->dir[3 * (size_t)n + 2] : 0;
  bdlm_status s = upload(w + lay.dir_at, h->dir.data(), h->dir.size() * sizeof(int64_t), st);
  if (s == BDLM_OK && varlen_lpt_order()) {
    h->q = varlen_q_table(all, off, n, tq, tk);
    s = upload(q_tab, h->q.data(), h->q.size() * sizeof(int4), st);
    if (s == BDLM_OK && with_kv) {
      h->kv = varlen_kv_table(all, off, n, tk);
      s = upload(kv_tab, h->kv.data(), h->kv.size() * sizeof(int4), st);
    }
  }
  // free the host arrays behind the copies (or at once if nothing is in flight)
  e = cudaLaunchHostFunc(st, free_varlen_host_arrays, h);
  if (e != cudaSuccess) {
    cudaStreamSynchronize(st);
    delete h;
    return s != BDLM_OK ? s : cuda_fail(e, "cudaLaunchHostFunc");
  }
  if (s != BDLM_OK) return s;
  if (!varlen_lpt_order()) {
    const int64_t* ord = d_dir + 3 * (size_t)n + 3;
    e = launch_varlen_items(all, d_dir, ord, d_dir + n + 1, n, nq, 0, tq, tk, q_tab, st, launches);
    if (e == cudaSuccess && with_kv)
      e = launch_varlen_items(all, d_dir, ord, d_dir + 2 * (size_t)n + 2, n, nkv, 1, tq, tk, kv_tab, st, launches);
    if (e != cudaSuccess) return cuda_fail(e, "packed-batch item tables");
  }
  *vt = VarlenTabs{q_tab, with_kv ? kv_tab : nullptr, d_dir, nq, nkv};
  return BDLM_OK;
}

}  // namespace

void bdlm::set_last_error(const std::string& msg) { g_last_error = msg; }

extern "C" {

size_t bdlm_workspace_size(int op, int64_t L, int64_t B, int Hq, int Hkv, int d, int P) {
  (void)P;
  if (check_shape(L, B, Hq, Hkv, d) != BDLM_OK) return 0;
  switch (op) {
    case BDLM_OP_FWD:
    case BDLM_OP_FWD_SHARD:
    case BDLM_OP_BWD_SHARD:
      return kWsHeader;
    case BDLM_OP_BWD:
      return kWsHeader + 2 * (size_t)Hq * (size_t)L * sizeof(float);
    default:
      return 0;
  }
}

bdlm_status bdlm_attn_fwd(const void* Qc, const void* Kc, const void* Vc, const void* Qn, const void* Kn,
                          const void* Vn, int64_t L, int64_t B, int Hq, int Hkv, int d, float scale, void* Oc,
                          void* On, bdlm_dtype o_dtype, float* LSEc, float* LSEn, void* workspace, size_t ws_bytes,
                          bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    BDLM_CHECK(check_shape(L, B, Hq, Hkv, d));
    BDLM_CHECK(check_scale(scale));
    if (o_dtype != BDLM_BF16 && o_dtype != BDLM_F32) return fail(BDLM_ERR_INVALID_ARG, "bad o_dtype %d", (int)o_dtype);
    BDLM_CHECK(check_ptrs("bdlm_attn_fwd(Qc,Kc,Vc,Qn,Kn,Vn,Oc,On,LSEc,LSEn)",
                          {Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, LSEc, LSEn}));
    BDLM_CHECK(check_ws(workspace, ws_bytes, bdlm_workspace_size(BDLM_OP_FWD, L, B, Hq, Hkv, d, 1)));
    return fwd_common(Qc, Kc, Vc, Qn, Kn, Vn, L, B, Hq, Hkv, d, scale, 0, L, 1, Oc, On, o_dtype == BDLM_F32, LSEc,
                      LSEn, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
  });
}

bdlm_status bdlm_attn_fwd_shard(const void* Qc, const void* Kc, const void* Vc, const void* Qn, const void* Kn,
                                const void* Vn, int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                                int64_t kv_begin, int64_t kv_end, int include_local, float* Op_c, float* Op_n,
                                float* LSEp_c, float* LSEp_n, void* workspace, size_t ws_bytes, bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    BDLM_CHECK(check_shape(L, B, Hq, Hkv, d));
    BDLM_CHECK(check_scale(scale));
    if (kv_begin < 0 || kv_end < kv_begin || kv_end > L)
      return fail(BDLM_ERR_SHAPE, "clean key range [%lld, %lld) is not inside [0, %lld)", (long long)kv_begin,
                  (long long)kv_end, (long long)L);
    BDLM_CHECK(check_ptrs("bdlm_attn_fwd_shard(Qc,Kc,Vc,Qn,Kn,Vn,Op_c,Op_n,LSEp_c,LSEp_n)",
                          {Qc, Kc, Vc, Qn, Kn, Vn, Op_c, Op_n, LSEp_c, LSEp_n}));
    BDLM_CHECK(check_ws(workspace, ws_bytes, bdlm_workspace_size(BDLM_OP_FWD_SHARD, L, B, Hq, Hkv, d, 1)));
    return fwd_common(Qc, Kc, Vc, Qn, Kn, Vn, L, B, Hq, Hkv, d, scale, kv_begin, kv_end, include_local, Op_c, Op_n,
                      1, LSEp_c, LSEp_n, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
  });
}

bdlm_status bdlm_attn_fwd_shard_refmax(const void* Qc, const void* Kc, const void* Vc, const void* Qn,
                                       const void* Kn, const void* Vn, int64_t L, int64_t B, int Hq, int Hkv, int d,
                                       float scale, int64_t kv_begin, int64_t kv_end, int include_local,
                                       const float* Mref_c, const float* Mref_n, float* Op_c, float* Op_n,
                                       float* LSEp_c, float* LSEp_n, void* workspace, size_t ws_bytes,
                                       bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    BDLM_CHECK(check_shape(L, B, Hq, Hkv, d));
    BDLM_CHECK(check_scale(scale));
    if (kv_begin < 0 || kv_end < kv_begin || kv_end > L)
      return fail(BDLM_ERR_SHAPE, "clean key range [%lld, %lld) is not inside [0, %lld)", (long long)kv_begin,
                  (long long)kv_end, (long long)L);
    BDLM_CHECK(check_ptrs("bdlm_attn_fwd_shard_refmax(Qc,Kc,Vc,Qn,Kn,Vn,Mref_c,Mref_n,Op_c,Op_n,LSEp_c,LSEp_n)",
                          {Qc, Kc, Vc, Qn, Kn, Vn, Mref_c, Mref_n, Op_c, Op_n, LSEp_c, LSEp_n}));
    BDLM_CHECK(check_ws(workspace, ws_bytes, bdlm_workspace_size(BDLM_OP_FWD_SHARD, L, B, Hq, Hkv, d, 1)));
    const FwdRef ref{Mref_c, Mref_n};
    return fwd_common(Qc, Kc, Vc, Qn, Kn, Vn, L, B, Hq, Hkv, d, scale, kv_begin, kv_end, include_local, Op_c, Op_n,
                      1, LSEp_c, LSEp_n, workspace, ws_bytes, static_cast<cudaStream_t>(stream), nullptr, &ref);
  });
}

}  // extern "C"

namespace {

// The clean key range and, for rank-local tensors with the local partial,
// whole corrupted blocks (a corrupted row reads its whole block's keys, which
// the rank's corrupted K / V must hold).
bdlm_status check_rows_call(int64_t L, int64_t B, int64_t kv_begin, int64_t kv_end, int include_local,
                            const int64_t* rows, bool local) {
  if (kv_begin < 0 || kv_end < kv_begin || kv_end > L)
    return fail(BDLM_ERR_SHAPE, "clean key range [%lld, %lld) is not inside [0, %lld)", (long long)kv_begin,
                (long long)kv_end, (long long)L);
  BDLM_CHECK(check_rows(rows, L));
  if (local && include_local && rows[3] > rows[2] && (rows[2] % B || (rows[3] % B && rows[3] != L)))
    return fail(BDLM_ERR_SHAPE,
                "rank-local corrupted rows [%lld, %lld) must be whole blocks of %lld (their keys are read)",
                (long long)rows[2], (long long)rows[3], (long long)B);
  return BDLM_OK;
}

bdlm_status fwd_rows_impl(const char* name, const void* Qc, const void* Kc, const void* Vc, const void* Qn,
                          const void* Kn, const void* Vn, int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                          int64_t kv_begin, int64_t kv_end, int include_local, const int64_t* rows, bool local,
                          float* Op_c, float* Op_n, float* LSEp_c, float* LSEp_n, void* workspace, size_t ws_bytes,
                          bdlm_stream stream) {
  BDLM_CHECK(check_shape(L, B, Hq, Hkv, d));
  BDLM_CHECK(check_scale(scale));
  BDLM_CHECK(check_rows_call(L, B, kv_begin, kv_end, include_local, rows, local));
  BDLM_CHECK(check_ptrs(name, {Qc, Kc, Vc, Qn, Kn, Vn, Op_c, Op_n, LSEp_c, LSEp_n}));
  BDLM_CHECK(check_ws(workspace, ws_bytes, bdlm_workspace_size(BDLM_OP_FWD_SHARD, L, B, Hq, Hkv, d, 1)));
  const RowRange rr = row_range(rows, L, local, kv_begin, kv_end);
  return fwd_common(Qc, Kc, Vc, Qn, Kn, Vn, L, B, Hq, Hkv, d, scale, kv_begin, kv_end, include_local, Op_c, Op_n, 1,
                    LSEp_c, LSEp_n, workspace, ws_bytes, static_cast<cudaStream_t>(stream), nullptr, nullptr, &rr);
}

bdlm_status bwd_rows_impl(const char* name, const void* Qc, const void* Kc, const void* Vc, const void* Qn,
                          const void* Kn, const void* Vn, const void* dOc, const void* dOn, const float* LSEc,
                          const float* LSEn, const float* Dc, const float* Dn, int64_t L, int64_t B, int Hq, int Hkv,
                          int d, float scale, int64_t kv_begin, int64_t kv_end, int include_local,
                          const int64_t* rows, bool local, float* dQc_acc, float* dQn_acc, float* dKc_acc,
                          float* dVc_acc, float* dKn_acc, float* dVn_acc, void* workspace, size_t ws_bytes,
                          bdlm_stream stream) {
  BDLM_CHECK(check_shape(L, B, Hq, Hkv, d));
  BDLM_CHECK(check_scale(scale));
  BDLM_CHECK(check_rows_call(L, B, kv_begin, kv_end, include_local, rows, local));
  BDLM_CHECK(check_ptrs(name, {Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn}));
  BDLM_CHECK(check_ptrs(name, {dQc_acc, dQn_acc, dKc_acc, dVc_acc, dKn_acc, dVn_acc}));
  BDLM_CHECK(check_ws(workspace, ws_bytes, bdlm_workspace_size(BDLM_OP_BWD_SHARD, L, B, Hq, Hkv, d, 1)));
  DeviceInfo info;
  BDLM_CHECK(device_info(info));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  BDLM_CHECK(clear_status(workspace, st));
  BwdParams p = bwd_params(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn, L, B, Hq, Hkv, d, scale, kv_begin,
                           kv_end, include_local, info.sms);
  p.rows = row_range(rows, L, local, kv_begin, kv_end);
  p.rows_call = 1;
  p.dQc = dQc_acc; p.dQn = dQn_acc; p.dKc = dKc_acc; p.dVc = dVc_acc; p.dKn = dKn_acc; p.dVn = dVn_acc;
  p.g_f32 = 1;
  p.dq_accumulate = 1;
  p.dkv_accumulate = 1;
  int launches = 0;
  bdlm_status vs = BDLM_OK;
  cudaError_t e = launch_backward_passes(p, info, workspace, st, &launches, &vs);
  if (vs != BDLM_OK) return vs;
  return finish(e, launches, "row-restricted backward launch");
}

}  // namespace

extern "C" {

bdlm_status bdlm_attn_fwd_shard_rows(const void* Qc, const void* Kc, const void* Vc, const void* Qn,
                                     const void* Kn, const void* Vn, int64_t L, int64_t B, int Hq, int Hkv, int d,
                                     float scale, int64_t kv_begin, int64_t kv_end, int include_local,
                                     int64_t rows_c_begin, int64_t rows_c_end, int64_t rows_n_begin,
                                     int64_t rows_n_end, float* Op_c, float* Op_n, float* LSEp_c, float* LSEp_n,
                                     void* workspace, size_t ws_bytes, bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    const int64_t rows[4] = {rows_c_begin, rows_c_end, rows_n_begin, rows_n_end};
    return fwd_rows_impl("bdlm_attn_fwd_shard_rows(Qc,Kc,Vc,Qn,Kn,Vn,Op_c,Op_n,LSEp_c,LSEp_n)", Qc, Kc, Vc, Qn, Kn,
                         Vn, L, B, Hq, Hkv, d, scale, kv_begin, kv_end, include_local, rows, false, Op_c, Op_n,
                         LSEp_c, LSEp_n, workspace, ws_bytes, stream);
  });
}

bdlm_status bdlm_attn_fwd_rank(const void* Qc, const void* Kc, const void* Vc, const void* Qn, const void* Kn,
                               const void* Vn, int64_t L, int64_t B, int Hq, int Hkv, int d, float scale,
                               int64_t kv_begin, int64_t kv_end, int include_local, int64_t rows_c_begin,
                               int64_t rows_c_end, int64_t rows_n_begin, int64_t rows_n_end, float* Op_c,
                               float* Op_n, float* LSEp_c, float* LSEp_n, void* workspace, size_t ws_bytes,
                               bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    const int64_t rows[4] = {rows_c_begin, rows_c_end, rows_n_begin, rows_n_end};
    return fwd_rows_impl("bdlm_attn_fwd_rank(Qc,Kc,Vc,Qn,Kn,Vn,Op_c,Op_n,LSEp_c,LSEp_n)", Qc, Kc, Vc, Qn, Kn, Vn, L,
                         B, Hq, Hkv, d, scale, kv_begin, kv_end, include_local, rows, true, Op_c, Op_n, LSEp_c,
                         LSEp_n, workspace, ws_bytes, stream);
  });
}

bdlm_status bdlm_lse_merge(int n_parts, const float* const* O_parts, const float* const* LSE_parts, int64_t rows,
                           int H, int d, void* O, bdlm_dtype o_dtype, float* LSE, bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    if (n_parts < 1 || n_parts > kMaxParts)
      return fail(BDLM_ERR_INVALID_ARG, "n_parts=%d must be in [1, %d]", n_parts, kMaxParts);
    if (!O_parts || !LSE_parts) return fail(BDLM_ERR_INVALID_ARG, "null partial pointer array");
    if (rows <= 0 || H <= 0) return fail(BDLM_ERR_SHAPE, "rows=%lld and H=%d must be positive", (long long)rows, H);
    if (d != 64 && d != 128) return fail(BDLM_ERR_SHAPE, "head dim d=%d must be 64 or 128", d);
    if (o_dtype != BDLM_BF16 && o_dtype != BDLM_F32) return fail(BDLM_ERR_INVALID_ARG, "bad o_dtype %d", (int)o_dtype);
    BDLM_CHECK(check_ptrs("bdlm_lse_merge(O)", {O}));
    if (LSE && !aligned16(LSE)) return fail(BDLM_ERR_ALIGN, "LSE output not 16-byte aligned");
    MergeParams p;
    for (int i = 0; i < n_parts; ++i) {
      BDLM_CHECK(check_ptrs("bdlm_lse_merge(O_parts[i], LSE_parts[i])", {O_parts[i], LSE_parts[i]}));
      p.O[i] = O_parts[i];
      p.LSE[i] = LSE_parts[i];
    }
    for (int i = n_parts; i < kMaxParts; ++i) p.O[i] = p.LSE[i] = nullptr;
    DeviceInfo info;
    BDLM_CHECK(device_info(info));
    p.n = n_parts;
    p.rows = rows;
    p.H = H;
    p.d = d;
    p.out = O;
    p.out_f32 = o_dtype == BDLM_F32;
    p.lse_out = LSE;
    int launches = 0;
    ScopedKernelTimer tm(K_MERGE, static_cast<cudaStream_t>(stream));
    cudaError_t e = launch_merge(p, static_cast<cudaStream_t>(stream), &launches);
    tm.stop();
    return finish(e, launches, "merge launch");
  });
}

bdlm_status bdlm_bwd_preprocess(const void* O, bdlm_dtype o_dtype, const void* dO, int64_t rows, int H, int d,
                                float* D, bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    if (rows <= 0 || H <= 0) return fail(BDLM_ERR_SHAPE, "rows=%lld and H=%d must be positive", (long long)rows, H);
    if (d != 64 && d != 128) return fail(BDLM_ERR_SHAPE, "head dim d=%d must be 64 or 128", d);
    if (o_dtype != BDLM_BF16 && o_dtype != BDLM_F32) return fail(BDLM_ERR_INVALID_ARG, "bad o_dtype %d", (int)o_dtype);
    BDLM_CHECK(check_ptrs("bdlm_bwd_preprocess(O,dO,D)", {O, dO, D}));
    DeviceInfo info;
    BDLM_CHECK(device_info(info));
    int launches = 0;
    ScopedKernelTimer tm(K_PREP, static_cast<cudaStream_t>(stream));
    cudaError_t e = launch_preprocess(O, o_dtype == BDLM_F32, dO, rows, H, d, D, static_cast<cudaStream_t>(stream),
                                      &launches, info.sms);
    tm.stop();
    return finish(e, launches, "preprocess launch");
  });
}

bdlm_status bdlm_attn_bwd(const void* Qc, const void* Kc, const void* Vc, const void* Qn, const void* Kn,
                          const void* Vn, const void* Oc, const void* On, const void* dOc, const void* dOn,
                          const float* LSEc, const float* LSEn, int64_t L, int64_t B, int Hq, int Hkv, int d,
                          float scale, void* dQc, void* dKc, void* dVc, void* dQn, void* dKn, void* dVn,
                          bdlm_dtype g_dtype, void* workspace, size_t ws_bytes, bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    BDLM_CHECK(check_shape(L, B, Hq, Hkv, d));
    BDLM_CHECK(check_scale(scale));
    if (g_dtype != BDLM_BF16 && g_dtype != BDLM_F32) return fail(BDLM_ERR_INVALID_ARG, "bad g_dtype %d", (int)g_dtype);
    BDLM_CHECK(check_ptrs("bdlm_attn_bwd(Qc,Kc,Vc,Qn,Kn,Vn,Oc,On,dOc,dOn,LSEc,LSEn)",
                          {Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, dOc, dOn, LSEc, LSEn}));
    BDLM_CHECK(check_ptrs("bdlm_attn_bwd(dQc,dKc,dVc,dQn,dKn,dVn)", {dQc, dKc, dVc, dQn, dKn, dVn}));
    BDLM_CHECK(check_ws(workspace, ws_bytes, bdlm_workspace_size(BDLM_OP_BWD, L, B, Hq, Hkv, d, 1)));
    DeviceInfo info;
    BDLM_CHECK(device_info(info));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float* Dc = reinterpret_cast<float*>(static_cast<char*>(workspace) + kWsHeader);
    float* Dn = Dc + (size_t)Hq * L;
    BDLM_CHECK(clear_status(workspace, st));
    int launches = 0;
    cudaError_t e;
    {
      ScopedKernelTimer tm(K_PREP, st);
      e = launch_preprocess(Oc, 0, dOc, L, Hq, d, Dc, st, &launches, info.sms);
    }
    if (e == cudaSuccess) {
      ScopedKernelTimer tm(K_PREP, st);
      e = launch_preprocess(On, 0, dOn, L, Hq, d, Dn, st, &launches, info.sms);
    }
    BwdParams p = bwd_params(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn, L, B, Hq, Hkv, d, scale, 0, L, 1,
                             info.sms);
    p.dQc = dQc; p.dQn = dQn; p.dKc = dKc; p.dVc = dVc; p.dKn = dKn; p.dVn = dVn;
    p.g_f32 = g_dtype == BDLM_F32;
    bdlm_status vs = BDLM_OK;
    if (e == cudaSuccess) e = launch_backward_passes(p, info, workspace, st, &launches, &vs);
    if (vs != BDLM_OK) return vs;
    return finish(e, launches, "backward launch");
  });
}

bdlm_status bdlm_attn_bwd_shard(const void* Qc, const void* Kc, const void* Vc, const void* Qn, const void* Kn,
                                const void* Vn, const void* dOc, const void* dOn, const float* LSEc,
                                const float* LSEn, const float* Dc, const float* Dn, int64_t L, int64_t B, int Hq,
                                int Hkv, int d, float scale, int64_t kv_begin, int64_t kv_end, int include_local,
                                float* dQc_acc, float* dQn_acc, float* dKc, float* dVc, float* dKn, float* dVn,
                                void* workspace, size_t ws_bytes, bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    BDLM_CHECK(check_shape(L, B, Hq, Hkv, d));
    BDLM_CHECK(check_scale(scale));
    if (kv_begin < 0 || kv_end < kv_begin || kv_end > L)
      return fail(BDLM_ERR_SHAPE, "clean key range [%lld, %lld) is not inside [0, %lld)", (long long)kv_begin,
                  (long long)kv_end, (long long)L);
    BDLM_CHECK(check_ptrs("bdlm_attn_bwd_shard(Qc,Kc,Vc,Qn,Kn,Vn,dOc,dOn,LSEc,LSEn,Dc,Dn)",
                          {Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn}));
    BDLM_CHECK(check_ptrs("bdlm_attn_bwd_shard(dQc_acc,dQn_acc,dKc,dVc,dKn,dVn)",
                          {dQc_acc, dQn_acc, dKc, dVc, dKn, dVn}));
    BDLM_CHECK(check_ws(workspace, ws_bytes, bdlm_workspace_size(BDLM_OP_BWD_SHARD, L, B, Hq, Hkv, d, 1)));
    DeviceInfo info;
    BDLM_CHECK(device_info(info));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    BDLM_CHECK(clear_status(workspace, st));
    BwdParams p = bwd_params(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn, L, B, Hq, Hkv, d, scale, kv_begin,
                             kv_end, include_local, info.sms);
    p.dQc = dQc_acc; p.dQn = dQn_acc; p.dKc = dKc; p.dVc = dVc; p.dKn = dKn; p.dVn = dVn;
    p.g_f32 = 1;
    p.dq_accumulate = 1;
    int launches = 0;
    bdlm_status vs = BDLM_OK;
    cudaError_t e = launch_backward_passes(p, info, workspace, st, &launches, &vs);
    if (vs != BDLM_OK) return vs;
    return finish(e, launches, "sharded backward launch");
  });
}

bdlm_status bdlm_attn_bwd_shard_rows(const void* Qc, const void* Kc, const void* Vc, const void* Qn,
                                     const void* Kn, const void* Vn, const void* dOc, const void* dOn,
                                     const float* LSEc, const float* LSEn, const float* Dc, const float* Dn, int64_t L,
                                     int64_t B, int Hq, int Hkv, int d, float scale, int64_t kv_begin,
                                     int64_t kv_end, int include_local, int64_t rows_c_begin, int64_t rows_c_end,
                                     int64_t rows_n_begin, int64_t rows_n_end, float* dQc_acc, float* dQn_acc,
                                     float* dKc_acc, float* dVc_acc, float* dKn_acc, float* dVn_acc, void* workspace,
                                     size_t ws_bytes, bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    const int64_t rows[4] = {rows_c_begin, rows_c_end, rows_n_begin, rows_n_end};
    return bwd_rows_impl("bdlm_attn_bwd_shard_rows(tensors, accumulators)", Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc,
                         LSEn, Dc, Dn, L, B, Hq, Hkv, d, scale, kv_begin, kv_end, include_local, rows, false, dQc_acc,
                         dQn_acc, dKc_acc, dVc_acc, dKn_acc, dVn_acc, workspace, ws_bytes, stream);
  });
}

bdlm_status bdlm_attn_bwd_rank(const void* Qc, const void* Kc, const void* Vc, const void* Qn, const void* Kn,
                               const void* Vn, const void* dOc, const void* dOn, const float* LSEc,
                               const float* LSEn, const float* Dc, const float* Dn, int64_t L, int64_t B, int Hq,
                               int Hkv, int d, float scale, int64_t kv_begin, int64_t kv_end, int include_local,
                               int64_t rows_c_begin, int64_t rows_c_end, int64_t rows_n_begin, int64_t rows_n_end,
                               float* dQc_acc, float* dQn_acc, float* dKc_acc, float* dVc_acc, float* dKn_acc,
                               float* dVn_acc, void* workspace, size_t ws_bytes, bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    const int64_t rows[4] = {rows_c_begin, rows_c_end, rows_n_begin, rows_n_end};
    return bwd_rows_impl("bdlm_attn_bwd_rank(tensors, accumulators)", Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn,
                         Dc, Dn, L, B, Hq, Hkv, d, scale, kv_begin, kv_end, include_local, rows, true, dQc_acc,
                         dQn_acc, dKc_acc, dVc_acc, dKn_acc, dVn_acc, workspace, ws_bytes, stream);
  });
}

int64_t bdlm_worklist(int64_t L, int64_t B, int Hq, int Hkv, int tile_q, int tile_k, int64_t kv_begin,
                      int64_t kv_end, int include_local, int32_t* out, int64_t cap) {
  try {
    if (L <= 0 || B <= 0 || L % B || Hq <= 0 || Hkv <= 0 || Hq % Hkv || tile_q <= 0 || tile_k <= 0) return -1;
    if (kv_begin < 0 || kv_end < kv_begin || kv_end > L) return -1;
    if (cap > 0 && !out) return -1;
    Geom g{L, B, Hq, Hkv, kv_begin, kv_end, include_local ? 1 : 0};
    g.naive_order = naive_schedule();
    const int64_t n = q_items(g, tile_q);
    for (int64_t i = 0; i < n && i < cap; ++i) {
      const QItem it = q_item(g, tile_q, i);
      const int64_t r0 = it.qtile * tile_q, r1 = imin64(r0 + tile_q, L);
      const QTileRanges q = qtile_ranges(g, it.stream, r0, r1, tile_k);
      int32_t* o = out + 8 * i;
      o[0] = it.stream;
      o[1] = it.head;
      o[2] = (int32_t)it.qtile;
      o[3] = (int32_t)q.c0;
      o[4] = (int32_t)q.c1;
      o[5] = (int32_t)q.n0;
      o[6] = (int32_t)q.n1;
      o[7] = (int32_t)((q.c1 - q.c0) + (q.n1 - q.n0));
    }
    return n;
  } catch (...) {
    return -1;
  }
}

bdlm_status bdlm_sync_status(void* workspace, bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    if (!workspace) return fail(BDLM_ERR_WORKSPACE, "workspace is null");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t word = 0;
    e = cudaMemcpy(&word, workspace, 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
    e = cudaMemset(workspace, 0, 4);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
    if (word != 0)
      return fail(BDLM_ERR_TIMEOUT, "device wait limit expired (status 0x%x, wait site %u)", word, word & 0xffu);
    return BDLM_OK;
  });
}

bdlm_status bdlm_watchdog_selftest(void* workspace, size_t ws_bytes, uint32_t limit_us, bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    BDLM_CHECK(check_ws(workspace, ws_bytes, kWsHeader));
    if (limit_us == 0 || limit_us > 10000000u) return fail(BDLM_ERR_INVALID_ARG, "limit_us=%u out of (0, 1e7]", limit_us);
    DeviceInfo info;
    BDLM_CHECK(device_info(info));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    BDLM_CHECK(clear_status(workspace, st));
    cudaError_t e = launch_watchdog(static_cast<uint32_t*>(workspace), (uint64_t)limit_us * 1000ull, st);
    g_launches.fetch_add(1);
    if (e != cudaSuccess) return cuda_fail(e, "watchdog launch");
    return bdlm_sync_status(workspace, stream);
  });
}

bdlm_status bdlm_timing_enable(int on) {
  timing().on.store(on != 0);
  return BDLM_OK;
}

int64_t bdlm_timing_report(char* buf, int64_t cap, int reset) {
  try {
    Timing& t = timing();
    std::lock_guard<std::mutex> lock(t.mu);
    bool cuda_ok = true;
    for (auto& pd : t.pending) {
      float ms = 0.f;
      if (cudaEventSynchronize(pd.b) != cudaSuccess || cudaEventElapsedTime(&ms, pd.a, pd.b) != cudaSuccess)
        cuda_ok = false;
      t.total_ms[pd.kind] += ms;
      t.count[pd.kind] += 1;
      t.pool.push_back(pd.a);
      t.pool.push_back(pd.b);
    }
    t.pending.clear();
    std::string out;
    for (int k = 0; k < K_COUNT; ++k) {
      if (!t.count[k]) continue;
      char line[160];
      snprintf(line, sizeof(line), "%s %llu %.6f\n", kKindNames[k], (unsigned long long)t.count[k], t.total_ms[k]);
      out += line;
    }
    if (buf && cap > 0) {
      const size_t n = out.size() < (size_t)(cap - 1) ? out.size() : (size_t)(cap - 1);
      memcpy(buf, out.data(), n);
      buf[n] = 0;
    }
    if (reset) {
      for (int k = 0; k < K_COUNT; ++k) {
        t.total_ms[k] = 0.0;
        t.count[k] = 0;
      }
    }
    return cuda_ok ? (int64_t)out.size() : -1;
  } catch (...) {
    return -1;
  }
}


// ------------------------------------------------------------ packed batch
size_t bdlm_workspace_size_varlen(int op, const int64_t* seq_offsets, int n_seqs, int Hq, int Hkv, int d) {
  try {
    if (op != BDLM_OP_FWD && op != BDLM_OP_BWD) return 0;
    int64_t T;
    if (check_varlen(seq_offsets, n_seqs, 0, Hq, Hkv, d, &T) != BDLM_OK) return 0;
    return varlen_layout(op, seq_offsets, n_seqs, Hq, Hkv, T).total;
  } catch (...) {
    return 0;
  }
}

bdlm_status bdlm_attn_fwd_varlen(const void* Qc, const void* Kc, const void* Vc, const void* Qn, const void* Kn,
                                 const void* Vn, const int64_t* seq_offsets, int n_seqs, int64_t B, int Hq,
                                 int Hkv, int d, float scale, void* Oc, void* On, bdlm_dtype o_dtype, float* LSEc,
                                 float* LSEn, void* workspace, size_t ws_bytes, bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    int64_t T;
    BDLM_CHECK(check_varlen(seq_offsets, n_seqs, B, Hq, Hkv, d, &T));
    BDLM_CHECK(check_scale(scale));
    if (o_dtype != BDLM_BF16 && o_dtype != BDLM_F32) return fail(BDLM_ERR_INVALID_ARG, "bad o_dtype %d", (int)o_dtype);
    BDLM_CHECK(check_ptrs("bdlm_attn_fwd_varlen(Qc,Kc,Vc,Qn,Kn,Vn,Oc,On,LSEc,LSEn)",
                          {Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, LSEc, LSEn}));
    const VarlenLayout lay = varlen_layout(BDLM_OP_FWD, seq_offsets, n_seqs, Hq, Hkv, T);
    BDLM_CHECK(check_ws(workspace, ws_bytes, lay.total));
    DeviceInfo info;
    BDLM_CHECK(device_info(info));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Geom all{T, B, Hq, Hkv, 0, T, 1};
    all.naive_order = naive_schedule();
    all.round_items = info.sms;
    VarlenTabs vt;
    int launches = 0;
    BDLM_CHECK(varlen_tables(all, seq_offsets, n_seqs, kFwdItemRows, false, lay, static_cast<char*>(workspace), st,
                             &launches, &vt));
    g_launches.fetch_add((uint64_t)launches);
    return fwd_common(Qc, Kc, Vc, Qn, Kn, Vn, T, B, Hq, Hkv, d, scale, 0, T, 1, Oc, On, o_dtype == BDLM_F32, LSEc,
                      LSEn, workspace, ws_bytes, st, &vt);
  });
}

bdlm_status bdlm_attn_bwd_varlen(const void* Qc, const void* Kc, const void* Vc, const void* Qn, const void* Kn,
                                 const void* Vn, const void* Oc, const void* On, const void* dOc, const void* dOn,
                                 const float* LSEc, const float* LSEn, const int64_t* seq_offsets, int n_seqs,
                                 int64_t B, int Hq, int Hkv, int d, float scale, void* dQc, void* dKc, void* dVc,
                                 void* dQn, void* dKn, void* dVn, bdlm_dtype g_dtype, void* workspace, size_t ws_bytes,
                                 bdlm_stream stream) {
  return guarded([&]() -> bdlm_status {
    int64_t T;
    BDLM_CHECK(check_varlen(seq_offsets, n_seqs, B, Hq, Hkv, d, &T));
    BDLM_CHECK(check_scale(scale));
    if (g_dtype != BDLM_BF16 && g_dtype != BDLM_F32) return fail(BDLM_ERR_INVALID_ARG, "bad g_dtype %d", (int)g_dtype);
    BDLM_CHECK(check_ptrs("bdlm_attn_bwd_varlen(Qc,Kc,Vc,Qn,Kn,Vn,Oc,On,dOc,dOn,LSEc,LSEn)",
                          {Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, dOc, dOn, LSEc, LSEn}));
    BDLM_CHECK(check_ptrs("bdlm_attn_bwd_varlen(dQc,dKc,dVc,dQn,dKn,dVn)", {dQc, dKc, dVc, dQn, dKn, dVn}));
    const VarlenLayout lay = varlen_layout(BDLM_OP_BWD, seq_offsets, n_seqs, Hq, Hkv, T);
    BDLM_CHECK(check_ws(workspace, ws_bytes, lay.total));
    DeviceInfo info;
    BDLM_CHECK(device_info(info));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* w = static_cast<char*>(workspace);
    float* Dc = reinterpret_cast<float*>(w + kWsHeader);
    float* Dn = Dc + (size_t)Hq * T;
    Geom all{T, B, Hq, Hkv, 0, T, 1};
    all.naive_order = naive_schedule();
    all.round_items = info.sms;
    VarlenTabs vt;
    int tab_launches = 0;
    BDLM_CHECK(varlen_tables(all, seq_offsets, n_seqs, kBwdTile, true, lay, w, st, &tab_launches, &vt));
    g_launches.fetch_add((uint64_t)tab_launches);
    BDLM_CHECK(clear_status(workspace, st));
    int launches = 0;
    cudaError_t e;
    {
      ScopedKernelTimer tm(K_PREP, st);
      e = launch_preprocess(Oc, 0, dOc, T, Hq, d, Dc, st, &launches, info.sms);
    }
    if (e == cudaSuccess) {
      ScopedKernelTimer tm(K_PREP, st);
      e = launch_preprocess(On, 0, dOn, T, Hq, d, Dn, st, &launches, info.sms);
    }
    BwdParams p = bwd_params(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn, T, B, Hq, Hkv, d, scale, 0, T, 1,
                             info.sms);
    p.dQc = dQc; p.dQn = dQn; p.dKc = dKc; p.dVc = dVc; p.dKn = dKn; p.dVn = dVn;
    p.g_f32 = g_dtype == BDLM_F32;
    bdlm_status vs = BDLM_OK;
    if (e == cudaSuccess) e = launch_backward_passes(p, info, workspace, st, &launches, &vs, &vt);
    if (vs != BDLM_OK) return vs;
    return finish(e, launches, "varlen backward launch");
  });
}

uint64_t bdlm_kernel_launches(void) { return g_launches.load(); }

const char* bdlm_last_error(void) { return g_last_error.c_str(); }

const char* bdlm_version(void) { return "bdlm_attn 0.1 (sm_103a)"; }

}  // extern "C"
