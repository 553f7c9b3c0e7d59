// api.cu -- C ABI of libtsa (declared in include/tsa.h).
//
// Host-side validation, workspace layout and the launch sequence of each
// entry point.  Nothing here allocates device memory, synchronises or prints.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include "../../include/tsa.h"
#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {
int scan_tile_rows();
int scan_grid_rows(bool q8);
}  // namespace tsa

using namespace tsa;

namespace {

thread_local std::string g_err;
thread_local cudaEvent_t g_stage[4] = {nullptr, nullptr, nullptr, nullptr};
thread_local TraceBuf g_trace = {nullptr, nullptr, 0};
// Fault injection for tests: the wait limit of the next key scan on this
// thread, whose CTA 0 then withholds its first tile copy (0: off).
thread_local long long g_stall_ns = 0;
std::atomic<unsigned long long> g_launches{0};

// Count a kernel launch of this library once it has been issued.
cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

// Record stage event i on stream st when stage timing is on.
cudaError_t stage_mark(int i, cudaStream_t st) {
  if (!g_stage[i]) return cudaSuccess;
  return cudaEventRecord(g_stage[i], st);
}

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}
int ok() {
  g_err.clear();
  return TSA_OK;
}
int cuda_fail(cudaError_t e, const char* what) {
  return fail(TSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr size_t kAlign = 256;
size_t up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// Dense pair list capacity per head: every position once plus the sentinel
// padding of at most 7 slots per (CTA, warp, unit visit) run.
int64_t dense_stride_for(int64_t l_cap) {
  return (int64_t)up((size_t)(l_cap > 0 ? l_cap : 1) + 65536, 64);
}

int num_sms() {
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!sms[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = v > 0 ? v : 148;
  }
  return sms[dev];
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }


// Device pointers of the exact top-K machinery (key scan + finish).
struct SelWs {
  int* status;
  uint32_t* tile_ctr;    // counters: zero before a call, cleared by its finish kernel
  int32_t* dense_n;
  uint32_t* emit_key;    // persist between calls (any content is safe)
  float* emit_margin;
  uint2* dense;
  int64_t dense_stride;
  uint64_t* spill;
  float* wz;
  int wz_stride;
  uint32_t* hist16;      // decode layouts only (nullptr elsewhere): zero before a call
};

// Workspace of one decode call (offsets from the base).  [zero_begin,
// zero_end) holds the counters that start every call at zero; the hint
// bins after them persist.
struct DecodeLayout {
  size_t zero_begin, status, tile_ctr, dense_n, hist16, zero_end;
  size_t emit_key, emit_margin, wz, dense, spill, total;
  int64_t dense_stride;
  int wz_stride;
};

DecodeLayout decode_layout(int B, int Hq, int Hkv, int64_t l_cap, int n_init, int n_recent) {
  DecodeLayout L{};
  const size_t rows = (size_t)B * Hq;
  (void)Hkv;
  L.dense_stride = dense_stride_for(l_cap);
  int64_t win = (int64_t)n_init + n_recent;
  if (win > l_cap) win = l_cap;
  L.wz_stride = (int)(win > 0 ? win : 1);
  size_t o = 0;
  L.zero_begin = o;
  L.status = o; o = up(o + 4);
  L.tile_ctr = o; o = up(o + 4);
  L.dense_n = o; o = up(o + rows * kCtrStride * 4);
  L.hist16 = o; o = up(o + rows * kH16Bins * 4);
  L.zero_end = o;
  L.emit_key = o; o = up(o + rows * 4);
  L.emit_margin = o; o = up(o + rows * 4);
  L.wz = o; o = up(o + rows * (size_t)L.wz_stride * 4);
  L.dense = o; o = up(o + rows * (size_t)L.dense_stride * 8);
  L.spill = o; o = up(o + rows * (size_t)L.dense_stride * 8);
  L.total = o;
  return L;
}

// Argument block of the key scan over workspace w.
ScanArgs scan_args(const uint16_t* q, const KvView& view, const int32_t* lens, int64_t len_host,
                   int B, int Hq, int n_init, int n_recent, float scale,
                   const int32_t* head_active, int active_value, const SelWs& w) {
  ScanArgs s{};
  s.q = q;
  s.kv = view;
  s.lens = lens;
  s.len_host = len_host;
  s.B = B;
  s.Hq = Hq;
  s.scale = scale;
  s.n_init = n_init;
  s.n_recent = n_recent;
  s.head_active = head_active;
  s.active_value = active_value;
  s.tile_ctr = w.tile_ctr;
  s.emit_key = w.emit_key;
  s.dense = w.dense;
  s.dense_n = w.dense_n;
  s.dense_stride = w.dense_stride;
  s.wz = w.wz;
  s.wz_stride = w.wz_stride;
  s.status = w.status;
  s.hist16 = w.hist16;
  s.trace = g_trace;
  s.wait_ns = g_stall_ns;
  s.stall_first_copy = g_stall_ns > 0;
  g_stall_ns = 0;  // one call only
  return s;
}

// Finish-kernel arguments common to both entry points.
FinishArgs finish_args(const uint16_t* q, const KvView& view, int Hq, float scale, int K,
                       const SelWs& w) {
  FinishArgs f{};
  f.q = q;
  f.kv = view;
  f.Hq = Hq;
  f.scale = scale;
  f.K = K;
  f.emit_key = w.emit_key;
  f.emit_margin = w.emit_margin;
  f.tile_ctr = w.tile_ctr;
  f.status = w.status;
  f.dense = w.dense;
  f.dense_n = w.dense_n;
  f.dense_stride = w.dense_stride;
  f.spill = w.spill;
  f.wz = w.wz;
  f.wz_stride = w.wz_stride;
  f.hist16 = w.hist16;
  f.trace = g_trace;
  return f;
}

// Persistent scan grid: one CTA per SM, at most one per tile.
int scan_grid(int B, const KvView& view, int64_t max_len, bool q8 = false) {
  const int64_t tr = scan_grid_rows(q8);
  const int64_t tiles = (int64_t)B * view.Hkv * ((max_len + tr - 1) / tr);
  int64_t grid = num_sms();
  if (grid > tiles) grid = tiles;
  if (grid < 1) grid = 1;
  return (int)grid;
}

int check_kv(const tsa_kv* kv, int B, int Hkv) {
  if (!kv) return fail(TSA_ERR_INVALID_ARG, "kv is NULL");
  if (!kv->k || !kv->v) return fail(TSA_ERR_INVALID_ARG, "kv->k / kv->v is NULL");
  if (!aligned(kv->k, 16) || !aligned(kv->v, 16))
    return fail(TSA_ERR_INVALID_ARG, "kv->k / kv->v must be 16-byte aligned");
  if (kv->l_cap < 0) return fail(TSA_ERR_INVALID_ARG, "kv->l_cap < 0");
  if (kv->l_cap >= (int64_t)1 << 31) return fail(TSA_ERR_INVALID_ARG, "kv->l_cap >= 2^31");
  if (kv->page_table) {
    const int ps = kv->page_size;
    if (ps < 16 || ps > 256 || (ps & (ps - 1)))
      return fail(TSA_ERR_INVALID_ARG, "page_size %d: must be a power of two in [16, 256]", ps);
    if (kv->max_pages <= 0) return fail(TSA_ERR_INVALID_ARG, "max_pages must be > 0");
    if ((int64_t)kv->max_pages * ps != kv->l_cap)
      return fail(TSA_ERR_INVALID_ARG, "paged cache: l_cap must equal max_pages*page_size");
  }
  (void)B;
  (void)Hkv;
  return TSA_OK;
}

KvView make_view(const tsa_kv* kv, int Hkv) {
  KvView v{};
  v.k = static_cast<const uint16_t*>(kv->k);
  v.v = static_cast<const uint16_t*>(kv->v);
  v.page_table = kv->page_table;
  v.page_shift = 0;
  if (kv->page_table)
    while ((1 << v.page_shift) < kv->page_size) ++v.page_shift;
  v.max_pages = kv->max_pages;
  v.l_cap = kv->l_cap;
  v.Hkv = Hkv;
  v.seq_rows = (int64_t)Hkv * kv->l_cap;
  v.pt_stride = kv->max_pages;
  return v;
}

int check_heads(int B, int Hq, int Hkv, int d) {
  if (d != kD) return fail(TSA_ERR_INVALID_ARG, "d = %d: only d = 128 is compiled", d);
  if (B < 0 || Hq <= 0 || Hkv <= 0) return fail(TSA_ERR_INVALID_ARG, "B/Hq/Hkv out of range");
  if (Hq % Hkv) return fail(TSA_ERR_INVALID_ARG, "Hq %% Hkv != 0 (Hq=%d Hkv=%d)", Hq, Hkv);
  if (Hq / Hkv > kMaxGroup)
    return fail(TSA_ERR_INVALID_ARG, "group size %d > %d", Hq / Hkv, kMaxGroup);
  if ((int64_t)B * Hkv > kMaxUnits)
    return fail(TSA_ERR_INVALID_ARG, "B*Hkv = %lld > %d", (long long)B * Hkv, kMaxUnits);
  if ((int64_t)B * Hq > 65535)
    return fail(TSA_ERR_INVALID_ARG, "B*Hq = %lld > 65535", (long long)B * Hq);
  return TSA_OK;
}

// Every host check of sparse_attn_decode except the workspace's.
int check_decode(const void* q, const tsa_kv* kv, const int32_t* lens, int B, int Hq, int Hkv,
                 int d, int K, int n_init, int n_recent, float scale, const float* out) {
  int rc = check_heads(B, Hq, Hkv, d);
  if (rc) return rc;
  if ((rc = check_kv(kv, B, Hkv))) return rc;
  if (B == 0) return TSA_OK;
  if (!q || !out || !lens) return fail(TSA_ERR_INVALID_ARG, "q, out and lens must be non-NULL");
  if (!aligned(q, 16)) return fail(TSA_ERR_INVALID_ARG, "q must be 16-byte aligned");
  if (!aligned(out, 16)) return fail(TSA_ERR_INVALID_ARG, "out must be 16-byte aligned");
  if (K < 0 || n_init < 0 || n_recent < 0)
    return fail(TSA_ERR_INVALID_ARG, "K, n_init, n_recent must be >= 0");
  if (!std::isfinite(scale)) return fail(TSA_ERR_INVALID_ARG, "scale must be finite");
  return TSA_OK;
}

}  // namespace

namespace tsa {
// Sets this thread's error message for an entry point defined in another
// translation unit of the library; returns `code`.
int report_error(int code, const char* msg) { return fail(code, "%s", msg); }
// The host checks of sparse_attn_decode other than the workspace's (TSA_OK,
// or the error code with this thread's message set).
int validate_decode(const void* q, const tsa_kv* kv, const int32_t* lens, int B, int Hq,
                    int Hkv, int d, int K, int n_init, int n_recent, float scale,
                    const float* out) {
  return check_decode(q, kv, lens, B, Hq, Hkv, d, K, n_init, n_recent, scale, out);
}
// Bytes at the start of a decode workspace that must be zero before a call.
size_t decode_zero_bytes(int B, int Hq, int Hkv, int64_t l_cap, int K, int n_init, int n_recent) {
  (void)K;
  return decode_layout(B, Hq, Hkv, l_cap, n_init, n_recent).zero_end;
}
}  // namespace tsa

extern "C" {

const char* tsa_last_error(void) { return g_err.c_str(); }

const char* tsa_version(void) { return "tsa 0.1 (sm_103a)"; }

unsigned long long tsa_kernel_launches(void) {
  return g_launches.load(std::memory_order_relaxed);
}

int tsa_set_stage_events(void* const* events, int n) {
  if (events && n > 0 && n < 4)
    return fail(TSA_ERR_INVALID_ARG, "tsa_set_stage_events needs 4 events");
  for (int i = 0; i < 4; ++i)
    g_stage[i] = (events && n >= 4) ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  return ok();
}

int tsa_set_trace(void* buf, size_t bytes) {
  if (!buf || bytes < 64 + sizeof(TraceRec)) {
    g_trace = {nullptr, nullptr, 0};
    return ok();
  }
  if (!aligned(buf, 64)) return fail(TSA_ERR_INVALID_ARG, "trace buffer must be 64-byte aligned");
  g_trace.count = static_cast<uint32_t*>(buf);
  g_trace.rec = reinterpret_cast<TraceRec*>(static_cast<uint8_t*>(buf) + 64);
  g_trace.cap = (uint32_t)((bytes - 64) / sizeof(TraceRec));
  return ok();
}

size_t tsa_decode_workspace_size(int B, int Hq, int Hkv, int d, int64_t l_cap, int K,
                                 int n_init, int n_recent) {
  (void)d;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || l_cap < 0 || K < 0 || n_init < 0 || n_recent < 0)
    return 0;
  return decode_layout(B, Hq, Hkv, l_cap, n_init, n_recent).total;
}

}  // extern "C"

namespace {

// The decode step's launches on workspace layout Lw: lengths from `lens`
// (device) or, without it, len_host; the static window given as the number
// of leading (n_init) and trailing (n_recent) positions of each sequence's
// cache.
// The quantised scan's inputs: the key codes and this call's query
// preparation in the workspace.
struct Q8Run {
  uint8_t* codes;
  const float* kscale;
  float* kerr;
  int n_new;
  size_t qh, qts, eps;  // workspace offsets
};

int decode_run(const void* q, const KvView& view, const int32_t* lens, int64_t len_host, int B,
               int Hq, int K, int n_init, int n_recent, float scale, float* out, float* lse_out,
               int32_t* topk_idx, float* topk_score, const DecodeLayout& Lw, void* workspace,
               cudaStream_t st, const Q8Run* q8 = nullptr) {
  // The workspace counters start at zero: the caller zeroes a new workspace
  // once and every call's finish kernel clears them again for the next call,
  // so no memset sits between consecutive calls and the key scan can be
  // launched as a programmatic dependent of the previous call's kernels.
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = stage_mark(0, st);
  if (e != cudaSuccess) return cuda_fail(e, "event record");
  SelWs w{};
  w.status = reinterpret_cast<int*>(ws + Lw.status);
  w.tile_ctr = reinterpret_cast<uint32_t*>(ws + Lw.tile_ctr);
  w.emit_key = reinterpret_cast<uint32_t*>(ws + Lw.emit_key);
  w.emit_margin = reinterpret_cast<float*>(ws + Lw.emit_margin);
  w.dense = reinterpret_cast<uint2*>(ws + Lw.dense);
  w.dense_n = reinterpret_cast<int32_t*>(ws + Lw.dense_n);
  w.dense_stride = Lw.dense_stride;
  w.spill = reinterpret_cast<uint64_t*>(ws + Lw.spill);
  w.wz = reinterpret_cast<float*>(ws + Lw.wz);
  w.wz_stride = Lw.wz_stride;
  if (!q8)  // the plain scan's fine histogram of the emitted pairs
    w.hist16 = reinterpret_cast<uint32_t*>(ws + Lw.hist16);

  // 1. key scan (logits, emitted pairs, window logits); with key codes,
  // after the query preparation (and the coding of the newest rows)
  const bool quant = q8 && view.l_cap > 0;
  if (quant) {
    Q8PrepArgs p{};
    p.q = static_cast<const uint16_t*>(q);
    p.kv = view;
    p.codes = q8->codes;
    p.kscale = q8->kscale;
    p.kerr = q8->kerr;
    p.lens = lens;
    p.len_host = len_host;
    p.B = B;
    p.Hq = Hq;
    p.n_new = q8->n_new;
    p.scale = scale;
    p.qh = reinterpret_cast<uint16_t*>(ws + q8->qh);
    p.qts = reinterpret_cast<float*>(ws + q8->qts);
    p.eps = reinterpret_cast<float*>(ws + q8->eps);
    if ((e = counted(launch_q8_prep(p, st, true))) != cudaSuccess)
      return cuda_fail(e, "query preparation launch");
  }
  if (view.l_cap > 0) {
    ScanArgs s = scan_args(static_cast<const uint16_t*>(q), view, lens, len_host, B, Hq, n_init,
                           n_recent, scale, nullptr, 0, w);
    if (quant) {
      s.codes = q8->codes;
      s.qh = reinterpret_cast<const uint16_t*>(ws + q8->qh);
      s.qts = reinterpret_cast<const float*>(ws + q8->qts);
      s.q8_new = q8->n_new;
    }
    if ((e = counted(launch_scan(s, scan_grid(B, view, view.l_cap, quant), st, true))) !=
        cudaSuccess)
      return cuda_fail(e, "scan launch");
  }
  if ((e = stage_mark(1, st)) != cudaSuccess) return cuda_fail(e, "event record");
  if ((e = stage_mark(2, st)) != cudaSuccess) return cuda_fail(e, "event record");
  // 2-3. exact top-K outside the window, window + selected partials, gamma merge
  {
    FinishArgs f = finish_args(static_cast<const uint16_t*>(q), view, Hq, scale, K, w);
    f.lens = lens;
    f.len_host = len_host;
    f.B = B;
    f.n_init = n_init;
    f.n_recent = n_recent;
    f.out = out;
    f.lse_out = lse_out;
    f.topk_idx = topk_idx;
    f.topk_score = topk_score;
    f.topk_stride = K;
    if (quant) {  // the emitted pairs rescored exactly, the window logits
      Q8RescoreArgs r{};
      r.q = static_cast<const uint16_t*>(q);
      r.kv = view;
      r.lens = lens;
      r.len_host = len_host;
      r.B = B;
      r.Hq = Hq;
      r.scale = scale;
      r.n_init = n_init;
      r.n_recent = n_recent;
      r.dense = w.dense;
      r.dense_n = w.dense_n;
      r.dense_stride = w.dense_stride;
      r.emit_key = w.emit_key;
      r.eps = reinterpret_cast<const float*>(ws + q8->eps);
      r.wz = w.wz;
      r.wz_stride = w.wz_stride;
      r.trace = g_trace;
      if ((e = counted(launch_q8_rescore(r, 2 * num_sms(), st))) != cudaSuccess)
        return cuda_fail(e, "rescore launch");
      f.q8_eps = r.eps;
    }
    if ((e = counted(launch_finish(f, st))) != cudaSuccess) return cuda_fail(e, "finish launch");
  }
  if ((e = stage_mark(3, st)) != cudaSuccess) return cuda_fail(e, "event record");
  return ok();
}

// attend_set's workspace: the finish kernel's counters and per-head state
// (the path words are zero: every head "reuses" its given set) and a spill
// area of the set's size per head.
struct AttendLayout {
  size_t status, tile_ctr, dense_n, path, emit_key, emit_margin, zero_end, spill, total;
  int64_t stride;
};
AttendLayout attend_layout(int B, int Hq, int M) {
  AttendLayout L{};
  const size_t rows = (size_t)B * Hq;
  L.stride = (int64_t)up((size_t)(M > 0 ? M : 1) + 64, 64);
  size_t o = 0;
  L.status = o; o = up(o + 4);
  L.tile_ctr = o; o = up(o + 4);
  L.dense_n = o; o = up(o + rows * kCtrStride * 4);
  L.path = o; o = up(o + rows * 4);
  L.emit_key = o; o = up(o + rows * 4);
  L.emit_margin = o; o = up(o + rows * 4);
  L.zero_end = o;
  L.spill = o; o = up(o + rows * (size_t)L.stride * 8);
  L.total = o;
  return L;
}

}  // namespace

extern "C" {

int sparse_attn_decode(const void* q, const tsa_kv* kv, const int32_t* lens, int B, int Hq,
                       int Hkv, int d, int K, int n_init, int n_recent, float scale, float* out,
                       float* lse_out, int32_t* topk_idx, float* topk_score, void* workspace,
                       size_t ws_bytes, void* stream) {
  int rc = check_decode(q, kv, lens, B, Hq, Hkv, d, K, n_init, n_recent, scale, out);
  if (rc) return rc;
  if (B == 0) return ok();
  const DecodeLayout Lw = decode_layout(B, Hq, Hkv, kv->l_cap, n_init, n_recent);
  if (!workspace || !aligned(workspace, kAlign))
    return fail(TSA_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  if (ws_bytes < Lw.total)
    return fail(TSA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", ws_bytes, Lw.total);
  return decode_run(q, make_view(kv, Hkv), lens, 0, B, Hq, K, n_init, n_recent, scale, out,
                    lse_out, topk_idx, topk_score, Lw, workspace, static_cast<cudaStream_t>(stream));
}

int sparse_attn_decode_shard(const void* q, const tsa_kv* kv, int64_t shard_len,
                             int64_t pos_offset, int64_t global_len, int Hq, int Hkv, int d, int K,
                             int n_init, int n_recent, float scale, float* out, float* lse_out,
                             int32_t* topk_idx, float* topk_score, void* workspace,
                             size_t ws_bytes, void* stream) {
  int rc = check_heads(1, Hq, Hkv, d);
  if (rc) return rc;
  if ((rc = check_kv(kv, 1, Hkv))) return rc;
  if (!q || !out) return fail(TSA_ERR_INVALID_ARG, "q and out must be non-NULL");
  if (!aligned(q, 16) || !aligned(out, 16))
    return fail(TSA_ERR_INVALID_ARG, "q / out must be 16-byte aligned");
  if (K < 0 || n_init < 0 || n_recent < 0)
    return fail(TSA_ERR_INVALID_ARG, "K, n_init, n_recent must be >= 0");
  if (!std::isfinite(scale)) return fail(TSA_ERR_INVALID_ARG, "scale must be finite");
  if (shard_len < 0 || shard_len > kv->l_cap)
    return fail(TSA_ERR_INVALID_ARG, "shard_len %lld outside [0, l_cap]", (long long)shard_len);
  if (pos_offset < 0 || pos_offset + shard_len > global_len)
    return fail(TSA_ERR_INVALID_ARG, "shard [%lld, %lld) outside [0, global_len = %lld)",
                (long long)pos_offset, (long long)(pos_offset + shard_len), (long long)global_len);
  const DecodeLayout Lw = decode_layout(1, Hq, Hkv, kv->l_cap, n_init, n_recent);
  if (!workspace || !aligned(workspace, kAlign))
    return fail(TSA_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  if (ws_bytes < Lw.total)
    return fail(TSA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", ws_bytes, Lw.total);
  // The global window [0, n_init) u [global_len - n_recent, global_len)
  // meets the shard [pos_offset, pos_offset + shard_len) in a prefix and a
  // suffix of it: n_init - pos_offset leading and
  // n_recent - (global_len - pos_offset - shard_len) trailing positions.
  auto clampl = [&](int64_t x) { return x < 0 ? 0 : (x > shard_len ? shard_len : x); };
  const int ni = (int)clampl((int64_t)n_init - pos_offset);
  const int nr = (int)clampl((int64_t)n_recent - (global_len - pos_offset - shard_len));
  return decode_run(q, make_view(kv, Hkv), nullptr, shard_len, 1, Hq, K, ni, nr, scale, out,
                    lse_out, topk_idx, topk_score, Lw, workspace, static_cast<cudaStream_t>(stream));
}

// ---- int8 key codes and the quantised decode ----

namespace {
struct Q8Layout {
  DecodeLayout d;
  size_t qh, qts, eps, total;
};
Q8Layout decode_q8_layout(int B, int Hq, int Hkv, int64_t l_cap, int n_init, int n_recent) {
  Q8Layout L{};
  L.d = decode_layout(B, Hq, Hkv, l_cap, n_init, n_recent);
  const size_t rows = (size_t)B * Hq;
  size_t o = L.d.total;
  L.qh = o; o = up(o + rows * kD * 2);
  L.qts = o; o = up(o + rows * 4);
  L.eps = o; o = up(o + rows * 4);
  L.total = o;
  return L;
}
int check_kq8(const tsa_kq8* kq) {
  if (!kq || !kq->codes || !kq->scale || !kq->err)
    return fail(TSA_ERR_INVALID_ARG, "kq, kq->codes, kq->scale and kq->err must be non-NULL");
  if (!aligned(kq->codes, 16)) return fail(TSA_ERR_INVALID_ARG, "kq->codes must be 16-byte aligned");
  if (!aligned(kq->scale, 4) || !aligned(kq->err, 4))
    return fail(TSA_ERR_INVALID_ARG, "kq->scale / kq->err must be 4-byte aligned");
  return TSA_OK;
}
}  // namespace

size_t tsa_decode_q8_workspace_size(int B, int Hq, int Hkv, int d, int64_t l_cap, int K,
                                    int n_init, int n_recent) {
  (void)d;
  (void)K;
  if (B < 0 || Hq <= 0 || l_cap < 0) return 0;
  return decode_q8_layout(B, Hq, Hkv, l_cap, n_init, n_recent).total;
}

int tsa_quantize_keys(const tsa_kv* kv, const tsa_kq8* kq, const int32_t* lens, int B, int Hkv,
                      int d, int64_t n_tail, int fit, void* stream) {
  if (d != kD) return fail(TSA_ERR_INVALID_ARG, "d = %d: only d = 128 is compiled", d);
  if (B < 0 || Hkv <= 0) return fail(TSA_ERR_INVALID_ARG, "B/Hkv out of range");
  int rc = check_kv(kv, B, Hkv);
  if (rc) return rc;
  if ((rc = check_kq8(kq))) return rc;
  if (fit != 0 && fit != 1) return fail(TSA_ERR_INVALID_ARG, "fit must be 0 or 1");
  if (!fit && n_tail < 0) return fail(TSA_ERR_INVALID_ARG, "n_tail must be >= 0");
  if ((int64_t)B * Hkv > 65535) return fail(TSA_ERR_INVALID_ARG, "B*Hkv > 65535");
  if (B == 0) return ok();
  if (!lens) return fail(TSA_ERR_INVALID_ARG, "lens must be non-NULL");
  const KvView view = make_view(kv, Hkv);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (fit) {
    const size_t bytes = (size_t)B * Hkv * kD * 4;
    if ((e = cudaMemsetAsync(kq->scale, 0, bytes, st)) != cudaSuccess)
      return cuda_fail(e, "memset");
    if ((e = cudaMemsetAsync(kq->err, 0, bytes, st)) != cudaSuccess)
      return cuda_fail(e, "memset");
  }
  e = launch_q8_quantize(view, lens, B, fit ? 0 : n_tail, fit != 0,
                         static_cast<uint8_t*>(kq->codes), kq->scale, kq->err, st);
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  const int64_t rows = fit ? view.l_cap : (n_tail < view.l_cap ? n_tail : view.l_cap);
  if (rows > 0) g_launches.fetch_add(fit ? 3 : 1, std::memory_order_relaxed);
  return ok();
}

int sparse_attn_decode_q8(const void* q, const tsa_kv* kv, const tsa_kq8* kq, int n_new,
                          const int32_t* lens, int B, int Hq, int Hkv, int d, int K, int n_init,
                          int n_recent, float scale, float* out, float* lse_out,
                          int32_t* topk_idx, float* topk_score, void* workspace, size_t ws_bytes,
                          void* stream) {
  int rc = check_decode(q, kv, lens, B, Hq, Hkv, d, K, n_init, n_recent, scale, out);
  if (rc) return rc;
  if ((rc = check_kq8(kq))) return rc;
  if (n_new < 0) return fail(TSA_ERR_INVALID_ARG, "n_new must be >= 0");
  if ((int64_t)B * Hq > kQ8MaxHeads)
    return fail(TSA_ERR_INVALID_ARG, "B*Hq = %lld > %d for the quantised scan",
                (long long)B * Hq, kQ8MaxHeads);
  if (B == 0) return ok();
  const Q8Layout Lq = decode_q8_layout(B, Hq, Hkv, kv->l_cap, n_init, n_recent);
  if (!workspace || !aligned(workspace, kAlign))
    return fail(TSA_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  if (ws_bytes < Lq.total)
    return fail(TSA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", ws_bytes, Lq.total);
  Q8Run r{};
  r.codes = static_cast<uint8_t*>(kq->codes);
  r.kscale = kq->scale;
  r.kerr = kq->err;
  r.n_new = n_new;
  r.qh = Lq.qh;
  r.qts = Lq.qts;
  r.eps = Lq.eps;
  return decode_run(q, make_view(kv, Hkv), lens, 0, B, Hq, K, n_init, n_recent, scale, out,
                    lse_out, topk_idx, topk_score, Lq.d, workspace,
                    static_cast<cudaStream_t>(stream), &r);
}

size_t tsa_attend_set_workspace_size(int B, int Hq, int M) {
  if (B <= 0 || Hq <= 0 || M < 1) return 0;
  return attend_layout(B, Hq, M).total;
}

int attend_set(const void* q, const tsa_kv* kv, int B, int Hq, int Hkv, int d,
               const int32_t* positions, const int32_t* counts, int M, float scale, float* out,
               float* lse_out, void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_heads(B, Hq, Hkv, d);
  if (rc) return rc;
  if ((rc = check_kv(kv, B, Hkv))) return rc;
  if (B == 0) return ok();
  if (M < 1 || M > (1 << 24)) return fail(TSA_ERR_INVALID_ARG, "M must be in [1, 2^24]");
  if (!q || !out || !positions || !counts)
    return fail(TSA_ERR_INVALID_ARG, "q, positions, counts and out must be non-NULL");
  if (!aligned(q, 16) || !aligned(out, 16))
    return fail(TSA_ERR_INVALID_ARG, "q / out must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(TSA_ERR_INVALID_ARG, "scale must be finite");
  const AttendLayout Lw = attend_layout(B, Hq, M);
  if (!workspace || !aligned(workspace, kAlign))
    return fail(TSA_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  if (ws_bytes < Lw.total)
    return fail(TSA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", ws_bytes, Lw.total);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // Every head takes the finish kernel's given-set path (a ReTopK reuse head
  // without the FIFO push): its rows are rescored, all of them are selected
  // (K = M >= count), and softmax.V runs over them without a window.
  SelWs w{};
  w.status = reinterpret_cast<int*>(ws + Lw.status);
  w.tile_ctr = reinterpret_cast<uint32_t*>(ws + Lw.tile_ctr);
  w.emit_key = reinterpret_cast<uint32_t*>(ws + Lw.emit_key);
  w.emit_margin = reinterpret_cast<float*>(ws + Lw.emit_margin);
  w.dense = nullptr;
  w.dense_n = reinterpret_cast<int32_t*>(ws + Lw.dense_n);
  w.dense_stride = Lw.stride;
  w.spill = reinterpret_cast<uint64_t*>(ws + Lw.spill);
  w.wz = nullptr;
  w.wz_stride = 1;
  const KvView view = make_view(kv, Hkv);
  FinishArgs f = finish_args(static_cast<const uint16_t*>(q), view, Hq, scale, M, w);
  f.lens = nullptr;
  f.len_host = kv->l_cap;  // positions must lie below l_cap
  f.B = B;
  f.out = out;
  f.lse_out = lse_out;
  f.topk_stride = M;
  f.path = reinterpret_cast<const int32_t*>(ws + Lw.path);
  f.mcand = counts;
  f.cand = reinterpret_cast<const uint32_t*>(positions);
  f.cand_cap = M;
  cudaError_t e = counted(launch_finish(f, static_cast<cudaStream_t>(stream)));
  if (e != cudaSuccess) return cuda_fail(e, "attend_set launch");
  return ok();
}

int tsa_workspace_status(void* workspace, int clear, void* stream) {
  if (!workspace || !aligned(workspace, kAlign))
    return fail(TSA_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int word = 0;  // the status word sits at offset 0 of both workspace layouts
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (clear && word) {
    e = cudaMemsetAsync(workspace, 0, sizeof word, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
  }
  if (word & kStatusTimeout)
    return fail(TSA_ERR_TIMEOUT,
                "a bounded device wait expired: the outputs of the calls since the last "
                "status read are NaN");
  if (word & kStatusBadLength)
    return fail(TSA_ERR_DEVICE_CHECK,
                "a sequence length outside [0, l_cap] was clamped to that range");
  if (word & kStatusCheck)
    return fail(TSA_ERR_DEVICE_CHECK,
                "an internal consistency check of a top-K selection failed (status 0x%x)", word);
  if (word) return fail(TSA_ERR_DEVICE_CHECK, "device status word 0x%x", word);
  return ok();
}

int tsa_inject_scan_stall(long long wait_limit_ns) {
  if (wait_limit_ns < 0 || wait_limit_ns > kWaitLimitNs)
    return fail(TSA_ERR_INVALID_ARG, "wait_limit_ns must be in [0, %lld]",
                (long long)kWaitLimitNs);
  g_stall_ns = wait_limit_ns;
  return ok();
}

int lse_merge(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b,
              float* o_out, float* lse_out, int rows, int d, void* stream) {
  if (rows < 0 || d < 1 || d > 1024) return fail(TSA_ERR_INVALID_ARG, "rows/d out of range");
  if (rows == 0) return ok();
  if (!o_a || !lse_a || !o_b || !lse_b || !o_out || !lse_out)
    return fail(TSA_ERR_INVALID_ARG, "NULL pointer");
  cudaError_t e = counted(launch_lse_merge(o_a, lse_a, o_b, lse_b, o_out, lse_out, rows, d,
                                   static_cast<cudaStream_t>(stream)));
  if (e != cudaSuccess) return cuda_fail(e, "lse_merge launch");
  return ok();
}

}  // extern "C"

// ===================================================================== ReTopK
struct tsa_retopk {
  uint32_t magic;
  int Hq, Hkv, K, C, R, W, T_r;
  float tau;
  int64_t max_len;
  float* qbar;       // [Hq][C][128]
  int32_t* sup;      // [Hq][C][K]
  int32_t* sup_n;    // [Hq][C]
  int64_t t;
  int fifo_head;
  int fresh;         // FIFO entry written by this handle's latest step (-1: none since init)
  bool initialised;
};

namespace {
constexpr uint32_t kMagic = 0x52544b31u;  // "RTK1"

struct RetopkLayout {
  size_t zero_begin, status, tile_ctr, dense_n, gbitmap, zero_end;
  size_t emit_key, emit_margin, wz, dense, spill, qbar_new, path, cand, mcand, lens, seqs, total;
  int64_t dense_stride, gbitmap_stride;
  int cand_cap;
};

// The selector keeps its candidate bitmap (one bit per cache position, plus a
// second level of one bit per 32-bit word) in one CTA's shared memory while
// that fits in 192 KiB; longer caches keep the bitmap in the workspace and
// only the second level in shared memory (192 KiB of it: 50 M positions).
constexpr int64_t kSmemBitmapBytes = (int64_t)192 * 1024;
bool bitmap_in_smem(int64_t len) {
  const int64_t words = (len + 31) / 32;
  return (words + (words + 31) / 32) * 4 <= kSmemBitmapBytes;
}
constexpr int64_t kMaxRetopkLen = kSmemBitmapBytes * 8 * 32;  // second level in 192 KiB

// Workspace of a step over up to n sequences of handles shaped like s.
RetopkLayout retopk_layout(const tsa_retopk* s, int n) {
  RetopkLayout L{};
  const size_t H = (size_t)n * s->Hq;
  L.dense_stride = dense_stride_for(s->max_len);
  L.cand_cap = s->R * s->K + s->W;
  size_t o = 0;
  L.zero_begin = o;
  L.status = o; o = up(o + 4);
  L.tile_ctr = o; o = up(o + 4);
  L.dense_n = o; o = up(o + H * kCtrStride * 4);
  // the bitmap of long caches (zero once; every step leaves it zero)
  L.gbitmap_stride = bitmap_in_smem(s->max_len) ? 0 : (int64_t)up((size_t)(s->max_len + 31) / 32, 64);
  L.gbitmap = o; o = up(o + H * (size_t)L.gbitmap_stride * 4);
  L.zero_end = o;
  L.emit_key = o; o = up(o + H * 4);
  L.emit_margin = o; o = up(o + H * 4);
  L.wz = o; o = up(o + 64);  // no window on this path
  L.dense = o; o = up(o + H * (size_t)L.dense_stride * 8);
  L.spill = o; o = up(o + H * (size_t)L.dense_stride * 8);
  L.qbar_new = o; o = up(o + H * kD * 4);
  L.path = o; o = up(o + H * 4);
  L.cand = o; o = up(o + H * (size_t)L.cand_cap * 4);
  L.mcand = o; o = up(o + H * 4);
  L.lens = o; o = up(o + (size_t)n * 4);
  L.seqs = o; o = up(o + (size_t)n * sizeof(RetopkSeq));
  L.total = o;
  return L;
}

size_t state_bytes(int Hq, int K, int C) {
  return up((size_t)Hq * C * kD * 4) + up((size_t)Hq * C * K * 4) + up((size_t)Hq * C * 4);
}

int check_state(const tsa_retopk* s) {
  if (!s || s->magic != kMagic) return fail(TSA_ERR_STATE, "invalid ReTopK handle");
  return TSA_OK;
}

}  // namespace

extern "C" {

size_t retopk_state_size(int Hq, int d, int K, int C) {
  if (Hq <= 0 || d != kD || K <= 0 || C <= 0) return 0;
  return state_bytes(Hq, K, C);
}

int retopk_create(tsa_retopk** st, int Hq, int Hkv, int d, int K, int C, int R, int W, float tau,
                  int T_r, int64_t max_len, void* state_mem, size_t state_bytes_) {
  if (!st) return fail(TSA_ERR_INVALID_ARG, "st is NULL");
  *st = nullptr;
  int rc = check_heads(1, Hq, Hkv, d);
  if (rc) return rc;
  if (K < 1) return fail(TSA_ERR_INVALID_ARG, "K must be >= 1");
  if (C < 1 || C > 64) return fail(TSA_ERR_INVALID_ARG, "C must be in [1, 64]");
  if (R < 1 || R > C) return fail(TSA_ERR_INVALID_ARG, "R must be in [1, C]");
  if (W < 0) return fail(TSA_ERR_INVALID_ARG, "W must be >= 0");
  if (T_r < 1) return fail(TSA_ERR_INVALID_ARG, "T_r must be >= 1");
  if (std::isnan(tau)) return fail(TSA_ERR_INVALID_ARG, "tau is NaN");
  if (max_len < 1 || max_len > kMaxRetopkLen)
    return fail(TSA_ERR_INVALID_ARG, "max_len must be in [1, %lld]", (long long)kMaxRetopkLen);
  if ((int64_t)R * K + W > 8192)
    return fail(TSA_ERR_INVALID_ARG, "R*K + W = %lld > 8192", (long long)R * K + W);
  if (!state_mem || !aligned(state_mem, kAlign))
    return fail(TSA_ERR_INVALID_ARG, "state_mem NULL or not 256-byte aligned");
  if (state_bytes_ < state_bytes(Hq, K, C))
    return fail(TSA_ERR_INVALID_ARG, "state_mem too small (%zu < %zu)", state_bytes_,
                state_bytes(Hq, K, C));
  tsa_retopk* s = new (std::nothrow) tsa_retopk();
  if (!s) return fail(TSA_ERR_INVALID_ARG, "out of host memory");
  s->magic = kMagic;
  s->Hq = Hq;
  s->Hkv = Hkv;
  s->K = K;
  s->C = C;
  s->R = R;
  s->W = W;
  s->T_r = T_r;
  s->tau = tau;
  s->max_len = max_len;
  uint8_t* m = static_cast<uint8_t*>(state_mem);
  s->qbar = reinterpret_cast<float*>(m);
  s->sup = reinterpret_cast<int32_t*>(m + up((size_t)Hq * C * kD * 4));
  s->sup_n = reinterpret_cast<int32_t*>(m + up((size_t)Hq * C * kD * 4) + up((size_t)Hq * C * K * 4));
  s->t = 0;
  s->fifo_head = 0;
  s->fresh = -1;
  s->initialised = false;
  *st = s;
  return ok();
}

int retopk_init(tsa_retopk* st, const void* prefill_q, const int32_t* prefill_supports,
                const int32_t* prefill_counts, void* stream) {
  int rc = check_state(st);
  if (rc) return rc;
  if (!prefill_q || !prefill_supports || !prefill_counts)
    return fail(TSA_ERR_INVALID_ARG, "NULL prefill pointer");
  RetopkInitArgs a{};
  a.prefill_q = static_cast<const uint16_t*>(prefill_q);
  a.prefill_sup = prefill_supports;
  a.prefill_n = prefill_counts;
  a.Hq = st->Hq;
  a.C = st->C;
  a.K = st->K;
  a.cache_qbar = st->qbar;
  a.cache_sup = st->sup;
  a.cache_sup_n = st->sup_n;
  cudaError_t e = counted(launch_retopk_init(a, static_cast<cudaStream_t>(stream)));
  if (e != cudaSuccess) return cuda_fail(e, "retopk init launch");
  st->t = 0;
  st->fifo_head = 0;
  st->fresh = -1;  // the init kernel completes before the next step's selector starts
  st->initialised = true;
  return ok();
}

size_t retopk_workspace_size(const tsa_retopk* st) {
  if (!st || st->magic != kMagic) return 0;
  return retopk_layout(st, 1).total;
}

size_t retopk_batched_workspace_size(const tsa_retopk* st, int n_max) {
  if (!st || st->magic != kMagic || n_max < 1 || n_max > kMaxRetopkBatch) return 0;
  return retopk_layout(st, n_max).total;
}

int retopk_step_batched(tsa_retopk* const* sts, int n, const void* q, const tsa_kv* kv,
                        const int64_t* lens, float scale, float* out, int32_t* support_out,
                        int32_t* path_out, int32_t* mcand_out, int32_t* cand_out, float* lse_out,
                        void* workspace, size_t ws_bytes, void* stream) {
  if (!sts || n < 1 || n > kMaxRetopkBatch)
    return fail(TSA_ERR_INVALID_ARG, "n must be in [1, %d] with a handle array", kMaxRetopkBatch);
  if (!lens) return fail(TSA_ERR_INVALID_ARG, "lens (host array) is NULL");
  const tsa_retopk* s0 = sts[0];
  int rc = check_state(s0);
  if (rc) return rc;
  for (int b = 0; b < n; ++b) {
    const tsa_retopk* sb = sts[b];
    if ((rc = check_state(sb))) return rc;
    if (!sb->initialised) return fail(TSA_ERR_STATE, "handle %d: retopk_init has not been called", b);
    if (sb->Hq != s0->Hq || sb->Hkv != s0->Hkv || sb->K != s0->K || sb->C != s0->C ||
        sb->R != s0->R || sb->W != s0->W || sb->T_r != s0->T_r || sb->tau != s0->tau ||
        sb->max_len != s0->max_len)
      return fail(TSA_ERR_INVALID_ARG, "handle %d: sizes and hyper-parameters differ from handle 0", b);
    for (int c = 0; c < b; ++c)
      if (sts[c] == sb || sts[c]->qbar == sb->qbar)
        return fail(TSA_ERR_INVALID_ARG, "handles %d and %d share their state", c, b);
  }
  if ((rc = check_heads(n, s0->Hq, s0->Hkv, kD))) return rc;
  if ((rc = check_kv(kv, n, s0->Hkv))) return rc;
  if (!q || !out) return fail(TSA_ERR_INVALID_ARG, "q and out must be non-NULL");
  if (!aligned(q, 16) || !aligned(out, 16))
    return fail(TSA_ERR_INVALID_ARG, "q/out must be 16-byte aligned");
  int64_t lmax = 0;
  for (int b = 0; b < n; ++b) {
    if (lens[b] < 1 || lens[b] > kv->l_cap || lens[b] > s0->max_len)
      return fail(TSA_ERR_INVALID_ARG, "lens[%d] = %lld outside [1, min(l_cap, max_len)]", b,
                  (long long)lens[b]);
    lmax = lens[b] > lmax ? lens[b] : lmax;
  }
  if (!std::isfinite(scale)) return fail(TSA_ERR_INVALID_ARG, "scale must be finite");
  if (!workspace || !aligned(workspace, kAlign))
    return fail(TSA_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  // The layout follows from the workspace's capacity (the most sequences its
  // ws_bytes hold), not from this call's n: calls with different n then see
  // every counter and per-row state at the same place.
  int ncap = 0;
  for (int c = 1; c <= kMaxRetopkBatch && retopk_layout(s0, c).total <= ws_bytes; ++c) ncap = c;
  if (ncap < n)
    return fail(TSA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", ws_bytes,
                retopk_layout(s0, n).total);
  const RetopkLayout Lw = retopk_layout(s0, ncap);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // As on the decode path, the workspace counters start at zero (the caller
  // zeroes a new workspace once; every step's finish kernel clears them), so
  // the three kernels form one chain of programmatic dependents.
  cudaError_t e = stage_mark(0, s);
  if (e != cudaSuccess) return cuda_fail(e, "event record");
  const KvView view = make_view(kv, s0->Hkv);
  const int Hq = s0->Hq;
  int32_t* path = reinterpret_cast<int32_t*>(ws + Lw.path);
  float* qbar_new = reinterpret_cast<float*>(ws + Lw.qbar_new);
  int32_t* lens_ws = reinterpret_cast<int32_t*>(ws + Lw.lens);
  RetopkSeq* seq_ws = reinterpret_cast<RetopkSeq*>(ws + Lw.seqs);
  SelWs w{};
  w.status = reinterpret_cast<int*>(ws + Lw.status);
  w.tile_ctr = reinterpret_cast<uint32_t*>(ws + Lw.tile_ctr);
  w.emit_key = reinterpret_cast<uint32_t*>(ws + Lw.emit_key);
  w.emit_margin = reinterpret_cast<float*>(ws + Lw.emit_margin);
  w.dense = reinterpret_cast<uint2*>(ws + Lw.dense);
  w.dense_n = reinterpret_cast<int32_t*>(ws + Lw.dense_n);
  w.dense_stride = Lw.dense_stride;
  w.spill = reinterpret_cast<uint64_t*>(ws + Lw.spill);
  w.wz = reinterpret_cast<float*>(ws + Lw.wz);
  w.wz_stride = 1;

  // 1. selector: cosine recall, path decision, candidate union, per (sequence, head)
  {
    RetopkSelArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.n = n;
    for (int b = 0; b < n; ++b) {
      const tsa_retopk* sb = sts[b];
      a.seq[b].qbar = sb->qbar;
      a.seq[b].sup = sb->sup;
      a.seq[b].sup_n = sb->sup_n;
      a.seq[b].L = lens[b];
      a.seq[b].fifo_head = sb->fifo_head;
      a.seq[b].refresh = (sb->t % sb->T_r) == 0;
      a.seq[b].fresh = sb->fresh;
    }
    a.Hq = Hq;
    a.C = s0->C;
    a.R = s0->R;
    a.K = s0->K;
    a.W = s0->W;
    a.tau = s0->tau;
    a.bitmap_words = (int)((lmax + 31) / 32);
    a.qbar_new = qbar_new;
    a.path = path;
    a.cand = reinterpret_cast<uint32_t*>(ws + Lw.cand);
    a.mcand = reinterpret_cast<int32_t*>(ws + Lw.mcand);
    a.cand_cap = Lw.cand_cap;
    a.path_out = path_out;
    a.mcand_out = mcand_out;
    a.cand_out = cand_out;
    a.lens_ws = lens_ws;
    a.seq_ws = seq_ws;
    a.trace = g_trace;
    // the bitmap (or, for a long cache, only its second level: the bitmap is
    // the workspace's) in shared memory
    const size_t l2w = (size_t)(a.bitmap_words + 31) / 32;
    const bool in_smem = bitmap_in_smem(lmax);
    a.gbitmap = in_smem ? nullptr : reinterpret_cast<uint32_t*>(ws + Lw.gbitmap);
    a.gbitmap_stride = Lw.gbitmap_stride;
    const size_t smem = up((in_smem ? (size_t)a.bitmap_words + l2w : l2w) * 4, 16);
    if ((e = counted(launch_retopk_selector(a, smem, s))) != cudaSuccess)
      return cuda_fail(e, "retopk selector launch");
  }
  // 2. exact-path heads: key scan over all keys (no window): the emitted
  //    pairs; it waits for the selector (paths and lengths) before it starts
  if ((e = counted(launch_scan(scan_args(static_cast<const uint16_t*>(q), view, lens_ws, 0, n,
                                         Hq, 0, 0, scale, path, 1, w),
                               scan_grid(n, view, lmax), s, true))) != cudaSuccess)
    return cuda_fail(e, "scan launch");
  if ((e = stage_mark(1, s)) != cudaSuccess) return cuda_fail(e, "event record");
  if ((e = stage_mark(2, s)) != cudaSuccess) return cuda_fail(e, "event record");
  // 3. every head: exact top-K (of its pairs; a reuse head rescores A_t
  //    itself), softmax.V over S_t (no window), and the FIFO push of
  //    (qbar_t, S_t) -- S_t is written into the entry it overwrites
  {
    FinishArgs f = finish_args(static_cast<const uint16_t*>(q), view, Hq, scale, s0->K, w);
    f.lens = lens_ws;
    f.B = n;
    f.n_init = 0;
    f.n_recent = 0;
    f.out = out;
    f.lse_out = lse_out;
    f.topk_idx = support_out;
    f.topk_score = nullptr;
    f.topk_stride = s0->K;
    f.path = path;
    f.mcand = reinterpret_cast<const int32_t*>(ws + Lw.mcand);
    f.cand = reinterpret_cast<const uint32_t*>(ws + Lw.cand);
    f.cand_cap = Lw.cand_cap;
    f.push_qbar = qbar_new;
    f.seqs = seq_ws;
    f.C = s0->C;
    if ((e = counted(launch_finish(f, s))) != cudaSuccess) return cuda_fail(e, "finish launch");
  }
  if ((e = stage_mark(3, s)) != cudaSuccess) return cuda_fail(e, "event record");
  for (int b = 0; b < n; ++b) {
    tsa_retopk* sb = sts[b];
    sb->t += 1;
    sb->fresh = sb->fifo_head;  // overwritten by this step's finish kernel
    sb->fifo_head = (sb->fifo_head + 1) % sb->C;
  }
  return ok();
}

int retopk_step(tsa_retopk* st, const void* q, const tsa_kv* kv, int64_t len, float scale,
                float* out, int32_t* support_out, int32_t* path_out, int32_t* mcand_out,
                int32_t* cand_out, float* lse_out, void* workspace, size_t ws_bytes,
                void* stream) {
  int rc = check_state(st);
  if (rc) return rc;
  if (!st->initialised) return fail(TSA_ERR_STATE, "retopk_init has not been called");
  if ((rc = check_kv(kv, 1, st->Hkv))) return rc;
  if (len < 1 || len > kv->l_cap || len > st->max_len)
    return fail(TSA_ERR_INVALID_ARG, "len %lld outside [1, min(l_cap, max_len)]", (long long)len);
  tsa_retopk* one[1] = {st};
  const int64_t lens[1] = {len};
  return retopk_step_batched(one, 1, q, kv, lens, scale, out, support_out, path_out, mcand_out,
                             cand_out, lse_out, workspace, ws_bytes, stream);
}

size_t retopk_prefill_workspace_size(int C, int Hq, int Hkv, int d, int64_t l_cap, int K) {
  (void)d;
  if (C <= 0 || Hq <= 0 || Hkv <= 0 || l_cap < 0 || K <= 0) return 0;
  // the decode workspace of C sequences without a window, plus the
  // attention outputs the finish kernel writes (not returned)
  return decode_layout(C, Hq, Hkv, l_cap, 0, 0).total + up((size_t)C * Hq * kD * 4);
}

int retopk_prefill_supports(const void* q_prefill, const tsa_kv* kv, int64_t L0, int C, int Hq,
                            int Hkv, int d, int K, float scale, int32_t* supports,
                            int32_t* counts, void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_heads(C, Hq, Hkv, d);
  if (rc) return rc;
  if ((rc = check_kv(kv, 1, Hkv))) return rc;
  if (C < 1) return fail(TSA_ERR_INVALID_ARG, "C must be >= 1");
  if (K < 1) return fail(TSA_ERR_INVALID_ARG, "K must be >= 1");
  if (L0 < C || L0 > kv->l_cap)
    return fail(TSA_ERR_INVALID_ARG, "L0 = %lld outside [C, l_cap]", (long long)L0);
  if (!q_prefill || !supports) return fail(TSA_ERR_INVALID_ARG, "q_prefill and supports must be non-NULL");
  if (!aligned(q_prefill, 16)) return fail(TSA_ERR_INVALID_ARG, "q_prefill must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(TSA_ERR_INVALID_ARG, "scale must be finite");
  const DecodeLayout Lw = decode_layout(C, Hq, Hkv, kv->l_cap, 0, 0);
  const size_t need = retopk_prefill_workspace_size(C, Hq, Hkv, d, kv->l_cap, K);
  if (!workspace || !aligned(workspace, kAlign))
    return fail(TSA_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  if (ws_bytes < need)
    return fail(TSA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", ws_bytes, need);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // The C queries are C sequences of one batch that all read the cache of
  // sequence 0 (sequence stride 0); query c sees positions [0, L0 - C + c].
  KvView view = make_view(kv, Hkv);
  view.seq_rows = 0;
  view.pt_stride = 0;
  SelWs w{};
  w.status = reinterpret_cast<int*>(ws + Lw.status);
  w.tile_ctr = reinterpret_cast<uint32_t*>(ws + Lw.tile_ctr);
  w.emit_key = reinterpret_cast<uint32_t*>(ws + Lw.emit_key);
  w.emit_margin = reinterpret_cast<float*>(ws + Lw.emit_margin);
  w.dense = reinterpret_cast<uint2*>(ws + Lw.dense);
  w.dense_n = reinterpret_cast<int32_t*>(ws + Lw.dense_n);
  w.dense_stride = Lw.dense_stride;
  w.spill = reinterpret_cast<uint64_t*>(ws + Lw.spill);
  w.wz = reinterpret_cast<float*>(ws + Lw.wz);
  w.wz_stride = Lw.wz_stride;
  w.hist16 = reinterpret_cast<uint32_t*>(ws + Lw.hist16);
  const int64_t len0 = L0 - C + 1;
  cudaError_t e;
  {
    ScanArgs sa = scan_args(static_cast<const uint16_t*>(q_prefill), view, nullptr, len0, C, Hq,
                            0, 0, scale, nullptr, 0, w);
    sa.len_step = 1;
    if ((e = counted(launch_scan(sa, scan_grid(C, view, L0), st, true))) != cudaSuccess)
      return cuda_fail(e, "scan launch");
  }
  {
    FinishArgs f = finish_args(static_cast<const uint16_t*>(q_prefill), view, Hq, scale, K, w);
    f.lens = nullptr;
    f.len_host = len0;
    f.len_step = 1;
    f.B = C;
    f.n_init = 0;
    f.n_recent = 0;
    f.out = reinterpret_cast<float*>(ws + Lw.total);
    f.lse_out = nullptr;
    f.topk_idx = supports;
    f.topk_score = nullptr;
    f.topk_stride = K;
    f.counts_out = counts;
    if ((e = counted(launch_finish(f, st))) != cudaSuccess) return cuda_fail(e, "finish launch");
  }
  return ok();
}

int retopk_get_counters(const tsa_retopk* st, int64_t* t, int32_t* fifo_head) {
  int rc = check_state(st);
  if (rc) return rc;
  if (t) *t = st->t;
  if (fifo_head) *fifo_head = st->fifo_head;
  return ok();
}

int retopk_set_counters(tsa_retopk* st, int64_t t, int32_t fifo_head) {
  int rc = check_state(st);
  if (rc) return rc;
  if (t < 0 || fifo_head < 0 || fifo_head >= st->C)
    return fail(TSA_ERR_INVALID_ARG, "counters out of range");
  st->t = t;
  st->fifo_head = fifo_head;
  st->initialised = true;
  return ok();
}

int retopk_destroy(tsa_retopk* st) {
  if (!st) return ok();
  if (st->magic != kMagic) return fail(TSA_ERR_STATE, "invalid ReTopK handle");
  st->magic = 0;
  delete st;
  return ok();
}

}  // extern "C"
