// rf_api.cu -- the C ABI of librf.so: argument validation, dispatch to the
// kernel launchers, error strings and the device status word.
//
// Every entry point checks its arguments on the host before touching CUDA;
// an invalid call launches nothing and returns RF_ERR_INVALID with a
// thread-local message (rf_last_error). No entry point allocates device
// memory or synchronises, except rf_device_status which exists to do so.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>

#include "rf_internal.h"

namespace {

thread_local char g_err[512] = {0};
thread_local uint8_t* g_visited = nullptr;
thread_local int64_t g_visited_len = 0;
thread_local int g_fault_site = 0;

// The device status word (one per device that loads the library).
__device__ int g_status_word = 0;
rf::SymbolCache g_status_cache;

// Driver calls that identify the current context, looked up once through the
// runtime (the library links no driver import). Null when unavailable.
using CtxGetCurrentFn = int (*)(void** ctx);
using CtxGetIdFn = int (*)(void* ctx, unsigned long long* id);

struct CtxFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const CtxFns& ctx_fns() {
  static const CtxFns fns = [] {
    CtxFns f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<CtxGetIdFn>(p);
    return f;
  }();
  return fns;
}

// Unique id of the calling thread's current context; 0 when there is none
// or it cannot be read (then nothing is cached).
unsigned long long current_ctx_id() {
  const CtxFns& f = ctx_fns();
  if (f.get_current == nullptr || f.get_id == nullptr) return 0;
  void* ctx = nullptr;
  if (f.get_current(&ctx) != 0 || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (f.get_id(ctx, &id) != 0) return 0;
  return id;
}

rf_status fail(rf_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

rf_status ok() {
  g_err[0] = 0;
  return RF_OK;
}

rf_status cuda_fail(cudaError_t e, const char* what) {
  return fail(RF_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

namespace rf {

void* symbol_address(const void* symbol, SymbolCache& cache, cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  const bool slot = dev >= 0 && dev < 128;
  unsigned long long id = current_ctx_id();
  if (slot && id != 0) {
    std::lock_guard<std::mutex> g(cache.mu);
    if (cache.ctx_id[dev] == id && cache.ptr[dev] != nullptr) return cache.ptr[dev];
  }
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, symbol);
  if (*err != cudaSuccess) return nullptr;
  id = current_ctx_id();  // the lookup may have made the primary context current
  if (slot && id != 0) {
    std::lock_guard<std::mutex> g(cache.mu);
    cache.ctx_id[dev] = id;
    cache.ptr[dev] = p;
  }
  return p;
}

int* status_word() {
  cudaError_t e = cudaSuccess;
  return static_cast<int*>(symbol_address(&g_status_word, g_status_cache, &e));
}

rf_status set_last_error(rf_status st, const char* msg) { return fail(st, "%s", msg); }

rf_status check_decode_args(const char* who, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, int B, int H, int Hkv, int Sk,
                            int d, float scale, int nsplit, rf_dtype dt) {
  if (B < 1 || H < 1 || Hkv < 1 || Sk < 1 || d < 1) return fail(RF_ERR_INVALID, "%s: bad sizes", who);
  if (H % Hkv != 0) return fail(RF_ERR_INVALID, "%s: H %% Hkv != 0", who);
  if (H / Hkv > 16) return fail(RF_ERR_UNSUPPORTED, "%s: H/Hkv > 16", who);
  if (nsplit < 1 || nsplit > Sk) return fail(RF_ERR_INVALID, "%s: need 1 <= nsplit <= Sk", who);
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(RF_ERR_INVALID, "%s: scale must be finite and > 0", who);
  if (dt != RF_F32 && dt != RF_BF16) return fail(RF_ERR_INVALID, "%s: dtype", who);
  if (dt != RF_BF16 || (d != 64 && d != 128))
    return fail(RF_ERR_UNSUPPORTED, "%s: bf16 with d in {64,128} only", who);
  if (int64_t(B) * Hkv * Sk * d * 2 > (int64_t(1) << 46))
    return fail(RF_ERR_INVALID, "%s: tensors too large", who);
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr)
    return fail(RF_ERR_INVALID, "%s: NULL pointer", who);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(RF_ERR_INVALID, "%s: pointers must be 16-byte aligned", who);
  if (lse != nullptr && !aligned(lse, 4))
    return fail(RF_ERR_INVALID, "%s: lse must be 4-byte aligned", who);
  return RF_OK;
}

uint8_t* debug_visited(int64_t* len) {
  if (len != nullptr) *len = g_visited_len;
  return g_visited;
}

}  // namespace rf

namespace {

// Validation shared by the attention entry points; fills `a`. *empty: Sq is
// 0 (nothing to launch).
rf_status attn_prepare(const char* fn, const void* q, const void* k, const void* v, void* o,
                       float* lse, int B, int H, int Hkv, int Sq, int Sk, int d, float scale,
                       int causal, const rf_blockmask* bm, rf_dtype dt, rf::AttnArgs& a,
                       bool* empty) {
  *empty = false;
  if (B < 1 || H < 1 || Hkv < 1 || Sq < 0 || Sk < 0 || d < 1)
    return fail(RF_ERR_INVALID, "%s: bad sizes B=%d H=%d Hkv=%d Sq=%d Sk=%d d=%d", fn, B, H,
                Hkv, Sq, Sk, d);
  if (Sq > (1 << 30) || Sk > (1 << 30))
    return fail(RF_ERR_INVALID, "%s: Sq and Sk must be <= 2^30", fn);
  if (H % Hkv != 0) return fail(RF_ERR_INVALID, "%s: H %% Hkv != 0", fn);
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(RF_ERR_INVALID, "%s: scale must be finite and > 0", fn);
  if (causal != 0 && causal != 1) return fail(RF_ERR_INVALID, "%s: causal must be 0/1", fn);
  if (dt != RF_F32 && dt != RF_BF16) return fail(RF_ERR_INVALID, "%s: bad dtype", fn);
  if (dt == RF_BF16 && d != 64 && d != 128)
    return fail(RF_ERR_UNSUPPORTED, "%s: bf16 supports d in {64,128}, got %d", fn, d);
  if (dt == RF_F32 && (d % 4 != 0 || d > 256))
    return fail(RF_ERR_UNSUPPORTED, "%s: f32 supports d %% 4 == 0, d <= 256", fn);
  const int64_t esz = dt == RF_F32 ? 4 : 2;
  if (int64_t(B) * H * Sq * d * esz > (int64_t(1) << 46) ||
      int64_t(B) * Hkv * Sk * d * esz > (int64_t(1) << 46))
    return fail(RF_ERR_INVALID, "%s: tensors too large", fn);
  const int nqt = static_cast<int>(cdiv(Sq, 128)), nkt = static_cast<int>(cdiv(Sk, 128));
  if (bm != nullptr) {
    if (bm->tile_q != 128 || bm->tile_k != 128)
      return fail(RF_ERR_INVALID, "%s: blockmask tiles must be 128x128", fn);
    if (bm->nqt != nqt || bm->nkt != nkt)
      return fail(RF_ERR_INVALID, "%s: blockmask nqt/nkt (%d,%d) != (%d,%d)", fn, bm->nqt,
                  bm->nkt, nqt, nkt);
    if (bm->per_head != 0 && bm->per_head != 1)
      return fail(RF_ERR_INVALID, "%s: blockmask per_head must be 0/1", fn);
    if (Sq > 0 && Sk > 0 && (bm->row_ptr == nullptr || bm->col_idx == nullptr))
      return fail(RF_ERR_INVALID, "%s: blockmask lists are NULL", fn);
    if (bm->tile_bits != nullptr && bm->bits == nullptr)
      return fail(RF_ERR_INVALID, "%s: blockmask tile_bits without bits", fn);
    if (bm->bits != nullptr && !aligned(bm->bits, 8))
      return fail(RF_ERR_INVALID, "%s: blockmask bits must be 8-byte aligned", fn);
    if (bm->cta_order != nullptr && !aligned(bm->cta_order, 4))
      return fail(RF_ERR_INVALID, "%s: blockmask cta_order must be 4-byte aligned", fn);
  }
  if (Sq == 0) {
    *empty = true;
    return ok();
  }
  if (q == nullptr || o == nullptr || (Sk > 0 && (k == nullptr || v == nullptr)))
    return fail(RF_ERR_INVALID, "%s: NULL tensor pointer", fn);
  if (!aligned(q, 16) || !aligned(o, 16) || (Sk > 0 && (!aligned(k, 16) || !aligned(v, 16))))
    return fail(RF_ERR_INVALID, "%s: q/k/v/o must be 16-byte aligned", fn);
  if (lse != nullptr && !aligned(lse, 4))
    return fail(RF_ERR_INVALID, "%s: lse must be 4-byte aligned", fn);
  int64_t vlen = 0;
  uint8_t* visited = rf::debug_visited(&vlen);
  if (visited != nullptr && vlen < int64_t(B) * H * nqt * nkt)
    return fail(RF_ERR_INVALID, "%s: visited buffer too small", fn);
  int* st = rf::status_word();
  if (st == nullptr) return fail(RF_ERR_CUDA, "%s: no CUDA device", fn);

  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.B = B; a.H = H; a.Hkv = Hkv; a.Sq = Sq; a.Sk = Sk; a.d = d;
  a.scale = scale; a.causal = causal;
  a.row_ptr = bm ? bm->row_ptr : nullptr;
  a.col_idx = bm ? bm->col_idx : nullptr;
  a.per_head = bm ? bm->per_head : 0;
  a.tile_bits = bm ? bm->tile_bits : nullptr;
  a.bits = bm && bm->tile_bits ? bm->bits : nullptr;
  a.nqt = nqt; a.nkt = nkt;
  a.cta_order = bm ? bm->cta_order : nullptr;
  a.visited = visited;
  a.status = st;
  return ok();
}

}  // namespace

extern "C" {

const char* rf_last_error(void) { return g_err; }

int rf_version(void) { return 1; }

rf_status rf_debug_set_visited(uint8_t* visited, int64_t visited_len) {
  if (visited != nullptr && visited_len <= 0)
    return fail(RF_ERR_INVALID, "rf_debug_set_visited: visited_len must be > 0");
  g_visited = visited;
  g_visited_len = visited ? visited_len : 0;
  return ok();
}

rf_status rf_debug_inject_fault(int site) {
  if (site != 0 && site != 1) return fail(RF_ERR_INVALID, "rf_debug_inject_fault: unknown site");
  g_fault_site = site;
  return ok();
}

rf_status rf_device_status(rf_stream stream, int* code) {
  if (code == nullptr) return fail(RF_ERR_INVALID, "rf_device_status: code is NULL");
  *code = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "rf_device_status: stream synchronize");
  int* w = rf::status_word();
  if (w == nullptr) return fail(RF_ERR_CUDA, "rf_device_status: no device status word");
  int v = 0;
  e = cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "rf_device_status: read");
  const int zero = 0;
  e = cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "rf_device_status: clear");
  *code = v;
  if (v == 0) return ok();
  const int kind = v >> 16;
  if (kind == rf::kDevTimeout)
    return fail(RF_ERR_TIMEOUT, "device wait gave up (code 0x%x)", v);
  return fail(RF_ERR_INVALID, "device detected invalid data (code 0x%x)", v);
}

rf_status rf_softmax_rows(const void* x, void* y, int64_t rows, int64_t cols, rf_dtype dt,
                          rf_stream stream) {
  if (rows < 0 || cols < 0) return fail(RF_ERR_INVALID, "rf_softmax_rows: negative size");
  if (dt != RF_F32 && dt != RF_BF16) return fail(RF_ERR_INVALID, "rf_softmax_rows: bad dtype");
  if (rows == 0 || cols == 0) return ok();
  if (x == nullptr || y == nullptr) return fail(RF_ERR_INVALID, "rf_softmax_rows: NULL pointer");
  if (rows > INT32_MAX) return fail(RF_ERR_INVALID, "rf_softmax_rows: rows > 2^31-1");
  if (cols > (int64_t(1) << 40)) return fail(RF_ERR_INVALID, "rf_softmax_rows: cols too large");
  int* st = rf::status_word();
  if (st == nullptr) return fail(RF_ERR_CUDA, "rf_softmax_rows: no CUDA device");
  cudaError_t e = rf::launch_softmax_rows(x, y, rows, cols, dt,
                                          reinterpret_cast<cudaStream_t>(stream), st,
                                          g_fault_site == 1);
  if (e != cudaSuccess) return cuda_fail(e, "rf_softmax_rows: launch");
  return ok();
}

rf_status rf_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Hkv, int Sq, int Sk, int d, float scale, int causal,
                      const rf_blockmask* bm, rf_dtype dt, rf_stream stream) {
  rf::AttnArgs a{};
  bool empty = false;
  const rf_status pst = attn_prepare("rf_attn_fwd", q, k, v, o, lse, B, H, Hkv, Sq, Sk, d, scale,
                                     causal, bm, dt, a, &empty);
  if (pst != RF_OK || empty) return pst;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dt == RF_F32) {
    e = rf::launch_attn_simt_f32(a, s);
  } else {
    const char* why = nullptr;
    e = rf::launch_attn_tc_bf16(a, s, &why);
    if (e != cudaSuccess && why != nullptr)
      return fail(RF_ERR_CUDA, "rf_attn_fwd: %s: %s", why, cudaGetErrorString(e));
  }
  if (e != cudaSuccess) return cuda_fail(e, "rf_attn_fwd: launch");
  return ok();
}

rf_status rf_attn_fwd_rowwise(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int Hkv, int Sq, int Sk, int d, float scale,
                              int causal, const rf_blockmask* bm, rf_dtype dt, rf_stream stream) {
  if (d != 64 && d != 128)
    return fail(RF_ERR_UNSUPPORTED, "rf_attn_fwd_rowwise: d must be 64 or 128, got %d", d);
  rf::AttnArgs a{};
  bool empty = false;
  const rf_status pst = attn_prepare("rf_attn_fwd_rowwise", q, k, v, o, lse, B, H, Hkv, Sq, Sk,
                                     d, scale, causal, bm, dt, a, &empty);
  if (pst != RF_OK || empty) return pst;
  cudaError_t e = rf::launch_attn_rowwise(a, dt, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rf_attn_fwd_rowwise: launch");
  return ok();
}

size_t rf_decode_workspace_bytes(int B, int H, int nsplit, int d) {
  if (B < 1 || H < 1 || nsplit < 1 || d < 1) return 0;
  const size_t n = size_t(B) * H * nsplit * (size_t(d) + 1) * sizeof(float);
  return (n + 255) / 256 * 256;
}

rf_status rf_attn_decode_splitk(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int Hkv, int Sk, int d, float scale, int nsplit,
                                float* ws, size_t ws_bytes, rf_dtype dt, rf_stream stream) {
  const rf_status chk = rf::check_decode_args("rf_attn_decode_splitk", q, k, v, o, lse, B, H, Hkv,
                                              Sk, d, scale, nsplit, dt);
  if (chk != RF_OK) return chk;
  if (ws == nullptr) return fail(RF_ERR_INVALID, "rf_attn_decode_splitk: NULL pointer");
  if (!aligned(ws, 16))
    return fail(RF_ERR_INVALID, "rf_attn_decode_splitk: pointers must be 16-byte aligned");
  if (ws_bytes < rf_decode_workspace_bytes(B, H, nsplit, d))
    return fail(RF_ERR_INVALID, "rf_attn_decode_splitk: workspace too small (%zu < %zu)",
                ws_bytes, rf_decode_workspace_bytes(B, H, nsplit, d));
  int* st = rf::status_word();
  if (st == nullptr) return fail(RF_ERR_CUDA, "rf_attn_decode_splitk: no CUDA device");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* o_part = ws;
  float* lse_part = ws + size_t(B) * H * nsplit * d;
  cudaError_t e = rf::launch_decode_partials(q, k, v, o_part, lse_part, B, H, Hkv, Sk, d, scale,
                                             nsplit, s, st);
  if (e != cudaSuccess) return cuda_fail(e, "rf_attn_decode_splitk: partials launch");
  e = rf::launch_splitk_merge(o_part, lse_part, o, lse, int64_t(B) * H, nsplit, d, dt, s);
  if (e != cudaSuccess) return cuda_fail(e, "rf_attn_decode_splitk: merge launch");
  return ok();
}

rf_status rf_attn_decode_partials(const void* q, const void* k, const void* v, float* ws,
                                  size_t ws_bytes, int B, int H, int Hkv, int Sk, int d,
                                  float scale, int nsplit, rf_dtype dt, rf_stream stream) {
  const char* fn = "rf_attn_decode_partials";
  // o is not written: q stands in for it in the shared checks
  const rf_status chk =
      rf::check_decode_args(fn, q, k, v, q, nullptr, B, H, Hkv, Sk, d, scale, nsplit, dt);
  if (chk != RF_OK) return chk;
  if (ws == nullptr) return fail(RF_ERR_INVALID, "%s: NULL pointer", fn);
  if (!aligned(ws, 16)) return fail(RF_ERR_INVALID, "%s: ws must be 16-byte aligned", fn);
  if (ws_bytes < rf_decode_workspace_bytes(B, H, nsplit, d))
    return fail(RF_ERR_INVALID, "%s: workspace too small (%zu < %zu)", fn, ws_bytes,
                rf_decode_workspace_bytes(B, H, nsplit, d));
  int* st = rf::status_word();
  if (st == nullptr) return fail(RF_ERR_CUDA, "%s: no CUDA device", fn);
  float* o_part = ws;
  float* lse_part = ws + size_t(B) * H * nsplit * d;
  cudaError_t e = rf::launch_decode_partials(q, k, v, o_part, lse_part, B, H, Hkv, Sk, d, scale,
                                             nsplit, reinterpret_cast<cudaStream_t>(stream), st);
  if (e != cudaSuccess) return cuda_fail(e, "rf_attn_decode_partials: launch");
  return ok();
}

rf_status rf_splitk_merge(const float* o_part, const float* lse_part, void* o, float* lse,
                          int64_t rows, int nsplit, int d, rf_dtype out_dt, rf_stream stream) {
  if (rows < 0 || nsplit < 1 || d < 1 || d > 1024)
    return fail(RF_ERR_INVALID, "rf_splitk_merge: bad sizes");
  if (out_dt != RF_F32 && out_dt != RF_BF16)
    return fail(RF_ERR_INVALID, "rf_splitk_merge: bad dtype");
  if (rows == 0) return ok();
  if (rows > INT32_MAX) return fail(RF_ERR_INVALID, "rf_splitk_merge: rows > 2^31-1");
  if (o_part == nullptr || lse_part == nullptr || o == nullptr)
    return fail(RF_ERR_INVALID, "rf_splitk_merge: NULL pointer");
  if (!aligned(o_part, 4) || !aligned(lse_part, 4) || !aligned(o, out_dt == RF_F32 ? 4 : 2) ||
      (lse != nullptr && !aligned(lse, 4)))
    return fail(RF_ERR_INVALID, "rf_splitk_merge: misaligned pointer");
  cudaError_t e = rf::launch_splitk_merge(o_part, lse_part, o, lse, rows, nsplit, d, out_dt,
                                          reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rf_splitk_merge: launch");
  return ok();
}

rf_status rf_splitk_merge_strided(const float* o_part, const float* lse_part, void* o, float* lse,
                                  int64_t rows, int nsplit, int d, int64_t o_split_stride,
                                  int64_t o_row_stride, int64_t lse_split_stride,
                                  int64_t lse_row_stride, rf_dtype out_dt, rf_stream stream) {
  const char* fn = "rf_splitk_merge_strided";
  if (rows < 0 || nsplit < 1 || d < 1 || d > 1024)
    return fail(RF_ERR_INVALID, "%s: bad sizes", fn);
  if (out_dt != RF_F32 && out_dt != RF_BF16) return fail(RF_ERR_INVALID, "%s: bad dtype", fn);
  if (o_split_stride < 0 || o_row_stride < 0 || lse_split_stride < 0 || lse_row_stride < 0)
    return fail(RF_ERR_INVALID, "%s: strides must be >= 0", fn);
  if (rows == 0) return ok();
  if (rows > INT32_MAX) return fail(RF_ERR_INVALID, "%s: rows > 2^31-1", fn);
  if (o_part == nullptr || lse_part == nullptr || o == nullptr)
    return fail(RF_ERR_INVALID, "%s: NULL pointer", fn);
  if (!aligned(o_part, 4) || !aligned(lse_part, 4) || !aligned(o, out_dt == RF_F32 ? 4 : 2) ||
      (lse != nullptr && !aligned(lse, 4)))
    return fail(RF_ERR_INVALID, "%s: misaligned pointer", fn);
  cudaError_t e = rf::launch_splitk_merge_strided(
      o_part, lse_part, o, lse, rows, nsplit, d, o_split_stride, o_row_stride, lse_split_stride,
      lse_row_stride, out_dt, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rf_splitk_merge_strided: launch");
  return ok();
}

rf_status rf_blockmask_build(const uint8_t* dense, int nheads, int nqt, int nkt, int32_t* row_ptr,
                             int32_t* col_idx, int64_t col_cap, rf_stream stream) {
  if (nheads < 1 || nqt < 1 || nkt < 1 || col_cap < 0)
    return fail(RF_ERR_INVALID, "rf_blockmask_build: bad sizes");
  if (int64_t(nheads) * nqt * nkt > INT32_MAX)
    return fail(RF_ERR_INVALID, "rf_blockmask_build: mask larger than 2^31-1 tiles");
  if (dense == nullptr || row_ptr == nullptr || (col_cap > 0 && col_idx == nullptr))
    return fail(RF_ERR_INVALID, "rf_blockmask_build: NULL pointer");
  if (!aligned(row_ptr, 4) || (col_idx != nullptr && !aligned(col_idx, 4)))
    return fail(RF_ERR_INVALID, "rf_blockmask_build: misaligned output");
  int* st = rf::status_word();
  if (st == nullptr) return fail(RF_ERR_CUDA, "rf_blockmask_build: no CUDA device");
  cudaError_t e = rf::launch_blockmask_build(dense, nheads, nqt, nkt, row_ptr, col_idx, col_cap,
                                             reinterpret_cast<cudaStream_t>(stream), st);
  if (e != cudaSuccess) return cuda_fail(e, "rf_blockmask_build: launch");
  return ok();
}

rf_status rf_blockmask_counts(const rf_blockmask* bm, int B, int H, int Sq, int Sk, int causal,
                              int64_t* counts, rf_stream stream) {
  const char* fn = "rf_blockmask_counts";
  if (B < 1 || H < 1 || Sq < 0 || Sk < 0 || Sq > (1 << 30) || Sk > (1 << 30))
    return fail(RF_ERR_INVALID, "%s: bad sizes B=%d H=%d Sq=%d Sk=%d", fn, B, H, Sq, Sk);
  if (causal != 0 && causal != 1) return fail(RF_ERR_INVALID, "%s: causal must be 0/1", fn);
  if (counts == nullptr || !aligned(counts, 8))
    return fail(RF_ERR_INVALID, "%s: counts must be an 8-byte aligned device int64[3]", fn);
  const int nqt = static_cast<int>(cdiv(Sq, 128)), nkt = static_cast<int>(cdiv(Sk, 128));
  if (bm != nullptr) {
    if (bm->tile_q != 128 || bm->tile_k != 128)
      return fail(RF_ERR_INVALID, "%s: blockmask tiles must be 128x128", fn);
    if (bm->nqt != nqt || bm->nkt != nkt)
      return fail(RF_ERR_INVALID, "%s: blockmask nqt/nkt (%d,%d) != (%d,%d)", fn, bm->nqt,
                  bm->nkt, nqt, nkt);
    if (bm->per_head != 0 && bm->per_head != 1)
      return fail(RF_ERR_INVALID, "%s: blockmask per_head must be 0/1", fn);
    if (Sq > 0 && Sk > 0 && (bm->row_ptr == nullptr || bm->col_idx == nullptr))
      return fail(RF_ERR_INVALID, "%s: blockmask lists are NULL", fn);
    if (bm->tile_bits != nullptr && bm->bits == nullptr)
      return fail(RF_ERR_INVALID, "%s: blockmask tile_bits without bits", fn);
    if (bm->bits != nullptr && !aligned(bm->bits, 8))
      return fail(RF_ERR_INVALID, "%s: blockmask bits must be 8-byte aligned", fn);
  }
  int* st = rf::status_word();
  if (st == nullptr) return fail(RF_ERR_CUDA, "%s: no CUDA device", fn);
  cudaError_t e = rf::launch_blockmask_counts(
      bm ? bm->row_ptr : nullptr, bm ? bm->col_idx : nullptr, bm ? bm->tile_bits : nullptr,
      bm ? bm->bits : nullptr, bm ? bm->per_head : 0, B, H, Sq, Sk, causal, counts,
      reinterpret_cast<cudaStream_t>(stream), st);
  if (e != cudaSuccess) return cuda_fail(e, "rf_blockmask_counts: launch");
  return ok();
}

int64_t rf_blockmask_cta_order_len(int B, int H, int Sq) {
  if (B < 1 || H < 1 || Sq < 1 || Sq > (1 << 30)) return 0;
  const int64_t pairs = cdiv(cdiv(Sq, 128), 2);
  return int64_t(B) * H * cdiv(pairs, 2);
}

rf_status rf_blockmask_cta_order(const rf_blockmask* bm, int B, int H, int Sq, int32_t* order,
                                 int64_t cap, rf_stream stream) {
  const char* fn = "rf_blockmask_cta_order";
  if (B < 1 || H < 1 || Sq < 1 || Sq > (1 << 30))
    return fail(RF_ERR_INVALID, "%s: bad sizes B=%d H=%d Sq=%d", fn, B, H, Sq);
  if (bm == nullptr || bm->row_ptr == nullptr || !aligned(bm->row_ptr, 4))
    return fail(RF_ERR_INVALID, "%s: blockmask with a 4-byte aligned row_ptr required", fn);
  const int nqt = static_cast<int>(cdiv(Sq, 128));
  if (bm->tile_q != 128 || bm->tile_k != 128 || bm->nqt != nqt)
    return fail(RF_ERR_INVALID, "%s: blockmask tiles must be 128x128 with nqt = %d", fn, nqt);
  if (bm->per_head != 0 && bm->per_head != 1)
    return fail(RF_ERR_INVALID, "%s: blockmask per_head must be 0/1", fn);
  const int64_t items = rf_blockmask_cta_order_len(B, H, Sq);
  if (items > INT32_MAX) return fail(RF_ERR_INVALID, "%s: too many work items", fn);
  if (order == nullptr || !aligned(order, 4) || cap < items)
    return fail(RF_ERR_INVALID, "%s: order must be a 4-byte aligned device int32[%lld]", fn,
                static_cast<long long>(items));
  cudaError_t e = rf::launch_cta_order(bm->row_ptr, bm->per_head, nqt, B * H, order, items,
                                       reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rf_blockmask_cta_order: launch");
  return ok();
}

rf_status rf_blockmask_build_elements(const uint8_t* dense, int nheads, int Sq, int Sk,
                                      int32_t* row_ptr, int32_t* col_idx, int32_t* tile_bits,
                                      uint64_t* bits, int64_t bits_cap, int32_t* n_partial,
                                      rf_stream stream) {
  if (nheads < 1 || Sq < 1 || Sk < 1 || bits_cap < 0)
    return fail(RF_ERR_INVALID, "rf_blockmask_build_elements: bad sizes");
  const int64_t ntiles = int64_t(nheads) * cdiv(Sq, 128) * cdiv(Sk, 128);
  if (ntiles > INT32_MAX / 2)
    return fail(RF_ERR_INVALID, "rf_blockmask_build_elements: more than 2^30 tiles");
  if (dense == nullptr || row_ptr == nullptr || col_idx == nullptr || tile_bits == nullptr)
    return fail(RF_ERR_INVALID, "rf_blockmask_build_elements: NULL pointer");
  if (!aligned(row_ptr, 4) || !aligned(col_idx, 4) || !aligned(tile_bits, 4) ||
      (bits != nullptr && !aligned(bits, 8)) || (n_partial != nullptr && !aligned(n_partial, 4)))
    return fail(RF_ERR_INVALID, "rf_blockmask_build_elements: misaligned output");
  int* st = rf::status_word();
  if (st == nullptr) return fail(RF_ERR_CUDA, "rf_blockmask_build_elements: no CUDA device");
  cudaError_t e = rf::launch_blockmask_build_elements(dense, nheads, Sq, Sk, row_ptr, col_idx,
                                                      tile_bits, bits, bits_cap, n_partial,
                                                      reinterpret_cast<cudaStream_t>(stream), st);
  if (e != cudaSuccess) return cuda_fail(e, "rf_blockmask_build_elements: launch");
  return ok();
}

rf_status rf_moe_route(const void* logits, int64_t T, int E, int k, int renorm, int32_t* idx,
                       float* w, float* lse, rf_dtype dt, rf_stream stream) {
  if (T < 0) return fail(RF_ERR_INVALID, "rf_moe_route: negative T");
  if (dt != RF_F32 && dt != RF_BF16) return fail(RF_ERR_INVALID, "rf_moe_route: bad dtype");
  if (E < 1 || E > 1024) return fail(RF_ERR_INVALID, "rf_moe_route: need 1 <= E <= 1024");
  if (k < 1 || k > E || k > 32) return fail(RF_ERR_INVALID, "rf_moe_route: need 1 <= k <= min(E, 32)");
  if (renorm != 0 && renorm != 1) return fail(RF_ERR_INVALID, "rf_moe_route: renorm must be 0 or 1");
  if (T == 0) return ok();
  if (logits == nullptr || idx == nullptr || w == nullptr)
    return fail(RF_ERR_INVALID, "rf_moe_route: NULL pointer");
  if (cdiv(T, 8) > INT32_MAX) return fail(RF_ERR_INVALID, "rf_moe_route: T too large");
  cudaError_t e = rf::launch_moe_route(logits, T, E, k, renorm, idx, w, lse, dt,
                                       reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rf_moe_route: launch");
  return ok();
}

rf_status rf_row_moments(const void* x, int64_t rows, int64_t cols, float eps, float* mean,
                         float* var, void* y, rf_dtype dt, rf_stream stream) {
  if (rows < 0 || cols < 0) return fail(RF_ERR_INVALID, "rf_row_moments: negative size");
  if (dt != RF_F32 && dt != RF_BF16) return fail(RF_ERR_INVALID, "rf_row_moments: bad dtype");
  if (!(eps >= 0.f) || !std::isfinite(eps))
    return fail(RF_ERR_INVALID, "rf_row_moments: eps must be finite and >= 0");
  if (rows == 0 || cols == 0) return ok();
  if (x == nullptr) return fail(RF_ERR_INVALID, "rf_row_moments: x is NULL");
  if (rows > INT32_MAX) return fail(RF_ERR_INVALID, "rf_row_moments: rows > 2^31-1");
  if (cols > (int64_t(1) << 40)) return fail(RF_ERR_INVALID, "rf_row_moments: cols too large");
  cudaError_t e = rf::launch_row_moments(x, rows, cols, eps, mean, var, y, dt,
                                         reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rf_row_moments: launch");
  return ok();
}

rf_status rf_moment_of_inertia(const float* points, const float* masses, int64_t sets,
                               int64_t n, float* total_mass, float* center, float* inertia,
                               rf_stream stream) {
  if (sets < 0 || n < 0) return fail(RF_ERR_INVALID, "rf_moment_of_inertia: negative size");
  if (sets > INT32_MAX) return fail(RF_ERR_INVALID, "rf_moment_of_inertia: sets > 2^31-1");
  if (n > (int64_t(1) << 40)) return fail(RF_ERR_INVALID, "rf_moment_of_inertia: n too large");
  if (sets == 0) return ok();
  if (n > 0 && points == nullptr)
    return fail(RF_ERR_INVALID, "rf_moment_of_inertia: points is NULL");
  if (!aligned(points, 4) || !aligned(masses, 4))
    return fail(RF_ERR_INVALID, "rf_moment_of_inertia: points and masses must be 4-byte aligned");
  cudaError_t e = rf::launch_moment_of_inertia(points, masses, sets, n, total_mass, center,
                                               inertia, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rf_moment_of_inertia: launch");
  return ok();
}

rf_status rf_rowquant_e4m3(const void* x, int64_t rows, int64_t K, uint8_t* q, float* scale,
                           rf_dtype dt, rf_stream stream) {
  if (rows < 0 || K < 0) return fail(RF_ERR_INVALID, "rf_rowquant_e4m3: negative size");
  if (dt != RF_F32 && dt != RF_BF16) return fail(RF_ERR_INVALID, "rf_rowquant_e4m3: bad dtype");
  if (rows == 0) return ok();
  if (K == 0 || K % 16 != 0) return fail(RF_ERR_UNSUPPORTED, "rf_rowquant_e4m3: K must be a positive multiple of 16");
  if (K * (dt == RF_F32 ? 4 : 2) > 64 * 1024)
    return fail(RF_ERR_UNSUPPORTED, "rf_rowquant_e4m3: rows longer than 64 KB");
  if (rows > INT32_MAX) return fail(RF_ERR_INVALID, "rf_rowquant_e4m3: rows > 2^31-1");
  if (x == nullptr || q == nullptr || scale == nullptr)
    return fail(RF_ERR_INVALID, "rf_rowquant_e4m3: NULL pointer");
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scale, 4))
    return fail(RF_ERR_INVALID, "rf_rowquant_e4m3: x and q must be 16-byte aligned");
  cudaError_t e = rf::launch_rowquant_e4m3(x, rows, K, q, scale, dt,
                                           reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rf_rowquant_e4m3: launch");
  return ok();
}

rf_status rf_fp8_gemm(const uint8_t* a, const float* sa, const uint8_t* w, const float* sw, void* c,
                      int M, int N, int K, rf_stream stream) {
  if (M < 0 || N < 0 || K < 0) return fail(RF_ERR_INVALID, "rf_fp8_gemm: negative size");
  if (M == 0 || N == 0) return ok();
  if (M % 128 != 0 || N % 256 != 0 || K % 128 != 0 || K == 0)
    return fail(RF_ERR_UNSUPPORTED,
                "rf_fp8_gemm: M must be a multiple of 128, N of 256, K a positive multiple of 128");
  if (a == nullptr || sa == nullptr || w == nullptr || sw == nullptr || c == nullptr)
    return fail(RF_ERR_INVALID, "rf_fp8_gemm: NULL pointer");
  if (!aligned(a, 16) || !aligned(w, 16) || !aligned(c, 16) || !aligned(sa, 4) || !aligned(sw, 4))
    return fail(RF_ERR_INVALID, "rf_fp8_gemm: a, w, c must be 16-byte aligned");
  if (int64_t(M / 128) * (N / 256) > INT32_MAX)
    return fail(RF_ERR_INVALID, "rf_fp8_gemm: too many tiles");
  int* st = rf::status_word();
  if (st == nullptr) return fail(RF_ERR_CUDA, "rf_fp8_gemm: no CUDA device");
  const char* why = nullptr;
  cudaError_t e = rf::launch_fp8_gemm(a, sa, w, sw, c, M, N, K,
                                      reinterpret_cast<cudaStream_t>(stream), st, &why);
  if (e != cudaSuccess && why != nullptr)
    return fail(RF_ERR_CUDA, "rf_fp8_gemm: %s: %s", why, cudaGetErrorString(e));
  if (e != cudaSuccess) return cuda_fail(e, "rf_fp8_gemm: launch");
  return ok();
}

size_t rf_mla_decode_workspace_bytes(int B, int nsplit) {
  return rf_decode_workspace_bytes(B, 128, nsplit, 512);
}

rf_status rf_mla_decode(const void* q, const void* kv, void* o, float* lse, int B, int Sk,
                        float scale, int nsplit, float* ws, size_t ws_bytes, rf_stream stream) {
  if (B < 1 || Sk < 1) return fail(RF_ERR_INVALID, "rf_mla_decode: bad sizes");
  if (nsplit < 1 || nsplit > Sk) return fail(RF_ERR_INVALID, "rf_mla_decode: need 1 <= nsplit <= Sk");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(RF_ERR_INVALID, "rf_mla_decode: scale must be finite and > 0");
  if (int64_t(B) * nsplit * 2 > INT32_MAX) return fail(RF_ERR_INVALID, "rf_mla_decode: too many splits");
  if (int64_t(B) * Sk * 576 * 2 > (int64_t(1) << 46))
    return fail(RF_ERR_INVALID, "rf_mla_decode: tensors too large");
  if (q == nullptr || kv == nullptr || o == nullptr || ws == nullptr)
    return fail(RF_ERR_INVALID, "rf_mla_decode: NULL pointer");
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(o, 16) || !aligned(ws, 16))
    return fail(RF_ERR_INVALID, "rf_mla_decode: pointers must be 16-byte aligned");
  if (lse != nullptr && !aligned(lse, 4))
    return fail(RF_ERR_INVALID, "rf_mla_decode: lse must be 4-byte aligned");
  if (ws_bytes < rf_mla_decode_workspace_bytes(B, nsplit))
    return fail(RF_ERR_INVALID, "rf_mla_decode: workspace too small (%zu < %zu)", ws_bytes,
                rf_mla_decode_workspace_bytes(B, nsplit));
  int* st = rf::status_word();
  if (st == nullptr) return fail(RF_ERR_CUDA, "rf_mla_decode: no CUDA device");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* o_part = ws;
  float* lse_part = ws + size_t(B) * 128 * nsplit * 512;
  const char* why = nullptr;
  cudaError_t e = rf::launch_mla_decode_partials(q, kv, o_part, lse_part, B, Sk, nsplit, scale, s,
                                                 st, &why);
  if (e != cudaSuccess && why != nullptr)
    return fail(RF_ERR_CUDA, "rf_mla_decode: %s: %s", why, cudaGetErrorString(e));
  if (e != cudaSuccess) return cuda_fail(e, "rf_mla_decode: partials launch");
  e = rf::launch_splitk_merge(o_part, lse_part, o, lse, int64_t(B) * 128, nsplit, 512, RF_BF16, s);
  if (e != cudaSuccess) return cuda_fail(e, "rf_mla_decode: merge launch");
  return ok();
}

}  // extern "C"
