// attn_host.cu -- attention forward on host buffers: the copies in and out
// overlap the kernels.
//
// rf_attn_fwd_host takes Q, K, V and returns O and LSE in host memory. The
// work is cut into chunks of whole (batch, KV-head group) slices, which are
// independent problems of the same kind (RedFuser technical summary, section
// 3: partitions of the single-segment strategy need no merge when they do not
// share a reduction axis). Chunk c moves through three streams:
//   copy-in stream:      Q_c, K_c, V_c host -> device slot c % 2
//   compute stream c % 2: rf_attn_fwd on the slot
//   copy-out stream:     O_c, LSE_c device slot -> host
// so that the copy-in of chunk c + 1, the kernel of chunk c and the copy-out
// of chunk c - 1 run at the same time. The kernels of consecutive chunks are
// on two streams, so the next chunk's CTAs start on the SMs that the current
// chunk's last partial wave leaves idle (a chunk is a few waves; one CTA of
// the attention kernel fills an SM's shared memory, so CTAs of the two
// kernels never share an SM). Two slots of device workspace, owned by the
// caller, hold the chunks in flight. Events order the streams; the caller's
// stream waits for the last copy-out, so the call is ordered on it like any
// other entry point and nothing here synchronises the host.
#include <cstdio>
#include <mutex>

#include "rf_internal.h"

namespace rf {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kTargetChunks = 8;

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// KV heads per chunk: the largest divisor of Hkv that still gives about
// kTargetChunks chunks over the batch (whole batch elements when B is large).
int kv_heads_per_chunk(int B, int Hkv) {
  const int want = (kTargetChunks + B - 1) / B;  // chunks per batch element
  for (int parts = 1; parts <= Hkv; ++parts)
    if (Hkv % parts == 0 && parts >= want) return Hkv / parts;
  return 1;
}

// Device bytes of one slot: Q, K, V, O and LSE of one chunk, 256-byte aligned.
struct SlotLayout {
  size_t q, k, v, o, lse, total;
};

SlotLayout slot_layout(int H, int Hkv, int Sq, int Sk, int d, int hkv_c, size_t esz) {
  const int hq_c = hkv_c * (H / Hkv);
  SlotLayout L{};
  L.q = 0;
  L.k = L.q + align256(size_t(hq_c) * Sq * d * esz);
  L.v = L.k + align256(size_t(hkv_c) * Sk * d * esz);
  L.o = L.v + align256(size_t(hkv_c) * Sk * d * esz);
  L.lse = L.o + align256(size_t(hq_c) * Sq * d * esz);
  L.total = L.lse + align256(size_t(hq_c) * Sq * sizeof(float));
  return L;
}

// Streams and events of one device, created on first use and kept for the
// life of the process; the mutex covers enqueueing (an event may be recorded
// again once the waits on its previous record have been enqueued).
struct DeviceQueues {
  std::mutex mu;
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr, comp[2] = {nullptr, nullptr};
  cudaEvent_t entry = nullptr, loaded[2] = {nullptr, nullptr}, computed[2] = {nullptr, nullptr},
              stored[2] = {nullptr, nullptr};
};
DeviceQueues g_queues[kMaxDevices];

cudaError_t queues_init(DeviceQueues& Q) {
  if (Q.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&Q.in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&Q.out, cudaStreamNonBlocking);
  for (int i = 0; i < 2 && e == cudaSuccess; ++i)
    e = cudaStreamCreateWithFlags(&Q.comp[i], cudaStreamNonBlocking);
  cudaEvent_t* evs[7] = {&Q.entry, &Q.loaded[0], &Q.loaded[1], &Q.computed[0],
                         &Q.computed[1], &Q.stored[0], &Q.stored[1]};
  for (int i = 0; i < 7 && e == cudaSuccess; ++i)
    e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming);
  if (e == cudaSuccess) Q.ready = true;
  return e;
}

}  // namespace
}  // namespace rf

extern "C" size_t rf_attn_fwd_host_workspace_bytes(int B, int H, int Hkv, int Sq, int Sk, int d,
                                                   rf_dtype dt) {
  if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || Sq < 0 || Sk < 0 || d < 1) return 0;
  if (dt != RF_F32 && dt != RF_BF16) return 0;
  const size_t esz = dt == RF_F32 ? 4 : 2;
  const int hkv_c = rf::kv_heads_per_chunk(B, Hkv);
  return 2 * rf::slot_layout(H, Hkv, Sq, Sk, d, hkv_c, esz).total;
}

extern "C" rf_status rf_attn_fwd_host(const void* q, const void* k, const void* v, void* o,
                                      float* lse, int B, int H, int Hkv, int Sq, int Sk, int d,
                                      float scale, int causal, const rf_blockmask* blockmask,
                                      rf_dtype dt, void* ws, size_t ws_bytes, rf_stream stream) {
  using namespace rf;
  if (B < 1 || H < 1 || Hkv < 1 || Sq < 0 || Sk < 0 || d < 1 || H % Hkv != 0)
    return set_last_error(RF_ERR_INVALID, "rf_attn_fwd_host: bad sizes");
  if (dt != RF_F32 && dt != RF_BF16)
    return set_last_error(RF_ERR_INVALID, "rf_attn_fwd_host: bad dtype");
  if (Sq == 0) return rf_attn_fwd(q, k, v, o, lse, B, H, Hkv, Sq, Sk, d, scale, causal,
                                  blockmask, dt, stream);
  if (q == nullptr || o == nullptr || (Sk > 0 && (k == nullptr || v == nullptr)))
    return set_last_error(RF_ERR_INVALID, "rf_attn_fwd_host: NULL host pointer");
  int64_t vlen = 0;
  if (debug_visited(&vlen) != nullptr)
    return set_last_error(RF_ERR_INVALID,
                          "rf_attn_fwd_host: the visited-tile debug buffer is not supported here");
  const size_t need = rf_attn_fwd_host_workspace_bytes(B, H, Hkv, Sq, Sk, d, dt);
  if (ws == nullptr || ws_bytes < need || reinterpret_cast<uintptr_t>(ws) % 256 != 0)
    return set_last_error(RF_ERR_INVALID,
                          "rf_attn_fwd_host: workspace must be 256-byte aligned and hold "
                          "rf_attn_fwd_host_workspace_bytes() bytes");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return set_last_error(RF_ERR_CUDA, "rf_attn_fwd_host: no CUDA device");

  const size_t esz = dt == RF_F32 ? 4 : 2;
  const int G = H / Hkv;
  const int hkv_c = kv_heads_per_chunk(B, Hkv), hq_c = hkv_c * G;
  const int per_b = Hkv / hkv_c, chunks = B * per_b;
  const SlotLayout L = slot_layout(H, Hkv, Sq, Sk, d, hkv_c, esz);
  const int nqt = (Sq + 127) / 128;
  const size_t q_bytes = size_t(hq_c) * Sq * d * esz, kv_bytes = size_t(hkv_c) * Sk * d * esz;
  const size_t lse_bytes = size_t(hq_c) * Sq * sizeof(float);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  DeviceQueues& Qs = g_queues[dev];
  std::lock_guard<std::mutex> guard(Qs.mu);
  cudaError_t e = queues_init(Qs);
#define RF_CK(call, what)                                                        \
  do {                                                                           \
    if ((e = (call)) != cudaSuccess) {                                           \
      char msg[160];                                                             \
      snprintf(msg, sizeof(msg), "rf_attn_fwd_host: %s: %s", what, cudaGetErrorString(e)); \
      return set_last_error(RF_ERR_CUDA, msg);                                   \
    }                                                                            \
  } while (0)
  RF_CK(e, "stream/event setup");
  // nothing is copied before the caller's earlier work on its stream is done
  RF_CK(cudaEventRecord(Qs.entry, s), "record");
  RF_CK(cudaStreamWaitEvent(Qs.in, Qs.entry, 0), "wait");
  RF_CK(cudaStreamWaitEvent(Qs.out, Qs.entry, 0), "wait");
  for (int i = 0; i < 2; ++i) RF_CK(cudaStreamWaitEvent(Qs.comp[i], Qs.entry, 0), "wait");
  for (int c = 0; c < chunks; ++c) {
    const int slot = c & 1;
    const int b = c / per_b, g0 = (c % per_b) * hkv_c, h0 = g0 * G;
    unsigned char* base = static_cast<unsigned char*>(ws) + slot * L.total;
    const size_t q_off = (size_t(b) * H + h0) * Sq * d * esz;
    const size_t kv_off = (size_t(b) * Hkv + g0) * Sk * d * esz;
    // a slot is refilled once its previous chunk has been copied out
    if (c >= 2) RF_CK(cudaStreamWaitEvent(Qs.in, Qs.stored[slot], 0), "wait");
    RF_CK(cudaMemcpyAsync(base + L.q, static_cast<const unsigned char*>(q) + q_off, q_bytes,
                          cudaMemcpyHostToDevice, Qs.in), "copy in");
    if (Sk > 0) {
      RF_CK(cudaMemcpyAsync(base + L.k, static_cast<const unsigned char*>(k) + kv_off, kv_bytes,
                            cudaMemcpyHostToDevice, Qs.in), "copy in");
      RF_CK(cudaMemcpyAsync(base + L.v, static_cast<const unsigned char*>(v) + kv_off, kv_bytes,
                            cudaMemcpyHostToDevice, Qs.in), "copy in");
    }
    RF_CK(cudaEventRecord(Qs.loaded[slot], Qs.in), "record");
    cudaStream_t cs = Qs.comp[slot];
    RF_CK(cudaStreamWaitEvent(cs, Qs.loaded[slot], 0), "wait");
    rf_blockmask bm_c;
    const rf_blockmask* bmp = nullptr;
    if (blockmask != nullptr) {
      bm_c = *blockmask;
      bm_c.cta_order = nullptr;  // an order for the whole problem does not fit a chunk's grid
      if (bm_c.per_head && bm_c.row_ptr != nullptr)
        bm_c.row_ptr += (int64_t(b) * H + h0) * nqt;  // this chunk's heads
      bmp = &bm_c;
    }
    const rf_status st = rf_attn_fwd(base + L.q, base + L.k, base + L.v, base + L.o,
                                     lse ? reinterpret_cast<float*>(base + L.lse) : nullptr, 1,
                                     hq_c, hkv_c, Sq, Sk, d, scale, causal, bmp, dt,
                                     reinterpret_cast<rf_stream>(cs));
    if (st != RF_OK) return st;  // message set by rf_attn_fwd
    RF_CK(cudaEventRecord(Qs.computed[slot], cs), "record");
    RF_CK(cudaStreamWaitEvent(Qs.out, Qs.computed[slot], 0), "wait");
    RF_CK(cudaMemcpyAsync(static_cast<unsigned char*>(o) + q_off, base + L.o, q_bytes,
                          cudaMemcpyDeviceToHost, Qs.out), "copy out");
    if (lse != nullptr)
      RF_CK(cudaMemcpyAsync(lse + (size_t(b) * H + h0) * Sq, base + L.lse, lse_bytes,
                            cudaMemcpyDeviceToHost, Qs.out), "copy out");
    RF_CK(cudaEventRecord(Qs.stored[slot], Qs.out), "record");
  }
  // the caller's stream resumes after the last copy out (which follows every
  // kernel: each chunk's copy out waits for its kernel, and the copy-out
  // stream is in order)
  RF_CK(cudaStreamWaitEvent(s, Qs.stored[(chunks - 1) & 1], 0), "wait");
#undef RF_CK
  return set_last_error(RF_OK, "");
}
