// decode_noalloc.cu -- split-K decode for callers that cannot allocate.
//
// rf_attn_decode_splitk needs a device workspace for the per-split partials,
// which the caller allocates. Some callers cannot call cudaMalloc: a plug-in
// loaded into a host process whose runtime owns every byte of device memory,
// or a latency-critical serving loop whose policy forbids allocation once it
// has started. For them this file provides rf_attn_decode_splitk_noalloc,
// which takes the partials from a fixed-size array that lives in the
// library's own device image (file-scope __device__ storage, reserved on every
// GPU that loads the library and held until the process exits) and then runs
// exactly the allocating entry point's kernels on it.
//
// The array's name, used in host code, stands for a host-side shadow, not a
// device address. The device address is looked up with cudaGetSymbolAddress
// (with the device current) and cached per device, tagged with the current
// context's unique id: after cudaDeviceReset, or once the primary context has
// been released and created again, the module is loaded anew and the array
// may sit elsewhere, so a changed id forces a new lookup.
#include <cstdio>

#include "rf_internal.h"

namespace {

// Largest workspace the array holds: 16 MiB (4 Mi floats). The split-K decode
// workload B=16, H=32, nsplit=32, d=128 needs 8.45 MB of it.
constexpr size_t kScratchBytes = size_t(16) << 20;

__device__ __align__(256) float g_decode_scratch[kScratchBytes / sizeof(float)];

rf::SymbolCache g_scratch_cache;

}  // namespace

extern "C" rf_status rf_attn_decode_splitk_noalloc(const void* q, const void* k, const void* v,
                                                   void* o, float* lse, int B, int H, int Hkv,
                                                   int Sk, int d, float scale, int nsplit,
                                                   rf_dtype dt, rf_stream stream) {
  // every argument is checked on the host before any CUDA call
  const rf_status chk = rf::check_decode_args("rf_attn_decode_splitk_noalloc", q, k, v, o, lse,
                                              B, H, Hkv, Sk, d, scale, nsplit, dt);
  if (chk != RF_OK) return chk;
  const size_t need = rf_decode_workspace_bytes(B, H, nsplit, d);
  if (need > kScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "rf_attn_decode_splitk_noalloc: partials need %zu bytes, more than the %zu-byte "
             "static workspace (use rf_attn_decode_splitk with a caller workspace)",
             need, kScratchBytes);
    return rf::set_last_error(RF_ERR_INVALID, msg);
  }
  cudaError_t e = cudaSuccess;
  float* ws = static_cast<float*>(rf::symbol_address(g_decode_scratch, g_scratch_cache, &e));
  if (ws == nullptr) {
    char msg[200];
    snprintf(msg, sizeof(msg), "rf_attn_decode_splitk_noalloc: static workspace lookup: %s",
             cudaGetErrorString(e));
    return rf::set_last_error(RF_ERR_CUDA, msg);
  }
  // On success every partial the merge reads was written earlier in the same
  // call, so the array needs no clearing between calls. A partials CTA that
  // gives up on a timed-out wait returns without writing its split; O and LSE
  // are then undefined (they may mix in an earlier call's partials) and
  // rf_device_status reports RF_ERR_TIMEOUT.
  return rf_attn_decode_splitk(q, k, v, o, lse, B, H, Hkv, Sk, d, scale, nsplit, ws, kScratchBytes,
                               dt, stream);
}
