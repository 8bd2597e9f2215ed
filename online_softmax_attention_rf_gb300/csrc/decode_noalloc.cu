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
// device address, so the device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached.
#include <atomic>
#include <cstdio>

#include "rf_internal.h"

namespace {

// Largest workspace the array holds: 16 MiB (4 Mi floats). The split-K decode
// workload B=16, H=32, nsplit=32, d=128 needs 8.45 MB of it.
constexpr size_t kScratchBytes = size_t(16) << 20;

__device__ __align__(256) float g_decode_scratch[kScratchBytes / sizeof(float)];

std::atomic<float*> g_scratch_addr[128];

// Device address of the array on the current device, looked up on first use.
float* scratch_address(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev >= 0 && dev < 128) {
    float* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p != nullptr) return p;
  }
  float* p = nullptr;
  *err = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_decode_scratch);
  if (*err != cudaSuccess) return nullptr;
  if (dev >= 0 && dev < 128) g_scratch_addr[dev].store(p, std::memory_order_release);
  return p;
}

}  // namespace

extern "C" rf_status rf_attn_decode_splitk_noalloc(const void* q, const void* k, const void* v,
                                                   void* o, float* lse, int B, int H, int Hkv,
                                                   int Sk, int d, float scale, int nsplit,
                                                   rf_dtype dt, rf_stream stream) {
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
  float* ws = scratch_address(&e);
  if (ws == nullptr) {
    char msg[200];
    snprintf(msg, sizeof(msg), "rf_attn_decode_splitk_noalloc: static workspace lookup: %s",
             cudaGetErrorString(e));
    return rf::set_last_error(RF_ERR_CUDA, msg);
  }
  // every partial the kernels read is written by them first in the same call,
  // so nothing in the array needs clearing between calls
  return rf_attn_decode_splitk(q, k, v, o, lse, B, H, Hkv, Sk, d, scale, nsplit, ws, kScratchBytes,
                               dt, stream);
}
