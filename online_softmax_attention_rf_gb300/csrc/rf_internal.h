// rf_internal.h -- declarations shared by the host entry points and the
// kernel translation units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "rf.h"

// Upper bound on any single device-side wait (mbarrier phase, TMEM, peer).
// Far above any legitimate wait in these kernels (microseconds), far below a
// watchdog: a wait that exceeds it records a status code and unwinds.
#define RF_WAIT_LIMIT_NS 2000000000ull

namespace rf {

// Device status word codes: (kind << 16) | (kernel << 8) | site.
enum DevKind : int { kDevTimeout = 1, kDevBadList = 2, kDevCapacity = 3 };
enum DevKernel : int {
  kKerSoftmax = 1,
  kKerAttnSimt = 2,
  kKerAttnTc = 3,
  kKerDecode = 4,
  kKerMerge = 5,
  kKerBlockmask = 6,
  kKerFp8 = 7,
  kKerMla = 8
};

__host__ __device__ constexpr int dev_code(int kind, int kernel, int site) {
  return (kind << 16) | (kernel << 8) | site;
}

// Device address of the status word for the current device (nullptr on error).
int* status_word();

// Device addresses of one __device__ variable, one per device, each tagged
// with the unique id of the context it was looked up in. A context that was
// torn down and created again (cudaDeviceReset, a primary context released
// and retained) gets a new id and may hold the variable at another address,
// so a tag that no longer matches the current context forces a new lookup.
struct SymbolCache {
  std::mutex mu;
  unsigned long long ctx_id[128] = {};
  void* ptr[128] = {};
};

// Device address of `symbol` (the host-side name of a __device__ variable of
// this library) in the calling thread's current context: the cached address
// when the context's id matches, else cudaGetSymbolAddress (which makes the
// device's primary context current if none is). Returns nullptr and sets
// *err on failure.
void* symbol_address(const void* symbol, SymbolCache& cache, cudaError_t* err);

// Host-side checks shared by rf_attn_decode_splitk and its allocation-free
// variant: everything but the workspace. `who` names the entry point in the
// message. Makes no CUDA call.
rf_status check_decode_args(const char* who, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, int B, int H, int Hkv, int Sk,
                            int d, float scale, int nsplit, rf_dtype dt);

// Sets this thread's rf_last_error() message and returns st.
rf_status set_last_error(rf_status st, const char* msg);

// Visited-tile debug buffer for the calling host thread (nullptr = off).
uint8_t* debug_visited(int64_t* len);

// Arguments of one attention-forward launch (validated on the host).
struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, Hkv, Sq, Sk, d;
  float scale;
  int causal;
  // block-sparse lists (row_ptr == nullptr: dense)
  const int32_t* row_ptr;
  const int32_t* col_idx;
  int per_head;
  // inner level of the two-level mask (tile_bits == nullptr: all tiles full)
  const int32_t* tile_bits;
  const uint64_t* bits;
  int nqt, nkt;
  const int32_t* cta_order;  // optional work order of the tensor-core kernel (nullptr: head-major)
  uint8_t* visited;  // optional debug output, [B*H*nqt*nkt]
  int* status;
};

// Each launcher validates nothing (the entry points do) and returns the
// launch error, if any.
// skip_first_copy: fault injection (rf_debug_inject_fault site 1).
cudaError_t launch_softmax_rows(const void* x, void* y, int64_t rows, int64_t cols,
                                rf_dtype dt, cudaStream_t s, int* status,
                                bool skip_first_copy = false);
cudaError_t launch_attn_simt_f32(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_attn_tc_bf16(const AttnArgs& a, cudaStream_t s, const char** why);
cudaError_t launch_attn_rowwise(const AttnArgs& a, rf_dtype dt, cudaStream_t s);
cudaError_t launch_decode_partials(const void* q, const void* k, const void* v, float* o_part,
                                   float* lse_part, int B, int H, int Hkv, int Sk, int d,
                                   float scale, int nsplit, cudaStream_t s, int* status);
cudaError_t launch_splitk_merge(const float* o_part, const float* lse_part, void* o, float* lse,
                                int64_t rows, int nsplit, int d, rf_dtype out_dt,
                                cudaStream_t s);
// Partial s of row r at o_part + s * o_split + r * o_row and
// lse_part[s * l_split + r * l_row] (element strides).
cudaError_t launch_splitk_merge_strided(const float* o_part, const float* lse_part, void* o,
                                        float* lse, int64_t rows, int nsplit, int d,
                                        int64_t o_split, int64_t o_row, int64_t l_split,
                                        int64_t l_row, rf_dtype out_dt, cudaStream_t s);
cudaError_t launch_blockmask_build(const uint8_t* dense, int nheads, int nqt, int nkt,
                                   int32_t* row_ptr, int32_t* col_idx, int64_t col_cap,
                                   cudaStream_t s, int* status);
cudaError_t launch_rowquant_e4m3(const void* x, int64_t rows, int64_t K, uint8_t* q, float* scale,
                                 rf_dtype dt, cudaStream_t s);
cudaError_t launch_fp8_gemm(const uint8_t* a, const float* sa, const uint8_t* w, const float* sw,
                            void* c, int M, int N, int K, cudaStream_t s, int* status,
                            const char** why);
cudaError_t launch_mla_decode_partials(const void* q, const void* kv, float* o_part,
                                       float* lse_part, int B, int Sk, int nsplit, float scale,
                                       cudaStream_t s, int* status, const char** why);
cudaError_t launch_moe_route(const void* logits, int64_t T, int E, int k, int renorm,
                             int32_t* idx, float* w, float* lse, rf_dtype dt, cudaStream_t s);
cudaError_t launch_moment_of_inertia(const float* points, const float* masses, int64_t sets,
                                     int64_t n, float* total, float* centre, float* inertia,
                                     cudaStream_t s);
cudaError_t launch_row_moments(const void* x, int64_t rows, int64_t cols, float eps, float* mean,
                               float* var, void* y, rf_dtype dt, cudaStream_t s);
// order[c] for c < items: the double items whose listed tiles exceed twice
// the mean first, then the others, both ascending (one CTA).
cudaError_t launch_cta_order(const int32_t* row_ptr, int per_head, int nqt, int BH, int32_t* order,
                             int64_t items, cudaStream_t s);
cudaError_t launch_blockmask_counts(const int32_t* row_ptr, const int32_t* col_idx,
                                    const int32_t* tile_bits, const uint64_t* bits, int per_head,
                                    int B, int H, int Sq, int Sk, int causal, int64_t* counts,
                                    cudaStream_t s, int* status);
cudaError_t launch_blockmask_build_elements(const uint8_t* dense, int nheads, int Sq, int Sk,
                                            int32_t* row_ptr, int32_t* col_idx,
                                            int32_t* tile_bits, uint64_t* bits, int64_t bits_cap,
                                            int32_t* n_partial, cudaStream_t s, int* status);

}  // namespace rf
