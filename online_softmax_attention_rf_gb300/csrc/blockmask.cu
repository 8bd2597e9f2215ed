// blockmask.cu -- dense tile mask -> row-compressed (BSR) tile lists.
//
// Accelerating Sparse Transformer Inference on GPU (STOF), Méthodologie,
// unified MHA module: the mask is kept as row-compressed lists of outer tiles,
// so that the attention kernel skips absent tiles entirely. The FLASHLIGHT
// summary (Risultati) notes that building block masks at run time is itself
// a cost; this kernel does it on the device in one launch.
//
// One CTA: (1) one warp per row counts the present tiles with ballots,
// (2) the CTA scans the counts into row_ptr, (3) one warp per row writes the
// column indices in ascending order (ballot + prefix popcount).
#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads) blockmask_build_kernel(
    const uint8_t* __restrict__ dense, int64_t nrows, int nkt, int32_t* __restrict__ row_ptr,
    int32_t* __restrict__ col_idx, int64_t col_cap, int* status) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = kThreads / 32;
  // (1) counts into row_ptr[r + 1]
  for (int64_t r = warp; r < nrows; r += nw) {
    const uint8_t* row = dense + r * nkt;
    int cnt = 0;
    for (int c0 = 0; c0 < nkt; c0 += 32) {
      const int c = c0 + lane;
      cnt += __popc(__ballot_sync(0xffffffffu, c < nkt && row[c] != 0));
    }
    if (lane == 0) row_ptr[r + 1] = cnt;
  }
  if (threadIdx.x == 0) {
    row_ptr[0] = 0;
    carry = 0;
  }
  __syncthreads();
  // (2) inclusive scan of row_ptr[1 .. nrows], 1024 rows at a time
  for (int64_t base = 0; base < nrows; base += kThreads) {
    const int64_t r = base + threadIdx.x;
    int32_t v = r < nrows ? row_ptr[r + 1] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int32_t w = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += t;
      }
      warp_tot[lane] = w;  // inclusive per-warp totals
    }
    __syncthreads();
    const int32_t add = carry + (warp > 0 ? warp_tot[warp - 1] : 0);
    if (r < nrows) row_ptr[r + 1] = v + add;
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_tot[nw - 1];
    __syncthreads();
  }
  // (3) column indices, ascending within each row
  bool overflow = false;
  for (int64_t r = warp; r < nrows; r += nw) {
    const uint8_t* row = dense + r * nkt;
    int64_t pos = row_ptr[r];
    for (int c0 = 0; c0 < nkt; c0 += 32) {
      const int c = c0 + lane;
      const bool set = c < nkt && row[c] != 0;
      const unsigned bal = __ballot_sync(0xffffffffu, set);
      if (set) {
        const int64_t at = pos + __popc(bal & ((1u << lane) - 1u));
        if (at < col_cap)
          col_idx[at] = c;
        else
          overflow = true;
      }
      pos += __popc(bal);
    }
  }
  if (overflow) record_status(status, dev_code(kDevCapacity, kKerBlockmask, 1));
}

}  // namespace

cudaError_t launch_blockmask_build(const uint8_t* dense, int nheads, int nqt, int nkt,
                                   int32_t* row_ptr, int32_t* col_idx, int64_t col_cap,
                                   cudaStream_t s, int* status) {
  blockmask_build_kernel<<<1, kThreads, 0, s>>>(dense, int64_t(nheads) * nqt, nkt, row_ptr,
                                                col_idx, col_cap, status);
  return cudaGetLastError();
}

}  // namespace rf
