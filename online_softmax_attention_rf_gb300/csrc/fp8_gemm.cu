// fp8_gemm.cu -- per-row FP8 absmax quantisation and the GEMM over the codes.
//
// RedFuser: An Automatic Operator Fusion Framework for Cascaded Reductions on
// AI Accelerators -- technical summary, sections 1 and 4: FP8 quantisation
// followed by GEMM is a cascade of reductions (the row's absolute maximum,
// then the dot products over the codes it scales).
//
// Quantisation (one CTA per row, the row staged once in shared memory by
// 16-byte cp.async): amax = max |x| over the row (block reduction), then each
// element becomes the E4M3 code of float32(x) * (448 / amax), rounded to
// nearest even and saturated (cvt.rn.satfinite.e4m3x2.f32); the row's scale is
// amax / 448 (an all-zero row: codes 0, scale 1). The row is read from HBM
// once and the codes written once.
//
// GEMM: C[m, n] = sa[m] * sw[n] * sum_k A[m, k] W[n, k] with A [M, K] and
// W [N, K] E4M3 codes (both K-major), C bf16 [M, N], in 128 x 256 tiles of
// C. Persistent: one CTA per SM walks the tiles (grouped 16 row tiles wide
// so that the tiles in flight share operands in L2). A TMA producer (one
// lane) streams 128-byte-deep K slices of A (128 rows) and W (256 rows) into
// a 4-stage ring with 128-byte swizzle and an L2 evict-last hint; one lane
// issues tcgen05.mma kind::f8f6f4 (M = 128, N = 256, K = 32 per instruction)
// into one of two f32 accumulators of 256 tensor-memory columns each and
// releases every stage with a commit; four epilogue warps read a finished
// accumulator (tcgen05.ld, lane = row), apply both scales and write bf16
// with an evict-first hint while the next tile accumulates in the other
// buffer. Every wait is bounded; on expiry the status word records the site
// and the roles unwind.
#include <cudaTypedefs.h>

#include <mutex>

#include "rf_device.cuh"

namespace rf {
namespace {

// ------------------------------------------------------------ quantisation

constexpr int kQThreads = 256;
constexpr int kQRowBytes = 64 * 1024;  // rows staged in shared memory

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

// Two float32 values -> two E4M3 codes (first value in the low byte).
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void unit8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}
__device__ __forceinline__ void unit8(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Row of K elements (K % 16 == 0, rows 16-byte aligned) staged in shared
// memory; eight elements per thread step.
template <typename T>
__global__ void __launch_bounds__(kQThreads) rowquant_kernel(const T* __restrict__ x, int64_t K,
                                                             uint8_t* __restrict__ q,
                                                             float* __restrict__ scale) {
  extern __shared__ __align__(16) unsigned char qrow[];
  __shared__ float red[kQThreads / 32];
  const int64_t row = blockIdx.x;
  const unsigned char* src = reinterpret_cast<const unsigned char*>(x + row * K);
  const int nunits = static_cast<int>(K * int64_t(sizeof(T)) / 16);
  for (int u = threadIdx.x; u < nunits; u += kQThreads) cp_async16(qrow + 16 * u, src + 16 * u);
  cp_async_wait_all();
  __syncthreads();
  const T* xs = reinterpret_cast<const T*>(qrow);
  // reduction 1: the row's absolute maximum
  float amax = 0.f;
  for (int64_t c = int64_t(threadIdx.x) * 8; c < K; c += int64_t(kQThreads) * 8) {
    float v[8];
    unit8(xs + c, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  // the codes of x * (448 / amax), rounded in float32
  const bool zero = !(amax > 0.f);
  const float inv = zero ? 0.f : 448.f / amax;
  if (threadIdx.x == 0) scale[row] = zero ? 1.f : amax / 448.f;
  uint8_t* qr = q + row * K;
  for (int64_t c = int64_t(threadIdx.x) * 8; c < K; c += int64_t(kQThreads) * 8) {
    float v[8];
    unit8(xs + c, v);
    uint2 out;
    out.x = uint32_t(e4m3x2(v[0] * inv, v[1] * inv)) |
            (uint32_t(e4m3x2(v[2] * inv, v[3] * inv)) << 16);
    out.y = uint32_t(e4m3x2(v[4] * inv, v[5] * inv)) |
            (uint32_t(e4m3x2(v[6] * inv, v[7] * inv)) << 16);
    *reinterpret_cast<uint2*>(qr + c) = out;
  }
}

// ------------------------------------------------------------ GEMM

constexpr int kGM = 128;          // rows of A per tile
constexpr int kGN = 256;          // rows of W (columns of C) per tile
constexpr int kGK = 128;          // K bytes (codes) per stage: one 128-byte swizzle row
constexpr int kGStages = 4;
constexpr int kGThreads = 192;    // warp 0 producer, warp 1 MMA + TMEM, warps 2-5 epilogue
constexpr int kGGroup = 16;       // row tiles per group of the tile order
constexpr int kABytes = kGM * kGK;
constexpr int kBBytes = kGN * kGK;
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kGStages * kABytes;
constexpr int kOffBar = kOffB + kGStages * kBBytes;
constexpr int kGSmem = kOffBar + 256 + 1024;  // + alignment slack

struct GBars {
  uint64_t full[kGStages];
  uint64_t empty[kGStages];
  uint64_t acc_full[2];   // accumulator buffer b holds a finished tile
  uint64_t acc_empty[2];  // the epilogue has read buffer b (one arrival per epilogue warp)
  uint64_t mma_idle;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(GBars) <= 256, "GEMM barriers exceed their block");

// kind::f8f6f4 instruction descriptor: D f32, A = B = E4M3 (format 0), both
// K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2-D TMA load with an L2 cache policy (the operands are re-read by the
// CTAs working on neighbouring tiles).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(pol)
      : "memory");
}

// Tile t of the persistent walk -> (m0, n0): groups of kGGroup row tiles,
// column tiles outermost within a group, so the tiles in flight at once
// share a few row and column tiles in L2.
__device__ __forceinline__ void tile_coords(int t, int mt, int nt, int& m0, int& n0) {
  const int per_group = kGGroup * nt;
  const int g = t / per_group, r = t % per_group;
  const int rows = min(kGGroup, mt - g * kGGroup);
  m0 = (g * kGGroup + r % rows) * kGM;
  n0 = (r / rows) * kGN;
}

// Persistent: CTA c takes tiles c, c + gridDim.x, ... The K-slice ring runs
// on across tiles; accumulator buffer (j mod 2) of the CTA's j-th tile is
// reused once the epilogue has read it, so a tile's epilogue overlaps the
// next tile's MMAs.
__global__ void __launch_bounds__(kGThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_w, const float* __restrict__ sa,
                    const float* __restrict__ sw, __nv_bfloat16* __restrict__ C, int M, int N,
                    int K, int* status) {
  extern __shared__ unsigned char gsmem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(gsmem_raw) + 1023) & ~uintptr_t(1023));
  GBars& bar = *reinterpret_cast<GBars*>(smem + kOffBar);
  const uint32_t s_base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = M / kGM, nt = N / kGN;
  const int ntiles = mt * nt;
  const int nk = K / kGK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(&bar.full[s], 1);
      mbar_init(&bar.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar.acc_full[b], 1);
      mbar_init(&bar.acc_empty[b], 4);
    }
    mbar_init(&bar.mma_idle, 1);
    bar.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bar.tmem_base, 2 * kGN);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bar.tmem_base;
  volatile int* abort_flag = &bar.abort_flag;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tensormap(&tm_a);
      prefetch_tensormap(&tm_w);
      const uint64_t keep = policy_evict_last();
      bool ok = true;
      int seq = 0;  // K slices issued (all tiles)
      for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
        int m0, n0;
        tile_coords(t, mt, nt, m0, n0);
        for (int kt = 0; ok && kt < nk; ++kt, ++seq) {
          const int s = seq % kGStages;
          if (seq >= kGStages)
            ok = mbar_wait(&bar.empty[s], ((seq / kGStages) - 1) & 1, status,
                           dev_code(kDevTimeout, kKerFp8, 1), abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&bar.full[s], kABytes + kBBytes);
          tma_load_2d(smem + kOffA + s * kABytes, &tm_a, &bar.full[s], kt * kGK, m0, keep);
          tma_load_2d(smem + kOffB + s * kBBytes, &tm_w, &bar.full[s], kt * kGK, n0, keep);
        }
      }
      // never leave with copies in flight: the last load into each stage
      for (int j = max(0, seq - kGStages); j < seq; ++j)
        mbar_wait(&bar.full[j % kGStages], (j / kGStages) & 1, status,
                  dev_code(kDevTimeout, kKerFp8, 2), nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(kGM, kGN);
      bool ok = true;
      bool issued = false;
      int seq = 0;
      int j = 0;  // this CTA's tiles so far
      for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x, ++j) {
        const int b = j & 1;
        const uint32_t acc = tmem + b * kGN;
        if (j >= 2)  // the epilogue has read this buffer's previous tile
          ok = mbar_wait(&bar.acc_empty[b], ((j >> 1) - 1) & 1, status,
                         dev_code(kDevTimeout, kKerFp8, 6), abort_flag);
        if (!ok) break;
        tc_fence_after_sync();
        for (int kt = 0; ok && kt < nk; ++kt, ++seq) {
          const int s = seq % kGStages;
          ok = mbar_wait(&bar.full[s], (seq / kGStages) & 1, status,
                         dev_code(kDevTimeout, kKerFp8, 3), abort_flag);
          if (!ok) break;
          tc_fence_after_sync();
          const uint64_t a_desc = sdesc_sw128(s_base + kOffA + s * kABytes, 16, 1024);
          const uint64_t b_desc = sdesc_sw128(s_base + kOffB + s * kBBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kGK / 32; ++kk)  // 32 codes = 32 bytes per instruction
            mma_e4m3(acc, a_desc + uint64_t(kk * 2), b_desc + uint64_t(kk * 2), idesc,
                     (kt > 0 || kk > 0) ? 1u : 0u);
          issued = true;
          mma_commit(&bar.empty[s]);
        }
        if (ok) mma_commit(&bar.acc_full[b]);
      }
      // never leave with MMAs in flight (their operands live in this CTA)
      if (issued) {
        mma_commit(&bar.mma_idle);
        mbar_wait(&bar.mma_idle, 0, status, dev_code(kDevTimeout, kKerFp8, 4), nullptr);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lanes 32*quad .. +31
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint64_t drop = policy_evict_first();
    int j = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++j) {
      const int b = j & 1;
      if (!mbar_wait_warp(&bar.acc_full[b], (j >> 1) & 1, status,
                          dev_code(kDevTimeout, kKerFp8, 5), abort_flag))
        break;
      tc_fence_after_sync();
      int m0, n0;
      tile_coords(t, mt, nt, m0, n0);
      const int row = m0 + quad * 32 + lane;
      const float sr = sa[row];
      __nv_bfloat16* crow = C + int64_t(row) * N + n0;
#pragma unroll 1
      for (int c0 = 0; c0 < kGN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32_wait(tmem + b * kGN + lane_off + c0, r);
        uint32_t packed[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          packed[e >> 1] = pack_bf16x2(__uint_as_float(r[e]) * sr * sw[n0 + c0 + e],
                                       __uint_as_float(r[e + 1]) * sr * sw[n0 + c0 + e + 1]);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          st_global_policy(reinterpret_cast<uint4*>(crow + c0) + q4,
                           make_uint4(packed[4 * q4], packed[4 * q4 + 1], packed[4 * q4 + 2],
                                      packed[4 * q4 + 3]),
                           drop);
      }
      // this warp's reads of the buffer are complete (tcgen05.wait::ld above)
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.acc_empty[b]);
    }
  }

  // ---------------------------------------------------------- teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 2 * kGN);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// [rows, K] bytes, 128-byte swizzle, boxes of 128 bytes x box_rows rows.
bool make_map_u8(CUtensorMap* m, const void* base, int K, int rows, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kGK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_rowquant_e4m3(const void* x, int64_t rows, int64_t K, uint8_t* q, float* scale,
                                 rf_dtype dt, cudaStream_t s) {
  const int64_t row_bytes = K * (dt == RF_F32 ? 4 : 2);
  if (row_bytes > kQRowBytes) return cudaErrorInvalidValue;
  const int smem = static_cast<int>(row_bytes);
  if (dt == RF_F32) {
    if (smem > 46 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(rowquant_kernel<float>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kQRowBytes);
      if (e != cudaSuccess) return e;
    }
    rowquant_kernel<float><<<static_cast<unsigned>(rows), kQThreads, smem, s>>>(
        static_cast<const float*>(x), K, q, scale);
  } else {
    if (smem > 46 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(rowquant_kernel<__nv_bfloat16>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kQRowBytes);
      if (e != cudaSuccess) return e;
    }
    rowquant_kernel<__nv_bfloat16><<<static_cast<unsigned>(rows), kQThreads, smem, s>>>(
        static_cast<const __nv_bfloat16*>(x), K, q, scale);
  }
  return cudaGetLastError();
}

cudaError_t launch_fp8_gemm(const uint8_t* a, const float* sa, const uint8_t* w, const float* sw,
                            void* c, int M, int N, int K, cudaStream_t s, int* status,
                            const char** why) {
  CUtensorMap ma, mw;
  if (!make_map_u8(&ma, a, K, M, kGM) || !make_map_u8(&mw, w, K, N, kGN)) {
    *why = "tensor map encoding failed";
    return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(fp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kGSmem);
  if (e != cudaSuccess) {
    *why = "shared memory attribute";
    return e;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    *why = "device attributes";
    return cudaErrorInvalidValue;
  }
  const int64_t tiles = int64_t(M / kGM) * (N / kGN);
  const int64_t grid = tiles < sms ? tiles : sms;  // persistent: one CTA per SM
  fp8_gemm_kernel<<<static_cast<unsigned>(grid), kGThreads, kGSmem, s>>>(
      ma, mw, sa, sw, static_cast<__nv_bfloat16*>(c), M, N, K, status);
  return cudaGetLastError();
}

}  // namespace rf
