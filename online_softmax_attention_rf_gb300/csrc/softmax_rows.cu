// softmax_rows.cu -- row softmax, the pure two-reduction cascade.
//
// RedFuser (An Automatic Operator Fusion Framework for Cascaded Reductions
// on AI Accelerators), technical summary section 1: softmax is a cascade of
// reductions (maximum, then sum of exponentials) where each waits for the
// root of the one before; section 2: fusing the chain means the input is
// loaded once; section 3: single-segment (one CTA) and multi-segment
// (partition, then merge the partial results) strategies.
//
// Shapes of the kernel:
//  * on chip, one CTA per row (row <= 64 KB): the row is copied into
//    shared memory once (cp.async.bulk, 16 KB pieces, each with its own
//    mbarrier so the maximum starts on the first piece), then
//    m = max, p = exp(x - m) written back in place with l = sum p, and
//    y = p / l stored -- 1 read + 1 write of HBM per element;
//  * longer rows, one cluster of 2..8 CTAs per row (multi-segment), about
//    128 KB of the row per CTA: each thread folds its elements into a running
//    (m, l) (the incremental form, O(1) state), the CTAs exchange their
//    (m_c, l_c) through distributed shared memory and combine them as
//    L = sum_c l_c exp(m_c - M), and a second pass over the slice, back to
//    front, writes y. The first pass loads with an L2 evict-last policy and
//    the second with evict-first; with three CTAs per SM the slices resident
//    at once fit in the 126 MB L2, so the second read comes from L2 and HBM
//    sees 1 read + 1 write per element (0.99 x on 1 MiB rows). Keeping the slice in shared memory
//    instead measured slower on this GPU: a 128 KB slice leaves one CTA per
//    SM, only 120 SMs can hold clusters of 8 such CTAs, and with the slice
//    resident too little of the next row can be in flight (a persistent
//    cluster ring with a producer warp reached 4.3 TB/s on 1 MiB rows,
//    against 5.6 TB/s here).
// x and y may alias: every element is read before the thread that writes it
// writes it.
#include <cooperative_groups.h>

#include "rf_device.cuh"

namespace cg = cooperative_groups;

namespace rf {
namespace {

constexpr int kThreads = 512;
// Largest slice one CTA holds on chip: 64 KB, so that three CTAs share an SM
// and one CTA's loads overlap another's stores. Long rows give each CTA of a
// cluster about as much.
constexpr int kSliceBytes = 64 * 1024;
constexpr int kPiece = 16384;            // bytes per bulk copy / mbarrier
constexpr int kMaxPieces = kSliceBytes / kPiece;
// CTAs per row for long rows: the portable cluster size. Eight CTAs with
// 128 KB of a 1 MiB row each measured 2.6 % faster than sixteen with 64 KB
// (fewer CTAs wait at each exchange), and four were 17 % slower.
constexpr int kMaxCluster = 8;

template <typename T>
__device__ __forceinline__ float to_f(T v) {
  return static_cast<float>(v);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Block-wide reductions; `red` holds one float per warp.
__device__ __forceinline__ float block_max(float x, float* red) {
  x = warp_max(x);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = x;
  __syncthreads();
  const float r = (threadIdx.x & 31) < nw ? red[threadIdx.x & 31] : kNegInf;
  return warp_max(r);
}

__device__ __forceinline__ float block_sum(float x, float* red) {
  x = warp_sum(x);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = x;
  __syncthreads();
  const float r = (threadIdx.x & 31) < nw ? red[threadIdx.x & 31] : 0.f;
  return warp_sum(r);
}

// exp(x - m) for a finite shift m; exp(-inf - m) = 0.
__device__ __forceinline__ float exp_shift(float x, float m) { return ex2_approx((x - m) * kLog2e); }

// Cluster barrier halves (barrier.cluster): arrive is non-blocking, wait
// returns once every CTA of the cluster has arrived.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Combine this CTA's (m, l) with the other CTAs of its cluster through
// distributed shared memory; every thread gets the row's (M, L). Each CTA
// pushes its pair into slot [rank] of every peer's `pairs` (one remote store
// per peer, issued by threads 0..nc-1 at once), then one cluster barrier
// makes the stores visible and every thread reads its own CTA's array. The
// caller has arrived (relaxed) on the cluster barrier at kernel start, so the
// first wait here only confirms that every peer is running before its shared
// memory is written; no CTA reads a peer's memory after the second barrier,
// so CTAs may leave as soon as they are done.
__device__ __forceinline__ void cluster_combine(float m, float l, float2* pairs, float& M,
                                                float& L) {
  cg::cluster_group cl = cg::this_cluster();
  const unsigned nc = cl.num_blocks();
  cluster_wait_acquire();  // phase 0: every peer has started
  if (threadIdx.x < nc) *cl.map_shared_rank(pairs + cl.block_rank(), threadIdx.x) = make_float2(m, l);
  cluster_arrive_release();
  cluster_wait_acquire();  // phase 1: every pair has landed here
  M = kNegInf;
  for (unsigned c = 0; c < nc; ++c) M = fmaxf(M, pairs[c].x);
  L = 0.f;
  if (M != kNegInf)
    for (unsigned c = 0; c < nc; ++c) {
      const float2 q = pairs[c];
      if (q.x != kNegInf) L += q.y * ex2_approx((q.x - M) * kLog2e);
    }
}

// Shared-memory-resident row. Row blockIdx is staged in dynamic shared
// memory as T; float input keeps the probabilities in place, bf16 input keeps
// x and recomputes the exp.
// fault != 0 (test aid): CTA 0 arms its first piece's barrier but never
// issues that copy, so its waits run out and it unwinds.
template <typename T>
__global__ void __launch_bounds__(kThreads) softmax_rows_onchip(const T* x, T* y, int64_t cols,
                                                                int bulk, int* status, int fault) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  T* xs = reinterpret_cast<T*>(smem_raw);
  __shared__ float red[32];
  __shared__ uint64_t bars[kMaxPieces];
  __shared__ int abort_flag;
  const int64_t row = blockIdx.x;
  const int64_t n = cols;
  const T* xr = x + row * cols;
  T* yr = y + row * cols;
  constexpr int kPerPiece = kPiece / sizeof(T);
  const int npieces = n > 0 ? static_cast<int>((n + kPerPiece - 1) / kPerPiece) : 0;

  // ---- stage the slice
  if (threadIdx.x == 0) abort_flag = 0;
  if (bulk) {
    if (threadIdx.x == 0) {
      for (int i = 0; i < npieces; ++i) mbar_init(&bars[i], 1);
      fence_barrier_init();
      const uint64_t pol = policy_evict_first();
      for (int i = 0; i < npieces; ++i) {
        const int64_t e0 = int64_t(i) * kPerPiece;
        const uint32_t bytes = static_cast<uint32_t>(min64(kPerPiece, n - e0) * sizeof(T));
        mbar_arrive_expect_tx(&bars[i], bytes);
        if (!(fault && blockIdx.x == 0 && i == 0)) bulk_load(xs + e0, xr + e0, bytes, &bars[i], pol);
      }
    }
  } else {
    for (int64_t e = threadIdx.x; e < n; e += kThreads) xs[e] = xr[e];
  }
  __syncthreads();
  // ---- reduction 1: maximum (piece by piece as the copies land)
  float m = kNegInf;
  bool ok = true;
  for (int i = 0; i < npieces; ++i) {
    if (bulk && !(ok = mbar_wait_warp(&bars[i], 0, status, dev_code(kDevTimeout, kKerSoftmax, 1),
                                      &abort_flag)))
      break;
    const int64_t e1 = min64(n, int64_t(i + 1) * kPerPiece);
    for (int64_t e = int64_t(i) * kPerPiece + threadIdx.x; e < e1; e += kThreads)
      m = fmaxf(m, to_f(xs[e]));
  }
  m = block_max(m, red);
  const float ms = (m == kNegInf) ? 0.f : m;
  // ---- reduction 2: sum of exp(x - m); float input keeps p in place
  float l = 0.f;
  if (ok) {
    if constexpr (sizeof(T) == 4) {
      for (int64_t e = threadIdx.x; e < n; e += kThreads) {
        const float p = exp_shift(xs[e], ms);
        xs[e] = p;
        l += p;
      }
    } else {
      for (int64_t e = threadIdx.x; e < n; e += kThreads) l += exp_shift(to_f(xs[e]), ms);
    }
  }
  l = block_sum(l, red);
  const float scale = l > 0.f ? 1.f / l : 0.f;
  if (abort_flag) {  // uniform: set before the last block reduction
    // never leave with copies in flight
    if (bulk && threadIdx.x == 0)
      for (int i = 0; i < npieces; ++i)
        if (!(fault && blockIdx.x == 0 && i == 0))  // the copy that was never issued
          mbar_wait(&bars[i], 0, status, dev_code(kDevTimeout, kKerSoftmax, 2), nullptr);
    return;
  }
  // ---- y = p * scale, 16-byte stores where the slice allows
  if constexpr (sizeof(T) == 4) {
    if (bulk) {
      const float4* ps = reinterpret_cast<const float4*>(xs);
      float4* yv = reinterpret_cast<float4*>(yr);
      for (int64_t e = threadIdx.x; e < n / 4; e += kThreads) {
        float4 v = ps[e];
        v.x *= scale; v.y *= scale; v.z *= scale; v.w *= scale;
        yv[e] = v;
      }
      for (int64_t e = (n / 4) * 4 + threadIdx.x; e < n; e += kThreads) yr[e] = xs[e] * scale;
    } else {
      for (int64_t e = threadIdx.x; e < n; e += kThreads) yr[e] = xs[e] * scale;
    }
  } else {
    if (bulk) {
      const uint4* xv = reinterpret_cast<const uint4*>(xs);
      uint4* yv = reinterpret_cast<uint4*>(yr);
      for (int64_t e = threadIdx.x; e < n / 8; e += kThreads) {
        const uint4 w = xv[e];
        const uint32_t in[4] = {w.x, w.y, w.z, w.w};
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = exp_shift(__uint_as_float(in[j] << 16), ms) * scale;
          const float hi = exp_shift(__uint_as_float(in[j] & 0xffff0000u), ms) * scale;
          out[j] = pack_bf16x2(lo, hi);
        }
        yv[e] = make_uint4(out[0], out[1], out[2], out[3]);
      }
      for (int64_t e = (n / 8) * 8 + threadIdx.x; e < n; e += kThreads)
        yr[e] = __float2bfloat16_rn(exp_shift(to_f(xs[e]), ms) * scale);
    } else {
      for (int64_t e = threadIdx.x; e < n; e += kThreads)
        yr[e] = __float2bfloat16_rn(exp_shift(to_f(xs[e]), ms) * scale);
    }
  }
}

// Unpack one 16-byte vector into floats.
__device__ __forceinline__ void unpack16(const uint4& w, float (&v)[4]) {
  v[0] = __uint_as_float(w.x); v[1] = __uint_as_float(w.y);
  v[2] = __uint_as_float(w.z); v[3] = __uint_as_float(w.w);
}
__device__ __forceinline__ void unpack16(const uint4& w, float (&v)[8]) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(in[j] << 16);
    v[2 * j + 1] = __uint_as_float(in[j] & 0xffff0000u);
  }
}

// Fold k values into a running (m, l): one rescale per group, when the
// group's maximum exceeds m.
template <int K>
__device__ __forceinline__ void fold(const float (&v)[K], float& m, float& l) {
  float vm = v[0];
#pragma unroll
  for (int j = 1; j < K; ++j) vm = fmaxf(vm, v[j]);
  if (vm > m) {
    l = (m == kNegInf) ? 0.f : l * ex2_approx((m - vm) * kLog2e);
    m = vm;
  }
  if (m != kNegInf) {
#pragma unroll
    for (int j = 0; j < K; ++j) l += exp_shift(v[j], m);
  }
}

// Long rows, one cluster per row, slice [seg0, seg1) per CTA. With `vec16`
// the slice is read as 16-byte vectors, four per thread in flight, pass 1
// with an L2 evict-last policy so that pass 2 (evict-first, like the stores
// of y) finds it in L2.
template <typename T>
__global__ void __launch_bounds__(kThreads) softmax_rows_stream(const T* x, T* y, int64_t cols,
                                                                int64_t seg_len, int vec16) {
  constexpr int V = 16 / sizeof(T);  // elements per vector
  // vectors in flight per thread: as many as fit in 40 registers (6 float,
  // 5 bf16), which leaves three 512-thread CTAs per SM. On 1 MiB float rows
  // this measured 6140 GB/s against 5690 with four in flight (32 registers,
  // four CTAs per SM: more slices resident, more of them re-read from DRAM)
  // and 5235 with seven (two CTAs per SM).
  constexpr int U = sizeof(T) == 4 ? 6 : 5;
  const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
  __shared__ float red[32];
  __shared__ float2 pairs[kMaxCluster];
  const int nc = static_cast<int>(cg::this_cluster().num_blocks());
  cluster_arrive_relaxed();  // phase 0 of cluster_combine
  const int64_t row = blockIdx.x / nc;
  const int64_t c = blockIdx.x % nc;
  const int64_t seg0 = min64(cols, c * seg_len);
  const int64_t seg1 = min64(cols, seg0 + seg_len);
  const T* xr = x + row * cols;
  T* yr = y + row * cols;
  // pass 1: per-thread running (m, l), rescaled whenever m grows
  float m = kNegInf, l = 0.f;
  if (vec16) {  // seg0 and seg1 are multiples of V
    const uint4* xv = reinterpret_cast<const uint4*>(xr + seg0);
    const int64_t nv = (seg1 - seg0) / V;
    for (int64_t b = threadIdx.x; b < nv; b += U * kThreads) {
      uint4 w[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (b + u * kThreads < nv) w[u] = ld_global_policy(xv + b + u * kThreads, keep);
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (b + u * kThreads < nv) {
          float v[V];
          unpack16(w[u], v);
          fold(v, m, l);
        }
    }
  } else {
    for (int64_t e = seg0 + threadIdx.x; e < seg1; e += kThreads) {
      const float v[1] = {to_f(xr[e])};
      fold(v, m, l);
    }
  }
  // merge the threads' states: block max, then rescaled block sum
  const float bm = block_max(m, red);
  float lt = (m == kNegInf) ? 0.f : l * ex2_approx((m - bm) * kLog2e);
  lt = block_sum(lt, red);
  float M, L;
  cluster_combine(bm, lt, pairs, M, L);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const float Ms = (M == kNegInf) ? 0.f : M;
  // pass 2: write y
  if (vec16) {
    const uint4* xv = reinterpret_cast<const uint4*>(xr + seg0);
    uint4* yv = reinterpret_cast<uint4*>(yr + seg0);
    const int64_t nv = (seg1 - seg0) / V;
    // back to front: the last vectors pass 1 loaded are the likeliest still in L2
    const int64_t nblk = (nv + U * kThreads - 1) / (U * kThreads);
    for (int64_t bb = nblk - 1; bb >= 0; --bb) {
      const int64_t b = bb * U * kThreads + threadIdx.x;
      uint4 w[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (b + u * kThreads < nv) w[u] = ld_global_policy(xv + b + u * kThreads, drop);
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (b + u * kThreads < nv) {
          float v[V];
          unpack16(w[u], v);
          uint4 o;
          if constexpr (V == 4) {
            o = make_uint4(__float_as_uint(exp_shift(v[0], Ms) * inv),
                           __float_as_uint(exp_shift(v[1], Ms) * inv),
                           __float_as_uint(exp_shift(v[2], Ms) * inv),
                           __float_as_uint(exp_shift(v[3], Ms) * inv));
          } else {
            uint32_t p[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
              p[j] = pack_bf16x2(exp_shift(v[2 * j], Ms) * inv, exp_shift(v[2 * j + 1], Ms) * inv);
            o = make_uint4(p[0], p[1], p[2], p[3]);
          }
          st_global_policy(yv + b + u * kThreads, o, drop);
        }
    }
  } else {
    for (int64_t e = seg0 + threadIdx.x; e < seg1; e += kThreads)
      yr[e] = static_cast<T>(exp_shift(to_f(xr[e]), Ms) * inv);
  }
}

template <typename T>
cudaError_t launch_typed(const T* x, T* y, int64_t rows, int64_t cols, cudaStream_t s,
                         int* status, bool fault) {
  constexpr int64_t cap = kSliceBytes / sizeof(T);  // elements per CTA
  constexpr int64_t vec = 16 / sizeof(T);
  // bulk copies and vector loads need 16-byte aligned rows of whole vectors
  const bool aligned = (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(y) % 16 == 0) && cols % vec == 0;
  if (cols <= cap) {
    const size_t smem = size_t((cols * sizeof(T) + 15) / 16 * 16);
    cudaError_t e = cudaFuncSetAttribute(softmax_rows_onchip<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSliceBytes);
    if (e != cudaSuccess) return e;
    softmax_rows_onchip<T><<<static_cast<unsigned>(rows), kThreads, smem, s>>>(
        x, y, cols, aligned ? 1 : 0, status, fault ? 1 : 0);
    return cudaGetLastError();
  }
  // one cluster per row, slices of about 128 KB, at most kMaxCluster CTAs
  // (1 MiB float rows: 8 x 128 KB, which measured 2.6 % faster than
  // 16 x 64 KB; 512 KB bf16 rows: 4 x 128 KB, 12 % faster than 8 x 64 KB)
  constexpr int64_t slice = 2 * cap;
  const int nc = static_cast<int>(min64(kMaxCluster, max64(2, (cols + slice - 1) / slice)));
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = s;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  int64_t seg = (cols + nc - 1) / nc;
  seg = (seg + vec - 1) / vec * vec;
  attr[0].val.clusterDim.x = nc;
  cfg.gridDim = dim3(static_cast<unsigned>(rows * nc));
  return cudaLaunchKernelEx(&cfg, softmax_rows_stream<T>, x, y, cols, seg, aligned ? 1 : 0);
}

}  // namespace

cudaError_t launch_softmax_rows(const void* x, void* y, int64_t rows, int64_t cols, rf_dtype dt,
                                cudaStream_t s, int* status, bool skip_first_copy) {
  if (rows * kMaxCluster > 0x7fffffffLL) return cudaErrorInvalidValue;  // grid size
  if (dt == RF_F32)
    return launch_typed<float>(static_cast<const float*>(x), static_cast<float*>(y), rows, cols,
                               s, status, skip_first_copy);
  return launch_typed<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(x),
                                     static_cast<__nv_bfloat16*>(y), rows, cols, s, status,
                                     skip_first_copy);
}

}  // namespace rf
