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
//  * longer rows, one cluster of 2..8 CTAs per row (multi-segment): each
//    thread folds its elements into a running (m, l) (the incremental form,
//    O(1) state), the CTAs exchange their (m_c, l_c) through distributed
//    shared memory and combine them as L = sum_c l_c exp(m_c - M), then y is
//    written. When the row splits into 16-byte-aligned slices of at most
//    128 KB, the slice stays on chip (softmax_rows_ring: persistent clusters
//    over the rows, a ring of 16 KB pieces filled by a producer warp, the
//    next row's loads overlapping this row's exchange and stores): 1 read +
//    1 write of HBM per element. Otherwise (unaligned rows, slices over
//    128 KB) a second pass re-reads the slice, the first pass loading with an
//    L2 evict-last policy so that the second mostly finds it in L2.
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
  constexpr int U = 4;               // vectors in flight per thread
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
    for (int64_t b = threadIdx.x; b < nv; b += U * kThreads) {
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

// ---------------------------------------------------------------------------
// Long rows with the slice kept on chip: persistent clusters and a ring.
//
// One cluster of nc CTAs per row (multi-segment strategy), each CTA holding
// its slice of cols / nc elements (at most kRingSliceBytes) in shared memory
// from the moment it lands until y is written: 1 read + 1 write of HBM per
// element. A grid of co-resident clusters walks the rows (cluster c takes
// rows c, c + nclusters, ...), and the slice streams through a ring of
// kRingSlots pieces of kPiece bytes, filled by one producer warp with bulk
// copies: as soon as the normalisation of row r has read a piece, its slot
// takes the next row's data, so the loads of row r + 1 overlap the stores of
// row r and the cluster exchange, and HBM never waits on one CTA's phases.
//
// Per row, the 16 consumer warps
//  (A) fold each piece into a per-thread running (m, l) as it lands (the
//      incremental form, O(1) state), then combine the threads (named
//      barrier 1, consumers only);
//  (B) push the CTA's (m_c, l_c) into every peer's shared memory and meet at
//      one cluster barrier (all threads of the cluster, the producer warp
//      included); every CTA then combines L = sum_c l_c exp(m_c - M);
//  (C) read their own elements of each piece again from shared memory,
//      write y = exp(x - M) / L from registers, and release the slot.
// Each thread reads in (C) exactly the elements it read in (A), so the
// phases need no CTA barrier between them.
//
// Ordering of the exchange: CTA a writes peer b's pairs[r & 1] for row r
// only after a's wait on the barrier of row r - 1, which b passes only after
// reading its pairs[(r - 2) & 1]; so a slot is never overwritten before it is
// read. No CTA leaves before the barrier of its last row, after which no peer
// writes its shared memory. After a timed-out wait a CTA stops its work
// (abort flag) but keeps meeting every cluster barrier, so its peers finish.
constexpr int kRingSlots = 13;                        // 13 x 16 KB = 208 KB
constexpr int kRingSliceBytes = 128 * 1024;           // at most 8 pieces per slice
constexpr int kRingConsumers = 512;                   // 16 warps
constexpr int kRingThreads = kRingConsumers + 32;     // + the producer warp

struct RingSmem {
  unsigned char data[kRingSlots][kPiece];
  uint64_t full[kRingSlots];
  uint64_t empty[kRingSlots];
  float2 pairs[2][kMaxCluster];
  float red[2][32];
  int abort_flag;
};

// Consumer-only (named barrier 1) reductions over the 16 consumer warps.
__device__ __forceinline__ float consumers_max(float x, float* red) {
  x = warp_max(x);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  asm volatile("bar.sync 1, %0;" ::"n"(kRingConsumers) : "memory");
  return warp_max((threadIdx.x & 31) < kRingConsumers / 32 ? red[threadIdx.x & 31] : kNegInf);
}
__device__ __forceinline__ float consumers_sum(float x, float* red) {
  x = warp_sum(x);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  asm volatile("bar.sync 1, %0;" ::"n"(kRingConsumers) : "memory");
  return warp_sum((threadIdx.x & 31) < kRingConsumers / 32 ? red[threadIdx.x & 31] : 0.f);
}

template <typename T>
__global__ void __launch_bounds__(kRingThreads, 1) softmax_rows_ring(const T* x, T* y,
                                                                    int64_t rows, int64_t cols,
                                                                    int* status) {
  constexpr int V = 16 / sizeof(T);  // elements per 16-byte vector
  extern __shared__ __align__(128) unsigned char ring_raw[];
  RingSmem& sm = *reinterpret_cast<RingSmem*>(ring_raw);
  cg::cluster_group cl = cg::this_cluster();
  const int nc = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int64_t ncl = gridDim.x / nc, cid = blockIdx.x / nc;
  const int64_t seg = cols / nc;                                  // elements of the slice
  const uint32_t slice_bytes = static_cast<uint32_t>(seg * sizeof(T));
  const int npieces = static_cast<int>((slice_bytes + kPiece - 1) / kPiece);
  const int64_t my_rows = cid < rows ? (rows - 1 - cid) / ncl + 1 : 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRingSlots; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kRingConsumers / 32);
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  cluster_arrive_relaxed();  // the start-up phase: every peer is running

  if (warp == kRingConsumers / 32) {
    // ---------------- producer warp: bulk copies into the ring
    const uint64_t pol = policy_evict_first();
    int64_t g = 0;  // pieces issued so far
    for (int64_t it = 0; it < my_rows; ++it) {
      // Row it's pieces may need slots that row it - 1's step (C) frees;
      // the consumers reach (C) once this warp has arrived on the barrier
      // of row it - 1, which it did at the end of the previous iteration.
      if (lane == 0 && !sm.abort_flag) {
        const T* src = x + (cid + it * ncl) * cols + rank * seg;
        for (int pc = 0; pc < npieces; ++pc, ++g) {
          const int slot = static_cast<int>(g % kRingSlots);
          const int64_t use = g / kRingSlots;
          if (use > 0 && !mbar_wait(&sm.empty[slot], static_cast<uint32_t>((use - 1) & 1),
                                    status, dev_code(kDevTimeout, kKerSoftmax, 5),
                                    &sm.abort_flag))
            break;
          const uint32_t off = static_cast<uint32_t>(pc) * kPiece;
          const uint32_t bytes = min(static_cast<uint32_t>(kPiece), slice_bytes - off);
          mbar_arrive_expect_tx(&sm.full[slot], bytes);
          bulk_load(sm.data[slot], reinterpret_cast<const unsigned char*>(src) + off, bytes,
                    &sm.full[slot], pol);
        }
      }
      __syncwarp();
      cluster_wait_acquire();     // the barrier before row it's exchange (start-up or row it - 1)
      cluster_arrive_relaxed();   // row it's barrier: the producer publishes nothing
    }
    cluster_wait_acquire();       // the last barrier
    // never leave with copies in flight: the last fill of every used slot
    if (lane == 0)
      for (int64_t k = (g > kRingSlots ? g - kRingSlots : 0); k < g; ++k)
        mbar_wait(&sm.full[k % kRingSlots], static_cast<uint32_t>((k / kRingSlots) & 1), status,
                  dev_code(kDevTimeout, kKerSoftmax, 6), nullptr);
    return;
  }

  // ---------------- consumer warps
  const uint64_t drop = policy_evict_first();
  int64_t g0 = 0;  // the row's first piece in the ring sequence
  for (int64_t it = 0; it < my_rows; ++it, g0 += npieces) {
    const int64_t row = cid + it * ncl;
    // (A) local (m, l), piece by piece as they land
    float m = kNegInf, l = 0.f;
    if (!sm.abort_flag) {
      for (int pc = 0; pc < npieces; ++pc) {
        const int64_t g = g0 + pc;
        const int slot = static_cast<int>(g % kRingSlots);
        if (!mbar_wait_warp(&sm.full[slot], static_cast<uint32_t>((g / kRingSlots) & 1), status,
                            dev_code(kDevTimeout, kKerSoftmax, 7), &sm.abort_flag))
          break;
        const int nv = static_cast<int>(min(static_cast<uint32_t>(kPiece),
                                            slice_bytes - static_cast<uint32_t>(pc) * kPiece) /
                                        16);
        const uint4* pv = reinterpret_cast<const uint4*>(sm.data[slot]);
#pragma unroll
        for (int u = 0; u < kPiece / 16 / kRingConsumers; ++u) {
          const int e = threadIdx.x + u * kRingConsumers;
          if (e < nv) {
            float v[V];
            unpack16(pv[e], v);
            fold(v, m, l);
          }
        }
      }
    }
    const float bm = consumers_max(m, sm.red[0]);
    const float lt = consumers_sum(m == kNegInf ? 0.f : l * ex2_approx((m - bm) * kLog2e),
                                   sm.red[1]);
    // (B) exchange (m_c, l_c) with the peers. Before the first row: wait
    // for the start-up phase (every peer is running). Before row it >= 1 the
    // wait on row it - 1's barrier (below, last row) already showed that
    // every peer has read pairs[(it - 2) & 1].
    if (it == 0) cluster_wait_acquire();
    float2* pairs = sm.pairs[it & 1];
    if (threadIdx.x < nc) *cl.map_shared_rank(pairs + rank, threadIdx.x) = make_float2(bm, lt);
    cluster_arrive_release();
    cluster_wait_acquire();  // this row's pairs have all landed
    float M = kNegInf;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, pairs[c].x);
    float L = 0.f;
    if (M != kNegInf)
      for (int c = 0; c < nc; ++c)
        if (pairs[c].x != kNegInf) L += pairs[c].y * ex2_approx((pairs[c].x - M) * kLog2e);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const float Ms = (M == kNegInf) ? 0.f : M;
    // (C) y from the slice on chip; release each piece's slot
    uint4* yv = reinterpret_cast<uint4*>(y + row * cols + rank * seg);
    for (int pc = 0; pc < npieces; ++pc) {
      const int64_t g = g0 + pc;
      const int slot = static_cast<int>(g % kRingSlots);
      if (!sm.abort_flag) {
        const int nv = static_cast<int>(min(static_cast<uint32_t>(kPiece),
                                            slice_bytes - static_cast<uint32_t>(pc) * kPiece) /
                                        16);
        const uint4* pv = reinterpret_cast<const uint4*>(sm.data[slot]);
#pragma unroll
        for (int u = 0; u < kPiece / 16 / kRingConsumers; ++u) {
          const int e = threadIdx.x + u * kRingConsumers;
          if (e < nv) {
            float v[V];
            unpack16(pv[e], v);
            uint4 o;
            if constexpr (V == 4) {
              o = make_uint4(__float_as_uint(exp_shift(v[0], Ms) * inv),
                             __float_as_uint(exp_shift(v[1], Ms) * inv),
                             __float_as_uint(exp_shift(v[2], Ms) * inv),
                             __float_as_uint(exp_shift(v[3], Ms) * inv));
            } else {
              uint32_t q[4];
#pragma unroll
              for (int j = 0; j < 4; ++j)
                q[j] = pack_bf16x2(exp_shift(v[2 * j], Ms) * inv,
                                   exp_shift(v[2 * j + 1], Ms) * inv);
              o = make_uint4(q[0], q[1], q[2], q[3]);
            }
            st_global_policy(yv + int64_t(pc) * (kPiece / 16) + e, o, drop);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);
    }
  }
  if (my_rows == 0) cluster_wait_acquire();  // the start-up phase
  // after the last row's barrier no peer writes this CTA's memory any more
}

// Persistent ring launch: as many clusters as can be resident at once (at
// most one per row). cudaErrorNotSupported: no cluster of this shape fits, the
// caller streams instead.
template <typename T>
cudaError_t launch_ring(const T* x, T* y, int64_t rows, int64_t cols, int nc, cudaStream_t s,
                        int* status) {
  const size_t smem = sizeof(RingSmem);
  cudaError_t e = cudaFuncSetAttribute(softmax_rows_ring<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = s;
  cfg.blockDim = dim3(kRingThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.gridDim = dim3(static_cast<unsigned>(nc));
  int active = 0;
  e = cudaOccupancyMaxActiveClusters(&active, softmax_rows_ring<T>, &cfg);
  if (e != cudaSuccess) return e;
  if (active < 1) return cudaErrorNotSupported;
  const int64_t ncl = min64(rows, active);
  cfg.gridDim = dim3(static_cast<unsigned>(ncl * nc));
  return cudaLaunchKernelEx(&cfg, softmax_rows_ring<T>, x, y, rows, cols, status);
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
  // one cluster per row, about one slice per CTA up to kMaxCluster CTAs
  const int nc = static_cast<int>(min64(kMaxCluster, max64(2, (cols + cap - 1) / cap)));
  // slices that fit the ring and split the row exactly: keep them on chip
  if (aligned && cols % (int64_t(nc) * vec) == 0 &&
      (cols / nc) * int64_t(sizeof(T)) <= kRingSliceBytes) {
    cudaError_t e = launch_ring<T>(x, y, rows, cols, nc, s, status);
    if (e != cudaErrorNotSupported) return e;
  }
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
