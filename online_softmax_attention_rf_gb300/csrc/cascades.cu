// cascades.cu -- other cascaded reductions on the same algebra.
//
// RedFuser: An Automatic Operator Fusion Framework for Cascaded Reductions on
// AI Accelerators -- technical summary, section 1: besides attention, routing
// in Mixture-of-Experts models and normalisation layers are cascades of
// reductions, each needing the root of the one before; section 4: MoE routing
// is one of the evaluated workloads; the Korean page's results add variance
// (non-ML) workloads.
//
// MoE routing (one warp per token): the softmax's maximum and sum of
// exponentials, then k rounds of arg-max over the logits (top-k of the
// probabilities are the top-k logits: exp is increasing), ties going to the
// lower expert index. Lane l holds the contiguous experts [EPL l, EPL l + EPL)
// (the logits arrive as 16-byte vectors), so expert order is lane order: in a
// round, one single-instruction warp reduction (redux.sync) over
// order-preserving integer keys gives the largest key, and the lowest lane
// holding it (a ballot and find-first-set) holds the lowest expert index
// with it. Each lane keeps its best and second-best remaining experts (an
// ascending scan with strict comparisons keeps the lower slot first); the
// winner moves to its second best and rescans its slots only when it wins
// again with the second best not yet known (for random logits, well under
// one rescan per token). The token's logits are read once.
//
// Row moments (one CTA per row): each thread folds its elements into a
// (count, mean, M2) state, four or eight at a time (two passes over
// registers, then the pairwise merge of Chan, Golub and LeVeque), the states
// merge across the warp and the CTA by the same rule (multi-segment
// strategy, merge step), and var = M2 / n. With an output, a second pass
// writes (x - mean) / sqrt(var + eps). Rows of up to 64 KB are staged in
// shared memory, float rows of up to 32768 elements otherwise stay in
// registers between the two (x is read once); longer rows are read a second
// time, from L2, where the first pass left them with an evict-last policy.
//
// Moment of inertia (one CTA per point set; the Korean page's non-ML
// workload): the total mass and centre of mass, then the sum of m |r - c|^2
// about that centre, in one read of the points: mass-weighted (W, c, M2)
// states of four points (two passes over registers), merged pairwise with
// the masses as weights.
#include "rf_device.cuh"

namespace rf {
namespace {

// ------------------------------------------------------------------ MoE routing

template <typename T>
__device__ __forceinline__ float load_f(const T* p) {
  return static_cast<float>(*p);
}

// Order-preserving map of a float to an unsigned key (a larger float gives
// a larger key; -0 is taken as +0 so that the two tie, as they compare).
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// The lane's best and second-best remaining experts in the order (larger
// key first, then lower slot): an ascending scan with strict comparisons.
// Real experts have keys >= 1; key 0 / slot EPL means none.
template <int EPL>
__device__ __forceinline__ void top2(const uint32_t (&key)[EPL], uint32_t taken, uint32_t& k1,
                                     int& s1, uint32_t& k2, int& s2) {
  k1 = 0u;
  k2 = 0u;
  s1 = EPL;
  s2 = EPL;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const uint32_t k = ((taken >> i) & 1u) ? 0u : key[i];
    const bool gt1 = k > k1, gt2 = k > k2;
    k2 = gt1 ? k1 : (gt2 ? k : k2);
    s2 = gt1 ? s1 : (gt2 ? i : s2);
    k1 = gt1 ? k : k1;
    s1 = gt1 ? i : s1;
  }
}

// Lane r < k holds the r-th selected expert (index ri, key rk): its
// probability exp(x - m) / s, renormalised over the k selected if asked.
__device__ __forceinline__ void route_store(int lane, int64_t t, int k, int renorm, uint32_t rk,
                                            int ri, float m, float s, int32_t* idx_out,
                                            float* w_out, float* lse_out) {
  const float p = lane < k ? expf(key_value(rk) - m) / s : 0.f;
  float wsum = p;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  if (lane < k) {
    idx_out[t * k + lane] = ri;
    w_out[t * k + lane] = renorm ? p / wsum : p;
  }
  if (lse_out != nullptr && lane == 0) lse_out[t] = m + logf(s);
}

// Lane l's EPL logits: 16-byte vector loads when the row allows (vec), else
// one element at a time; experts past E are -inf.
template <typename T, int EPL>
__device__ __forceinline__ void load_block(const T* row, int lane, int E, bool vec,
                                           float (&x)[EPL]) {
  const int e0 = lane * EPL;
  constexpr int V = 16 / sizeof(T);
  if (vec && e0 + EPL <= E && EPL % V == 0) {
    const uint4* src = reinterpret_cast<const uint4*>(row + e0);
#pragma unroll
    for (int j = 0; j < EPL / V; ++j) {
      const uint4 w = src[j];
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
      if constexpr (V == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) x[j * 4 + i] = __uint_as_float(u[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[j * 8 + 2 * i] = __uint_as_float(u[i] << 16);
          x[j * 8 + 2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        }
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) x[i] = e0 + i < E ? load_f(row + e0 + i) : kNegInf;
  }
}

template <typename T, int EPL>
__global__ void __launch_bounds__(256) moe_route_kernel(const T* __restrict__ logits, int64_t T_,
                                                        int E, int k, int renorm, int vec,
                                                        int32_t* __restrict__ idx_out,
                                                        float* __restrict__ w_out,
                                                        float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T_) return;  // whole warps leave together
  // real experts get keys >= 1; padding gets 0 and is never selected
  float x[EPL];
  load_block<T, EPL>(logits + t * E, lane, E, vec != 0, x);
  uint32_t key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) key[i] = lane * EPL + i < E ? max(order_key(x[i]), 1u) : 0u;
  uint32_t taken = 0u, k1, k2;
  int s1, s2;
  top2<EPL>(key, taken, k1, s1, k2, s2);
  bool second_known = true;
  // reduction 1: the maximum (the first round's winning key)
  uint32_t wk = __reduce_max_sync(0xffffffffu, k1);
  const float m = key_value(wk);
  // reduction 2: sum of exp(x - m) (exp(-inf) = 0 for padding). x - m is
  // rounded once before the scaling by log2 e, so the hardware exp2 keeps a
  // relative error near 1e-6 even when the logits are far from zero.
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) s += ex2_approx((x[i] - m) * kLog2e);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  // reduction 3, k rounds: the largest remaining key, then the lowest lane
  // holding it (= the lowest expert index: lanes hold ascending blocks, and a
  // lane's best is its lowest slot among equal keys). Every remaining key is
  // >= 1, so a lane with nothing left (best key 0) never matches.
  int ri = 0;
  uint32_t rk = 0u;
  for (int r = 0; r < k; ++r) {
    if (r > 0) wk = __reduce_max_sync(0xffffffffu, k1);
    const uint32_t hold = __ballot_sync(0xffffffffu, k1 == wk);
    const int wl = __ffs(hold) - 1;
    const int wi = wl * EPL + __shfl_sync(0xffffffffu, s1, wl);
    if (lane == wl) {
      taken |= 1u << s1;
      if (second_known) {
        k1 = k2;
        s1 = s2;
        second_known = false;
      } else {
        top2<EPL>(key, taken, k1, s1, k2, s2);
        second_known = true;
      }
    }
    if (lane == r) {
      ri = wi;
      rk = wk;
    }
  }
  route_store(lane, t, k, renorm, rk, ri, m, s, idx_out, w_out, lse_out);
}

template <typename T, int EPL>
cudaError_t launch_route(const T* x, int64_t T_, int E, int k, int renorm, int32_t* idx,
                         float* w, float* lse, cudaStream_t s) {
  const unsigned blocks = static_cast<unsigned>((T_ + 7) / 8);
  // rows start 16-byte aligned when the base does and E fills whole vectors
  const int vec = reinterpret_cast<uintptr_t>(x) % 16 == 0 && E % (16 / sizeof(T)) == 0;
  moe_route_kernel<T, EPL><<<blocks, 256, 0, s>>>(x, T_, E, k, renorm, vec, idx, w, lse);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_route_t(const T* x, int64_t T_, int E, int k, int renorm, int32_t* idx,
                           float* w, float* lse, cudaStream_t s) {
  if (E <= 64) return launch_route<T, 2>(x, T_, E, k, renorm, idx, w, lse, s);
  if (E <= 128) return launch_route<T, 4>(x, T_, E, k, renorm, idx, w, lse, s);
  if (E <= 256) return launch_route<T, 8>(x, T_, E, k, renorm, idx, w, lse, s);
  if (E <= 512) return launch_route<T, 16>(x, T_, E, k, renorm, idx, w, lse, s);
  return launch_route<T, 32>(x, T_, E, k, renorm, idx, w, lse, s);
}

// ------------------------------------------------------------------ row moments

struct Moments {
  float n, mean, m2;
};

// Pairwise merge (Chan, Golub and LeVeque).
__device__ __forceinline__ Moments merge(Moments a, Moments b) {
  if (b.n == 0.f) return a;  // also keeps delta^2 * 0 from making NaN
  if (a.n == 0.f) return b;
  const float n = a.n + b.n;
  const float delta = b.mean - a.mean, fb = b.n / n;
  return {n, a.mean + delta * fb, a.m2 + b.m2 + delta * delta * a.n * fb};
}

// (count, mean, M2) of eight values: two passes over registers.
__device__ __forceinline__ Moments chunk8(const float (&v)[8]) {
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += v[j];
  const float mean = s * 0.125f;
  float q = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) q += (v[j] - mean) * (v[j] - mean);
  return {8.f, mean, q};
}

__device__ __forceinline__ Moments shfl_merge(Moments a, int o) {
  Moments b;
  b.n = __shfl_xor_sync(0xffffffffu, a.n, o);
  b.mean = __shfl_xor_sync(0xffffffffu, a.mean, o);
  b.m2 = __shfl_xor_sync(0xffffffffu, a.m2, o);
  return merge(a, b);
}

__device__ __forceinline__ void load8(const float* p, float (&v)[8], uint64_t pol) {
  const uint4 a = ld_global_policy(reinterpret_cast<const uint4*>(p), pol);
  const uint4 b = ld_global_policy(reinterpret_cast<const uint4*>(p) + 1, pol);
  v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
  v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
  v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
  v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8], uint64_t pol) {
  const uint4 a = ld_global_policy(reinterpret_cast<const uint4*>(p), pol);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8], uint64_t pol) {
  st_global_policy(reinterpret_cast<uint4*>(p),
                   make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                              __float_as_uint(v[3])), pol);
  st_global_policy(reinterpret_cast<uint4*>(p) + 1,
                   make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]), __float_as_uint(v[6]),
                              __float_as_uint(v[7])), pol);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8], uint64_t pol) {
  st_global_policy(reinterpret_cast<uint4*>(p),
                   make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                              pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7])), pol);
}

constexpr int kMomThreads = 512;

// vec8: the row is 16-byte aligned and cols % 8 == 0 (eight-element chunks).
template <typename T>
__global__ void __launch_bounds__(kMomThreads) row_moments_kernel(const T* __restrict__ x,
                                                                  int64_t cols, float eps,
                                                                  float* __restrict__ mean_out,
                                                                  float* __restrict__ var_out,
                                                                  T* __restrict__ y, int vec8) {
  __shared__ Moments part[kMomThreads / 32];
  __shared__ float stats[2];
  const int64_t row = blockIdx.x;
  const T* xr = x + row * cols;
  const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
  const uint64_t pol1 = y != nullptr ? keep : drop;  // keep the row for the second pass
  Moments st{0.f, 0.f, 0.f};
  if (vec8) {
    for (int64_t c = int64_t(threadIdx.x) * 8; c < cols; c += int64_t(kMomThreads) * 8) {
      float v[8];
      load8(xr + c, v, pol1);
      st = merge(st, chunk8(v));
    }
  } else {
    for (int64_t c = threadIdx.x; c < cols; c += kMomThreads) {
      const float v = static_cast<float>(xr[c]);
      st = merge(st, Moments{1.f, v, 0.f});
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) st = shfl_merge(st, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = st;
  __syncthreads();
  if (threadIdx.x < 32) {
    Moments w = threadIdx.x < kMomThreads / 32 ? part[threadIdx.x] : Moments{0.f, 0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = shfl_merge(w, o);
    if (threadIdx.x == 0) {
      const float var = w.n > 0.f ? w.m2 / w.n : 0.f;
      stats[0] = w.mean;
      stats[1] = var;
      if (mean_out != nullptr) mean_out[row] = w.mean;
      if (var_out != nullptr) var_out[row] = var;
    }
  }
  if (y == nullptr) return;
  __syncthreads();
  const float mean = stats[0], inv = rsqrtf(stats[1] + eps);
  T* yr = y + row * cols;
  if (vec8) {
    for (int64_t c = int64_t(threadIdx.x) * 8; c < cols; c += int64_t(kMomThreads) * 8) {
      float v[8];
      load8(xr + c, v, drop);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = (v[j] - mean) * inv;
      store8(yr + c, v, drop);
    }
  } else {
    for (int64_t c = threadIdx.x; c < cols; c += kMomThreads)
      yr[c] = static_cast<T>((static_cast<float>(xr[c]) - mean) * inv);
  }
}

// Rows of up to NCH * 8 * kMomThreads elements (vec8 rows only; used for
// float rows too long for shared memory, up to 32768 elements): each thread
// holds its NCH eight-element chunks in registers from the load to the
// normalised store, so x is read from HBM exactly once.
template <typename T, int NCH>
__global__ void __launch_bounds__(kMomThreads) row_moments_regs_kernel(
    const T* __restrict__ x, int64_t cols, float eps, float* __restrict__ mean_out,
    float* __restrict__ var_out, T* __restrict__ y) {
  __shared__ Moments part[kMomThreads / 32];
  __shared__ float stats[2];
  const int64_t row = blockIdx.x;
  const T* xr = x + row * cols;
  const uint64_t drop = policy_evict_first();
  float v[NCH][8];
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int64_t c = (int64_t(j) * kMomThreads + threadIdx.x) * 8;
    if (c < cols) load8(xr + c, v[j], drop);
  }
  Moments st{0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int64_t c = (int64_t(j) * kMomThreads + threadIdx.x) * 8;
    if (c < cols) st = merge(st, chunk8(v[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) st = shfl_merge(st, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = st;
  __syncthreads();
  if (threadIdx.x < 32) {
    Moments w = threadIdx.x < kMomThreads / 32 ? part[threadIdx.x] : Moments{0.f, 0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = shfl_merge(w, o);
    if (threadIdx.x == 0) {
      const float var = w.n > 0.f ? w.m2 / w.n : 0.f;
      stats[0] = w.mean;
      stats[1] = var;
      if (mean_out != nullptr) mean_out[row] = w.mean;
      if (var_out != nullptr) var_out[row] = var;
    }
  }
  if (y == nullptr) return;
  __syncthreads();
  const float mean = stats[0], inv = rsqrtf(stats[1] + eps);
  T* yr = y + row * cols;
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int64_t c = (int64_t(j) * kMomThreads + threadIdx.x) * 8;
    if (c < cols) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[j][i] = (v[j][i] - mean) * inv;
      store8(yr + c, v[j], drop);
    }
  }
}

// 16-byte asynchronous global -> shared copies (completion is a hardware
// wait on the thread's own copy groups; no spin loop).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;\n"
               :: "r"(smem_u32(dst)), "l"(src), "l"(pol) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

// Four or eight values of one 16-byte unit (f32 / bf16).
__device__ __forceinline__ int unit_vals(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  return 4;
}
__device__ __forceinline__ int unit_vals(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
  return 8;
}
__device__ __forceinline__ void unit_store(float* p, const float (&v)[8], uint64_t pol) {
  st_global_policy(reinterpret_cast<uint4*>(p),
                   make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                              __float_as_uint(v[3])), pol);
}
__device__ __forceinline__ void unit_store(__nv_bfloat16* p, const float (&v)[8], uint64_t pol) {
  store8(p, v, pol);
}

// (count, mean, M2) of the N = 4 or 8 values of a unit: two passes over
// registers.
template <int N>
__device__ __forceinline__ Moments chunk_n(const float (&v)[8]) {
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < N; ++j) s += v[j];
  const float mean = s * (1.f / N);
  float q = 0.f;
#pragma unroll
  for (int j = 0; j < N; ++j) q += (v[j] - mean) * (v[j] - mean);
  return {float(N), mean, q};
}

constexpr int kSmemThreads = 256;
constexpr int kSmemRowBytes = 64 * 1024;

// Rows of up to 64 KB (vec8 rows): the CTA copies its row into shared
// memory in 16-byte units (unit u by thread u mod 256, so a quarter-warp
// touches 128 contiguous bytes: no bank conflicts), takes the moments from
// there and writes the normalised row from there: x is read from HBM once.
// Small CTAs and no registers held across the copy let about seven rows
// per SM be in flight.
template <typename T>
__global__ void __launch_bounds__(kSmemThreads) row_moments_smem_kernel(
    const T* __restrict__ x, int64_t cols, float eps, float* __restrict__ mean_out,
    float* __restrict__ var_out, T* __restrict__ y) {
  extern __shared__ __align__(16) unsigned char srow[];
  __shared__ Moments part[kSmemThreads / 32];
  __shared__ float stats[2];
  constexpr int kPer = 16 / sizeof(T);
  const int64_t row = blockIdx.x;
  const int nunits = static_cast<int>(cols / kPer);
  const unsigned char* src = reinterpret_cast<const unsigned char*>(x + row * cols);
  const uint64_t drop = policy_evict_first();
  for (int u = threadIdx.x; u < nunits; u += kSmemThreads)
    cp_async16(srow + 16 * u, src + 16 * int64_t(u), drop);
  cp_async_wait_all();
  __syncthreads();
  const T* xs = reinterpret_cast<const T*>(srow);
  Moments st{0.f, 0.f, 0.f};
  for (int u = threadIdx.x; u < nunits; u += kSmemThreads) {
    float v[8];
    unit_vals(xs + u * kPer, v);
    st = merge(st, chunk_n<kPer>(v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) st = shfl_merge(st, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = st;
  __syncthreads();
  if (threadIdx.x < 32) {
    Moments w = threadIdx.x < kSmemThreads / 32 ? part[threadIdx.x] : Moments{0.f, 0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = shfl_merge(w, o);
    if (threadIdx.x == 0) {
      const float var = w.n > 0.f ? w.m2 / w.n : 0.f;
      stats[0] = w.mean;
      stats[1] = var;
      if (mean_out != nullptr) mean_out[row] = w.mean;
      if (var_out != nullptr) var_out[row] = var;
    }
  }
  if (y == nullptr) return;
  __syncthreads();
  const float mean = stats[0], inv = rsqrtf(stats[1] + eps);
  T* yr = y + row * cols;
  for (int u = threadIdx.x; u < nunits; u += kSmemThreads) {
    float v[8];
    unit_vals(xs + u * kPer, v);
#pragma unroll
    for (int j = 0; j < kPer; ++j) v[j] = (v[j] - mean) * inv;
    unit_store(yr + int64_t(u) * kPer, v, drop);
  }
}

template <typename T>
cudaError_t launch_moments_t(const T* x, int64_t rows, int64_t cols, float eps, float* mean,
                             float* var, T* y, bool vec8, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>(rows);
  const int64_t per_pass = int64_t(8) * kMomThreads;
  const int64_t nch = (cols + per_pass - 1) / per_pass;
  const int64_t row_bytes = cols * int64_t(sizeof(T));
  if (vec8 && row_bytes <= kSmemRowBytes) {
    const int smem = static_cast<int>(row_bytes);
    if (smem > 46 * 1024) {  // with the kernel's static shared memory, past the 48 KB default
      cudaError_t e = cudaFuncSetAttribute(row_moments_smem_kernel<T>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemRowBytes);
      if (e != cudaSuccess) return e;
    }
    row_moments_smem_kernel<T><<<grid, kSmemThreads, smem, s>>>(x, cols, eps, mean, var, y);
  } else if (sizeof(T) == 4 && vec8 && nch <= 8) {
    // float rows of 64 to 128 KB
    row_moments_regs_kernel<T, 8><<<grid, kMomThreads, 0, s>>>(x, cols, eps, mean, var, y);
  } else {
    row_moments_kernel<T><<<grid, kMomThreads, 0, s>>>(x, cols, eps, mean, var, y, vec8 ? 1 : 0);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------ moment of inertia

// (W, c, M2) of point masses: total mass, weighted mean position, and the
// sum of m |r - c|^2.
struct WMoments {
  float w, cx, cy, cz, m2;
};

__device__ __forceinline__ WMoments wmerge(WMoments a, WMoments b) {
  if (b.w == 0.f) return a;
  if (a.w == 0.f) return b;
  const float w = a.w + b.w, f = b.w / w;
  const float dx = b.cx - a.cx, dy = b.cy - a.cy, dz = b.cz - a.cz;
  return {w, a.cx + dx * f, a.cy + dy * f, a.cz + dz * f,
          a.m2 + b.m2 + (dx * dx + dy * dy + dz * dz) * a.w * f};
}

__device__ __forceinline__ WMoments wshfl_merge(WMoments a, int o) {
  WMoments b;
  b.w = __shfl_xor_sync(0xffffffffu, a.w, o);
  b.cx = __shfl_xor_sync(0xffffffffu, a.cx, o);
  b.cy = __shfl_xor_sync(0xffffffffu, a.cy, o);
  b.cz = __shfl_xor_sync(0xffffffffu, a.cz, o);
  b.m2 = __shfl_xor_sync(0xffffffffu, a.m2, o);
  return wmerge(a, b);
}

// Four point masses: two passes over registers (centre, then M2).
__device__ __forceinline__ WMoments chunk4(const float (&x)[12], const float (&m)[4]) {
  const float w = (m[0] + m[1]) + (m[2] + m[3]);
  if (w == 0.f) return {0.f, 0.f, 0.f, 0.f, 0.f};
  float sx = 0.f, sy = 0.f, sz = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    sx = fmaf(m[i], x[3 * i], sx);
    sy = fmaf(m[i], x[3 * i + 1], sy);
    sz = fmaf(m[i], x[3 * i + 2], sz);
  }
  const float inv = 1.f / w;
  const float cx = sx * inv, cy = sy * inv, cz = sz * inv;
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float dx = x[3 * i] - cx, dy = x[3 * i + 1] - cy, dz = x[3 * i + 2] - cz;
    q = fmaf(m[i], dx * dx + dy * dy + dz * dz, q);
  }
  return {w, cx, cy, cz, q};
}

constexpr int kInertiaThreads = 256;

// One CTA per point set. vec4: the set's points and masses start 16-byte
// aligned and n % 4 == 0 (four points = three float4, four masses = one).
__global__ void __launch_bounds__(kInertiaThreads) inertia_kernel(
    const float* __restrict__ pts, const float* __restrict__ mass, int64_t n, int vec4,
    float* __restrict__ total, float* __restrict__ centre, float* __restrict__ inertia) {
  __shared__ WMoments part[kInertiaThreads / 32];
  const int64_t set = blockIdx.x;
  const float* ps = pts + set * n * 3;
  const float* ms = mass != nullptr ? mass + set * n : nullptr;
  const uint64_t drop = policy_evict_first();
  WMoments st{0.f, 0.f, 0.f, 0.f, 0.f};
  if (vec4) {
#pragma unroll 2
    for (int64_t c = threadIdx.x; c < n / 4; c += kInertiaThreads) {
      float x[12], m[4];
      const uint4* p4 = reinterpret_cast<const uint4*>(ps + c * 12);
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const uint4 u = ld_global_policy(p4 + j, drop);
        x[4 * j] = __uint_as_float(u.x);
        x[4 * j + 1] = __uint_as_float(u.y);
        x[4 * j + 2] = __uint_as_float(u.z);
        x[4 * j + 3] = __uint_as_float(u.w);
      }
      if (ms != nullptr) {
        const uint4 u = ld_global_policy(reinterpret_cast<const uint4*>(ms + c * 4), drop);
        m[0] = __uint_as_float(u.x);
        m[1] = __uint_as_float(u.y);
        m[2] = __uint_as_float(u.z);
        m[3] = __uint_as_float(u.w);
      } else {
        m[0] = m[1] = m[2] = m[3] = 1.f;
      }
      st = wmerge(st, chunk4(x, m));
    }
  } else {
    for (int64_t i = threadIdx.x; i < n; i += kInertiaThreads) {
      const float mi = ms != nullptr ? ms[i] : 1.f;
      st = wmerge(st, WMoments{mi, ps[3 * i], ps[3 * i + 1], ps[3 * i + 2], 0.f});
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) st = wshfl_merge(st, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = st;
  __syncthreads();
  if (threadIdx.x < 32) {
    WMoments w = threadIdx.x < kInertiaThreads / 32 ? part[threadIdx.x]
                                                     : WMoments{0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = wshfl_merge(w, o);
    if (threadIdx.x == 0) {
      if (total != nullptr) total[set] = w.w;
      if (centre != nullptr) {
        centre[3 * set] = w.cx;
        centre[3 * set + 1] = w.cy;
        centre[3 * set + 2] = w.cz;
      }
      if (inertia != nullptr) inertia[set] = w.m2;
    }
  }
}

}  // namespace

cudaError_t launch_moe_route(const void* logits, int64_t T_, int E, int k, int renorm,
                             int32_t* idx, float* w, float* lse, rf_dtype dt, cudaStream_t s) {
  if (dt == RF_F32)
    return launch_route_t(static_cast<const float*>(logits), T_, E, k, renorm, idx, w, lse, s);
  return launch_route_t(static_cast<const __nv_bfloat16*>(logits), T_, E, k, renorm, idx, w, lse,
                        s);
}

cudaError_t launch_row_moments(const void* x, int64_t rows, int64_t cols, float eps, float* mean,
                               float* var, void* y, rf_dtype dt, cudaStream_t s) {
  const size_t esz = dt == RF_F32 ? 4 : 2;
  const bool vec8 = reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                    (y == nullptr || reinterpret_cast<uintptr_t>(y) % 16 == 0) &&
                    (cols * esz) % 16 == 0 && cols % 8 == 0;
  if (dt == RF_F32)
    return launch_moments_t(static_cast<const float*>(x), rows, cols, eps, mean, var,
                            static_cast<float*>(y), vec8, s);
  return launch_moments_t(static_cast<const __nv_bfloat16*>(x), rows, cols, eps, mean, var,
                          static_cast<__nv_bfloat16*>(y), vec8, s);
}

cudaError_t launch_moment_of_inertia(const float* points, const float* masses, int64_t sets,
                                     int64_t n, float* total, float* centre, float* inertia,
                                     cudaStream_t s) {
  const bool vec4 = n % 4 == 0 && reinterpret_cast<uintptr_t>(points) % 16 == 0 &&
                    (masses == nullptr || reinterpret_cast<uintptr_t>(masses) % 16 == 0);
  inertia_kernel<<<static_cast<unsigned>(sets), kInertiaThreads, 0, s>>>(
      points, masses, n, vec4 ? 1 : 0, total, centre, inertia);
  return cudaGetLastError();
}

}  // namespace rf
