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
// lower expert index. Each lane keeps its best remaining expert; a round is
// two single-instruction warp reductions (redux.sync) over order-preserving
// integer keys of the logits -- the largest key, then the lowest index
// holding it. With up to eight experts per lane, each lane sorts its slots
// once (a sorting network) and the winner pops the head of its list; with
// more, the winning lane rescans its slots. The token's logits are read once.
//
// Row moments (one CTA per row): each thread folds its elements into a
// (count, mean, M2) state, eight at a time (two passes over eight registers,
// then the pairwise merge of Chan, Golub and LeVeque), the states merge across
// the warp and the CTA by the same rule (multi-segment strategy, merge step),
// and var = M2 / n. With an output, a second pass writes (x - mean) /
// sqrt(var + eps). Rows of up to 32768 elements stay in registers between the
// two (x is read once); longer rows are read a second time, from L2, where
// the first pass left them with an evict-last policy.
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

// The lane's best remaining expert: the largest key, the lowest slot on ties
// (slots are in ascending expert order). No slot left: key 0, slot EPL.
template <int EPL>
__device__ __forceinline__ void local_best(const uint32_t (&key)[EPL], uint32_t taken,
                                           uint32_t& bk, int& bs) {
  bk = 0u;
  bs = EPL;
#pragma unroll
  for (int i = EPL - 1; i >= 0; --i) {
    if (!((taken >> i) & 1u) && key[i] >= bk) {
      bk = key[i];
      bs = i;
    }
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

// Up to 32 experts per lane: the winning lane of a round rescans its slots.
template <typename T, int EPL>
__global__ void __launch_bounds__(256) moe_route_kernel(const T* __restrict__ logits, int64_t T_,
                                                        int E, int k, int renorm,
                                                        int32_t* __restrict__ idx_out,
                                                        float* __restrict__ w_out,
                                                        float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T_) return;  // whole warps leave together
  const T* row = logits + t * E;
  // lane l holds experts l, l + 32, ... (coalesced loads); padding slots are
  // marked taken so that they are never selected
  uint32_t key[EPL];
  float x[EPL];
  uint32_t taken = 0u;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    x[i] = e < E ? load_f(row + e) : kNegInf;
    key[i] = order_key(x[i]);
    if (e >= E) taken |= 1u << i;
  }
  uint32_t bk;
  int bs;
  local_best<EPL>(key, taken, bk, bs);
  // reduction 1: the maximum (the first selection round's winner)
  uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
  const float m = key_value(wk);
  // reduction 2: sum of exp(x - m) (exp(-inf) = 0 for padding)
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) s += expf(x[i] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  // reduction 3, k rounds: the largest remaining key, then the lowest expert
  // index among the lanes holding it
  int ri = 0;
  uint32_t rk = 0u;
  for (int r = 0; r < k; ++r) {
    if (r > 0) wk = __reduce_max_sync(0xffffffffu, bk);
    const int cand = (bk == wk && bs < EPL) ? lane + 32 * bs : 0x7fffffff;
    const int wi = __reduce_min_sync(0xffffffffu, cand);
    if (wi == lane + 32 * bs) {  // the winning lane drops its best and finds the next
      taken |= 1u << bs;
      local_best<EPL>(key, taken, bk, bs);
    }
    if (lane == r) {
      ri = wi;
      rk = wk;
    }
  }
  route_store(lane, t, k, renorm, rk, ri, m, s, idx_out, w_out, lse_out);
}

// Compare-exchange for a descending order of (key, then lower slot first).
__device__ __forceinline__ void cex(uint32_t& ka, uint32_t& sa, uint32_t& kb, uint32_t& sb) {
  const bool sw = kb > ka || (kb == ka && sb < sa);
  const uint32_t k0 = sw ? kb : ka, s0 = sw ? sb : sa;
  kb = sw ? ka : kb;
  sb = sw ? sa : sb;
  ka = k0;
  sa = s0;
}

// Sorting networks on 2, 4 and 8 inputs (1, 5 and 19 comparators; the
// 8-input one has depth 6), checked on every 0-1 input.
template <int EPL>
__device__ __forceinline__ void sort_lane(uint32_t (&k)[EPL], uint32_t (&s)[EPL]) {
#define RF_CEX(a, b) cex(k[a], s[a], k[b], s[b])
  if constexpr (EPL == 2) {
    RF_CEX(0, 1);
  } else if constexpr (EPL == 4) {
    RF_CEX(0, 1); RF_CEX(2, 3); RF_CEX(0, 2); RF_CEX(1, 3); RF_CEX(1, 2);
  } else {
    static_assert(EPL == 8, "sorted lanes hold 2, 4 or 8 experts");
    RF_CEX(0, 2); RF_CEX(1, 3); RF_CEX(4, 6); RF_CEX(5, 7);
    RF_CEX(0, 4); RF_CEX(1, 5); RF_CEX(2, 6); RF_CEX(3, 7);
    RF_CEX(0, 1); RF_CEX(2, 3); RF_CEX(4, 5); RF_CEX(6, 7);
    RF_CEX(2, 4); RF_CEX(3, 5);
    RF_CEX(1, 4); RF_CEX(3, 6);
    RF_CEX(1, 2); RF_CEX(3, 4); RF_CEX(5, 6);
  }
#undef RF_CEX
}

// Up to 8 experts per lane: each lane sorts its slots once; a round's
// winning lane pops the head of its sorted list (no rescan).
template <typename T, int EPL>
__global__ void __launch_bounds__(256) moe_route_sorted_kernel(
    const T* __restrict__ logits, int64_t T_, int E, int k, int renorm,
    int32_t* __restrict__ idx_out, float* __restrict__ w_out, float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T_) return;  // whole warps leave together
  const T* row = logits + t * E;
  // real experts get keys >= 1; padding gets 0 and sorts last, never selected
  float x[EPL];
  uint32_t key[EPL], sl[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    x[i] = e < E ? load_f(row + e) : kNegInf;
    key[i] = e < E ? max(order_key(x[i]), 1u) : 0u;
    sl[i] = i;
  }
  sort_lane<EPL>(key, sl);
  uint32_t packed = 0u;  // sorted slots, four bits each, head in the low bits
#pragma unroll
  for (int i = 0; i < EPL; ++i) packed |= sl[i] << (4 * i);
  // reduction 1: the maximum (the first round's winning key)
  uint32_t wk = __reduce_max_sync(0xffffffffu, key[0]);
  const float m = key_value(wk);
  // reduction 2: sum of exp(x - m)
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) s += expf(x[i] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  // reduction 3, k rounds (every remaining key is >= 1, so an exhausted
  // lane, whose head key is 0, never matches)
  int ri = 0;
  uint32_t rk = 0u;
  for (int r = 0; r < k; ++r) {
    if (r > 0) wk = __reduce_max_sync(0xffffffffu, key[0]);
    const int my_e = lane + 32 * int(packed & 15u);
    const int wi = __reduce_min_sync(0xffffffffu, key[0] == wk ? my_e : 0x7fffffff);
    if (wi == my_e && key[0] == wk) {  // pop the head
#pragma unroll
      for (int i = 0; i < EPL - 1; ++i) key[i] = key[i + 1];
      key[EPL - 1] = 0u;
      packed >>= 4;
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
  if constexpr (EPL <= 8)
    moe_route_sorted_kernel<T, EPL><<<blocks, 256, 0, s>>>(x, T_, E, k, renorm, idx, w, lse);
  else
    moe_route_kernel<T, EPL><<<blocks, 256, 0, s>>>(x, T_, E, k, renorm, idx, w, lse);
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

// Rows of up to NCH * 8 * kMomThreads elements (vec8 rows only): each thread
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

template <typename T>
cudaError_t launch_moments_t(const T* x, int64_t rows, int64_t cols, float eps, float* mean,
                             float* var, T* y, bool vec8, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>(rows);
  const int64_t per_pass = int64_t(8) * kMomThreads;
  const int64_t nch = (cols + per_pass - 1) / per_pass;
  if (vec8 && nch <= 1)
    row_moments_regs_kernel<T, 1><<<grid, kMomThreads, 0, s>>>(x, cols, eps, mean, var, y);
  else if (vec8 && nch <= 2)
    row_moments_regs_kernel<T, 2><<<grid, kMomThreads, 0, s>>>(x, cols, eps, mean, var, y);
  else if (vec8 && nch <= 4)
    row_moments_regs_kernel<T, 4><<<grid, kMomThreads, 0, s>>>(x, cols, eps, mean, var, y);
  else if (vec8 && nch <= 8)
    row_moments_regs_kernel<T, 8><<<grid, kMomThreads, 0, s>>>(x, cols, eps, mean, var, y);
  else
    row_moments_kernel<T><<<grid, kMomThreads, 0, s>>>(x, cols, eps, mean, var, y, vec8 ? 1 : 0);
  return cudaGetLastError();
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

}  // namespace rf
