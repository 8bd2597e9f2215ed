// decode.cu -- split-K decode partials and the log-sum-exp merge.
//
// RedFuser (An Automatic Operator Fusion Framework for Cascaded Reductions
// on AI Accelerators), section 3: the multi-segment strategy partitions the
// input for parallelism and merges the partial results; FlashDecoding is a
// special case of it. Each CTA owns one (batch, kv-head, split): it streams
// that split's K and V once from HBM and keeps, for every query head of the
// group, the incremental state (m, l, acc) of section 2 (running max, running
// sum, accumulator rescaled by exp(m_old - m_new)). It writes the split's
// normalised partial O_s = acc / l and lse_s = m + ln l; the merge kernel then
// combines the splits with LSE = log sum_s exp(lse_s) and
// O = sum_s exp(lse_s - LSE) O_s (the monoid merge of two states).
//
// Memory path (HBM-bound): one producer lane streams 16 KB K and V chunks
// with cp.async.bulk into a 3-stage shared-memory ring (mbarrier
// transaction counts, L2 evict-first); four consumer warps split each chunk.
// Inside a warp, lane l owns head-dim elements [l*D/32, (l+1)*D/32): partial
// dot products of a batch of keys against every query head of the group are
// reduced across lanes by a reduce-scatter (halving exchange), which leaves
// two finished scores per lane instead of broadcasting all of them.
#include <type_traits>

#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kChunkBytes = 16384;  // bytes of K (and of V) per stage

template <int D>
struct DecodeShape {
  static constexpr int CH = kChunkBytes / (D * 2);  // keys per chunk
  static constexpr int DPL = D / 32;                // head-dim elements per lane
};

// Shared-memory layout of one CTA.
template <int D>
struct DecodeSmem {
  __nv_bfloat16 k[kStages][DecodeShape<D>::CH * D];
  __nv_bfloat16 v[kStages][DecodeShape<D>::CH * D];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  float pbuf[kConsumerWarps][64];
  int abort_flag;
};

// One halving step of the reduce-scatter: lanes whose bit `OFF` is set keep
// the upper HALF values, the others the lower ones, each adding its partner's.
template <int HALF, int OFF>
__device__ __forceinline__ void rs_step(float (&x)[64]) {
  const bool upper = (threadIdx.x & OFF) != 0;
#pragma unroll
  for (int i = 0; i < HALF; ++i) {
    const float send = upper ? x[i] : x[i + HALF];
    const float keep = upper ? x[i + HALF] : x[i];
    x[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
  }
}

// Reduce-scatter of 64 values over the 32 lanes of a warp: afterwards lane l
// holds the warp-wide sums of values 2l and 2l+1 in x[0], x[1].
__device__ __forceinline__ void reduce_scatter64(float (&x)[64]) {
  rs_step<32, 16>(x);
  rs_step<16, 8>(x);
  rs_step<8, 4>(x);
  rs_step<4, 2>(x);
  rs_step<2, 1>(x);
}

// v[g] for a runtime head index g, without indexing a register array.
template <int GP>
__device__ __forceinline__ float pick(const float (&v)[GP], int g) {
  float r = 0.f;
#pragma unroll
  for (int i = 0; i < GP; ++i) r = (i == g) ? v[i] : r;
  return r;
}

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

// This lane's D/32 elements of a bf16 row as D/64 packed float pairs.
template <int D>
__device__ __forceinline__ void load_row_pairs(const __nv_bfloat16* row, float2 (&out)[D / 64]) {
  const int lane = threadIdx.x & 31;
  if constexpr (D == 128) {
    const uint2 w = *reinterpret_cast<const uint2*>(row + lane * 4);
    bf16x2_to_f32(w.x, out[0].x, out[0].y);
    bf16x2_to_f32(w.y, out[1].x, out[1].y);
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(row + lane * 2);
    bf16x2_to_f32(w, out[0].x, out[0].y);
  }
}

template <int D>
__device__ __forceinline__ void load_row_slice(const __nv_bfloat16* row, float (&out)[D / 32]) {
  const int lane = threadIdx.x & 31;
  if constexpr (D == 128) {
    const uint2 w = *reinterpret_cast<const uint2*>(row + lane * 4);
    bf16x2_to_f32(w.x, out[0], out[1]);
    bf16x2_to_f32(w.y, out[2], out[3]);
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(row + lane * 2);
    bf16x2_to_f32(w, out[0], out[1]);
  }
}

// GP = query heads per kv head, padded to 4, 8 or 16; G = real count.
template <int D, int GP>
__global__ void __launch_bounds__(kThreads) decode_partials_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, float* __restrict__ o_part,
    float* __restrict__ lse_part, int H, int Hkv, int Sk, int nsplit, float scale_log2,
    int* status) {
  using S = DecodeShape<D>;
  constexpr int CH = S::CH, DPL = S::DPL;
  constexpr int KB = 64 / GP;                 // keys per warp batch (64 scores)
  constexpr int KPW = CH / kConsumerWarps;    // keys per warp per chunk
  static_assert(KPW % KB == 0, "batch must divide a warp's share of a chunk");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  DecodeSmem<D>& sm = *reinterpret_cast<DecodeSmem<D>*>(smem_raw);

  const int G = H / Hkv;
  const int split = blockIdx.x % nsplit;
  const int bk = blockIdx.x / nsplit;  // b * Hkv + hk
  const int b = bk / Hkv, hk = bk % Hkv;
  const int per = Sk / nsplit;
  const int key0 = split * per;
  const int key1 = (split == nsplit - 1) ? Sk : key0 + per;
  const int nkeys = key1 - key0;
  const int nchunks = (nkeys + CH - 1) / CH;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __nv_bfloat16* kbase = k + (int64_t(bk) * Sk + key0) * D;
  const __nv_bfloat16* vbase = v + (int64_t(bk) * Sk + key0) * D;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumerWarps);
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------- producer: one lane streams K/V chunks
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int last[kStages] = {-1, -1, -1};
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kStages;
        if (!mbar_wait(&sm.empty[s], ((c / kStages) & 1) ^ 1, status,
                       dev_code(kDevTimeout, kKerDecode, 1), &sm.abort_flag))
          break;
        const int n = min(CH, nkeys - c * CH);
        const uint32_t bytes = static_cast<uint32_t>(n) * D * 2;
        mbar_arrive_expect_tx(&sm.full[s], 2 * bytes);
        bulk_load(sm.k[s], kbase + int64_t(c) * CH * D, bytes, &sm.full[s], pol);
        bulk_load(sm.v[s], vbase + int64_t(c) * CH * D, bytes, &sm.full[s], pol);
        last[s] = c;
      }
      // never leave with copies in flight
      for (int s = 0; s < kStages; ++s)
        if (last[s] >= 0)
          mbar_wait(&sm.full[s], (last[s] / kStages) & 1, status,
                    dev_code(kDevTimeout, kKerDecode, 2), nullptr);
    }
    __syncwarp();
    __syncthreads();  // pairs with the consumers' barrier before the combine
    return;
  }

  // ---------------- consumers
  // query slice of every head in the group, pre-scaled into log2 units
  float qv[GP][DPL];
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    if (g < G) {
      const int h = hk * G + g;
      load_row_slice<D>(q + (int64_t(b) * H + h) * D, qv[g]);
#pragma unroll
      for (int e = 0; e < DPL; ++e) qv[g][e] *= scale_log2;
    } else {
#pragma unroll
      for (int e = 0; e < DPL; ++e) qv[g][e] = 0.f;
    }
  }
  // state: running max per head (all lanes), lane-partial sums for the two
  // heads this lane scores, accumulators [head][own head-dim slice]
  constexpr int DP2 = DPL / 2;  // packed float pairs per lane
  float2 q2[GP][DP2];
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int e = 0; e < DP2; ++e) q2[g][e] = make_float2(qv[g][2 * e], qv[g][2 * e + 1]);
  float m[GP], lpart[2] = {0.f, 0.f};
  float2 acc[GP][DP2];
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    m[g] = kNegInf;
#pragma unroll
    for (int e = 0; e < DP2; ++e) acc[g][e] = make_float2(0.f, 0.f);
  }
  // this lane's two scores are (key 2l/GP, head 2l%GP) and (.., +1)
  const int my_key = (2 * lane) / GP;
  const int my_g = (2 * lane) % GP;
  float* pb = sm.pbuf[warp];

  for (int c = 0; c < nchunks; ++c) {
    const int s = c % kStages;
    if (!mbar_wait_warp(&sm.full[s], (c / kStages) & 1, status,
                        dev_code(kDevTimeout, kKerDecode, 3), &sm.abort_flag))
      break;
    const int n = min(CH, nkeys - c * CH);
    const __nv_bfloat16* kc = sm.k[s];
    const __nv_bfloat16* vc = sm.v[s];
#pragma unroll 1
    for (int kb = warp * KPW; kb < (warp + 1) * KPW; kb += KB) {
      if (kb >= n) break;
      // partial dot products: part[key * GP + g]
      float part[64];
#pragma unroll
      for (int j = 0; j < KB; ++j) {
        float2 kr[DP2];
        load_row_pairs<D>(kc + (kb + j) * D, kr);
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          float2 a = __fmul2_rn(q2[g][0], kr[0]);
#pragma unroll
          for (int e = 1; e < DP2; ++e) a = ffma2(q2[g][e], kr[e], a);
          part[j * GP + g] = a.x + a.y;
        }
      }
      reduce_scatter64(part);
      // my two scores (log2 units); keys past the split are masked
      const bool valid = kb + my_key < n;
      float s0 = valid && my_g < G ? part[0] : kNegInf;
      float s1 = valid && my_g + 1 < G ? part[1] : kNegInf;
      // tile max per head: lanes with equal (lane % (GP/2)) hold the same heads
      float mx0 = s0, mx1 = s1;
#pragma unroll
      for (int off = GP / 2; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      float alpha[GP];
      bool grow = false;
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        const float tm = __shfl_sync(0xffffffffu, (g & 1) ? mx1 : mx0, g >> 1);
        const float mn = fmaxf(m[g], tm);
        alpha[g] = (mn == kNegInf || m[g] == mn) ? 1.f : ex2_approx(m[g] - mn);
        grow |= (mn != m[g]);
        m[g] = mn;
      }
      const float ms0 = pick<GP>(m, my_g);
      const float ms1 = pick<GP>(m, my_g + 1);
      const float p0 = (s0 == kNegInf) ? 0.f : ex2_approx(s0 - ms0);
      const float p1 = (s1 == kNegInf) ? 0.f : ex2_approx(s1 - ms1);
      if (__any_sync(0xffffffffu, grow)) {
        lpart[0] *= pick<GP>(alpha, my_g);
        lpart[1] *= pick<GP>(alpha, my_g + 1);
#pragma unroll
        for (int g = 0; g < GP; ++g)
#pragma unroll
          for (int e = 0; e < DP2; ++e)
            acc[g][e] = __fmul2_rn(acc[g][e], make_float2(alpha[g], alpha[g]));
      }
      lpart[0] += p0;
      lpart[1] += p1;
      // broadcast the batch's probabilities, then acc += p * V
      *reinterpret_cast<float2*>(pb + 2 * lane) = make_float2(p0, p1);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < KB; ++j) {
        if (kb + j >= n) break;
        float2 vr[DP2];
        load_row_pairs<D>(vc + (kb + j) * D, vr);
#pragma unroll
        for (int g4 = 0; g4 < GP; g4 += 4) {
          const float4 p = *reinterpret_cast<const float4*>(pb + j * GP + g4);
          const float pp[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int e = 0; e < DP2; ++e)
              acc[g4 + u][e] = ffma2(make_float2(pp[u], pp[u]), vr[e], acc[g4 + u][e]);
        }
      }
      __syncwarp();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
  }
  // finish the lane-partial sums: heads (my_g, my_g+1) over lanes sharing them
#pragma unroll
  for (int off = GP / 2; off < 32; off <<= 1) {
    lpart[0] += __shfl_xor_sync(0xffffffffu, lpart[0], off);
    lpart[1] += __shfl_xor_sync(0xffffffffu, lpart[1], off);
  }
  float l[GP];
#pragma unroll
  for (int g = 0; g < GP; ++g) l[g] = __shfl_sync(0xffffffffu, (g & 1) ? lpart[1] : lpart[0], g >> 1);

  // combine the four consumer warps (disjoint key subsets) through shared
  // memory, reusing the K stages (every copy has landed and been consumed)
  __syncthreads();
  float* cm = reinterpret_cast<float*>(sm.k[0]);           // [warps][GP]
  float* cl = cm + kConsumerWarps * GP;                     // [warps][GP]
  float* ca = cl + kConsumerWarps * GP;                     // [warps][GP][D]
  if (lane == 0)
    for (int g = 0; g < GP; ++g) {
      cm[warp * GP + g] = m[g];
      cl[warp * GP + g] = l[g];
    }
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int e = 0; e < DP2; ++e)
      *reinterpret_cast<float2*>(ca + (warp * GP + g) * D + lane * DPL + 2 * e) = acc[g][e];
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32));
  if (sm.abort_flag) return;
  for (int t = threadIdx.x; t < G * D; t += kConsumerWarps * 32) {
    const int g = t / D, col = t % D;
    float M = kNegInf;
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cm[w * GP + g]);
    float L = 0.f, O = 0.f;
    if (M != kNegInf)
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = cm[w * GP + g];
        if (mw == kNegInf) continue;
        const float f = ex2_approx(mw - M);
        L += cl[w * GP + g] * f;
        O += ca[(w * GP + g) * D + col] * f;
      }
    const int64_t row = int64_t(b) * H + hk * G + g;
    o_part[(row * nsplit + split) * D + col] = L > 0.f ? O / L : 0.f;
    if (col == 0) lse_part[row * nsplit + split] = L > 0.f ? (M + log2f(L)) * kLn2 : kNegInf;
  }
}

// One warp per output row: LSE = log sum_s exp(lse_s); O = sum_s w_s O_s.
// Lane s computes split s's weight exp(lse_s - LSE) once (32 splits at a time)
// and the weights are broadcast by shuffles; each lane then accumulates its
// columns with 16-byte loads when the row allows it.
// Partial s of row r sits at o_part[s * o_split + r * o_row] (d floats) and
// lse_part[s * l_split + r * l_row]: row-major [rows, nsplit] as the decode
// workspace stores it, or split-major [nsplit, rows] as gathered from ranks.
struct MergeStrides {
  int64_t o_split, o_row, l_split, l_row;
};

__device__ __forceinline__ float merge_max(const float* lp, int nsplit, int64_t l_split) {
  const int lane = threadIdx.x & 31;
  float M = kNegInf;
  for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, lp[s * l_split]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  return M;
}

// kCPW chunks (of 128 columns with float4 access, else 32) per warp, kBatch
// live splits per round of loads: kCPW * kBatch loads in flight per lane.
template <typename TO, bool kVec4, int kCPW, int kBatch>
__global__ void __launch_bounds__(128, kCPW == 1 ? 8 : 4) splitk_merge_kernel(const float* __restrict__ o_part,
                                                           const float* __restrict__ lse_part,
                                                           TO* __restrict__ o,
                                                           float* __restrict__ lse, int64_t rows,
                                                           int nsplit, int d,
                                                           const MergeStrides st) {
  // one warp per (row, group of kCPW chunks): a wide row's chunks load in
  // parallel; each warp forms the row's weights itself
  constexpr int kCols = kVec4 ? 128 : 32;
  const int groups = (d + kCPW * kCols - 1) / (kCPW * kCols);
  const int64_t wid = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t row = wid / groups;
  const int group = static_cast<int>(wid - row * groups);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* lp = lse_part + row * st.l_row;
  const float M = merge_max(lp, nsplit, st.l_split);
  // sum of exp(lse_s - M)
  float tot = 0.f;
  if (M != kNegInf)
    for (int s = lane; s < nsplit; s += 32) tot += expf(lp[s * st.l_split] - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const float LSE = (M != kNegInf) ? M + logf(tot) : kNegInf;
  const float* op = o_part + row * st.o_row;
  // The splits of weight 0 are neither loaded nor added (their partials may
  // hold anything, or never have been written). The others are taken in
  // batches of up to kBatch, in ascending order, found from a ballot of the
  // weights; each batch's loads are issued before any of them is used, so a
  // row with few live splits costs one round trip to memory.
  using V = typename std::conditional<kVec4, float4, float>::type;
  int c[kCPW];
  bool col[kCPW];
  V acc[kCPW];
#pragma unroll
  for (int i = 0; i < kCPW; ++i) {
    c[i] = (group * kCPW + i) * kCols + (kVec4 ? 4 * lane : lane);
    col[i] = c[i] < d;
    acc[i] = V{};
  }
  for (int s0 = 0; s0 < nsplit; s0 += 32) {
    const int s = s0 + lane;
    const float ls = s < nsplit ? lp[s * st.l_split] : kNegInf;
    const float w = (ls == kNegInf || M == kNegInf) ? 0.f : expf(ls - LSE);
    unsigned live = __ballot_sync(0xffffffffu, w != 0.f);
    while (live != 0u) {
      int idx[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        idx[j] = live != 0u ? __ffs(live) - 1 : -1;  // warp-uniform
        live &= live - 1u;
      }
      float wk[kBatch];
      V v[kBatch][kCPW];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) wk[j] = __shfl_sync(0xffffffffu, w, idx[j] < 0 ? 0 : idx[j]);
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
#pragma unroll
        for (int i = 0; i < kCPW; ++i) {
          v[j][i] = V{};
          if (col[i] && idx[j] >= 0)
            v[j][i] = *reinterpret_cast<const V*>(op + int64_t(s0 + idx[j]) * st.o_split + c[i]);
        }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (idx[j] < 0) continue;
#pragma unroll
        for (int i = 0; i < kCPW; ++i) {
          if constexpr (kVec4) {
            acc[i].x = fmaf(wk[j], v[j][i].x, acc[i].x);
            acc[i].y = fmaf(wk[j], v[j][i].y, acc[i].y);
            acc[i].z = fmaf(wk[j], v[j][i].z, acc[i].z);
            acc[i].w = fmaf(wk[j], v[j][i].w, acc[i].w);
          } else {
            acc[i] = fmaf(wk[j], v[j][i], acc[i]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kCPW; ++i) {
    if (!col[i]) continue;
    TO* orow = o + row * d + c[i];
    if constexpr (kVec4) {
      orow[0] = static_cast<TO>(acc[i].x);
      orow[1] = static_cast<TO>(acc[i].y);
      orow[2] = static_cast<TO>(acc[i].z);
      orow[3] = static_cast<TO>(acc[i].w);
    } else {
      orow[0] = static_cast<TO>(acc[i]);
    }
  }
  if (lane == 0 && group == 0 && lse != nullptr) lse[row] = LSE;
}

template <int D, int GP>
cudaError_t launch_gp(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                      int B, int H, int Hkv, int Sk, float scale, int nsplit, cudaStream_t s,
                      int* status) {
  const size_t smem = sizeof(DecodeSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(decode_partials_kernel<D, GP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t grid = int64_t(B) * Hkv * nsplit;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  decode_partials_kernel<D, GP><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), o_part, lse_part, H, Hkv, Sk, nsplit,
      scale * kLog2e, status);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                     int B, int H, int Hkv, int Sk, float scale, int nsplit, cudaStream_t s,
                     int* status) {
  const int G = H / Hkv;
  if (G <= 4) return launch_gp<D, 4>(q, k, v, o_part, lse_part, B, H, Hkv, Sk, scale, nsplit, s, status);
  if (G <= 8) return launch_gp<D, 8>(q, k, v, o_part, lse_part, B, H, Hkv, Sk, scale, nsplit, s, status);
  return launch_gp<D, 16>(q, k, v, o_part, lse_part, B, H, Hkv, Sk, scale, nsplit, s, status);
}

}  // namespace

cudaError_t launch_decode_partials(const void* q, const void* k, const void* v, float* o_part,
                                   float* lse_part, int B, int H, int Hkv, int Sk, int d,
                                   float scale, int nsplit, cudaStream_t s, int* status) {
  if (d == 128) return launch_d<128>(q, k, v, o_part, lse_part, B, H, Hkv, Sk, scale, nsplit, s, status);
  return launch_d<64>(q, k, v, o_part, lse_part, B, H, Hkv, Sk, scale, nsplit, s, status);
}

cudaError_t launch_splitk_merge_strided(const float* o_part, const float* lse_part, void* o,
                                        float* lse, int64_t rows, int nsplit, int d,
                                        int64_t o_split, int64_t o_row, int64_t l_split,
                                        int64_t l_row, rf_dtype out_dt, cudaStream_t s) {
  const int warps = 4;
  const MergeStrides st{o_split, o_row, l_split, l_row};
  const bool vec = d % 4 == 0 && reinterpret_cast<uintptr_t>(o_part) % 16 == 0 &&
                   o_split % 4 == 0 && o_row % 4 == 0;
  // rows up to 128 columns: one chunk per warp, eight live splits per round;
  // wider rows (float4): four chunks per warp, four live splits per round
  const bool wide = vec && d > 128;
  const int64_t cols = !vec ? 32 : wide ? 512 : 128;   // columns per warp
  const int64_t grid = (rows * ((d + cols - 1) / cols) + warps - 1) / warps;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const unsigned g = static_cast<unsigned>(grid);
  const unsigned t = warps * 32;
  auto run = [&](auto* out) {
    using TO = typename std::remove_pointer<decltype(out)>::type;
    if (wide)
      splitk_merge_kernel<TO, true, 4, 4><<<g, t, 0, s>>>(o_part, lse_part, out, lse, rows, nsplit, d, st);
    else if (vec)
      splitk_merge_kernel<TO, true, 1, 8><<<g, t, 0, s>>>(o_part, lse_part, out, lse, rows, nsplit, d, st);
    else
      splitk_merge_kernel<TO, false, 1, 8><<<g, t, 0, s>>>(o_part, lse_part, out, lse, rows, nsplit, d, st);
  };
  if (out_dt == RF_F32)
    run(static_cast<float*>(o));
  else
    run(static_cast<__nv_bfloat16*>(o));
  return cudaGetLastError();
}

cudaError_t launch_splitk_merge(const float* o_part, const float* lse_part, void* o, float* lse,
                                int64_t rows, int nsplit, int d, rf_dtype out_dt, cudaStream_t s) {
  return launch_splitk_merge_strided(o_part, lse_part, o, lse, rows, nsplit, d, d,
                                     int64_t(nsplit) * d, 1, nsplit, out_dt, s);
}

}  // namespace rf
