// attn_simt.cu -- exact float32 attention forward, one warp per query row.
//
// The same single-pass cascade as the tensor-core kernel (running max m,
// running sum l and accumulator acc per row, rescaled by exp(m_old - m_new)
// at each key tile; RedFuser, section 2, incremental computation; FLASHLIGHT,
// Metodologia item 3), in plain float32 FFMA arithmetic so that float32
// inputs keep float32 accuracy (no TF32 rounding anywhere).
//
// Shape of the kernel (STOF, Méthodologie, row-wise kernel): the query is
// split by rows, one warp owns one row, the reductions are warp shuffles and
// no inter-warp synchronisation enters the arithmetic. The eight warps of a
// CTA share K/V sub-tiles of 32 * KPL keys staged in shared memory (KPL = 4,
// 2, 1 keys per lane for d <= 64, 128, 256, so one staging round covers a
// whole 128-key mask tile at d <= 64). Each lane scores its KPL keys as KPL
// independent dot products (16-byte reads of K rows padded to d + 4 floats:
// conflict-free); the warp's probabilities go to shared memory and each lane
// accumulates its output columns from them with two partial sums. Masked
// 128 x 128 tiles are skipped entirely: the CTA walks the same tile list
// (dense range, causal range, or block-sparse row) the tensor-core kernel
// walks; inside a partial tile of a two-level mask each key's bit in its
// 8 x 8 inner block decides (STOF, two-level storage format).
#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kRows = 8;       // query rows (warps) per CTA
constexpr int kTile = 128;     // mask tile side

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

// Shared-memory floats for head dimension d and KPL keys per lane.
__host__ __device__ constexpr int simt_smem_floats(int d, int kpl) {
  return 32 * kpl * (d + 4)      // K sub-tile, rows padded
         + 32 * kpl * d          // V sub-tile
         + kRows * d             // the CTA's query rows
         + kRows * 32 * kpl;     // each warp's probabilities
}

// DCH = ceil(d / 32): output columns owned by each lane (lane + 32 t).
// KPL: keys per lane in a sub-tile of 32 * KPL keys.
// 16-byte asynchronous global -> shared copy; with `in` false nothing is
// read and the 16 bytes are zero-filled. And the wait for all of this
// thread's copies (a hardware wait, not a spin loop).
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool in) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(in ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

template <int DCH, int KPL>
__global__ void __launch_bounds__(kRows * 32) attn_simt_f32_kernel(const AttnArgs a) {
  constexpr int kSub = 32 * KPL;
  extern __shared__ float smem[];
  const int d = a.d, dk = a.d + 4;
  float* Ks = smem;                 // [kSub][d + 4]
  float* Vs = Ks + kSub * dk;       // [kSub][d]
  float* Qs = Vs + kSub * d;        // [kRows][d]
  float* Ps = Qs + kRows * d;       // [kRows][kSub]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrb = (a.Sq + kRows - 1) / kRows;
  const int rb = blockIdx.x % nrb;
  const int bh = blockIdx.x / nrb;
  const int b = bh / a.H, h = bh % a.H;
  const int hk = h / (a.H / a.Hkv);
  const int r0 = rb * kRows, r1 = min(a.Sq, r0 + kRows);
  const int i = r0 + warp;
  const bool row_ok = i < a.Sq;
  const float* qg = static_cast<const float*>(a.q) + (int64_t(bh) * a.Sq + i) * d;
  const float* kg = static_cast<const float*>(a.k) + int64_t(b * a.Hkv + hk) * a.Sk * d;
  const float* vg = static_cast<const float*>(a.v) + int64_t(b * a.Hkv + hk) * a.Sk * d;
  float* pw = Ps + warp * kSub;

  // the query row by asynchronous copies too: the first sub-tile's wait
  // covers it, so Q, K and V cost one round trip
  if (row_ok)
    for (int c = 4 * lane; c < d; c += 128) cp_async16_zfill(Qs + warp * d + c, qg + c, true);

  // keys visible to the CTA's last row bound every tile it may touch
  const int64_t shift = int64_t(a.Sk) - a.Sq;  // bottom-right causal alignment
  const int64_t kend = a.causal ? min64(a.Sk, int64_t(r1) + shift) : a.Sk;
  const int64_t row_kend = a.causal ? min64(a.Sk, int64_t(i) + 1 + shift) : a.Sk;
  const int qt = r0 / kTile;
  int beg = 0, end = 0;
  const int32_t* cols = nullptr;
  if (a.row_ptr != nullptr) {
    const int32_t* rp = a.row_ptr + (a.per_head ? int64_t(bh) * a.nqt : 0) + qt;
    beg = rp[0];
    end = rp[1];
    cols = a.col_idx;
  } else {
    end = kend > 0 ? static_cast<int>((kend + kTile - 1) / kTile) : 0;
  }

  float m = kNegInf, l = 0.f;
  float acc[DCH];
#pragma unroll
  for (int t = 0; t < DCH; ++t) acc[t] = 0.f;

  int prev = -1;
  for (int n = beg; n < end; ++n) {
    int kt = n;
    if (cols != nullptr) {
      kt = cols[n];
      if (kt < 0 || kt >= a.nkt || kt <= prev) {  // malformed list: record and stop
        if (threadIdx.x == 0) record_status(a.status, dev_code(kDevBadList, kKerAttnSimt, 1));
        break;
      }
      prev = kt;
    }
    if (int64_t(kt) * kTile >= kend) break;  // beyond every causal row: ascending list ends
    if (a.visited != nullptr && threadIdx.x == 0)
      a.visited[(int64_t(bh) * a.nqt + qt) * a.nkt + kt] = 1;
    // a partial tile of a two-level mask: its inner 8 x 8 bitmaps decide
    const int pb = (cols != nullptr && a.tile_bits != nullptr) ? a.tile_bits[n] : -1;
    for (int sub = 0; sub < kTile / kSub; ++sub) {
      const int k0 = kt * kTile + sub * kSub;
      if (k0 >= kend) break;
      __syncthreads();  // the previous sub-tile is consumed
      // K and V rows by asynchronous 16-byte copies, all of a thread's in
      // flight at once (keys past Sk are filled with zeros)
      const int d4 = d / 4;
      for (int e = threadIdx.x; e < kSub * d4; e += kRows * 32) {
        const int r = e / d4, c = (e % d4) * 4;
        const int key = k0 + r;
        const bool in = key < a.Sk;
        const int64_t off = in ? int64_t(key) * d + c : 0;
        cp_async16_zfill(Ks + r * dk + c, kg + off, in);
        cp_async16_zfill(Vs + r * d + c, vg + off, in);
      }
      cp_async_wait_all();
      __syncthreads();
      if (!row_ok) continue;
      // scores of this row against keys k0 + lane + 32 j, j < KPL
      float s[KPL];
      bool vis[KPL];
#pragma unroll
      for (int j = 0; j < KPL; ++j) {
        const int key = k0 + lane + 32 * j;
        vis[j] = key < row_kend;
        if (vis[j] && pb >= 0) {
          const int rr = i - qt * kTile, cc = key - kt * kTile;
          const uint64_t w = a.bits[int64_t(pb) * 256 + (rr >> 3) * (kTile / 8) + (cc >> 3)];
          vis[j] = (w >> ((rr & 7) * 8 + (cc & 7))) & 1;
        }
        s[j] = 0.f;
      }
      const float* qr = Qs + warp * d;
      for (int c = 0; c < d; c += 4) {
        const float4 q4 = *reinterpret_cast<const float4*>(qr + c);
#pragma unroll
        for (int j = 0; j < KPL; ++j) {
          const float4 k4 = *reinterpret_cast<const float4*>(Ks + (lane + 32 * j) * dk + c);
          s[j] = fmaf(q4.x, k4.x, s[j]);
          s[j] = fmaf(q4.y, k4.y, s[j]);
          s[j] = fmaf(q4.z, k4.z, s[j]);
          s[j] = fmaf(q4.w, k4.w, s[j]);
        }
      }
      float smax = kNegInf;
#pragma unroll
      for (int j = 0; j < KPL; ++j) {
        s[j] = vis[j] ? s[j] * a.scale : kNegInf;
        smax = fmaxf(smax, s[j]);
      }
      // online update: m' = max(m, max s); alpha = exp(m - m'); p = exp(s - m')
      const float mn = fmaxf(m, warp_max(smax));
      if (mn == kNegInf) continue;  // nothing visible to this row yet
      const float alpha = (m == kNegInf) ? 0.f : expf(m - mn);
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < KPL; ++j) {
        const float pj = (s[j] == kNegInf) ? 0.f : expf(s[j] - mn);
        pw[lane + 32 * j] = pj;
        psum += pj;
      }
      l = l * alpha + warp_sum(psum);
      __syncwarp();
#pragma unroll
      for (int t = 0; t < DCH; ++t) {
        const int c = lane + 32 * t;
        if (c < d) {
          float a0 = 0.f, a1 = 0.f;
          for (int k = 0; k < kSub; k += 2) {
            a0 = fmaf(pw[k], Vs[k * d + c], a0);
            a1 = fmaf(pw[k + 1], Vs[(k + 1) * d + c], a1);
          }
          acc[t] = acc[t] * alpha + (a0 + a1);
        }
      }
      __syncwarp();  // pw is rewritten by the next sub-tile
      m = mn;
    }
  }
  cp_async_wait_all();  // a row with no visible tile still issued its Q copies
  if (!row_ok) return;
  float* og = static_cast<float*>(a.o) + (int64_t(bh) * a.Sq + i) * d;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int t = 0; t < DCH; ++t) {
    const int c = lane + 32 * t;
    if (c < d) og[c] = acc[t] * inv;
  }
  if (lane == 0 && a.lse != nullptr)
    a.lse[int64_t(bh) * a.Sq + i] = l > 0.f ? m + logf(l) : kNegInf;
}

// O = 0 and lse = -inf everywhere (no keys at all).
__global__ void attn_fill_empty(uint32_t* o_words, int64_t n_words, float* lse, int64_t nrows) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n_words; e += stride)
    o_words[e] = 0u;
  if (lse != nullptr)
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < nrows; e += stride)
      lse[e] = kNegInf;
}

template <int DCH, int KPL>
cudaError_t launch_dch(const AttnArgs& a, cudaStream_t s) {
  const size_t smem = size_t(simt_smem_floats(a.d, KPL)) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(attn_simt_f32_kernel<DCH, KPL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t nrb = (a.Sq + kRows - 1) / kRows;
  const int64_t grid = nrb * a.B * a.H;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  attn_simt_f32_kernel<DCH, KPL><<<static_cast<unsigned>(grid), kRows * 32, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_empty(const AttnArgs& a, size_t elem_bytes, cudaStream_t s) {
  const int64_t rows = int64_t(a.B) * a.H * a.Sq;
  const int64_t words = rows * a.d * static_cast<int64_t>(elem_bytes) / 4;
  attn_fill_empty<<<1184, 256, 0, s>>>(static_cast<uint32_t*>(a.o), words, a.lse, rows);
  return cudaGetLastError();
}

cudaError_t launch_attn_simt_f32(const AttnArgs& a, cudaStream_t s) {
  if (a.Sk == 0) return launch_attn_empty(a, sizeof(float), s);
  switch ((a.d + 31) / 32) {
    case 1: return launch_dch<1, 4>(a, s);
    case 2: return launch_dch<2, 4>(a, s);
    case 3: return launch_dch<3, 2>(a, s);
    case 4: return launch_dch<4, 2>(a, s);
    case 5: return launch_dch<5, 1>(a, s);
    case 6: return launch_dch<6, 1>(a, s);
    case 7: return launch_dch<7, 1>(a, s);
    default: return launch_dch<8, 1>(a, s);
  }
}

}  // namespace rf
