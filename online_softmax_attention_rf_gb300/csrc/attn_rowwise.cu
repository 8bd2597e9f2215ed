// attn_rowwise.cu -- STOF's row-wise attention kernel (one warp per query row).
//
// Accelerating Sparse Transformer Inference on GPU (STOF), Méthodologie,
// unified MHA module, dual-kernel strategy: for highly sparse masks and short
// sequences, Q is split into rows, each row is reduced with warp-level
// shuffles and no synchronisation between warps is needed. Here a warp owns
// one query row and visits only its visible keys: the listed outer tiles of
// its query tile (all of a full tile's keys, the set bits of a partial
// tile's 8 x 8 inner bitmaps, and the causal limit), 32 keys at a time. Lane
// i scores the batch's i-th key against the query row (kept in shared memory
// and read by broadcast), so scores need no reduction; the batch maximum and
// sum take one warp reduction each, and the lanes, which own D/32 head
// dimensions of the accumulator, add the batch's value rows with
// shuffle-broadcast weights -- the incremental update of (m, l, acc)
// (RedFuser, section 2: O(1) state per row, rescaled by exp(m_old - m_new)).
// Everything is float32 (bf16 inputs are widened exactly), with exp2/log2 and
// the scale times log2 e folded into q.
#include "rf_device.cuh"

namespace rf {
namespace {

// query rows per CTA (all in one 128-row tile); each warp stages 32 key and
// 32 value rows (8 to 32 KB), so small CTAs keep several per SM
constexpr int kRowWarps = 4;

template <typename T, int DPL>
struct Vec;
template <>
struct Vec<__nv_bfloat16, 2> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[2]) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    v[0] = __uint_as_float(w << 16);
    v[1] = __uint_as_float(w & 0xffff0000u);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[2]) {
    *reinterpret_cast<uint32_t*>(p) = pack_bf16x2(v[0], v[1]);
  }
};
template <>
struct Vec<__nv_bfloat16, 4> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[4]) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(w.x << 16);
    v[1] = __uint_as_float(w.x & 0xffff0000u);
    v[2] = __uint_as_float(w.y << 16);
    v[3] = __uint_as_float(w.y & 0xffff0000u);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[4]) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
  }
};
template <>
struct Vec<float, 2> {
  static __device__ __forceinline__ void load(const float* p, float (&v)[2]) {
    const float2 w = *reinterpret_cast<const float2*>(p);
    v[0] = w.x;
    v[1] = w.y;
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[2]) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
  }
};
template <>
struct Vec<float, 4> {
  static __device__ __forceinline__ void load(const float* p, float (&v)[4]) {
    const float4 w = *reinterpret_cast<const float4*>(p);
    v[0] = w.x;
    v[1] = w.y;
    v[2] = w.z;
    v[3] = w.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};

struct RowParams {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, Hkv, Sq, Sk;
  float scale_log2;
  int causal;
  const int32_t* row_ptr;  // nullptr: dense (every key tile listed)
  const int32_t* col_idx;
  const int32_t* tile_bits;
  const uint64_t* bits;
  int per_head, nqt, nkt;
};

// State of one row: running max m (log2 units), sum l, accumulator slice.
template <int DPL>
struct RowState {
  float m, l, acc[DPL];
};

// Rows of the batch's keys and values are staged in shared memory as 16-byte
// units; unit c of row r is stored at position c ^ (r & 7) of the row, so
// that the units one instruction touches fall in distinct bank groups.
__device__ __forceinline__ int swz(int r, int c) { return c ^ (r & 7); }

// 16-byte asynchronous global -> shared copy (L1-cached) and the wait for
// all of this thread's copies (a hardware wait, not a spin loop).
__device__ __forceinline__ void cp_async_ca16(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

// Dot product of the (scaled) query row (shared memory, read by broadcast)
// with staged key row r.
__device__ __forceinline__ float dot_row(const float* qs, const __nv_bfloat16* ks, int r, int D) {
  float s0 = 0.f, s1 = 0.f;
  const uint4* k4 = reinterpret_cast<const uint4*>(ks + r * D);
#pragma unroll 4
  for (int c = 0; c < D / 8; ++c) {
    const uint4 w = k4[swz(r, c)];
    const float4 qa = reinterpret_cast<const float4*>(qs)[2 * c];
    const float4 qb = reinterpret_cast<const float4*>(qs)[2 * c + 1];
    s0 = fmaf(qa.x, __uint_as_float(w.x << 16), s0);
    s1 = fmaf(qa.y, __uint_as_float(w.x & 0xffff0000u), s1);
    s0 = fmaf(qa.z, __uint_as_float(w.y << 16), s0);
    s1 = fmaf(qa.w, __uint_as_float(w.y & 0xffff0000u), s1);
    s0 = fmaf(qb.x, __uint_as_float(w.z << 16), s0);
    s1 = fmaf(qb.y, __uint_as_float(w.z & 0xffff0000u), s1);
    s0 = fmaf(qb.z, __uint_as_float(w.w << 16), s0);
    s1 = fmaf(qb.w, __uint_as_float(w.w & 0xffff0000u), s1);
  }
  return s0 + s1;
}
__device__ __forceinline__ float dot_row(const float* qs, const float* ks, int r, int D) {
  float s0 = 0.f, s1 = 0.f;
  const float4* k4 = reinterpret_cast<const float4*>(ks + r * D);
#pragma unroll 4
  for (int c = 0; c < D / 4; ++c) {
    const float4 w = k4[swz(r, c)];
    const float4 qa = reinterpret_cast<const float4*>(qs)[c];
    s0 = fmaf(qa.x, w.x, s0);
    s1 = fmaf(qa.y, w.y, s1);
    s0 = fmaf(qa.z, w.z, s0);
    s1 = fmaf(qa.w, w.w, s1);
  }
  return s0 + s1;
}

// One batch of n <= 32 keys, lane i holding key i. The warp copies the key
// and value rows into its shared buffers whole lines at a time (kUnits / 32
// rows per instruction), then each lane scores its own key (no reduction),
// the batch maximum and sum take one warp reduction each, and the lanes'
// accumulator slices add the value rows one key at a time.
template <typename T, int DPL>
__device__ __forceinline__ void run_batch(const float* qs, const T* kb, const T* vb, int lane,
                                          int my_key, int n, RowState<DPL>& st, T* ksm, T* vsm) {
  constexpr int D = 32 * DPL;
  constexpr int kPer = 16 / sizeof(T);       // elements per 16-byte unit
  constexpr int kUnits = D / kPer;           // units per row (8, 16 or 32)
  constexpr int kRowsPer = 32 / kUnits;      // rows per copy instruction
  const int c = lane % kUnits;
#pragma unroll 4
  for (int r0 = 0; r0 < 32; r0 += kRowsPer) {
    const int r = r0 + lane / kUnits;
    const int key = __shfl_sync(0xffffffffu, my_key, r);
    if (r < n) {
      const int64_t off = int64_t(key) * D + c * kPer;
      cp_async_ca16(ksm + r * D + swz(r, c) * kPer, kb + off);
      cp_async_ca16(vsm + r * D + swz(r, c) * kPer, vb + off);
    }
  }
  cp_async_wait_all();
  __syncwarp();
  const bool valid = lane < n;
  const float s = valid ? dot_row(qs, ksm, lane, D) : kNegInf;
  float mb = s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
  const float m_new = fmaxf(st.m, mb);
  const float alpha = st.m == kNegInf ? 0.f : exp2f(st.m - m_new);
  const float p = valid ? exp2f(s - m_new) : 0.f;
  float ps = p;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
  st.l = st.l * alpha + ps;
#pragma unroll
  for (int e = 0; e < DPL; ++e) st.acc[e] *= alpha;
  // lane l's DPL elements of row i: unit (l * DPL) / kPer, offset within it
  const int my_unit = (lane * DPL) / kPer, my_off = (lane * DPL) % kPer;
#pragma unroll 4
  for (int i = 0; i < n; ++i) {
    const float pi = __shfl_sync(0xffffffffu, p, i);
    float vv[DPL];
    Vec<T, DPL>::load(vsm + i * D + swz(i, my_unit) * kPer + my_off, vv);
#pragma unroll
    for (int e = 0; e < DPL; ++e) st.acc[e] = fmaf(pi, vv[e], st.acc[e]);
  }
  __syncwarp();  // the buffers are refilled by the next batch
  st.m = m_new;
}

// Appends the keys base + (set bits of `bits`) to the pending batch (lane i
// takes the i-th), running the batch whenever it fills. Lane l owns bit l:
// a set bit of rank j goes to batch slot nk + j through the warp's slots in
// shared memory.
template <typename T, int DPL>
__device__ __forceinline__ void take_keys(uint32_t bits, int base, const float* qs, const T* kb,
                                          const T* vb, int lane, int* slots, int& my_key, int& nk,
                                          RowState<DPL>& st, T* ksm, T* vsm) {
  while (bits != 0u) {
    const int cnt = __popc(bits);
    const int take = min(cnt, 32 - nk);
    const bool mine = (bits >> lane) & 1u;
    const int rank = __popc(bits & ((1u << lane) - 1u));
    if (mine && rank < take) slots[nk + rank] = base + lane;
    __syncwarp();
    if (lane >= nk && lane < nk + take) my_key = slots[lane];
    __syncwarp();  // the slots are rewritten by the next word
    nk += take;
    bits = __ballot_sync(0xffffffffu, mine && rank >= take);
    if (nk == 32) {
      run_batch<T, DPL>(qs, kb, vb, lane, my_key, 32, st, ksm, vsm);
      nk = 0;
    }
  }
}

template <typename T, int DPL>
__global__ void __launch_bounds__(32 * kRowWarps) attn_rowwise_kernel(const RowParams p) {
  constexpr int D = 32 * DPL;
  __shared__ __align__(16) float q_sh[kRowWarps][D];
  __shared__ int slot_sh[kRowWarps][32];
  extern __shared__ __align__(16) unsigned char kvbuf_raw[];  // [warps][2][32][D] of T
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nrb = (p.Sq + kRowWarps - 1) / kRowWarps;
  const int bh = static_cast<int>(blockIdx.x / nrb);
  const int row = static_cast<int>(blockIdx.x % nrb) * kRowWarps + wid;
  if (row >= p.Sq) return;  // whole warps leave together; no CTA-wide barrier follows
  const int b = bh / p.H, h = bh % p.H;
  const int bk = b * p.Hkv + h / (p.H / p.Hkv);
  const T* qr = static_cast<const T*>(p.q) + (int64_t(bh) * p.Sq + row) * D;
  const T* kb = static_cast<const T*>(p.k) + int64_t(bk) * p.Sk * D;
  const T* vb = static_cast<const T*>(p.v) + int64_t(bk) * p.Sk * D;
  float* qs = q_sh[wid];
  T* ksm = reinterpret_cast<T*>(kvbuf_raw) + wid * 2 * 32 * D;
  T* vsm = ksm + 32 * D;
  {
    float qv[DPL];
    Vec<T, DPL>::load(qr + lane * DPL, qv);
#pragma unroll
    for (int e = 0; e < DPL; ++e) qs[lane * DPL + e] = qv[e] * p.scale_log2;
    __syncwarp();
  }
  RowState<DPL> st;
  st.m = kNegInf;
  st.l = 0.f;
#pragma unroll
  for (int e = 0; e < DPL; ++e) st.acc[e] = 0.f;

  const int row_lim = p.causal ? min(p.Sk, row + 1 + (p.Sk - p.Sq)) : p.Sk;
  const int qt = row / 128, r = row % 128;
  int n0 = 0, n1 = p.nkt;  // list entries of this query tile
  const int32_t* cols = nullptr;
  const int32_t* tbits = nullptr;
  if (p.row_ptr != nullptr) {
    const int64_t li = (p.per_head ? int64_t(bh) * p.nqt : 0) + qt;
    n0 = p.row_ptr[li];
    n1 = p.row_ptr[li + 1];
    cols = p.col_idx;
    tbits = p.tile_bits;
  }
  int my_key = 0;  // lane i: the i-th key of the pending batch
  int nk = 0;
  for (int n = n0; n < n1; ++n) {
    const int u = cols != nullptr ? cols[n] : n;
    const int k0 = u * 128;
    if (k0 >= row_lim) {
      if (cols == nullptr) break;  // a dense range is ascending
      continue;
    }
    const int lim = min(128, row_lim - k0);
    // this row's 128 key bits of tile u (bit c of word c / 32 = key k0 + c)
    auto lim_word = [&](int c0) -> uint32_t {
      return lim >= c0 + 32 ? ~0u : (lim > c0 ? (1u << (lim - c0)) - 1u : 0u);
    };
    uint32_t w0 = lim_word(0), w1 = lim_word(32), w2 = lim_word(64), w3 = lim_word(96);
    const int pb = tbits != nullptr ? tbits[n] : -1;
    if (pb >= 0) {
      // one byte of each of the 16 inner 8 x 8 blocks this row crosses:
      // lane c < 16 loads block c's byte, groups of four lanes OR their
      // bytes into one word, and the four words are broadcast
      const uint8_t* rb =
          reinterpret_cast<const uint8_t*>(p.bits + int64_t(pb) * 256 + (r >> 3) * 16) + (r & 7);
      uint32_t part = lane < 16 ? uint32_t(rb[lane * 8]) << (8 * (lane & 3)) : 0u;
      part |= __shfl_xor_sync(0xffffffffu, part, 1);
      part |= __shfl_xor_sync(0xffffffffu, part, 2);
      w0 &= __shfl_sync(0xffffffffu, part, 0);
      w1 &= __shfl_sync(0xffffffffu, part, 4);
      w2 &= __shfl_sync(0xffffffffu, part, 8);
      w3 &= __shfl_sync(0xffffffffu, part, 12);
    }
    // visible keys in ascending order, batched
    take_keys<T, DPL>(w0, k0, qs, kb, vb, lane, slot_sh[wid], my_key, nk, st, ksm, vsm);
    take_keys<T, DPL>(w1, k0 + 32, qs, kb, vb, lane, slot_sh[wid], my_key, nk, st, ksm, vsm);
    take_keys<T, DPL>(w2, k0 + 64, qs, kb, vb, lane, slot_sh[wid], my_key, nk, st, ksm, vsm);
    take_keys<T, DPL>(w3, k0 + 96, qs, kb, vb, lane, slot_sh[wid], my_key, nk, st, ksm, vsm);
  }
  if (nk > 0) run_batch<T, DPL>(qs, kb, vb, lane, my_key, nk, st, ksm, vsm);

  float out[DPL];
  const float inv = st.l > 0.f ? 1.f / st.l : 0.f;
#pragma unroll
  for (int e = 0; e < DPL; ++e) out[e] = st.acc[e] * inv;
  T* orow = static_cast<T*>(p.o) + (int64_t(bh) * p.Sq + row) * D;
  Vec<T, DPL>::store(orow + lane * DPL, out);
  if (p.lse != nullptr && lane == 0)
    p.lse[int64_t(bh) * p.Sq + row] = st.l > 0.f ? (st.m + log2f(st.l)) * kLn2 : kNegInf;
}

template <typename T, int DPL>
cudaError_t launch_t(const RowParams& p, cudaStream_t s) {
  const int64_t nrb = (p.Sq + kRowWarps - 1) / kRowWarps;
  const int64_t grid = nrb * p.B * p.H;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int smem = kRowWarps * 2 * 32 * 32 * DPL * static_cast<int>(sizeof(T));
  if (smem > 40 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(attn_rowwise_kernel<T, DPL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  attn_rowwise_kernel<T, DPL><<<static_cast<unsigned>(grid), 32 * kRowWarps, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_rowwise(const AttnArgs& a, rf_dtype dt, cudaStream_t s) {
  RowParams p{};
  p.q = a.q;
  p.k = a.k;
  p.v = a.v;
  p.o = a.o;
  p.lse = a.lse;
  p.B = a.B;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.scale_log2 = a.scale * kLog2e;
  p.causal = a.causal;
  p.row_ptr = a.row_ptr;
  p.col_idx = a.col_idx;
  p.tile_bits = a.tile_bits;
  p.bits = a.bits;
  p.per_head = a.per_head;
  p.nqt = a.nqt;
  p.nkt = a.nkt;
  const bool f32 = dt == RF_F32;
  if (a.d == 64)
    return f32 ? launch_t<float, 2>(p, s) : launch_t<__nv_bfloat16, 2>(p, s);
  return f32 ? launch_t<float, 4>(p, s) : launch_t<__nv_bfloat16, 4>(p, s);
}

}  // namespace rf
