// mla_decode.cu -- multi-head latent attention (MLA) decode on the tcgen05
// tensor cores, split over the key sequence and merged by log-sum-exp.
//
// RedFuser: An Automatic Operator Fusion Framework for Cascaded Reductions on
// AI Accelerators -- technical summary, section 4 (MLA is one of the
// evaluated workloads; the generated kernel is compared with FlashMLA) and
// section 3 (multi-segment strategy: each segment keeps the O(1) state
// (m, l, acc) of the incremental form, the segments merge by log-sum-exp).
//
// The absorbed decode form: every batch element has one latent key-value head
// kv [Sk, 576] (512 latent columns + 64 rotary ones) shared by the 128 query
// heads q [128, 576] of its single query token; scores s = scale q . kv, and
// the values are the latent columns, v = kv[:, :512]. Per (batch, split, half)
// one CTA:
//   tensor memory: O_half [128 heads x 256 value columns] f32, two score tiles
//     S [128 x 32 keys] f32, two P tiles [128 x 32] bf16 (352 of 512 columns;
//     the full 128 x 512 accumulator alone would fill tensor memory, so the
//     two halves of the value columns go to two CTAs, each forming the
//     scores itself);
//   shared memory: q [128 x 576] (144 KB, loaded once) and a 2-stage ring of
//     32-key kv tiles (36 KB each), all 128-byte swizzled, K-major;
//   S_b = q kv_tile^T (36 MMAs, K = 576), the softmax (one thread per head,
//     TMEM lane = head) forms P_b, then O_half += P_b V_half (two TS-MMAs,
//     P from tensor memory, V the tile's latent columns read as an MN-major
//     operand); the next tile's scores are computed while the softmax works.
// The partial (O, LSE) of a split is written in the split-K workspace layout
// and merged by the split-K merge kernel. Every wait is bounded.
#include <cudaTypedefs.h>

#include <mutex>

#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kMH = 128;        // query heads (rows of every tile)
constexpr int kMD = 576;        // key dimension (latent + rotary)
constexpr int kMV = 512;        // value dimension (latent)
constexpr int kMVH = 256;       // value columns per CTA
constexpr int kMN = 32;         // keys per tile
constexpr int kMChunks = kMD / 64;             // 64-column swizzle chunks of a row
constexpr int kQChunk = kMH * 128;             // 16 KB: one chunk of q
constexpr int kKVChunk = kMN * 128;            // 4 KB: one chunk of a kv tile
constexpr int kKVTile = kMChunks * kKVChunk;   // 36 KB
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kMChunks * kQChunk;
constexpr int kOffBar = kOffKV + 2 * kKVTile;
constexpr int kMSmem = kOffBar + 256 + 1024;   // + alignment slack
constexpr int kMThreads = 192;  // warps 0-3 softmax, 4 producer + TMEM, 5 MMA issuer
constexpr int kWarpProd = 4;
constexpr int kWarpMma = 5;
// tensor-memory columns
constexpr uint32_t kTmO = 0;
constexpr uint32_t kTmS = kMVH;                // S_b at kTmS + 32 b
constexpr uint32_t kTmP = kMVH + 2 * kMN;      // P_b at kTmP + 16 b
constexpr float kRescale = 8.0f;               // log2 units (stale max kept below)

struct MBars {
  uint64_t q_full;
  uint64_t kv_full[2];
  uint64_t kv_empty[2];
  uint64_t s_full[2];   // S_b holds the scores of the tile using buffer b
  uint64_t p_full[2];   // P_b written by the four softmax warps
  uint64_t pv_done;     // the latest P.V has completed
  uint64_t o_done;
  uint64_t mma_idle;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(MBars) <= 256, "MLA barriers exceed their block");

struct MParams {
  int B, Sk, nsplit;
  float scale_log2;
  float* o_part;    // [B * 128, nsplit, 512]
  float* lse_part;  // [B * 128, nsplit]
  int* status;
};

// Store 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0],"
      " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// S = q tile^T: 36 K steps of 16 (four per 64-column chunk, 32 bytes apart).
__device__ __forceinline__ void issue_scores(uint32_t tm_s, uint32_t q_base, uint32_t kv_base) {
  constexpr uint32_t idesc = idesc_bf16_f32(kMH, kMN, 0);
#pragma unroll
  for (int kk = 0; kk < kMD / 16; ++kk) {
    const uint32_t qa = q_base + (kk >> 2) * kQChunk + (kk & 3) * 32;
    const uint32_t ka = kv_base + (kk >> 2) * kKVChunk + (kk & 3) * 32;
    mma_bf16(tm_s, sdesc_sw128(qa, 16, 1024), sdesc_sw128(ka, 16, 1024), idesc,
             kk > 0 ? 1u : 0u);
  }
}

// O_half (+)= P V_half: A = P from tensor memory (8 columns per 16 keys), B =
// the tile's value columns [256 half, +256) as an MN-major operand (64-column
// chunks kKVChunk apart, 8-key groups 1024 bytes apart).
__device__ __forceinline__ void issue_values(uint32_t tm_o, uint32_t tm_p, uint32_t kv_base,
                                             int half, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kMH, kMVH, 1);
  const uint32_t vb = kv_base + half * 4 * kKVChunk;
#pragma unroll
  for (int kk = 0; kk < kMN / 16; ++kk)
    mma_bf16_ts(tm_o, tm_p + kk * 8, sdesc_sw128(vb + kk * 16 * 128, kKVChunk, 1024), idesc,
                (kk > 0 || accumulate) ? 1u : 0u);
}

__global__ void __launch_bounds__(kMThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_kv, const MParams p) {
  extern __shared__ unsigned char msmem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(msmem_raw) + 1023) & ~uintptr_t(1023));
  MBars& bar = *reinterpret_cast<MBars*>(smem + kOffBar);
  const uint32_t s_base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA -> (batch, split, value half)
  const int half = static_cast<int>(blockIdx.x & 1);
  const int split = static_cast<int>((blockIdx.x >> 1) % p.nsplit);
  const int b = static_cast<int>((blockIdx.x >> 1) / p.nsplit);
  const int per = p.Sk / p.nsplit;
  const int key0 = split * per;
  const int key1 = (split == p.nsplit - 1) ? p.Sk : key0 + per;
  const int ntiles = (key1 - key0 + kMN - 1) / kMN;

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.kv_full[i], 1);
      mbar_init(&bar.kv_empty[i], 1);
      mbar_init(&bar.s_full[i], 1);
      mbar_init(&bar.p_full[i], 4);
    }
    mbar_init(&bar.pv_done, 1);
    mbar_init(&bar.o_done, 1);
    mbar_init(&bar.mma_idle, 1);
    bar.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpProd) {
    tmem_alloc(&bar.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bar.tmem_base;
  volatile int* abort_flag = &bar.abort_flag;

  if (warp == kWarpProd) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_kv);
      mbar_arrive_expect_tx(&bar.q_full, kMChunks * kQChunk);
      for (int c = 0; c < kMChunks; ++c)
        tma_load_3d(smem + kOffQ + c * kQChunk, &tm_q, &bar.q_full, c * 64, 0, b);
      bool ok = true;
      int j = 0;
      for (; ok && j < ntiles; ++j) {
        const int s = j & 1;
        if (j >= 2)
          ok = mbar_wait(&bar.kv_empty[s], ((j >> 1) - 1) & 1, p.status,
                         dev_code(kDevTimeout, kKerMla, 1), abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bar.kv_full[s], kKVTile);
        for (int c = 0; c < kMChunks; ++c)
          tma_load_3d(smem + kOffKV + s * kKVTile + c * kKVChunk, &tm_kv, &bar.kv_full[s], c * 64,
                      key0 + j * kMN, b);
      }
      // never leave with copies in flight
      mbar_wait(&bar.q_full, 0, p.status, dev_code(kDevTimeout, kKerMla, 2), nullptr);
      for (int i = max(0, j - 2); i < j; ++i)
        mbar_wait(&bar.kv_full[i & 1], (i >> 1) & 1, p.status, dev_code(kDevTimeout, kKerMla, 2),
                  nullptr);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t q_base = s_base + kOffQ;
      bool ok = mbar_wait(&bar.q_full, 0, p.status, dev_code(kDevTimeout, kKerMla, 3), abort_flag);
      bool issued = false;
      // scores of tile 0
      if (ok && (ok = mbar_wait(&bar.kv_full[0], 0, p.status, dev_code(kDevTimeout, kKerMla, 4),
                                abort_flag))) {
        tc_fence_after_sync();
        issue_scores(tmem + kTmS, q_base, s_base + kOffKV);
        mma_commit(&bar.s_full[0]);
        issued = true;
      }
      for (int j = 0; ok && j < ntiles; ++j) {
        const int s = j & 1, s1 = (j + 1) & 1;
        // the next tile's scores (its S buffer was read by softmax j - 1,
        // whose P.V was issued in the previous iteration)
        if (j + 1 < ntiles) {
          if (!(ok = mbar_wait(&bar.kv_full[s1], ((j + 1) >> 1) & 1, p.status,
                               dev_code(kDevTimeout, kKerMla, 4), abort_flag)))
            break;
          tc_fence_after_sync();
          issue_scores(tmem + kTmS + s1 * kMN, q_base, s_base + kOffKV + s1 * kKVTile);
          mma_commit(&bar.s_full[s1]);
        }
        // P_j is in tensor memory
        if (!(ok = mbar_wait(&bar.p_full[s], (j >> 1) & 1, p.status,
                             dev_code(kDevTimeout, kKerMla, 5), abort_flag)))
          break;
        tc_fence_after_sync();
        issue_values(tmem + kTmO, tmem + kTmP + s * 16, s_base + kOffKV + s * kKVTile, half,
                     j > 0);
        mma_commit(&bar.kv_empty[s]);
        mma_commit(&bar.pv_done);
      }
      if (ok) mma_commit(&bar.o_done);
      // never leave with MMAs in flight
      if (issued) {
        mma_commit(&bar.mma_idle);
        mbar_wait(&bar.mma_idle, 0, p.status, dev_code(kDevTimeout, kKerMla, 6), nullptr);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- softmax (thread = head)
    const int h = threadIdx.x;  // 0..127, TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float m_run = kNegInf, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j & 1;
      ok = mbar_wait_warp(&bar.s_full[s], (j >> 1) & 1, p.status, dev_code(kDevTimeout, kKerMla, 7),
                          abort_flag);
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t sr[32];
      tmem_ld32_wait(tmem + kTmS + s * kMN + lane_off, sr);
      const int lim = min(kMN, key1 - (key0 + j * kMN));
      float mx = kNegInf;
#pragma unroll
      for (int c = 0; c < kMN; ++c) {
        if (c >= lim) sr[c] = __float_as_uint(kNegInf);
        mx = fmaxf(mx, __uint_as_float(sr[c]));
      }
      const float m_new = fmaxf(m_run, mx * p.scale_log2);
      const bool resc = m_new > m_run + kRescale;
      const float m_use = resc ? m_new : m_run;
      const float alpha = resc ? ex2_approx(m_run - m_new) : 1.f;
      float sum = 0.f;
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < kMN; c += 2) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c]), p.scale_log2, -m_use));
        const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), p.scale_log2, -m_use));
        sum += p0 + p1;
        pk[c >> 1] = pack_bf16x2(p0, p1);
      }
      l_run = l_run * alpha + sum;
      m_run = m_use;
      // P_j (its buffer was last read by P.V j - 2, which the commit that
      // signalled S_j tracks)
      tmem_st16(tmem + kTmP + s * 16 + lane_off, pk);
      tmem_wait_st();
      // O *= alpha once the previous P.V has completed
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        ok = mbar_wait_warp(&bar.pv_done, (j - 1) & 1, p.status, dev_code(kDevTimeout, kKerMla, 8),
                            abort_flag);
        if (!ok) break;
        tc_fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < kMVH; c += 32) {
          uint32_t ov[32];
          tmem_ld32_wait(tmem + kTmO + c + lane_off, ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32_wait(tmem + kTmO + c + lane_off, ov);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.p_full[s]);
    }
    // epilogue: the split's O (this half of the value columns) and LSE
    if (ok)
      ok = mbar_wait_warp(&bar.o_done, 0, p.status, dev_code(kDevTimeout, kKerMla, 9), abort_flag);
    if (ok) {
      tc_fence_after_sync();
      const int64_t row = int64_t(b) * kMH + h;
      float* op = p.o_part + (row * p.nsplit + split) * kMV + half * kMVH;
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
      for (int c = 0; c < kMVH; c += 32) {
        uint32_t ov[32];
        tmem_ld32_wait(tmem + kTmO + c + lane_off, ov);
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(op + c + e) =
              make_float4(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv,
                          __uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
      }
      if (half == 0)
        p.lse_part[row * p.nsplit + split] =
            l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : kNegInf;
    }
  }

  // ---------------------------------------------------------- teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpProd) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
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

// [B, rows, 576] bf16, 128-byte swizzle, boxes of 64 columns x box_rows rows.
bool make_map_mla(CUtensorMap* m, const void* base, int rows, int B, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kMD), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kMD) * 2,
                                 static_cast<cuuint64_t>(rows) * kMD * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_mla_decode_partials(const void* q, const void* kv, float* o_part,
                                       float* lse_part, int B, int Sk, int nsplit, float scale,
                                       cudaStream_t s, int* status, const char** why) {
  CUtensorMap mq, mkv;
  if (!make_map_mla(&mq, q, kMH, B, kMH) || !make_map_mla(&mkv, kv, Sk, B, kMN)) {
    *why = "tensor map encoding failed";
    return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kMSmem);
  if (e != cudaSuccess) {
    *why = "shared memory attribute";
    return e;
  }
  MParams p{};
  p.B = B;
  p.Sk = Sk;
  p.nsplit = nsplit;
  p.scale_log2 = scale * kLog2e;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.status = status;
  const int64_t grid = int64_t(B) * nsplit * 2;
  mla_decode_kernel<<<static_cast<unsigned>(grid), kMThreads, kMSmem, s>>>(mq, mkv, p);
  return cudaGetLastError();
}

}  // namespace rf
