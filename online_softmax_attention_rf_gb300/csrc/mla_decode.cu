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
//     S [128 x 64 keys] f32 (P [128 x 64] bf16 is written over the first 32
//     columns of its S), and the first 256 columns of q [128 x 256] bf16 (all
//     512 columns; the full 128 x 512 accumulator alone would fill tensor
//     memory, so the two halves of the value columns go to two CTAs, each
//     forming the scores itself);
//   shared memory: the other 320 columns of q (80 KB, loaded once) and a
//     2-stage ring of 64-key kv tiles (72 KB each), all 128-byte swizzled,
//     K-major; each tile is also prefetched into L2 two tiles ahead. A slot
//     holds a tile in two parts that are released at different times: X, the
//     five 64-column chunks only the scores read (the other value half and
//     the rotary columns), free once the scores are done, and H, this CTA's
//     four value-half chunks, free once P.V is done. The scores take X
//     first, so the next-but-one tile's H part has their duration to land;
//   S_b = q kv_tile^T (36 MMAs of K = 16: the first 16 take q from tensor
//     memory, the last 20 from shared memory), the softmax (one thread per
//     head, TMEM lane = head) forms P_b, then O_half += P_b V_half (four
//     TS-MMAs, P from tensor memory, V the tile's latent columns read as an
//     MN-major operand); the next tile's scores are computed while the
//     softmax works.
// An M = 128, K = 16 MMA takes about 55 cycles for any N up to 64 (64 at
// N = 128, where the arithmetic starts to bound it), so 64-key tiles halve
// the score MMAs' time per key against 32-key ones; q in tensor memory frees
// the shared memory that 64-key tiles need.
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
constexpr int kMN = 64;         // keys per tile
constexpr int kMChunks = kMD / 64;             // 64-column swizzle chunks of a row
constexpr int kMXC = kMChunks - 4;             // chunks in a slot's X part (H holds 4)
constexpr int kMQT = 4;                        // q chunks in tensor memory (K steps 0-15)
constexpr int kMQS = kMChunks - kMQT;          // q chunks in shared memory (K steps 16-35)
constexpr int kMStages = 2;                    // kv ring depth
constexpr int kMPrefetch = 2;                  // L2 prefetch distance, in tiles
constexpr int kQChunk = kMH * 128;             // 16 KB: one chunk of q
constexpr int kKVChunk = kMN * 128;            // 8 KB: one chunk of a kv tile
constexpr int kKVTile = kMChunks * kKVChunk;   // 72 KB
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kMQS * kQChunk;
constexpr int kOffBar = kOffKV + kMStages * kKVTile;
constexpr int kOffQStage = kOffKV + (kMStages - 1) * kKVTile;  // q's TMEM chunks, at first
static_assert(kMQT * kQChunk <= kKVTile, "q staging exceeds a ring slot");
constexpr int kMSmem = kOffBar + 256 + 1024;   // + alignment slack
// The epilogue stages each head's O row (256 floats) in the idle kv ring,
// rows 1040 bytes apart: a quarter-warp's 16-byte stores then fall in eight
// different bank groups.
constexpr int kStageRow = kMVH * 4 + 16;
static_assert(kMH * kStageRow <= kMStages * kKVTile, "O staging exceeds the kv ring");
static_assert(kMSmem <= 227 * 1024, "MLA shared memory exceeds a CTA's limit");
constexpr int kMThreads = 192;  // warps 0-3 softmax, 4 producer + TMEM, 5 MMA issuer
constexpr int kWarpProd = 4;
constexpr int kWarpMma = 5;
// tensor-memory columns
constexpr uint32_t kTmO = 0;
constexpr uint32_t kTmS = kMVH;                // S_b at kTmS + 64 b, P_b over its first 32
constexpr uint32_t kTmQ = kTmS + 2 * kMN;      // q columns [0, 256): 8 columns per K step
static_assert(kTmQ + kMQT * 32 == 512, "MLA tensor-memory columns");
static_assert(kMQT % 2 == 0, "q chunks go to tensor memory in pairs");
constexpr float kRescale = 8.0f;               // log2 units (stale max kept below)

struct MBars {
  uint64_t q_full;      // q's shared-memory chunks have landed
  uint64_t q_stage;     // q's tensor-memory chunks have landed in the last ring slot
  uint64_t q_tmem;      // q's tensor-memory columns are written (four softmax warps)
  uint64_t x_full[kMStages];    // a slot's X part has landed
  uint64_t x_empty[kMStages];   // the scores that read it have completed
  uint64_t h_full[kMStages];    // a slot's H part has landed
  uint64_t h_empty[kMStages];   // the P.V that read it has completed
  uint64_t s_full[2];   // S_b holds the scores of the tile using buffer b
  uint64_t p_full[2];   // P_b (over S_b) written by the four softmax warps
  uint64_t pv_done;     // the latest P.V has completed
  uint64_t o_done;
  uint64_t mma_idle;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(MBars) <= 256, "MLA barriers exceed their block");

struct MParams {
  const __nv_bfloat16* q;  // [B, 128, 576]
  int B, Sk, nsplit;
  float scale_log2;
  float* o_part;    // [B * 128, nsplit, 512]
  float* lse_part;  // [B * 128, nsplit]
  int* status;
};

// Warm L2 with a box of a tensor (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// Contiguous bulk copy shared -> global, tracked by this thread's bulk group.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_store_row(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}

// Commit this thread's bulk stores and wait until they have read their source
// (the CTA may then exit; the writes complete before the grid does).
__device__ __forceinline__ void bulk_store_drain() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Chunk i of a slot's X part: the other value half's four chunks, then the
// rotary chunk 8.
__host__ __device__ constexpr int x_chunk(int i, int half) { return i < 4 ? (half ? i : 4 + i) : 8; }

// Part of S = q tile^T: for each chunk c of the part, four K steps of 16
// (32 bytes apart in the swizzled rows), q from tensor memory for c < kMQT and
// from shared memory otherwise. The X part starts the accumulation. kHalf is
// a template argument so that every chunk index and operand choice is fixed
// at compile time (the issuing thread's instructions per MMA count); the
// operand descriptors are the part's and q's base descriptors plus constant
// address offsets (a descriptor holds the shared address >> 4 in its low 14
// bits, and every offset here stays inside the shared window).
template <bool kX, int kHalf>
__device__ __forceinline__ void issue_score_part(uint32_t tm_s, uint32_t tm_q, uint64_t qd,
                                                 uint64_t pd) {
  constexpr uint32_t idesc = idesc_bf16_f32(kMH, kMN, 0);
  constexpr int n = kX ? kMXC : 4;
#pragma unroll
  for (int i = 0; i < n; ++i) {
    const int c = kX ? x_chunk(i, kHalf) : 4 * kHalf + i;
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const int kk = 4 * c + k4;
      const uint64_t kd = pd + static_cast<uint64_t>((i * kKVChunk + k4 * 32) >> 4);
      const uint32_t acc = (kX && i == 0 && k4 == 0) ? 0u : 1u;
      if (c < kMQT)
        mma_bf16_ts(tm_s, tm_q + kk * 8, kd, idesc, acc);
      else
        mma_bf16(tm_s, qd + static_cast<uint64_t>(((c - kMQT) * kQChunk + k4 * 32) >> 4), kd,
                 idesc, acc);
    }
  }
}

// O_half (+)= P V_half: A = P from tensor memory (8 columns per 16 keys), B =
// the H part (this CTA's 256 value columns) as an MN-major operand (64-column
// chunks kKVChunk apart, 8-key groups 1024 bytes apart).
__device__ __forceinline__ void issue_values(uint32_t tm_o, uint32_t tm_p, uint64_t vd,
                                             bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kMH, kMVH, 1);
#pragma unroll
  for (int kk = 0; kk < kMN / 16; ++kk)
    mma_bf16_ts(tm_o, tm_p + kk * 8, vd + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc,
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
    mbar_init(&bar.q_stage, 1);
    mbar_init(&bar.q_tmem, 4);
    for (int i = 0; i < kMStages; ++i) {
      mbar_init(&bar.x_full[i], 1);
      mbar_init(&bar.x_empty[i], 1);
      mbar_init(&bar.h_full[i], 1);
      mbar_init(&bar.h_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
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
      // q's tensor-memory chunks are staged in the last ring slot, which its
      // first tile takes only after the softmax warps have copied them out
      mbar_arrive_expect_tx(&bar.q_stage, kMQT * kQChunk);
      for (int c = 0; c < kMQT; ++c)
        tma_load_3d(smem + kOffQStage + c * kQChunk, &tm_q, &bar.q_stage, c * 64, 0, b);
      mbar_arrive_expect_tx(&bar.q_full, kMQS * kQChunk);
      for (int c = 0; c < kMQS; ++c)
        tma_load_3d(smem + kOffQ + c * kQChunk, &tm_q, &bar.q_full, (kMQT + c) * 64, 0, b);
      for (int jj = 1; jj < kMPrefetch && jj < ntiles; ++jj)
        for (int c = 0; c < kMChunks; ++c)
          tma_prefetch_l2_3d(&tm_kv, c * 64, key0 + jj * kMN, b);
      bool ok = true;
      int nx = 0, nh = 0;  // tiles whose X / H parts were requested
      for (int j = 0; ok && j < ntiles; ++j) {
        const int s = j % kMStages;
        const int par = ((j / kMStages) - 1) & 1;
        unsigned char* slot = smem + kOffKV + s * kKVTile;
        if (j >= kMStages)
          ok = mbar_wait(&bar.x_empty[s], par, p.status, dev_code(kDevTimeout, kKerMla, 1),
                         abort_flag);
        else if (j == kMStages - 1)
          ok = mbar_wait(&bar.q_tmem, 0, p.status, dev_code(kDevTimeout, kKerMla, 11), abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bar.x_full[s], kMXC * kKVChunk);
        for (int i = 0; i < kMXC; ++i)
          tma_load_3d(slot + i * kKVChunk, &tm_kv, &bar.x_full[s], x_chunk(i, half) * 64,
                      key0 + j * kMN, b);
        ++nx;
        if (j >= kMStages)
          ok = mbar_wait(&bar.h_empty[s], par, p.status, dev_code(kDevTimeout, kKerMla, 13),
                         abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bar.h_full[s], 4 * kKVChunk);
        for (int i = 0; i < 4; ++i)
          tma_load_3d(slot + (kMXC + i) * kKVChunk, &tm_kv, &bar.h_full[s], (4 * half + i) * 64,
                      key0 + j * kMN, b);
        ++nh;
        if (j + kMPrefetch < ntiles)
          for (int c = 0; c < kMChunks; ++c)
            tma_prefetch_l2_3d(&tm_kv, c * 64, key0 + (j + kMPrefetch) * kMN, b);
      }
      // never leave with copies in flight
      mbar_wait(&bar.q_full, 0, p.status, dev_code(kDevTimeout, kKerMla, 2), nullptr);
      mbar_wait(&bar.q_stage, 0, p.status, dev_code(kDevTimeout, kKerMla, 2), nullptr);
      for (int i = max(0, nx - kMStages); i < nx; ++i)
        mbar_wait(&bar.x_full[i % kMStages], (i / kMStages) & 1, p.status,
                  dev_code(kDevTimeout, kKerMla, 2), nullptr);
      for (int i = max(0, nh - kMStages); i < nh; ++i)
        mbar_wait(&bar.h_full[i % kMStages], (i / kMStages) & 1, p.status,
                  dev_code(kDevTimeout, kKerMla, 2), nullptr);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t q_base = s_base + kOffQ;
      bool ok = mbar_wait(&bar.q_full, 0, p.status, dev_code(kDevTimeout, kKerMla, 3), abort_flag);
      if (ok)
        ok = mbar_wait(&bar.q_tmem, 0, p.status, dev_code(kDevTimeout, kKerMla, 10), abort_flag);
      bool issued = false;
      const uint64_t qd = sdesc_sw128(q_base, 16, 1024);
      // descriptors of the ring slots' X part, H part (K-major) and H part as
      // the MN-major value operand; slot 1 is kKVTile bytes after slot 0
      static_assert(kMStages == 2, "the descriptor selection below assumes two slots");
      const uint64_t xd0 = sdesc_sw128(s_base + kOffKV, 16, 1024);
      const uint64_t hd0 = sdesc_sw128(s_base + kOffKV + kMXC * kKVChunk, 16, 1024);
      const uint64_t vd0 = sdesc_sw128(s_base + kOffKV + kMXC * kKVChunk, kKVChunk, 1024);
      constexpr uint64_t kSlotStep = kKVTile >> 4;
      // S_t: the X part (then its slot part is released), then the H part
      auto scores = [&](int t) -> bool {
        const int ks = t % kMStages, par = (t / kMStages) & 1;
        const uint32_t tm_s = tmem + kTmS + (t & 1) * kMN;
        const uint64_t xk = xd0 + (ks ? kSlotStep : 0), hk = hd0 + (ks ? kSlotStep : 0);
        if (!mbar_wait(&bar.x_full[ks], par, p.status, dev_code(kDevTimeout, kKerMla, 4),
                       abort_flag))
          return false;
        tc_fence_after_sync();
        issued = true;
        if (half)
          issue_score_part<true, 1>(tm_s, tmem + kTmQ, qd, xk);
        else
          issue_score_part<true, 0>(tm_s, tmem + kTmQ, qd, xk);
        mma_commit(&bar.x_empty[ks]);
        if (!mbar_wait(&bar.h_full[ks], par, p.status, dev_code(kDevTimeout, kKerMla, 14),
                       abort_flag))
          return false;
        tc_fence_after_sync();
        if (half)
          issue_score_part<false, 1>(tm_s, tmem + kTmQ, qd, hk);
        else
          issue_score_part<false, 0>(tm_s, tmem + kTmQ, qd, hk);
        mma_commit(&bar.s_full[t & 1]);
        return true;
      };
      if (ok) ok = scores(0);
      for (int j = 0; ok && j < ntiles; ++j) {
        const int s = j & 1;                 // S and P buffers
        const int ks = j % kMStages;         // ring slot
        // the next tile's scores (its S buffer was read by softmax j - 1,
        // whose P.V was issued in the previous iteration)
        if (j + 1 < ntiles && !(ok = scores(j + 1))) break;
        // P_j is in tensor memory
        if (!(ok = mbar_wait(&bar.p_full[s], (j >> 1) & 1, p.status,
                             dev_code(kDevTimeout, kKerMla, 5), abort_flag)))
          break;
        tc_fence_after_sync();
        issue_values(tmem + kTmO, tmem + kTmS + s * kMN, vd0 + (ks ? kSlotStep : 0), j > 0);
        mma_commit(&bar.h_empty[ks]);
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
    // q columns [0, 256) of head h into tensor memory from the staged
    // chunks: the 32-bit words of the bf16 row in order are the A operand's
    // layout (two elements per column, the lower column in the low half).
    // A staged row is 128-byte swizzled: its 16-byte unit u sits at unit
    // u ^ (h & 7), so eight consecutive heads read eight bank groups.
    bool ok = mbar_wait_warp(&bar.q_stage, 0, p.status, dev_code(kDevTimeout, kKerMla, 12),
                             abort_flag);
    if (ok) {
      const unsigned char* qs = smem + kOffQStage + h * 128;
#pragma unroll 1
      for (int c = 0; c < kMQT; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = *reinterpret_cast<const uint4*>(qs + c * kQChunk + ((u ^ (h & 7)) << 4));
          w[4 * u] = v.x;
          w[4 * u + 1] = v.y;
          w[4 * u + 2] = v.z;
          w[4 * u + 3] = v.w;
        }
        tmem_st32(tmem + kTmQ + c * 32 + lane_off, w);
      }
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.q_tmem);
    }
    float m_run = kNegInf, l_run = 0.f;
    for (int j = 0; ok && j < ntiles; ++j) {
      const int s = j & 1;
      ok = mbar_wait_warp(&bar.s_full[s], (j >> 1) & 1, p.status, dev_code(kDevTimeout, kKerMla, 7),
                          abort_flag);
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t sr[kMN];
      tmem_ld64_wait(tmem + kTmS + s * kMN + lane_off, sr);
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
      uint32_t pk[kMN / 2];
#pragma unroll
      for (int c = 0; c < kMN; c += 2) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c]), p.scale_log2, -m_use));
        const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), p.scale_log2, -m_use));
        sum += p0 + p1;
        pk[c >> 1] = pack_bf16x2(p0, p1);
      }
      l_run = l_run * alpha + sum;
      m_run = m_use;
      // P_j over the first half of S_j (this thread has read its row of S_j;
      // P.V j - 2 read the previous P there before S_j was computed)
      tmem_st32(tmem + kTmS + s * kMN + lane_off, pk);
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
      // The row goes through shared memory and leaves as one 1 KB bulk
      // copy (each thread's own row, so no barrier between them): the kv
      // ring is idle here, since every tile landed before its MMAs and the
      // last P.V has completed.
      float* stage = reinterpret_cast<float*>(smem + kOffKV + h * kStageRow);
#pragma unroll 1
      for (int c = 0; c < kMVH; c += 64) {
        uint32_t ov[64];
        tmem_ld64_wait(tmem + kTmO + c + lane_off, ov);
#pragma unroll
        for (int e = 0; e < 64; e += 4)
          *reinterpret_cast<float4*>(stage + c + e) =
              make_float4(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv,
                          __uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
      }
      fence_proxy_async_smem();
      bulk_store_row(op, stage, kMVH * 4);
      bulk_store_drain();
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
  p.q = static_cast<const __nv_bfloat16*>(q);
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
