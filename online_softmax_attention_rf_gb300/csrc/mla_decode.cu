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
// the values are the latent columns, v = kv[:, :512]. The kernel is
// persistent: one CTA per SM, half of them per half of the value columns. The
// B * nsplit key segments are dealt out in order, a contiguous run of them per
// CTA (the two halves' CTAs of a run are neighbours and walk the same keys).
// Within a run, the consecutive segments of one batch element have contiguous
// keys; the CTA folds them into one online-softmax state and writes one
// partial, in the first segment's slot, and the other slots get LSE = -inf,
// which the merge skips. So q is loaded, and O written, once per batch element
// of a run instead of once per segment. Per CTA:
//   tensor memory: O_half [128 heads x 256 value columns] f32, one score tile
//     S [128 x 128 keys] f32 (P [128 x 128] bf16 is written over its first 64
//     columns), and the first 256 columns of q [128 x 256] bf16 (all 512
//     columns; the full 128 x 512 accumulator alone would fill tensor memory,
//     so the two halves of the value columns go to two CTAs, each forming the
//     scores itself);
//   shared memory: the other 320 columns of q (80 KB, loaded once per batch
//     element) and one slot for a 128-key kv tile (144 KB), all 128-byte
//     swizzled, K-major; each tile is also prefetched into L2 two tiles
//     ahead. The slot holds a tile in two parts that are released at
//     different times: X, the five 64-column chunks only the scores read (the
//     other value half and the rotary columns), free once the scores are
//     done, and H, this CTA's four value-half chunks, free once P.V is done.
//     The scores take X first, so the next tile's X part lands while the H
//     part's scores, the softmax and P.V run, and its H part while the next
//     X part's scores run. q's tensor-memory chunks are staged in the H part;
//   per tile: S = q kv_tile^T (36 MMAs of N = 128, K = 16: for the value half
//     whose X part holds chunks 0-3, 16 of them take q from tensor memory),
//     the softmax (one thread per head, TMEM lane = head) forms P over S,
//     then O_half += P V_half (eight TS-MMAs, P from tensor memory, V the
//     tile's latent columns read as an MN-major operand). The next tile's
//     scores are issued after that P.V and overwrite S in tensor-pipe order.
// An M = 128, K = 16 MMA takes about 55 cycles for any N up to 64 and 64 at
// N = 128, so 128-key tiles give the score MMAs twice the work per
// instruction for ~16 % more time; with one S buffer the softmax does not
// overlap the MMAs, which costs less than the halved MMA count saves (64-key
// tiles in two buffers, overlapped: ~4.0k cycles per 64 keys; one 128-key
// tile: ~4.5k).
// The partial (O, LSE) is written in the split-K workspace layout and merged
// by the split-K merge kernel. Between two batch elements of a run, the
// producer loads the next q's shared-memory chunks once the previous scores
// are done, and takes the slot (q's staged chunks, then tiles) once the
// previous O has left it. Every wait is bounded.
#include <cudaTypedefs.h>

#include <mutex>

#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kMH = 128;        // query heads (rows of every tile)
constexpr int kMD = 576;        // key dimension (latent + rotary)
constexpr int kMV = 512;        // value dimension (latent)
constexpr int kMVH = 256;       // value columns per CTA
constexpr int kMN = 128;        // keys per tile
constexpr int kMChunks = kMD / 64;             // 64-column swizzle chunks of a row
constexpr int kMXC = kMChunks - 4;             // chunks in a slot's X part (H holds 4)
constexpr int kMQT = 4;                        // q chunks in tensor memory (K steps 0-15)
constexpr int kMQS = kMChunks - kMQT;          // q chunks in shared memory (K steps 16-35)
constexpr int kMPrefetch = 2;                  // L2 prefetch distance, in tiles
constexpr int kQChunk = kMH * 128;             // 16 KB: one chunk of q
constexpr int kKVChunk = kMN * 128;            // 16 KB: one chunk of a kv tile
constexpr int kKVTile = kMChunks * kKVChunk;   // 144 KB
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kMQS * kQChunk;
constexpr int kOffBar = kOffKV + kKVTile;
constexpr int kOffQStage = kOffKV + kMXC * kKVChunk;  // q's TMEM chunks, in the H part at first
static_assert(kMQT * kQChunk <= 4 * kKVChunk, "q staging exceeds the H part");
constexpr int kMSmem = kOffBar + 256 + 1024;   // + alignment slack
// The epilogue stages each head's O row (256 floats) in the idle kv slot,
// rows 1040 bytes apart: a quarter-warp's 16-byte stores then fall in eight
// different bank groups.
constexpr int kStageRow = kMVH * 4 + 16;
static_assert(kMH * kStageRow <= kKVTile, "O staging exceeds the kv slot");
static_assert(kMSmem <= 227 * 1024, "MLA shared memory exceeds a CTA's limit");
constexpr int kMThreads = 192;  // warps 0-3 softmax, 4 producer + TMEM, 5 MMA issuer
constexpr int kWarpProd = 4;
constexpr int kWarpMma = 5;
// tensor-memory columns
constexpr uint32_t kTmO = 0;
constexpr uint32_t kTmS = kMVH;                // S, and P over its first 64 columns
constexpr uint32_t kTmQ = kTmS + kMN;          // q columns [0, 256): 8 columns per K step
static_assert(kTmQ + kMQT * 32 == 512, "MLA tensor-memory columns");
static_assert(kMQT % 2 == 0, "q chunks go to tensor memory in pairs");
constexpr float kRescale = 8.0f;               // log2 units (stale max kept below)

struct MBars {
  uint64_t q_full;      // q's shared-memory chunks have landed
  uint64_t q_stage;     // q's tensor-memory chunks have landed in the H part
  uint64_t q_tmem;      // q's tensor-memory columns are written (four softmax warps)
  uint64_t x_full;      // the slot's X part has landed
  uint64_t x_empty;     // the scores that read it have completed
  uint64_t h_full;      // the slot's H part has landed
  uint64_t h_empty;     // the P.V that read it has completed
  uint64_t s_full;      // S holds the scores of the current tile
  uint64_t p_full;      // P (over S) written by the four softmax warps
  uint64_t pv_done;     // the latest P.V has completed
  uint64_t o_done;      // a segment's MMAs have completed
  uint64_t epi_done;    // a segment's O has left the slot (four softmax warps)
  uint64_t mma_idle;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(MBars) <= 256, "MLA barriers exceed their block");

struct MParams {
  const __nv_bfloat16* q;  // [B, 128, 576]
  int B, Sk, nsplit;
  int64_t units;    // B * nsplit key segments (per value half)
  int64_t runs;     // CTAs per value half; CTA c takes segments [c U / R, (c + 1) U / R)
  float scale_log2;
  float* o_part;    // [B * 128, nsplit, 512]
  float* lse_part;  // [B * 128, nsplit]
  int* status;
};

// The consecutive key segments of one batch element within a CTA's run: their
// keys are contiguous, so the CTA folds them into one online-softmax state and
// writes one partial, in the slot of the first segment.
struct MSeg {
  int b, s0, s1;          // batch element, first and last segment
  int key0, key1, ntiles; // keys [key0, key1), 64-key tiles
  int64_t next;           // the run's next segment
};

__device__ __forceinline__ MSeg mla_segment(const MParams& p, int64_t u, int64_t u1) {
  MSeg g;
  g.b = static_cast<int>(u / p.nsplit);
  const int64_t first = int64_t(g.b) * p.nsplit;
  const int64_t end = min(u1, first + p.nsplit);
  g.s0 = static_cast<int>(u - first);
  g.s1 = static_cast<int>(end - 1 - first);
  const int per = p.Sk / p.nsplit;
  g.key0 = g.s0 * per;
  g.key1 = (g.s1 == p.nsplit - 1) ? p.Sk : (g.s1 + 1) * per;
  g.ntiles = (g.key1 - g.key0 + kMN - 1) / kMN;
  g.next = end;
  return g;
}

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
  // CTA -> (value half, run of key segments); the two halves' CTAs of a run
  // are neighbours, so each kv tile is read from DRAM once and from L2 once
  const int half = static_cast<int>(blockIdx.x & 1);
  const int64_t run = blockIdx.x >> 1;
  const int64_t u0 = run * p.units / p.runs, u1 = (run + 1) * p.units / p.runs;

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_stage, 1);
    mbar_init(&bar.q_tmem, 4);
    mbar_init(&bar.x_full, 1);
    mbar_init(&bar.x_empty, 1);
    mbar_init(&bar.h_full, 1);
    mbar_init(&bar.h_empty, 1);
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.p_full, 4);
    mbar_init(&bar.pv_done, 1);
    mbar_init(&bar.o_done, 1);
    mbar_init(&bar.epi_done, 4);
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
  // Every role walks the same segments. The n-th tile of the CTA (counted
  // over all its segments) completes phase n of the slot, S and P barriers;
  // segment k completes phase k of the q, o_done and epi_done barriers.

  if (warp == kWarpProd) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_kv);
      bool ok = true;
      int nq = 0, nqs = 0;   // q loads issued (shared part, staged part)
      int nx = 0, nh = 0;    // X / H parts requested
      int k = 0;
      for (int64_t u = u0; ok && u < u1; ++k) {
        const MSeg g = mla_segment(p, u, u1);
        // q's shared-memory chunks: once the previous segment's scores are done
        if (k > 0 && !(ok = mbar_wait(&bar.o_done, (k - 1) & 1, p.status,
                                      dev_code(kDevTimeout, kKerMla, 15), abort_flag)))
          break;
        mbar_arrive_expect_tx(&bar.q_full, kMQS * kQChunk);
        for (int c = 0; c < kMQS; ++c)
          tma_load_3d(smem + kOffQ + c * kQChunk, &tm_q, &bar.q_full, (kMQT + c) * 64, 0, g.b);
        ++nq;
        // the slot: once the previous segment's O has left it. q's
        // tensor-memory chunks are staged in the H part, which the segment's
        // first tile takes only after the softmax warps have copied them out.
        if (k > 0 && !(ok = mbar_wait(&bar.epi_done, (k - 1) & 1, p.status,
                                      dev_code(kDevTimeout, kKerMla, 16), abort_flag)))
          break;
        mbar_arrive_expect_tx(&bar.q_stage, kMQT * kQChunk);
        for (int c = 0; c < kMQT; ++c)
          tma_load_3d(smem + kOffQStage + c * kQChunk, &tm_q, &bar.q_stage, c * 64, 0, g.b);
        ++nqs;
        if (k == 0)
          for (int jj = 1; jj < kMPrefetch && jj < g.ntiles; ++jj)
            for (int c = 0; c < kMChunks; ++c)
              tma_prefetch_l2_3d(&tm_kv, c * 64, g.key0 + jj * kMN, g.b);
        const bool more = g.next < u1;
        const MSeg gn = more ? mla_segment(p, g.next, u1) : g;
        unsigned char* slot = smem + kOffKV;
        for (int j = 0; ok && j < g.ntiles; ++j) {
          if (nx >= 1)
            ok = mbar_wait(&bar.x_empty, (nx - 1) & 1, p.status,
                           dev_code(kDevTimeout, kKerMla, 1), abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&bar.x_full, kMXC * kKVChunk);
          for (int i = 0; i < kMXC; ++i)
            tma_load_3d(slot + i * kKVChunk, &tm_kv, &bar.x_full, x_chunk(i, half) * 64,
                        g.key0 + j * kMN, g.b);
          ++nx;
          if (nh >= 1)
            ok = mbar_wait(&bar.h_empty, (nh - 1) & 1, p.status,
                           dev_code(kDevTimeout, kKerMla, 13), abort_flag);
          if (ok && j == 0)
            ok = mbar_wait(&bar.q_tmem, k & 1, p.status, dev_code(kDevTimeout, kKerMla, 11),
                           abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&bar.h_full, 4 * kKVChunk);
          for (int i = 0; i < 4; ++i)
            tma_load_3d(slot + (kMXC + i) * kKVChunk, &tm_kv, &bar.h_full,
                        (4 * half + i) * 64, g.key0 + j * kMN, g.b);
          ++nh;
          // L2 prefetch kMPrefetch tiles ahead, into the next segment near the end
          const int jp = j + kMPrefetch;
          if (jp < g.ntiles) {
            for (int c = 0; c < kMChunks; ++c)
              tma_prefetch_l2_3d(&tm_kv, c * 64, g.key0 + jp * kMN, g.b);
          } else if (more && jp - g.ntiles < gn.ntiles) {
            for (int c = 0; c < kMChunks; ++c)
              tma_prefetch_l2_3d(&tm_kv, c * 64, gn.key0 + (jp - g.ntiles) * kMN, gn.b);
          }
        }
        u = g.next;
      }
      // never leave with copies in flight
      if (nq > 0)
        mbar_wait(&bar.q_full, (nq - 1) & 1, p.status, dev_code(kDevTimeout, kKerMla, 2), nullptr);
      if (nqs > 0)
        mbar_wait(&bar.q_stage, (nqs - 1) & 1, p.status, dev_code(kDevTimeout, kKerMla, 2),
                  nullptr);
      if (nx > 0)
        mbar_wait(&bar.x_full, (nx - 1) & 1, p.status, dev_code(kDevTimeout, kKerMla, 2),
                  nullptr);
      if (nh > 0)
        mbar_wait(&bar.h_full, (nh - 1) & 1, p.status, dev_code(kDevTimeout, kKerMla, 2),
                  nullptr);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t q_base = s_base + kOffQ;
      bool ok = true, issued = false;
      const uint64_t qd = sdesc_sw128(q_base, 16, 1024);
      // descriptors of the slot's X part, H part (K-major) and H part as the
      // MN-major value operand
      const uint64_t xd = sdesc_sw128(s_base + kOffKV, 16, 1024);
      const uint64_t hd = sdesc_sw128(s_base + kOffKV + kMXC * kKVChunk, 16, 1024);
      const uint64_t vd = sdesc_sw128(s_base + kOffKV + kMXC * kKVChunk, kKVChunk, 1024);
      const uint32_t tm_s = tmem + kTmS;
      int n = 0;  // tiles before
      int k = 0;
      for (int64_t u = u0; ok && u < u1; ++k) {
        const MSeg g = mla_segment(p, u, u1);
        ok = mbar_wait(&bar.q_full, k & 1, p.status, dev_code(kDevTimeout, kKerMla, 3), abort_flag);
        if (ok)
          ok = mbar_wait(&bar.q_tmem, k & 1, p.status, dev_code(kDevTimeout, kKerMla, 10),
                         abort_flag);
        for (int j = 0; ok && j < g.ntiles; ++j, ++n) {
          const int par = n & 1;
          // S = q tile^T: the X part (then released), then the H part. S
          // overwrites P of the previous tile, whose P.V was issued before.
          if (!(ok = mbar_wait(&bar.x_full, par, p.status, dev_code(kDevTimeout, kKerMla, 4),
                               abort_flag)))
            break;
          tc_fence_after_sync();
          issued = true;
          if (half)
            issue_score_part<true, 1>(tm_s, tmem + kTmQ, qd, xd);
          else
            issue_score_part<true, 0>(tm_s, tmem + kTmQ, qd, xd);
          mma_commit(&bar.x_empty);
          if (!(ok = mbar_wait(&bar.h_full, par, p.status, dev_code(kDevTimeout, kKerMla, 14),
                               abort_flag)))
            break;
          tc_fence_after_sync();
          if (half)
            issue_score_part<false, 1>(tm_s, tmem + kTmQ, qd, hd);
          else
            issue_score_part<false, 0>(tm_s, tmem + kTmQ, qd, hd);
          mma_commit(&bar.s_full);
          // P_j is in tensor memory
          if (!(ok = mbar_wait(&bar.p_full, par, p.status, dev_code(kDevTimeout, kKerMla, 5),
                               abort_flag)))
            break;
          tc_fence_after_sync();
          issue_values(tmem + kTmO, tm_s, vd, j > 0);
          mma_commit(&bar.h_empty);
          mma_commit(&bar.pv_done);
        }
        if (ok) mma_commit(&bar.o_done);
        u = g.next;
      }
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
    bool ok = true;
    int n = 0;  // tiles before
    int k = 0;
    for (int64_t u = u0; ok && u < u1; ++k) {
      const MSeg g = mla_segment(p, u, u1);
      // q columns [0, 256) of head h into tensor memory from the staged
      // chunks: the 32-bit words of the bf16 row in order are the A operand's
      // layout (two elements per column, the lower column in the low half).
      // A staged row is 128-byte swizzled: its 16-byte unit u sits at unit
      // u ^ (h & 7), so eight consecutive heads read eight bank groups.
      if (!(ok = mbar_wait_warp(&bar.q_stage, k & 1, p.status, dev_code(kDevTimeout, kKerMla, 12),
                                abort_flag)))
        break;
      {
        const unsigned char* qs = smem + kOffQStage + h * 128;
#pragma unroll 1
        for (int c = 0; c < kMQT; ++c) {
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint4 v = *reinterpret_cast<const uint4*>(qs + c * kQChunk + ((e ^ (h & 7)) << 4));
            w[4 * e] = v.x;
            w[4 * e + 1] = v.y;
            w[4 * e + 2] = v.z;
            w[4 * e + 3] = v.w;
          }
          tmem_st32(tmem + kTmQ + c * 32 + lane_off, w);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.q_tmem);
      }
      float m_run = kNegInf, l_run = 0.f;
      for (int j = 0; ok && j < g.ntiles; ++j, ++n) {
        ok = mbar_wait_warp(&bar.s_full, n & 1, p.status, dev_code(kDevTimeout, kKerMla, 7),
                            abort_flag);
        if (!ok) break;
        tc_fence_after_sync();
        uint32_t sr[kMN];
        tmem_ld128_wait(tmem + kTmS + lane_off, sr);
        const int lim = min(kMN, g.key1 - (g.key0 + j * kMN));  // the same in every thread
        if (lim < kMN) {
#pragma unroll
          for (int c = 0; c < kMN; ++c)
            if (c >= lim) sr[c] = __float_as_uint(kNegInf);
        }
        // row maximum: eight independent partial maxima, three inputs per max
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = kNegInf;
#pragma unroll
        for (int c = 0; c < kMN; c += 2)
          m8[(c >> 1) & 7] =
              fmax3(m8[(c >> 1) & 7], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
        const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                               fmaxf(m8[6], m8[7]));
        const float m_new = fmaxf(m_run, mx * p.scale_log2);
        const bool resc = m_new > m_run + kRescale;
        const float m_use = resc ? m_new : m_run;
        const float alpha = resc ? ex2_approx(m_run - m_new) : 1.f;
        // p = 2^(s c - m) on column pairs (packed FMA and adds, four partial
        // sums); P over the first 64 columns of S (all of S has been read)
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 nm2 = make_float2(-m_use, -m_use);
        float2 s4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) s4[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const float2 x = ffma2(make_float2(__uint_as_float(sr[64 * hf + c]),
                                               __uint_as_float(sr[64 * hf + c + 1])),
                                   sc2, nm2);
            const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            s4[(c >> 1) & 3] = fadd2(s4[(c >> 1) & 3], pp);
            pk[c >> 1] = pack_bf16x2(pp.x, pp.y);
          }
          tmem_st32(tmem + kTmS + 32 * hf + lane_off, pk);
        }
        const float2 st = fadd2(fadd2(s4[0], s4[1]), fadd2(s4[2], s4[3]));
        const float sum = st.x + st.y;
        l_run = l_run * alpha + sum;
        m_run = m_use;
        tmem_wait_st();
        // O *= alpha once the previous P.V has completed (it has: the scores
        // that this tile's S came from were issued after it)
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          ok = mbar_wait_warp(&bar.pv_done, (n - 1) & 1, p.status,
                              dev_code(kDevTimeout, kKerMla, 8), abort_flag);
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
        if (lane == 0) mbar_arrive(&bar.p_full);
      }
      // epilogue: the segment's O (this half of the value columns) and LSE
      if (!ok ||
          !(ok = mbar_wait_warp(&bar.o_done, k & 1, p.status, dev_code(kDevTimeout, kKerMla, 9),
                                abort_flag)))
        break;
      tc_fence_after_sync();
      const int64_t row = int64_t(g.b) * kMH + h;
      float* op = p.o_part + (row * p.nsplit + g.s0) * kMV + half * kMVH;
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      // The row goes through shared memory and leaves as one 1 KB bulk copy
      // (each thread's own row, so no barrier between them): the kv slot is
      // idle here, since every tile of the segment landed before its MMAs,
      // the last P.V has completed, and the producer loads nothing into the
      // slot before epi_done.
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
      // the partial sits in the first segment's slot; the others hold no
      // payload and a -inf LSE, which the merge skips
      if (half == 0) {
        float* lp = p.lse_part + row * p.nsplit;
        lp[g.s0] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : kNegInf;
        for (int t = g.s0 + 1; t <= g.s1; ++t) lp[t] = kNegInf;
      }
      bulk_store_drain();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.epi_done);
      u = g.next;
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
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 2) {
    *why = "device attributes";
    return cudaErrorInvalidValue;
  }
  MParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.B = B;
  p.Sk = Sk;
  p.nsplit = nsplit;
  p.units = int64_t(B) * nsplit;
  // persistent: one CTA per SM, half of them per value half
  p.runs = p.units < sms / 2 ? p.units : sms / 2;
  p.scale_log2 = scale * kLog2e;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.status = status;
  const int64_t grid = 2 * p.runs;
  mla_decode_kernel<<<static_cast<unsigned>(grid), kMThreads, kMSmem, s>>>(mq, mkv, p);
  return cudaGetLastError();
}

}  // namespace rf
