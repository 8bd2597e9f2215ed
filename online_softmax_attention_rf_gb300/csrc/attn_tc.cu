// attn_tc.cu -- bf16 attention forward on the tcgen05 tensor cores.
//
// The cascaded reduction max -> sum exp -> normalised P.V of safe-softmax
// attention, fused into one pass over K and V in the incremental form
// (RedFuser: An Automatic Operator Fusion Framework for Cascaded Reductions
// on AI Accelerators, section 2: O(1) on-chip state per row; section 3:
// single-segment strategy, one CTA per query tile, FlashAttention as a special
// case). The max is taken straight from the Q K^T accumulator (FLASHLIGHT,
// Metodologia item 2), the running sum and accumulator are rescaled by
// exp(m_old - m_new) (item 3), and the head dimension is one tile (item 4).
// Masked 128 x 128 tiles are never visited (STOF, Méthodologie: block-sparse
// outer tiles in row-compressed lists; skipped, not zeroed); inside a partial
// tile of the two-level format the 8 x 8 inner bitmaps mask single keys.
//
// Each CTA runs two work items back to back; an item is two 128-row query
// tiles of one (batch, head) sharing one K/V stream, and a CTA pairs a heavy
// and a light item of one head so causal work is even across CTAs. Tensor
// memory, barriers and the pipeline stay live across the items, the second
// item's Q tiles load as soon as the last QK of the first has read each, and
// the second item's first QK is issued before the first item's epilogue.
// Warp roles (352 threads):
//   warps 0-3  softmax group 0 (query tile 0: thread r owns row r, TMEM lane r)
//   warps 4-7  softmax group 1 (query tile 1)
//   warp 8     TMEM allocator; TMA producer (one lane): Q tiles, then K/V
//              tiles into a shared-memory ring
//   warps 9-10 MMA issuers of query tiles 0 and 1 (one lane each)
// Each query tile has its own issuer. The tensor pipe accepts only a few MMAs
// ahead of the one executing, so an issuing thread stalls for about as long
// as its MMAs run; with one issuer per tile the two tiles' MMA streams are
// independent and one tile's softmax overlaps the other's MMAs. An issuer
// waits for the K/V tiles of its next block while its softmax group works,
// because shared-memory waits are slow while the tensor core streams operands
// from shared memory; it takes P from its group at a named barrier, which is
// cheap, and pushes each block of MMAs (P.V, then the next Q K^T) under a
// lock so that the two tiles' blocks reach the pipe whole and in turn.
// Tensor memory (512 columns): S0 | S1 (128 f32 columns each) | O0 | O1 (D each).
// P_t (bf16, two per column) is written back into tensor memory and is the A
// operand of the P.V MMA, so that MMA reads only V from shared memory: at
// D = 128 P_t overwrites the first half of S_t, at D = 64 it has its own
// columns after O1. Shared memory: Q0, Q1 (128-byte swizzled K-major) and the
// K/V ring (each slot one 128 x D tile; V is read as an MN-major operand).
//
// Per key tile u of query tile t:
//   MMA:     S_t = Q_t K_u^T                      (tcgen05.mma, f32 in TMEM)
//   softmax: m' = max(m, rowmax S); p = exp2(S*c - m'); l = a*l + rowsum p;
//            if the max grew by more than 2^8, O_t *= a = exp2(m - m') (in TMEM)
//            else the stale max is kept (a = 1; exact, since l and O share it);
//            P_t = bf16(p) into tensor memory
//   MMA:     O_t += P_t V_u, then at once S_t = Q_t K_next^T
// Epilogue: O = O_t / l (bf16), LSE = (m + log2 l) ln 2.
//
// Reuse of S_t's columns for P_t relies on the tensor pipe executing one
// thread's MMAs in issue order: QK_t(u+1) (which overwrites S_t) is issued after
// PV_t(u) (which reads P_t from it) by the same thread, as in the published
// Blackwell attention kernels; the commit that signals S_t(u+1) tracks PV_t(u)
// as well, so the softmax only writes P_t(u+1) after PV_t(u) has completed.
// A K/V slot is released when both groups are done with it: each group either
// commits its MMAs that read the slot or, for a key tile only the other group
// needs, arrives once the tile has landed.
//
// Every wait is bounded (RF_WAIT_LIMIT_NS); on expiry the kernel records a
// status code, the other roles notice the abort flag, and the CTA unwinds,
// waits for its own copies and MMAs, and frees its tensor memory. The five
// warps of a query tile (its four softmax warps and its issuer) decide to
// unwind together, at a reducing named barrier, so no warp is ever left
// waiting at a barrier the others have abandoned.
#include <cudaTypedefs.h>

#include <mutex>

#include "rf_device.cuh"

namespace rf {

cudaError_t launch_attn_empty(const AttnArgs& a, size_t elem_bytes, cudaStream_t s);

namespace {

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows > 256x
constexpr int kBM = 128;                   // query rows per tile
constexpr int kBN = 128;                   // keys per tile
constexpr int kThreads = 352;
constexpr int kWarpLoad = 8;
constexpr int kWarpIssue = 9;              // warps 9 and 10: MMA issuers of tiles 0 and 1
constexpr int kChunk = 16384;              // one 128-row x 64-column bf16 swizzle block

template <int D>
struct Layout {
  static constexpr int kTileBytes = kBM * D * 2;  // one Q, K or V tile
  static constexpr int kStages = (D == 128) ? 5 : 8;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + 2 * kTileBytes;
  static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
  static constexpr int kBarBytes = 256;
  // a split item's hand-over from group 1 to group 0: m and l of 128 rows
  static constexpr int kOffXch = kOffBar + kBarBytes;
  static constexpr int kXchBytes = 2 * kBM * 4;
  static constexpr int kBytes = kOffXch + kXchBytes + 1024;  // + alignment slack
  static constexpr uint32_t kTmemS = 0;        // S0 at 0, S1 at 128
  static constexpr uint32_t kTmemO = 2 * kBN;  // O0 at 256, O1 at 256 + D
  // P_t: on S_t's first 64 columns at D = 128 (S_t is read into registers
  // before P_t is written); after O1 at D = 64
  __host__ __device__ static constexpr uint32_t tmem_p(int t) {
    return D == 128 ? kTmemS + t * kBN : kTmemO + 2 * D + t * 64;
  }
};

struct Bars {
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t s_full[2];
  uint64_t o_done[2];
  uint64_t mma_idle[2];
  uint32_t tmem_base;
  int abort_flag;
  int issue_lock;  // held by a group while it pushes one block of MMAs
  int item_x;      // this CTA's double item (the work order's entry), -1: none
  uint64_t split_ready;  // split item: group 1's O, m and l are final (its 4 softmax warps)
  uint64_t split_read;   // split item: group 0 has read them (its 4 softmax warps)
};
static_assert(sizeof(Bars) <= Layout<64>::kBarBytes && sizeof(Bars) <= Layout<128>::kBarBytes,
              "barrier block overflows its shared-memory slot");
static_assert(Layout<64>::kBytes <= 227 * 1024 && Layout<128>::kBytes <= 227 * 1024,
              "attention shared memory exceeds a CTA's limit");

// Key-tile list of one query tile: dense/causal range or a block-sparse row.
struct TileList {
  const int32_t* cols;  // nullptr: range [0, n)
  int n;                // entries (after causal truncation and validation)
  const int32_t* tb;    // inner-level bitmap index per entry (-1: full); nullptr: all full
  int stride = 1;       // 2 in a split item's view: every second entry of a list
  __device__ __forceinline__ int at(int i) const { return cols ? cols[i * stride] : i; }
  __device__ __forceinline__ int bitmap(int i) const { return tb ? tb[i * stride] : -1; }
};

struct Params {
  int B, H, Hkv, Sq, Sk;
  float scale_log2;
  int causal;
  const int32_t* row_ptr;
  const int32_t* col_idx;
  const int32_t* tile_bits;  // two-level mask: bitmap index per list entry, or nullptr
  const uint64_t* bits;      // 256 words (8 x 8 blocks) per partial tile
  int per_head, nqt, nkt, pairs;
  const int32_t* cta_order;  // work order: CTA c takes double item cta_order[c]; nullptr: c
  __nv_bfloat16* o;
  float* lse;
  uint8_t* visited;
  int* status;
};

// The list of query tile qt of head bh; every role computes it identically.
// Block-sparse rows are truncated at the first entry that is out of range, not
// strictly ascending, or beyond the last causally visible key.
__device__ TileList tile_list(const Params& p, int bh, int qt, bool record) {
  TileList L{nullptr, 0, nullptr};
  if (qt >= p.nqt) return L;
  const int64_t q_end = min64(p.Sq, int64_t(qt + 1) * kBM);
  const int64_t kend = p.causal ? min64(p.Sk, q_end + (int64_t(p.Sk) - p.Sq)) : p.Sk;
  if (kend <= 0) return L;
  const int ntiles = static_cast<int>((kend + kBN - 1) / kBN);
  if (p.row_ptr == nullptr) {
    L.n = ntiles;
    return L;
  }
  const int32_t* rp = p.row_ptr + (p.per_head ? int64_t(bh) * p.nqt : 0) + qt;
  const int beg = rp[0], end = rp[1];
  L.cols = p.col_idx + beg;
  L.tb = p.tile_bits != nullptr ? p.tile_bits + beg : nullptr;
  int n = 0, prev = -1;
  for (int i = beg; i < end; ++i) {
    const int c = p.col_idx[i];
    if (c < 0 || c >= p.nkt || c <= prev) {
      if (record) record_status(p.status, dev_code(kDevBadList, kKerAttnTc, 1));
      break;
    }
    if (c >= ntiles) break;
    prev = c;
    ++n;
  }
  if (end < beg && record) record_status(p.status, dev_code(kDevBadList, kKerAttnTc, 2));
  L.n = n;
  return L;
}

// Merge cursor over the union of two ascending lists.
struct UnionIter {
  TileList l0, l1;
  int i0 = 0, i1 = 0;
  __device__ __forceinline__ bool next(int& u, bool& need0, bool& need1) {
    const int a = i0 < l0.n ? l0.at(i0) : 0x7fffffff;
    const int b = i1 < l1.n ? l1.at(i1) : 0x7fffffff;
    if (a == 0x7fffffff && b == 0x7fffffff) return false;
    u = min(a, b);
    need0 = (a == u);
    need1 = (b == u);
    i0 += need0;
    i1 += need1;
    return true;
  }
  // Whether the next entry exists and is needed by tile t (not consumed).
  __device__ __forceinline__ bool next_is(int t) const {
    const int a = i0 < l0.n ? l0.at(i0) : 0x7fffffff;
    const int b = i1 < l1.n ? l1.at(i1) : 0x7fffffff;
    if (a == 0x7fffffff && b == 0x7fffffff) return false;
    return t == 0 ? a <= b : b <= a;
  }
};

// Named barrier of one group -- its four softmax warps and its issuer warp,
// 160 threads, id 1 + t -- that also ORs a predicate over the group: every
// thread gets the same answer.
__device__ __forceinline__ bool group_sync_or(int t, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 160, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(1 + t)
      : "memory");
  return r != 0;
}

// The MMA issue lock. An issuer pushes each block of its MMAs (P.V and the
// next Q K^T) while holding it, so the two tiles' blocks reach the tensor pipe
// whole and in turn rather than interleaved: the groups then stay half a
// period apart, each one's softmax running under the other's MMAs. It is
// taken only after every wait the block needs, so its holder never waits on
// the other group. Acquisition is bounded like every other wait.
__device__ __forceinline__ bool issue_lock(int* lk, int* status, int code,
                                           volatile int* abort_flag) {
  if (atomicCAS(lk, 0, 1) == 0) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(32);
    if (atomicCAS(lk, 0, 1) == 0) return true;
    if (*abort_flag || globaltimer_ns() - t0 > RF_WAIT_LIMIT_NS) {
      record_status(status, code);
      *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ void issue_unlock(int* lk) { atomicExch(lk, 0); }

// Shared-memory descriptors are built once; an MMA step only adds a constant
// offset (in 16-byte units) to the start-address field, which cannot carry
// out of its 14 bits because shared memory ends below 256 KB.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tm_s, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, 0);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kChunk + (kk & 3) * 32) >> 4);
    mma_bf16(tm_s, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O_t (+)= P_t V: A = P_t from tensor memory (8 columns per 16 keys),
// B = V from shared memory as an MN-major operand.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tm_o, uint32_t tm_p, uint64_t v_desc,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, D, 1);
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>((kk * 16 * 128) >> 4);
    mma_bf16_ts(tm_o, tm_p + kk * 8, v_desc + off, idesc, (kk > 0 || accumulate) ? 1u : 0u);
  }
}

// Work items of one CTA. An item is a pair of query tiles of one head; CTA x
// takes two items of head x / ceil(pairs / 2): the pair counted j from the top
// (heavy under causal masking: later tiles see more keys) and the pair counted
// j from the bottom (light), so every CTA carries about the same causal work
// and the hardware's CTA scheduler balances the rest. CTAs run head-major,
// which keeps each head's K/V in L2 while its CTAs run; a mask's work order
// (cta_order, rf_blockmask_cta_order) may move the long double items to the
// front: x is the CTA's double item, read once at the kernel's start
// (item_x), -1 for an order entry outside the double items. Returns false
// when the CTA has no k-th item.
__device__ __forceinline__ int item_of_cta(const Params& p) {
  if (p.cta_order == nullptr) return static_cast<int>(blockIdx.x);
  const int x = p.cta_order[blockIdx.x];
  const int64_t n = int64_t((p.pairs + 1) / 2) * p.B * p.H;
  if (x < 0 || x >= n) {
    record_status(p.status, dev_code(kDevBadList, kKerAttnTc, 3));
    return -1;
  }
  return x;
}

// One work item of a CTA: the query tile of each softmax group (>= nqt: the
// group has none), or, for a split item, one query tile for both groups,
// which take alternate entries of its list and merge their states at the end.
struct Item {
  int bh;
  int q0, q1;
  bool split;
  __device__ __forceinline__ int q(int t) const { return t ? q1 : q0; }
};

// Raw length of query tile qt's list (before any truncation); 0 past the end.
__device__ __forceinline__ int list_len(const Params& p, int bh, int qt) {
  if (qt >= p.nqt) return 0;
  const int32_t* rp = p.row_ptr + (p.per_head ? int64_t(bh) * p.nqt : 0) + qt;
  return rp[1] - rp[0];
}

// The k-th item of double item x: the pair (2 (pairs - 1 - j), + 1), then
// the pair (2 j, + 1) when it differs. In launches with a two-level mask, a
// pair whose one tile lists more than 3 times its partner's entries plus 8
// (the query tile holding a mask's global rows, next to a band tile) becomes
// two items: the long tile split over both groups, then the other tile alone.
// Otherwise the long tile's group works alone while the other group idles
// after its few tiles. Every role computes the same sequence. Returns false
// when the CTA has no k-th item.
template <bool kInner>
__device__ bool cta_item(const Params& p, int x, int k, Item& it) {
  if (x < 0) return false;
  const int half = (p.pairs + 1) / 2;
  const int j = x % half;
  it.bh = x / half;
  it.split = false;
  if constexpr (!kInner) {
    if (k == 0) {
      it.q0 = 2 * (p.pairs - 1 - j);
      it.q1 = it.q0 + 1;
      return true;
    }
    if (k == 1 && j != p.pairs - 1 - j) {
      it.q0 = 2 * j;
      it.q1 = it.q0 + 1;
      return true;
    }
    return false;
  }
  const int npairs = j != p.pairs - 1 - j ? 2 : 1;
  int idx = 0;
  for (int s = 0; s < npairs; ++s) {
    const int a = s == 0 ? 2 * (p.pairs - 1 - j) : 2 * j, b = a + 1;
    int lng = -1, shrt = -1;
    if (p.row_ptr != nullptr) {
      const int la = list_len(p, it.bh, a), lb = list_len(p, it.bh, b);
      if (la > 3 * lb + 8) {
        lng = a;
        shrt = b;
      } else if (lb > 3 * la + 8) {
        lng = b;
        shrt = a;
      }
    }
    if (lng >= 0) {
      if (idx++ == k) {
        it.q0 = it.q1 = lng;
        it.split = true;
        return true;
      }
      if (shrt < p.nqt && idx++ == k) {
        it.q0 = shrt;
        it.q1 = p.nqt;
        it.split = false;
        return true;
      }
    } else if (idx++ == k) {
      it.q0 = a;
      it.q1 = b;
      it.split = false;
      return true;
    }
  }
  return false;
}

// Group t's list in item `it`: its tile's list, or, for a split item, the
// entries at positions t, t + 2, ... of the shared tile's list (only group
// 0's view records list faults).
template <bool kInner>
__device__ __forceinline__ TileList group_list(const Params& p, const Item& it, int t,
                                               bool record) {
  if (!kInner || !it.split) return tile_list(p, it.bh, it.q(t), record);
  TileList L = tile_list(p, it.bh, it.q0, record && t == 0);
  if (L.cols != nullptr) {
    L.cols += t;
    if (L.tb != nullptr) L.tb += t;
    L.n = (L.n - t + 1) / 2;
    L.stride = 2;
  } else {
    L.n = 0;  // not reached: items are split only in launches with lists
  }
  return L;
}

// kInner: the launch carries a two-level mask (inner 8 x 8 bitmaps); the
// other launches are compiled without that code path.
template <int D, bool kInner>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using L = Layout<D>;
  constexpr int NS = L::kStages;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bar = *reinterpret_cast<Bars*>(smem + L::kOffBar);
  const uint32_t s_base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bar.kv_full[i], 1);
      mbar_init(&bar.kv_empty[i], 2);  // one release per softmax group
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar.q_full[t], 1);
      mbar_init(&bar.q_empty[t], 1);
      mbar_init(&bar.s_full[t], 1);
      mbar_init(&bar.o_done[t], 1);
      mbar_init(&bar.mma_idle[t], 1);
    }
    bar.abort_flag = 0;
    bar.issue_lock = 0;
    bar.item_x = item_of_cta(p);
    mbar_init(&bar.split_ready, 4);
    mbar_init(&bar.split_read, 4);
    fence_barrier_init();
  }
  if (warp == kWarpLoad) {
    tmem_alloc(&bar.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  const int cta_x = bar.item_x;
  tc_fence_after_sync();
  const uint32_t tmem = bar.tmem_base;
  volatile int* abort_flag = &bar.abort_flag;

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    // Per item: the first K/V pair, then Q0 and Q1 (each once the previous
    // item's last QK on it has completed), then the remaining K/V pairs.
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      int seq = 0;
      int q_loads[2] = {0, 0};
      bool ok = true;
      Item d;
      for (int item = 0; ok && cta_item<kInner>(p, cta_x, item, d); ++item) {
        const int bh = d.bh;
        const int bk = (bh / p.H) * p.Hkv + (bh % p.H) / (p.H / p.Hkv);
        UnionIter it{group_list<kInner>(p, d, 0, false), group_list<kInner>(p, d, 1, false)};
        const int nt[2] = {it.l0.n, it.l1.n};
        int u;
        bool n0, n1;
        bool first = true;
        while (ok && it.next(u, n0, n1)) {
          for (int kv = 0; kv < 2 && ok; ++kv, ++seq) {
            const int slot = seq % NS;
            ok = mbar_wait(&bar.kv_empty[slot], ((seq / NS) & 1) ^ 1, p.status,
                           dev_code(kDevTimeout, kKerAttnTc, 10), abort_flag);
            if (!ok) break;
            mbar_arrive_expect_tx(&bar.kv_full[slot], L::kTileBytes);
            unsigned char* dst = smem + L::kOffKV + slot * L::kTileBytes;
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(dst + c * kChunk, kv == 0 ? &tm_k : &tm_v, &bar.kv_full[slot], c * 64,
                          u * kBN, bk);
          }
          if (first && ok) {
            first = false;
            for (int t = 0; t < 2 && ok; ++t) {
              if (nt[t] == 0) continue;
              if (q_loads[t] > 0)
                ok = mbar_wait(&bar.q_empty[t], (q_loads[t] - 1) & 1, p.status,
                               dev_code(kDevTimeout, kKerAttnTc, 12), abort_flag);
              if (!ok) break;
              mbar_arrive_expect_tx(&bar.q_full[t], L::kTileBytes);
              for (int c = 0; c < D / 64; ++c)
                tma_load_3d(smem + L::kOffQ + t * L::kTileBytes + c * kChunk, &tm_q,
                            &bar.q_full[t], c * 64, d.q(t) * kBM, bh);
              ++q_loads[t];
            }
          }
        }
      }
      // never leave with copies in flight: the last load into each slot
      for (int sq = max(0, seq - NS); sq < seq; ++sq)
        mbar_wait(&bar.kv_full[sq % NS], (sq / NS) & 1, p.status,
                  dev_code(kDevTimeout, kKerAttnTc, 11), nullptr);
      for (int t = 0; t < 2; ++t)
        if (q_loads[t] > 0)
          mbar_wait(&bar.q_full[t], (q_loads[t] - 1) & 1, p.status,
                    dev_code(kDevTimeout, kKerAttnTc, 13), nullptr);
    }
    __syncwarp();
  } else if (warp >= kWarpIssue) {
    // ------------------------------------------------------------ MMA issuers
    // Warp kWarpIssue + t issues and commits the MMAs of query tile t from its
    // first lane; the other lanes only keep the warp in the group barriers.
    const int t = warp - kWarpIssue;
    bool ok = true;
    // Q_t and the K/V ring as MMA operands: K slots K-major, V slots MN-major
    // (64-column blocks kChunk bytes apart); slot s starts s * kTileBytes in.
    const uint64_t q_desc = sdesc_sw128(s_base + L::kOffQ + t * L::kTileBytes, 16, 1024);
    const uint64_t k_desc0 = sdesc_sw128(s_base + L::kOffKV, 16, 1024);
    const uint64_t v_desc0 = sdesc_sw128(s_base + L::kOffKV, kChunk, 1024);
    const uint32_t mm_s = tmem + L::kTmemS + t * kBN;
    const uint32_t mm_o = tmem + L::kTmemO + t * D;
    const uint32_t mm_p = tmem + L::tmem_p(t);
    UnionIter it{};                      // the current item's union of both tiles' lists
    int seq = 0;                         // K/V sequence number of the next union entry
    int vseq = 0;                        // V tile of the entry whose QK was issued last
    int nq = 0;                          // items whose Q_t was waited for
    int n_iss = 0;                       // entries of this item issued (QK) so far
    int started = -1;                    // last item whose first QK was issued
    bool issued_any = false;
    Item icur{};                         // item the issuer is on
#define RF_WAIT(b, par, site)                                                        \
  mbar_wait(&bar.b, (par), p.status, dev_code(kDevTimeout, kKerAttnTc, site), abort_flag)
#define RF_SLOT(sq) (static_cast<uint64_t>((((sq) % NS) * L::kTileBytes) >> 4))
    // Next union entry this group needs; entries only the other group needs
    // are released (both slots) once they have landed. False at the item's end.
    auto advance = [&](int& u, int& kseq) -> bool {
      int uu;
      bool n0, n1;
      while (it.next(uu, n0, n1)) {
        const int ks = seq;
        seq += 2;
        if (t == 0 ? n0 : n1) {
          u = uu;
          kseq = ks;
          return true;
        }
        for (int e = 0; e < 2; ++e) {
          if (!(ok = RF_WAIT(kv_full[(ks + e) % NS], ((ks + e) / NS) & 1, 20))) return false;
          mbar_arrive(&bar.kv_empty[(ks + e) % NS]);
        }
      }
      return false;
    };
#define RF_LOCK() issue_lock(&bar.issue_lock, p.status, dev_code(kDevTimeout, kKerAttnTc, 23), abort_flag)
    // The next entry this group needs, with its K tile landed; false at the
    // item's end or on failure (ok).
    auto next_k = [&](int& u, int& kseq) -> bool {
      if (!advance(u, kseq)) return false;
      return (ok = RF_WAIT(kv_full[kseq % NS], (kseq / NS) & 1, 21));
    };
    // Commits after S_t = Q_t K_u^T (K in slot kseq) has been issued, the
    // one the softmax waits for first; they track every earlier MMA of this
    // thread, so they need not hold the lock.
    auto qk_commits = [&](int u, int kseq, int n) {
      mma_commit(&bar.s_full[t]);
      mma_commit(&bar.kv_empty[kseq % NS]);
      if (++n_iss == n) mma_commit(&bar.q_empty[t]);  // the item's last read of Q_t
      vseq = kseq + 1;
      if (p.visited != nullptr)
        p.visited[(int64_t(icur.bh) * p.nqt + icur.q(t)) * p.nkt + u] = 1;
    };
    // Item k: wait for its Q_t and issue its first QK (or, when this group
    // has no key tile in it, release all of its entries).
    auto start_item = [&](int k) {
      started = k;
      if (!cta_item<kInner>(p, cta_x, k, icur)) return;
      it = UnionIter{group_list<kInner>(p, icur, 0, t == 0),
                     group_list<kInner>(p, icur, 1, t == 1)};
      n_iss = 0;
      const int n = t == 0 ? it.l0.n : it.l1.n;
      if (n == 0) {
        int u, kseq;
        advance(u, kseq);  // releases every entry; returns false
        return;
      }
      if (!(ok = RF_WAIT(q_full[t], nq & 1, 22))) return;
      ++nq;
      int u, kseq;
      if (next_k(u, kseq) && (ok = RF_LOCK())) {
        tc_fence_after_sync();
        issue_qk<D>(mm_s, q_desc, k_desc0 + RF_SLOT(kseq));
        issue_unlock(&bar.issue_lock);
        issued_any = true;
        qk_commits(u, kseq, n);
      }
    };

    // The same items, lists and group barriers as the softmax warps.
    Item d;
    for (int item = 0; cta_item<kInner>(p, cta_x, item, d); ++item) {
      const TileList list = group_list<kInner>(p, d, t, false);
      if (lane == 0 && started < item) start_item(item);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      for (int jj = 0; jj < list.n; ++jj) {
        // Prepare this step's MMA block while the softmax runs: wait for V_u
        // and, when the next union entry is this group's, for that entry's K
        // tile, and consume the entry. Blocking on that K tile before this
        // step's P.V is safe: with no skipped entry between, its slot was
        // freed by releases committed in earlier blocks.
        const bool last = jj + 1 == list.n;
        int u2 = 0, k2 = 0;
        bool fast = false;
        if (lane == 0 && ok && (ok = RF_WAIT(kv_full[vseq % NS], (vseq / NS) & 1, 24)) && !last &&
            it.next_is(t) && (ok = RF_WAIT(kv_full[seq % NS], (seq / NS) & 1, 21))) {
          advance(u2, k2);  // consumes exactly that entry
          fast = true;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        // P_t is in tensor memory
        if (group_sync_or(t, !ok)) {
          ok = false;
          break;
        }
        if (lane == 0 && (ok = RF_LOCK())) {
          // O_t += P_t V_u, then the next QK of this group in the same block
          // when it was prepared above, or the end of the item. Only the MMAs
          // are issued under the lock; the commits follow it, S first. P.V is
          // issued before any wait that may block: the next K tile, or a tile
          // this group skips, may be loaded only into the slot this P.V
          // releases.
          tc_fence_after_sync();
          issue_pv<D>(mm_o, mm_p, v_desc0 + RF_SLOT(vseq), jj > 0);
          if (fast) issue_qk<D>(mm_s, q_desc, k_desc0 + RF_SLOT(k2));
          issue_unlock(&bar.issue_lock);
          const int v_done = vseq;
          if (fast) {
            qk_commits(u2, k2, list.n);
            mma_commit(&bar.kv_empty[v_done % NS]);
          } else {
            mma_commit(&bar.kv_empty[v_done % NS]);
            if (last) {
              mma_commit(&bar.o_done[t]);
            } else if (next_k(u2, k2) && (ok = RF_LOCK())) {
              tc_fence_after_sync();
              issue_qk<D>(mm_s, q_desc, k_desc0 + RF_SLOT(k2));
              issue_unlock(&bar.issue_lock);
              qk_commits(u2, k2, list.n);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (group_sync_or(t, !ok)) {  // after the item's steps
        ok = false;
        break;
      }
      // while the softmax warps write this item's output: release the
      // entries after this group's last, and start the next item
      if (lane == 0 && list.n > 0) {
        int u2, k2;
        advance(u2, k2);
        if (ok) start_item(item + 1);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (group_sync_or(t, !ok)) {  // after the item's epilogue
        ok = false;
        break;
      }
    }
#undef RF_WAIT
#undef RF_SLOT
#undef RF_LOCK
    // never leave with MMAs in flight (their operands live in this CTA)
    if (lane == 0 && issued_any) {
      mma_commit(&bar.mma_idle[t]);
      mbar_wait(&bar.mma_idle[t], 0, p.status, dev_code(kDevTimeout, kKerAttnTc, 28), nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax groups
    const int t = warp >> 2;             // query tile of this group
    const int r = threadIdx.x & 127;     // row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tm_s = tmem + L::kTmemS + t * kBN + lane_off;
    const uint32_t tm_o = tmem + L::kTmemO + t * D + lane_off;
    const uint32_t tm_p = tmem + L::tmem_p(t) + lane_off;
    const int shift = p.Sk - p.Sq;       // Sq, Sk <= 2^30: no overflow below
    int j = 0;                           // S tiles consumed (all items)
    int o_items = 0;                     // items whose final P.V was waited for
    int n_split = 0;                     // split items so far
    bool ok = true;
    // Every exit from the loops below is decided at a group barrier that the
    // group's issuer warp joins too, so the five warps always leave together.
    Item d;
    for (int item = 0; cta_item<kInner>(p, cta_x, item, d); ++item) {
      const int bh = d.bh;
      const int qt = d.q(t);
      const int row = qt * kBM + r;
      const TileList list = group_list<kInner>(p, d, t, false);
      const int row_lim = p.causal ? min(p.Sk, row + 1 + shift) : p.Sk;
      const int tile_first_lim = p.causal ? min(p.Sk, qt * kBM + 1 + shift) : p.Sk;
      float m_run = kNegInf, l_run = 0.f;
      for (int jj = 0; jj < list.n; ++jj, ++j) {
        const int u = list.at(jj);
        // A partial tile of a two-level mask: this row's 128 key bits, one
        // byte from each of the 16 inner 8 x 8 blocks it crosses, gathered
        // while S is being computed.
        const int pb = kInner ? list.bitmap(jj) : -1;
        uint32_t mw0 = ~0u, mw1 = ~0u, mw2 = ~0u, mw3 = ~0u;
        if (kInner && pb >= 0) {
          const uint8_t* rb = reinterpret_cast<const uint8_t*>(
                                  p.bits + int64_t(pb) * 256 + (r >> 3) * 16) + (r & 7);
          uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int cb = 0; cb < 16; ++cb) w[cb >> 2] |= uint32_t(rb[cb * 8]) << (8 * (cb & 3));
          mw0 = w[0]; mw1 = w[1]; mw2 = w[2]; mw3 = w[3];
        }
        if (ok)
          ok = mbar_wait_warp(&bar.s_full[t], j & 1, p.status,
                              dev_code(kDevTimeout, kKerAttnTc, 30), abort_flag);
        if (ok) {
          tc_fence_after_sync();
          // element mask only where the tile crosses the causal diagonal or Sk
          const int k0 = u * kBN;
          const int lim = (k0 + kBN > tile_first_lim) ? max(0, min(kBN, row_lim - k0)) : kBN;
          // pass 1: row maximum over all 128 columns (one TMEM read), 8
          // independent partial maxima, two columns per step (max is exact,
          // so the order does not matter)
          float mx;
          uint32_t sr[128];
          {
            tmem_ld128_wait(tm_s, sr);
            if (lim < kBN) {
#pragma unroll
              for (int c = 0; c < kBN; ++c)
                if (c >= lim) sr[c] = __float_as_uint(kNegInf);
            }
            if (kInner && pb >= 0) {
#pragma unroll
              for (int c = 0; c < kBN; ++c) {
                const uint32_t w = c < 32 ? mw0 : c < 64 ? mw1 : c < 96 ? mw2 : mw3;
                if (!((w >> (c & 31)) & 1u)) sr[c] = __float_as_uint(kNegInf);
              }
            }
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m8[i] = kNegInf;
#pragma unroll
            for (int c = 0; c < kBN; c += 2)
              m8[(c >> 1) & 7] = fmax3(m8[(c >> 1) & 7], __uint_as_float(sr[c]),
                                       __uint_as_float(sr[c + 1]));
            mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                       fmaxf(m8[6], m8[7]));
          }
          const float m_new = (mx == kNegInf) ? m_run : fmaxf(m_run, mx * p.scale_log2);
          const bool resc = m_new > m_run + kRescaleThreshold;
          const float m_use = resc ? m_new : m_run;
          const float alpha = resc ? ex2_approx(m_run - m_new) : 1.f;
          const float sh = (m_use == kNegInf) ? 0.f : m_use;
          // pass 2: p = exp2(s * c - m) two columns at a time (packed FMA),
          // row sum in 4 packed partial sums, P as bf16 pairs (column j =
          // keys 2j, 2j+1); half h writes P columns [32h, 32h + 32). Without
          // an inner mask S is read again in two halves of 64 (as fast as
          // keeping pass 1's registers, and lighter on them); with one, pass
          // 1's masked scores are reused. At D = 128 P overwrites S_t's first
          // 64 columns, which pass 1 and half 0 have read.
          const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
          const float2 nsh2 = make_float2(-sh, -sh);
          float2 s4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) s4[i] = make_float2(0.f, 0.f);
if constexpr (kInner) {
            // two-level masks: the masked scores of pass 1 are reused from
            // registers (10 % faster on the two-level workload than
            // masking a second read)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
              for (int c = 0; c < 64; c += 2) {
                const float2 x = ffma2(make_float2(__uint_as_float(sr[64 * h + c]),
                                                   __uint_as_float(sr[64 * h + c + 1])),
                                       sc2, nsh2);
                const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                s4[(c >> 1) & 3] = fadd2(s4[(c >> 1) & 3], pp);
                sr[32 * h + (c >> 1)] = pack_bf16x2(pp.x, pp.y);
              }
              tmem_st32(tm_p + 32 * h, *reinterpret_cast<const uint32_t(*)[32]>(&sr[32 * h]));
            }
          } else {
  #pragma unroll 1
            for (int h = 0; h < 2; ++h) {
              uint32_t sh1[64];
              tmem_ld64_wait(tm_s + 64 * h, sh1);
              if (lim < kBN) {
  #pragma unroll
                for (int c = 0; c < 64; ++c)
                  if (64 * h + c >= lim) sh1[c] = __float_as_uint(kNegInf);
              }
              if (kInner && pb >= 0) {
                const uint32_t wa = h ? mw2 : mw0, wb = h ? mw3 : mw1;
  #pragma unroll
                for (int c = 0; c < 64; ++c)
                  if (!(((c < 32 ? wa : wb) >> (c & 31)) & 1u)) sh1[c] = __float_as_uint(kNegInf);
              }
  #pragma unroll
              for (int c = 0; c < 64; c += 2) {
                const float2 x = ffma2(
                    make_float2(__uint_as_float(sh1[c]), __uint_as_float(sh1[c + 1])), sc2, nsh2);
                const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                s4[(c >> 1) & 3] = fadd2(s4[(c >> 1) & 3], pp);
                sh1[c >> 1] = pack_bf16x2(pp.x, pp.y);
              }
              tmem_st32(tm_p + 32 * h, *reinterpret_cast<const uint32_t(*)[32]>(&sh1[0]));
            }
          }
          tmem_wait_st();
          const float2 st = fadd2(fadd2(s4[0], s4[1]), fadd2(s4[2], s4[3]));
          l_run = l_run * alpha + (st.x + st.y);
          m_run = m_use;
          // O_t *= alpha; the previous P.V on O_t has completed (the commit
          // that signalled this S tracks it)
          if (jj > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t ov[32];
              tmem_ld32_wait(tm_o + c, ov);
#pragma unroll
              for (int e = 0; e < 32; ++e)
                ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
              tmem_st32_wait(tm_o + c, ov);
            }
          }
          tc_fence_before_sync();
        }
        // P_t (and any rescale of O_t) is in tensor memory for all 128 rows;
        // the group's issuer warp takes it from here
        if (group_sync_or(t, !ok)) {
          ok = false;
          break;
        }
      }
      // the issuer has committed the item's last P.V (or given up)
      if (group_sync_or(t, !ok)) {
        ok = false;
        break;
      }
      // epilogue: O = acc / l, LSE = (m + log2 l) ln 2. The next item's first
      // P.V on O_t is issued only after this group's next P is written, i.e.
      // after the TMEM reads below.
      if constexpr (kInner) {
        if (d.split) {
          // A split item: group 1's state over the odd entries goes to group
          // 0 (m and l through shared memory, O_1 read from tensor memory in
          // the same lanes), which merges it with its own over the even
          // entries and writes the rows. Group 1 then waits until group 0 has
          // read them before its next item can overwrite O_1. The waits are
          // bounded like every other.
          if (list.n > 0) {
            ok = mbar_wait_warp(&bar.o_done[t], o_items & 1, p.status,
                                dev_code(kDevTimeout, kKerAttnTc, 32), abort_flag);
            ++o_items;
          }
          float* xm = reinterpret_cast<float*>(smem + L::kOffXch);
          float* xl = xm + kBM;
          const uint32_t sp = n_split & 1;
          ++n_split;
          if (t == 1) {
            if (ok) {
              tc_fence_after_sync();
              xm[r] = m_run;
              xl[r] = l_run;
              tc_fence_before_sync();
              __syncwarp();
              if ((threadIdx.x & 31) == 0) mbar_arrive(&bar.split_ready);
              ok = mbar_wait_warp(&bar.split_read, sp, p.status,
                                  dev_code(kDevTimeout, kKerAttnTc, 34), abort_flag);
            }
          } else {
            if (ok)
              ok = mbar_wait_warp(&bar.split_ready, sp, p.status,
                                  dev_code(kDevTimeout, kKerAttnTc, 35), abort_flag);
            if (ok) {
              tc_fence_after_sync();
              const bool row_ok = row < p.Sq;
              const float m1 = xm[r], l1 = xl[r];
              const float m = fmaxf(m_run, m1);
              const float a0 = m_run == kNegInf ? 0.f : ex2_approx(m_run - m);
              const float a1 = m1 == kNegInf ? 0.f : ex2_approx(m1 - m);
              const float l = a0 * l_run + a1 * l1;
              const float inv = l > 0.f ? 1.f / l : 0.f;
              // a group without entries leaves its O columns unwritten: its
              // weight is 0 and its values are never used
              const float w0 = a0 * inv, w1 = a1 * inv;
              const uint32_t tm_o1 = tmem + L::kTmemO + D + lane_off;
              __nv_bfloat16* og = p.o + (int64_t(bh) * p.Sq + row) * D;
#pragma unroll 1
              for (int c = 0; c < D; c += 32) {
                uint32_t o0[32], o1[32];
                tmem_ld32_wait(tm_o + c, o0);
                tmem_ld32_wait(tm_o1 + c, o1);
                if (row_ok) {
                  float v[32];
#pragma unroll
                  for (int e = 0; e < 32; ++e)
                    v[e] = (w0 != 0.f ? w0 * __uint_as_float(o0[e]) : 0.f) +
                           (w1 != 0.f ? w1 * __uint_as_float(o1[e]) : 0.f);
#pragma unroll
                  for (int e = 0; e < 32; e += 8) {
                    uint4 w;
                    w.x = pack_bf16x2(v[e], v[e + 1]);
                    w.y = pack_bf16x2(v[e + 2], v[e + 3]);
                    w.z = pack_bf16x2(v[e + 4], v[e + 5]);
                    w.w = pack_bf16x2(v[e + 6], v[e + 7]);
                    *reinterpret_cast<uint4*>(og + c + e) = w;
                  }
                }
              }
              tc_fence_before_sync();
              if (row_ok && p.lse != nullptr)
                p.lse[int64_t(bh) * p.Sq + row] = l > 0.f ? (m + log2f(l)) * kLn2 : kNegInf;
              __syncwarp();
              if ((threadIdx.x & 31) == 0) mbar_arrive(&bar.split_read);
            }
          }
          if (group_sync_or(t, !ok)) {
            ok = false;
            break;
          }
          continue;
        }
      }
      const bool row_ok = row < p.Sq && qt < p.nqt;
      __nv_bfloat16* og = p.o + (int64_t(bh) * p.Sq + row) * D;
      if (list.n > 0) {
        ok = mbar_wait_warp(&bar.o_done[t], o_items & 1, p.status,
                            dev_code(kDevTimeout, kKerAttnTc, 32), abort_flag);
        ++o_items;
      }
      if (list.n > 0 && ok) {
        tc_fence_after_sync();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t ov[32];
          tmem_ld32_wait(tm_o + c, ov);
          if (row_ok) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(ov[e + 4]) * inv, __uint_as_float(ov[e + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(ov[e + 6]) * inv, __uint_as_float(ov[e + 7]) * inv);
              *reinterpret_cast<uint4*>(og + c + e) = w;
            }
          }
        }
        tc_fence_before_sync();
        if (row_ok && p.lse != nullptr)
          p.lse[int64_t(bh) * p.Sq + row] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : kNegInf;
      } else if (list.n == 0 && row_ok) {
        // no visible key for any row of this tile
        for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(og + c) = make_uint4(0, 0, 0, 0);
        if (p.lse != nullptr) p.lse[int64_t(bh) * p.Sq + row] = kNegInf;
      }
      if (group_sync_or(t, !ok)) {
        ok = false;
        break;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpLoad) {
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

// [BH, S, D] bf16, 128-byte swizzle, boxes of 64 columns x 128 rows.
bool make_map(CUtensorMap* m, const void* base, int D, int S, int BH) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(S) * D * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool kInner>
cudaError_t launch_d(const AttnArgs& a, cudaStream_t s, const char** why) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, D, a.Sq, a.B * a.H) || !make_map(&mk, a.k, D, a.Sk, a.B * a.Hkv) ||
      !make_map(&mv, a.v, D, a.Sk, a.B * a.Hkv)) {
    *why = "tensor map encoding failed";
    return cudaErrorInvalidValue;
  }
  constexpr int smem = Layout<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, kInner>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) {
    *why = "shared memory attribute";
    return e;
  }

  Params p{};
  p.B = a.B; p.H = a.H; p.Hkv = a.Hkv; p.Sq = a.Sq; p.Sk = a.Sk;
  p.scale_log2 = a.scale * kLog2e;
  p.causal = a.causal;
  p.row_ptr = a.row_ptr; p.col_idx = a.col_idx; p.per_head = a.per_head;
  p.tile_bits = a.tile_bits; p.bits = a.bits;
  p.nqt = a.nqt; p.nkt = a.nkt;
  p.pairs = (a.nqt + 1) / 2;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.visited = a.visited;
  p.cta_order = a.cta_order;
  p.status = a.status;
  const int64_t items = int64_t(p.pairs) * a.B * a.H;
  if (items > 0x7fffffffLL) {
    *why = "too many work items";
    return cudaErrorInvalidConfiguration;
  }
  // two items (a heavy and a light query-tile pair of one head) per CTA
  const int64_t grid = int64_t((p.pairs + 1) / 2) * a.B * a.H;
  attn_tc_kernel<D, kInner><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tc_bf16(const AttnArgs& a, cudaStream_t s, const char** why) {
  if (a.Sk == 0) return launch_attn_empty(a, 2, s);
  const bool inner = a.tile_bits != nullptr;
  if (a.d == 128) return inner ? launch_d<128, true>(a, s, why) : launch_d<128, false>(a, s, why);
  return inner ? launch_d<64, true>(a, s, why) : launch_d<64, false>(a, s, why);
}

}  // namespace rf
