// blockmask.cu -- dense tile mask -> row-compressed (BSR) tile lists.
//
// Accelerating Sparse Transformer Inference on GPU (STOF), Méthodologie,
// unified MHA module: the mask is kept as row-compressed lists of outer tiles,
// so that the attention kernel skips absent tiles entirely. The FLASHLIGHT
// summary (Risultati) notes that building block masks at run time is itself
// a cost; this kernel does it on the device in one launch.
//
// One CTA: (1) one warp per row counts the present tiles with ballots,
// (2) the CTA scans the counts into row_ptr, (3) one warp per row writes the
// column indices in ascending order (ballot + prefix popcount).
//
// The two-level form (same page, storage format: outer tiles full or
// partial, one 64-bit bitmap per 8 x 8 inner block of a partial tile) is
// built from a dense element mask in three launches: one CTA per outer tile
// classifies it; one CTA lists the non-empty tiles and numbers the partial
// ones in list order; one CTA per listed partial tile writes its 256 words.
#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads) blockmask_build_kernel(
    const uint8_t* __restrict__ dense, int64_t nrows, int nkt, int32_t* __restrict__ row_ptr,
    int32_t* __restrict__ col_idx, int64_t col_cap, int* status) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = kThreads / 32;
  // (1) counts into row_ptr[r + 1]
  for (int64_t r = warp; r < nrows; r += nw) {
    const uint8_t* row = dense + r * nkt;
    int cnt = 0;
    for (int c0 = 0; c0 < nkt; c0 += 32) {
      const int c = c0 + lane;
      cnt += __popc(__ballot_sync(0xffffffffu, c < nkt && row[c] != 0));
    }
    if (lane == 0) row_ptr[r + 1] = cnt;
  }
  if (threadIdx.x == 0) {
    row_ptr[0] = 0;
    carry = 0;
  }
  __syncthreads();
  // (2) inclusive scan of row_ptr[1 .. nrows], 1024 rows at a time
  for (int64_t base = 0; base < nrows; base += kThreads) {
    const int64_t r = base + threadIdx.x;
    int32_t v = r < nrows ? row_ptr[r + 1] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int32_t w = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += t;
      }
      warp_tot[lane] = w;  // inclusive per-warp totals
    }
    __syncthreads();
    const int32_t add = carry + (warp > 0 ? warp_tot[warp - 1] : 0);
    if (r < nrows) row_ptr[r + 1] = v + add;
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_tot[nw - 1];
    __syncthreads();
  }
  // (3) column indices, ascending within each row
  bool overflow = false;
  for (int64_t r = warp; r < nrows; r += nw) {
    const uint8_t* row = dense + r * nkt;
    int64_t pos = row_ptr[r];
    for (int c0 = 0; c0 < nkt; c0 += 32) {
      const int c = c0 + lane;
      const bool set = c < nkt && row[c] != 0;
      const unsigned bal = __ballot_sync(0xffffffffu, set);
      if (set) {
        const int64_t at = pos + __popc(bal & ((1u << lane) - 1u));
        if (at < col_cap)
          col_idx[at] = c;
        else
          overflow = true;
      }
      pos += __popc(bal);
    }
  }
  if (overflow) record_status(status, dev_code(kDevCapacity, kKerBlockmask, 1));
}

// CTA-wide exclusive scan helper state: inclusive per-warp totals.
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t* warp_tot,
                                                        int32_t* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += t;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t w = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  const int32_t excl = x - v + (warp > 0 ? warp_tot[warp - 1] : 0);
  *total = warp_tot[nw - 1];
  __syncthreads();
  return excl;
}

constexpr int kTile = 128, kInner = 8;
enum : int32_t { kEmpty = 0, kFull = 1, kPartial = 2 };

// E1: class of outer tile blockIdx.x = (n * nqt + qt) * nkt + kt, into state[].
__global__ void __launch_bounds__(256) tile_class_kernel(const uint8_t* __restrict__ dense,
                                                         int Sq, int Sk, int nqt, int nkt,
                                                         int32_t* __restrict__ state) {
  __shared__ int n_set, n_in;
  const int64_t tile = blockIdx.x;
  const int kt = static_cast<int>(tile % nkt);
  const int qt = static_cast<int>((tile / nkt) % nqt);
  const int64_t n = tile / (int64_t(nkt) * nqt);
  if (threadIdx.x == 0) n_set = n_in = 0;
  __syncthreads();
  const int r1 = min(kTile, Sq - qt * kTile), c1 = min(kTile, Sk - kt * kTile);
  const uint8_t* base = dense + (n * Sq + int64_t(qt) * kTile) * Sk + int64_t(kt) * kTile;
  int set = 0;
  for (int e = threadIdx.x; e < r1 * kTile; e += blockDim.x) {
    const int r = e / kTile, c = e % kTile;
    if (c < c1) set += base[int64_t(r) * Sk + c] != 0;
  }
  atomicAdd(&n_set, set);
  if (threadIdx.x == 0) n_in = r1 * c1;
  __syncthreads();
  if (threadIdx.x == 0)
    state[tile] = n_set == 0 ? kEmpty : (n_set == n_in ? kFull : kPartial);
}

// E2 (one CTA): row_ptr and col_idx from the states (still in tile_bits),
// then tile_bits[n] = the partial tile's number in list order, or -1.
__global__ void __launch_bounds__(1024) two_level_lists_kernel(
    int64_t nrows, int nkt, int32_t* __restrict__ row_ptr, int32_t* __restrict__ col_idx,
    int32_t* __restrict__ tile_bits, int64_t bits_cap, int32_t* n_partial, int* status) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  constexpr int32_t kPartialFlag = 1 << 30;
  // counts per row of outer tiles
  for (int64_t r = warp; r < nrows; r += nw) {
    int cnt = 0;
    for (int c0 = 0; c0 < nkt; c0 += 32) {
      const int c = c0 + lane;
      cnt += __popc(__ballot_sync(0xffffffffu, c < nkt && tile_bits[r * nkt + c] != kEmpty));
    }
    if (lane == 0) row_ptr[r + 1] = cnt;
  }
  if (threadIdx.x == 0) {
    row_ptr[0] = 0;
    carry = 0;
  }
  __syncthreads();
  for (int64_t b0 = 0; b0 < nrows; b0 += blockDim.x) {
    const int64_t r = b0 + threadIdx.x;
    int32_t tot;
    const int32_t v = r < nrows ? row_ptr[r + 1] : 0;
    const int32_t ex = block_exclusive_scan(v, warp_tot, &tot);
    if (r < nrows) row_ptr[r + 1] = carry + ex + v;
    __syncthreads();
    if (threadIdx.x == 0) carry += tot;
    __syncthreads();
  }
  // column indices; the partial flag rides in bit 30 until numbered
  for (int64_t r = warp; r < nrows; r += nw) {
    int64_t pos = row_ptr[r];
    for (int c0 = 0; c0 < nkt; c0 += 32) {
      const int c = c0 + lane;
      const int32_t st = c < nkt ? tile_bits[r * nkt + c] : kEmpty;
      const unsigned bal = __ballot_sync(0xffffffffu, st != kEmpty);
      if (st != kEmpty)
        col_idx[pos + __popc(bal & ((1u << lane) - 1u))] = c | (st == kPartial ? kPartialFlag : 0);
      pos += __popc(bal);
    }
  }
  __syncthreads();  // every state has been read; tile_bits is free
  const int64_t nnz = row_ptr[nrows];
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int64_t b0 = 0; b0 < nnz; b0 += blockDim.x) {
    const int64_t i = b0 + threadIdx.x;
    const int32_t ci = i < nnz ? col_idx[i] : 0;
    const int32_t flag = (ci & kPartialFlag) ? 1 : 0;
    int32_t tot;
    const int32_t ex = block_exclusive_scan(flag, warp_tot, &tot);
    if (i < nnz) {
      tile_bits[i] = flag ? carry + ex : -1;
      col_idx[i] = ci & ~kPartialFlag;
    }
    __syncthreads();
    if (threadIdx.x == 0) carry += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (n_partial != nullptr) *n_partial = carry;
    if (carry > bits_cap) record_status(status, dev_code(kDevCapacity, kKerBlockmask, 2));
  }
}

// E3: the 256 words of listed entry blockIdx.x, if it is a partial tile.
__global__ void __launch_bounds__(256) tile_bits_kernel(const uint8_t* __restrict__ dense,
                                                        int Sq, int Sk, int nqt, int64_t nrows,
                                                        const int32_t* __restrict__ row_ptr,
                                                        const int32_t* __restrict__ col_idx,
                                                        const int32_t* __restrict__ tile_bits,
                                                        uint64_t* __restrict__ bits,
                                                        int64_t bits_cap) {
  const int64_t i = blockIdx.x;
  if (i >= row_ptr[nrows]) return;
  const int32_t p = tile_bits[i];
  if (p < 0 || p >= bits_cap) return;
  // the row of outer tiles holding entry i: last r with row_ptr[r] <= i
  int64_t lo = 0, hi = nrows - 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) / 2;
    if (row_ptr[mid] <= i) lo = mid; else hi = mid - 1;
  }
  const int64_t n = lo / nqt;
  const int qt = static_cast<int>(lo % nqt), kt = col_idx[i];
  const int br = threadIdx.x / (kTile / kInner), bc = threadIdx.x % (kTile / kInner);
  uint64_t w = 0;
  for (int r = 0; r < kInner; ++r) {
    const int row = qt * kTile + br * kInner + r;
    if (row >= Sq) break;
    const uint8_t* src = dense + (n * Sq + row) * Sk;
    for (int c = 0; c < kInner; ++c) {
      const int col = kt * kTile + bc * kInner + c;
      if (col < Sk && src[col] != 0) w |= uint64_t(1) << (r * kInner + c);
    }
  }
  bits[int64_t(p) * 256 + threadIdx.x] = w;
}


// The tensor-core attention kernel's work order for a mask. Double item x
// (head n = x / half, j = x % half, half = ceil(pairs / 2)) holds the query-tile
// pair counted j from the top and the pair counted j from the bottom; its
// work is the number of tiles listed for those (up to four) query tiles.
// order[c], c < items: the items whose work exceeds twice the mean (w * items
// > 2 * total) first, then the others, both ascending -- a stable partition,
// so without such items the order is the identity. One CTA of 1024 threads:
// a sum, a count, then chunks of 1024 items with block-wide exclusive scans.
__device__ __forceinline__ int64_t order_work(const int32_t* row_ptr, int per_head, int nqt,
                                              int pairs, int half, int64_t x) {
  const int64_t n = x / half;
  const int j = static_cast<int>(x % half);
  const int64_t base = per_head ? n * nqt : 0;
  const int qa = 2 * (pairs - 1 - j), qb = 2 * j;
  int64_t w = 0;
  for (int t = 0; t < 2; ++t) {
    if (qa + t < nqt) w += row_ptr[base + qa + t + 1] - row_ptr[base + qa + t];
    if (qb != qa && qb + t < nqt) w += row_ptr[base + qb + t + 1] - row_ptr[base + qb + t];
  }
  return w;
}

__device__ __forceinline__ int64_t block_sum_1024(int64_t v, int64_t* sh) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();  // sh is reused by consecutive calls
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  int64_t t = 0;
  for (int w = 0; w < 32; ++w) t += sh[w];
  return t;
}

__global__ void __launch_bounds__(1024) cta_order_kernel(const int32_t* __restrict__ row_ptr,
                                                         int per_head, int nqt, int BH,
                                                         int32_t* __restrict__ order,
                                                         int64_t items) {
  __shared__ int64_t sh[32];
  __shared__ int wh[32], wl[32];
  const int pairs = (nqt + 1) / 2, half = (pairs + 1) / 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t part = 0;
  for (int64_t x = threadIdx.x; x < items; x += 1024)
    part += order_work(row_ptr, per_head, nqt, pairs, half, x);
  const int64_t total = block_sum_1024(part, sh);
  int64_t nh = 0;
  for (int64_t x = threadIdx.x; x < items; x += 1024)
    nh += order_work(row_ptr, per_head, nqt, pairs, half, x) * items > 2 * total ? 1 : 0;
  const int64_t heavy_total = block_sum_1024(nh, sh);
  int64_t heavy_base = 0, light_base = heavy_total;
  for (int64_t x0 = 0; x0 < items; x0 += 1024) {
    const int64_t x = x0 + threadIdx.x;
    const bool in = x < items;
    const bool heavy = in && order_work(row_ptr, per_head, nqt, pairs, half, x) * items > 2 * total;
    const bool light = in && !heavy;
    const unsigned bh = __ballot_sync(0xffffffffu, heavy), bl = __ballot_sync(0xffffffffu, light);
    __syncthreads();  // wh / wl of the previous chunk have been read
    if (lane == 0) {
      wh[warp] = __popc(bh);
      wl[warp] = __popc(bl);
    }
    __syncthreads();
    int ph = 0, pl = 0, th = 0, tl = 0;
    for (int w = 0; w < 32; ++w) {
      if (w < warp) {
        ph += wh[w];
        pl += wl[w];
      }
      th += wh[w];
      tl += wl[w];
    }
    const unsigned below = (1u << lane) - 1u;
    if (heavy) order[heavy_base + ph + __popc(bh & below)] = static_cast<int32_t>(x);
    if (light) order[light_base + pl + __popc(bl & below)] = static_cast<int32_t>(x);
    heavy_base += th;
    light_base += tl;
  }
}
}  // namespace

// Inputs of the analytic kernel selector, counted over the tile lists the
// attention kernels walk (STOF, Méthodologie, unified MHA module: the choice
// between the row-wise and block-wise kernels is taken from the sparsity).
// One CTA per list row (a query tile of a head); warp w takes the row's
// entries w, w + 8, ... For each entry it counts the visible (query, key)
// pairs of the tile: a full tile by the closed form of each row's causal
// limit, a partial tile (two-level mask) as the popcount of its 256 inner
// 8 x 8 words with the causal limit applied bit-wise. An entry is counted as
// listed when it holds a visible pair (the attention kernels skip the others),
// and as partial when it is also partial in the encoding. Without lists the
// row is the dense or causal range of key tiles. Counts of a list shared by
// all heads (or of no list) are multiplied by `mult` = B * H.
__global__ void __launch_bounds__(256) blockmask_counts_kernel(
    const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col_idx,
    const int32_t* __restrict__ tile_bits, const uint64_t* __restrict__ bits, int nqt, int nkt,
    int Sq, int Sk, int causal, int64_t mult, unsigned long long* counts, int* status) {
  __shared__ unsigned long long red[3][8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t lrow = blockIdx.x;          // list row: head * nqt + query tile
  const int qt = static_cast<int>(lrow % nqt);
  const int64_t shift = int64_t(Sk) - Sq;   // bottom-right causal alignment
  int beg = 0, end = nkt;
  if (row_ptr != nullptr) {
    beg = row_ptr[lrow];
    end = row_ptr[lrow + 1];
  }
  unsigned long long listed = 0, partial = 0, pairs = 0;
  for (int n = beg + warp; n < end; n += 8) {
    const int kt = row_ptr != nullptr ? col_idx[n] : n;
    if (kt < 0 || kt >= nkt) {
      if (lane == 0) record_status(status, dev_code(kDevBadList, kKerBlockmask, 3));
      continue;
    }
    const int pb = tile_bits != nullptr ? tile_bits[n] : -1;
    const int64_t k0 = int64_t(kt) * kTile;
    unsigned long long cnt = 0;
    if (pb < 0) {
      const int64_t k1 = min64(Sk, k0 + kTile);
      for (int rr = lane; rr < kTile; rr += 32) {
        const int64_t r = int64_t(qt) * kTile + rr;
        if (r >= Sq) break;
        const int64_t lim = causal ? min64(k1, r + 1 + shift) : k1;
        if (lim > k0) cnt += static_cast<unsigned long long>(lim - k0);
      }
    } else {
      const uint64_t* w = bits + int64_t(pb) * 256;
      for (int wi = lane; wi < 256; wi += 32) {
        uint64_t word = w[wi];
        if (causal) {
          // bit 8 r + c is row qt*128 + 8 rb + r, key k0 + 8 cb + c
          const int rb = wi >> 4, cb = wi & 15;
          uint64_t keep = 0;
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const int64_t last = int64_t(qt) * kTile + 8 * rb + r + shift - (k0 + 8 * cb);
            const uint64_t byte = last < 0 ? 0u : last >= 7 ? 0xffu : ((1u << (last + 1)) - 1u);
            keep |= byte << (8 * r);
          }
          word &= keep;
        }
        cnt += static_cast<unsigned long long>(__popcll(word));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (cnt > 0) {
      listed += 1;
      partial += pb >= 0 ? 1 : 0;
      pairs += cnt;
    }
  }
  if (lane == 0) {
    red[0][warp] = listed;
    red[1][warp] = partial;
    red[2][warp] = pairs;
  }
  __syncthreads();
  if (threadIdx.x < 3) {
    unsigned long long t = 0;
    for (int w = 0; w < 8; ++w) t += red[threadIdx.x][w];
    if (t != 0) atomicAdd(counts + threadIdx.x, t * static_cast<unsigned long long>(mult));
  }
}

cudaError_t launch_cta_order(const int32_t* row_ptr, int per_head, int nqt, int BH, int32_t* order,
                             int64_t items, cudaStream_t s) {
  if (items <= 0) return cudaSuccess;
  cta_order_kernel<<<1, 1024, 0, s>>>(row_ptr, per_head, nqt, BH, order, items);
  return cudaGetLastError();
}

cudaError_t launch_blockmask_counts(const int32_t* row_ptr, const int32_t* col_idx,
                                    const int32_t* tile_bits, const uint64_t* bits, int per_head,
                                    int B, int H, int Sq, int Sk, int causal, int64_t* counts,
                                    cudaStream_t s, int* status) {
  cudaError_t e = cudaMemsetAsync(counts, 0, 3 * sizeof(int64_t), s);
  if (e != cudaSuccess || Sq == 0 || Sk == 0) return e;
  const int nqt = (Sq + kTile - 1) / kTile, nkt = (Sk + kTile - 1) / kTile;
  const bool each_head = row_ptr != nullptr && per_head;
  const int64_t rows = (each_head ? int64_t(B) * H : 1) * nqt;
  const int64_t mult = each_head ? 1 : int64_t(B) * H;
  if (rows > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  blockmask_counts_kernel<<<static_cast<unsigned>(rows), 256, 0, s>>>(
      row_ptr, col_idx, tile_bits, bits, nqt, nkt, Sq, Sk, causal, mult,
      reinterpret_cast<unsigned long long*>(counts), status);
  return cudaGetLastError();
}

cudaError_t launch_blockmask_build_elements(const uint8_t* dense, int nheads, int Sq, int Sk,
                                            int32_t* row_ptr, int32_t* col_idx,
                                            int32_t* tile_bits, uint64_t* bits, int64_t bits_cap,
                                            int32_t* n_partial, cudaStream_t s, int* status) {
  const int nqt = (Sq + kTile - 1) / kTile, nkt = (Sk + kTile - 1) / kTile;
  const int64_t ntiles = int64_t(nheads) * nqt * nkt, nrows = int64_t(nheads) * nqt;
  tile_class_kernel<<<static_cast<unsigned>(ntiles), 256, 0, s>>>(dense, Sq, Sk, nqt, nkt,
                                                                   tile_bits);
  // without bitmaps (bits == nullptr) only the lists and the count are built
  two_level_lists_kernel<<<1, 1024, 0, s>>>(nrows, nkt, row_ptr, col_idx, tile_bits,
                                            bits != nullptr ? bits_cap : INT64_MAX, n_partial,
                                            status);
  if (bits != nullptr)
    tile_bits_kernel<<<static_cast<unsigned>(ntiles), 256, 0, s>>>(
        dense, Sq, Sk, nqt, nrows, row_ptr, col_idx, tile_bits, bits, bits_cap);
  return cudaGetLastError();
}

cudaError_t launch_blockmask_build(const uint8_t* dense, int nheads, int nqt, int nkt,
                                   int32_t* row_ptr, int32_t* col_idx, int64_t col_cap,
                                   cudaStream_t s, int* status) {
  blockmask_build_kernel<<<1, kThreads, 0, s>>>(dense, int64_t(nheads) * nqt, nkt, row_ptr,
                                                col_idx, col_cap, status);
  return cudaGetLastError();
}

}  // namespace rf
