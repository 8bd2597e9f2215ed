// attn_select.cu -- the analytic choice between the block-wise (tensor-core)
// and the row-wise attention kernels.
//
// Accelerating Sparse Transformer Inference on GPU (STOF), Méthodologie,
// unified MHA module, kernel selection: an analytic model picks the row-wise
// or the block-wise kernel from the mask's sparsity and the sequence length.
// Here both kernels' times are estimated from the work each one does and the
// way it fills the GPU:
//   block-wise: a CTA per pair of query-tile pairs; a CTA's time is its share
//     of the listed 128 x 128 tiles (a partial tile costing more: its inner
//     bitmaps are applied element by element) plus a cost per work item;
//     CTAs run in waves of one per SM, so short sequences leave SMs idle;
//   row-wise: a warp per query row; each visible (query, key) pair costs a
//     fixed amount of SM time (in proportion to d), plus a cost per row and
//     per (row, listed tile) visit; the work spreads over all SMs.
// The constants were fitted by non-negative least squares to 62 timings of
// both kernels on GB300 (sequences of 128 to 4096, 1 to 256 heads, d 64 and
// 128, dense causal, tile masks, and scattered element masks of density 0.2
// to 5 %), each timed from the host call (so the fixed terms include the call
// overhead): median relative error 2 % (block-wise) and 7 % (row-wise). The
// choice matches the faster measured kernel in 49 of the 62 cases; the other
// 13 are launch-bound sizes (at most 256 tokens and 16 heads) where the two
// kernels are within 15 % of each other. On GB300 the tensor-core kernel is
// the faster one from 512 tokens or 64 heads up, by 2 to 70 times.
#include <cmath>

#include "rf_internal.h"

namespace {

// block-wise: fixed seconds per call, per listed full / partial tile of a
// CTA, and per work item of a CTA
constexpr double kBlockFixed = 25.05e-6;
constexpr double kBlockTile = 0.819e-6;
constexpr double kBlockPartialTile = 1.165e-6;
constexpr double kBlockItem = 4.316e-6;
// row-wise: fixed seconds per call; SM-seconds per visible pair (d = 64), per
// row, and per (row, listed tile) visit
constexpr double kRowFixed = 30.90e-6;
constexpr double kRowPair = 4.04e-9;
constexpr double kRowRow = 1.226e-7;
constexpr double kRowVisit = 2.478e-8;

}  // namespace

namespace rf {

bool attn_estimate(int B, int H, int Sq, int Sk, int d, int64_t listed_tiles,
                   int64_t partial_tiles, int64_t visible_pairs, int num_sms, double* t_block,
                   double* t_row) {
  if (B < 1 || H < 1 || Sq < 1 || Sk < 0 || (d != 64 && d != 128) || listed_tiles < 0 ||
      partial_tiles < 0 || partial_tiles > listed_tiles || visible_pairs < 0 || num_sms < 1)
    return false;
  const double heads = double(B) * H;
  const int64_t nqt = (int64_t(Sq) + 127) / 128;
  const int64_t pairs = (nqt + 1) / 2;
  const double ctas = heads * double((pairs + 1) / 2);
  const double items_per_cta = pairs > 1 ? 2.0 : 1.0;
  const double waves = std::ceil(ctas / num_sms);
  const double full = double(listed_tiles - partial_tiles), part = double(partial_tiles);
  // a CTA's time: its share of the listed tiles (both query tiles of an
  // item counted) plus the items' start and epilogue
  const double per_cta = (full * kBlockTile + part * kBlockPartialTile) / ctas +
                         items_per_cta * kBlockItem;
  *t_block = kBlockFixed + waves * per_cta;
  const double rows = heads * Sq;
  const double visits = double(listed_tiles) * 128.0;  // rows of a tile walk its list
  *t_row = kRowFixed + (double(visible_pairs) * kRowPair * (d / 64.0) + rows * kRowRow +
                        visits * kRowVisit) / num_sms;
  return true;
}

}  // namespace rf

extern "C" int rf_attn_choose_kernel(int B, int H, int Sq, int Sk, int d, int64_t listed_tiles,
                                     int64_t partial_tiles, int64_t visible_pairs, int num_sms) {
  double tb = 0.0, tr = 0.0;
  if (!rf::attn_estimate(B, H, Sq, Sk, d, listed_tiles, partial_tiles, visible_pairs, num_sms,
                         &tb, &tr))
    return -1;
  return tr < tb ? RF_KERNEL_ROWWISE : RF_KERNEL_BLOCKWISE;
}

extern "C" int rf_attn_estimate_us(int B, int H, int Sq, int Sk, int d, int64_t listed_tiles,
                                   int64_t partial_tiles, int64_t visible_pairs, int num_sms,
                                   double* block_us, double* row_us) {
  double tb = 0.0, tr = 0.0;
  if (block_us == nullptr || row_us == nullptr ||
      !rf::attn_estimate(B, H, Sq, Sk, d, listed_tiles, partial_tiles, visible_pairs, num_sms,
                         &tb, &tr))
    return RF_ERR_INVALID;
  *block_us = tb * 1e6;
  *row_us = tr * 1e6;
  return RF_OK;
}
