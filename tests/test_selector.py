"""The analytic kernel selector (host logic, no GPU).

STOF, Méthodologie, unified MHA module, kernel selection: the row-wise kernel
for highly sparse masks on short sequences, the block-wise kernel otherwise.
rf_attn_choose_kernel / rf_attn_estimate_us are pure host functions of the
library. Their inputs (listed tiles, partial tiles, visible pairs) come from
rf_blockmask_counts on the device; here they are counted by enumeration, and
tests/test_gpu_selector.py checks the device counts against the same
enumeration.
"""

import numpy as np
import pytest

from online_softmax_attention_rf_gb300 import api, build, inputs


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    api.lib()


def brute_counts(B, H, Sq, Sk, causal, em):
    """Counts by enumerating tiles (em [nh, Sq, Sk] after any causal limit)."""
    listed = partial = 0
    for hm in em:
        for qt in range(-(-Sq // 128)):
            for kt in range(-(-Sk // 128)):
                blk = hm[qt * 128:(qt + 1) * 128, kt * 128:(kt + 1) * 128]
                if blk.any():
                    listed += 1
                    partial += int(not blk.all())
    scale = B * H if em.shape[0] == 1 else 1
    return listed * scale, partial * scale, int(em.sum()) * scale


def test_invalid_arguments():
    assert api.lib().rf_attn_choose_kernel(0, 1, 1, 1, 64, 1, 0, 1, 152) == -1
    assert api.lib().rf_attn_choose_kernel(1, 1, 1, 1, 96, 1, 0, 1, 152) == -1
    assert api.lib().rf_attn_choose_kernel(1, 1, 1, 1, 64, 1, 2, 1, 152) == -1   # partial > listed
    assert api.lib().rf_attn_choose_kernel(1, 1, 1, 1, 64, 1, 0, 1, 0) == -1
    with pytest.raises(api.RFError):
        api.estimate_us(1, 1, 1, 1, 64, -1, 0, 1, 152)


def test_long_dense_and_block_sparse_pick_the_block_kernel():
    for name in ("mha_prefill", "gqa_long", "block_sparse"):
        w = inputs.WORKLOADS[name]
        B, H, S, d = w["B"], w["H"], w["Sq"], w["d"]
        nqt = inputs.n_tiles(S)
        if name == "block_sparse":
            tm = inputs.window_random_tile_mask(nqt, w["window"], w["frac"], w["seed"])
            listed, visible = int(tm.sum()) * B * H, int(tm.sum()) * 128 * 128 * B * H
        else:
            listed = nqt * (nqt + 1) // 2 * B * H
            visible = S * (S + 1) // 2 * B * H
        assert api.choose_kernel(B, H, S, S, d, listed, 0, visible, 152) == \
            api.RF_KERNEL_BLOCKWISE, name


def test_scattered_short_workload_picks_the_block_kernel():
    """At 1024 tokens and 256 heads the tensor-core kernel is the faster one
    on GB300 (0.19 ms against 0.93 ms for the row-wise kernel)."""
    w = inputs.WORKLOADS["scattered_short"]
    em = inputs.scattered_mask(w["Sq"], w["window"], w["n_global"], w["density"], w["seed"])
    counts = brute_counts(w["B"], w["H"], w["Sq"], w["Sk"], False, em[None])
    assert api.choose_kernel(w["B"], w["H"], w["Sq"], w["Sk"], w["d"], *counts, num_sms=152) == \
        api.RF_KERNEL_BLOCKWISE


def test_tiny_scattered_masks_pick_the_row_kernel():
    """A highly sparse mask on a short sequence with one head: the block-wise
    kernel would run one CTA on one of 152 SMs; the model picks row-wise."""
    em = inputs.scattered_mask(256, 4, 2, 0.002, 3)
    counts = brute_counts(1, 1, 256, 256, False, em[None])
    assert api.choose_kernel(1, 1, 256, 256, 64, *counts, num_sms=152) == api.RF_KERNEL_ROWWISE


def test_estimates_are_monotone():
    base = dict(B=8, H=16, Sq=2048, Sk=2048, d=64)
    b0, r0 = api.estimate_us(*base.values(), 1000, 0, 10 ** 7, 152)
    b1, r1 = api.estimate_us(*base.values(), 2000, 0, 10 ** 7, 152)
    b2, r2 = api.estimate_us(*base.values(), 2000, 1000, 2 * 10 ** 7, 152)
    assert b1 > b0 and r1 > r0          # more listed tiles: both slower
    assert b2 > b1 and r2 > r1          # partial tiles and more pairs
    b3, r3 = api.estimate_us(*base.values(), 2000, 0, 10 ** 7, 76)
    assert b3 >= b1 and r3 > r1         # fewer SMs
