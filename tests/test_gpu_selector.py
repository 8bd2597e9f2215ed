"""The kernel selector's inputs counted on the device (rf_blockmask_counts).

STOF, Méthodologie, unified MHA module: the row-wise / block-wise choice is
taken from the mask's sparsity. The device counts (listed tiles holding a
visible pair, partial tiles among them, visible pairs) must equal an
enumeration of the mask, for dense, causal, tile-level and two-level masks,
shared and per head, with ragged edges.
"""

import numpy as np
import pytest
import torch

from online_softmax_attention_rf_gb300 import api, inputs
from tests.test_selector import brute_counts

pytestmark = pytest.mark.gpu


def _causal(Sq, Sk, causal):
    if not causal:
        return np.ones((Sq, Sk), dtype=bool)
    return np.arange(Sk)[None, :] <= np.arange(Sq)[:, None] + (Sk - Sq)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq,Sk", [(300, 420), (420, 300), (128, 128), (1000, 1000)])
def test_element_mask_counts(cuda_device, causal, Sq, Sk):
    rng = np.random.default_rng(Sq + Sk)
    em = rng.random((2, Sq, Sk)) < 0.01
    em[:, :128, :128] = True                            # one full tile per head
    em[1, -5:, -7:] = True                              # a ragged corner
    bm = api.BlockMask.from_dense_elements(em)
    got = api.selector_counts(1, 2, Sq, Sk, causal, bm)
    vis = em & _causal(Sq, Sk, causal)[None]
    listed, _, pairs = brute_counts(1, 2, Sq, Sk, causal, vis)
    # partial: listed after the causal limit and partial in the encoding
    nqt, nkt = -(-Sq // 128), -(-Sk // 128)
    partial = 0
    for h in range(2):
        for qt in range(nqt):
            for kt in range(nkt):
                rs, cs = slice(qt * 128, (qt + 1) * 128), slice(kt * 128, (kt + 1) * 128)
                if vis[h, rs, cs].any() and not em[h, rs, cs].all():
                    partial += 1
    assert got == (listed, partial, pairs)
    assert api.device_status() == 0


@pytest.mark.parametrize("causal", [False, True])
def test_tile_mask_counts_shared_and_per_head(cuda_device, causal):
    Sq, Sk = 300, 700
    rng = np.random.default_rng(5)
    tm = rng.random((3, 6)) < 0.5
    # tile-level lists have no inner level: no tile is partial in the
    # encoding (the causal element mask inside a listed tile costs nothing)
    full = np.repeat(np.repeat(tm, 128, 0), 128, 1)[:Sq, :Sk] & _causal(Sq, Sk, causal)
    got = api.selector_counts(2, 3, Sq, Sk, causal, api.BlockMask.from_dense(tm))
    listed, _, pairs = brute_counts(2, 3, Sq, Sk, causal, full[None])
    assert got == (listed, 0, pairs)
    tmh = rng.random((6, 3, 6)) < 0.4
    fullh = np.repeat(np.repeat(tmh, 128, 1), 128, 2)[:, :Sq, :Sk] & _causal(Sq, Sk, causal)
    got = api.selector_counts(2, 3, Sq, Sk, causal, api.BlockMask.from_dense(tmh))
    listed, _, pairs = brute_counts(2, 3, Sq, Sk, causal, fullh)
    assert got == (listed, 0, pairs)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq,Sk", [(300, 420), (4096, 4096), (1, 65536)])
def test_dense_counts(cuda_device, causal, Sq, Sk):
    got = api.selector_counts(4, 8, Sq, Sk, causal)
    vis = _causal(Sq, Sk, causal)
    nqt, nkt = -(-Sq // 128), -(-Sk // 128)
    listed = sum(bool(vis[qt * 128:(qt + 1) * 128, kt * 128:(kt + 1) * 128].any())
                 for qt in range(nqt) for kt in range(nkt))
    assert got == (listed * 32, 0, int(vis.sum()) * 32)


def test_workload_counts(cuda_device):
    """The scattered_short workload: device counts equal the enumeration, and
    the selector picks the block-wise kernel there."""
    w = inputs.WORKLOADS["scattered_short"]
    em = inputs.scattered_mask(w["Sq"], w["window"], w["n_global"], w["density"], w["seed"])
    bm = api.BlockMask.from_dense_elements(em)
    got = api.selector_counts(w["B"], w["H"], w["Sq"], w["Sk"], False, bm)
    assert got == brute_counts(w["B"], w["H"], w["Sq"], w["Sk"], False, em[None])
    assert api.choose_kernel(w["B"], w["H"], w["Sq"], w["Sk"], w["d"], *got) == \
        api.RF_KERNEL_BLOCKWISE


def test_empty_and_bad_lists(cuda_device):
    assert api.selector_counts(1, 1, 0, 100, False) == (0, 0, 0)
    # an out-of-range tile index is skipped and reported on the device
    row_ptr = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
    col_idx = torch.tensor([0, 5], dtype=torch.int32, device="cuda")
    bm = api.BlockMask(row_ptr, col_idx, 1, 2, 0)
    got = api.selector_counts(1, 1, 128, 256, False, bm)
    assert got == (1, 0, 128 * 128)
    with pytest.raises(api.RFError) as e:
        api.device_status()
    assert e.value.status == api.RF_ERR_INVALID
    assert api.device_status() == 0     # reading clears it
