"""The tensor-core kernel's work order for a mask (rf_blockmask_cta_order).

A mask whose query tiles differ a lot in listed tiles (global query rows that
attend to every key, as in STOF's sparse patterns) leaves one long CTA per
head; the order moves those double items to the front. The order must be the
stable partition an enumeration of the lists gives, and the attention output
must not depend on it (each work item computes the same rows either way).
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from online_softmax_attention_rf_gb300 import api, inputs
from tests.helpers import TOL_BF16_LSE, TOL_BF16_O, assert_close, f64

pytestmark = pytest.mark.gpu


def _expected_order(row_ptr, per_head, nqt, B, H):
    """Double items whose listed tiles exceed twice the mean first, then the
    rest, both ascending -- from the lists, in Python integers."""
    pairs = (nqt + 1) // 2
    half = (pairs + 1) // 2
    rp = [int(x) for x in row_ptr]
    work = []
    for x in range(B * H * half):
        n, j = divmod(x, half)
        base = n * nqt if per_head else 0
        qs = {2 * (pairs - 1 - j), 2 * (pairs - 1 - j) + 1, 2 * j, 2 * j + 1}
        work.append(sum(rp[base + q + 1] - rp[base + q] for q in qs if q < nqt))
    total, items = sum(work), len(work)
    heavy = [x for x in range(items) if work[x] * items > 2 * total]
    light = [x for x in range(items) if work[x] * items <= 2 * total]
    return heavy + light, heavy


def _global_band_mask(S, band, glob, nheads=None):
    """[S, S] (shared lists), or [nheads, S, S] (lists per head)."""
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    m = (np.abs(i - j) <= band) | (j < glob) | (i < glob)
    return m if nheads is None else np.broadcast_to(m, (nheads, S, S)).copy()


@pytest.mark.parametrize("per_head", [False, True])
def test_order_is_the_stable_partition(cuda_device, per_head):
    B, H, S = 2, 3, 4096
    em = _global_band_mask(S, 64, 16, B * H if per_head else None)
    if per_head:
        em[4, 2000:2010, :] = True               # one head with a second long query tile
    bm = api.BlockMask.from_dense_elements(em)
    order = bm.cta_order(B, H, S).cpu().numpy()
    expect, heavy = _expected_order(bm.row_ptr.cpu().numpy(), bm.per_head, bm.nqt, B, H)
    assert len(heavy) > 0                        # the global rows make the pair of tile 0 long
    assert order.tolist() == expect
    assert sorted(order.tolist()) == list(range(len(expect)))


def test_order_is_identity_without_long_items(cuda_device):
    B, H, S = 1, 4, 1536
    tm = np.asarray(inputs.random_tile_mask(S // 128, S // 128, 0.5, 3))   # shared lists
    bm = api.BlockMask.from_dense(tm)
    expect, heavy = _expected_order(bm.row_ptr.cpu().numpy(), bm.per_head, bm.nqt, B, H)
    assert not heavy
    assert bm.cta_order(B, H, S).cpu().numpy().tolist() == list(range(len(expect)))
    # the library writes every entry
    n = int(api.lib().rf_blockmask_cta_order_len(B, H, S))
    order = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    st = bm.as_struct()
    api._check(api.lib().rf_blockmask_cta_order(ctypes.byref(st), B, H, S, api._ptr(order), n,
                                                api._stream()))
    assert order.cpu().numpy().tolist() == expect == list(range(n))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_attention_does_not_depend_on_the_order(cuda_device, causal, d):
    B, H, Hkv, S = 1, 2, 1, 4096
    em = _global_band_mask(S, 64, 24)
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, S, S, d, 7 + d, "bf16"))
    scale = inputs.default_scale(d)
    bm = api.BlockMask.from_dense_elements(em)
    assert len(_expected_order(bm.row_ptr.cpu().numpy(), 0, bm.nqt, B, H)[1]) > 0
    o1, l1 = api.attn_fwd(q, k, v, scale, causal, bm)            # in the mask's order
    o2 = torch.empty_like(q)
    l2 = torch.empty(B, H, S, dtype=torch.float32, device="cuda")
    plain = bm.as_struct()                                       # head-major order
    api._check(api.lib().rf_attn_fwd(api._ptr(q), api._ptr(k), api._ptr(v), api._ptr(o2),
                                     api._ptr(l2), B, H, Hkv, S, S, d, float(scale),
                                     1 if causal else 0, ctypes.byref(plain), api.RF_BF16,
                                     api._stream()))
    assert api.device_status() == 0
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)
    # and both equal the definition
    o_ref, lse_ref = oracle.attention(f64(q), f64(k), f64(v), scale, causal, elem_mask=em)
    assert_close(o1, o_ref, TOL_BF16_O, "O")
    assert_close(l1, lse_ref, TOL_BF16_LSE, "LSE")


def test_order_entry_out_of_range_is_reported(cuda_device):
    B, H, S = 1, 1, 512
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, H, S, S, 64, 5, "bf16"))
    bm = api.BlockMask.from_dense(np.ones((S // 128, S // 128), dtype=bool))
    n = int(api.lib().rf_blockmask_cta_order_len(B, H, S))
    bad = torch.full((n,), n + 3, dtype=torch.int32, device="cuda")
    bm.cta_orders[(B, H, S)] = bad
    api.attn_fwd(q, k, v, None, False, bm)
    with pytest.raises(api.RFError) as e:
        api.device_status()
    assert e.value.status == api.RF_ERR_INVALID
    assert api.device_status() == 0
