"""STOF's row-wise attention kernel and the kernel selector on the GPU.

Accelerating Sparse Transformer Inference on GPU (STOF), Méthodologie, unified
MHA module: the row-wise kernel (one warp per query row, warp shuffles, no
inter-warp synchronisation) computes the same attention as the block-wise one;
an analytic model picks between them. Every case compares with the float64
oracle (dense, causal with Sq != Sk, grouped-query heads, tile masks shared and
per head, two-level element masks, rows with no visible key, no keys at all).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from online_softmax_attention_rf_gb300 import api, inputs
from tests.helpers import TOL_BF16_LSE, TOL_BF16_O, TOL_F32, assert_close, f64

pytestmark = pytest.mark.gpu


def _tols(dtype):
    return (TOL_F32, TOL_F32) if dtype == "f32" else (TOL_BF16_O, TOL_BF16_LSE)


def _compare(B, H, Hkv, Sq, Sk, d, causal, dtype, seed, tile_mask=None, elem_mask=None):
    q, k, v = inputs.make_qkv(B, H, Hkv, Sq, Sk, d, seed, dtype)
    bm = None
    if tile_mask is not None:
        bm = api.BlockMask.from_dense(tile_mask)
    elif elem_mask is not None:
        bm = api.BlockMask.from_dense_elements(elem_mask)
    scale = 1.0 / math.sqrt(d)
    o, lse = api.attn_fwd_rowwise(q.cuda(), k.cuda(), v.cuda(), scale, causal, bm)
    assert api.device_status() == 0
    o_ref, lse_ref = oracle.attention(f64(q), f64(k), f64(v), scale, causal, tile_mask=tile_mask,
                                      elem_mask=elem_mask)
    to, tl = _tols(dtype)
    assert_close(o, o_ref, to, "O")
    assert_close(lse, lse_ref, tl, "LSE")
    return o, lse


@pytest.mark.parametrize("B,H,Hkv,Sq,Sk,d,causal,dtype", [
    (1, 2, 1, 130, 300, 64, False, "bf16"),
    (2, 4, 2, 256, 256, 128, True, "bf16"),
    (1, 1, 1, 77, 1000, 64, True, "f32"),
    (1, 2, 2, 300, 129, 128, False, "f32"),
    (2, 2, 1, 200, 520, 64, True, "bf16"),
    (1, 3, 3, 9, 5, 128, True, "bf16"),        # fewer keys than a batch of eight
])
def test_rowwise_dense_matches_oracle(cuda_device, B, H, Hkv, Sq, Sk, d, causal, dtype):
    _compare(B, H, Hkv, Sq, Sk, d, causal, dtype, Sq + Sk)


@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_rowwise_tile_masks(cuda_device, per_head, causal):
    Sq, Sk = 384, 520
    nqt, nkt = inputs.n_tiles(Sq), inputs.n_tiles(Sk)
    tm = np.asarray(inputs.random_tile_mask(nqt, nkt, 0.5, 3, nheads=4 if per_head else None))
    _compare(2, 2, 1, Sq, Sk, 64, causal, "bf16", 4, tile_mask=tm)


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 64)])
def test_rowwise_two_level_masks(cuda_device, dtype, d):
    S = 300
    em = np.stack([inputs.scattered_mask(S, 5, 3, 0.05, s) for s in range(2)])   # per head
    em[1, 17, :] = False                                                        # a row with no key
    o, lse = _compare(1, 2, 2, S, S, d, False, dtype, 6, elem_mask=em)
    assert torch.all(o[0, 1, 17].float() == 0) and torch.isinf(lse[0, 1, 17])


def test_rowwise_two_level_causal_shared(cuda_device):
    S = 260
    em = inputs.scattered_mask(S, 8, 4, 0.1, 9)
    _compare(2, 2, 1, S, S, 64, True, "bf16", 7, elem_mask=em)


def test_rowwise_no_keys(cuda_device):
    q = torch.randn(1, 2, 5, 64, device="cuda").to(torch.bfloat16)
    k = torch.empty(1, 2, 0, 64, device="cuda", dtype=torch.bfloat16)
    o, lse = api.attn_fwd_rowwise(q, k, k)
    assert api.device_status() == 0
    assert torch.all(o.float() == 0) and torch.all(torch.isinf(lse)) and torch.all(lse < 0)


def test_rowwise_equals_blockwise_on_a_tile_mask(cuda_device):
    """Both kernels on the same inputs: equal within the bf16 output bound
    (the block kernel rounds P to bf16 before P.V, the row kernel does not)."""
    Sq = Sk = 512
    tm = np.asarray(inputs.random_tile_mask(4, 4, 0.6, 2))
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 4, 2, Sq, Sk, 128, 3, "bf16"))
    bm = api.BlockMask.from_dense(tm)
    o1, l1 = api.attn_fwd(q, k, v, None, True, bm)
    o2, l2 = api.attn_fwd_rowwise(q, k, v, None, True, bm)
    assert api.device_status() == 0
    assert (o1.float() - o2.float()).abs().max().item() <= 2 * TOL_BF16_O
    fin = torch.isfinite(l1)
    assert torch.equal(fin, torch.isfinite(l2))
    assert (l1[fin] - l2[fin]).abs().max().item() <= 2 * TOL_BF16_LSE


def test_auto_selection_and_full_size_sampled(cuda_device):
    """The scattered short-sequence workload at full size: the selector picks
    the block-wise kernel (the faster one on GB300 at this size), and sampled
    rows of both kernels match the oracle."""
    w = inputs.WORKLOADS["scattered_short"]
    q, k, v, scale, extras = inputs.workload_inputs("scattered_short")
    em = extras["elem_mask"]
    bm = api.BlockMask.from_dense_elements(em)
    counts = api.selector_counts(w["B"], w["H"], w["Sq"], w["Sk"], False, bm)
    assert api.choose_kernel(w["B"], w["H"], w["Sq"], w["Sk"], w["d"], *counts) == \
        api.RF_KERNEL_BLOCKWISE
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_auto, l_auto = api.attn_fwd(qd, kd, vd, scale, False, bm, kernel="auto")
    o_row, l_row = api.attn_fwd_rowwise(qd, kd, vd, scale, False, bm)
    o_blk, l_blk = api.attn_fwd(qd, kd, vd, scale, False, bm)
    assert api.device_status() == 0
    assert torch.equal(o_auto, o_blk) and torch.equal(l_auto, l_blk)
    rows = sorted(set(np.random.default_rng(0).choice(w["Sq"], 48, replace=False).tolist()
                      + [0, w["n_global"] - 1, w["n_global"], w["Sq"] - 1]))
    for b, h in [(0, 0), (15, 15)]:
        o_ref, lse_ref = oracle.attention(f64(q[b:b + 1, h:h + 1]), f64(k[b:b + 1, h:h + 1]),
                                          f64(v[b:b + 1, h:h + 1]), scale, False, rows=rows,
                                          elem_mask=em)
        for o, lse, name in ((o_row, l_row, "row"), (o_blk, l_blk, "block")):
            assert_close(o[b, h, rows], o_ref[0, 0], TOL_BF16_O, "%s O" % name)
            assert_close(lse[b, h, rows], lse_ref[0, 0], TOL_BF16_LSE, "%s LSE" % name)


def test_auto_selection_tiny_picks_rowwise(cuda_device):
    """One head of 256 tokens under a highly sparse mask: "auto" runs the
    row-wise kernel (bit-identical to calling it) and matches the oracle."""
    em = inputs.scattered_mask(256, 4, 2, 0.002, 3)
    q, k, v = inputs.make_qkv(1, 1, 1, 256, 256, 64, 12, "bf16")
    bm = api.BlockMask.from_dense_elements(em)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_auto, l_auto = api.attn_fwd(qd, kd, vd, None, False, bm, kernel="auto")
    o_row, l_row = api.attn_fwd_rowwise(qd, kd, vd, None, False, bm)
    assert api.device_status() == 0
    assert torch.equal(o_auto, o_row) and torch.equal(l_auto, l_row)
    o_ref, lse_ref = oracle.attention(f64(q), f64(k), f64(v), 1 / 8, False, elem_mask=em)
    assert_close(o_row, o_ref, TOL_BF16_O, "O")
    assert_close(l_row, lse_ref, TOL_BF16_LSE, "LSE")
