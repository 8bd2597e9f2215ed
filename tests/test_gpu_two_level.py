"""Two-level (outer tile lists + inner 8x8 bitmaps) masks on the GPU.

Accelerating Sparse Transformer Inference on GPU (STOF), Méthodologie, unified
MHA module, two-level storage format: outer tiles are listed in BSR rows and
marked full or partial; the valid elements of a partial tile are one 64-bit
bitmap per 8x8 inner block. The device encoder (rf_blockmask_build_elements)
must produce exactly the oracle's encoding, and attention under the encoded
mask must equal the oracle's attention under the dense element mask.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from online_softmax_attention_rf_gb300 import api, inputs
from tests.helpers import TOL_BF16_LSE, TOL_BF16_O, TOL_F32, assert_close, f64

pytestmark = pytest.mark.gpu


def _element_mask(nheads, Sq, Sk, seed):
    """Random element mask with empty, full and partial outer tiles, and
    inner blocks that are empty, full and mixed."""
    rng = np.random.default_rng(seed)
    m = np.zeros((nheads, Sq, Sk), dtype=bool)
    nqt, nkt = -(-Sq // 128), -(-Sk // 128)
    for h in range(nheads):
        for qt in range(nqt):
            for kt in range(nkt):
                kind = rng.integers(0, 4)           # 0 empty, 1 full, 2-3 partial
                rs = slice(qt * 128, (qt + 1) * 128)
                cs = slice(kt * 128, (kt + 1) * 128)
                if kind == 1:
                    m[h, rs, cs] = True
                elif kind >= 2:
                    blk = m[h, rs, cs]
                    inner = rng.random((16, 16)) < 0.5       # which 8x8 blocks are touched
                    dense = rng.random(blk.shape) < rng.choice([0.2, 0.7])
                    sel = np.repeat(np.repeat(inner, 8, 0), 8, 1)[:blk.shape[0], :blk.shape[1]]
                    blk[:] = dense & sel
    return m


@pytest.mark.parametrize("nheads,Sq,Sk", [(1, 256, 384), (3, 300, 200), (2, 129, 1000)])
def test_device_encoder_matches_oracle(cuda_device, nheads, Sq, Sk):
    m = _element_mask(nheads, Sq, Sk, nheads * 1000 + Sq)
    bm = api.BlockMask.from_dense_elements(m)
    assert api.device_status() == 0
    rp, ci, tb, bits = oracle.two_level_encode(m)
    got_rp = bm.row_ptr.cpu().numpy()
    assert np.array_equal(got_rp, rp)
    nnz = int(rp[-1])
    assert np.array_equal(bm.col_idx.cpu().numpy()[:nnz], ci)
    assert np.array_equal(bm.tile_bits.cpu().numpy()[:nnz], tb)
    got_bits = bm.bits.cpu().numpy().view(np.uint64)[:bits.shape[0]]
    assert np.array_equal(got_bits, bits)


def _run(B, H, Hkv, Sq, Sk, d, causal, dtype, m, seed):
    q, k, v = inputs.make_qkv(B, H, Hkv, Sq, Sk, d, seed, dtype)
    bm = api.BlockMask.from_dense_elements(m)
    o, lse = api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), None, causal, bm)
    assert api.device_status() == 0
    o_ref, lse_ref = oracle.attention(f64(q), f64(k), f64(v), 1.0 / math.sqrt(d), causal,
                                      elem_mask=m)
    return o, lse, o_ref, lse_ref


@pytest.mark.parametrize("B,H,Hkv,Sq,Sk,d,causal,dtype,per_head", [
    (1, 2, 1, 384, 384, 128, False, "bf16", True),
    (2, 2, 2, 300, 520, 64, True, "bf16", True),
    (1, 4, 2, 256, 256, 128, True, "bf16", False),
    (1, 2, 2, 200, 260, 64, False, "f32", True),
    (1, 1, 1, 130, 300, 32, True, "f32", False),
])
def test_two_level_attention_matches_oracle(cuda_device, B, H, Hkv, Sq, Sk, d, causal, dtype,
                                            per_head):
    m = _element_mask(B * H if per_head else 1, Sq, Sk, Sq + Sk + d)
    if not per_head:
        m = m[0]
    o, lse, o_ref, lse_ref = _run(B, H, Hkv, Sq, Sk, d, causal, dtype, m, 7)
    if dtype == "f32":
        assert_close(o, o_ref, TOL_F32, "O")
        assert_close(lse, lse_ref, TOL_F32, "LSE")
    else:
        assert_close(o, o_ref, TOL_BF16_O, "O")
        assert_close(lse, lse_ref, TOL_BF16_LSE, "LSE")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_rows_masked_out_by_bitmaps(cuda_device, dtype):
    """Rows whose every key is removed by the inner bitmaps get O = 0 and
    LSE = -inf even though their outer tiles are listed."""
    Sq, Sk, d = 256, 256, 64
    m = np.ones((Sq, Sk), dtype=bool)
    m[5, :] = False                      # one row sees nothing
    m[130:140, :] = False                # ten rows of the second query tile
    m[200, 3] = False                    # a single element
    o, lse, o_ref, lse_ref = _run(1, 2, 1, Sq, Sk, d, False, dtype, m, 9)
    tol = (TOL_F32, TOL_F32) if dtype == "f32" else (TOL_BF16_O, TOL_BF16_LSE)
    assert_close(o, o_ref, tol[0], "O")
    assert_close(lse, lse_ref, tol[1], "LSE")
    for r in [5, 130, 139]:
        assert torch.all(o[:, :, r].float() == 0)
        assert torch.all(torch.isinf(lse[:, :, r])) and torch.all(lse[:, :, r] < 0)


def test_whole_tiles_equal_the_tile_mask_path(cuda_device):
    """An element mask made of whole tiles lists only full tiles and gives
    bit-identical results to the outer-level (tile) mask of the same tiles."""
    Sq = Sk = 512
    tm = inputs.random_tile_mask(4, 4, 0.5, 3, nheads=2)
    em = np.repeat(np.repeat(np.asarray(tm, bool), 128, 1), 128, 2)
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 2, 2, Sq, Sk, 128, 5, "bf16"))
    bm2 = api.BlockMask.from_dense_elements(em)
    assert (bm2.tile_bits[:int(bm2.row_ptr[-1])] == -1).all()
    o2, l2 = api.attn_fwd(q, k, v, None, True, bm2)
    o1, l1 = api.attn_fwd(q, k, v, None, True, api.BlockMask.from_dense(tm))
    assert api.device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
