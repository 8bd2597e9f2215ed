"""rf_attn_fwd on the GPU against the float64 oracle, element by element.

Shapes span several 128 x 128 tiles with ragged tails, causal alignment with
Sq != Sk (including rows that see no key), grouped-query heads, head dims 64
and 128 on the tensor-core path, and float32 on the exact SIMT path; the
block-sparse cases check the skipped-tile set bit-exactly.
"""

import numpy as np
import pytest
import torch

import oracle
from online_softmax_attention_rf_gb300 import api, inputs
from tests.helpers import assert_close, bf16_tols, f64

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Hkv, Sq, Sk, d, causal, dtype
    (1, 1, 1, 128, 128, 128, False, "bf16"),
    (1, 2, 1, 300, 300, 128, True, "bf16"),
    (2, 4, 2, 257, 513, 128, True, "bf16"),
    (1, 2, 2, 513, 257, 128, True, "bf16"),      # Sq > Sk: first rows see nothing
    (1, 8, 2, 384, 640, 64, False, "bf16"),
    (2, 3, 3, 200, 1000, 64, True, "bf16"),
    (1, 2, 2, 70, 45, 128, False, "bf16"),       # one partial tile each
    (1, 1, 1, 1, 700, 128, False, "bf16"),       # a single query row
    (1, 1, 1, 128, 128, 64, False, "f32"),
    (2, 4, 2, 150, 333, 64, True, "f32"),
    (1, 2, 1, 97, 40, 100, True, "f32"),
    (1, 1, 1, 64, 200, 256, False, "f32"),
    # the SIMT kernel's other widths: 4 keys per lane (d <= 64), 2 (d <= 128),
    # 1 (d <= 256), with ragged rows and keys, causal and grouped heads
    (1, 2, 1, 45, 300, 4, True, "f32"),
    (2, 2, 2, 130, 129, 32, False, "f32"),
    (1, 4, 2, 200, 260, 128, True, "f32"),
    (1, 1, 1, 70, 333, 160, False, "f32"),
    (1, 2, 1, 33, 190, 200, True, "f32"),
    (1, 1, 1, 9, 257, 224, False, "f32"),
]


def _run(B, H, Hkv, Sq, Sk, d, causal, dtype, seed, tile_mask=None, amp=1.0):
    q, k, v = inputs.make_qkv(B, H, Hkv, Sq, Sk, d, seed, dtype, amp)
    scale = inputs.default_scale(d)
    bm = api.BlockMask.from_dense(tile_mask) if tile_mask is not None else None
    o, lse = api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale, causal, bm)
    assert api.device_status() == 0
    o_ref, lse_ref = oracle.attention(f64(q), f64(k), f64(v), scale, causal, tile_mask)
    return o, lse, o_ref, lse_ref


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_attention_matches_oracle(cuda_device, case):
    B, H, Hkv, Sq, Sk, d, causal, dtype = case
    o, lse, o_ref, lse_ref = _run(B, H, Hkv, Sq, Sk, d, causal, dtype, seed=11)
    tol_o, tol_l = bf16_tols(o.dtype)
    assert_close(o, o_ref, tol_o, "O")
    assert_close(lse, lse_ref, tol_l, "LSE")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse_matches_oracle(cuda_device, dtype, causal):
    B, H, S, d = 1, 2, 1100, 64
    nqt = inputs.n_tiles(S)
    tm = inputs.window_random_tile_mask(nqt, window=3, frac=0.3, seed=5)
    o, lse, o_ref, lse_ref = _run(B, H, H, S, S, d, causal, dtype, 12, tm)
    tol_o, tol_l = bf16_tols(o.dtype)
    assert_close(o, o_ref, tol_o, "O")
    assert_close(lse, lse_ref, tol_l, "LSE")


def test_block_sparse_per_head_lists(cuda_device):
    B, H, Sq, Sk, d = 2, 2, 640, 900, 128
    tm = inputs.random_tile_mask(inputs.n_tiles(Sq), inputs.n_tiles(Sk), 0.4, 7, nheads=B * H)
    tm[0, 2, :] = False                                  # a query tile with no key tile
    o, lse, o_ref, lse_ref = _run(B, H, H, Sq, Sk, d, False, "bf16", 13, tm)
    assert_close(o, o_ref, 2e-2, "O")
    assert_close(lse, lse_ref, 1e-3, "LSE")


def _visited(B, H, Hkv, Sq, Sk, d, causal, dtype, tm):
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, Sq, Sk, d, 3, dtype))
    nqt, nkt = inputs.n_tiles(Sq), inputs.n_tiles(Sk)
    buf = torch.zeros(B * H * nqt * nkt, dtype=torch.uint8, device="cuda")
    api.set_debug_visited(buf)
    try:
        bm = api.BlockMask.from_dense(tm) if tm is not None else None
        api.attn_fwd(q, k, v, None, causal, bm)
        assert api.device_status() == 0
    finally:
        api.set_debug_visited(None)
    return buf.cpu().numpy().reshape(B * H, nqt, nkt).astype(bool)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("Sq,Sk,causal,use_tm", [
    (1000, 1000, True, False), (300, 900, True, False), (900, 300, True, False),
    (1100, 1100, False, True), (1100, 1100, True, True), (640, 1000, True, True)])
def test_skipped_tiles_are_exactly_the_masked_ones(cuda_device, dtype, Sq, Sk, causal, use_tm):
    tm = None
    if use_tm:
        tm = inputs.random_tile_mask(inputs.n_tiles(Sq), inputs.n_tiles(Sk), 0.35, Sq + Sk)
    got = _visited(1, 2, 1, Sq, Sk, 64, causal, dtype, tm)
    want = oracle.visited_tiles(Sq, Sk, causal, tm, 128)
    for n in range(got.shape[0]):
        assert np.array_equal(got[n], want), (n, np.argwhere(got[n] != want)[:5])


def test_no_keys_gives_zero_and_neg_inf(cuda_device):
    for dtype in (torch.bfloat16, torch.float32):
        q = torch.randn(1, 2, 5, 64, device="cuda").to(dtype)
        k = torch.empty(1, 2, 0, 64, device="cuda", dtype=dtype)
        o, lse = api.attn_fwd(q, k, k, 0.125)
        assert torch.all(o == 0) and torch.all(lse == -float("inf"))


def test_deterministic(cuda_device):
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 4, 2, 700, 700, 128, 21, "bf16"))
    o1, l1 = api.attn_fwd(q, k, v, None, True)
    o2, l2 = api.attn_fwd(q, k, v, None, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_large_score_shift(cuda_device):
    # q and k with amplitude 2.8 give scores of standard deviation ~8 (11 in
    # log2 units): the running max grows by more than 2^8 between key tiles,
    # so the in-TMEM rescale of O runs. V keeps unit amplitude so that the
    # bf16 rounding of O stays inside the tolerance.
    q, k, _ = inputs.make_qkv(1, 2, 2, 512, 1024, 64, 17, "bf16", 2.8)
    _, _, v = inputs.make_qkv(1, 2, 2, 512, 1024, 64, 18, "bf16", 1.0)
    scale = inputs.default_scale(64)
    o, lse = api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale, True)
    o_ref, lse_ref = oracle.attention(f64(q), f64(k), f64(v), scale, True)
    assert_close(o, o_ref, 2e-2, "O")
    assert_close(lse, lse_ref, 1e-3, "LSE")


def test_malformed_block_list_is_reported(cuda_device):
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 1, 1, 256, 256, 64, 1, "bf16"))
    row_ptr = torch.tensor([0, 1, 3], dtype=torch.int32, device="cuda")
    col_idx = torch.tensor([0, 1, 7], dtype=torch.int32, device="cuda")   # 7 is out of range
    bm = api.BlockMask(row_ptr, col_idx, 2, 2, 0)
    api.attn_fwd(q, k, v, None, False, bm)
    with pytest.raises(api.RFError) as e:
        api.device_status()
    assert e.value.status == api.RF_ERR_INVALID
    assert api.device_status() == 0     # reading clears it


@pytest.mark.parametrize("B,H,Hkv,Sq,Sk,d,causal,dtype,use_tm,with_lse", [
    (8, 4, 2, 300, 500, 128, True, "bf16", False, True),     # whole batch elements per chunk
    (1, 8, 8, 257, 257, 64, False, "bf16", False, True),     # one kv head per chunk
    (2, 6, 3, 200, 640, 128, True, "bf16", True, True),      # GQA + per-head block lists
    (3, 2, 1, 129, 70, 64, False, "f32", False, False),      # SIMT path, no LSE
    (2, 4, 2, 150, 0, 128, False, "bf16", False, True),      # no keys
])
def test_attn_fwd_host_equals_device(cuda_device, B, H, Hkv, Sq, Sk, d, causal, dtype, use_tm,
                                     with_lse):
    """The host-buffer entry point computes exactly what rf_attn_fwd computes:
    per-chunk launches do the same per-row work, so results are bit-identical."""
    q, k, v = inputs.make_qkv(B, H, Hkv, Sq, Sk, d, 17, dtype)
    bm = None
    if use_tm:
        tm = inputs.random_tile_mask(inputs.n_tiles(Sq), inputs.n_tiles(Sk), 0.5, 5, nheads=B * H)
        bm = api.BlockMask.from_dense(tm)
    o_d, lse_d = api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), None, causal, bm)
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o_h, lse_h = api.attn_fwd_host(qp, kp, vp, None, causal, bm, with_lse=with_lse)
    torch.cuda.current_stream().synchronize()
    assert api.device_status() == 0
    assert torch.equal(o_h, o_d.cpu())
    if with_lse:
        assert torch.equal(lse_h, lse_d.cpu())
    else:
        assert lse_h is None
