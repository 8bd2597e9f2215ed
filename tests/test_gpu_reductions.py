"""Split-K decode, the log-sum-exp merge, row softmax and the block-list build
on the GPU against the float64 oracle."""

import math

import numpy as np
import pytest
import torch

import oracle
from online_softmax_attention_rf_gb300 import api, inputs
from tests.helpers import (TOL_BF16_LSE, TOL_BF16_O, TOL_BF16_SOFTMAX, TOL_F32, assert_close,
                           f64)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,Hkv,Sk,d,nsplit", [
    (2, 8, 2, 5000, 128, 7),       # G = 4, ragged last split
    (1, 4, 4, 3000, 128, 3),       # G = 1 (padded to 4)
    (2, 16, 2, 4096, 64, 16),      # G = 8, d = 64
    (1, 16, 1, 999, 128, 5),       # G = 16
    (1, 2, 1, 100, 64, 100),       # one key per split
    (3, 6, 2, 130, 128, 1),        # G = 3, a single split
])
def test_decode_matches_oracle(cuda_device, B, H, Hkv, Sk, d, nsplit):
    q, k, v = inputs.make_qkv(B, H, Hkv, 1, Sk, d, 31, "bf16")
    scale = inputs.default_scale(d)
    ws_bytes = api.decode_workspace_bytes(B, H, nsplit, d)
    ws = torch.empty(ws_bytes // 4, dtype=torch.float32, device="cuda")
    o, lse = api.attn_decode_splitk(q.cuda(), k.cuda(), v.cuda(), nsplit, scale, ws)
    assert api.device_status() == 0
    # the merged result equals the unsplit definition ...
    o_ref, lse_ref = oracle.attention(f64(q), f64(k), f64(v), scale)
    assert_close(o, o_ref, TOL_BF16_O, "O")
    assert_close(lse, lse_ref, TOL_BF16_LSE, "LSE")
    # ... and the stored partials equal the per-split definition
    n = B * H * nsplit
    op_ref, lp_ref = oracle.decode_partials(f64(q), f64(k), f64(v), scale, nsplit)
    assert_close(ws[:n * d].view(B, H, nsplit, d), op_ref, 5e-3, "O_s")
    assert_close(ws[n * d:n * d + n].view(B, H, nsplit), lp_ref, TOL_BF16_LSE, "lse_s")


def test_decode_split_count_does_not_change_the_result(cuda_device):
    q, k, v = (t.cuda() for t in inputs.make_qkv(2, 8, 2, 1, 8192, 128, 32, "bf16"))
    o1, l1 = api.attn_decode_splitk(q, k, v, 1)
    for ns in (2, 8, 32, 128):
        o, l = api.attn_decode_splitk(q, k, v, ns)
        assert_close(o, f64(o1), TOL_BF16_O, "O nsplit=%d" % ns)
        assert_close(l, f64(l1), TOL_BF16_LSE, "LSE nsplit=%d" % ns)


def test_decode_equals_prefill_row(cuda_device):
    # FlashDecoding and FlashAttention are special cases of one form: the
    # decode of one query row equals the prefill kernel on that row
    q, k, v = (t.cuda() for t in inputs.make_qkv(2, 8, 2, 1, 3000, 128, 33, "bf16"))
    od, ld = api.attn_decode_splitk(q, k, v, 6)
    op, lp = api.attn_fwd(q, k, v)
    assert_close(od, f64(op), TOL_BF16_O, "O")
    assert_close(ld, f64(lp), TOL_BF16_LSE, "LSE")


def _partials(rows, nsplit, d, seed):
    rng = np.random.default_rng(seed)
    o_part = rng.standard_normal((rows, nsplit, d)).astype(np.float32)
    lse_part = (rng.standard_normal((rows, nsplit)) * 3).astype(np.float32)
    lse_part[1, 3] = -np.inf                   # an empty split
    lse_part[2, :] = -np.inf                   # a row with nothing at all
    lse_part[3, :] += 80.0                     # large values must not overflow
    return o_part, lse_part


@pytest.mark.parametrize("rows,nsplit,d", [
    (5, 4, 64), (37, 32, 128), (9, 7, 100), (4, 130, 33),
    # rows wider than 128 columns: four 128-column chunks per warp, four live
    # splits per round of loads (partial chunk groups at 260 and 1000)
    (6, 16, 512), (5, 9, 260), (4, 40, 1024), (7, 5, 1000),
    (5, 6, 513),              # no float4 access: 32-column chunks
])
def test_merge_matches_oracle(cuda_device, rows, nsplit, d):
    o_part, lse_part = _partials(rows, nsplit, d, rows)
    o, lse = api.splitk_merge(torch.from_numpy(o_part).cuda(), torch.from_numpy(lse_part).cuda(),
                              torch.float32)
    o_ref, lse_ref = oracle.merge_partials(o_part, lse_part)
    assert_close(o, o_ref, TOL_F32, "O")
    # rows with |LSE| of order 1-10 at 1e-5 absolute; row 3 (every split
    # shifted by +80, |LSE| ~ 90, where one float32 ulp is 7.6e-6) at 1e-5
    # relative to |LSE|
    small = np.ones(rows, dtype=bool)
    small[3] = False
    assert_close(lse.cpu()[torch.from_numpy(small)], lse_ref[small], TOL_F32, "LSE")
    assert_close(lse.cpu()[3:4], lse_ref[3:4], TOL_F32 * max(1.0, abs(float(lse_ref[3]))),
                 "LSE (row 3, relative)")
    ob, _ = api.splitk_merge(torch.from_numpy(o_part).cuda(), torch.from_numpy(lse_part).cuda(),
                             torch.bfloat16)
    assert_close(ob, o_ref, 8e-3 * max(1.0, float(np.abs(o_ref).max())), "O bf16")



@pytest.mark.parametrize("nsplit,d", [(20, 128), (40, 64), (13, 33), (16, 512), (37, 1000)])
def test_merge_ignores_payload_of_empty_splits(cuda_device, nsplit, d):
    # splits in the 8-wide load batches and in the tail after them, with
    # lse = -inf and a NaN/inf payload: the merged rows stay finite and equal
    # the oracle's merge of the remaining splits
    rows = 6
    o_part, lse_part = _partials(rows, nsplit, d, 100 + nsplit)
    empty = [1, 3, nsplit - 1, nsplit // 2]
    for s in empty:
        lse_part[0, s] = -np.inf
        o_part[0, s, :] = np.nan
        lse_part[4, s] = -np.inf
        o_part[4, s, ::2] = np.inf
    o_ref, lse_ref = oracle.merge_partials(np.nan_to_num(o_part, nan=0.0, posinf=0.0), lse_part)
    for dt in (torch.float32, torch.bfloat16):
        o, lse = api.splitk_merge(torch.from_numpy(o_part).cuda(),
                                  torch.from_numpy(lse_part).cuda(), dt)
        keep = [0, 1, 4, 5]                    # row 2 is all -inf, row 3 is shifted by +80
        tol = TOL_F32 if dt == torch.float32 else 8e-3 * max(1.0, float(np.abs(o_ref).max()))
        assert torch.isfinite(o.float()).all()
        assert_close(o[keep], o_ref[keep], tol, "O")
        assert_close(lse[keep], lse_ref[keep], TOL_F32, "LSE")

SOFTMAX_SHAPES = [
    (7, 33), (64, 1000), (3, 1), (16, 16384), (2, 32768), (3, 40000), (2, 262144),
    (1, 300001), (2, 600000), (5, 4099), (300, 32768), (200, 40000)]


@pytest.mark.parametrize("rows,cols", SOFTMAX_SHAPES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_softmax_rows_matches_oracle(cuda_device, rows, cols, dtype):
    x = inputs.make_rows(rows, cols, rows * 7 + cols, dtype, 3.0)
    y = api.softmax_rows(x.cuda())
    assert api.device_status() == 0
    y_ref = oracle.softmax_rows(f64(x))
    assert_close(y, y_ref, TOL_F32 if dtype == "f32" else TOL_BF16_SOFTMAX, "y")


def test_softmax_rows_edge_values(cuda_device):
    x = torch.randn(4, 5000) * 2
    x[0, 100:] = -math.inf            # masked tail
    x[1, :] = -math.inf               # nothing visible: zeros
    x[2, 7] = 1e4                     # one dominant entry
    y = api.softmax_rows(x.cuda())
    y_ref = oracle.softmax_rows(f64(x))
    assert_close(y, y_ref, TOL_F32, "y")
    # in place
    xc = x.cuda()
    api.softmax_rows(xc, out=xc)
    assert_close(xc, y_ref, TOL_F32, "y in place")


@pytest.mark.parametrize("cols", [40000, 80000, 262144, 600000])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_softmax_rows_long_rows_masked_in_place(cuda_device, cols, dtype):
    """Rows longer than 64 KB take the cluster path (2 to 8 CTAs per row of
    about 128 KB each, each streaming its slice twice: 80000 float columns
    give clusters of 3, 40000 columns and the bf16 rows up to 80000 columns
    clusters of 2, 262144 bf16 columns clusters of 4, the longer rows
    clusters of 8): whole slices of -inf, a row with one visible entry and a
    row with none must combine correctly, in place as well."""
    x = inputs.make_rows(3, cols, cols + 11, dtype, 3.0)
    x[0, cols // 3:] = -math.inf          # later CTAs see only -inf
    x[1, :] = -math.inf                   # nothing visible: zeros
    x[2, :] = -math.inf
    x[2, cols - 5] = 0.5                  # one visible entry, in the last slice
    y_ref = oracle.softmax_rows(f64(x))
    xc = x.cuda()
    api.softmax_rows(xc, out=xc)
    assert api.device_status() == 0
    assert_close(xc, y_ref, TOL_F32 if dtype == "f32" else TOL_BF16_SOFTMAX, "y in place")


def test_blockmask_build_matches_enumeration(cuda_device):
    tm = inputs.random_tile_mask(50, 77, 0.3, 9, nheads=3)
    tm[1, 4, :] = False
    tm[2, 0, :] = True
    bm = api.BlockMask.from_dense(tm)
    assert api.device_status() == 0
    row_ptr, col_idx = oracle.bsr_from_tile_mask(tm)
    got_rp = bm.row_ptr.cpu().numpy()
    assert np.array_equal(got_rp, row_ptr)
    assert np.array_equal(bm.col_idx.cpu().numpy()[:row_ptr[-1]], col_idx)


def test_blockmask_build_block_sparse_workload(cuda_device):
    w = inputs.WORKLOADS["block_sparse"]
    tm = inputs.window_random_tile_mask(inputs.n_tiles(w["Sq"]), w["window"], w["frac"], w["seed"])
    bm = api.BlockMask.from_dense(tm)
    row_ptr, col_idx = oracle.bsr_from_tile_mask(tm)
    assert int(bm.row_ptr[-1]) == 1722 == row_ptr[-1]
    assert np.array_equal(bm.col_idx.cpu().numpy()[:1722], col_idx)


def test_blockmask_build_capacity_is_reported(cuda_device):
    dense = torch.ones(1, 4, 4, dtype=torch.uint8, device="cuda")
    row_ptr = torch.empty(5, dtype=torch.int32, device="cuda")
    col_idx = torch.full((10,), -1, dtype=torch.int32, device="cuda")
    api.blockmask_build(dense, row_ptr, col_idx)
    with pytest.raises(api.RFError):
        api.device_status()
    assert row_ptr.tolist() == [0, 4, 8, 12, 16]
    assert col_idx.tolist() == [0, 1, 2, 3, 0, 1, 2, 3, 0, 1]
