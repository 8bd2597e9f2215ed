"""The named workloads at full size, in the launch configuration bench.py
times, checked on sampled outputs the oracle computes one by one (first,
last, tile-boundary and random rows of a few heads), plus properties that hold
at any size (every output finite; every row sees at least one key)."""

import numpy as np
import pytest
import torch

import oracle
from online_softmax_attention_rf_gb300 import api, inputs
from tests.helpers import TOL_BF16_LSE, TOL_BF16_O, TOL_F32, assert_close, f64

pytestmark = pytest.mark.gpu


def _sample_rows(S, seed):
    fixed = [0, 1, 2, 127, 128, 129, S // 2, S - 129, S - 128, S - 2, S - 1]
    rnd = np.random.default_rng(seed).integers(0, S, 5).tolist()
    return sorted({r for r in fixed + rnd if 0 <= r < S})


def _check_prefill(name, heads):
    w = inputs.WORKLOADS[name]
    q, k, v, scale, extras = inputs.workload_inputs(name)
    tm = extras.get("tile_mask")
    bm = api.BlockMask.from_dense(tm) if tm is not None else None
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = api.attn_fwd(qd, kd, vd, scale, w["causal"], bm)
    assert api.device_status() == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    del qd, kd, vd
    G = w["H"] // w["Hkv"]
    rows = _sample_rows(w["Sq"], w["seed"])
    tol_o, tol_l = (TOL_F32, TOL_F32) if w["dtype"] == "f32" else (TOL_BF16_O, TOL_BF16_LSE)
    for b, h in heads:
        o_ref, lse_ref = oracle.attention(
            f64(q[b:b + 1, h:h + 1]), f64(k[b:b + 1, h // G:h // G + 1]),
            f64(v[b:b + 1, h // G:h // G + 1]), scale, w["causal"], tm, 128, rows)
        assert_close(o[b, h, rows], o_ref[0, 0], tol_o, "%s O (b=%d,h=%d)" % (name, b, h))
        assert_close(lse[b, h, rows], lse_ref[0, 0], tol_l, "%s LSE (b=%d,h=%d)" % (name, b, h))


def test_tiny_fp32_full(cuda_device):
    q, k, v, scale, _ = inputs.workload_inputs("tiny_fp32")
    o, lse = api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale, False)
    o_ref, lse_ref = oracle.attention(f64(q), f64(k), f64(v), scale)
    assert_close(o, o_ref, TOL_F32, "O")
    assert_close(lse, lse_ref, TOL_F32, "LSE")


def test_mha_prefill_sampled(cuda_device):
    _check_prefill("mha_prefill", [(0, 0), (1, 17), (3, 31)])


def test_gqa_long_sampled(cuda_device):
    _check_prefill("gqa_long", [(0, 0), (0, 9), (0, 63)])


def test_block_sparse_sampled(cuda_device):
    _check_prefill("block_sparse", [(0, 0), (1, 15)])


def test_two_level_sampled(cuda_device):
    """The element-masked (two-level) workload at full size: encoder on the
    device, attention, sampled rows of two heads against the oracle."""
    w = inputs.WORKLOADS["two_level"]
    q, k, v, scale, extras = inputs.workload_inputs("two_level")
    em = extras["elem_mask"]
    bm = api.BlockMask.from_dense_elements(em)
    o, lse = api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale, False, bm)
    assert api.device_status() == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    rows = _sample_rows(w["Sq"], w["seed"]) + [w["n_global"] - 1, w["n_global"], 5000]
    rows = sorted(set(rows))
    for b, h in [(0, 0), (1, 15)]:
        o_ref, lse_ref = oracle.attention(f64(q[b:b + 1, h:h + 1]), f64(k[b:b + 1, h:h + 1]),
                                          f64(v[b:b + 1, h:h + 1]), scale, False, rows=rows,
                                          elem_mask=em)
        assert_close(o[b, h, rows], o_ref[0, 0], TOL_BF16_O, "two_level O (b=%d,h=%d)" % (b, h))
        assert_close(lse[b, h, rows], lse_ref[0, 0], TOL_BF16_LSE, "two_level LSE (b=%d,h=%d)" % (b, h))


def test_decode_splitk_sampled(cuda_device):
    w = inputs.WORKLOADS["decode_splitk"]
    q, k, v, scale, _ = inputs.workload_inputs("decode_splitk")
    o, lse = api.attn_decode_splitk(q.cuda(), k.cuda(), v.cuda(), w["nsplit"], scale)
    assert api.device_status() == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    G = w["H"] // w["Hkv"]
    for b, hk in [(0, 0), (7, 3), (15, 7)]:
        hs = slice(hk * G, (hk + 1) * G)
        o_ref, lse_ref = oracle.attention(f64(q[b:b + 1, hs]), f64(k[b:b + 1, hk:hk + 1]),
                                          f64(v[b:b + 1, hk:hk + 1]), scale)
        assert_close(o[b:b + 1, hs], o_ref, TOL_BF16_O, "decode O (b=%d,hk=%d)" % (b, hk))
        assert_close(lse[b:b + 1, hs], lse_ref, TOL_BF16_LSE, "decode LSE (b=%d,hk=%d)" % (b, hk))


@pytest.mark.parametrize("name", list(inputs.SOFTMAX_WORKLOADS))
def test_softmax_rows_sampled(cuda_device, name):
    w = inputs.SOFTMAX_WORKLOADS[name]
    x = inputs.make_rows(w["rows"], w["cols"], w["seed"])
    y = api.softmax_rows(x.cuda())
    assert api.device_status() == 0
    rows = [0, 1, w["rows"] // 2, w["rows"] - 1]
    assert_close(y[rows], oracle.softmax_rows(f64(x[rows])), TOL_F32, name)
    # every row sums to one (a property at any size)
    s = y.double().sum(dim=1)
    assert torch.allclose(s, torch.ones_like(s), atol=1e-4)


def _visited_full(name, make_blockmask, want_tiles):
    """Runs a full-size workload exactly as bench.py launches it, recording
    the tiles each query tile's MMA issuer visits, and compares all heads
    with the oracle's set of tiles holding a visible pair (STOF,
    Méthodologie: masked tiles are skipped entirely)."""
    w = inputs.WORKLOADS[name]
    q, k, v, scale, extras = inputs.workload_inputs(name)
    nqt, nkt = inputs.n_tiles(w["Sq"]), inputs.n_tiles(w["Sk"])
    nheads = w["B"] * w["H"]
    buf = torch.zeros(nheads * nqt * nkt, dtype=torch.uint8, device="cuda")
    bm = make_blockmask(extras)
    api.set_debug_visited(buf)
    try:
        api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale, w["causal"], bm)
        assert api.device_status() == 0
    finally:
        api.set_debug_visited(None)
    got = buf.cpu().numpy().reshape(nheads, nqt, nkt).astype(bool)
    want = want_tiles(w, extras)
    for n in range(nheads):
        bad = np.argwhere(got[n] != want)
        assert bad.size == 0, "%s head %d: %d tiles differ, first %s" % (
            name, n, len(bad), bad[:5].tolist())
    return want


def test_block_sparse_skip_set_full_size(cuda_device):
    want = _visited_full(
        "block_sparse", lambda ex: api.BlockMask.from_dense(ex["tile_mask"]),
        lambda w, ex: oracle.visited_tiles(w["Sq"], w["Sk"], w["causal"], ex["tile_mask"], 128))
    assert int(want.sum()) == 1722           # the workload's tile count per head


def test_two_level_skip_set_full_size(cuda_device):
    want = _visited_full(
        "two_level", lambda ex: api.BlockMask.from_dense_elements(ex["elem_mask"]),
        lambda w, ex: oracle.visited_tiles(w["Sq"], w["Sk"], w["causal"],
                                           elem_mask=ex["elem_mask"]))
    # the visited set is exactly the set of listed tiles of the encoding
    w = inputs.WORKLOADS["two_level"]
    rp, _, _, _ = oracle.two_level_encode(inputs.band_global_mask(w["Sq"], w["band"],
                                                                  w["n_global"]))
    assert int(want.sum()) == int(rp[-1])
