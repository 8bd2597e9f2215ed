"""Other cascaded reductions on the GPU against the float64 oracle.

RedFuser: An Automatic Operator Fusion Framework for Cascaded Reductions on AI
Accelerators -- technical summary, section 1 (MoE routing and normalisation
layers are cascades of reductions) and section 4 (MoE routing workload); the
Korean page's results (variance workloads).

MoE routing: the selected expert indices must equal the oracle's exactly (the
selection is taken on the logits as given, in both), the weights and the
log-sum-exp within the float32 bound. Row moments: mean, variance and the
normalised rows within bounds derived from float32 rounding (below).
"""

import numpy as np
import pytest
import torch

import oracle
from online_softmax_attention_rf_gb300 import api, inputs
from tests.helpers import TOL_BF16_O, TOL_F32, assert_close, f64

pytestmark = pytest.mark.gpu

# Row moments tolerance: float32 unit roundoff u = 2^-24 times a growth bound
# K = 256 (eight-term chunk sums, then about log2(n) pairwise merge levels,
# with headroom). mean: K u (|mean| + sigma); var: K u var (1 + |mean|/sigma);
# y: K u ((|mean| + sigma)/sigma + |y|), the first term from the mean's error
# seen in units of sigma, the second from the scale's.
U32 = 2.0 ** -24
K_GROWTH = 256


def _route(logits, k, renorm):
    idx, w, lse = api.moe_route(logits.cuda(), k, renorm)
    assert api.device_status() == 0
    ridx, rw, rlse = oracle.moe_route(f64(logits), k, renorm)
    return idx.cpu().numpy(), w, lse, ridx, rw, rlse


@pytest.mark.parametrize("T,E,k,dtype,renorm", [
    (1000, 256, 8, "f32", True),
    (777, 60, 6, "bf16", False),
    (513, 1024, 32, "f32", False),
    (300, 8, 8, "f32", True),          # k = E
    (64, 1, 1, "f32", False),          # one expert
    (999, 300, 4, "bf16", True),
    (100, 33, 32, "f32", False),       # E not a multiple of 32
    (9, 128, 2, "bf16", True),         # fewer tokens than a CTA holds
])
def test_moe_route_matches_oracle(cuda_device, T, E, k, dtype, renorm):
    x = inputs.make_logits(T, E, T + E + k, dtype, amp=2.0)
    idx, w, lse, ridx, rw, rlse = _route(x, k, renorm)
    assert np.array_equal(idx, ridx)
    assert_close(w, rw, TOL_F32, "w")
    assert_close(lse, rlse, TOL_F32, "lse")


@pytest.mark.parametrize("E", [64, 128, 256, 512])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_moe_route_ties_go_to_the_lower_index(cuda_device, dtype, E):
    x = inputs.make_logits(500, E, 3, dtype, ties=True)
    idx, w, lse, ridx, rw, rlse = _route(x, 8, False)
    assert np.array_equal(idx, ridx)
    assert_close(w, rw, TOL_F32, "w")
    # equal logits within a token's selection appear in ascending index order
    xs = f64(x)
    for t in range(0, 500, 37):
        vals = xs[t, idx[t]]
        for a in range(7):
            if vals[a] == vals[a + 1]:
                assert idx[t, a] < idx[t, a + 1]


def test_moe_route_offset_and_masked_experts(cuda_device):
    """Logits far from zero (the maximum subtraction keeps exp in range) and
    experts masked with -inf (weight 0; chosen last, lower index first)."""
    T, E, k = 400, 128, 8
    x = inputs.make_logits(T, E, 11, "f32", amp=2.0) + 1000.0
    x[::3, 5:120] = float("-inf")         # every third token: only 13 finite experts
    x[1::7, :] = float("-inf")
    x[1::7, 77] = 0.0                     # one finite expert, then masked ones
    idx, w, lse, ridx, rw, rlse = _route(x, k, False)
    assert np.array_equal(idx, ridx)
    assert_close(w, rw, TOL_F32, "w")
    assert_close(lse, rlse, TOL_F32 * 10, "lse")   # |lse| ~ 1000: half an ulp is 3e-5


def test_moe_route_without_lse_and_renorm_consistency(cuda_device):
    x = inputs.make_logits(256, 256, 4, "f32", amp=2.0).cuda()
    i1, w1, l1 = api.moe_route(x, 8, False)
    i2, w2, l2 = api.moe_route(x, 8, True, with_lse=False)
    assert l2 is None
    assert torch.equal(i1, i2)
    torch.testing.assert_close(w2, w1 / w1.sum(1, keepdim=True), rtol=1e-6, atol=1e-7)
    assert torch.allclose(w2.sum(1), torch.ones(256, device="cuda"), atol=1e-6)


def test_moe_route_full_size_sampled(cuda_device):
    """The routing workload (131072 tokens, 256 experts, top 8) in the launch
    configuration the benchmark times; the oracle checks 4096 sampled tokens."""
    c = inputs.CASCADE_WORKLOADS["moe_route"]
    x = inputs.make_logits(c["T"], c["E"], c["seed"], c["dtype"], c["amp"])
    idx, w, lse = api.moe_route(x.cuda(), c["k"], c["renorm"])
    assert api.device_status() == 0
    rows = np.random.default_rng(0).choice(c["T"], 4096, replace=False)
    ridx, rw, rlse = oracle.moe_route(f64(x)[rows], c["k"], c["renorm"])
    assert np.array_equal(idx.cpu().numpy()[rows], ridx)
    assert_close(w.cpu()[rows], rw, TOL_F32, "w")
    assert_close(lse.cpu()[rows], rlse, TOL_F32, "lse")


def _check_moments(x, mean, var, y, eps):
    rmean, rvar, ry = oracle.row_moments(f64(x), eps)
    sig = np.sqrt(rvar)
    tol_m = K_GROWTH * U32 * (np.abs(rmean) + sig) + 1e-30
    err_m = np.abs(f64(mean) - rmean)
    assert (err_m <= tol_m).all(), "mean: worst err/tol %.3g" % (err_m / tol_m).max()
    tol_v = K_GROWTH * U32 * rvar * (1 + np.abs(rmean) / np.maximum(sig, 1e-30)) + 1e-30
    err_v = np.abs(f64(var) - rvar)
    assert (err_v <= tol_v).all(), "var: worst err/tol %.3g" % (err_v / tol_v).max()
    if y is None:
        return
    if x.dtype == torch.bfloat16:
        assert_close(y, ry, TOL_BF16_O, "y")
        return
    rel = np.where(sig > 0, (np.abs(rmean) + sig) / np.maximum(sig, 1e-30), 1.0)
    tol_y = K_GROWTH * U32 * (rel[:, None] + np.abs(ry))
    err_y = np.abs(f64(y) - ry)
    assert (err_y <= tol_y).all(), "y: worst err/tol %.3g" % (err_y / tol_y).max()


@pytest.mark.parametrize("rows,cols", [(33, 1), (17, 7), (64, 8), (40, 1000), (16, 4096),
                                       (6, 4104), (8, 8192), (4, 12288), (3, 20000),
                                       (2, 32768), (5, 20001), (3, 65536)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_row_moments_matches_oracle(cuda_device, rows, cols, dtype):
    x = inputs.make_moment_rows(rows, cols, rows * 7 + cols, dtype, amp=1.5, offset=3.0)
    mean, var, y = api.row_moments(x.cuda(), 1e-5)
    assert api.device_status() == 0
    _check_moments(x, mean, var, y, 1e-5)


def test_row_moments_statistics_only_and_in_place(cuda_device):
    x = inputs.make_moment_rows(100, 2048, 5, "f32", offset=-2.0)
    xd = x.cuda()
    m1, v1, y1 = api.row_moments(xd, 1e-3, normalize=False)
    assert y1 is None
    m2, v2, y2 = api.row_moments(xd, 1e-3, out=xd)          # y aliases x
    assert api.device_status() == 0
    assert torch.equal(m1, m2) and torch.equal(v1, v2)
    _check_moments(x, m2, v2, y2, 1e-3)


def test_row_moments_large_offset(cuda_device):
    """mean/sigma = 1000: the one-pass sum of squares would lose every
    digit of the variance here; the merged (count, mean, M2) states do not."""
    x = inputs.make_moment_rows(32, 8192, 6, "f32", amp=1.0, offset=1000.0)
    mean, var, y = api.row_moments(x.cuda(), 0.0)
    _check_moments(x, mean, var, y, 0.0)
    rvar = oracle.row_moments(f64(x))[1]
    assert np.abs(f64(var) / rvar - 1).max() < 1e-3


def test_row_moments_unaligned_rows(cuda_device):
    """A view starting one element in (no 16-byte alignment) takes the
    element-wise path and gives the same statistics."""
    base = inputs.make_moment_rows(1, 64 * 1000 + 1, 8, "f32").cuda()
    x = base[0, 1:].view(64, 1000)
    mean, var, y = api.row_moments(x, 1e-5)
    _check_moments(x.cpu(), mean, var, y, 1e-5)


def test_row_moments_full_size_sampled(cuda_device):
    c = inputs.CASCADE_WORKLOADS["row_moments"]
    x = inputs.make_moment_rows(c["rows"], c["cols"], c["seed"], c["dtype"], c["amp"],
                                c["offset"])
    mean, var, y = api.row_moments(x.cuda(), c["eps"])
    assert api.device_status() == 0
    rows = np.random.default_rng(1).choice(c["rows"], 64, replace=False)
    _check_moments(x[rows], mean.cpu()[rows], var.cpu()[rows], y.cpu()[rows], c["eps"])


def _check_inertia(points, masses, M, c, I):
    """Bounds from float32 rounding: K u times the magnitudes involved
    (u = 2^-24, K = 256 as above); sigma = sqrt(I / M) is the spread."""
    rM, rc, rI = oracle.moment_of_inertia(f64(points), None if masses is None else f64(masses))
    sig = np.sqrt(np.where(rM > 0, rI / np.where(rM > 0, rM, 1), 0))
    cn = np.abs(rc).max(axis=1)
    assert (np.abs(f64(M) - rM) <= K_GROWTH * U32 * rM + 1e-30).all()
    tol_c = K_GROWTH * U32 * (cn + sig) + 1e-30
    assert (np.abs(f64(c) - rc).max(axis=1) <= tol_c).all(), "centre"
    tol_i = K_GROWTH * U32 * rI * (1 + cn / np.maximum(sig, 1e-30)) + 1e-30
    err = np.abs(f64(I) - rI)
    assert (err <= tol_i).all(), "inertia: worst err/tol %.3g" % (err / tol_i).max()


@pytest.mark.parametrize("sets,n", [(5, 1), (7, 3), (3, 4), (4, 1000), (2, 4096), (3, 4097),
                                    (8, 100000)])
@pytest.mark.parametrize("unit", [False, True])
def test_moment_of_inertia_matches_oracle(cuda_device, sets, n, unit):
    points, masses = inputs.make_point_sets(sets, n, sets * 31 + n, amp=2.0, offset=5.0)
    if unit:
        masses = None
    M, c, I = api.moment_of_inertia(points.cuda(), None if unit else masses.cuda())
    assert api.device_status() == 0
    _check_inertia(points, masses, M, c, I)


def test_moment_of_inertia_zero_mass_and_unaligned(cuda_device):
    points, masses = inputs.make_point_sets(3, 2049, 4, amp=1.0, offset=-3.0)
    masses[1] = 0.0                                   # a set without mass
    pd, md = points.cuda(), masses.cuda()
    M, c, I = api.moment_of_inertia(pd, md)
    assert api.device_status() == 0
    assert M[1].item() == 0 and torch.all(c[1] == 0) and I[1].item() == 0
    _check_inertia(points, masses, M, c, I)
    # a view one point in (12-byte offset): the element-wise path
    flat = pd.reshape(-1)[3:3 + 3 * 2048 * 3].view(3, 2048, 3)
    mflat = md.reshape(-1)[1:1 + 3 * 2048].view(3, 2048)
    M3, c3, I3 = api.moment_of_inertia(flat, mflat)
    assert api.device_status() == 0
    _check_inertia(flat.cpu(), mflat.cpu(), M3, c3, I3)


def test_moment_of_inertia_full_size_sampled(cuda_device):
    w = inputs.CASCADE_WORKLOADS["inertia"]
    points, masses = inputs.make_point_sets(w["sets"], w["n"], w["seed"], w["amp"], w["offset"])
    M, c, I = api.moment_of_inertia(points.cuda(), masses.cuda())
    assert api.device_status() == 0
    sets = np.random.default_rng(2).choice(w["sets"], 64, replace=False)
    _check_inertia(points[sets], masses[sets], M.cpu()[sets], c.cpu()[sets], I.cpu()[sets])
