"""Pins of the oracle's other cascaded reductions (``oracle/cascades.py``,
``oracle/incremental.py`` moment states): brute force with explicit loops,
library routines (torch.topk / softmax, numpy var), closed forms, invariants,
and planted mistakes that a pin must catch."""

import math

import numpy as np
import pytest
import torch

import oracle
import oracle.cascades as oc


def _brute_route(row, k, renorm):
    E = len(row)
    m = max(row)
    e = [math.exp(v - m) for v in row]
    s = math.fsum(e)
    left = list(range(E))
    idx = []
    for _ in range(k):
        best = left[0]
        for j in left[1:]:
            if row[j] > row[best]:            # strict: the lower index wins ties
                best = j
        idx.append(best)
        left.remove(best)
    w = [e[j] / s for j in idx]
    if renorm:
        tot = math.fsum(w)
        w = [x / tot for x in w]
    return idx, w, m + math.log(s)


@pytest.mark.parametrize("renorm", [False, True])
def test_moe_route_brute_force(renorm):
    rng = np.random.default_rng(1)
    x = rng.normal(size=(7, 11)) * 3
    x[2, 4] = x[2, 9] = x[2].max() + 1          # a tie at the top
    idx, w, lse = oracle.moe_route(x, 4, renorm)
    for t in range(7):
        bi, bw, bl = _brute_route(x[t].tolist(), 4, renorm)
        assert idx[t].tolist() == bi
        np.testing.assert_allclose(w[t], bw, rtol=1e-13, atol=1e-15)
        assert abs(lse[t] - bl) < 1e-12


def test_moe_route_library():
    """Distinct logits: torch.topk's indices and torch.softmax's values."""
    x = torch.randn(50, 64, dtype=torch.float64, generator=torch.Generator().manual_seed(2))
    idx, w, lse = oracle.moe_route(x.numpy(), 6)
    tv, ti = torch.topk(x, 6, dim=1, largest=True, sorted=True)
    assert np.array_equal(idx, ti.numpy())
    p = torch.softmax(x, dim=1)
    np.testing.assert_allclose(w, torch.gather(p, 1, ti).numpy(), rtol=1e-13)
    np.testing.assert_allclose(lse, torch.logsumexp(x, 1).numpy(), rtol=1e-13)


def test_moe_route_ties_and_special_cases():
    x = np.array([[0.0, 1.0, 1.0, 1.0, -2.0]])
    idx, w, _ = oracle.moe_route(x, 3)
    assert idx.tolist() == [[1, 2, 3]]                        # equal logits: lower index first
    idx, w, _ = oracle.moe_route(x, 5)
    assert sorted(idx[0].tolist()) == list(range(5))           # k = E: a permutation
    np.testing.assert_allclose(w.sum(), 1.0, rtol=1e-14)
    u = np.zeros((1, 8))
    idx, w, lse = oracle.moe_route(u, 2, True)                 # uniform: first two, 1/2 each
    assert idx.tolist() == [[0, 1]] and np.allclose(w, 0.5) and abs(lse[0] - math.log(8)) < 1e-14


def test_moe_route_shift_invariance():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(20, 32))
    a = oracle.moe_route(x, 5, False)
    b = oracle.moe_route(x + 17.25, 5, False)
    assert np.array_equal(a[0], b[0])
    np.testing.assert_allclose(a[1], b[1], rtol=1e-12)
    np.testing.assert_allclose(b[2] - a[2], 17.25, rtol=1e-12)


def test_row_moments_library_and_closed_forms():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(9, 1000)) * 5 + 3
    mean, var, y = oracle.row_moments(x, eps=0.0)
    np.testing.assert_allclose(mean, x.mean(axis=1), rtol=1e-13)
    np.testing.assert_allclose(var, np.var(x, axis=1), rtol=1e-12)      # population variance
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose((y * y).mean(axis=1), 1.0, rtol=1e-12)
    m2, v2, y2 = oracle.row_moments(np.array([[2.0, 6.0], [5.0, 5.0]]), eps=0.0 + 1e-30)
    assert m2.tolist() == [4.0, 5.0] and v2.tolist() == [4.0, 0.0]     # ((a-b)/2)^2; constant row
    assert np.all(y2[1] == 0.0)


def test_row_moments_shift_and_scale():
    x = np.random.default_rng(5).normal(size=(3, 257))
    _, v, _ = oracle.row_moments(x)
    _, vs, _ = oracle.row_moments(x + 1e3)
    _, vc, _ = oracle.row_moments(3.0 * x)
    np.testing.assert_allclose(vs, v, rtol=1e-9)
    np.testing.assert_allclose(vc, 9.0 * v, rtol=1e-12)


@pytest.mark.parametrize("chunk", [1, 7, 128, 1000])
def test_moment_states_merge_to_the_two_pass_result(chunk):
    """The pairwise (count, mean, M2) merge the GPU uses reaches the
    two-pass definition for any chunking, and merges associatively."""
    x = np.random.default_rng(6).normal(size=3001) * 2 + 10
    st = (0, 0.0, 0.0)
    for c0 in range(0, x.size, chunk):
        st = oracle.moments_merge(st, oracle.moments_state(x[c0:c0 + chunk]))
    mean, var, _ = oracle.row_moments(x[None])
    assert st[0] == x.size
    assert abs(st[1] - mean[0]) < 1e-12 and abs(st[2] / st[0] - var[0]) < 1e-10
    a, b, c = (oracle.moments_state(p) for p in np.split(x[:3000], 3))
    l = oracle.moments_merge(oracle.moments_merge(a, b), c)
    r = oracle.moments_merge(a, oracle.moments_merge(b, c))
    assert abs(l[1] - r[1]) < 1e-12 and abs(l[2] - r[2]) < 1e-8


def _brute_inertia(points, masses):
    """Python-math loops: total mass, centre of mass, then sum m |r - c|^2."""
    M = math.fsum(masses)
    k = len(points[0])
    c = [math.fsum(m * p[j] for p, m in zip(points, masses)) / M for j in range(k)]
    I = math.fsum(m * math.fsum((p[j] - c[j]) ** 2 for j in range(k))
                  for p, m in zip(points, masses))
    return M, c, I


def test_inertia_brute_force():
    rng = np.random.default_rng(7)
    r = rng.normal(size=(3, 9, 3)) * 2 + 5
    m = rng.random((3, 9)) + 0.1
    M, c, I = oracle.moment_of_inertia(r, m)
    for s in range(3):
        bM, bc, bI = _brute_inertia(r[s].tolist(), m[s].tolist())
        assert abs(M[s] - bM) < 1e-12 and np.allclose(c[s], bc, rtol=1e-13)
        assert abs(I[s] - bI) < 1e-11 * bI


def test_inertia_closed_forms():
    # two point masses: I = m1 m2 / (m1 + m2) d^2
    M, c, I = oracle.moment_of_inertia([[[0.0, 0.0, 0.0], [0.0, 0.0, 2.0]]], [[1.0, 3.0]])
    assert M[0] == 4.0 and np.allclose(c[0], [0, 0, 1.5]) and abs(I[0] - 3.0) < 1e-14
    # N unit masses on a circle of radius R: centre 0, I = N R^2
    t = np.arange(12) * (2 * np.pi / 12)
    ring = np.stack([3.0 * np.cos(t), 3.0 * np.sin(t), np.zeros(12)], axis=1)[None]
    M, c, I = oracle.moment_of_inertia(ring)
    assert np.allclose(c[0], 0, atol=1e-14) and abs(I[0] - 12 * 9.0) < 1e-12
    # zero total mass
    M, c, I = oracle.moment_of_inertia(np.ones((1, 4, 3)), np.zeros((1, 4)))
    assert M[0] == 0 and np.all(c[0] == 0) and I[0] == 0


def test_inertia_parallel_axis_translation_and_variance():
    rng = np.random.default_rng(8)
    r = rng.normal(size=(4, 50, 3)) + np.array([10.0, -4.0, 2.0])
    m = rng.random((4, 50))
    M, c, I = oracle.moment_of_inertia(r, m)
    about_origin = (m * (r * r).sum(axis=2)).sum(axis=1)          # parallel-axis theorem
    np.testing.assert_allclose(about_origin, I + M * (c * c).sum(axis=1), rtol=1e-12)
    M2, c2, I2 = oracle.moment_of_inertia(r + 7.5, m)               # translation
    np.testing.assert_allclose(I2, I, rtol=1e-10)
    np.testing.assert_allclose(c2, c + 7.5, rtol=1e-13)
    Mu, cu, Iu = oracle.moment_of_inertia(r)                          # unit masses
    np.testing.assert_allclose(Iu, 50 * np.var(r, axis=1).sum(axis=1), rtol=1e-12)


@pytest.mark.parametrize("chunk", [1, 5, 64])
def test_weighted_states_merge_to_the_two_pass_result(chunk):
    rng = np.random.default_rng(9)
    r = rng.normal(size=(301, 3)) * 3 + 20
    m = rng.random(301) + 0.01
    st = (0.0, np.zeros(3), 0.0)
    for c0 in range(0, 301, chunk):
        st = oracle.weighted_merge(st, oracle.weighted_state(r[c0:c0 + chunk], m[c0:c0 + chunk]))
    M, c, I = oracle.moment_of_inertia(r[None], m[None])
    assert abs(st[0] - M[0]) < 1e-10 and np.allclose(st[1], c[0], rtol=1e-12)
    assert abs(st[2] - I[0]) < 1e-9 * I[0]
    a, b, d = (oracle.weighted_state(r[i:i + 100], m[i:i + 100]) for i in (0, 100, 200))
    left = oracle.weighted_merge(oracle.weighted_merge(a, b), d)
    right = oracle.weighted_merge(a, oracle.weighted_merge(b, d))
    assert abs(left[2] - right[2]) < 1e-9 * left[2]


def _all_finite_e4m3():
    """Every finite E4M3 value, decoded by torch's float8_e4m3fn (codes 0x7f
    and 0xff are NaN)."""
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return codes, vals


def test_e4m3_against_torch():
    codes, vals = _all_finite_e4m3()
    assert np.array_equal(oracle.e4m3_round(vals), vals)          # representable values stay
    pos = vals >= 0
    assert np.array_equal(oracle.e4m3_code(vals[pos & (vals > 0)]), codes[pos & (vals > 0)])
    # midpoints between neighbours (ties to even) and random values in range
    u = np.unique(np.abs(vals))
    mids = (u[1:] + u[:-1]) / 2
    rng = np.random.default_rng(10)
    probe = np.concatenate([mids, -mids, rng.uniform(-448, 448, 2000),
                            rng.uniform(-1, 1, 2000) * 2.0 ** -5])
    want = torch.from_numpy(probe).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3_round(probe), want)
    # codes of everything, signs and signed zeros included (tiny values round to +-0)
    probe = np.concatenate([probe, [-1e-5, 1e-5, -0.0, 0.0], -vals[vals > 0]])
    codes_t = torch.from_numpy(probe).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_code(oracle.e4m3_round(probe)), codes_t)


def test_e4m3_saturates():
    v = np.array([448.0, 449.0, 464.0, 480.0, 1e6, -1e30])
    assert np.array_equal(oracle.e4m3_round(v), [448, 448, 448, 448, 448, -448])


def test_rowquant_properties():
    rng = np.random.default_rng(11)
    x = (rng.normal(size=(6, 300)) * np.array([1e-3, 1, 7, 100, 3e4, 1])[:, None]).astype(np.float32)
    x[5] = 0.0
    q, sc = oracle.rowquant_e4m3(x)
    assert np.all(np.abs(q[:5]).max(axis=1) == 448.0)              # the absmax element maps to 448
    assert np.all(q[5] == 0) and sc[5] == 1.0
    amax = np.abs(x[:5]).max(axis=1)
    np.testing.assert_allclose(sc[:5], amax / 448.0, rtol=1e-7)
    # dequantised error: half a unit in the last of 3 mantissa bits, or half
    # the subnormal spacing, in units of the scale
    err = np.abs(q[:5] * sc[:5, None] - x[:5])
    bound = 2.0 ** -4 * np.abs(x[:5]) + 2.0 ** -10 * sc[:5, None] * 1.0001
    assert np.all(err <= bound)
    # exact scaling by a power of two leaves the codes unchanged
    q2, sc2 = oracle.rowquant_e4m3(x * np.float32(8.0))
    assert np.array_equal(q2, q) and np.allclose(sc2[:5], sc[:5] * 8, rtol=0)


def test_rowquant_float32_decision_agrees_with_float64_away_from_ties():
    """The oracle forms the scaled value x * (448 / amax) in float32 (the one
    place where it takes the kernel's precision, because the result decides
    an integer code). Taken in float64 it differs by at most a few float32
    ulps, so the codes must agree except where the float64 product lies
    within that distance of a rounding tie between two E4M3 values."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((64, 4096)) * rng.uniform(1e-2, 1e2, (64, 1))).astype(np.float32)
    x[3, :100] = np.float32(448.0) * np.arange(100, dtype=np.float32) / np.float32(7.0)
    q32, _ = oracle.rowquant_e4m3(x)
    x64 = x.astype(np.float64)
    p64 = x64 * (448.0 / np.abs(x64).max(axis=1))[:, None]
    q64 = oracle.e4m3_round(p64)
    _, vals = _all_finite_e4m3()
    u = np.unique(np.abs(vals))
    mids = (u[1:] + u[:-1]) / 2
    a = np.abs(p64)
    j = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    dist = np.minimum(np.abs(a - mids[j - 1]), np.abs(a - mids[j]))
    near_tie = dist <= 4 * 2.0 ** -24 * a
    differ = q32 != q64
    assert not np.any(differ & ~near_tie)
    assert differ.sum() <= near_tie.sum() and differ.mean() < 1e-3


def test_fp8_gemm_definition():
    rng = np.random.default_rng(12)
    a = rng.normal(size=(5, 64)).astype(np.float32)
    w = rng.normal(size=(3, 64)).astype(np.float32)
    qa, sa = oracle.rowquant_e4m3(a)
    qw, sw = oracle.rowquant_e4m3(w)
    c = oracle.fp8_gemm(qa, sa, qw, sw)
    for i in range(5):
        for j in range(3):
            ref = math.fsum(float(qa[i, k]) * float(qw[j, k]) for k in range(64))
            assert abs(c[i, j] - float(sa[i]) * float(sw[j]) * ref) < 1e-9 * (1 + abs(c[i, j]))
    np.testing.assert_allclose(c, (qa * sa[:, None]) @ (qw * sw[:, None]).T, rtol=1e-12)
    np.testing.assert_allclose(c, a @ w.T, rtol=0.2, atol=2.0)   # close to the unquantised product


def _pins():
    yield lambda: test_moe_route_brute_force(True)
    yield test_moe_route_ties_and_special_cases
    yield test_row_moments_library_and_closed_forms
    yield test_inertia_brute_force
    yield test_inertia_closed_forms
    yield test_inertia_parallel_axis_translation_and_variance
    yield test_e4m3_against_torch
    yield test_e4m3_saturates
    yield test_rowquant_properties


def _mutant_route_ties_upward(logits, k, renorm=False):
    x = np.asarray(logits, dtype=np.float64)
    flipped = x[:, ::-1]
    idx, w, lse = _orig_route(flipped, k, renorm)
    return (x.shape[1] - 1 - idx).astype(np.int32), w, lse


def _mutant_route_no_renorm(logits, k, renorm=False):
    return _orig_route(logits, k, False)


def _mutant_sample_variance(x, eps=1e-5):
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[1]
    mean = x.sum(axis=1) / n
    d = x - mean[:, None]
    var = (d * d).sum(axis=1) / (n - 1)
    return mean, var, d / np.sqrt(var + eps)[:, None]


def _mutant_inertia_about_origin(points, masses=None):
    M, c, I = _orig_inertia(points, masses)
    r = np.asarray(points, dtype=np.float64)
    m = np.ones(r.shape[:2]) if masses is None else np.asarray(masses, dtype=np.float64)
    return M, c, (m * (r * r).sum(axis=2)).sum(axis=1)


def _mutant_inertia_unweighted_centre(points, masses=None):
    r = np.asarray(points, dtype=np.float64)
    m = np.ones(r.shape[:2]) if masses is None else np.asarray(masses, dtype=np.float64)
    c = r.mean(axis=1)
    return m.sum(axis=1), c, (m * ((r - c[:, None]) ** 2).sum(axis=2)).sum(axis=1)


def _mutant_e4m3_half_away(v):
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.clip(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6, 8)
    qn = np.exp2(e - 3)
    return np.sign(v) * np.minimum(np.floor(a / qn + 0.5) * qn, 448.0)


def _mutant_e4m3_no_saturation(v):
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.clip(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6, None)
    qn = np.exp2(e - 3)
    return np.sign(v) * np.round(a / qn) * qn


_orig_route = oc.moe_route
_orig_inertia = oc.moment_of_inertia
_orig_e4m3 = oc.e4m3_round


@pytest.mark.parametrize("target,mutant", [
    ("moe_route", _mutant_route_ties_upward), ("moe_route", _mutant_route_no_renorm),
    ("row_moments", _mutant_sample_variance),
    ("moment_of_inertia", _mutant_inertia_about_origin),
    ("moment_of_inertia", _mutant_inertia_unweighted_centre),
    ("e4m3_round", _mutant_e4m3_half_away), ("e4m3_round", _mutant_e4m3_no_saturation)])
def test_pins_catch_planted_mistakes(monkeypatch, target, mutant):
    monkeypatch.setattr(oracle, target, mutant)
    if target == "e4m3_round":      # rowquant_e4m3 calls it through its own module
        monkeypatch.setattr(oc, target, mutant)
    failures = 0
    for pin in _pins():
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures > 0
