"""Plain float64 definitions of other cascaded reductions.

TEST INFRASTRUCTURE ONLY: imported by ``tests/`` and ``bench.py``'s CPU
baseline; never by the product.

Sources (page title, section):

* RedFuser: An Automatic Operator Fusion Framework for Cascaded Reductions on
  AI Accelerators -- technical summary, section 1 "Problématique": besides
  attention, the key examples of cascaded reductions are normalisation
  layers, routing in Mixture-of-Experts models and FP8 quantisation; section
  4 "Résultats Expérimentaux": MoE routing and FP8 Quant + GEMM workloads;
  the Korean page, results: variance and moment-of-inertia (non-ML)
  workloads.

Readings where the pages are silent (the pages name these workloads but
give no formula, format or precision; each reading below is the plainest
one for a workload given by name):

* MoE routing: p = softmax(logits) over the experts of one token; the k
  experts with the largest p are selected, in descending order, ties broken
  towards the lower expert index; their weights are p (``renorm`` False) or
  p divided by the sum of the k selected p (``renorm`` True). Because exp is
  increasing, the k largest p are the k largest logits, so the selection is
  taken on the logits as given (no rounding enters it).
* Row moments: mean = sum(x) / n, then var = sum((x - mean)^2) / n (the
  population variance, the one normalisation layers use); the normalised row
  is (x - mean) / sqrt(var + eps).
* Moment of inertia (the Korean page's non-ML workload): for a set of point
  masses m_i at positions r_i, the total mass M = sum m_i and the centre of
  mass c = sum m_i r_i / M (reduction 1), then the moment of inertia about
  the centre of mass, I = sum m_i |r_i - c|^2 (reduction 2, which needs c):
  the scalar (polar) moment, the trace-free reading being the plainest one
  for a workload given only by name.
* FP8 quantisation + GEMM (named only): per-row absmax quantisation to FP8
  E4M3 (the format with 4 exponent bits, bias 7, 3 mantissa bits, largest
  finite value 448, subnormals down to 2^-9): amax = max |x| over the row
  (reduction 1); the row is scaled by 448 / amax and rounded to the nearest
  E4M3 value, ties to even, magnitudes past 448 saturating to 448; the row's
  dequantisation scale is amax / 448 (an all-zero row: codes 0, scale 1).
  The pages fix no precision for the scaled value. Because the rounding
  decides an integer code, the oracle takes that one decision in float32,
  the precision in which the kernel forms it: inv = float32(448) /
  float32(amax), then float32(x) * inv. Everything else (amax, the E4M3
  rounding of that product, the GEMM) is exact or float64. Taken in float64
  instead, the scaled value differs from the float32 one by at most about
  two float32 ulps, so the codes agree except where the product lies within
  that distance of a rounding tie between two E4M3 values (a pin checks
  exactly this). The GEMM (reduction 2, over the quantised values) is
  C[m, n] = sa[m] * sw[n] * sum_k qa[m, k] qw[n, k], in float64 here.
"""

import numpy as np


def moe_route(logits, k, renorm=False):
    """Top-k softmax routing of each token (row), float64, three steps.

    logits [T, E] (any float dtype, cast exactly). Returns (idx int32 [T, k],
    w float64 [T, k], lse float64 [T]).
    """
    x = np.asarray(logits, dtype=np.float64)
    T, E = x.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    # step 1: softmax over the experts, by its definition (max, sum, divide)
    m = x.max(axis=1)
    e = np.exp(x - m[:, None])
    s = e.sum(axis=1)
    p = e / s[:, None]
    # step 2: the k largest logits, descending; equal logits: lower index first
    idx = np.empty((T, k), dtype=np.int32)
    cols = np.arange(E)
    for t in range(T):
        order = np.lexsort((cols, -x[t]))   # primary key -x, secondary index
        idx[t] = order[:k]
    # step 3: their probabilities, renormalised over the selection if asked
    w = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    if renorm:
        w = w / w.sum(axis=1, keepdims=True)
    return idx, w, m + np.log(s)


def row_moments(x, eps=1e-5):
    """Per-row mean and population variance, two passes (mean first), and
    the normalised rows. x [R, n] -> (mean [R], var [R], y [R, n])."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[1]
    mean = x.sum(axis=1) / n                           # reduction 1
    d = x - mean[:, None]
    var = (d * d).sum(axis=1) / n                      # reduction 2, needs reduction 1
    y = d / np.sqrt(var + eps)[:, None]
    return mean, var, y


def moment_of_inertia(points, masses=None):
    """Per point set: total mass, centre of mass, and the moment of inertia
    about the centre of mass, by the two-pass definition in float64.

    points [S, N, k] (any float dtype, cast exactly), masses [S, N] (None:
    unit masses). Returns (M [S], c [S, k], I [S]); a set of total mass 0
    gives c = 0 and I = 0.
    """
    r = np.asarray(points, dtype=np.float64)
    S, N, k = r.shape
    m = np.ones((S, N)) if masses is None else np.asarray(masses, dtype=np.float64)
    M = m.sum(axis=1)                                             # reduction 1
    safe = np.where(M != 0, M, 1.0)
    c = np.where((M != 0)[:, None], (m[:, :, None] * r).sum(axis=1) / safe[:, None], 0.0)
    d = r - c[:, None, :]
    I = np.where(M != 0, (m * (d * d).sum(axis=2)).sum(axis=1), 0.0)   # reduction 2
    return M, c, I


E4M3_MAX = 448.0


def e4m3_round(v):
    """Nearest E4M3 value of float64 v (ties to even), saturating at 448,
    from the format's definition: normal numbers 2^e (1 + m/8), e in
    [-6, 8], subnormals m * 2^-9."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)                       # below 2^-6: the subnormal spacing 2^-9
    quantum = np.exp2(e - 3)
    q = np.round(a / quantum) * quantum         # numpy rounds halves to even
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, v)                    # zeros keep their sign


def e4m3_code(v):
    """The 8-bit code (sign, exponent, mantissa) of E4M3 values; the sign bit
    is kept for zero (a negative value that rounds to zero is -0, 0x80)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    sign = np.signbit(v).astype(np.uint8) << 7
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    normal = a >= 2.0 ** -6
    exp_field = np.where(normal, e + 7, 0).astype(np.int64)
    mant = np.where(normal, a / np.exp2(e) - 1.0, a / 2.0 ** -9) * np.where(normal, 8, 1)
    return (sign | (exp_field << 3).astype(np.uint8) | np.rint(mant).astype(np.uint8)).astype(
        np.uint8)


def rowquant_e4m3(x):
    """Per-row absmax quantisation of x [R, K] (any float dtype) to E4M3.
    Returns (q float64 [R, K] of E4M3 values, scale float32 [R])."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.abs(x32).max(axis=1)                                    # reduction 1
    safe = np.where(amax > 0, amax, np.float32(1.0)).astype(np.float32)
    inv = (np.float32(E4M3_MAX) / safe).astype(np.float32)
    prod = (x32 * inv[:, None]).astype(np.float32)                    # float32, as the kernel
    q = e4m3_round(prod.astype(np.float64))
    q = np.where((amax > 0)[:, None], q, 0.0)
    scale = np.where(amax > 0, safe / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    return q, scale


def fp8_gemm(qa, sa, qw, sw):
    """C = diag(sa) (qa qw^T) diag(sw) in float64 (reduction 2 over k)."""
    qa = np.asarray(qa, dtype=np.float64)
    qw = np.asarray(qw, dtype=np.float64)
    return (np.asarray(sa, np.float64)[:, None] * (qa @ qw.T)) * np.asarray(sw, np.float64)[None]
