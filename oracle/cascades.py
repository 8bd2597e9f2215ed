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

Readings where the pages are silent (each listed in the design notes):

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
