"""Float64 run of the incremental (online) form, used to check the derivation.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages state the incremental form only in words:

* RedFuser: An Automatic Operator Fusion Framework for Cascaded Reductions on
  AI Accelerators -- section 2 "Méthodologie", incremental computation:
  partial results are updated as new input arrives, so on-chip state falls
  from O(L) to O(1); the feasibility conditions are a decomposable F_i, a
  commutative monoid and distributivity of the reduction over the combining
  operator.
* Riepilogo Tecnico: FLASHLIGHT -- "Metodologia", item 3 (algebraic
  transformation): keep running accumulators for the maximum and the sum and
  rescale the sum whenever the running maximum changes, using
  e^(x-y) = e^x / e^y.

Written out, the state per query row is (m, l, acc), starting at
(-inf, 0, 0). A tile of keys with scores s updates it as

    m'   = max(m, max_tile s)
    a    = exp(m - m')
    l'   = a * l   + sum_tile exp(s - m')
    acc' = a * acc + sum_tile exp(s - m') * v

and the result is O = acc / l, LSE = m + ln l. When m' is still -inf (no
visible key yet) the update uses a = 1 and exp(s - m') = 0. Two states merge
by the same rule (the monoid the multi-segment strategy relies on).

This module is not the oracle: it exists so that a test can show that the
online form equals the three-pass definition in ``three_pass.py`` for any
tiling, which is what licenses the GPU to use it.
"""

import numpy as np

NEG_INF = -np.inf


def _shift(m):
    """The maximum used for the exponentials: m itself, or 0 while m = -inf."""
    return np.where(m > NEG_INF, m, 0.0)


def init_state(R, dv):
    return (np.full(R, NEG_INF), np.zeros(R), np.zeros((R, dv)))


def update(state, s, v):
    """Fold one key tile (scores s [R, T] with -inf where masked, v [T, dv])."""
    m, l, acc = state
    tile_max = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], NEG_INF)
    m_new = np.maximum(m, tile_max)
    a = np.where(m_new > NEG_INF, np.exp(m - _shift(m_new)), 1.0)
    p = np.exp(s - _shift(m_new)[:, None])
    return (m_new, a * l + p.sum(axis=1), a[:, None] * acc + p @ v)


def merge(x, y):
    """Combine two states over disjoint key sets."""
    m1, l1, a1 = x
    m2, l2, a2 = y
    m = np.maximum(m1, m2)
    ms = _shift(m)
    w1 = np.where(m1 > NEG_INF, np.exp(m1 - ms), 0.0)
    w2 = np.where(m2 > NEG_INF, np.exp(m2 - ms), 0.0)
    return (m, w1 * l1 + w2 * l2, w1[:, None] * a1 + w2[:, None] * a2)


def finish(state):
    m, l, acc = state
    seen = l > 0
    o = np.zeros_like(acc)
    o[seen] = acc[seen] / l[seen][:, None]
    lse = np.full(l.shape, NEG_INF)
    lse[seen] = m[seen] + np.log(l[seen])
    return o, lse


def incremental_attention(q, k, v, scale, vis, tile):
    """One head: q [R, d], k [Sk, d], v [Sk, dv], vis [R, Sk] bool.

    Processes the keys in tiles of ``tile`` (any size >= 1) with the update
    above and returns (o [R, dv], lse [R]).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    state = init_state(q.shape[0], v.shape[1])
    for j0 in range(0, k.shape[0], tile):
        j1 = min(j0 + tile, k.shape[0])
        s = scale * (q @ k[j0:j1].T)
        s = np.where(vis[:, j0:j1], s, NEG_INF)
        state = update(state, s, v[j0:j1])
    return finish(state)


# ---------------------------------------------------------------- moments
# The mean -> centred-sum-of-squares cascade in incremental form: a chunk's
# state is (n, mean, M2) with M2 = sum (x - mean)^2; two states merge as
#   n = na + nb, delta = mean_b - mean_a, mean = mean_a + delta * nb / n,
#   M2 = M2_a + M2_b + delta^2 * na * nb / n
# (the pairwise update of Chan, Golub and LeVeque), and var = M2 / n. This is
# the multi-segment form the GPU uses; it is checked against the two-pass
# definition in row_moments.

def moments_state(x):
    x = np.asarray(x, dtype=np.float64)
    n = x.size
    if n == 0:
        return (0, 0.0, 0.0)
    mean = x.sum() / n
    return (n, mean, float(((x - mean) ** 2).sum()))


def moments_merge(a, b):
    na, ma, qa = a
    nb, mb, qb = b
    n = na + nb
    if n == 0:
        return (0, 0.0, 0.0)
    delta = mb - ma
    return (n, ma + delta * nb / n, qa + qb + delta * delta * na * nb / n)


def weighted_state(points, masses):
    """(W, c, M2) of one chunk of point masses: W = sum m, c the weighted
    mean position, M2 = sum m |r - c|^2 (two passes over the chunk)."""
    r = np.asarray(points, dtype=np.float64).reshape(-1, np.shape(points)[-1])
    m = np.asarray(masses, dtype=np.float64).reshape(-1)
    W = m.sum()
    if W == 0:
        return (0.0, np.zeros(r.shape[1]), 0.0)
    c = (m[:, None] * r).sum(axis=0) / W
    return (W, c, float((m * ((r - c) ** 2).sum(axis=1)).sum()))


def weighted_merge(a, b):
    """Pairwise merge of (W, c, M2) states: the mass-weighted form of the
    count merge above (weights in place of counts)."""
    wa, ca, qa = a
    wb, cb, qb = b
    W = wa + wb
    if wb == 0:
        return a
    if wa == 0:
        return b
    delta = np.asarray(cb) - np.asarray(ca)
    return (W, ca + delta * (wb / W), qa + qb + float(delta @ delta) * wa * wb / W)
