"""Pins of the float64 oracle against things other than itself (CPU only).

Each pin is chosen so that a plausible mistake in the oracle (a dropped
scale, a wrong head mapping, top-left instead of bottom-right causal
alignment, log2 instead of ln, a transposed operand, a wrong split bound)
fails at least one of them; ``test_pins_catch_planted_mistakes`` plants such
mistakes in the oracle and checks that they are caught.

Pins used (the pages print no worked example and no error bound):
* brute force with Python ``math`` on tiny shapes;
* float64 library routines: ``torch.softmax``, ``torch.logsumexp`` and
  ``scaled_dot_product_attention`` with its own causal masks (top-left for
  square shapes, ``causal_lower_right`` for Sq != Sk);
* closed forms: a hand-solved 1x2 case, uniform scores, one dominant key,
  the first causal row;
* invariants: probabilities sum to one, invariance to a constant shift of a
  row's scores, split-K merge equal to the unsplit result, merge associative
  and commutative, GQA equal to MHA with repeated K/V heads, the online form
  equal to the three-pass form for any tiling;
* enumeration for the visited-tile set and the block-sparse row lists.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import three_pass as oa
from oracle import incremental as oi
from online_softmax_attention_rf_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

TOL = 1e-12
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _close(a, b, tol=TOL):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), "non-finite pattern differs"
    assert np.array_equal(a[~fin], b[~fin])
    if fin.any():
        err = np.max(np.abs(a[fin] - b[fin]) / np.maximum(1.0, np.abs(b[fin])))
        assert err <= tol, err


# --------------------------------------------------------------------------
# brute force with Python math


def _brute_visible(Sq, Sk, causal, tm, tile, em=None):
    """Visibility by explicit loops: bottom-right causal means the last query
    row sees every key and each earlier row one key fewer; an element mask
    removes single keys."""
    vis = [[True] * Sk for _ in range(Sq)]
    if em is not None:
        for i in range(Sq):
            for j in range(Sk):
                if not em[i][j]:
                    vis[i][j] = False
    for i in range(Sq):
        if causal:
            n_seen = Sk - (Sq - 1 - i)          # keys seen by row i
            for j in range(Sk):
                if j >= n_seen:
                    vis[i][j] = False
        if tm is not None:
            for j in range(Sk):
                if not tm[i // tile][j // tile]:
                    vis[i][j] = False
    return vis


def _brute_head(q, k, v, scale, vis):
    Sq, d = len(q), len(q[0])
    Sk, dv = len(k), len(v[0])
    o, lse = [], []
    for i in range(Sq):
        s = {}
        for j in range(Sk):
            if vis[i][j]:
                s[j] = scale * math.fsum(q[i][c] * k[j][c] for c in range(d))
        if not s:
            o.append([0.0] * dv)
            lse.append(-math.inf)
            continue
        m = max(s.values())
        l = math.fsum(math.exp(x - m) for x in s.values())
        o.append([math.fsum(math.exp(s[j] - m) / l * v[j][c] for j in s) for c in range(dv)])
        lse.append(m + math.log(l))
    return o, lse


def _brute_attention(q, k, v, scale, causal=False, tm=None, tile=2, em=None):
    B, H, Sq, _ = q.shape
    _, Hkv, Sk, _ = k.shape
    G = H // Hkv
    o = np.zeros((B, H, Sq, v.shape[-1]))
    lse = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            tmh = None if tm is None else (tm if tm.ndim == 2 else tm[b * H + h])
            emh = None if em is None else (em if em.ndim == 2 else em[b * H + h]).tolist()
            vis = _brute_visible(Sq, Sk, causal, None if tmh is None else tmh.tolist(), tile, emh)
            ob, lb = _brute_head(q[b, h].tolist(), k[b, h // G].tolist(), v[b, h // G].tolist(),
                                 scale, vis)
            o[b, h], lse[b, h] = ob, lb
    return o, lse


BRUTE_CASES = [
    # B, H, Hkv, Sq, Sk, d, causal, tile-mask
    (1, 1, 1, 5, 7, 3, False, False),
    (2, 2, 1, 6, 6, 4, True, False),
    (1, 4, 2, 4, 8, 2, True, False),
    (1, 2, 2, 8, 5, 3, True, False),     # Sq > Sk: early rows see nothing
    (2, 3, 3, 7, 8, 4, False, True),
    (1, 2, 1, 8, 8, 3, True, True),
]


@pytest.mark.parametrize("causal,per_head", [(False, False), (True, True)])
def test_brute_force_element_mask(causal, per_head):
    """Attention under an element mask (STOF's inner level) equals explicit
    loops that drop every masked (query, key) pair."""
    B, H, Hkv, Sq, Sk, d = 1, 2, 1, 6, 7, 3
    q, k, v = _rand((B, H, Sq, d), 11), _rand((B, Hkv, Sk, d), 12), _rand((B, Hkv, Sk, d), 13)
    rng = np.random.default_rng(14)
    em = rng.random((B * H, Sq, Sk) if per_head else (Sq, Sk)) < 0.5
    o, lse = oracle.attention(q, k, v, 0.9, causal, elem_mask=em)
    ob, lb = _brute_attention(q, k, v, 0.9, causal, None, 2, em)
    _close(o, ob)
    _close(lse, lb)


def test_element_mask_special_cases():
    """An all-true element mask changes nothing; one that is constant over
    each tile is the same as the tile mask."""
    B, H, Sq, Sk, d, tile = 1, 2, 9, 10, 4, 3
    q, k, v = _rand((B, H, Sq, d), 21), _rand((B, H, Sk, d), 22), _rand((B, H, Sk, d), 23)
    base = oracle.attention(q, k, v, 0.5, True)
    allt = oracle.attention(q, k, v, 0.5, True, elem_mask=np.ones((Sq, Sk), bool))
    _close(allt[0], base[0])
    _close(allt[1], base[1])
    tm = np.random.default_rng(24).random((-(-Sq // tile), -(-Sk // tile))) < 0.5
    em = np.repeat(np.repeat(tm, tile, 0), tile, 1)[:Sq, :Sk]
    a = oracle.attention(q, k, v, 0.5, False, tm, tile)
    b = oracle.attention(q, k, v, 0.5, False, elem_mask=em)
    _close(a[0], b[0])
    _close(a[1], b[1])


def test_two_level_format_examples():
    """The words the pages describe: one uint64 per 8x8 inner block of a
    partial outer tile (bit 8r + c = element (r, c), the reading taken);
    full tiles carry no bitmap; a tile with no valid element is not listed."""
    m = np.zeros((1, 256, 384), bool)
    m[0, 0, :8] = True                 # tile (0,0): first row of inner block (0,0)
    m[0, 9, 16] = True                 # tile (0,0): inner block (1,2), element (1,0)
    m[0, 128:, 256:] = True            # tile (1,2): full
    m[0, 130, 131] = True              # tile (1,1): inner block (0,0), element (2,3)
    rp, ci, tb, bits = oracle.two_level_encode(m)
    assert rp.tolist() == [0, 1, 3] and ci.tolist() == [0, 1, 2] and tb.tolist() == [0, 1, -1]
    w0 = bits[0]
    assert int(w0[0]) == 0xFF and int(w0[1 * 16 + 2]) == 1 << 8
    assert np.count_nonzero(w0) == 2
    assert int(bits[1][0]) == 1 << (2 * 8 + 3) and np.count_nonzero(bits[1]) == 1
    # a block whose 64 elements are all valid is the all-ones word
    m2 = np.zeros((1, 128, 128), bool)
    m2[0, 8:16, 16:24] = True
    assert int(oracle.two_level_encode(m2)[3][0][1 * 16 + 2]) == 0xFFFFFFFFFFFFFFFF


@pytest.mark.parametrize("shape,density", [((2, 300, 200), 0.02), ((1, 129, 257), 0.5),
                                           ((3, 64, 64), 0.9)])
def test_two_level_round_trip(shape, density):
    rng = np.random.default_rng(int(density * 100) + shape[1])
    m = rng.random(shape) < density
    m[0, :, :64] = True                # whole tiles valid: listed as full
    rp, ci, tb, bits = oracle.two_level_encode(m)
    assert (oracle.two_level_decode(rp, ci, tb, bits, *shape) == m).all()
    # listed tiles are exactly the tiles holding a valid element
    tiles = np.zeros((shape[0], -(-shape[1] // 128), -(-shape[2] // 128)), bool)
    for h, i, j in zip(*np.nonzero(m)):
        tiles[h, i // 128, j // 128] = True
    rp2, ci2 = oracle.bsr_from_tile_mask(tiles)
    assert np.array_equal(rp, rp2) and np.array_equal(ci, ci2)


@pytest.mark.parametrize("case", BRUTE_CASES)
def test_brute_force_tiny(case):
    B, H, Hkv, Sq, Sk, d, causal, use_tm = case
    q = _rand((B, H, Sq, d), 1)
    k = _rand((B, Hkv, Sk, d), 2)
    v = _rand((B, Hkv, Sk, d + 1), 3)
    tile = 2
    tm = None
    if use_tm:
        tm = np.random.default_rng(4).random((B * H, -(-Sq // tile), -(-Sk // tile))) < 0.6
    scale = 0.7
    o, lse = oracle.attention(q, k, v, scale, causal, tm, tile)
    ob, lb = _brute_attention(q, k, v, scale, causal, tm, tile)
    _close(o, ob)
    _close(lse, lb)


def test_closed_form_one_row():
    # q = (1, 0); keys (1, 0) and (0, 1); values (1, 2) and (3, 4); scale 1.
    # scores (1, 0): p = (e, 1) / (1 + e); O = (e + 3, 2e + 4) / (1 + e);
    # LSE = ln(1 + e).
    e = math.e
    q = np.array([[[[1.0, 0.0]]]])
    k = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    v = np.array([[[[1.0, 2.0], [3.0, 4.0]]]])
    o, lse = oracle.attention(q, k, v, 1.0)
    _close(o[0, 0, 0], [(e + 3) / (1 + e), (2 * e + 4) / (1 + e)])
    _close(lse[0, 0, 0], math.log(1 + e))


# --------------------------------------------------------------------------
# float64 library routines


def _torch_reference(q, k, v, scale, causal, tm=None, tile=128):
    """softmax(QK^T scale + mask) V and logsumexp, float64 torch on CPU."""
    q, k, v = (torch.from_numpy(np.asarray(x, np.float64)) for x in (q, k, v))
    G = q.shape[1] // k.shape[1]
    k = k.repeat_interleave(G, dim=1)
    v = v.repeat_interleave(G, dim=1)
    s = torch.matmul(q, k.transpose(-1, -2)) * scale
    Sq, Sk = s.shape[-2:]
    keep = torch.ones(Sq, Sk, dtype=torch.bool)
    if causal:
        keep = torch.ones(Sq, Sk, dtype=torch.bool).tril(diagonal=Sk - Sq)
    keep = keep.expand(s.shape).clone()
    if tm is not None:
        t = torch.from_numpy(np.asarray(tm, bool))
        t = t.repeat_interleave(tile, -2).repeat_interleave(tile, -1)[..., :Sq, :Sk]
        if t.dim() == 3:
            t = t.reshape(s.shape[0], s.shape[1], Sq, Sk)
        keep = keep & t
    s = s.masked_fill(~keep, -math.inf)
    lse = torch.logsumexp(s, dim=-1)
    p = torch.softmax(s, dim=-1).nan_to_num(0.0)
    return (p @ v).numpy(), lse.numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_torch_softmax_library(causal):
    B, H, Hkv, S, d = 2, 4, 2, 300, 64
    q = _rand((B, H, S, d), 10)
    k = _rand((B, Hkv, S, d), 11)
    v = _rand((B, Hkv, S, d), 12)
    o, lse = oracle.attention(q, k, v, 0.125, causal)
    ot, lt = _torch_reference(q, k, v, 0.125, causal)
    _close(o, ot)
    _close(lse, lt)


def test_torch_tile_mask_library():
    B, H, S, d, tile = 1, 2, 512, 32, 128
    q, k, v = _rand((B, H, S, d), 13), _rand((B, H, S, d), 14), _rand((B, H, S, d), 15)
    tm = inputs.window_random_tile_mask(4, window=2, frac=0.5, seed=3)
    o, lse = oracle.attention(q, k, v, 0.2, False, tm, tile)
    ot, lt = _torch_reference(q, k, v, 0.2, False, tm, tile)
    _close(o, ot)
    _close(lse, lt)


def test_sdpa_top_left_causal_square():
    # torch's own causal mask (is_causal, top-left) coincides with bottom-right
    # alignment when Sq == Sk
    q, k, v = (_rand((2, 3, 129, 16), s) for s in (20, 21, 22))
    o, _ = oracle.attention(q, k, v, 0.25, causal=True)
    t = [torch.from_numpy(x) for x in (q, k, v)]
    ot = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=True, scale=0.25)
    _close(o, ot.numpy())


def test_sdpa_latent_kv_heads():
    """Multi-head latent attention decode as the oracle computes it: many
    query heads against one key head whose first dv columns are the values
    (d_qk = latent + rope, d_v = latent), pinned by torch's SDPA with the
    key head broadcast and v the key's leading columns."""
    B, H, Sk, d, dv = 2, 8, 150, 24, 16
    q = _rand((B, H, 1, d), 33)
    kv = _rand((B, 1, Sk, d), 34)
    o, lse = oracle.attention(q, kv, kv[..., :dv], 0.2)
    tq = torch.from_numpy(q)
    tk = torch.from_numpy(kv).expand(B, H, Sk, d)
    ot = torch.nn.functional.scaled_dot_product_attention(tq, tk, tk[..., :dv], scale=0.2)
    _close(o, ot.numpy())
    s = 0.2 * (tq @ tk.transpose(-1, -2))
    _close(lse, torch.logsumexp(s, dim=-1).numpy())


def test_sdpa_lower_right_causal():
    # bottom-right alignment for Sq != Sk, pinned by torch's causal_lower_right
    from torch.nn.attention.bias import causal_lower_right
    Sq, Sk = 37, 101
    q, k, v = _rand((1, 2, Sq, 8), 30), _rand((1, 2, Sk, 8), 31), _rand((1, 2, Sk, 8), 32)
    o, _ = oracle.attention(q, k, v, 0.3, causal=True)
    t = [torch.from_numpy(x) for x in (q, k, v)]
    ot = torch.nn.functional.scaled_dot_product_attention(
        *t, attn_mask=causal_lower_right(Sq, Sk), scale=0.3)
    _close(o, ot.numpy())


# --------------------------------------------------------------------------
# closed forms and invariants


def test_probabilities_sum_to_one():
    # with V = identity, O is the probability matrix P itself (Sq <= Sk, so
    # every causal row sees at least one key)
    Sq, Sk, d = 30, 33, 8
    q, k = _rand((1, 1, Sq, d), 40), _rand((1, 1, Sk, d), 41)
    eye = np.eye(Sk)[None, None]
    for causal in (False, True):
        p, _ = oracle.attention(q, k, eye, 0.5, causal)
        assert np.all(p >= 0)
        _close(p.sum(-1), np.ones((1, 1, Sq)))


def test_shift_invariance():
    # an extra column (c/scale in q, 1 in k) adds c to every score of a row
    Sq, Sk, d, scale, c = 20, 50, 16, 0.125, 3.75
    q, k, v = _rand((1, 2, Sq, d), 50), _rand((1, 2, Sk, d), 51), _rand((1, 2, Sk, d), 52)
    o, lse = oracle.attention(q, k, v, scale, True)
    q2 = np.concatenate([q, np.full((1, 2, Sq, 1), c / scale)], -1)
    k2 = np.concatenate([k, np.ones((1, 2, Sk, 1))], -1)
    o2, lse2 = oracle.attention(q2, k2, v, scale, True)
    _close(o2, o)
    _close(lse2, lse + c)


def test_uniform_scores_give_mean_of_v():
    Sk = 77
    q, v = _rand((2, 3, 5, 8), 60), _rand((2, 3, Sk, 8), 61)
    o, lse = oracle.attention(q, np.zeros((2, 3, Sk, 8)), v, 0.3)
    _close(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape))
    _close(lse, np.full(lse.shape, math.log(Sk)))


def test_dominant_score_selects_its_value_row():
    Sk, j0, scale = 64, 41, 0.125
    q = np.zeros((1, 1, 1, 4))
    q[..., 0] = 1.0
    k = _rand((1, 1, Sk, 4), 70, 1e-3)
    k[0, 0, j0, 0] = 1e3
    v = _rand((1, 1, Sk, 6), 71)
    o, lse = oracle.attention(q, k, v, scale)
    _close(o[0, 0, 0], v[0, 0, j0], 1e-12)
    s0 = scale * float(q[0, 0, 0] @ k[0, 0, j0])
    _close(lse[0, 0, 0], s0, 1e-12)


def test_causal_first_row():
    S = 31
    q, k, v = _rand((1, 2, S, 8), 80), _rand((1, 2, S, 8), 81), _rand((1, 2, S, 8), 82)
    o, lse = oracle.attention(q, k, v, 0.4, causal=True)
    _close(o[:, :, 0], v[:, :, 0])
    _close(lse[:, :, 0], 0.4 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]))


def test_rows_without_visible_keys():
    # causal with Sq > Sk: rows i < Sq - Sk see no key
    Sq, Sk = 10, 4
    q, k, v = _rand((1, 1, Sq, 4), 90), _rand((1, 1, Sk, 4), 91), _rand((1, 1, Sk, 4), 92)
    o, lse = oracle.attention(q, k, v, 1.0, causal=True)
    assert np.all(o[0, 0, :Sq - Sk] == 0) and np.all(lse[0, 0, :Sq - Sk] == -np.inf)
    assert np.all(np.isfinite(lse[0, 0, Sq - Sk:]))
    # an empty tile mask hides every key
    o, lse = oracle.attention(q, k, v, 1.0, False, np.zeros((1, 1), bool), tile=16)
    assert np.all(o == 0) and np.all(lse == -np.inf)


def test_gqa_equals_mha_with_repeated_heads():
    B, H, Hkv, S, d = 2, 8, 2, 45, 16
    q, k, v = _rand((B, H, S, d), 100), _rand((B, Hkv, S, d), 101), _rand((B, Hkv, S, d), 102)
    o, lse = oracle.attention(q, k, v, 0.25, True)
    rep = H // Hkv
    o2, lse2 = oracle.attention(q, np.repeat(k, rep, 1), np.repeat(v, rep, 1), 0.25, True)
    _close(o, o2)
    _close(lse, lse2)


# --------------------------------------------------------------------------
# split-K partials and the log-sum-exp merge


@pytest.mark.parametrize("Sk,nsplit", [(4096, 32), (1000, 7), (33, 33), (50, 1)])
def test_split_merge_equals_unsplit(Sk, nsplit):
    B, H, Hkv, d = 2, 8, 2, 16
    q, k, v = _rand((B, H, 1, d), 110), _rand((B, Hkv, Sk, d), 111), _rand((B, Hkv, Sk, d), 112)
    op, lp = oracle.decode_partials(q, k, v, 0.25, nsplit)
    o, lse = oracle.merge_partials(op, lp)
    ou, lu = oracle.attention(q, k, v, 0.25)
    _close(o, ou[:, :, 0])
    _close(lse, lu[:, :, 0])


def test_split_bounds():
    assert oracle.split_bounds(65536, 32)[5] == (10240, 12288)
    b = oracle.split_bounds(1000, 7)
    assert b[0] == (0, 142) and b[-1] == (852, 1000)
    assert all(b[i][1] == b[i + 1][0] for i in range(6))
    with pytest.raises(ValueError):
        oracle.split_bounds(3, 4)


def test_merge_associative_commutative_and_identity():
    R, d = 6, 5
    parts = [(_rand((R, d), 120 + i), _rand((R,), 130 + i, 4.0)) for i in range(4)]
    o_all, l_all = oracle.merge_partials(np.stack([p[0] for p in parts], 1),
                                         np.stack([p[1] for p in parts], 1))

    def m2(a, b):
        return oracle.merge_partials(np.stack([a[0], b[0]], 1), np.stack([a[1], b[1]], 1))

    left = m2(m2(m2(parts[0], parts[1]), parts[2]), parts[3])
    right = m2(parts[0], m2(parts[1], m2(parts[2], parts[3])))
    perm = m2(m2(parts[3], parts[1]), m2(parts[2], parts[0]))
    for o, l in (left, right, perm):
        _close(o, o_all)
        _close(l, l_all)
    # (O = 0, lse = -inf) is the identity; an all -inf row merges to (0, -inf)
    ident = (np.zeros((R, d)), np.full(R, -np.inf))
    o, l = m2(parts[0], ident)
    _close(o, parts[0][0])
    _close(l, parts[0][1])
    o, l = m2(ident, ident)
    assert np.all(o == 0) and np.all(l == -np.inf)


def test_merge_closed_form_two_splits():
    # lse = (0, ln 3): weights 1/4, 3/4; LSE = ln 4
    o, lse = oracle.merge_partials(np.array([[[1.0, 0.0], [0.0, 1.0]]]),
                                   np.array([[0.0, math.log(3.0)]]))
    _close(o[0], [0.25, 0.75])
    _close(lse[0], math.log(4.0))


# --------------------------------------------------------------------------
# the online form reaches the three-pass result (the derivation the GPU uses)


@pytest.mark.parametrize("tile", [1, 7, 128, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_incremental_form_equals_three_pass(tile, causal):
    Sq, Sk, d = 70, 300, 16
    q, k, v = _rand((Sq, d), 140, 2.0), _rand((Sk, d), 141, 2.0), _rand((Sk, d), 142)
    vis = oracle.visible_mask(Sq, Sk, causal)
    o, lse = oi.incremental_attention(q, k, v, 0.3, vis, tile)
    o3, l3 = oracle.attention(q[None, None], k[None, None], v[None, None], 0.3, causal)
    _close(o, o3[0, 0])
    _close(lse, l3[0, 0])


def test_incremental_states_merge_as_a_monoid():
    Sq, Sk, d = 9, 120, 8
    q, k, v = _rand((Sq, d), 150), _rand((Sk, d), 151), _rand((Sk, d), 152)

    def state(a, b):
        st = oi.init_state(Sq, d)
        return oi.update(st, 0.5 * (q @ k[a:b].T), v[a:b])

    whole = oi.finish(state(0, Sk))
    x, y, z = state(0, 40), state(40, 41), state(41, Sk)
    for st in (oi.merge(oi.merge(x, y), z), oi.merge(x, oi.merge(y, z)), oi.merge(z, oi.merge(y, x)),
               oi.merge(oi.init_state(Sq, d), oi.merge(x, oi.merge(y, z)))):
        o, l = oi.finish(st)
        _close(o, whole[0])
        _close(l, whole[1])


# --------------------------------------------------------------------------
# row softmax


def test_softmax_rows_brute_and_library():
    x = _rand((7, 33), 160, 5.0)
    y = oracle.softmax_rows(x)
    for r in range(7):
        m = max(x[r])
        e = [math.exp(t - m) for t in x[r]]
        tot = math.fsum(e)
        _close(y[r], [t / tot for t in e])
    _close(y, torch.softmax(torch.from_numpy(x), -1).numpy())
    _close(y.sum(1), np.ones(7))
    _close(oracle.softmax_rows(x + 123.0), y)   # shift invariance


def test_softmax_rows_masked_entries():
    x = _rand((3, 10), 170)
    x[0, 3:] = -np.inf
    x[2, :] = -np.inf
    y = oracle.softmax_rows(x)
    _close(y[0, :3], torch.softmax(torch.from_numpy(x[0, :3]), -1).numpy())
    assert np.all(y[0, 3:] == 0) and np.all(y[2] == 0)


# --------------------------------------------------------------------------
# visited tiles and block-sparse row lists


def _brute_visited(Sq, Sk, causal, tm, tile):
    vis = _brute_visible(Sq, Sk, causal, None if tm is None else tm.tolist(), tile)
    nqt, nkt = -(-Sq // tile), -(-Sk // tile)
    out = np.zeros((nqt, nkt), bool)
    for i in range(Sq):
        for j in range(Sk):
            if vis[i][j]:
                out[i // tile, j // tile] = True
    return out


@pytest.mark.parametrize("Sq,Sk,causal,use_tm", [
    (20, 20, True, False), (13, 29, True, False), (29, 13, True, False),
    (24, 24, False, True), (21, 30, True, True)])
def test_visited_tiles_by_enumeration(Sq, Sk, causal, use_tm):
    tile = 4
    tm = None
    if use_tm:
        tm = np.random.default_rng(Sq * Sk).random((-(-Sq // tile), -(-Sk // tile))) < 0.5
    got = oracle.visited_tiles(Sq, Sk, causal, tm, tile)
    assert np.array_equal(got, _brute_visited(Sq, Sk, causal, tm, tile))


def test_visited_tiles_causal_square_is_lower_triangle():
    got = oracle.visited_tiles(1024, 1024, True, None, 128)
    assert np.array_equal(got, np.tril(np.ones((8, 8), bool)))


def test_bsr_from_tile_mask_by_enumeration():
    tm = np.random.default_rng(5).random((3, 6, 9)) < 0.4
    row_ptr, col_idx = oracle.bsr_from_tile_mask(tm)
    assert row_ptr[0] == 0 and row_ptr[-1] == tm.sum() and len(row_ptr) == 19
    r = 0
    for h in range(3):
        for i in range(6):
            cols = [j for j in range(9) if tm[h, i, j]]
            assert list(col_idx[row_ptr[r]:row_ptr[r + 1]]) == cols
            r += 1


def test_window_random_mask_counts():
    # 128 tiles per side: window (0 <= i-j <= 7) holds 996 tiles, 7260 lower
    # tiles remain and 726 of them are drawn: 1722 in all
    tm = inputs.window_random_tile_mask(128, 8, 0.1, 4)
    i, j = np.nonzero(tm)
    assert tm.sum() == 1722
    assert np.all(i >= j)
    assert (((i - j) <= 7)).sum() == 996
    assert np.array_equal(tm, inputs.window_random_tile_mask(128, 8, 0.1, 4))


# --------------------------------------------------------------------------
# stored regression values (written by tests/golden/make_golden.py, oracle only)


def test_golden_fixture():
    with open(os.path.join(GOLDEN, "oracle_small_cases.json")) as f:
        cases = json.load(f)["cases"]
    assert cases
    for c in cases:
        q, k, v = (np.array(c[n], np.float64) for n in ("q", "k", "v"))
        tm = None if c["tile_mask"] is None else np.array(c["tile_mask"], bool)
        o, lse = oracle.attention(q, k, v, c["scale"], c["causal"], tm, c["tile"])
        _close(o, np.array(c["o"]), 1e-13)
        _close(lse, np.array(c["lse"], dtype=np.float64), 1e-13)


# --------------------------------------------------------------------------
# planted mistakes are caught


def _mutant_no_scale(q, k, v, scale, vis):
    return _orig_three_pass(q, k, v, 1.0, vis)


def _mutant_log2(q, k, v, scale, vis):
    o, lse = _orig_three_pass(q, k, v, scale, vis)
    return o, lse / math.log(2.0)


def _mutant_transposed_v(q, k, v, scale, vis):
    o, lse = _orig_three_pass(q, k, v[::-1], scale, vis)
    return o, lse


def _mutant_no_normalise(q, k, v, scale, vis):
    o, lse = _orig_three_pass(q, k, v, scale, vis)
    return o * 1.5, lse


_orig_three_pass = oa._three_pass
_orig_visible = oa.visible_mask


def _mutant_top_left(Sq, Sk, causal, tile_mask=None, tile=128, rows=None, elem_mask=None):
    vis = _orig_visible(Sq, Sk, False, tile_mask, tile, rows, elem_mask)
    if causal:
        rows = np.arange(Sq) if rows is None else np.asarray(rows)
        vis &= np.arange(Sk)[None, :] <= rows[:, None]
    return vis


def _mutant_no_elem_mask(Sq, Sk, causal, tile_mask=None, tile=128, rows=None, elem_mask=None):
    return _orig_visible(Sq, Sk, causal, tile_mask, tile, rows)


def _pins():
    yield lambda: test_brute_force_element_mask(True, True)
    yield lambda: test_brute_force_tiny(BRUTE_CASES[1])
    yield lambda: test_brute_force_tiny(BRUTE_CASES[3])
    yield test_closed_form_one_row
    yield test_sdpa_lower_right_causal
    yield test_uniform_scores_give_mean_of_v


@pytest.mark.parametrize("target,mutant", [
    ("_three_pass", _mutant_no_scale), ("_three_pass", _mutant_log2),
    ("_three_pass", _mutant_transposed_v), ("_three_pass", _mutant_no_normalise),
    ("visible_mask", _mutant_top_left), ("visible_mask", _mutant_no_elem_mask)])
def test_pins_catch_planted_mistakes(monkeypatch, target, mutant):
    monkeypatch.setattr(oa, target, mutant)
    failures = 0
    for pin in _pins():
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures >= 1, "no pin caught the planted mistake"
