"""MLA decode (absorbed form) on the tensor cores against the float64 oracle.

RedFuser page, section 4 (MLA workload) and section 3 (multi-segment
strategy): 128 query heads of one token attend to one latent key-value head
(576 key columns, the first 512 are the values); split over the keys, each
split's partial (O, LSE) on the tensor cores, merged by log-sum-exp. The
oracle is the plain attention definition with one key head and values equal
to the keys' leading 512 columns. Tolerances: bf16 O 2e-2, LSE 1e-3.
"""

import math

import numpy as np
import pytest

import oracle
from online_softmax_attention_rf_gb300 import api, inputs
from tests.helpers import TOL_BF16_LSE, TOL_BF16_O, assert_close, f64

pytestmark = pytest.mark.gpu


def _oracle(q, kv, scale, batches=None):
    qb = f64(q)[:, :, None, :]
    kb = f64(kv)[:, None]
    if batches is not None:
        qb, kb = qb[batches], kb[batches]
    o, lse = oracle.attention(qb, kb, kb[..., :512], scale)
    return o[:, :, 0, :], lse[:, :, 0]


@pytest.mark.parametrize("B,Sk,nsplit,amp", [
    (1, 32, 1, 1.0),        # one tile
    (2, 100, 3, 1.0),       # ragged tails
    (1, 1000, 8, 1.0),
    (3, 513, 1, 1.0),       # 17 tiles in one split
    (1, 1, 1, 1.0),         # a single key
    (2, 700, 2, 4.0),       # q x 4: large scores, the running maximum moves, O is rescaled
    (1, 64, 1, 1.0),        # exactly one 64-key tile
    (2, 130, 1, 1.0),       # two full tiles and a 2-key tail
    (1, 2049, 3, 1.0),      # more tiles per split than ring stages, ragged splits
    (2, 20, 20, 1.0),       # one key per split
    (1, 130, 2, 8.0),       # q x 8: the running maximum jumps between tiles
    # more segments than CTAs per value half (one per two SMs): each CTA folds a
    # run of segments, and runs cross batch elements
    (10, 1000, 20, 1.0),    # runs of 2-3 segments of 50 keys
    (100, 300, 3, 1.0),     # runs of ~4 segments over 2-3 batch elements
    (1, 20000, 200, 4.0),   # one batch element, runs of 2-3 segments of 100 keys
    (40, 4096, 16, 1.0),    # runs of 8-9 segments of 256 keys
])
def test_mla_decode_matches_oracle(cuda_device, B, Sk, nsplit, amp):
    q, kv = inputs.make_mla(B, Sk, B * 100 + Sk)
    q = (q.float() * amp).to(q.dtype)      # scores grow with q; the values (|O| ~ 1) do not
    scale = 1.0 / math.sqrt(192.0)
    o, lse = api.mla_decode(q.cuda(), kv.cuda(), nsplit, scale)
    assert api.device_status() == 0
    bs = None if B <= 10 else [0, 1, B // 2, B - 2, B - 1]   # sampled rows of large batches
    o_ref, lse_ref = _oracle(q, kv, scale, bs)
    if bs is not None:
        o, lse = o[bs], lse[bs]
    assert_close(o, o_ref, TOL_BF16_O, "O")
    assert_close(lse, lse_ref, TOL_BF16_LSE, "LSE")


def test_mla_split_invariance(cuda_device):
    """Any split of the keys gives the same result (the merge is exact in
    real arithmetic): 1, 5 and 16 splits agree within the bf16 bound."""
    q, kv = inputs.make_mla(2, 2048, 9)
    qd, kd = q.cuda(), kv.cuda()
    outs = [api.mla_decode(qd, kd, n, 0.07) for n in (1, 5, 16)]
    assert api.device_status() == 0
    for o, lse in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= TOL_BF16_O
        assert (lse - outs[0][1]).abs().max().item() <= TOL_BF16_LSE


def test_mla_full_size_sampled(cuda_device):
    """The benchmark workload (B = 32, Sk = 8192, 16 splits) in its launch
    configuration; three batch elements (all heads) against the oracle."""
    w = inputs.MLA_WORKLOADS["mla_decode"]
    q, kv = inputs.make_mla(w["B"], w["Sk"], w["seed"], w["amp"])
    o, lse = api.mla_decode(q.cuda(), kv.cuda(), w["nsplit"], w["scale"])
    assert api.device_status() == 0
    for b in (0, 17, 31):
        o_ref, lse_ref = _oracle(q[b:b + 1], kv[b:b + 1], w["scale"])
        assert_close(o[b:b + 1], o_ref, TOL_BF16_O, "O (b=%d)" % b)
        assert_close(lse[b:b + 1], lse_ref, TOL_BF16_LSE, "LSE (b=%d)" % b)
