"""Key-sharded split-K decode on the GPU (RedFuser, section 3, multi-segment
strategy: partition the keys, compute each segment's partial, merge).

The partials step alone (rf_attn_decode_partials) against the oracle's
per-split results; the strided merge of split-major partials against the
oracle's merge and, bit for bit, against the row-major merge of the same
values; and the whole sharded decode on two gloo ranks sharing this GPU
(the exchange runs on the host, so no kernel waits on another rank) against
the unsplit attention.
"""

import json
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from online_softmax_attention_rf_gb300 import api, inputs
from tests.helpers import TOL_BF16_LSE, TOL_BF16_O, TOL_F32, assert_close, f64

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode_partials_match_oracle(cuda_device):
    B, H, Hkv, Sk, d, ns = 2, 8, 2, 3000, 128, 5
    q, k, v = inputs.make_qkv(B, H, Hkv, 1, Sk, d, 31, "bf16")
    scale = inputs.default_scale(d)
    op, lp = api.attn_decode_partials(q.cuda(), k.cuda(), v.cuda(), ns, scale)
    assert api.device_status() == 0
    op_ref, lp_ref = oracle.decode_partials(f64(q), f64(k), f64(v), scale, ns)
    assert_close(op, op_ref.reshape(B * H, ns, d), TOL_BF16_O, "o_s")
    assert_close(lp, lp_ref.reshape(B * H, ns), TOL_BF16_LSE, "lse_s")


@pytest.mark.parametrize("world,rows,d", [(2, 37, 128), (4, 5, 64), (3, 9, 100)])
def test_strided_merge_of_split_major_partials(cuda_device, world, rows, d):
    rng = np.random.default_rng(world * rows)
    o_all = rng.standard_normal((world, rows, d)).astype(np.float32)
    lse_all = (rng.standard_normal((world, rows)) * 3).astype(np.float32)
    lse_all[0, 1] = -np.inf                       # an empty shard for one row
    lse_all[:, 2] = -np.inf                       # a row no shard sees
    og, lg = torch.from_numpy(o_all).cuda(), torch.from_numpy(lse_all).cuda()
    o, lse = api.splitk_merge(og.permute(1, 0, 2), lg.permute(1, 0), torch.float32)
    o_ref, lse_ref = oracle.merge_partials(o_all.transpose(1, 0, 2), lse_all.T)
    assert_close(o, o_ref, TOL_F32, "O")
    assert_close(lse, lse_ref, TOL_F32, "LSE")
    # the same values row-major: the identical arithmetic, bit for bit
    o2, l2 = api.splitk_merge(og.permute(1, 0, 2).contiguous(), lg.permute(1, 0).contiguous(),
                              torch.float32)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, bounds, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from online_softmax_attention_rf_gb300 import dist as rfdist
    torch.cuda.set_device(0)
    dist.init_process_group("gloo")
    try:
        B, H, Hkv, Sk, d = 2, 16, 4, bounds[-1], 128
        q, k, v = inputs.make_qkv(B, H, Hkv, 1, Sk, d, 33, "bf16")
        a, e = bounds[rank], bounds[rank + 1]
        ks, vs = k[:, :, a:e].contiguous().cuda(), v[:, :, a:e].contiguous().cuda()
        o, lse = rfdist.decode_splitk_sharded(q.cuda(), ks, vs, 4, inputs.default_scale(d))
        assert api.device_status() == 0
        torch.save({"o": o.cpu(), "lse": lse.cpu()}, os.path.join(out_dir, "r%d.pt" % rank))
    finally:
        dist.destroy_process_group()


def test_sharded_decode_two_gloo_ranks_on_one_gpu(cuda_device, tmp_path):
    bounds = [0, 5000, 12000]                     # unequal shards
    mp.start_processes(_rank_main, args=(2, _free_port(), bounds, str(tmp_path)), nprocs=2,
                       join=True, start_method="spawn")
    q, k, v = inputs.make_qkv(2, 16, 4, 1, bounds[-1], 128, 33, "bf16")
    o_ref, lse_ref = oracle.attention(f64(q), f64(k), f64(v), inputs.default_scale(128))
    res = [torch.load(tmp_path / ("r%d.pt" % r)) for r in range(2)]
    for r in res:
        assert_close(r["o"], o_ref, TOL_BF16_O, "O")
        assert_close(r["lse"], lse_ref, TOL_BF16_LSE, "LSE")
    assert torch.equal(res[0]["o"], res[1]["o"]) and torch.equal(res[0]["lse"], res[1]["lse"])
