"""The N > 1 bench path on the CPU: two ranks over gloo.

The attention path shards by (batch, head, query tile) with no exchange, so
the multi-rank bench runs one replica per rank (weak scaling) and its only
collectives are the barrier around the timed region and the max over ranks
of the elapsed time. These tests run that host logic on two gloo ranks
(127.0.0.1 rendezvous), and the reference arm under torchrun, where rank 0
alone times the oracle and prints the line.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist, r, w, local = bench.dist_setup(world)
    try:
        assert (r, w, local) == (rank, world, rank)
        assert dist.get_backend() == "gloo"
        bench.barrier(dist)
        # each rank's own elapsed time; every rank gets the slowest
        got = bench.max_over_ranks(dist, 10.0 + 3.5 * rank)
        with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
            json.dump({"max": got}, f)
        bench.barrier(dist)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for rank in range(world):
        with open(tmp_path / ("rank%d.json" % rank)) as f:
            assert json.load(f)["max"] == 13.5


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    sys.path.insert(0, ROOT)
    import bench
    dist, rank, world, local = bench.dist_setup(1)
    assert dist is None and (rank, world, local) == (0, 1, 0)
    assert bench.max_over_ranks(None, 2.5) == 2.5
    bench.barrier(None)


def test_reference_arm_under_torchrun_prints_once():
    """torchrun with two ranks: rank 0 prints one JSON line with the oracle's
    number, rank 1 does no work, both exit 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 1
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # the same metric, unit, direction and workload as the product arm, so
    # that the two lines compare
    sys.path.insert(0, ROOT)
    import bench
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s"
    assert line["higher_is_better"] is True
    assert line["config"]["workload"] == bench.WORKLOAD


def _shard_rank_main(rank, world, port, out_dir):
    """One rank of the key-sharded decode, on the CPU: the oracle's partials
    of this rank's shard stand in for the GPU partials, the rank merges them
    into one float32 partial per row, and exchange_partials gathers those
    over gloo."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    from online_softmax_attention_rf_gb300 import dist as rfdist
    from online_softmax_attention_rf_gb300 import inputs
    dist.init_process_group("gloo")
    try:
        B, H, Hkv, Sk, d = 2, 8, 2, 1000, 64
        q, k, v = inputs.make_qkv(B, H, Hkv, 1, Sk, d, 4, "bf16")
        bounds = [0, 300, 1000] if world == 2 else None
        a, e = bounds[rank], bounds[rank + 1]
        scale = inputs.default_scale(d)
        op, lp = oracle.decode_partials(q.double().numpy(), k[:, :, a:e].double().numpy(),
                                        v[:, :, a:e].double().numpy(), scale, 3)
        o_r, lse_r = oracle.merge_partials(op, lp)               # [B, H, d], [B, H]
        o_r = torch.from_numpy(o_r.reshape(B * H, d).astype(np.float32))
        lse_r = torch.from_numpy(lse_r.reshape(B * H).astype(np.float32))
        o_all, lse_all = rfdist.exchange_partials(o_r, lse_r)
        assert o_all.shape == (world, B * H, d) and lse_all.shape == (world, B * H)
        assert torch.equal(o_all[rank], o_r) and torch.equal(lse_all[rank], lse_r)
        # merge of the gathered split-major partials (rows first)
        o, lse = oracle.merge_partials(o_all.permute(1, 0, 2).double().numpy(),
                                       lse_all.permute(1, 0).double().numpy())
        o_ref, lse_ref = oracle.attention(q.double().numpy(), k.double().numpy(),
                                          v.double().numpy(), scale)
        err_o = float(np.abs(o - o_ref.reshape(B * H, d)).max())
        err_l = float(np.abs(lse - lse_ref.reshape(B * H)).max())
        with open(os.path.join(out_dir, "shard%d.json" % rank), "w") as f:
            json.dump({"err_o": err_o, "err_l": err_l}, f)
    finally:
        dist.destroy_process_group()


def test_key_sharded_decode_exchange_on_two_gloo_ranks(tmp_path):
    """Keys split 300 / 700 between two ranks: after the all-gather every
    rank merges the same partials, and the merge equals the unsplit
    attention (to float32 rounding of the exchanged partials)."""
    world = 2
    mp.start_processes(_shard_rank_main, args=(world, _free_port(), str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    for rank in range(world):
        with open(tmp_path / ("shard%d.json" % rank)) as f:
            r = json.load(f)
        assert r["err_o"] <= 1e-6 and r["err_l"] <= 1e-5, r
