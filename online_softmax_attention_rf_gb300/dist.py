"""Split-K decode with the keys sharded across ranks (one GPU per rank).

RedFuser: An Automatic Operator Fusion Framework for Cascaded Reductions on AI
Accelerators, section 3 (multi-segment strategy): the reduction's input is
partitioned, each segment produces a partial result, and the partial results
are merged. For attention decode the segments are contiguous ranges of the
key-value cache, the partial result of a segment is its (O_s, lse_s) pair, and
the merge is the log-sum-exp rule LSE = log sum_s exp(lse_s),
O = sum_s exp(lse_s - LSE) O_s. The merge is a commutative monoid, so the
segments may be merged in any grouping: within a rank first, then across
ranks.

One call, on every rank of a process group:

1. ``rf_attn_decode_partials``: the partials of ``nsplit_local`` splits of
   this rank's shard of the keys (device);
2. ``rf_splitk_merge`` (float32 out): the rank's own (O_r, lse_r), one partial
   per query row (device);
3. one all-gather of (O_r, lse_r) over the group -- B*H*(d + 1) floats per
   rank, the only exchange on the path. With NCCL the device tensors are
   gathered in place; with gloo through host copies;
4. ``rf_splitk_merge_strided``: the gathered split-major [world, B*H, d]
   partials merged straight from that layout into O (bf16) and LSE.

Every rank ends with the full result. No peer-memory loads, no multicast.
"""

import torch

from . import api


def exchange_partials(o_r, lse_r, group=None):
    """All-gather one float32 partial per row from every rank.

    o_r [rows, d], lse_r [rows] (same shape on every rank) -> (o_all
    [world, rows, d], lse_all [world, rows]) in rank order, on the device of
    the inputs. With a gloo group the exchange goes through host memory."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    backend = dist.get_backend(group)
    dev = o_r.device
    if backend == "nccl":
        o_all = torch.empty((world,) + tuple(o_r.shape), dtype=o_r.dtype, device=dev)
        lse_all = torch.empty((world,) + tuple(lse_r.shape), dtype=lse_r.dtype, device=dev)
        dist.all_gather_into_tensor(o_all, o_r.contiguous(), group=group)
        dist.all_gather_into_tensor(lse_all, lse_r.contiguous(), group=group)
        return o_all, lse_all
    o_h, l_h = o_r.detach().cpu().contiguous(), lse_r.detach().cpu().contiguous()
    o_list = [torch.empty_like(o_h) for _ in range(world)]
    l_list = [torch.empty_like(l_h) for _ in range(world)]
    dist.all_gather(o_list, o_h, group=group)
    dist.all_gather(l_list, l_h, group=group)
    return torch.stack(o_list).to(dev), torch.stack(l_list).to(dev)


def decode_splitk_sharded(q, k_shard, v_shard, nsplit_local, scale=None, group=None,
                          out_dtype=torch.bfloat16):
    """Decode attention over keys sharded across the ranks of ``group``.

    q [B, H, 1, d] (the same on every rank); k_shard, v_shard [B, Hkv, Sk_r, d]:
    this rank's contiguous range of the keys (ranks may hold different
    lengths, each at least nsplit_local keys). Returns (o [B, H, 1, d] of
    ``out_dtype``, lse float32 [B, H, 1]), identical on every rank."""
    B, H, _, d = q.shape
    o_part, lse_part = api.attn_decode_partials(q, k_shard, v_shard, nsplit_local, scale)
    o_r, lse_r = api.splitk_merge(o_part, lse_part, torch.float32)
    o_all, lse_all = exchange_partials(o_r, lse_r, group)
    o, lse = api.splitk_merge(o_all.permute(1, 0, 2), lse_all.permute(1, 0), out_dtype)
    return o.view(B, H, 1, d), lse.view(B, H, 1)
