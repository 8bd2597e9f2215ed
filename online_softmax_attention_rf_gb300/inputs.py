"""Seeded synthetic inputs shared by the CUDA path and the CPU oracle.

This module holds none of the method's arithmetic: it only draws numbers and
builds masks, so that the oracle and the GPU consume identical bytes. The
workloads follow the attention shapes of the pages' evaluation (multi-head and
grouped-query prefill, split-K decode, block-sparse attention with the mask
families STOF evaluates: causal, sliding window, Longformer/Bigbird-like).
No dataset or trained weight is involved; every tensor is drawn here.

Recipe: ``torch.Generator().manual_seed(seed)`` on the CPU, ``torch.randn``
in float32 for Q, then K, then V (in that order, from one generator),
multiplied by ``amp`` and cast to the workload dtype.
"""

import math

import numpy as np
import torch

#: The named workloads. ``tile`` is the block-sparse tile side.
WORKLOADS = {
    # tiny exact case, fp32 in and out
    "tiny_fp32": dict(B=1, H=1, Hkv=1, Sq=128, Sk=128, d=64, causal=False,
                      dtype="f32", seed=0, amp=1.0),
    # multi-head causal prefill
    "mha_prefill": dict(B=4, H=32, Hkv=32, Sq=4096, Sk=4096, d=128, causal=True,
                        dtype="bf16", seed=1, amp=1.0),
    # grouped-query long-context causal prefill
    "gqa_long": dict(B=1, H=64, Hkv=8, Sq=32768, Sk=32768, d=128, causal=True,
                     dtype="bf16", seed=2, amp=0.5),
    # split-K decode, one query row per head
    "decode_splitk": dict(B=16, H=32, Hkv=8, Sq=1, Sk=65536, d=128, nsplit=32,
                          causal=False, dtype="bf16", seed=3, amp=1.0),
    # block-sparse: sliding window of 8 tiles, diagonal, 10% random lower tiles
    "block_sparse": dict(B=2, H=16, Hkv=16, Sq=16384, Sk=16384, d=64, causal=False,
                         dtype="bf16", seed=4, amp=1.0, tile=128, window=8, frac=0.1),
    # two-level (element) mask, Longformer-like: keys within `band` of the
    # query row, plus `n_global` global tokens (first keys, seen by every row;
    # first rows, which see every key)
    "two_level": dict(B=2, H=16, Hkv=16, Sq=16384, Sk=16384, d=64, causal=False,
                      dtype="bf16", seed=8, amp=1.0, band=256, n_global=64),
    # short sequences under a scattered (Bigbird-like) element mask: window
    # 16, 8 global tokens, 1 % random keys -- the row-wise kernel's regime
    "scattered_short": dict(B=16, H=16, Hkv=16, Sq=1024, Sk=1024, d=64, causal=False,
                            dtype="bf16", seed=11, amp=1.0, window=16, n_global=8,
                            density=0.01),
}

#: Row-softmax shapes (rows, cols): one row fits a CTA; one row spans a cluster.
SOFTMAX_WORKLOADS = {
    "rows_64k": dict(rows=16384, cols=16384, seed=5),
    "rows_1m": dict(rows=1024, cols=262144, seed=6),
}

#: Other cascaded reductions. MoE routing: router logits of a prefill batch
#: for a 256-expert, top-8 model (float32 logits, N(0, amp^2)). Row moments:
#: normalisation-layer rows (float32, N(offset, amp^2): a mean far from zero
#: relative to the spread is the case a one-pass sum of squares gets wrong).
#: Inertia: sets of point masses in 3-D.
CASCADE_WORKLOADS = {
    "moe_route": dict(T=131072, E=256, k=8, renorm=True, dtype="f32", seed=9, amp=2.0),
    "row_moments": dict(rows=16384, cols=8192, dtype="f32", seed=10, amp=1.0, offset=8.0,
                        eps=1e-5),
    # point sets: positions N(offset, amp^2) per coordinate, masses U(0.5, 1.5)
    "inertia": dict(sets=2048, n=32768, seed=12, amp=2.0, offset=5.0),
    # a linear layer in FP8: activations A [M, K] and weights W [N, K], bf16
    # N(0, 1) before per-row quantisation
    "fp8_gemm": dict(M=8192, N=8192, K=8192, seed=13),
}

#: MLA decode, absorbed form: 128 query heads of one token against one latent
#: head (512 latent + 64 rotary columns), values = the latent columns; scale
#: 1 / sqrt(128 + 64) (the unabsorbed query-key dimension).
MLA_WORKLOADS = {
    "mla_decode": dict(B=32, Sk=8192, nsplit=16, seed=14, amp=1.0,
                       scale=1.0 / math.sqrt(192.0)),
}

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def default_scale(d):
    """1/sqrt(d), the scale used by every workload."""
    return 1.0 / math.sqrt(d)


def make_qkv(B, H, Hkv, Sq, Sk, d, seed, dtype="bf16", amp=1.0, dv=None):
    """Q [B,H,Sq,d], K [B,Hkv,Sk,d], V [B,Hkv,Sk,dv] on the CPU, contiguous."""
    g = torch.Generator().manual_seed(seed)
    dv = d if dv is None else dv
    td = TORCH_DTYPES[dtype]
    q = (torch.randn(B, H, Sq, d, generator=g) * amp).to(td)
    k = (torch.randn(B, Hkv, Sk, d, generator=g) * amp).to(td)
    v = (torch.randn(B, Hkv, Sk, dv, generator=g) * amp).to(td)
    return q, k, v


def make_rows(rows, cols, seed, dtype="f32", amp=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, cols, generator=g) * amp).to(TORCH_DTYPES[dtype])


def make_logits(T, E, seed, dtype="f32", amp=1.0, ties=False):
    """Router logits [T, E]; ``ties`` draws small integers so that many are equal."""
    g = torch.Generator().manual_seed(seed)
    if ties:
        x = torch.randint(-3, 4, (T, E), generator=g).to(torch.float32)
    else:
        x = torch.randn(T, E, generator=g) * amp
    return x.to(TORCH_DTYPES[dtype])


def make_moment_rows(rows, cols, seed, dtype="f32", amp=1.0, offset=0.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, cols, generator=g) * amp + offset).to(TORCH_DTYPES[dtype])


def make_gemm_operands(M, N, K, seed, dtype="bf16"):
    """(A [M, K], W [N, K]) drawn N(0, 1) on the CPU, in that order."""
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(M, K, generator=g).to(TORCH_DTYPES[dtype])
    w = torch.randn(N, K, generator=g).to(TORCH_DTYPES[dtype])
    return a, w


def make_mla(B, Sk, seed, amp=1.0):
    """(q bf16 [B, 128, 576], kv bf16 [B, Sk, 576]) drawn N(0, amp^2), q first."""
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, 128, 576, generator=g) * amp).to(torch.bfloat16)
    kv = (torch.randn(B, Sk, 576, generator=g) * amp).to(torch.bfloat16)
    return q, kv


def make_point_sets(sets, n, seed, amp=1.0, offset=0.0):
    """(points float32 [sets, n, 3], masses float32 [sets, n])."""
    g = torch.Generator().manual_seed(seed)
    points = torch.randn(sets, n, 3, generator=g) * amp + offset
    masses = torch.rand(sets, n, generator=g) + 0.5
    return points, masses


def n_tiles(S, tile=128):
    return -(-S // tile)


def window_random_tile_mask(nqt, window=8, frac=0.1, seed=4):
    """bool [nqt, nqt]: sliding window, diagonal, and random lower tiles.

    Tile (i, j) is in the window when 0 <= i - j <= window - 1 (the diagonal
    is part of it). Of the strictly-lower tiles outside the window, listed in
    row-major order, round(frac * count) are drawn uniformly without
    replacement by ``numpy.random.default_rng(seed).choice``.
    """
    i = np.arange(nqt)[:, None]
    j = np.arange(nqt)[None, :]
    mask = (i - j >= 0) & (i - j <= window - 1)
    rest = np.argwhere(i - j >= window)          # row-major order
    k = int(round(frac * len(rest)))
    if k:
        pick = np.random.default_rng(seed).choice(len(rest), k, replace=False)
        sel = rest[pick]
        mask[sel[:, 0], sel[:, 1]] = True
    return mask


def band_global_mask(S, band, n_global, rows=None):
    """bool [len(rows), S] element mask: |i - j| <= band, or j < n_global, or
    i < n_global (all rows by default; built in row blocks to bound memory)."""
    rows = np.arange(S) if rows is None else np.asarray(rows)
    out = np.zeros((rows.size, S), dtype=bool)
    j = np.arange(S, dtype=np.int32)[None, :]
    for r0 in range(0, rows.size, 1024):
        i = rows[r0:r0 + 1024, None].astype(np.int32)
        out[r0:r0 + 1024] = (np.abs(i - j) <= band) | (j < n_global) | (i < n_global)
    return out


def scattered_mask(S, window, n_global, density, seed):
    """bool [S, S] element mask, Bigbird-like: keys within `window` of the
    query row, `n_global` global tokens (first keys and first rows), and
    random keys drawn independently with probability `density`."""
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    m = (np.abs(i - j) <= window) | (j < n_global) | (i < n_global)
    return m | (np.random.default_rng(seed).random((S, S)) < density)


def random_tile_mask(nqt, nkt, density, seed, nheads=None):
    """bool [nqt, nkt] (or [nheads, nqt, nkt]) with each tile present w.p. density."""
    rng = np.random.default_rng(seed)
    shape = (nqt, nkt) if nheads is None else (nheads, nqt, nkt)
    return rng.random(shape) < density


def workload_inputs(name):
    """(q, k, v, scale, extras) for a named workload, drawn on the CPU."""
    w = WORKLOADS[name]
    q, k, v = make_qkv(w["B"], w["H"], w["Hkv"], w["Sq"], w["Sk"], w["d"], w["seed"],
                       w["dtype"], w["amp"])
    extras = {}
    if name == "block_sparse":
        nqt = n_tiles(w["Sq"], w["tile"])
        extras["tile_mask"] = window_random_tile_mask(nqt, w["window"], w["frac"], w["seed"])
    if name == "two_level":
        extras["elem_mask"] = band_global_mask(w["Sq"], w["band"], w["n_global"])
    if name == "scattered_short":
        extras["elem_mask"] = scattered_mask(w["Sq"], w["window"], w["n_global"], w["density"],
                                             w["seed"])
    return q, k, v, default_scale(w["d"]), extras
