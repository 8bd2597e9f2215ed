"""Write oracle_small_cases.json: small inputs and the oracle's outputs.

The pages print no worked example, so no stored value here comes from them.
These fixtures are regression values: the inputs are drawn by NumPy with
fixed seeds and stored alongside the outputs, and the outputs are computed by
``oracle.attention`` alone. A change to the oracle's arithmetic that moves
any of them must name, in its commit message, the passage of the pages that
justifies it.

Run from the repository root:  python tests/golden/make_golden.py
"""

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402

CASES = [
    # name, B, H, Hkv, Sq, Sk, d, causal, tile, tile-mask density, scale
    ("dense", 1, 2, 2, 5, 6, 4, False, 2, None, 0.5),
    ("causal_gqa", 1, 4, 2, 6, 6, 3, True, 2, None, 0.6),
    ("causal_rect", 1, 1, 1, 7, 4, 2, True, 2, None, 1.0),
    ("tile_mask", 2, 1, 1, 6, 8, 3, False, 2, 0.5, 0.4),
]


def main():
    out = []
    for n, (name, B, H, Hkv, Sq, Sk, d, causal, tile, dens, scale) in enumerate(CASES):
        rng = np.random.default_rng(1000 + n)
        q = np.round(rng.standard_normal((B, H, Sq, d)), 6)
        k = np.round(rng.standard_normal((B, Hkv, Sk, d)), 6)
        v = np.round(rng.standard_normal((B, Hkv, Sk, d)), 6)
        tm = None
        if dens is not None:
            tm = rng.random((B * H, -(-Sq // tile), -(-Sk // tile))) < dens
        o, lse = oracle.attention(q, k, v, scale, causal, tm, tile)
        out.append(dict(
            name=name, scale=scale, causal=causal, tile=tile,
            q=q.tolist(), k=k.tolist(), v=v.tolist(),
            tile_mask=None if tm is None else tm.tolist(),
            o=o.tolist(), lse=[[[float(t) for t in r] for r in h] for h in lse]))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small_cases.json")
    with open(path, "w") as f:
        json.dump({"source": "oracle.attention (float64); inputs drawn by numpy, seeds 1000+i",
                   "cases": out}, f, indent=None)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
