"""Float64 CPU oracle for the fused online-softmax attention path.

TEST INFRASTRUCTURE ONLY. Nothing in the product package
``online_softmax_attention_rf_gb300`` imports this package, and the product
never falls back to it. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import it.

The oracle shares no code with the CUDA path: no kernels, headers, constant
tables, tiling or pre-/post-processing. It computes the plain definition of
each operation with NumPy in float64, three unfused passes per row, written
so that it can be checked against the pages by eye.

Modules
-------
``three_pass``   three-pass safe-softmax attention, row softmax, split-K
                 partials and their log-sum-exp merge, the set of tiles that
                 hold at least one visible (query, key) pair, the
                 block-sparse row lists of a tile mask, and the two-level
                 (outer lists + inner 8x8 bitmaps) encoding of an element
                 mask.
``incremental``  an independent float64 run of the incremental (online) form,
                 used only to check that the derivation the GPU follows
                 reaches the three-pass result; the same for the pairwise
                 merge of (count, mean, M2) moment states.
``cascades``     other cascaded reductions the pages name: top-k softmax
                 routing of Mixture-of-Experts tokens, per-row mean and
                 variance (normalisation statistics), the moment of
                 inertia of point sets about their centre of mass, and
                 per-row FP8 (E4M3) absmax quantisation with the GEMM over
                 the quantised values.

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` against brute force, closed forms, invariants
and library routines; none is "parity unpinned".
"""

from .three_pass import (  # noqa: F401
    NEG_INF,
    attention,
    bsr_from_tile_mask,
    decode_partials,
    merge_partials,
    softmax_rows,
    split_bounds,
    two_level_decode,
    two_level_encode,
    visible_mask,
    visited_tiles,
)
from .incremental import (  # noqa: F401
    incremental_attention,
    moments_merge,
    moments_state,
    weighted_merge,
    weighted_state,
)
from .cascades import (  # noqa: F401
    E4M3_MAX,
    e4m3_code,
    e4m3_round,
    fp8_gemm,
    moe_route,
    moment_of_inertia,
    row_moments,
    rowquant_e4m3,
)
