"""Plain float64 definitions of the attention path (three unfused passes).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference leg of ``bench.py``; never by the product.

Sources (page title, section):

* RedFuser: An Automatic Operator Fusion Framework for Cascaded Reductions on
  AI Accelerators -- technical summary, section 1 "Problématique": attention
  is a cascaded reduction, a safe softmax followed by a GEMM, where each
  reduction (maximum, then sum) waits for the root of the one before.
* same page, section 2 "Méthodologie", formal definition: a cascaded
  reduction is d_i = (+)_l F_i(X[l], D_i), D_i being the earlier results.
  For one query row the chain is d1 = max_j s_j, d2 = sum_j exp(s_j - d1),
  d3 = sum_j exp(s_j - d1) / d2 * v_j.
* same page, section 3 "Contributions", multi-segment strategy: the input is
  partitioned and the partial results are merged (split-K partials and their
  log-sum-exp merge below).
* Accelerating Sparse Transformer Inference on GPU (STOF) -- technical
  summary, "Méthodologie", unified MHA module: block-sparse outer tiles kept
  as row-compressed (BSR) lists; masked tiles are skipped entirely
  ("Énoncé du problème"). Same section, two-level storage format: outer
  tiles are "full" (every element valid) or "partial"; the valid elements of
  a partial tile are kept as one 64-bit bitmap per 8x8 inner block.

The oracle deliberately does NOT use the incremental (online) form the GPU
uses; it runs the definition: pass 1 row maximum, pass 2 sum of shifted
exponentials, pass 3 normalised P.V.

Readings where the pages are silent (none of these pages prints a formula,
a bit order or a layout; each reading below is the plainest one that the
rest of the pages' text supports):

* LSE is the natural log: LSE_i = m_i + ln l_i.
* Causal masking is bottom-right aligned: query row i sees key j iff
  j <= i + (Sk - Sq).
* A tile mask is a bool array over (query tile, key tile) of side ``tile``;
  a key is visible only if its tile is present (and, with causal, also
  causally visible).
* GQA: query head h reads key/value head h // (H // Hkv).
* A row with no visible key gives O = 0 and LSE = -inf.
* A row-softmax row whose entries are all -inf gives y = 0.
* An element mask is a bool array over (query row, key); a key is visible
  only if the element mask allows it as well as the tile mask and causality.
* Two-level format (the pages give no bit order): an outer tile is listed if
  it holds a valid element; it is full if every element of it that lies
  inside the Sq x Sk matrix is valid, else partial. The 16 x 16 inner blocks
  of a partial tile are stored row-major, 256 words per tile; bit 8 r + c of
  a word is element (r, c) of its 8 x 8 block (row-major bits). Elements
  outside the matrix have bit 0.
* Split-K: contiguous splits of Sk // nsplit keys, the last split taking the
  remainder.
"""

import numpy as np

NEG_INF = -np.inf

#: query rows processed together; bounds the float64 score block in memory
ROW_BLOCK = 256


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def visible_mask(Sq, Sk, causal, tile_mask=None, tile=128, rows=None, elem_mask=None):
    """bool [R, Sk]: True where query row i may attend key j.

    ``rows`` selects query rows (default: all Sq rows). ``tile_mask`` is a
    2-D bool array [ceil(Sq/tile), ceil(Sk/tile)] for one head;
    ``elem_mask`` a 2-D bool array [Sq, Sk] for one head.
    """
    rows = np.arange(Sq, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    i = rows[:, None]
    j = np.arange(Sk, dtype=np.int64)[None, :]
    vis = np.ones((rows.size, Sk), dtype=bool)
    if causal:
        vis &= j <= i + (Sk - Sq)
    if tile_mask is not None:
        tm = np.asarray(tile_mask, dtype=bool)
        vis &= tm[i // tile, j // tile]
    if elem_mask is not None:
        vis &= np.asarray(elem_mask, dtype=bool)[rows]
    return vis


def _head_tile_mask(tile_mask, b, h, H):
    """The mask of head (b, h): a 2-D mask is shared, a 3-D one is per head."""
    if tile_mask is None:
        return None
    tm = np.asarray(tile_mask, dtype=bool)
    return tm if tm.ndim == 2 else tm[b * H + h]


def _three_pass(q, k, v, scale, vis):
    """One head, a block of query rows: the definition in three passes.

    q [R, d], k [Sk, d], v [Sk, dv], vis [R, Sk] -> (o [R, dv], lse [R]).
    """
    # scores s_ij = scale * <q_i, k_j>; a library matmul forms the dot products
    s = scale * (q @ k.T)
    s = np.where(vis, s, NEG_INF)
    seen = vis.any(axis=1)
    # pass 1: row maximum (d1)
    m = np.full(q.shape[0], NEG_INF)
    if s.shape[1]:
        m = s.max(axis=1)
    # pass 2: sum of exponentials shifted by the maximum (d2)
    shift = np.where(seen, m, 0.0)
    e = np.exp(s - shift[:, None])  # masked entries: exp(-inf) = 0
    l = e.sum(axis=1)
    # pass 3: normalised probabilities times V (d3)
    p = e / np.where(seen, l, 1.0)[:, None]
    o = p @ v
    o[~seen] = 0.0
    lse = np.full(q.shape[0], NEG_INF)
    lse[seen] = m[seen] + np.log(l[seen])
    return o, lse


def attention(q, k, v, scale, causal=False, tile_mask=None, tile=128, rows=None, heads=None,
              elem_mask=None):
    """Safe-softmax attention, float64, plain definition.

    q [B, H, Sq, d]; k, v [B, Hkv, Sk, d(v)]; any float dtype (cast exactly
    to float64). ``tile_mask``: None, bool [nqt, nkt] shared by all heads, or
    bool [B*H, nqt, nkt] per head. ``elem_mask``: None, bool [Sq, Sk] shared
    or [B*H, Sq, Sk] per head. ``rows``: query-row indices to compute
    (default all). ``heads``: list of (b, h) to compute (default all).

    Returns (o, lse): with ``heads`` None, o [B, H, R, dv] and lse [B, H, R];
    otherwise o [n, R, dv] and lse [n, R] in the order of ``heads``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Sq, d = q.shape
    Bk, Hkv, Sk, dk = k.shape
    if Bk != B or dk != d or v.shape[:3] != k.shape[:3] or H % Hkv:
        raise ValueError("shape mismatch")
    G = H // Hkv
    rows = np.arange(Sq, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    all_heads = heads is None
    hl = [(b, h) for b in range(B) for h in range(H)] if all_heads else list(heads)
    dv = v.shape[-1]
    o = np.zeros((len(hl), rows.size, dv))
    lse = np.full((len(hl), rows.size), NEG_INF)
    for n, (b, h) in enumerate(hl):
        tm = _head_tile_mask(tile_mask, b, h, H)
        em = _head_tile_mask(elem_mask, b, h, H)
        kv = h // G
        for r0 in range(0, rows.size, ROW_BLOCK):
            rr = rows[r0:r0 + ROW_BLOCK]
            vis = visible_mask(Sq, Sk, causal, tm, tile, rr, em)
            o[n, r0:r0 + rr.size], lse[n, r0:r0 + rr.size] = _three_pass(
                q[b, h, rr], k[b, kv], v[b, kv], scale, vis)
    if all_heads:
        o = o.reshape(B, H, rows.size, dv)
        lse = lse.reshape(B, H, rows.size)
    return o, lse


def softmax_rows(x):
    """Row softmax y_j = exp(x_j - max x) / sum exp(x - max x), float64.

    The pure two-reduction cascade (max, then sum of exponentials) of the
    RedFuser page's problem statement; pass 1 maximum, pass 2 sum, then the
    normalisation. A row of all -inf gives y = 0.
    """
    x = _f64(x)
    y = np.zeros_like(x)
    for r0 in range(0, x.shape[0], 4096):
        xb = x[r0:r0 + 4096]
        m = xb.max(axis=1)                       # pass 1
        seen = m > NEG_INF
        shift = np.where(seen, m, 0.0)
        e = np.exp(xb - shift[:, None])
        l = e.sum(axis=1)                        # pass 2
        y[r0:r0 + 4096] = np.where(seen[:, None], e / np.where(seen, l, 1.0)[:, None], 0.0)
    return y


def split_bounds(Sk, nsplit):
    """[(start, end)] of the nsplit contiguous key splits.

    Each split holds Sk // nsplit keys; the last one also takes the
    remainder.
    """
    if nsplit < 1 or nsplit > Sk:
        raise ValueError("need 1 <= nsplit <= Sk")
    n = Sk // nsplit
    return [(s * n, (s + 1) * n if s < nsplit - 1 else Sk) for s in range(nsplit)]


def decode_partials(q, k, v, scale, nsplit):
    """Per-split attention results of one decode query row per head.

    q [B, H, 1, d]; k, v [B, Hkv, Sk, d]. Split s covers keys
    split_bounds(Sk, nsplit)[s]; its partial is the plain attention over
    those keys alone: O_s (normalised within the split) and lse_s.
    Returns o_part [B, H, nsplit, dv], lse_part [B, H, nsplit].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Sq, _ = q.shape
    if Sq != 1:
        raise ValueError("decode has one query row")
    dv = v.shape[-1]
    o_part = np.zeros((B, H, nsplit, dv))
    lse_part = np.zeros((B, H, nsplit))
    for s, (a, e) in enumerate(split_bounds(k.shape[2], nsplit)):
        o, lse = attention(q, k[:, :, a:e], v[:, :, a:e], scale)
        o_part[:, :, s] = o[:, :, 0]
        lse_part[:, :, s] = lse[:, :, 0]
    return o_part, lse_part


def merge_partials(o_part, lse_part):
    """Log-sum-exp merge of split results (multi-segment strategy).

    o_part [..., S, dv], lse_part [..., S] -> (o [..., dv], lse [...]):
    LSE = log sum_s exp(lse_s) and O = sum_s exp(lse_s - LSE) O_s. The sum
    is taken relative to max_s lse_s, which is the same number in exact
    arithmetic and cannot overflow. All lse_s = -inf gives O = 0, LSE = -inf.
    """
    o_part, lse_part = _f64(o_part), _f64(lse_part)
    mx = lse_part.max(axis=-1)
    seen = mx > NEG_INF
    shift = np.where(seen, mx, 0.0)
    tot = np.exp(lse_part - shift[..., None]).sum(axis=-1)
    lse = np.where(seen, shift + np.log(np.where(seen, tot, 1.0)), NEG_INF)
    w = np.exp(lse_part - np.where(seen, lse, 0.0)[..., None])
    w = np.where(seen[..., None], w, 0.0)
    o = (w[..., None] * o_part).sum(axis=-2)
    return o, lse


def visited_tiles(Sq, Sk, causal, tile_mask=None, tile=128, elem_mask=None):
    """bool [nqt, nkt]: tiles holding at least one visible (query, key) pair.

    This is the set of tiles a kernel that skips masked tiles must process
    (and the only ones it may process). ``tile_mask`` and ``elem_mask`` are
    2-D (one head).
    """
    nqt, nkt = -(-Sq // tile), -(-Sk // tile)
    out = np.zeros((nqt, nkt), dtype=bool)
    for qt in range(nqt):
        rows = np.arange(qt * tile, min(Sq, (qt + 1) * tile))
        vis = visible_mask(Sq, Sk, causal, tile_mask, tile, rows, elem_mask)
        colany = vis.any(axis=0)
        for kt in range(nkt):
            out[qt, kt] = colany[kt * tile:(kt + 1) * tile].any()
    return out


def bsr_from_tile_mask(tile_mask):
    """Row-compressed lists of a tile mask (STOF's outer-tile BSR index).

    tile_mask: bool [nqt, nkt] or [nheads, nqt, nkt]; the rows of all heads
    are listed one after another. Returns (row_ptr int32 [nrows + 1],
    col_idx int32 [nnz]) with the columns of each row in ascending order.
    """
    tm = np.asarray(tile_mask, dtype=bool)
    flat = tm.reshape(-1, tm.shape[-1])
    counts = [int(r.sum()) for r in flat]
    row_ptr = np.zeros(len(counts) + 1, dtype=np.int32)
    row_ptr[1:] = np.cumsum(counts)
    cols = [np.nonzero(r)[0] for r in flat]
    col_idx = np.concatenate(cols).astype(np.int32) if cols else np.zeros(0, np.int32)
    return row_ptr, col_idx


def two_level_encode(elem_mask, tile=128, inner=8):
    """STOF's two-level storage of an element mask (outer BSR + inner bitmaps).

    elem_mask: bool [nheads, Sq, Sk] or [Sq, Sk]. For each head and each row
    of outer tiles, the tiles that hold a valid element are listed in
    ascending column order (row_ptr, col_idx, as ``bsr_from_tile_mask``);
    tile_bits[n] is -1 for a full tile, else the index of its bitmap block
    in ``bits``, which holds (tile // inner)**2 words per partial tile:
    inner blocks row-major, bit inner*r + c of a word = element (r, c) of
    its block.
    Returns (row_ptr int32, col_idx int32, tile_bits int32, bits uint64 [P, nb*nb]).
    """
    em = np.asarray(elem_mask, dtype=bool)
    if em.ndim == 2:
        em = em[None]
    nh, Sq, Sk = em.shape
    nqt, nkt, nb = -(-Sq // tile), -(-Sk // tile), tile // inner
    weights = np.left_shift(np.uint64(1), np.arange(inner * inner, dtype=np.uint64))
    row_ptr, col_idx, tile_bits, bits = [0], [], [], []
    for h in range(nh):
        for qt in range(nqt):
            for kt in range(nkt):
                blk = em[h, qt * tile:(qt + 1) * tile, kt * tile:(kt + 1) * tile]
                if not blk.any():
                    continue
                col_idx.append(kt)
                if blk.all():
                    tile_bits.append(-1)
                    continue
                full = np.zeros((tile, tile), dtype=bool)   # outside the matrix: 0
                full[:blk.shape[0], :blk.shape[1]] = blk
                # [br, r, bc, c] -> [br, bc, r * inner + c]
                cells = full.reshape(nb, inner, nb, inner).transpose(0, 2, 1, 3)
                cells = cells.reshape(nb * nb, inner * inner)
                words = (cells.astype(np.uint64) * weights).sum(axis=1, dtype=np.uint64)
                tile_bits.append(len(bits))
                bits.append(words)
            row_ptr.append(len(col_idx))
    bits = np.stack(bits) if bits else np.zeros((0, nb * nb), np.uint64)
    return (np.asarray(row_ptr, np.int32), np.asarray(col_idx, np.int32),
            np.asarray(tile_bits, np.int32), bits.astype(np.uint64))


def two_level_decode(row_ptr, col_idx, tile_bits, bits, nheads, Sq, Sk, tile=128, inner=8):
    """The element mask [nheads, Sq, Sk] that a two-level encoding describes."""
    nqt, nkt, nb = -(-Sq // tile), -(-Sk // tile), tile // inner
    out = np.zeros((nheads, nqt * tile, nkt * tile), dtype=bool)
    for h in range(nheads):
        for qt in range(nqt):
            r = h * nqt + qt
            for n in range(row_ptr[r], row_ptr[r + 1]):
                kt = col_idx[n]
                dst = out[h, qt * tile:(qt + 1) * tile, kt * tile:(kt + 1) * tile]
                if tile_bits[n] < 0:
                    dst[:] = True
                    continue
                for blk in range(nb * nb):
                    br, bc = divmod(blk, nb)
                    w = int(bits[tile_bits[n], blk])
                    for e in range(inner * inner):
                        if (w >> e) & 1:
                            rr, cc = divmod(e, inner)
                            dst[br * inner + rr, bc * inner + cc] = True
    return out[:, :Sq, :Sk]
