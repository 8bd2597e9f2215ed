"""A CPU model of the barrier protocol of the tensor-core attention kernel.

attn_tc_kernel (csrc/attn_tc.cu) runs three kinds of roles per CTA: a TMA
producer that fills a ring of NS K/V tile slots in the order of the union of
two query tiles' key-tile lists, and for each query tile a softmax group plus
an MMA issuer. They synchronise only through mbarriers (kv_full / kv_empty per
slot, q_full / q_empty, s_full, o_done) and one issue lock. Every device wait
is bounded, so a protocol deadlock would show up as a timeout status; this
model finds such deadlocks on the CPU instead, before any GPU run.

Each role is a generator that yields the condition it waits on; a scheduler
runs any role whose condition holds (in a seeded random order, with MMA
commits delivered late or at once). If no role can move and not all are done,
the protocol deadlocks for those tile lists. The model follows the kernel's
order of operations per step:

  issuer:  wait V(u) landed; if the next union entry is this tile's, wait for
           its K and consume it  --  P ready  --  lock; P.V(u) [+ Q.K(next)];
           unlock; commit release of V(u) [, K(next), Q (last QK), S]; else
           on the last entry commit "O done", release the rest of the item's
           entries and start the next item; else wait for the next entry's K
           (releasing entries only the other tile needs) and issue its Q.K.
  producer: per union entry, wait for the slot to be released by both tiles,
           load K then V; after an item's first entry, load its Q tiles.

A planted mistake -- waiting for the next K tile before the P.V whose release
that load needs, the order an earlier kernel version had -- must deadlock.
"""

import random

import numpy as np
import pytest

from online_softmax_attention_rf_gb300 import inputs


class _Bar:
    """mbarrier with an arrival count and a phase counter."""

    def __init__(self, count):
        self.count, self.arrived, self.phase = count, 0, 0

    def arrive(self):
        self.arrived += 1
        if self.arrived == self.count:
            self.arrived, self.phase = 0, self.phase + 1

    def done(self, parity):
        return (self.phase & 1) != parity


def _tile_list(mask, bh, qt, nqt):
    if qt >= nqt:
        return []
    m = mask[bh if mask.shape[0] > 1 else 0, qt]
    return [int(c) for c in np.nonzero(m)[0]]


def _union(l0, l1):
    return [(u, u in l0, u in l1) for u in sorted(set(l0) | set(l1))]


def _cta_items(pairs, x):
    half = (pairs + 1) // 2
    j, bh = x % half, x // half
    items = [(bh, 2 * (pairs - 1 - j))]
    if j != pairs - 1 - j:
        items.append((bh, 2 * j))
    return items


def _run_cta(mask, nqt, items, NS, late_commits, rng, planted=False):
    """True if every role of one CTA finishes; False on deadlock."""
    kv_full = [_Bar(1) for _ in range(NS)]
    kv_empty = [_Bar(2) for _ in range(NS)]
    q_full, q_empty = [_Bar(1), _Bar(1)], [_Bar(1), _Bar(1)]
    s_full, o_done = [_Bar(1), _Bar(1)], [_Bar(1), _Bar(1)]
    met = {"sm": [0, 0], "is": [0, 0]}   # arrivals at each tile's group barrier
    lock = [0]
    pending = []
    split_ready, split_read = _Bar(1), _Bar(1)

    def commit(b):
        if late_commits:
            pending.append(b)
        else:
            b.arrive()

    def lists(k):
        if len(items[k]) == 3:                   # explicit lists (l0, l1, split)
            return items[k][0], items[k][1]
        bh, qt0 = items[k]
        return _tile_list(mask, bh, qt0, nqt), _tile_list(mask, bh, qt0 + 1, nqt)

    def is_split(k):
        return len(items[k]) == 3 and items[k][2]

    def producer():
        seq, q_loads = 0, [0, 0]
        for k in range(len(items)):
            l0, l1 = lists(k)
            first = True
            for _ in _union(l0, l1):
                for _kv in range(2):
                    slot, par = seq % NS, ((seq // NS) & 1) ^ 1
                    yield lambda slot=slot, par=par: kv_empty[slot].done(par)
                    kv_full[slot].arrive()
                    seq += 1
                if first:
                    first = False
                    for t, lt in enumerate((l0, l1)):
                        if not lt:
                            continue
                        if q_loads[t] > 0:
                            par = (q_loads[t] - 1) & 1
                            yield lambda t=t, par=par: q_empty[t].done(par)
                        q_full[t].arrive()
                        q_loads[t] += 1

    def group_barrier(t, side):
        """Rendezvous of a tile's softmax warps and its issuer."""
        other = "is" if side == "sm" else "sm"
        met[side][t] += 1
        mine = met[side][t]
        yield lambda: met[other][t] >= mine

    def softmax(t):
        j, o_items, n_split = 0, 0, 0
        for k in range(len(items)):
            n = len(lists(k)[t])
            for _ in range(n):
                par = j & 1
                yield lambda par=par: s_full[t].done(par)
                j += 1
                yield from group_barrier(t, "sm")     # P is in tensor memory
            yield from group_barrier(t, "sm")         # after the item's steps
            if n:                                     # epilogue
                par = o_items & 1
                yield lambda par=par: o_done[t].done(par)
                o_items += 1
            if is_split(k):                           # group 1 hands over to group 0
                par = n_split & 1
                n_split += 1
                if t == 1:
                    split_ready.arrive()
                    yield lambda par=par: split_read.done(par)
                else:
                    yield lambda par=par: split_ready.done(par)
                    split_read.arrive()
            yield from group_barrier(t, "sm")         # after the epilogue

    def issuer(t):
        st = dict(seq=0, vseq=0, nq=0, n_iss=0, started=-1, it=[])

        def wait_full(s_):
            return lambda: kv_full[s_ % NS].done((s_ // NS) & 1)

        def advance():
            while st["it"]:
                u, n0, n1 = st["it"].pop(0)
                ks = st["seq"]
                st["seq"] += 2
                if (n0, n1)[t]:
                    return ks
                for e in range(2):       # an entry only the other tile needs
                    yield wait_full(ks + e)
                    kv_empty[(ks + e) % NS].arrive()
            return None

        def next_k():
            ks = yield from advance()
            if ks is not None:
                yield wait_full(ks)
            return ks

        def take_lock():
            yield lambda: lock[0] == 0
            lock[0] = 1

        def qk_commits(ks, n):
            commit(s_full[t])
            commit(kv_empty[ks % NS])
            st["n_iss"] += 1
            if st["n_iss"] == n:
                commit(q_empty[t])
            st["vseq"] = ks + 1

        def start_item(k):
            st["started"] = k
            if k >= len(items):
                return
            l0, l1 = lists(k)
            st["it"], st["n_iss"] = _union(l0, l1), 0
            n = len((l0, l1)[t])
            if n == 0:
                yield from advance()
                return
            par = st["nq"] & 1
            yield lambda: q_full[t].done(par)
            st["nq"] += 1
            ks = yield from next_k()
            yield from take_lock()
            lock[0] = 0
            qk_commits(ks, n)

        for k in range(len(items)):
            n = len(lists(k)[t])
            if st["started"] < k:
                yield from start_item(k)
            for jj in range(n):
                last = jj + 1 == n
                vs = st["vseq"]
                yield wait_full(vs)
                fast = None
                it = st["it"]
                if not last and it and (it[0][1 + t] or planted):
                    # the kernel waits here only when the next union entry is
                    # this tile's; the planted mistake also skips others' entries
                    fast = yield from next_k()
                yield from group_barrier(t, "is")     # P is in tensor memory
                yield from take_lock()
                lock[0] = 0
                commit(kv_empty[vs % NS])
                if fast is not None:
                    qk_commits(fast, n)
                elif not last:
                    ks = yield from next_k()
                    yield from take_lock()
                    lock[0] = 0
                    qk_commits(ks, n)
                else:
                    commit(o_done[t])
            yield from group_barrier(t, "is")         # after the item's steps
            if n:
                yield from advance()                  # entries after this tile's last
                yield from start_item(k + 1)
            yield from group_barrier(t, "is")         # after the epilogue

    roles = {"producer": producer(), "sm0": softmax(0), "sm1": softmax(1),
             "is0": issuer(0), "is1": issuer(1)}
    waiting = {name: None for name in roles}
    done = set()
    while len(done) < len(roles):
        runnable = [n for n in roles if n not in done
                    and (waiting[n] is None or waiting[n]())]
        if pending and (not runnable or rng.random() < 0.5):
            pending.pop(0).arrive()      # an MMA batch completes
            continue
        if not runnable:
            return False
        name = rng.choice(runnable)
        try:
            waiting[name] = next(roles[name])
        except StopIteration:
            done.add(name)
    return True


def _run(mask, nqt, NS, late, seed, planted=False):
    pairs = (nqt + 1) // 2
    rng = random.Random(seed)
    for x in range(((pairs + 1) // 2) * mask.shape[0]):
        if not _run_cta(mask, nqt, _cta_items(pairs, x), NS, late, rng, planted):
            return False
    return True


def test_protocol_completes_on_the_block_sparse_test_masks():
    nqt, nkt = inputs.n_tiles(640), inputs.n_tiles(900)
    tm = np.asarray(inputs.random_tile_mask(nqt, nkt, 0.4, 7, nheads=4))
    tm[0, 2, :] = False          # a query tile with no key tile
    for late in (False, True):
        assert _run(tm, nqt, 5, late, 1)


@pytest.mark.parametrize("seed", range(6))
def test_protocol_completes_on_random_lists(seed):
    rng = np.random.default_rng(seed)
    for _ in range(60):
        nq, nk, nh = int(rng.integers(1, 9)), int(rng.integers(1, 12)), int(rng.integers(1, 3))
        mask = rng.random((nh, nq, nk)) < rng.random()
        assert _run(mask, nq, int(rng.choice([5, 8])), bool(rng.integers(0, 2)),
                    int(rng.integers(1 << 30))), (nq, nk, nh)


def test_protocol_completes_on_causal_lists():
    rng = np.random.default_rng(11)
    for nq in range(1, 12):
        for off in (-3, 0, 2):
            nk = max(1, nq + off)
            mask = np.array([[[c <= q + off for c in range(nk)] for q in range(nq)]])
            for NS in (5, 8):
                assert _run(mask, nq, NS, bool(rng.integers(0, 2)), int(rng.integers(1 << 30)))


def test_planted_order_deadlocks():
    """Waiting for the next K tile before issuing the P.V that releases its
    slot, whatever entries lie between, deadlocks on some lists; the model
    must see it (otherwise the tests above would prove nothing)."""
    rng = np.random.default_rng(3)
    found = False
    for _ in range(200):
        nq, nk = int(rng.integers(2, 9)), int(rng.integers(2, 12))
        mask = rng.random((1, nq, nk)) < 0.5
        if not _run(mask, nq, 5, False, 7, planted=True):
            found = True
            break
    assert found


def test_protocol_completes_with_many_items_per_cta():
    """The roles' loops take any number of items per CTA; chaining several
    heads' double items in one CTA (CTA c taking double items c, c + grid,
    ...) must complete too."""
    rng = np.random.default_rng(5)
    for _ in range(80):
        nq, nk, nh = int(rng.integers(1, 9)), int(rng.integers(1, 12)), int(rng.integers(1, 4))
        mask = rng.random((nh, nq, nk)) < rng.random()
        pairs = (nq + 1) // 2
        nx = ((pairs + 1) // 2) * nh
        for grid in (1, 2, 3):
            for c in range(min(grid, nx)):
                items = [it for x in range(c, nx, grid) for it in _cta_items(pairs, x)]
                assert _run_cta(mask, nq, items, int(rng.choice([5, 8])), bool(rng.integers(0, 2)),
                                random.Random(int(rng.integers(1 << 30)))), (nq, nk, nh, grid)


def _cta_items_split(mask, nqt, pairs, x):
    """The kernel's items for a launch with a two-level mask: a pair whose
    one tile lists more than 3 times its partner's entries plus 8 becomes a
    split item (both groups on the long tile, alternate entries) and then the
    other tile alone."""
    out = []
    for bh, a in _cta_items(pairs, x):
        la, lb = _tile_list(mask, bh, a, nqt), _tile_list(mask, bh, a + 1, nqt)
        if len(la) > 3 * len(lb) + 8 or len(lb) > 3 * len(la) + 8:
            lng, shrt = (la, lb) if len(la) > len(lb) else (lb, la)
            short_tile = a + 1 if lng is la else a
            out.append((lng[0::2], lng[1::2], True))
            if short_tile < nqt:
                out.append((shrt, [], False))
        else:
            out.append((la, lb, False))
    return out


@pytest.mark.parametrize("seed", range(4))
def test_protocol_completes_with_split_items(seed):
    """Masks with long query tiles (global rows) next to short ones: the
    split items' alternating lists, the lone short tiles and the hand-over
    between the two groups must complete in any timing."""
    rng = np.random.default_rng(100 + seed)
    n_split = 0
    for _ in range(40):
        nq, nk, nh = int(rng.integers(1, 9)), int(rng.integers(10, 40)), int(rng.integers(1, 3))
        mask = rng.random((nh, nq, nk)) < 0.08
        for h in range(nh):
            mask[h, int(rng.integers(0, nq))] = True     # a global query tile
        pairs = (nq + 1) // 2
        nx = ((pairs + 1) // 2) * nh
        for x in range(nx):
            items = _cta_items_split(mask, nq, pairs, x)
            n_split += sum(1 for it in items if it[2])
            assert _run_cta(mask, nq, items, int(rng.choice([5, 8])), bool(rng.integers(0, 2)),
                            random.Random(int(rng.integers(1 << 30)))), (nq, nk, nh, x)
    assert n_split > 0
