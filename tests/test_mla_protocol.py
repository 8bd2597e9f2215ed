"""A CPU model of the persistent MLA decode kernel's barrier protocol.

mla_decode_kernel (csrc/mla_decode.cu) runs three roles per CTA: a TMA
producer, one MMA-issuing thread and four softmax warps (one role here). A
CTA walks a run of key segments; the segments of one batch element form one
folded segment with its own q, online-softmax state and partial. The roles
synchronise only through mbarriers whose waits test a phase PARITY, so a
waiter must never fall two phases behind (it would then block, or pass on
the wrong phase). Every device wait is bounded, so a protocol fault would
show as a timeout status or, worse, as a silent data race; this model finds
both on the CPU.

Each role is a generator that yields the barrier phase it waits for; TMA
copies land in any order at random times, and the tensor pipe executes the
issuer's MMAs and commits in order at random times. At every wait the model
checks that the barrier is at the awaited phase or one past it, and every
access checks what the buffer holds: the kv slot's X and H parts (a kv tile,
q's staged chunks or the staged O rows), q in shared and in tensor memory, the
S / P tile and the O accumulator. Planted mistakes -- the producer taking the
slot for the next batch element before the previous O has left it, loading
the next q before the previous scores are done, or loading a tile's H part
over q's staged chunks before the softmax warps have copied them -- must be
caught.

RedFuser page, section 3 (multi-segment strategy: each segment's partial
state, merged by log-sum-exp) and section 4 (the MLA workload).
"""

import random

import pytest


class _Bar:
    def __init__(self, count):
        self.count, self.arrived, self.phase = count, 0, 0

    def arrive(self, n=1):
        for _ in range(n):
            self.arrived += 1
            if self.arrived == self.count:
                self.arrived, self.phase = 0, self.phase + 1


class _Fault(Exception):
    pass


def _check(cond, what):
    if not cond:
        raise _Fault(what)


def segments(B, Sk, nsplit, runs, run):
    """The folded segments of one run: (b, s0, s1, key0, key1, ntiles), the
    same arithmetic as the kernel's run bounds and mla_segment()."""
    units = B * nsplit
    u0, u1 = run * units // runs, (run + 1) * units // runs
    per = Sk // nsplit
    out, u = [], u0
    while u < u1:
        b = u // nsplit
        end = min(u1, (b + 1) * nsplit)
        s0, s1 = u - b * nsplit, end - 1 - b * nsplit
        key0 = s0 * per
        key1 = Sk if s1 == nsplit - 1 else (s1 + 1) * per
        out.append((b, s0, s1, key0, key1, (key1 - key0 + 63) // 64))
        u = end
    return out


def _run_cta(segs, rng, planted=None, p_resc=0.5):
    """True when every role of one CTA finishes; raises _Fault on a hazard or
    a phase that moved two past its waiter; False on deadlock."""
    B = {n: _Bar(c) for n, c in [("q_full", 1), ("q_stage", 1), ("q_tmem", 4), ("pv_done", 1),
                                 ("o_done", 1), ("epi_done", 4), ("mma_idle", 1),
                                 ("x_full", 1), ("x_empty", 1), ("h_full", 1), ("h_empty", 1),
                                 ("s_full", 1), ("p_full", 4)]}
    # X / H: what the slot's parts hold; S: the score tile ("S", seg, tile,
    # parts done), then P over it ("P", ...), then "used" once P.V has run
    st = {"X": None, "H": None, "qs": None, "qt": None, "S": None, "O": None,
          "o_read": set(), "q_copied": set(), "O_busy": False}
    tma, pipe = [], []          # copies in flight; the tensor pipe's queue

    def pending_reads(res):
        return any(op[0] == "mma" and res in op[1] for op in pipe)

    def wait(name, idx):
        return ("wait", name, idx)

    def tma_issue(target, tag, bar):
        _check(not pending_reads(target), "copy into %s while an MMA still reads it" % (target,))
        if target in ("X", "H"):
            _check(not st["O_busy"], "copy into the slot while O rows are stored from it")
        tma.append((target, tag, bar))

    def producer():
        n = 0
        for k, (b, s0, s1, k0, k1, nt) in enumerate(segs):
            if k > 0 and planted != "q_early":
                yield wait("o_done", k - 1)
            tma_issue("qs", k, "q_full")
            if k > 0 and planted != "no_epi_wait":
                yield wait("epi_done", k - 1)
            tma_issue("H", ("q", k), "q_stage")
            for j in range(nt):
                if n >= 1:
                    yield wait("x_empty", n - 1)
                tma_issue("X", (k, j), "x_full")
                if n >= 1:
                    yield wait("h_empty", n - 1)
                if j == 0 and planted != "h_over_q":
                    yield wait("q_tmem", k)
                _check(st["H"] != ("q", k) or k in st["q_copied"],
                       "tile copied over q's staged chunks before the softmax read them")
                tma_issue("H", (k, j), "h_full")
                n += 1

    def issuer():
        n = 0
        for k, (b, s0, s1, k0, k1, nt) in enumerate(segs):
            yield wait("q_full", k)
            yield wait("q_tmem", k)
            for j in range(nt):
                yield wait("x_full", n)
                pipe.append(("mma", ["X", "qs", "qt"], ("score_x", k, j)))
                pipe.append(("commit", "x_empty"))
                yield wait("h_full", n)
                pipe.append(("mma", ["H", "qs", "qt"], ("score_h", k, j)))
                pipe.append(("commit", "s_full"))
                yield wait("p_full", n)
                pipe.append(("mma", ["H", "P"], ("pv", k, j)))
                pipe.append(("commit", "h_empty"))
                pipe.append(("commit", "pv_done"))
                n += 1
            pipe.append(("commit", "o_done"))
        pipe.append(("commit", "mma_idle"))
        yield wait("mma_idle", 0)

    def softmax():
        n = 0
        for k, (b, s0, s1, k0, k1, nt) in enumerate(segs):
            yield wait("q_stage", k)
            _check(st["H"] == ("q", k), "q's staged chunks missing: %r" % (st["H"],))
            _check(not pending_reads("qt"), "q written to tensor memory under a running MMA")
            st["qt"] = k
            st["q_copied"].add(k)
            B["q_tmem"].arrive(4)
            for j in range(nt):
                yield wait("s_full", n)
                _check(st["S"] == ("S", k, j, 2), "S read before both score parts: %r" % (st["S"],))
                _check(not pending_reads("P"), "P written over a P that P.V still reads")
                st["S"] = ("P", k, j)
                if j > 0 and rng.random() < p_resc:
                    yield wait("pv_done", n - 1)
                    _check(not any(op[0] == "mma" and op[2][0] == "pv" for op in pipe),
                           "O rescaled under a running P.V")
                    _check(st["O"] == (k, j), "O rescaled before the previous P.V landed")
                B["p_full"].arrive(4)
                n += 1
            yield wait("o_done", k)
            _check(st["O"] == (k, nt), "epilogue before the last P.V: %r" % (st["O"],))
            _check(not any(t in ("X", "H") for t, _, _ in tma),
                   "O staged in the slot while a copy into it is in flight")
            _check(not pending_reads("X") and not pending_reads("H"),
                   "O staged in the slot under a running MMA")
            st["X"] = st["H"] = "O"
            st["o_read"].add(k)
            st["O_busy"] = True          # the bulk copies read the staged rows ...
            yield ("step",)
            st["O_busy"] = False         # ... until each thread's drain returns
            B["epi_done"].arrive(4)

    roles = {"producer": producer(), "issuer": issuer(), "softmax": softmax()}
    waiting = {r: None for r in roles}
    done = set()

    def ready(w):
        if w[0] == "step":
            return True
        _, name, idx = w
        ph = B[name].phase
        _check(idx <= ph <= idx + 1, "barrier %r at phase %d, waiter wants %d" % (name, ph, idx))
        return ph == idx + 1

    def step_role(r):
        try:
            waiting[r] = next(roles[r])
        except StopIteration:
            done.add(r)
            waiting[r] = None

    def run_pipe_head():
        op = pipe.pop(0)
        if op[0] == "commit":
            B[op[1]].arrive()
            return
        kind, k, t = op[2]
        if kind in ("score_x", "score_h"):
            part = "X" if kind == "score_x" else "H"
            _check(st[part] == (k, t), "scores of (%d, %d) read %s = %r" % (k, t, part, st[part]))
            _check(st["qs"] == k and st["qt"] == k, "scores with another segment's q")
            if kind == "score_x":
                _check(st["S"] is None or st["S"][0] == "used",
                       "S overwritten before its P was consumed: %r" % (st["S"],))
                st["S"] = ("S", k, t, 1)
            else:
                _check(st["S"] == ("S", k, t, 1), "score parts out of order")
                st["S"] = ("S", k, t, 2)
        else:  # pv
            _check(st["H"] == (k, t), "P.V read H = %r" % (st["H"],))
            _check(st["S"] == ("P", k, t), "P.V before P: %r" % (st["S"],))
            if t == 0:
                _check(k == 0 or (k - 1) in st["o_read"], "O overwritten before its epilogue")
                st["O"] = (k, 1)
            else:
                _check(st["O"] == (k, t), "P.V accumulates into %r" % (st["O"],))
                st["O"] = (k, t + 1)
            st["S"] = ("used", k, t)

    for r in roles:
        step_role(r)
    for _ in range(1_000_000):
        moves = [("role", r) for r in roles
                 if r not in done and (waiting[r] is None or ready(waiting[r]))]
        if tma:
            moves.append(("tma", None))
        if pipe:
            moves.append(("pipe", None))
        if not moves:
            return len(done) == len(roles)
        kind, r = rng.choice(moves)
        if kind == "role":
            step_role(r)
        elif kind == "tma":
            target, tag, bar = tma.pop(rng.randrange(len(tma)))
            st[target] = tag
            B[bar].arrive()
        else:
            run_pipe_head()
    raise AssertionError("model did not terminate")


_CASES = [
    # B, Sk, nsplit, runs
    (32, 8192, 16, 76),     # the benchmark workload: runs of 6 or 7 segments
    (32, 8192, 19, 76),
    (3, 513, 4, 5),
    (2, 100, 3, 4),
    (1, 1, 1, 1),
    (5, 130, 7, 3),         # one-tile and two-tile folded segments, runs over 3 batches
    (4, 2049, 3, 2),
    (7, 64, 64, 6),         # one key per segment
]


@pytest.mark.parametrize("B,Sk,nsplit,runs", _CASES)
def test_runs_cover_every_segment_once(B, Sk, nsplit, runs):
    seen = {}
    for r in range(runs):
        for b, s0, s1, k0, k1, nt in segments(B, Sk, nsplit, runs, r):
            assert 0 <= s0 <= s1 < nsplit and nt >= 1 and 0 <= k0 < k1 <= Sk
            for s in range(s0, s1 + 1):
                assert (b, s) not in seen
                seen[b, s] = r
    assert len(seen) == B * nsplit
    # the folded segments of a batch element tile its keys exactly
    for b in range(B):
        segs = sorted(g[3:5] for r in range(runs) for g in segments(B, Sk, nsplit, runs, r)
                      if g[0] == b)
        assert segs[0][0] == 0 and segs[-1][1] == Sk
        assert all(a[1] == c[0] for a, c in zip(segs, segs[1:]))


@pytest.mark.parametrize("B,Sk,nsplit,runs", _CASES)
def test_protocol_completes_without_hazards(B, Sk, nsplit, runs):
    rng = random.Random(B * 1000 + nsplit)
    picked = sorted({0, runs - 1, runs // 2} | set(rng.sample(range(runs), min(runs, 4))))
    for r in picked:
        segs = segments(B, Sk, nsplit, runs, r)
        for seed in range(6):
            assert _run_cta(segs, random.Random(seed * 7919 + r), p_resc=seed / 5)


@pytest.mark.parametrize("planted", ["no_epi_wait", "q_early", "h_over_q"])
def test_planted_mistakes_are_caught(planted):
    segs = segments(5, 130, 7, 3, 1)
    assert len(segs) >= 2
    caught = 0
    for seed in range(40):
        try:
            _run_cta(segs, random.Random(seed), planted=planted)
        except _Fault:
            caught += 1
    assert caught > 0
