"""Model check of the one-tile kernel's barrier protocol (csrc/fa_fwd1_sm103.cu), on the CPU.

The kernel's MMA warp issues, per key step g of a query tile, S(g + 1) and then P V(g) after
waiting for P(g); four softmax warps wait for S(g), write P(g) over it and arrive on the P
barrier, waiting for P V(g - 1) first only when they rescale O; at the end of a tile each
waits for the tile's last P V.  Every wait is an mbarrier parity wait, which can only tell
whether the phase of a given parity has completed: a waiter that meets its barrier two phases
past the phase it wants misreads it.

The model runs the MMA warp, the four softmax warps and an in-order tensor pipe as coroutines
under random schedules and checks that every wait that passes sees its event really done and
that the run ends.  Two barriers per event (key step g on barrier g % 2, phase (g / 2) % 2),
the kernel's scheme, must pass every schedule; one barrier per event is correct only while the
softmax waits for P V(g - 1) in every step, and fails without that wait.
"""
import random

import pytest


class _Bar:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def passed(self, parity):
        # mbarrier.try_wait.parity: true once the phase of this parity has completed, i.e.
        # while the current phase has the other parity
        return (self.phase & 1) != parity


class _Violation(Exception):
    pass


def _run(seed, two_barriers, wait_pv_every_step, warps=4, plant=None):
    rnd = random.Random(seed)
    tiles = [rnd.randint(1, 5) for _ in range(rnd.randint(1, 6))]
    nb = 2 if two_barriers else 1
    bar_s = [_Bar(1) for _ in range(2)]            # S buffers alternate in every scheme
    bar_p = [_Bar(warps) for _ in range(nb)]
    bar_pv = [_Bar(1) for _ in range(nb)]
    s_done, pv_done = set(), set()
    p_done = {w: set() for w in range(warps)}
    pipe = []

    def pick(bars, g):
        return bars[g & 1] if len(bars) == 2 else bars[0]

    def parity(bars, g):
        return ((g >> 1) & 1) if len(bars) == 2 else (g & 1)

    def mma():
        g = 0
        for nk in tiles:
            pipe.append(("S", g))
            yield
            for j in range(nk):
                gs = g + j
                if j + 1 < nk:
                    pipe.append(("S", gs + 1))
                    yield
                while plant != "mma_skips_p_wait" and not pick(bar_p, gs).passed(parity(bar_p, gs)):
                    yield "wait"
                if any(gs not in p_done[w] for w in range(warps)):
                    raise _Violation(f"MMA warp passed P({gs}) early")
                pipe.append(("PV", gs))
                yield
            g += nk

    def softmax(w):
        g = 0
        for nk in tiles:
            for j in range(nk):
                gs = g + j
                while plant != "softmax_skips_s_wait" and not bar_s[gs & 1].passed((gs >> 1) & 1):
                    yield "wait"
                if gs not in s_done:
                    raise _Violation(f"softmax warp {w} passed S({gs}) early")
                rescale = j > 0 and rnd.random() < 0.3
                if j > 0 and (rescale or wait_pv_every_step):
                    while not pick(bar_pv, gs - 1).passed(parity(bar_pv, gs - 1)):
                        yield "wait"
                    if gs - 1 not in pv_done:
                        raise _Violation(f"softmax warp {w} passed P V({gs - 1}) early")
                p_done[w].add(gs)
                pick(bar_p, gs).arrive()
                yield
            last = g + nk - 1
            while not pick(bar_pv, last).passed(parity(bar_pv, last)):
                yield "wait"
            if last not in pv_done:
                raise _Violation(f"softmax warp {w} read O before P V({last})")
            g += nk

    procs = [mma()] + [softmax(w) for w in range(warps)]
    alive = list(range(len(procs)))
    idle = 0
    while alive or pipe:
        choice = rnd.choice(alive + (["pipe"] if pipe else []))
        if choice == "pipe":
            kind, g = pipe.pop(0)   # in order, as the tensor pipe completes them
            if kind == "S":
                s_done.add(g)
                bar_s[g & 1].arrive()
            else:
                pv_done.add(g)
                pick(bar_pv, g).arrive()
            idle = 0
            continue
        try:
            idle = idle + 1 if next(procs[choice]) == "wait" else 0
        except StopIteration:
            alive.remove(choice)
            idle = 0
        if idle > 5000:
            return "deadlock"
    return "ok"


def _outcomes(seeds, **kw):
    out = {}
    for seed in range(seeds):
        try:
            r = _run(seed, **kw)
        except _Violation:
            r = "violation"
        out[r] = out.get(r, 0) + 1
    return out


def test_two_barriers_per_event_hold_under_every_schedule():
    """The kernel's scheme: P published without waiting for the previous P V, S / P / P V each
    on two alternating barriers."""
    assert _outcomes(600, two_barriers=True, wait_pv_every_step=False) == {"ok": 600}


def test_one_barrier_per_event_needs_the_per_step_wait():
    """With one barrier per event the protocol holds only while every step waits for the
    previous P V (the softmax cannot then run a step ahead of the MMA warp's wait)."""
    assert _outcomes(600, two_barriers=False, wait_pv_every_step=True) == {"ok": 600}
    broken = _outcomes(600, two_barriers=False, wait_pv_every_step=False)
    assert broken.get("violation", 0) + broken.get("deadlock", 0) > 300


@pytest.mark.parametrize("plant", ["softmax_skips_s_wait", "mma_skips_p_wait"])
def test_model_catches_a_planted_missing_wait(plant):
    """The checker itself: a role that skips one of its waits is caught on most schedules."""
    out = _outcomes(200, two_barriers=True, wait_pv_every_step=False, plant=plant)
    assert out.get("violation", 0) > 100


# ----------------------------------------------------------------------------------------------
# Staged output at D = 256: the one query buffer holds in turn Q(t) (until its copy into tensor
# memory completes: barQcp phase t) and the output rows of tile t - 1 (staged by the softmax once
# Q(t) has been copied: barStaged[(t - 1) % 2]); the Q producer stores those rows, signals that
# the stores have read them (barOread phase t - 1) and only then loads Q(t + 1).  The last tile
# has no next query copy to wait for: its epilogue waits for the read of the previous tile's rows
# instead.  The model checks that no query tile is overwritten before its copy completes, that
# rows are staged only over a copied query tile or read-out rows, stored only once staged, and
# never lost.  (A tile's last P V completes after its query copy: the tensor pipe runs them in
# issue order.)

def _run_staged(seed, two_staged_barriers=True, skip_copy_wait=False, last_waits_read=True):
    rnd = random.Random(seed)
    T = rnd.randint(1, 7)
    bar_q = _Bar(1)                     # Q(t) landed (phase t)
    bar_qcp = _Bar(1)                   # Q(t) copied into tensor memory (phase t)
    nst = 2 if two_staged_barriers else 1
    bar_st = [_Bar(1) for _ in range(nst)]   # rows of tile t staged (one arrival stands for the 4 warps)
    bar_or = _Bar(1)                    # rows of tile t read by their bulk stores (phase t)
    buf = {"holds": None}               # ("Q", t) or ("O", t) or None
    copied, staged, stored = set(), set(), set()
    inflight = []                       # async completions: ("load", t) / ("copy", t)

    def pick(t):
        return bar_st[t & 1] if nst == 2 else bar_st[0]

    def par(t):
        return ((t >> 1) & 1) if nst == 2 else (t & 1)

    def producer():
        for t in range(T):
            if t == 1:
                while not bar_qcp.passed(0):
                    yield "wait"
            if t >= 2:
                k = t - 2
                while not pick(k).passed(par(k)):
                    yield "wait"
                if buf["holds"] != ("O", k):
                    raise _Violation(f"store of O({k}) finds {buf['holds']}")
                stored.add(k)
                buf["holds"] = None                  # the stores have read the buffer
                bar_or.arrive()
                yield
            if buf["holds"] is not None and buf["holds"][0] == "Q" and buf["holds"][1] not in copied:
                raise _Violation(f"Q({t}) load over an uncopied {buf['holds']}")
            if buf["holds"] is not None and buf["holds"][0] == "O":
                raise _Violation(f"Q({t}) load over unstored {buf['holds']}")
            inflight.append(("load", t))
            yield
        for k in range(max(0, T - 2), T):
            while not pick(k).passed(par(k)):
                yield "wait"
            if buf["holds"] != ("O", k):
                raise _Violation(f"final store of O({k}) finds {buf['holds']}")
            stored.add(k)
            buf["holds"] = None
            bar_or.arrive()
            yield

    pv_done = set()

    def mma():
        for t in range(T):
            while not bar_q.passed(t & 1):
                yield "wait"
            if buf["holds"] != ("Q", t):
                raise _Violation(f"copy of Q({t}) finds {buf['holds']}")
            inflight.append(("copy", t))
            yield
            for _ in range(rnd.randint(0, 3)):       # the tile's key steps
                yield
            while t not in copied:                   # in-order pipe: the copy completes first
                yield "wait"
            pv_done.add(t)

    def softmax():
        for t in range(T):
            while t not in pv_done:
                yield "wait"
            if t + 1 < T and not skip_copy_wait:
                while not bar_qcp.passed((t + 1) & 1):
                    yield "wait"
            if t + 1 == T and t >= 1 and last_waits_read:
                while not bar_or.passed((t - 1) & 1):
                    yield "wait"
            h = buf["holds"]
            if t + 1 < T and h != ("Q", t + 1):
                raise _Violation(f"O({t}) staged over {h}")
            if h is not None and h[0] == "Q" and h[1] not in copied:
                raise _Violation(f"O({t}) staged over uncopied {h}")
            if h is not None and h[0] == "O":
                raise _Violation(f"O({t}) staged over unstored {h}")
            buf["holds"] = ("O", t)
            staged.add(t)
            pick(t).arrive()
            yield

    procs = [producer(), mma(), softmax()]
    alive = list(range(3))
    idle = 0
    while alive or inflight:
        choice = rnd.choice(alive + (["async"] if inflight else []))
        if choice == "async":
            kind, t = inflight.pop(rnd.randrange(len(inflight)))
            if kind == "load":
                buf["holds"] = ("Q", t)
                bar_q.arrive()
            else:
                copied.add(t)
                bar_qcp.arrive()
            idle = 0
            continue
        try:
            idle = idle + 1 if next(procs[choice]) == "wait" else 0
        except StopIteration:
            alive.remove(choice)
            idle = 0
        if idle > 5000:
            return "deadlock"
    if stored != set(range(T)):
        raise _Violation("rows lost")
    return "ok"


def _staged_outcomes(seeds, **kw):
    out = {}
    for seed in range(seeds):
        try:
            r = _run_staged(seed, **kw)
        except _Violation:
            r = "violation"
        out[r] = out.get(r, 0) + 1
    return out


def test_staged_output_protocol_holds():
    """The kernel's scheme: every query tile copied before the buffer is reused, every tile's
    rows staged over a copied query tile and stored exactly once, under every schedule."""
    assert _staged_outcomes(800) == {"ok": 800}


def test_staged_output_protocol_catches_planted_mistakes():
    """Staging without waiting for the next query tile's copy, or the last tile staging without
    waiting for the previous tile's rows to be read out, each fail."""
    nowait = _staged_outcomes(800, skip_copy_wait=True)
    assert nowait.get("violation", 0) > 100
    noread = _staged_outcomes(800, last_waits_read=False)
    assert noread.get("violation", 0) > 100
