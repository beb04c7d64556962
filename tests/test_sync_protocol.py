"""Deadlock freedom of the attention kernels' synchronisation protocol, checked on a model.

The forward kernel runs a TMA producer, one MMA-issuing thread per query tile and one element-wise
group per query tile; its two element-wise groups take turns (named-barrier ping-pong) on the key
tiles both query tiles see.  A ping-pong that paired the groups' i-th key tiles instead of the same
key tile could deadlock when the tiles' key ranges start at different tiles (packed segments): one
group waited for its turn while the shared K/V buffers waited for it.  The dQ kernel runs one
MMA-issuing thread that serves both query tiles in a fixed order (per key tile: each tile's dP after
its P, then each tile's dQ update and next S after its dS) and element-wise groups that run free;
with turns (phases = 2 below) it would be deadlock-free too, but measured no faster, so the kernel
has none.  The model follows the kernels' waits and releases step by step (MMAs complete as soon as
they are issued) and checks that every actor finishes, for random key ranges."""
import random

import pytest


def run(kind, ra, rb, valid1=True, NS=5, dq_turns=False):
    xa, wa = ra; xb, wb = rb if valid1 else (ra[0], ra[0])
    j0 = min(xa, xb) if valid1 else xa
    j1 = max(wa, wb) if valid1 else wa
    ranges = {0: (xa, wa), 1: (xb, wb)}
    inr = lambda t, j: ranges[t][0] <= j < ranges[t][1]
    n_iss = 2 if valid1 else 1
    ev = set()            # completed events
    cnt = {}              # counters (releases)
    def inc(k): cnt[k] = cnt.get(k, 0) + 1
    def get(k): return cnt.get(k, 0)
    pp_lo = max(xa, xb); pp_hi = min(wa, wb) if valid1 else pp_lo
    phases = (2 if dq_turns else 0) if kind == "dq" else 1
    n_pp = phases * max(0, pp_hi - pp_lo)
    give = {0: 0, 1: 0}   # arrivals received on barrier of group t
    def producer():
        if kind == "dq":
            for n, j in enumerate(range(j0, j1)):
                if n >= 2:
                    yield lambda: get(("k_rel", j - 2)) >= n_iss
                ev.add(("K", j))
                if n >= 1:
                    yield lambda: get(("v_rel", j - 1)) >= n_iss
                ev.add(("V", j))
        else:
            items = [("K", j) if i % 2 == 0 else ("V", j) for j in range(j0, j1) for i in (0, 1)]
            for it, item in enumerate(items):
                if it >= NS:
                    prev = items[it - NS]
                    yield lambda prev=prev: get(("rel",) + prev) >= n_iss
                ev.add(item)
    tiles = (0, 1) if valid1 else (0,)

    def issuer_dq():
        # one thread for both tiles: per key tile the dP of each tile (after its P), then the
        # dQ update and the next S of each tile (after its dS)
        yield lambda: ("K", j0) in ev
        for t in tiles:
            if inr(t, j0): ev.add(("S", t, j0))
        for j in range(j0, j1):
            yield lambda j=j: ("V", j) in ev
            for t in tiles:
                if inr(t, j):
                    yield lambda j=j, t=t: ("sfree", t, j) in ev
                    ev.add(("dP", t, j))
            inc(("v_rel", j)); inc(("v_rel", j))
            if j + 1 < j1:
                yield lambda j=j: ("K", j + 1) in ev
            for t in tiles:
                if inr(t, j):
                    yield lambda j=j, t=t: ("dsfull", t, j) in ev
                if inr(t, j + 1): ev.add(("S", t, j + 1))
            inc(("k_rel", j)); inc(("k_rel", j))

    def issuer(t):
        if kind == "dq":
            return
        else:
            yield lambda: ("K", j0) in ev
            if inr(t, j0): ev.add(("S", t, j0))
            inc(("rel", "K", j0))
            for j in range(j0, j1):
                yield lambda j=j: ("V", j) in ev
                if j + 1 < j1:
                    yield lambda j=j: ("K", j + 1) in ev
                if inr(t, j):
                    yield lambda j=j: ("P", t, j) in ev
                inc(("rel", "V", j))
                if inr(t, j + 1): ev.add(("S", t, j + 1))
                if j + 1 < j1: inc(("rel", "K", j + 1))
    def ew(t):
        n_give = n_pp if t == 0 else n_pp - 1
        state = {"turn": 0, "synced": 0}
        if t == 1 and n_pp > 0: give[0] += 1
        def take(pp):
            if pp:
                need = state["synced"] + 1
                yield lambda: give[t] >= need
                state["synced"] += 1
        def giv(pp):
            if pp:
                if state["turn"] < n_give: give[1 - t] += 1
                state["turn"] += 1
        for j in range(*ranges[t]):
            pp = phases > 0 and pp_lo <= j < pp_hi
            yield from take(pp)
            yield lambda j=j: ("S", t, j) in ev
            if kind == "dq":
                ev.add(("sfree", t, j))
                giv(pp)
                yield from take(pp)
                yield lambda j=j: ("dP", t, j) in ev
                ev.add(("dsfull", t, j))
                giv(pp)
            else:
                ev.add(("P", t, j))
                giv(pp)
    if kind == "dq":
        actors = [producer(), issuer_dq(), ew(0)]
        if valid1: actors += [ew(1)]
    else:
        actors = [producer(), issuer(0), ew(0)]
        if valid1: actors += [issuer(1), ew(1)]
    waits = [None] * len(actors)
    done = [False] * len(actors)
    while not all(done):
        progress = False
        for i, a in enumerate(actors):
            if done[i]: continue
            while waits[i] is None or waits[i]():
                try:
                    waits[i] = next(a); progress = True
                except StopIteration:
                    done[i] = True; break
            if done[i]: progress = True
        if not progress:
            return False
    return True



def test_known_offset_ranges_finish():
    assert run("dq", (0, 3), (2, 4))
    assert run("fwd", (0, 3), (5, 9))


@pytest.mark.parametrize("kind,dq_turns", [("dq", False), ("dq", True), ("fwd", False)])
def test_random_ranges_never_deadlock(kind, dq_turns):
    rng = random.Random(12345)
    for _ in range(3000):
        xa = rng.randint(0, 12); wa = xa + rng.randint(1, 12)
        xb = rng.randint(0, 12); wb = xb + rng.randint(1, 12)
        assert run(kind, (xa, wa), (xb, wb), rng.random() < 0.9, dq_turns=dq_turns), ((xa, wa), (xb, wb))


# dK/dV: one MMA issuer per element-wise group; the shared dK / dV accumulations stay in item
# order through token barriers; the element-wise groups take turns phase by phase.  With a window
# F, each group adds its accumulator to the global sums after its last item of every window that
# more items follow (once the Q-slot releases of the window's last two items show their MMAs
# complete), and group 0 hands the next window's first P^T over only after both groups have done
# so; the model also checks that no window's first dV MMA (which restarts the accumulators) is
# issued before both flushes of the previous window.
def run_dkdv_pp(N, NQ=3, NO=2, F=None, rng=None):
    ev = set()
    n_win = (N - 1) // F if F and N > 0 else 0
    Na, Nb = (N + 1) // 2, N // 2
    n_pp = 2 * min(Na, Nb)
    give = {0: 0, 1: 0}
    def producer():
        for n in range(N):
            if n >= NQ:
                yield lambda n=n: ("q_empty", n - NQ) in ev
            ev.add(("Q", n))
            if n >= NO:
                yield lambda n=n: ("o_empty", n - NO) in ev
            ev.add(("O", n))
    def issuer(g):
        if g >= N: return
        yield lambda: ("Q", g) in ev
        ev.add(("S", g))
        for n in range(g, N, 2):
            yield lambda n=n: ("P", n) in ev
            yield lambda n=n: ("O", n) in ev
            if n > 0:
                yield lambda n=n: ("dv_tok", n - 1) in ev
            if F and n % F == 0 and n > 0:   # restarts the accumulators
                w = n // F - 1
                assert ("flushed", 0, w) in ev and ("flushed", 1, w) in ev, (N, F, n)
            ev.add(("dv_tok", n))
            ev.add(("dP", n)); ev.add(("o_empty", n))
            yield lambda n=n: ("dS", n) in ev
            if n > 0:
                yield lambda n=n: ("dk_tok", n - 1) in ev
            ev.add(("dk_tok", n)); ev.add(("q_empty", n))
            if n + 2 < N:
                yield lambda n=n: ("Q", n + 2) in ev
                ev.add(("S", n + 2))
    def ew(g):
        n_give = n_pp if g == 0 else n_pp - 1
        st = {"turn": 0, "sync": 0}
        if g == 1 and n_pp > 0: give[0] += 1
        def take():
            if st["turn"] < n_pp:
                need = st["sync"] + 1
                yield lambda: give[g] >= need
                st["sync"] += 1
        def giv():
            if st["turn"] < n_pp:
                if st["turn"] < n_give: give[1 - g] += 1
            st["turn"] += 1
        for n in range(g, N, 2):
            yield from take()
            yield lambda n=n: ("S", n) in ev
            ev.add(("P", n)); giv()
            yield from take()
            yield lambda n=n: ("dP", n) in ev
            ev.add(("dS", n)); giv()
            if F and n % F == F - 2 + g and n // F < n_win:
                w = n // F
                m0, m1 = (w + 1) * F - 2, (w + 1) * F - 1
                yield lambda m0=m0, m1=m1: ("q_empty", m0) in ev and ("q_empty", m1) in ev
                # the sums read are complete: every MMA of the window has been issued
                assert all(("dk_tok", m) in ev for m in range(w * F, (w + 1) * F)), (N, F, w)
                ev.add(("flushed", g, w))
                if g == 0:
                    yield lambda w=w: ("flushed", 1, w) in ev
    actors = [producer(), issuer(0), issuer(1), ew(0), ew(1)]
    waits = [None] * len(actors); done = [False] * len(actors)
    if rng is not None:   # random interleaving: one step of a random runnable actor at a time
        while not all(done):
            ready = [i for i in range(len(actors)) if not done[i] and (waits[i] is None or waits[i]())]
            if not ready:
                return False
            i = rng.choice(ready)
            try:
                waits[i] = next(actors[i])
            except StopIteration:
                done[i] = True
        return True
    while not all(done):
        progress = False
        for i, a in enumerate(actors):
            if done[i]: continue
            while waits[i] is None or waits[i]():
                try:
                    waits[i] = next(a); progress = True
                except StopIteration:
                    done[i] = True; break
            if done[i]: progress = True
        if not progress: return False
    return True


def test_dkdv_two_issuers_never_deadlock():
    assert all(run_dkdv_pp(n) for n in range(0, 40))


@pytest.mark.parametrize("F", [2, 4, 6, 10])
def test_dkdv_flushed_windows_never_deadlock(F):
    assert all(run_dkdv_pp(n, F=F) for n in range(0, 40))
    rng = random.Random(F)
    for _ in range(300):
        assert run_dkdv_pp(rng.randrange(0, 30), F=F, rng=rng)
