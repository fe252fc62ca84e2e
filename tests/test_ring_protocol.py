"""A randomised model of the score CTA's barrier protocol in the decode attention kernel
(tc_attention.cuh): a producer fills a 3-stage ring with each segment's two query items and
then its pages; two issuer warps take alternate pages into two score buffers; the softmax warps
copy the query into TMEM, release it to both issuers and read every page's scores.

An mbarrier completes phase after phase; a wait names the parity of the phase it wants and
passes when the barrier's current phase has the other parity.  So a wait is only unambiguous
when its barrier is at most one phase ahead of the phase it names.  The model raises on a wait
that passes with the barrier two or more phases ahead (a spurious pass) and on a schedule that
stops making progress (a deadlock).

The kernel's protocol (a page's full barrier is one of (stage, issuer), a query item's one of
its stage, and a query-seen barrier that both issuers arrive on before the softmax releases
the next query) passes every schedule; sharing one full barrier per stage, or dropping the
query-seen barrier, fails some."""
import random

import pytest

STAGES, Q_ITEMS = 3, 2


class Spurious(Exception):
    pass


class Deadlock(Exception):
    pass


class Bar:
    """An mbarrier: `count` arrivals (plus any expected transaction bytes) complete a phase."""

    def __init__(self, count):
        self.count, self.pending, self.tx, self.done = count, count, 0, 0

    def arrive(self, tx=0):
        assert self.pending > 0, "over-arrival"
        self.pending -= 1
        self.tx += tx
        self._check()

    def complete_tx(self, tx):
        self.tx -= tx
        self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count

    def try_wait(self, phase):
        """Wait for phase `phase` (0-based) by its parity, as the hardware does."""
        ok = (self.done & 1) != (phase & 1)
        if ok and self.done <= phase:
            raise Spurious(f"phase {phase} passed with {self.done} completed")
        if ok and self.done > phase + 1:
            raise Spurious(f"phase {phase} passed with {self.done} completed (two or more ahead)")
        return ok


def run(segs, rnd, shared_full, qseen):
    full_q = [Bar(1) for _ in range(STAGES)]
    full_p = [[Bar(1) for _ in range(2)] for _ in range(STAGES)]
    empty = [Bar(1) for _ in range(STAGES)]
    sfull = [Bar(1) for _ in range(2)]
    sfree = [Bar(4) for _ in range(2)]
    qready, qseen_bar, done = Bar(4), Bar(2), Bar(2)
    events, now = [], [0]

    def later(fn):
        events.append((now[0] + rnd.randint(1, 40), fn))

    def wait(bar, phase):
        while not bar.try_wait(phase):
            yield

    def page_bar(stage, page):
        return full_q[stage] if shared_full else full_p[stage][page & 1]

    def producer():
        k = g = 0
        for npg in segs:
            for _ in range(Q_ITEMS):
                if k >= STAGES:
                    yield from wait(empty[k % STAGES], k // STAGES - 1)
                b = full_q[k % STAGES]
                b.arrive(tx=1)
                later(lambda b=b: b.complete_tx(1))
                k += 1
            for _ in range(npg):
                if k >= STAGES:
                    yield from wait(empty[k % STAGES], k // STAGES - 1)
                b = page_bar(k % STAGES, g)
                b.arrive(tx=1)
                later(lambda b=b: b.complete_tx(1))
                k += 1
                g += 1

    def issuer(me):
        k = g = 0
        seen = {}  # barrier -> phases this issuer has waited for
        for si, npg in enumerate(segs):
            yield from wait(qready, si)
            if qseen:
                qseen_bar.arrive()
            for qi in range(Q_ITEMS):
                if me == 0:
                    empty[(k + qi) % STAGES].arrive()
            k += Q_ITEMS
            for _ in range(npg):
                if (g & 1) == me:
                    st = k % STAGES
                    b = page_bar(st, g)
                    if shared_full:
                        phase = k // STAGES
                    else:
                        phase = seen.get(id(b), 0)
                        seen[id(b)] = phase + 1
                    yield from wait(b, phase)
                    if g >= 2:
                        yield from wait(sfree[me], (g >> 1) - 1)
                    for _ in range(rnd.randint(0, 8)):
                        yield
                    later(lambda st=st, me=me: (sfull[me].arrive(), empty[st].arrive()))
                k += 1
                g += 1
        done.arrive()

    def softmax_warps():
        k = g = 0
        seen = {}
        for si, npg in enumerate(segs):
            for _ in range(Q_ITEMS):
                b = full_q[k % STAGES]
                if shared_full:
                    phase = k // STAGES
                else:
                    phase = seen.get(id(b), 0)
                    seen[id(b)] = phase + 1
                yield from wait(b, phase)
                k += 1
            if qseen and si > 0:
                yield from wait(qseen_bar, si - 1)
            for _ in range(4):
                qready.arrive()
            for _ in range(npg):
                yield from wait(sfull[g & 1], g >> 1)
                for _ in range(rnd.randint(0, 10)):
                    yield
                for _ in range(4):
                    sfree[g & 1].arrive()
                g += 1
                k += 1

    parties = [producer(), issuer(0), issuer(1), softmax_warps()]
    alive = list(parties)
    starve = rnd.random() < 0.5  # stretches in which one party is not scheduled at all
    steps = 0
    while alive or events:
        steps += 1
        if steps > 200_000:
            raise Deadlock(f"segments {segs}")
        now[0] += 1
        for e in [e for e in events if e[0] <= now[0]]:
            events.remove(e)
            e[1]()
        rnd.shuffle(alive)
        pick = alive[: rnd.randint(1, len(alive))] if alive else []
        if starve and (now[0] // 300) % 2 == 1:
            slow = parties[(now[0] // 600) % len(parties)]
            pick = [p for p in pick if p is not slow]
        for p in pick:
            try:
                next(p)
            except StopIteration:
                alive.remove(p)
    assert done.done == 1


def schedules(n, seed0=0):
    for seed in range(seed0, seed0 + n):
        rnd = random.Random(seed)
        segs = [rnd.choice([1, 1, 2, 3, 5, 16, 33]) for _ in range(rnd.randint(1, 8))]
        yield seed, segs, rnd


def test_kernel_protocol_never_passes_early_or_deadlocks():
    for seed, segs, rnd in schedules(300):
        run(segs, rnd, shared_full=False, qseen=True)


@pytest.mark.parametrize("shared_full,qseen", [(True, True), (False, False)])
def test_simpler_protocols_fail(shared_full, qseen):
    """One full barrier per stage (both issuers skip each other's pages on it), or no
    query-seen barrier (an issuer with no page in a segment can fall two query phases
    behind): some schedule passes a wait early or deadlocks."""
    for seed, segs, rnd in schedules(400):
        try:
            run(segs, rnd, shared_full=shared_full, qseen=qseen)
        except (Spurious, Deadlock):
            return
    pytest.fail("no schedule exposed the simpler protocol")


def run_p_ring(n_pages, npbuf, rnd, rule):
    """The value CTA's P buffers: the softmax writes page g's P into buffer g % npbuf; the PVs
    complete in page order (one thread issues them and each commit covers all its earlier
    MMAs); a release warp waits for each PV in order and then arrives on the buffer's empty
    barrier (in the kernel a remote arrive with release semantics, waited on with a
    cluster-scope acquire, so a later buffer's phase also shows the earlier arrivals).
    rule "pairs" is the kernel's: an even page waits for the next page's buffer, which covers
    its own, and an odd page waits for nothing; "every" waits for each page's own buffer;
    "even_own" (wrong) waits only on even pages, for their own buffer.  Raises if a wait passes
    early or P is written over a buffer whose PV is still pending."""
    empty = [Bar(1) for _ in range(npbuf)]
    full = [Bar(1) for _ in range(npbuf)]
    pv_done = [False] * n_pages
    events, now, last_pv = [], [0], [0]

    def later(fn, at=None):
        events.append((at if at is not None else now[0] + rnd.randint(1, 30), fn))

    def wait(bar, phase):
        while not bar.try_wait(phase):
            yield

    def softmax_warps():
        for g in range(n_pages):
            for _ in range(rnd.randint(0, 6)):
                yield
            gw = {"every": g, "pairs": g + 1 if g % 2 == 0 else None,
                  "even_own": g if g % 2 == 0 else None}[rule]
            if gw is not None and gw >= npbuf:
                yield from wait(empty[gw % npbuf], gw // npbuf - 1)
            if g >= npbuf and not pv_done[g - npbuf]:
                raise Spurious(f"P of page {g} written while the PV of page {g - npbuf} is pending")
            later(lambda b=g % npbuf: full[b].arrive())  # the st.async bytes land

    def value_mma():
        for g in range(n_pages):
            yield from wait(full[g % npbuf], g // npbuf)
            for _ in range(rnd.randint(0, 8)):
                yield
            last_pv[0] = max(now[0] + rnd.randint(1, 30), last_pv[0] + 1)  # in page order
            later(lambda g=g: pv_done.__setitem__(g, True), at=last_pv[0])

    def release_warp():
        for g in range(n_pages):
            while not pv_done[g]:
                yield
            for _ in range(rnd.randint(0, 4)):
                yield
            empty[g % npbuf].arrive()

    parties = [softmax_warps(), value_mma(), release_warp()]
    alive = list(parties)
    steps = 0
    while alive or events:
        steps += 1
        if steps > 200_000:
            raise Deadlock(f"{n_pages} pages")
        now[0] += 1
        for e in [e for e in events if e[0] <= now[0]]:
            events.remove(e)
            e[1]()
        rnd.shuffle(alive)
        for p in (alive[: rnd.randint(1, len(alive))] if alive else []):
            try:
                next(p)
            except StopIteration:
                alive.remove(p)
    assert all(pv_done)


@pytest.mark.parametrize("npbuf", [2, 4])
def test_p_buffer_waits_every_other_page(npbuf):
    for seed in range(200):
        rnd = random.Random(seed)
        run_p_ring(rnd.randint(1, 40), npbuf, rnd, "pairs")
        run_p_ring(rnd.randint(1, 40), npbuf, rnd, "every")


def test_p_buffer_wrong_rule_fails():
    """Waiting on even pages for their own buffer only leaves the odd pages unguarded."""
    for seed in range(200):
        rnd = random.Random(seed)
        try:
            run_p_ring(rnd.randint(8, 40), 4, rnd, "even_own")
        except Spurious:
            return
    pytest.fail("no schedule exposed the wrong rule")
