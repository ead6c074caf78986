"""A model of the tensor-core expert kernel's barrier hand-offs, run under random schedules.

The kernel (csrc/expert_tc.cu) passes every operand through mbarriers whose waits test one
parity bit: a wait for a phase of parity p passes whenever the barrier's current phase has
the other parity, so a waiter that is two phases behind (or a whole ring lap ahead) cannot
tell.  This model replays the roles' loops with the same ring arithmetic (code producer,
activation-tile producer, MMA issuer, dequantiser sets taking units in turn, epilogue
warps), lets bulk copies land in any order and MMA commits arrive in issue order, and picks
the next runnable role at random.  It checks that

  - for every ring geometry the launcher can choose (int2/int4/int8 codes; 32-, 64- and
    128-row launches with one or two m-tiles per work item; code runs of 1, 2 or 4
    chunks), with the TMEM stages in use capped as the kernel caps them (kUnit * stages <=
    chunks of either ring) and no more dequantiser sets than stages, no schedule deadlocks
    and every wait passes on the phase it was meant for;
  - without the stage cap, the int8 64-row launch (six stages of two chunks against a ring
    of two 4-chunk code runs) has schedules in which a dequantiser set passes a code-ring
    wait one lap early; with three sets on two stages, a set passes a stage's done wait a
    lap early: the reasons for the two limits.
The model's barrier arithmetic does not depend on the m-tiles per item (a unit's chunks
carry both m-tiles' codes; the arrival counts are per chunk), only the geometry does.
"""
import random

import pytest

K_UNIT = 2          # chunks per TMEM stage hand-off
N_SETS = 3          # dequantiser sets
SMEM_RINGS = 220 * 1024
MAX_RUNS = 24
MAX_STAGES = 16


def launch_shape(nmax):
    """(m-tiles per item, accumulator buffers) of a launch of groups of <= nmax rows."""
    return {32: (2, 2), 64: (2, 1)}.get(nmax, (1, 2))


def geometry(bits, nmax, kc_gcd, capped=True, mt=None, accb=None):
    """The launch's rings, stages and dequantiser sets, as the kernel and its launcher
    size them."""
    if mt is None:
        mt, accb = launch_shape(nmax)
    stages = min(MAX_STAGES, (512 - accb * mt * nmax) // (32 * K_UNIT * mt))
    a_ring = 64 * 1024 if bits == 8 else 48 * 1024
    b_ring = SMEM_RINGS - a_ring
    if mt == 2:
        ra = 2 if kc_gcd % 2 == 0 else 1
    else:
        ra = 4 if kc_gcd % 4 == 0 else (2 if kc_gcd % 2 == 0 else 1)
    rb = ra if nmax == 32 else 1
    a_run = mt * ra * 128 * 64 * bits // 8
    b_stride = (rb + (1 if rb > 1 else 0)) * nmax * 128
    sa, sb = min(MAX_RUNS, a_ring // a_run), min(MAX_RUNS, b_ring // b_stride)
    st = min(stages, min(sa * ra, sb * rb) // K_UNIT) if capped else stages
    sets = min(N_SETS, st) if capped else N_SETS
    return dict(ST=st, SA=sa, ra=ra, SB=sb, rb=rb, sets=sets)


class Bar:
    """An mbarrier: an arrival count per phase, transaction bytes, a phase number."""
    changes = 0  # every arrival or landing, over all barriers (the scheduler's clock)

    def __init__(self, count):
        self.count, self.pending, self.tx, self.phase = count, count, 0, 0

    def arrive(self, expect_tx=0):
        Bar.changes += 1
        self.tx += expect_tx
        self.pending -= 1
        self._complete()

    def land(self, n=1):
        Bar.changes += 1
        self.tx -= n
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def passes(self, parity):  # mbarrier.try_wait.parity
        return (self.phase & 1) != parity


class Ring:
    def __init__(self, stages, per_run=1):
        self.stages, self.per_run, self.s, self.ph, self.j, self.n = stages, per_run, 0, 0, 0, 0

    def step(self):  # one chunk (or one run when per_run is 1)
        self.j += 1
        if self.j == self.per_run:
            self.j, self.n = 0, self.n + 1
            self.s += 1
            if self.s == self.stages:
                self.s, self.ph = 0, self.ph ^ 1


class EarlyPass(Exception):
    pass


def run_schedule(seed, ST, SA, ra, SB, rb, items, sets=N_SETS):
    """One random schedule; returns 'ok' or 'deadlock', raises EarlyPass on a wait that
    passed before the phase it stood for had completed."""
    rng = random.Random(seed)
    a_full, a_empty = [Bar(1) for _ in range(SA)], [Bar(4 * ra) for _ in range(SA)]
    b_full, b_empty = [Bar(1) for _ in range(SB)], [Bar(1) for _ in range(SB)]
    t_full, done = [Bar(4) for _ in range(ST)], [Bar(1) for _ in range(ST)]
    acc_full, acc_empty = [Bar(1), Bar(1)], [Bar(4), Bar(4)]
    copies, commits = [], []

    def wait(bar, parity, need):
        """Poll until the wait passes; `need` = the phase count the wait stands for."""
        while not bar.passes(parity):
            yield "blocked"
        if bar.phase < need:
            raise EarlyPass

    def producer(full, empty, per_run, stages):
        pos = Ring(stages)
        for kc_total in items:
            for _ in range(0, kc_total, per_run):
                yield from wait(empty[pos.s], pos.ph ^ 1, pos.n // stages)
                full[pos.s].arrive(expect_tx=1)
                copies.append(full[pos.s])
                pos.step()

    def issuer():
        t, b = Ring(ST), Ring(SB, rb)
        for n, kc_total in enumerate(items):
            yield from wait(acc_empty[n & 1], ((n >> 1) & 1) ^ 1, n >> 1)
            for ku in range(0, kc_total, K_UNIT):
                yield from wait(t_full[t.s], t.ph, t.n // ST + 1)
                for j in range(K_UNIT):
                    if b.j + 1 >= rb or ku + j + 1 >= kc_total:
                        commits.append(b_empty[b.s])
                    b.step()
                commits.append(done[t.s])
                t.step()
            commits.append(acc_full[n & 1])

    def dequantiser(my_set, q):
        t, a, b = Ring(ST), Ring(SA, ra), Ring(SB, rb)
        unit = 0
        for kc_total in items:
            for _ in range(0, kc_total, K_UNIT):
                if unit % sets == my_set:
                    yield from wait(done[t.s], t.ph ^ 1, t.n // ST)
                    for _ in range(K_UNIT):
                        yield from wait(a_full[a.s], a.ph, a.n // SA + 1)
                        a_empty[a.s].arrive()
                        if q == 0:
                            yield from wait(b_full[b.s], b.ph, b.n // SB + 1)
                        a.step()
                        b.step()
                    yield "step"
                    t_full[t.s].arrive()
                else:
                    for _ in range(K_UNIT):
                        a.step()
                        b.step()
                unit += 1
                t.step()

    def epilogue():
        for n, _ in enumerate(items):
            yield from wait(acc_full[n & 1], (n >> 1) & 1, (n >> 1) + 1)
            yield "step"
            acc_empty[n & 1].arrive()

    roles = [producer(a_full, a_empty, ra, SA), producer(b_full, b_empty, rb, SB), issuer()]
    roles += [epilogue() for _ in range(4)]
    roles += [dequantiser(s, q) for s in range(sets) for q in range(4)]
    live, blocked = list(roles), set()  # blocked: polled a failing wait since the last change
    while True:
        runnable = [r for r in live if id(r) not in blocked]
        choices = runnable + ["copy"] * (2 if copies else 0) + ["commit"] * (2 if commits else 0)
        if not choices:
            return "deadlock" if live else "ok"
        pick = rng.choice(choices)
        before = Bar.changes
        if pick == "copy":
            copies.pop(rng.randrange(len(copies))).land()
        elif pick == "commit":
            commits.pop(0).arrive()
        else:
            try:
                what = next(pick)
            except StopIteration:
                live.remove(pick)
                what = "step"
        if Bar.changes != before:
            blocked.clear()
        if pick not in ("copy", "commit") and what == "blocked":
            blocked.add(id(pick))


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("nmax,mt,accb", [(32, 2, 2), (64, 2, 1), (64, 2, 2), (128, 2, 1),
                                          (128, 1, 2)])
@pytest.mark.parametrize("kc_gcd", [32, 6, 3])
def test_capped_geometries_never_pass_early_or_deadlock(bits, nmax, mt, accb, kc_gcd):
    geo = geometry(bits, nmax, kc_gcd, mt=mt, accb=accb)
    assert geo["ST"] >= 2 and K_UNIT * geo["ST"] <= min(geo["SA"] * geo["ra"], geo["SB"] * geo["rb"])
    assert geo["sets"] <= geo["ST"]
    items = [kc_gcd * max(1, 12 // kc_gcd) * 2] * 3  # whole units, a few rings' worth
    for seed in range(12):
        assert run_schedule(seed, items=items, **geo) == "ok", (geo, seed)


def test_uncapped_int8_64_row_launch_passes_a_code_wait_a_lap_early():
    geo = geometry(8, 64, 32, capped=False, mt=1, accb=2)
    assert geo["ST"] * K_UNIT > geo["SA"] * geo["ra"]  # 12 chunks of stages, 8 of code ring
    early = 0
    for seed in range(40):
        try:
            run_schedule(seed, items=[32] * 4, **geo)
        except EarlyPass:
            early += 1
    assert early > 0
    capped = geometry(8, 64, 32, mt=1, accb=2)
    assert capped["ST"] == 4
    for seed in range(40):
        assert run_schedule(seed, items=[32] * 4, **capped) == "ok"


def test_more_sets_than_stages_pass_a_done_wait_a_lap_early():
    # a 64-row launch with two m-tiles per item and two accumulator buffers has two stages:
    # three sets would each come back to a stage only every sixth unit, after it turned
    # over twice
    geo = geometry(4, 64, 32, mt=2, accb=2)
    assert geo["ST"] == 2 and geo["sets"] == 2
    early = 0
    for seed in range(20):
        try:
            run_schedule(seed, items=[96] * 2, **dict(geo, sets=3))
        except EarlyPass:
            early += 1
    assert early > 0
    for seed in range(20):
        assert run_schedule(seed, items=[96] * 2, **geo) == "ok"
