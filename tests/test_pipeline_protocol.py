"""The weight-gradient kernel's barrier protocol, played out on the CPU under
random schedules.

The kernel moves every 64-row stage through three kinds of actors: TMA
producers (H and G, each with a ring of its own), converter warps (G from
shared memory into A slots in tensor memory) and one MMA issuer.  They hand
the stages to one another through mbarriers, whose waits test only the parity
of a phase.  A waiter that is two phases ahead of a barrier sees the parity of
an older phase and passes early.  This model runs the same hand-offs with the
kernel's ring sizes and warp counts (read from the source) and random copy,
MMA and scheduling delays, and checks that every reader sees the stage it
expects and that no copy or store lands on data still to be read.  A second
scheme, in which the converter groups take whole stages in turn from one
shared ring, must fail: that shows the model can see the hazard.
"""

import os
import random
import re

import pytest

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "long_context_attention_seqattn_gb300", "csrc", "wgrad_bf16.cu")


def kernel_constants():
    text = open(SRC).read()
    out = {}
    for name in ("kHStages", "kGStages", "kASlots", "kConvWarps"):
        m = re.search(r"constexpr int %s = (\d+);" % name, text)
        assert m, name
        out[name] = int(m.group(1))
    return out


class Race(Exception):
    pass


class Barrier:
    """mbarrier: `count` arrivals plus the expected transaction bytes complete
    a phase; try_wait.parity(P) passes once the phase count's parity differs
    from P."""

    def __init__(self, count):
        self.count, self.pending, self.tx, self.phases = count, count, 0, 0

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phases += 1
            self.pending = self.count

    def arrive(self):
        self.pending -= 1
        if self.pending < 0:
            raise Race("more arrivals than the barrier's count")
        self._complete()

    def arrive_expect_tx(self, n):
        self.tx += n
        self.arrive()

    def complete_tx(self, n):
        self.tx -= n
        self._complete()

    def passes(self, parity):
        return (self.phases & 1) != parity


def simulate(scheme, n_st, h_stages, g_stages, groups, a_slots, seed):
    """scheme "kernel": separate H and G rings, every converter group takes
    every stage (its share of the rows).  scheme "turns": one ring holding H
    and G, converter group p takes the stages s with s % groups == p."""
    rng = random.Random(seed)
    events = []
    clock = [0.0]

    def later(dt, fn):
        events.append((clock[0] + dt, len(events) + rng.random(), fn))

    shared = scheme == "turns"
    if shared:
        g_stages = h_stages
    h_full = [Barrier(1) for _ in range(h_stages)]
    h_empty = [Barrier(1) for _ in range(h_stages)]
    g_full = h_full if shared else [Barrier(1) for _ in range(g_stages)]
    g_empty = None if shared else [Barrier(groups) for _ in range(g_stages)]
    a_full = [Barrier(1 if shared else groups) for _ in range(a_slots)]
    a_empty = [Barrier(1) for _ in range(a_slots)]
    h_data = [None] * h_stages           # stage whose H has landed in the slot
    g_data = [None] * g_stages
    g_reads_due = [0] * g_stages
    a_data = [dict() for _ in range(a_slots)]   # converter group -> stage stored
    mma_busy_until = [0.0]

    def copy(data, st, s, bar, reads_due=None):
        if reads_due is not None and reads_due[st]:
            raise Race(f"copy of stage {s} into slot {st} with reads of the old stage due")
        data[st] = None

        def land():
            data[st] = s
            bar.complete_tx(1)
        later(rng.uniform(1, 30), land)

    def producer_h():
        for s in range(n_st):
            st = s % h_stages
            yield h_empty[st], ((s // h_stages) & 1) ^ 1
            h_full[st].arrive_expect_tx(2 if shared else 1)
            copy(h_data, st, s, h_full[st])
            if shared:
                copy(g_data, st, s, h_full[st])

    def producer_g():
        for s in range(n_st):
            st = s % g_stages
            yield g_empty[st], ((s // g_stages) & 1) ^ 1
            g_full[st].arrive_expect_tx(1)
            copy(g_data, st, s, g_full[st], g_reads_due)
            g_reads_due[st] = groups

    def mma():
        for s in range(n_st):
            st, sl = s % h_stages, s % a_slots
            yield h_full[st], (s // h_stages) & 1
            yield a_full[sl], (s // a_slots) & 1
            if h_data[st] != s:
                raise Race(f"MMA of stage {s} found H of stage {h_data[st]}")
            need = [s % groups] if shared else range(groups)
            for gi in need:
                if a_data[sl].get(gi) != s:
                    raise Race(f"MMA of stage {s} found A part {gi} of stage {a_data[sl].get(gi)}")
            start = max(clock[0], mma_busy_until[0])
            mma_busy_until[0] = start + rng.uniform(5, 20)

            def commit(st=st, sl=sl, s=s):      # the MMA ran: its operands must still be there
                if h_data[st] != s or (shared and g_data[st] != s):
                    raise Race(f"stage {s} overwritten before its MMA ran")
                if any(v != s for v in a_data[sl].values()):
                    raise Race(f"A slot {sl} overwritten before the MMA of stage {s} ran")
                h_empty[st].arrive()
                a_empty[sl].arrive()
            later(mma_busy_until[0] - clock[0], commit)

    def converter(gi):
        stages = range(gi, n_st, groups) if shared else range(n_st)
        for s in stages:
            st, sl = s % g_stages, s % a_slots
            yield a_empty[sl], ((s // a_slots) & 1) ^ 1
            yield g_full[st], (s // g_stages) & 1
            if g_data[st] != s:
                raise Race(f"converter group {gi} read stage {g_data[st]} expecting {s}")
            if not shared:
                g_reads_due[st] -= 1
                g_empty[st].arrive()
            a_data[sl][gi] = s
            a_full[sl].arrive()

    actors = [producer_h(), mma()] + [converter(g) for g in range(groups)]
    if not shared:
        actors.append(producer_g())
    waits = {a: next(a, None) for a in actors}
    waits = {a: w for a, w in waits.items() if w is not None}
    for _ in range(10 ** 6):
        ready = [a for a, (bar, par) in waits.items() if bar.passes(par)]
        if ready and (not events or rng.random() < 0.5):
            a = rng.choice(ready)
            w = next(a, None)
            if w is None:
                del waits[a]
            else:
                waits[a] = w
        elif events:
            events.sort(key=lambda e: (e[0], e[1]))
            t, _, fn = events.pop(0)
            clock[0] = max(clock[0], t)
            fn()
        else:
            break
    if waits:
        raise Race(f"deadlock: {len(waits)} actors still waiting")


def failures(scheme, trials, **kw):
    bad = []
    for seed in range(trials):
        try:
            simulate(scheme, seed=seed, **kw)
        except Race as e:
            bad.append(str(e))
    return bad


@pytest.mark.parametrize("n_st", [1, 2, 3, 5, 32])
def test_kernel_protocol_has_no_race(n_st):
    c = kernel_constants()
    bad = failures("kernel", 60, n_st=n_st, h_stages=c["kHStages"], g_stages=c["kGStages"],
                   groups=c["kConvWarps"] // 4, a_slots=c["kASlots"])
    assert not bad, bad[0]


@pytest.mark.parametrize("h_stages,g_stages,groups,a_slots", [(3, 3, 4, 4), (4, 2, 2, 4), (2, 4, 4, 8), (3, 2, 2, 8)])
def test_protocol_has_no_race_at_other_ring_sizes(h_stages, g_stages, groups, a_slots):
    bad = failures("kernel", 40, n_st=24, h_stages=h_stages, g_stages=g_stages, groups=groups, a_slots=a_slots)
    assert not bad, bad[0]


def test_groups_taking_stages_in_turn_race():
    """The scheme the kernel avoids: with one 3-stage ring and two converter
    groups taking alternate stages, some schedule lets a group pass a stage
    barrier on an older phase's parity."""
    bad = failures("turns", 60, n_st=32, h_stages=3, g_stages=3, groups=2, a_slots=4)
    assert bad and any("expecting" in b for b in bad)
