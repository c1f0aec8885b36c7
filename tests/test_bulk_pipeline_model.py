"""Barrier protocol of the 128-token-tile GEMM kernel (csrc/gemm.cu,
csrc/gemm_common.cuh), single-CTA and CTA-pair forms, checked on a model
(CPU).

Waits on an mbarrier test only the parity of a phase, so a wait is right
only if it starts after the phase before the one it wants has completed and
before the phase after it can complete.  The model runs every role as the
sequence of waits and arrivals the kernel takes, under adversarial
scheduling (copies land, and MMAs complete, only when a random draw lets
them, and some copies are held until nothing else can move), and counts
phases exactly.  A parity wait names the phase it means (n from 0, -1 for
"none yet") and tests n & 1, as the kernel's expressions do.

  * producer w of NPROD issues the groups gi with gi % NPROD == w into its
    sub-ring of SPS stages (stage (gi % NPROD) SPS + (gi / NPROD) % SPS, lap
    (gi / NPROD) / SPS): from a stage's second lap on it first waits for the
    stage's release (empty: 1 MMA commit + 4 dequant warps), then publishes
    the stage's sequence word gi + 1 and issues the copy;
  * dequant slot gi % NSLOT waits until the stage's sequence word is gi + 1
    (a value wait), then for the stage's copy (full) and for its A buffer
    (aempty, buffer gi % NABUF), then arrives on A-full (on the leading CTA's
    barrier in the pair form) and releases the stage;
  * the MMA issuer (each CTA's; the leading CTA's alone in the pair form),
    per fold chunk of up to 8 groups of a unit: waits for the chunk's
    accumulator (accempty), per group for its A buffer (afull: 4 arrivals, 8
    in the pair form), issues, and commits A-empty and the stage's empty
    barrier, and at the chunk's end the accumulator's full barrier; commits
    land when the MMAs before them complete, in issue order, and in the pair
    form on both CTAs' barriers;
  * the epilogue waits for each chunk's accumulator and releases it (on the
    leading CTA's barrier in the pair form: 16 arrivals, 32 there).
"""
import random

import pytest

NACC, FOLD, NABUF, NSLOT, NEPI = 2, 8, 4, 2, 16


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.done = count, count, 0

    def arrive(self, n):
        self.pending -= n
        assert self.pending >= 0, "more arrivals than the phase expects"
        if self.pending == 0:
            self.done += 1
            self.pending = self.count

    def passes(self, parity):
        return (self.done & 1) != parity


def make_schedule(T, G, P0):
    """The kernel's make_schedule: (T_dp, P, I_sk)."""
    if T >= P0:
        rem = T % P0
        T_sk = 0 if rem == 0 else min(T, rem + P0)
        return T - T_sk, P0, T_sk * G
    return 0, max(1, min(P0, (T * G + 3) // 4)), T * G


def worker_units(b, P, T, G, T_dp, I):
    """UnitIter's sequence for worker b (a CTA, or a CTA pair)."""
    units, t = [], b
    while t < T_dp:
        units.append((t, 0, G))
        t += P
    it, end = b * I // P, (b + 1) * I // P
    while it < end:
        sk, g0 = divmod(it, G)
        g1 = min(G, g0 + end - it)
        units.append((T_dp + sk, g0, g1))
        it += g1 - g0
    return units


def run(units, stages, nprod, pair, skip_seq_wait=False, local_release=False, hold=(), seed=0):
    """One worker (one CTA, or the two CTAs of a pair).  Returns (deadlocked,
    wrong passes)."""
    rng = random.Random(seed)
    sps = stages // nprod
    ctas = (0, 1) if pair else (0,)
    bars = {}
    for c in ctas:
        for s in range(stages):
            bars[c, "full", s], bars[c, "empty", s] = Bar(1), Bar(1 + 4)
        for a in range(NABUF):
            bars[c, "afull", a], bars[c, "aempty", a] = Bar(8 if pair else 4), Bar(1)
        for b in range(NACC):
            bars[c, "accfull", b], bars[c, "accempty", b] = Bar(1), Bar(2 * NEPI if pair else NEPI)
    seq = {(c, s): 0 for c in ctas for s in range(stages)}
    chunks, ngroups = [], 0  # per chunk: its groups' indices in the worker's order
    for _, g0, g1 in units:
        for c0 in range(g0, g1, FOLD):
            n = min(FOLD, g1 - c0)
            chunks.append(list(range(ngroups, ngroups + n)))
            ngroups += n

    def place(gi):
        k = gi // nprod
        return (gi % nprod) * sps + k % sps, k // sps

    inflight = []  # copies issued, not landed: (cta, stage, gi)
    mma_q = []  # MMA groups issued, not completed: (gi, commits after it)
    issued = set()

    def producer(c, w):
        for gi in range(w, ngroups, nprod):
            s, lap = place(gi)
            if lap:
                yield "wait", (c, "empty", s), lap - 1
            seq[c, s] = gi + 1
            inflight.append((c, s, gi))
            issued.add((c, gi))
            yield "step",

    def dequant(c, j):
        for gi in range(j, ngroups, NSLOT):
            s, lap = place(gi)
            a = gi % NABUF
            if not skip_seq_wait:
                yield "seq", (c, s), gi + 1
            yield "wait", (c, "full", s), lap
            yield "wait", (c, "aempty", a), gi // NABUF - 1
            yield "arrive", (0 if pair else c, "afull", a), 4
            yield "arrive", (c, "empty", s), 4

    def mma(c):
        gi = 0
        targets = ctas if pair else (c,)
        for ch, groups in enumerate(chunks):
            b = ch % NACC
            yield "wait", (c, "accempty", b), ch // NACC - 1
            for k, g in enumerate(groups):
                a = g % NABUF
                yield "wait", (c, "afull", a), g // NABUF
                commits = [(t, "aempty", a) for t in targets] + [(t, "empty", place(g)[0]) for t in targets]
                if k == len(groups) - 1:
                    commits += [(t, "accfull", b) for t in targets]
                mma_q.append((g, commits))
                yield "step",

    def epilogue(c):
        for ch in range(len(chunks)):
            b = ch % NACC
            yield "wait", (c, "accfull", b), ch // NACC
            yield "arrive", (0 if pair and not local_release else c, "accempty", b), NEPI

    roles = []
    for c in ctas:
        roles += [producer(c, w) for w in range(nprod)] + [dequant(c, j) for j in range(NSLOT)] + [epilogue(c)]
    roles += [mma(0)] if pair else [mma(c) for c in ctas]
    current, finished, wrong = [None] * len(roles), [False] * len(roles), []
    while not all(finished):
        moved = False
        free = [i for i, x in enumerate(inflight) if x[2] not in hold]
        if free and rng.random() < 0.5:
            c, s, _ = inflight.pop(free[rng.randrange(len(free))])
            bars[c, "full", s].arrive(1)
            moved = True
        if mma_q and rng.random() < 0.5:  # the oldest MMA group completes; its commits land
            _, commits = mma_q.pop(0)
            for key in commits:
                bars[key].arrive(1)
            moved = True
        for r in rng.sample(range(len(roles)), len(roles)):
            if finished[r]:
                continue
            if current[r] is None:
                try:
                    current[r] = next(roles[r])
                except StopIteration:
                    finished[r] = moved = True
                    continue
            op = current[r]
            if op[0] == "step":
                current[r], moved = None, True
            elif op[0] == "issued":
                if op[1] in issued:
                    current[r], moved = None, True
            elif op[0] == "seq":
                if seq[op[1]] == op[2]:
                    current[r], moved = None, True
            elif op[0] == "arrive":
                bars[op[1]].arrive(op[2])
                current[r], moved = None, True
            elif bars[op[1]].passes(op[2] & 1):
                bar = bars[op[1]]
                if bar.done != op[2] + 1:
                    wrong.append((op[1], op[2], bar.done))
                current[r], moved = None, True
        if not moved:
            if mma_q:
                _, commits = mma_q.pop(0)
                for key in commits:
                    bars[key].arrive(1)
            elif inflight:
                c, s, _ = inflight.pop(0)  # only held copies are left: land the oldest
                bars[c, "full", s].arrive(1)
            else:
                return True, wrong
    return False, wrong


# (form, stages, producers): the single-CTA kernel's five-stage ring, the
# pair kernel's two sub-rings of four
FORMS = [("single", 5, 1), ("pair", 8, 2)]


@pytest.mark.parametrize("form,stages,nprod", FORMS)
@pytest.mark.parametrize("M,N,K", [(128, 22016, 4096), (256, 4096, 14336), (200, 2048, 1024), (129, 512, 1152),
                                   (4096, 28672, 8192)])
def test_protocol_has_no_wrong_pass_and_no_deadlock(form, stages, nprod, M, N, K):
    pair = form == "pair"
    G, MT = K // 128, (M + 127) // 128
    T = MT * (N // (256 if pair else 128))
    T_dp, P, I = make_schedule(T, G, 76 if pair else 152)
    for b in sorted({0, 1, P // 2, P - 1}):
        units = worker_units(b, P, T, G, T_dp, I)[:6]  # the first units cover every transition
        ngroups = sum(g1 - g0 for _, g0, g1 in units)
        for seed, hold in [(0, ()), (1, ())] + [(2, (h,)) for h in range(min(ngroups, 6))]:
            dead, wrong = run(units, stages, nprod, pair, hold=hold, seed=seed)
            assert not dead, f"{form} worker {b} units {units} hold {hold}: deadlock"
            assert not wrong, f"{form} worker {b} units {units} hold {hold}: {wrong[:3]}"


def test_model_catches_a_skipped_sequence_wait():
    """Five stages shared by two dequant slots: a stage's consumer changes
    from lap to lap, so a slot that waited on the stage's parity without
    first checking the stage's sequence word could take a later lap's phase
    for its own (the copy for the group two laps on landing first)."""
    units = [(0, 0, 40)]
    found = any(run(units, 5, 1, False, skip_seq_wait=True, hold=(h,), seed=s)[1]
                for s in range(12) for h in range(10))
    assert found
    assert not any(run(units, 5, 1, False, hold=(h,), seed=s)[1] for s in range(12) for h in range(10))


def test_model_needs_the_pair_epilogue_on_the_leading_barrier():
    """In the pair form the leading CTA's accumulator-empty barrier counts
    both CTAs' epilogue warps (32): an epilogue that released the buffer on
    its own CTA's barrier instead would leave the issuer waiting for good."""
    units = [(0, 0, 24), (1, 0, 24)]
    assert run(units, 8, 2, True)[0] is False
    assert run(units, 8, 2, True, local_release=True)[0] is True
