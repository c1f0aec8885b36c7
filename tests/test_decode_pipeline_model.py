"""Barrier protocol of the decode GEMM kernel (csrc/gemm_decode.cu), checked on
a model (CPU).

The kernel's roles hand work to each other through mbarriers whose waits test
only the parity of a phase, so a wait is right only if it starts after the
phase before the one it wants has completed, and before the phase after it
can complete.  The model runs each role as a sequence of waits and arrivals,
in the order the kernel takes them, under adversarial scheduling (some copies
land only when nothing else can move), and counts phases exactly.  Each wait
names the phase it means (n, counted from 0; -1 for "none yet") and tests its
parity n & 1, which is what the kernel's parity expressions evaluate to.

  * producers: group gi (in the CTA's order) belongs to slot gi % NSLOT and
    goes to that slot's sub-ring of SPS stages; from a stage's second lap on,
    the copy first waits for the stage's release;
  * dequant slot j, per fold chunk (up to 8 * NSLOT consecutive groups of a
    unit): it waits for the chunk's accumulator to be free (also when it has
    no group in the chunk, then it only arrives); per own group it waits for
    the stage, releases it, waits until its previous group's MMAs are done,
    issues the group's MMAs, which complete on its MMA-done barrier, and after
    its last group of the chunk, on the chunk's accumulator barrier;
  * epilogue: waits for each chunk's accumulator and releases it.

Every parity wait must pass exactly on the phase it means, every stage must
still hold a group's bytes when its slot reads them, and no schedule may
deadlock.  Two planted mistakes must show: a slot skipping the accumulator
wait in chunks where it has no group (a wait passes a lap early), and a slot
releasing a stage before reading it (the stage is refilled under it).
"""
import random

import pytest

NACC, FOLD, NEPI = 2, 8, 4


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.done = count, count, 0

    def arrive(self, n):
        self.pending -= n
        assert self.pending >= 0, "more arrivals than the phase expects"
        if self.pending == 0:
            self.done += 1
            self.pending = self.count

    def passes(self, parity):  # mbarrier try_wait.parity: the phase of this parity has completed
        return (self.done & 1) != parity


def cta_units(b, P, T, G, T_dp):
    """The CTA's (tile, g0, g1) units: whole tiles round-robin, then its
    stream-K range of group iterations (csrc/gemm_common.cuh UnitIter)."""
    units, t = [], b
    while t < T_dp:
        units.append((t, 0, G))
        t += P
    n_it = (T - T_dp) * G
    it, end = b * n_it // P, (b + 1) * n_it // P
    while it < end:
        sk, g0 = divmod(it, G)
        g1 = min(G, g0 + end - it)
        units.append((T_dp + sk, g0, g1))
        it += g1 - g0
    return units


def schedule(M, N, K, P0=152):
    G, T = K // 128, N // 128
    if T >= P0:
        rem = T % P0
        T_sk = 0 if rem == 0 else min(T, rem + P0)
        return G, T, T - T_sk, P0
    return G, T, 0, max(1, min(P0, (T * G + 3) // 4))


def run(units, nslot, stages, skip_idle_wait=False, hold=(), seed=0, early_release=False):
    """Returns (deadlocked, list of wrong passes)."""
    rng = random.Random(seed)
    sps = stages // nslot
    ch_len = FOLD * nslot
    bars = {}
    for s in range(stages):
        bars["full", s], bars["empty", s] = Bar(1), Bar(4)
    for j in range(nslot):
        bars["mmadone", j] = Bar(1)
    for b in range(NACC):
        bars["accfull", b], bars["accempty", b] = Bar(nslot), Bar(NEPI)
    chunks, gi = [], 0  # (first group index, length)
    for _, g0, g1 in units:
        for c0 in range(g0, g1, ch_len):
            n = min(ch_len, g1 - c0)
            chunks.append((gi, n))
            gi += n
    place = {g: ((g % nslot) * sps + (g // nslot) % sps, (g // nslot) // sps) for g in range(gi)}
    inflight, issued = [], set()
    content = {}  # stage -> the pair whose bytes it holds (set as a copy lands)

    def producer():
        for g in range(gi):
            s, lap = place[g]
            if lap:
                yield "wait", ("empty", s), lap - 1
            inflight.append((s, g))
            issued.add(g)
            yield "step",

    def slot(j):
        nown = 0
        for ch, (gc0, n) in enumerate(chunks):
            b, lap_b = ch % NACC, ch // NACC
            mine = [gc0 + off for off in range(n) if (gc0 + off) % nslot == j]
            if mine or not skip_idle_wait:
                yield "wait", ("accempty", b), lap_b - 1
            if not mine:
                yield "arrive", ("accfull", b), 1
                continue
            for k, g in enumerate(mine):
                yield "issued", g
                s, lap = place[g]
                if early_release:  # planted: the stage is released before it is read
                    yield "arrive", ("empty", s), 4
                yield "wait", ("full", s), lap
                yield "check", s, g  # the stage still holds this group's bytes when it is read
                yield "wait", ("mmadone", j), nown - 1
                if not early_release:
                    yield "arrive", ("empty", s), 4
                yield "arrive", ("mmadone", j), 1
                if k == len(mine) - 1:
                    yield "arrive", ("accfull", b), 1
                nown += 1

    def epilogue():
        for ch in range(len(chunks)):
            b, lap_b = ch % NACC, ch // NACC
            yield "wait", ("accfull", b), lap_b
            yield "arrive", ("accempty", b), NEPI

    roles = [producer(), epilogue()] + [slot(j) for j in range(nslot)]
    current = [None] * len(roles)
    finished = [False] * len(roles)
    wrong = []
    while not all(finished):
        moved = False
        free = [i for i, (_, g) in enumerate(inflight) if g not in hold]
        if free and rng.random() < 0.5:
            s, k = inflight.pop(free[rng.randrange(len(free))])
            content[s] = k
            bars["full", s].arrive(1)
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
            elif op[0] == "issued":  # the group's copy has been issued (not a move until then)
                if op[1] in issued:
                    current[r], moved = None, True
            elif op[0] == "arrive":
                bars[op[1]].arrive(op[2])
                current[r], moved = None, True
            elif op[0] == "check":
                if content.get(op[1]) != op[2]:
                    wrong.append((("stage", op[1]), op[2], content.get(op[1])))
                current[r], moved = None, True
            elif bars[op[1]].passes(op[2] & 1):  # a wait for phase n tests parity n & 1
                bar = bars[op[1]]
                if bar.done != op[2] + 1:  # passed on a phase other than the one meant
                    wrong.append((op[1], op[2], bar.done))
                current[r], moved = None, True
        if not moved:
            if not inflight:
                return True, wrong
            s, k = inflight.pop(0)  # only held copies are left: land the oldest
            content[s] = k
            bars["full", s].arrive(1)
    return False, wrong


def config(M):
    """(NSLOT, STAGES) of the kernel's configuration for M tokens."""
    bn = 16 if M <= 16 else 32 if M <= 32 else 64
    nslot = 2 if bn == 64 else 4
    b_bytes = bn * 128 * 2
    fit = (227 * 1024 - 2048 - nslot * b_bytes) // 8448
    return nslot, min(fit, 24) // nslot * nslot


@pytest.mark.parametrize("M,N,K", [(16, 12288, 4096), (40, 1664, 1152), (64, 22016, 4096), (16, 19456, 8192),
                                   (1, 384, 1152), (32, 1280, 384), (16, 4096, 14336)])
def test_protocol_has_no_wrong_pass_and_no_deadlock(M, N, K):
    nslot, stages = config(M)
    G, T, T_dp, P = schedule(M, N, K)
    for b in sorted({0, 1, P // 2, P - 1} | set(range(0, P, max(1, P // 12)))):
        units = cta_units(b, P, T, G, T_dp)
        ngroups = sum(g1 - g0 for _, g0, g1 in units)
        for seed, hold in [(0, ()), (1, ())] + [(2, (h,)) for h in range(min(ngroups, 8))]:
            dead, wrong = run(units, nslot, stages, hold=hold, seed=seed)
            assert not dead, f"CTA {b} units {units} hold {hold}: deadlock"
            assert not wrong, f"CTA {b} units {units} hold {hold}: {wrong[:3]}"


def test_model_catches_a_skipped_accumulator_wait():
    """One-group units: each chunk has one group, so a slot is idle in three
    of every four chunks.  A slot that skipped the accumulator wait in its idle
    chunks would wait a lap ahead on an accumulator buffer when it next has a
    group, and pass early while the epilogue is still behind."""
    nslot, stages = config(16)
    units = [(t, 0, 1) for t in range(12)]
    found = any(run(units, nslot, stages, skip_idle_wait=True, hold=(h,), seed=s)[1]
                for s in range(8) for h in range(6))
    assert found
    assert not any(run(units, nslot, stages, hold=(h,), seed=s)[1] for s in range(8) for h in range(6))


def test_model_catches_a_stage_released_before_it_is_read():
    """A slot that released a stage before reading it would let the producer
    refill the stage under it: the model must see the stage holding another
    group's bytes when the slot reads it."""
    nslot, stages = config(16)
    units = [(0, 0, 32), (1, 0, 32)]
    found = False
    for s in range(8):
        for h in range(6):
            dead, wrong = run(units, nslot, stages, hold=(h,), seed=s, early_release=True)
            found |= dead or bool(wrong)
    assert found
    assert not any(run(units, nslot, stages, hold=(h,), seed=s)[1] for s in range(8) for h in range(6))


def sk_cta_of(it, P, I):
    """The CTA whose stream-K range holds group iteration it (the kernel's
    formula: CTA b's range is [floor(b I / P), floor((b + 1) I / P)))."""
    return ((it + 1) * P - 1) // I


@pytest.mark.parametrize("M,N,K", [(16, 12288, 4096), (16, 4096, 14336), (64, 22016, 4096), (1, 384, 1152),
                                   (40, 1664, 1152), (16, 19456, 8192), (8, 256, 512), (32, 128, 131072),
                                   (16, 38912, 4096)])
def test_stream_k_schedule_and_hand_off(M, N, K):
    """The decode kernel's work split covers every (tile, group) exactly once;
    a split tile's owner is the CTA holding its group 0, that part is the
    owner's last unit, and the CTAs it gathers from (blockIdx + 1 .. the CTA of
    the tile's last group) are exactly the other holders, each holding one
    part of the tile as a unit of its own; every such part is either the
    first unit of its CTA or that CTA's only unit, and no CTA holds two (one
    split-K slot per CTA)."""
    G, T, T_dp, P = schedule(M, N, K)
    seen = {}
    units_of = {b: cta_units(b, P, T, G, T_dp) for b in range(P)}
    for b, units in units_of.items():
        assert sum(1 for _, g0, _ in units if g0 > 0) <= 1
        for t, g0, g1 in units:
            assert 0 <= g0 < g1 <= G
            for g in range(g0, g1):
                assert (t, g) not in seen
                seen[t, g] = b
    assert len(seen) == T * G
    I = (T - T_dp) * G
    for t in range(T_dp, T):
        holders = sorted({seen[t, g] for g in range(G)})
        owner = seen[t, 0]
        if len(holders) == 1:
            continue
        assert units_of[owner][-1] == (t, 0, units_of[owner][-1][2])  # the owner's last unit
        b1 = sk_cta_of((t - T_dp) * G + G - 1, P, I)
        assert holders == list(range(owner, b1 + 1))
        for c in holders[1:]:
            parts = [u for u in units_of[c] if u[0] == t]
            assert len(parts) == 1 and parts[0][1] > 0
            assert units_of[c][0] == parts[0] or len(units_of[c]) == 1
