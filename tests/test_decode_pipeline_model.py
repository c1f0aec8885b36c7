"""Barrier protocol of the decode GEMM kernel (csrc/gemm_decode.cu), checked on
a model (CPU).

The kernel's roles hand work to each other through mbarriers whose waits test
only the parity of a phase, so a wait is right only if it starts after the
phase before the one it wants has completed, and before the phase after it
can complete.  The model runs each role as a sequence of waits and arrivals,
exactly as the kernel orders them, under adversarial scheduling (some copies
land only when nothing else can move), and counts phases exactly:

Each wait names the phase it means (n, counted from 0; -1 for "none yet")
and tests its parity n & 1, which is what the kernel's parity expressions
evaluate to.

  * producer: per group one copy into the owning slot's sub-ring of weight
    stages; from the second lap on it first waits for the stage's release;
  * dequant slot j: the groups at batch positions t = j (mod NSLOT) in each
    unit, plus the empty second place of a one-group batch it owns (a dummy
    that only waits for the A buffer and arrives); per group: wait for the
    stage, release it, wait for the A buffer, arrive on the batch;
  * MMA warp: per fold chunk of 8 groups it waits for an accumulator, per
    batch of two groups for the batch, then commits the A buffer, and at the
    chunk's end the accumulator;
  * epilogue: waits for each chunk's accumulator and releases it.

Every parity wait must pass exactly on the phase it means, and no schedule may
deadlock.  The same model with the earlier protocol (one ring shared by all
slots; a one-group batch's slot arriving twice instead of a dummy) shows a
wait passing a lap early, which is the race that protocol had on the GPU.
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


def run(units, nslot, stages, nbatch, old=False, hold=(), seed=0):
    """Returns (deadlocked, list of wrong passes)."""
    rng = random.Random(seed)
    sps = stages // nslot
    bars = {}
    for s in range(stages):
        bars["full", s], bars["empty", s] = Bar(1), Bar(4)
    for a in range(nbatch):
        bars["afull", a], bars["aempty", a] = Bar(8), Bar(1)
    for b in range(NACC):
        bars["accfull", b], bars["accempty", b] = Bar(1), Bar(NEPI)
    entries, t0, gi = [], 0, 0  # (t, gi or None for a dummy, nb)
    for _, g0, g1 in units:
        n = g1 - g0
        for off in range(n + n % 2):
            pos = off & 1
            real = off < n
            entries.append(dict(t=t0 + off, gi=gi if real else None, nb=min(2, n - (off - pos))))
            gi += real
        t0 += n + n % 2
    real = [e for e in entries if e["gi"] is not None]
    place = {}  # gi -> (stage, lap)
    count = [0] * nslot
    for e in real:
        j = e["t"] % nslot
        if old:
            place[e["gi"]] = (e["gi"] % stages, e["gi"] // stages)
        else:
            place[e["gi"]] = (j * sps + count[j] % sps, count[j] // sps)
        count[j] += 1
    inflight, issued = [], set()

    def producer():
        for e in real:
            s, lap = place[e["gi"]]
            if lap:
                yield "wait", ("empty", s), lap - 1
            inflight.append((s, e["gi"]))
            issued.add(e["gi"])
            yield "step",

    def slot(j):
        for e in entries:
            if e["t"] % nslot != j or (old and e["gi"] is None):
                continue
            bi = e["t"] >> 1
            a, lap_a = bi % nbatch, bi // nbatch
            if e["gi"] is not None:
                yield "issued", e["gi"]
                s, lap = place[e["gi"]]
                yield "wait", ("full", s), lap
                yield "arrive", ("empty", s), 4
            yield "wait", ("aempty", a), lap_a - 1
            yield "arrive", ("afull", a), 8 if (old and e["nb"] == 1) else 4

    def mma():
        bi = chunk = 0
        for _, g0, g1 in units:
            for c0 in range(g0, g1, FOLD):
                b, lap_b = chunk % NACC, chunk // NACC
                yield "wait", ("accempty", b), lap_b - 1
                for _ in range(c0, min(g1, c0 + FOLD), 2):
                    yield "wait", ("afull", bi % nbatch), bi // nbatch
                    yield "arrive", ("aempty", bi % nbatch), 1
                    bi += 1
                yield "arrive", ("accfull", b), 1
                chunk += 1

    def epilogue():
        chunk = 0
        for _, g0, g1 in units:
            for _ in range(g0, g1, FOLD):
                b, lap_b = chunk % NACC, chunk // NACC
                yield "wait", ("accfull", b), lap_b
                yield "arrive", ("accempty", b), NEPI
                chunk += 1

    roles = [producer(), mma(), epilogue()] + [slot(j) for j in range(nslot)]
    current = [None] * len(roles)
    finished = [False] * len(roles)
    wrong = []
    while not all(finished):
        moved = False
        free = [i for i, (_, g) in enumerate(inflight) if g not in hold]
        if free and rng.random() < 0.5:
            s, _ = inflight.pop(free[rng.randrange(len(free))])
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
            elif bars[op[1]].passes(op[2] & 1):  # a wait for phase n tests parity n & 1
                bar = bars[op[1]]
                if bar.done != op[2] + 1:  # passed on a phase other than the one meant
                    wrong.append((op[1], op[2], bar.done))
                current[r], moved = None, True
        if not moved:
            if not inflight:
                return True, wrong
            s, _ = inflight.pop(0)  # only held copies are left: land the oldest
            bars["full", s].arrive(1)
    return False, wrong


def config(M):
    bn = 16 if M <= 16 else 32 if M <= 32 else 64
    nslot = 2 if bn == 64 else 4
    stages = 16 if bn < 64 else 15
    nbatch = (512 - (2 * bn + 63) // 64 * 64) // 128
    return nslot, stages - stages % nslot, nbatch


@pytest.mark.parametrize("M,N,K", [(16, 12288, 4096), (40, 1664, 1152), (64, 22016, 4096), (16, 19456, 8192),
                                   (1, 384, 1152), (32, 1280, 384)])
def test_protocol_has_no_wrong_pass_and_no_deadlock(M, N, K):
    nslot, stages, nbatch = config(M)
    G, T, T_dp, P = schedule(M, N, K)
    for b in sorted({0, 1, P // 2, P - 1} | set(range(0, P, max(1, P // 12)))):
        units = cta_units(b, P, T, G, T_dp)
        ngroups = sum(g1 - g0 for _, g0, g1 in units)
        for seed, hold in [(0, ()), (1, ())] + [(2, (h,)) for h in range(min(ngroups, 8))]:
            dead, wrong = run(units, nslot, stages, nbatch, hold=hold, seed=seed)
            assert not dead, f"CTA {b} units {units} hold {hold}: deadlock"
            assert not wrong, f"CTA {b} units {units} hold {hold}: {wrong[:3]}"


def test_model_catches_the_earlier_protocol():
    """A CTA of the 16 x 12288 x 4096 decode schedule whose range is two
    odd-length units (groups 23..31 of one tile, 0..10 of the next): with one
    ring shared by the slots and a double arrival for one-group batches, a
    copy that lands late lets a slot's waits pass a lap early."""
    nslot, stages, nbatch = config(16)
    G, T, T_dp, P = schedule(16, 12288, 4096)
    units = cta_units(17, P, T, G, T_dp)
    assert [(g0, g1) for _, g0, g1 in units] == [(23, 32), (0, 11)]
    found = any(run(units, nslot, stages, nbatch, old=True, hold=(0,), seed=s)[1] for s in range(4))
    assert found
    assert not any(run(units, nslot, stages, nbatch, hold=(0,), seed=s)[1] for s in range(4))
