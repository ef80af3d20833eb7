"""Model check of the tensor-core GEMM's shared-memory ring protocol (k_gemm_tc.cu), on the CPU.

compute-sanitizer's race checks are not available for this kernel's GPU, so the protocol is checked
as a model: for each CTA of a cluster, the producer warp (raw weight boxes by TMA), the activation
loader (its share of every activation tile, multicast to all CTAs of the cluster), the MMA issuer
(whose commits free the activation slot in every CTA) and the 8 dequantising warps run as
coroutines over the kernel's loop structure, slot indices and barrier parities, with mbarriers
modelled by their phase, arrival and transaction counts (try_wait.parity p succeeds once the phase
of parity p has completed) and every copy and MMA completing after a random delay. For every ring
depth the kernel instantiates, with clusters of one and two CTAs, all K steps must finish without
a deadlock, every read must see the data of its own K step (every share of the activation tile),
and no slot may be overwritten while the MMAs of any CTA still read it.
"""
import random

import pytest


class Bar:
    """An mbarrier: `count` arrivals (and the expected transaction bytes) complete a phase."""

    def __init__(self, count):
        self.count, self.pending, self.tx, self.phase = count, count, 0, 0

    def arrive(self):
        self.pending -= 1
        self._check()

    def expect_tx(self, n):
        self.tx += n
        self.pending -= 1
        self._check()

    def complete_tx(self, n):
        self.tx -= n
        self._check()

    def _check(self):
        # the transaction count may go below zero for a while (a peer's multicast share can land
        # before this CTA's loader announced the step's bytes); arrivals may not
        assert self.pending >= 0, "barrier over-arrived"
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        return (self.phase & 1) != parity


def run(SA, SB, SR, nk, seed, CL=2, drop_loader_wait=False):
    """One cluster of CL CTAs running the K loop. Per CTA: SR raw-box slots (freed by the
    dequantising warps), SA dequantised-tile slots, SB activation slots. The activation tile of a
    step is loaded in CL shares, one by each CTA's loader, each share multicast to every CTA of the
    cluster; a CTA's activation slot is free once the MMAs of every CTA have read it (their commits
    arrive on every CTA's empty barrier)."""
    rnd = random.Random(seed)
    events, now = [], [0]

    def later(fn, lo, hi):
        events.append((now[0] + rnd.randint(lo, hi), fn))

    class Cta:
        def __init__(self):
            self.full_w = [Bar(1) for _ in range(SR)]
            self.empty_w = [Bar(8) for _ in range(SR)]
            self.full_b = [Bar(1) for _ in range(SB)]
            self.empty_b = [Bar(CL) for _ in range(SB)]
            self.full_a = [Bar(8) for _ in range(SA)]
            self.empty_a = [Bar(1) for _ in range(SA)]
            self.raw = [None] * SR
            self.shares = [dict() for _ in range(SB)]     # slot -> {share: step} landed
            self.atile = [[None] * 8 for _ in range(SA)]
            self.raw_readers = [set() for _ in range(SR)]
            self.reading_b, self.reading_a = set(), set()

    ctas = [Cta() for _ in range(CL)]

    def producer(c):
        C = ctas[c]

        def issue(j):
            s = j % SR
            assert not C.raw_readers[s], ("raw box overwritten before every warp read it", j)
            C.full_w[s].expect_tx(1)

            def land(s=s, j=j):
                C.raw[s] = j
                C.raw_readers[s] = set(range(8))
                C.full_w[s].complete_tx(1)
            later(land, 5, 60)
        for j in range(min(nk, SR)):
            issue(j)
        for j in range(SR, nk):
            while not C.empty_w[j % SR].done(((j // SR) - 1) & 1):
                yield
            issue(j)

    def loader(c):
        C = ctas[c]
        for j in range(nk):
            s = j % SB
            if j >= SB and not drop_loader_wait:
                while not C.empty_b[s].done(((j // SB) - 1) & 1):
                    yield
            C.full_b[s].expect_tx(CL)            # the whole tile: CL shares
            for d in range(CL):                  # this CTA's share, multicast to every CTA
                D = ctas[d]
                assert s not in D.reading_b, ("activation slot overwritten while an MMA reads it", j, d)

                def land(D=D, s=s, j=j, c=c):
                    D.shares[s][c] = j
                    D.full_b[s].complete_tx(1)
                later(land, 2, 50)
            yield

    def mma(c):
        C = ctas[c]
        for j in range(nk):
            s, a = j % SB, j % SA
            while not (C.full_a[a].done((j // SA) & 1) and C.full_b[s].done((j // SB) & 1)):
                yield
            assert all(C.shares[s].get(d) == j for d in range(CL)), ("activation tile", j, C.shares[s])
            assert all(t == j for t in C.atile[a]), ("dequantised tile", j)
            C.reading_b.add(s)
            C.reading_a.add(a)

            def finish(s=s, a=a):
                C.reading_b.discard(s)
                C.reading_a.discard(a)
                for D in ctas:                    # the commit arrives on every CTA's empty barrier
                    D.empty_b[s].arrive()
                C.empty_a[a].arrive()
            later(finish, 3, 30)
            yield

    def warp(c, w):
        C = ctas[c]
        for j in range(nk):
            r, a = j % SR, j % SA
            while not C.full_w[r].done((j // SR) & 1):
                yield
            if j >= SA:
                while not C.empty_a[a].done(((j // SA) - 1) & 1):
                    yield
            assert C.raw[r] == j, ("raw box", j)
            assert a not in C.reading_a, ("dequantised tile overwritten while an MMA reads it", j)
            C.atile[a][w] = j
            C.raw_readers[r].discard(w)
            yield
            C.full_a[a].arrive()
            C.empty_w[r].arrive()

    agents = []
    for c in range(CL):
        agents += [producer(c), loader(c), mma(c)] + [warp(c, w) for w in range(8)]
    alive = [True] * len(agents)
    for _ in range(400000):
        if not any(alive):
            return
        events.sort(key=lambda e: e[0])
        while events and events[0][0] <= now[0]:
            events.pop(0)[1]()
        order = list(range(len(agents)))
        rnd.shuffle(order)
        for i in order:
            if alive[i]:
                try:
                    next(agents[i])
                except StopIteration:
                    alive[i] = False
        now[0] += 1
    raise AssertionError("deadlock")


def ring_depths(qb_bytes, bn, mt):
    """(SA, SB, SR) as the kernel's Cfg<QT, BN, MT> computes them."""
    q4 = qb_bytes == 16
    a_bytes = mt * 128 * 64 * 2
    b_bytes = 2 * bn * 64 * 2
    rq_slot = (mt * 32 * (8 * qb_bytes + 16) + 1023) // 1024 * 1024
    sa = 3 if mt == 2 and q4 and bn == 64 else 2
    sr = 2 if mt == 2 and not q4 and bn == 128 else 3
    sb = min(6, (220 * 1024 - sa * a_bytes - sr * rq_slot) // b_bytes)
    assert sb >= 2
    assert sa * a_bytes + sb * b_bytes + sr * rq_slot + 1024 + 512 <= 227 * 1024
    return sa, sb, sr


# every tile shape the launcher picks from (BN tokens x MT weight tiles), for Q4_0 and Q8_0
SHAPES = [(qb, bn, mt) for qb in (16, 32) for bn, mt in ((64, 1), (64, 2), (128, 1), (128, 2), (256, 1))]


@pytest.mark.parametrize("qb_bytes,bn,mt", SHAPES)
@pytest.mark.parametrize("CL", [1, 2])
def test_ring_protocol(qb_bytes, bn, mt, CL):
    SA, SB, SR = ring_depths(qb_bytes, bn, mt)
    for nk in (1, 2, 3, 5, 7, 40):
        for seed in range(2):
            run(SA, SB, SR, nk, seed, CL=CL)


def test_model_catches_a_missing_wait():
    """The check is not vacuous: dropping the dequantising warps' wait for a free tile slot races."""
    import inspect
    src = inspect.getsource(run).replace("while not C.empty_a[a].done(((j // SA) - 1) & 1):", "while False:")
    ns = {"random": random, "Bar": Bar}
    exec(compile(src, "mutated", "exec"), ns)
    with pytest.raises(AssertionError):
        for seed in range(5):
            ns["run"](3, 6, 3, 40, seed)


def test_model_catches_a_loader_that_does_not_wait_for_the_cluster():
    """A loader that reuses an activation slot without waiting for every CTA's MMAs overwrites a
    tile a peer still reads."""
    with pytest.raises(AssertionError):
        for seed in range(20):
            run(2, 2, 3, 40, seed, CL=2, drop_loader_wait=True)
