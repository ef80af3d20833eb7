"""Model check of the tensor-core GEMM's shared-memory ring protocol (k_gemm_tc.cu), on the CPU.

compute-sanitizer's race checks are not available for this kernel's GPU, so the protocol is checked
as a model: the producer warp (raw weight boxes by TMA), the MMA issuer and the 8 dequantising /
activation-loading warps run as coroutines over the kernel's loop structure, slot indices and
barrier parities, with mbarriers modelled by their phase and arrival counts (try_wait.parity p
succeeds once the phase of parity p has completed) and every copy and MMA completing after a random
delay. For every ring depth the kernel instantiates, all K steps must finish without a deadlock,
every read must see the data of its own K step, and no slot may be overwritten while the MMAs of an
earlier step still read it.
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
        assert self.pending >= 0 and self.tx >= 0, "barrier over-arrived"
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        return (self.phase & 1) != parity


def run(SA, SB, SR, D, nk, seed):
    """One CTA's K loop: SR raw-box slots (freed by the dequantising warps), SB activation slots
    (freed by the MMA commit), SA dequantised-tile slots, activations D steps ahead."""
    rnd = random.Random(seed)
    full_w = [Bar(1) for _ in range(SR)]
    empty_w = [Bar(8) for _ in range(SR)]
    full_b = [Bar(8) for _ in range(SB)]
    empty_b = [Bar(1) for _ in range(SB)]
    full_a = [Bar(8) for _ in range(SA)]
    empty_a = [Bar(1) for _ in range(SA)]
    raw = [None] * SR                                  # step whose raw box a slot holds
    rows = [[None] * SB for _ in range(8)]             # step whose activation rows warp w put in a slot
    atile = [[None] * 8 for _ in range(SA)]            # step whose tile rows warp w dequantised
    raw_readers = [set() for _ in range(SR)]           # warps that still have to read a raw box
    reading_b, reading_a = set(), set()                # slots an MMA in flight reads
    events, now = [], [0]

    def later(fn, lo, hi):
        events.append((now[0] + rnd.randint(lo, hi), fn))

    def producer():
        def issue(j):
            s = j % SR
            assert not raw_readers[s], ("raw box overwritten before every warp read it", j)
            full_w[s].expect_tx(1)

            def land(s=s, j=j):
                raw[s] = j
                raw_readers[s] = set(range(8))
                full_w[s].complete_tx(1)
            later(land, 5, 60)
        for j in range(min(nk, SR)):
            issue(j)
        for j in range(SR, nk):
            while not empty_w[j % SR].done(((j // SR) - 1) & 1):
                yield
            issue(j)

    def mma():
        for j in range(nk):
            s, a = j % SB, j % SA
            while not (full_a[a].done((j // SA) & 1) and full_b[s].done((j // SB) & 1)):
                yield
            assert all(rows[w][s] == j for w in range(8)), ("activation tile", j)
            assert all(t == j for t in atile[a]), ("dequantised tile", j)
            reading_b.add(s)
            reading_a.add(a)

            def finish(s=s, a=a):
                reading_b.discard(s)
                reading_a.discard(a)
                empty_b[s].arrive()
                empty_a[a].arrive()
            later(finish, 3, 30)
            yield

    def warp(w):
        groups = []                                    # committed cp.async groups: landing flags

        def load_act(j):
            assert j % SB not in reading_b, ("activation slot overwritten while an MMA reads it", j)
            flag = {"landed": False}

            def land(s=j % SB, j=j, flag=flag):
                rows[w][s] = j
                flag["landed"] = True
            later(land, 2, 50)
            return [flag]
        for j in range(D):
            groups.append(load_act(j) if j < nk else [])
        for j in range(nk):
            r, b, a = j % SR, j % SB, j % SA
            while not full_w[r].done((j // SR) & 1):
                yield
            if j >= SA:
                while not empty_a[a].done(((j // SA) - 1) & 1):
                    yield
            assert raw[r] == j, ("raw box", j)
            assert a not in reading_a, ("dequantised tile overwritten while an MMA reads it", j)
            atile[a][w] = j
            raw_readers[r].discard(w)
            yield
            full_a[a].arrive()
            empty_w[r].arrive()
            while not all(f["landed"] for g in groups[:len(groups) - (D - 1)] for f in g):
                yield                                  # cp.async.wait_group D - 1
            full_b[b].arrive()
            jn = j + D
            g = []
            if jn < nk:
                if jn >= SB:
                    while not empty_b[jn % SB].done(((jn // SB) - 1) & 1):
                        yield
                g = load_act(jn)
            groups.append(g)

    agents = [producer(), mma()] + [warp(w) for w in range(8)]
    alive = [True] * len(agents)
    for _ in range(200000):
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
    """(SA, SB, SR, DB) as the kernel's Cfg<QT, BN, MT> computes them."""
    q4 = qb_bytes == 16
    a_bytes = mt * 128 * 64 * 2
    b_bytes = 2 * bn * 64 * 2
    rq_slot = (mt * 32 * (8 * qb_bytes + 16) + 1023) // 1024 * 1024
    sa = 3 if mt == 2 and q4 and bn == 64 else 2
    sr = 2 if mt == 2 and not q4 and bn == 128 else 3
    sb = min(6, (220 * 1024 - sa * a_bytes - sr * rq_slot) // b_bytes)
    db = sb - sa if sb - sa >= 2 else sb - 1
    assert sb >= 2 and db >= 1
    assert sa * a_bytes + sb * b_bytes + sr * rq_slot + 1024 + 512 <= 227 * 1024
    return sa, sb, sr, db


# every tile shape the launcher picks from (BN tokens x MT weight tiles), for Q4_0 and Q8_0
SHAPES = [(qb, bn, mt) for qb in (16, 32) for bn, mt in ((64, 1), (64, 2), (128, 1), (128, 2), (256, 1))]


@pytest.mark.parametrize("qb_bytes,bn,mt", SHAPES)
def test_ring_protocol(qb_bytes, bn, mt):
    SA, SB, SR, DB = ring_depths(qb_bytes, bn, mt)
    for nk in (1, 2, 3, 5, 7, 64):
        for seed in range(3):
            run(SA, SB, SR, DB, nk, seed)


def test_model_catches_a_missing_wait():
    """The check is not vacuous: dropping the dequantising warps' wait for a free tile slot races."""
    import inspect
    src = inspect.getsource(run).replace("while not empty_a[a].done(((j // SA) - 1) & 1):", "while False:")
    ns = {"random": random, "Bar": Bar}
    exec(compile(src, "mutated", "exec"), ns)
    with pytest.raises(AssertionError):
        for seed in range(5):
            ns["run"](3, 6, 3, 3, 64, seed)
