"""Model check, on the CPU, of the persistent decode step's in-CTA barrier protocol for the
weight-streaming phases (step_gemv in k_decode_step.cuh).

In each phase a CTA consumes its stages in pairs. All 8 warps compute both stages' dot products
into part[q] (q = pair & 1); one warp -- the pair's epilogue warp, rotating over the 8 warps --
then reads part[q] for the epilogues while the others go on. Hardware named barriers (which never
time out) order this:
  DONE(q): the epilogue warp and the feeding warp (warp 7) wait, the others only arrive;
  FREE(q): the epilogue warp arrives after reading part[q]; the other warps wait for that two
           pairs later, before they write part[q] again;
and at the end of the phase the FREE arrivals of the last two pairs are taken, then the whole
CTA meets. The warps are modelled as coroutines with random interleavings, over sequences of
phases of 0 to 9 pairs, and the test checks: no deadlock (a hang of real hardware), every
barrier generation holds arrivals of one pair only, part[q] holds exactly the pair an epilogue
reads (all 8 warps' products, not yet overwritten), the ring slots of a pair are refilled only
after every warp has read them, and every barrier is balanced when a phase ends. Planted
mistakes in the protocol are caught."""
import random

import pytest

N_WARPS = 8
FEED_WARP = 7
THREADS = 256


class Deadlock(Exception):
    pass


class Barriers:
    """bar.sync / bar.arrive over 256 threads: a generation completes when 8 warps have arrived."""

    def __init__(self):
        self.count = {}
        self.tag = {}
        self.gen = {}

    def arrive(self, bid, tag):
        c = self.count.get(bid, 0)
        if c == 0:
            self.tag[bid] = tag
        assert self.tag[bid] == tag, f"barrier {bid}: arrival for pair {tag} joins pair {self.tag[bid]}'s generation"
        c += 32
        if c == THREADS:
            self.count[bid] = 0
            self.gen[bid] = self.gen.get(bid, 0) + 1
        else:
            self.count[bid] = c
        return self.gen.get(bid, 0)

    def balanced(self):
        return all(c == 0 for c in self.count.values())


def warp_program(w, phases, st, mistake):
    """One warp's sequence of actions; yields ('sync', bid, tag) / ('arrive', bid, tag) / ('act', fn)."""
    for ph, n_pairs in enumerate(phases):
        for bi in range(n_pairs):
            q = bi & 1
            epi = w == (bi & (N_WARPS - 1)) if mistake != "two_epi_warps" else (w >> 1) == (bi & 3)
            was = bi >= 2 and (w == ((bi - 2) & (N_WARPS - 1)) if mistake != "two_epi_warps"
                               else (w >> 1) == ((bi - 2) & 3))
            if bi >= 2 and not was and mistake != "no_free_wait":
                yield ("sync", 4 + q, (ph, bi - 2))
            yield ("act", lambda w=w, ph=ph, bi=bi, q=q: st.write(w, ph, bi, q))
            if mistake == "epi_arrives_done" and epi:
                yield ("arrive", 2 + q, (ph, bi))
            elif epi or w == FEED_WARP:
                yield ("sync", 2 + q, (ph, bi))
            else:
                yield ("arrive", 2 + q, (ph, bi))
            if epi:
                yield ("act", lambda w=w, ph=ph, bi=bi, q=q: st.read(w, ph, bi, q))
                yield ("arrive", 4 + q, (ph, bi))
            if w == FEED_WARP:
                yield ("act", lambda ph=ph, bi=bi: st.refill(ph, bi))
        ends = range(max(0, n_pairs - 2), n_pairs) if mistake != "no_balance" else range(0)
        for j in ends:
            if (w != (j & (N_WARPS - 1))) if mistake != "two_epi_warps" else ((w >> 1) != (j & 3)):
                yield ("sync", 4 + (j & 1), (ph, j))
        yield ("sync", 1, (ph, "end"))
        yield ("act", lambda ph=ph: st.phase_end(ph))


class State:
    def __init__(self, bars):
        self.part = {0: {}, 1: {}}     # q -> {warp: (phase, pair)}
        self.read_pair = set()        # dots done: (phase, pair, warp)
        self.readers = {}             # (phase, pair) -> warps whose epilogue read is done
        self.two = False
        self.bars = bars

    def write(self, w, ph, bi, q):
        # the pair two back (same buffer) must have been read by its epilogue warp(s) already
        for (oph, obi) in set(self.part[q].values()):
            if (oph, obi) != (ph, bi) and not self.readers.get((oph, obi), set()) >= self.expected_readers(obi):
                raise AssertionError(f"warp {w} overwrites part[{q}] of pair {(oph, obi)} before its epilogue read it")
        self.part[q][w] = (ph, bi)
        self.read_pair.add((ph, bi, w))

    def expected_readers(self, bi):
        return {bi & (N_WARPS - 1)} if not self.two else {2 * (bi & 3), 2 * (bi & 3) + 1}

    def read(self, w, ph, bi, q):
        got = self.part[q]
        assert len(got) == N_WARPS and all(v == (ph, bi) for v in got.values()), \
            f"epilogue of pair {(ph, bi)} reads part[{q}] = {got}"
        self.readers.setdefault((ph, bi), set()).add(w)

    def refill(self, ph, bi):
        for w in range(N_WARPS):
            assert (ph, bi, w) in self.read_pair, f"slots of pair {(ph, bi)} refilled before warp {w} read them"

    def phase_end(self, ph):
        pass


def run(phases, seed, mistake=None):
    rng = random.Random(seed)
    bars = Barriers()
    st = State(bars)
    st.two = mistake == "two_epi_warps"
    progs = [warp_program(w, phases, st, mistake) for w in range(N_WARPS)]
    waiting = {}                     # warp -> (bid, gen it waits to complete)
    done = [False] * N_WARPS
    def step(w):
        if w in waiting:
            bid, g = waiting[w]
            if bars.gen.get(bid, 0) > g:
                del waiting[w]
            else:
                return False
        act = next(progs[w], None)
        if act is None:
            done[w] = True
            return True
        kind = act[0]
        if kind == "act":
            fn = act[1]
            fn()
            return True
        bid, tag = act[1], act[2]
        g_before = bars.gen.get(bid, 0)
        bars.arrive(bid, tag)
        if kind == "arrive":
            return True
        if bars.gen.get(bid, 0) == g_before:   # not complete yet: wait for this generation
            waiting[w] = (bid, g_before)
        return True

    guard = 0
    while not all(done):
        guard += 1
        assert guard < 10 ** 6
        live = [w for w in range(N_WARPS) if not done[w]]
        rng.shuffle(live)
        progressed = False
        for w in live[: rng.randint(1, len(live))]:
            if step(w):
                progressed = True
        if not progressed:
            # nobody in the chosen subset could move; try everyone before declaring a deadlock
            if not any(step(w) for w in live):
                raise Deadlock(f"all live warps blocked: {waiting}")
    assert bars.balanced(), bars.count
    return True


PHASE_SEQS = [[0, 1, 2, 3], [4, 5, 6, 7, 8, 9], [3, 0, 2, 1, 9, 4], [2, 2, 2], [1, 1, 1, 1, 5], [9, 9]]


@pytest.mark.parametrize("seq", PHASE_SEQS)
def test_protocol_holds(seq):
    for seed in range(40):
        run(seq, seed)


@pytest.mark.parametrize("mistake,err", [("no_free_wait", AssertionError), ("no_balance", (AssertionError, Deadlock)),
                                         ("epi_arrives_done", AssertionError),
                                         # two epilogue warps per pair that skip the FREE wait as a
                                         # pair: one may overwrite what its partner still reads
                                         ("two_epi_warps", AssertionError)])
def test_planted_mistakes_are_caught(mistake, err):
    caught = False
    for seed in range(200):
        try:
            run([5, 6, 3], seed, mistake)
        except err:
            caught = True
            break
    assert caught, mistake
