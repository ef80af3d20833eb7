"""Model check of the persistent decode step's synchronisation (k_decode_step.cuh), on the CPU.

The step is the one kernel whose CTAs wait on one another, so its protocol is checked as a model:
each CTA runs as a coroutine over the kernel's flow -- the stage ring filled at launch and refilled
after every consumed pair (slot k % slots, barrier parity (k / slots) & 1), the grid barriers
(a monotonic arrival counter), the per-KV-head counters each CTA publishes its QKV quads on
after its last QKV stage and the attention units wait for, the split merge by the last unit of a head (an arrival counter), and
the reset by the last CTA to finish -- with every bulk copy landing after a random delay and the
CTAs scheduled in random order. Over two launches in a row it checks that every consumed slot
holds the stage the consumer expects and none is refilled early, that each phase's input is
complete when it is staged and no buffer is overwritten while a CTA still has to read it, that a
unit starts only when its head's q, k and v rows are all written and a merge sees every split,
and that the counters are zero again for the next launch.
"""
import random

import pytest


class Bar:
    def __init__(self):
        self.phase, self.pending = 0, None

    def arm(self):                      # arrive.expect_tx by the feeding thread
        assert self.pending is None, "slot armed twice"
        self.pending = True

    def land(self):                     # the bulk copy's bytes complete the phase
        self.pending = None
        self.phase += 1

    def done(self, parity):
        return (self.phase & 1) != parity


def model(grid, slots, L, H, KV, hd, d, F, V, tps, ns, n_out, seed, launches=2):
    rnd = random.Random(seed)
    qw, kw = H * hd, KV * hd
    G = H // KV
    kvh_quads = (G + 2) * hd // 4
    # phases: per layer QKV, O, gate/up, down; then the head. stages = ceil(tasks / tps)
    tasks = [(qw + 2 * kw) // 4, d // 4, (F + 1) // 2, d // 4]
    n_st = []
    for _ in range(L):
        n_st += [-(-t // tps[i]) for i, t in enumerate(tasks)]
    n_st.append(-(-(V // 4) // tps[0]))
    n_ph = 4 * L + (1 if n_out else 0)

    def kvh_of(r0):                     # KV head of QKV row quad r0 (as the epilogue publishes it)
        if r0 < qw:
            return (r0 // hd) // G
        return ((r0 - qw) // hd) % KV

    shared = {"bar0": 0, "bar1": 0, "cnt": [0] * KV, "att": [0] * KV}
    events, now = [], [0]

    def later(fn):
        events.append((now[0] + rnd.randint(1, 30), fn))

    for launch in range(launches):
        assert shared["bar0"] == 0 and shared["bar1"] == 0 and shared["cnt"] == [0] * KV and shared["att"] == [0] * KV
        # what each phase wrote: epilogue completions per phase, per head quads of layer l,
        # staging completions per phase, the attention partials and merges
        written = [0] * (4 * L + 1)
        staged = [0] * (4 * L + 1)
        quads = [[0] * KV for _ in range(L)]
        partial = {}
        merged = {(l, h): False for l in range(L) for h in range(KV)}
        units = KV * ns

        def cta(c):
            n_bar = [0]                                             # this CTA's barriers so far
            full = [Bar() for _ in range(slots)]
            ring = [None] * slots
            consumed = set()
            cur = {"ph": 0, "st": c, "issued": 0}

            def feed_one():
                while cur["ph"] < n_ph and cur["st"] >= n_st[cur["ph"]]:
                    cur["ph"] += 1
                    cur["st"] = c
                if cur["ph"] >= n_ph:
                    return
                slot = cur["issued"] % slots
                assert ring[slot] is None or ring[slot] in consumed, ("slot refilled before it was used", c)
                full[slot].arm()
                tag = (cur["ph"], cur["st"])

                def land(slot=slot, tag=tag):
                    ring[slot] = tag
                    full[slot].land()
                later(land)
                cur["st"] += grid
                cur["issued"] += 1

            def grid_sync():
                n_bar[0] += 1
                shared["bar0"] += 1
                target = n_bar[0] * grid
                while shared["bar0"] < target:
                    yield

            k = [0]
            pub = [0] * KV                                          # quads not yet published

            def gemv(ph, prev_done):
                assert prev_done(), ("phase input incomplete when staged", ph, c)
                staged[ph] += 1
                yield
                st = c
                while st < n_st[ph]:
                    st2 = st + grid
                    two = st2 < n_st[ph]
                    for u in range(2 if two else 1):
                        slot = (k[0] + u) % slots
                        while not full[slot].done(((k[0] + u) // slots) & 1):
                            yield
                        assert ring[slot] == (ph, st if u == 0 else st2), ("wrong stage in slot", ph, c)
                        consumed.add(ring[slot])
                    yield                                           # the pair's CTA barrier
                    for s_ in ([st, st2] if two else [st]):        # epilogues
                        if ph < 4 * L and ph % 4 == 0:             # QKV: publish the quads
                            l = ph // 4
                            for e in range(tps[0]):
                                task = s_ * tps[0] + e
                                if task < tasks[0]:                # one epilogue thread per quad
                                    quads[l][kvh_of(4 * task)] += 1
                                    pub[kvh_of(4 * task)] += 1     # counted in shared memory
                                    yield
                        written[ph] += 1
                    feed_one()
                    if two:
                        feed_one()
                    k[0] += 2 if two else 1
                    st += 2 * grid
                if ph < 4 * L and ph % 4 == 0:                     # publish once per KV head
                    yield                                           # the CTA barrier
                    for h in range(KV):
                        if pub[h]:
                            shared["cnt"][h] += pub[h]
                            pub[h] = 0
                            yield

            def done_all(ph):
                return lambda: written[ph] == n_st[ph]

            for _ in range(slots):
                feed_one()
            yield from grid_sync()                                  # after the embedding
            has_unit = c < units
            u_kvh, u_sp = c % KV, c // KV
            for l in range(L):
                base = 4 * l
                yield from gemv(base, (lambda: True) if l == 0 else done_all(base - 1))
                if has_unit:
                    target = (l + 1) * kvh_quads
                    while shared["cnt"][u_kvh] < target:
                        yield
                    assert quads[l][u_kvh] == kvh_quads, ("unit started before its head's rows", l, c)
                    if ns == 1:
                        assert l == 0 or staged[base - 3] == grid, "o overwritten before every CTA staged it"
                        merged[(l, u_kvh)] = True
                    else:
                        assert l == 0 or merged[(l - 1, u_kvh)], "partial overwritten before the merge read it"
                        partial[(u_kvh, u_sp)] = l
                        prev = shared["att"][u_kvh]
                        shared["att"][u_kvh] += 1
                        yield
                        if prev == ns - 1:                          # the last split merges
                            assert all(partial.get((u_kvh, s)) == l for s in range(ns)), "merge missed a split"
                            assert l == 0 or staged[base - 3] == grid, "o overwritten before every CTA staged it"
                            merged[(l, u_kvh)] = True
                            shared["att"][u_kvh] = 0
                yield from grid_sync()
                yield from gemv(base + 1, lambda: all(merged[(l, h)] for h in range(KV)))
                yield from grid_sync()
                assert staged[base] == grid, "x overwritten before every CTA staged it"
                yield from gemv(base + 2, done_all(base + 1))
                yield from grid_sync()
                yield from gemv(base + 3, done_all(base + 2))
                yield from grid_sync()
            if n_out:
                yield from gemv(4 * L, done_all(4 * L - 1))
            prev = shared["bar1"]
            shared["bar1"] += 1
            if prev == grid - 1:                                    # the last CTA resets the counters
                shared["bar0"] = 0
                shared["bar1"] = 0
                shared["cnt"] = [0] * KV
            assert cur["issued"] == k[0], ("stages issued but never consumed", c)

        agents = [cta(c) for c in range(grid)]
        alive = [True] * grid
        for _ in range(100000):
            if not any(alive):
                break
            events.sort(key=lambda e: e[0])
            while events and events[0][0] <= now[0]:
                events.pop(0)[1]()
            order = list(range(grid))
            rnd.shuffle(order)
            for i in order:
                if alive[i]:
                    try:
                        next(agents[i])
                    except StopIteration:
                        alive[i] = False
            now[0] += 1
        else:
            raise AssertionError("deadlock")
        assert written[:n_ph] == n_st[:n_ph]
    return True


SHAPES = [
    # grid, slots, L, H, KV, hd, d, F, V, tps per phase kind (QKV, O, GU, down), splits, n_out
    (3, 3, 2, 4, 2, 8, 32, 16, 20, (2, 4, 2, 1), 1, 1),
    (5, 5, 2, 4, 2, 8, 32, 16, 20, (2, 4, 2, 1), 2, 1),
    (4, 4, 2, 8, 2, 8, 32, 24, 36, (4, 2, 2, 1), 2, 0),
    (7, 5, 3, 4, 1, 16, 48, 40, 44, (2, 4, 2, 1), 7, 1),
]


@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_decode_step_protocol(shape):
    grid, slots, L, H, KV, hd, d, F, V, tps, ns, n_out = SHAPES[shape]
    for seed in range(4):
        model(grid, slots, L, H, KV, hd, d, F, V, tps, ns, n_out, seed)


@pytest.mark.parametrize("wrong,right", [
    ("target = (l + 1) * kvh_quads", "target = l * kvh_quads + 1"),             # a unit starts on the first quads
    ('                shared["cnt"] = [0] * KV\n', ""),                          # counters left for the next launch
])
def test_model_catches_planted_mistakes(wrong, right):
    """The check is not vacuous: each planted protocol mistake fails it."""
    import inspect
    src = inspect.getsource(model)
    assert wrong in src
    ns_ = {"random": random, "Bar": Bar}
    exec(compile(src.replace(wrong, right), "mutated", "exec"), ns_)
    with pytest.raises(AssertionError):
        for seed in range(6):
            ns_["model"](*SHAPES[1][:-1], SHAPES[1][-1], seed)
