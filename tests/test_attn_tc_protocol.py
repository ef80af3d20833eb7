"""Model check of the tcgen05 prefill attention's pipeline protocol (k_attn_prefill_tc.cu), on the CPU.

compute-sanitizer is not available for this kernel's GPU, so its barrier protocol is checked as a
model, in the way of the GEMM ring model: the K/V producer (two TMA stages), the MMA issuer
(S_t = Q K_t^T into score buffer t % 2, then P_{t-1} V_{t-1} into O with P read from buffer
(t - 1) % 2) and the four softmax warps (a row quarter each: scores in, P written over them, O
rescaled once the previous product is done) run as coroutines over the kernel's loop structure,
stage and buffer indices and barrier parities. mbarriers are modelled by their phase, arrival and
transaction counts (try_wait.parity p succeeds once the phase of parity p has completed); the
MMAs of the issuing thread complete in issue order after random delays, and a commit arrives once
every MMA issued before it is done; copies land after random delays. For every key-tile count the
kernel meets, every wait must end (no deadlock), must wake on the phase it waits for (no parity
aliasing), every read must see the data of its own tile, and no stage, score buffer or O may be
written while an MMA or a warp still reads it. (The model also shows that the score buffer's
p_free wait is implied by the stage's: the same index, and the stage is refilled only after the
product that read both.)
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
        assert self.pending >= 0, "barrier over-arrived"
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, k):
        """Has the k-th phase (0-based) completed, as try_wait.parity(k & 1) sees it? The model
        also asserts that no later phase has completed yet (the parity would alias)."""
        ok = (self.phase & 1) != (k & 1)
        if ok:
            assert self.phase == k + 1, ("parity aliasing", k, self.phase)
        return ok


def run(n_kt, seed, skip_empty_kv=False, skip_o_done=False):
    rnd = random.Random(seed)
    events, now = [], [0]

    def later(fn, lo, hi):
        events.append((now[0] + rnd.randint(lo, hi), fn))

    full_kv, empty_kv = [Bar(1), Bar(1)], [Bar(1), Bar(1)]
    s_full, p_full, p_free = [Bar(1), Bar(1)], [Bar(4), Bar(4)], [Bar(1), Bar(1)]
    o_done, q_full = Bar(1), Bar(4)
    kv = [None, None]                 # tile held by each stage
    S = [None, None]                  # score buffer b: ("S", t) or ("P", t, warps written)
    O = {"tiles": -1}                 # last tile whose product O includes
    kv_readers = [set(), set()]       # in-flight MMAs reading a stage ("K" / "V")
    buf_readers = [set(), set()]      # in-flight readers of a score buffer
    o_busy = [0]                      # in-flight P.V products writing O
    q_ready = [0]
    mma_tail = [0]                    # completion time of the last MMA issued (in-order pipe)

    def mma_issue(fn, lo=3, hi=40):
        t = max(now[0], mma_tail[0]) + rnd.randint(lo, hi)
        mma_tail[0] = t
        events.append((t, fn))

    def commit(bar):
        # arrives once every MMA issued before it has completed
        events.append((mma_tail[0], bar.arrive))

    def producer():
        for j in range(n_kt):
            s = j & 1
            if j >= 2 and not skip_empty_kv:
                while not empty_kv[s].done((j >> 1) - 1):
                    yield
            assert not kv_readers[s], ("K/V stage overwritten while an MMA reads it", j)
            full_kv[s].expect_tx(2)

            def land(s=s, j=j):
                kv[s] = j
                full_kv[s].complete_tx(2)
            later(land, 5, 60)
            yield

    def mma():
        while not q_full.done(0):
            yield
        assert q_ready[0] == 4
        for t in range(n_kt + 1):
            if t < n_kt:
                s = b = t & 1
                while not full_kv[s].done(t >> 1):
                    yield
                if t >= 2:
                    while not p_free[b].done((t >> 1) - 1):
                        yield
                assert kv[s] == t, ("K of tile", t, kv[s])
                assert not buf_readers[b], ("score buffer overwritten while P is read", t)
                kv_readers[s].add("K")
                buf_readers[b].add("S-write")

                def s_done(s=s, b=b, t=t):
                    kv_readers[s].discard("K")
                    buf_readers[b].discard("S-write")
                    S[b] = ("S", t)
                mma_issue(s_done)
                commit(s_full[b])
            if t >= 1:
                u = t - 1
                s = b = u & 1
                while not p_full[b].done(u >> 1):
                    yield
                assert S[b] == ("P", u, 4), ("P of tile", u, S[b])
                assert kv[s] == u, ("V of tile", u, kv[s])
                kv_readers[s].add("V")
                buf_readers[b].add("P-read")
                o_busy[0] += 1

                def pv_done(s=s, b=b, u=u):
                    kv_readers[s].discard("V")
                    buf_readers[b].discard("P-read")
                    assert O["tiles"] == u - 1, ("P.V products out of order", u, O)
                    O["tiles"] = u
                    o_busy[0] -= 1
                mma_issue(pv_done)
                commit(empty_kv[s])
                commit(p_free[b])
                commit(o_done)
            yield

    def softmax(w):
        q_ready[0] += 1
        q_full.arrive()
        yield
        for j in range(n_kt):
            b = j & 1
            while not s_full[b].done(j >> 1):
                yield
            assert S[b] is not None and S[b][:2] == ("S", j) or (S[b][0] == "P" and S[b][1] == j), ("scores", j, S[b])
            yield
            # P over this warp's rows of the scores (the buffer is not read by any MMA now)
            assert "P-read" not in buf_readers[b] and "S-write" not in buf_readers[b], ("P written under an MMA", j)
            S[b] = ("P", j, (S[b][2] if S[b][0] == "P" else 0) + 1)
            yield
            if j > 0 and not skip_o_done:
                while not o_done.done(j - 1):
                    yield
            if j > 0:
                assert o_busy[0] == 0 and O["tiles"] == j - 1, ("O rescaled while a product writes it", j, O)
            p_full[b].arrive()
        while not o_done.done(n_kt - 1):
            yield
        assert O["tiles"] == n_kt - 1 and o_busy[0] == 0

    agents = [producer(), mma()] + [softmax(w) for w in range(4)]
    alive = [True] * len(agents)
    for _ in range(200000):
        if not any(alive):
            assert all(not r for r in kv_readers)
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


@pytest.mark.parametrize("n_kt", [1, 2, 3, 4, 7, 16])
def test_pipeline_protocol(n_kt):
    for seed in range(6):
        run(n_kt, seed)


def test_model_catches_a_stage_refilled_too_early():
    """Without the wait for the stage's P.V product, the next tile's copy lands under it."""
    with pytest.raises(AssertionError):
        for seed in range(30):
            run(8, seed, skip_empty_kv=True)


def test_model_catches_o_rescaled_under_a_product():
    """Without the wait for the previous P.V product, O is rescaled while that product writes it."""
    with pytest.raises(AssertionError):
        for seed in range(30):
            run(8, seed, skip_o_done=True)
