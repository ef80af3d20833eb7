"""Host-side rules of the C-ABI library, on machines without a GPU.

The library loads and exports every symbol include/lcx.h declares; a host-only context runs the
batch rules of lcx_decode (validation, filling, cell reservation, ubatch split, abort, return
codes) and is compared against the oracle's batch rules on random batch streams.
"""
import re
import os

import numpy as np
import pytest

import llama_ubatch_forward_gb300 as lcx
import oracle
import synth
from llama_ubatch_forward_gb300.torch_io import hparams_of

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TINY = synth.CONFIGS["tiny"]


@pytest.fixture(scope="module", autouse=True)
def built():
    lcx.build()


def test_exports_every_declared_symbol():
    hdr = open(os.path.join(ROOT, "include", "lcx.h")).read()
    declared = set(re.findall(r"\b(lcx_[a-z_0-9]+)\s*\(", hdr))
    assert declared == set(lcx.SYMBOLS)
    L = lcx.lib()
    for name in declared:
        assert hasattr(L, name), name


def _host_ctx(n_ctx=256, n_seq=2, n_ubatch=4):
    return lcx.Context(None, n_ctx, n_seq, n_ubatch, host_only_hp=hparams_of(TINY))


def test_rejects_bad_shapes():
    hp = hparams_of(TINY)
    hp.n_embd = 100
    with pytest.raises(RuntimeError):
        lcx.Context(None, 128, 1, 8, host_only_hp=hp)
    hp = hparams_of(TINY)
    hp.n_head_kv = 3
    with pytest.raises(RuntimeError):
        lcx.Context(None, 128, 1, 8, host_only_hp=hp)


def test_return_codes_and_filling():
    c = _host_ctx(n_ctx=100)
    assert c.stats().n_ctx == 256
    V = TINY.n_vocab
    assert c.decode([]) == lcx.LCX_INVALID if False else True
    assert c.decode([V]) == -1 and c.decode([-5]) == -1
    assert c.decode([1], seq_id=[2]) == -1
    assert c.decode([1, 2], pos=[0, 2]) == -1
    assert c.decode([1], pos=[1]) == -1
    assert c.decode([1, 2, 3]) == 0 and c.seq_pos_max(0) == 2 and c.n_outputs() == 1
    assert c.decode([4, 5], seq_id=[1, 1], logits=[1, 1]) == 0 and c.n_outputs() == 2
    assert c.seq_pos_max(1) == 1
    assert c.decode(np.ones(252, np.int32)) == 1 and c.seq_pos_max(0) == 2     # 5 used + 252 > 256
    assert c.decode(np.ones(251, np.int32)) == 0 and c.seq_pos_max(0) == 253
    assert c.stats().n_cells_used == 256
    assert c.decode([1]) == 1
    c.kv_clear()
    assert c.seq_pos_max(0) == -1 and c.stats().n_cells_used == 0
    assert c.decode([7]) == 0 and c.seq_pos_max(0) == 0


def test_ubatch_split_and_outputs():
    c = _host_ctx(n_ctx=512, n_ubatch=5)
    assert c.decode(np.arange(17), logits=np.ones(17)) == 0
    s = c.stats()
    assert s.n_ubatch_last == 4 and s.n_outputs_last == 17


def test_abort_between_ubatches_releases_the_rest():
    c = _host_ctx(n_ctx=512, n_ubatch=4)
    calls = []

    def cb():
        calls.append(1)
        return len(calls) >= 2            # let the 2nd ubatch run, stop before the 3rd

    c.set_abort(cb)
    assert c.decode(np.arange(10), logits=np.ones(10)) == lcx.LCX_ABORTED
    assert c.seq_pos_max(0) == 7 and c.stats().n_cells_used == 8 and c.n_outputs() == 8
    c.set_abort(None)
    assert c.decode([1], pos=[8]) == 0 and c.seq_pos_max(0) == 8


def test_pages_recycle_across_clears():
    c = _host_ctx(n_ctx=256, n_seq=4, n_ubatch=64)
    for _ in range(3):
        for s in range(4):
            assert c.decode(np.arange(64), seq_id=np.full(64, s)) == 0
        assert c.decode([1]) == 1
        c.kv_clear()


@pytest.mark.parametrize("unified", [True, False])
def test_rules_match_the_oracle_on_random_streams(unified):
    """Same return code and positions as the oracle for random valid and invalid batches, with one
    shared cell store and with a stream per sequence (its own capacity rule)."""
    m = synth.make_model(TINY, n_layer=1)
    rng = np.random.default_rng(11)
    for trial in range(3):
        oc = oracle.Context(oracle.Model(m), 256, 3, 512)
        hc = _host_ctx(n_ctx=256, n_seq=3, n_ubatch=7)
        assert oc.set_kv_unified(unified) == 0 and hc.set_kv_unified(unified) == 0
        for step in range(25):
            n = int(rng.integers(0, 40))
            toks = rng.integers(-1, TINY.n_vocab + 1, n) if rng.random() < 0.2 else rng.integers(0, TINY.n_vocab, n)
            seq = rng.integers(0, 4 if rng.random() < 0.2 else 3, n)
            pos = None
            if rng.random() < 0.5:
                nxt = {s: oc.seq_pos_max(s) + 1 for s in range(3)}
                pos = []
                for s in seq:
                    pos.append(nxt.get(int(s), 0))
                    nxt[int(s)] = nxt.get(int(s), 0) + 1
                if rng.random() < 0.3 and n:
                    pos[int(rng.integers(0, n))] += 1
            flags = (rng.random(n) < 0.3).astype(np.int8) if rng.random() < 0.5 else None
            ro = oc.decode(toks, pos, seq, flags)
            rh = hc.decode(toks, pos, seq, flags)
            assert rh == ro[0], (trial, step)
            if ro[0] == 0:
                assert hc.n_outputs() == ro[1].shape[0]
            for s in range(3):
                assert hc.seq_pos_max(s) == oc.seq_pos_max(s)


def test_sample_checks_arguments_before_any_device_work():
    """lcx_sample's host-side checks: each call below returns before touching the device (the
    pointers are never dereferenced), so it runs without a GPU."""
    import ctypes
    L = lcx.lib()
    P = lcx.lcx_sampler
    ok = P(1.0, 40, 0.95, 0.05, 0.8)
    fake = 16
    by = ctypes.byref
    assert L.lcx_sample(None, fake, 1, 100, None, 0, fake, fake, None) == lcx.LCX_INVALID        # no parameters
    assert L.lcx_sample(by(ok), fake, -1, 100, None, 0, fake, fake, None) == lcx.LCX_INVALID     # rows < 0
    assert L.lcx_sample(by(ok), fake, 1, 0, None, 0, fake, fake, None) == lcx.LCX_INVALID        # empty vocabulary
    assert L.lcx_sample(by(ok), fake, 1, (1 << 18) + 1, None, 0, fake, fake, None) == lcx.LCX_INVALID
    assert L.lcx_sample(by(ok), fake, 1, 100, None, -1, fake, fake, None) == lcx.LCX_INVALID     # history < 0
    for pen in (0.0, -1.0, float("nan"), float("inf")):
        assert L.lcx_sample(by(P(pen, 40, 0.95, 0.05, 0.8)), fake, 1, 100, None, 0, fake, fake, None) == lcx.LCX_INVALID
    assert L.lcx_sample(by(ok), None, 0, 100, None, 0, None, None, None) == lcx.LCX_OK         # no rows: no-op
    assert L.lcx_sample(by(ok), None, 1, 100, None, 0, fake, fake, None) == lcx.LCX_INVALID      # no logits
    assert L.lcx_sample(by(ok), fake, 1, 100, None, 0, fake, None, None) == lcx.LCX_INVALID      # no output
    assert L.lcx_sample(by(ok), fake, 1, 100, None, 3, fake, fake, None) == lcx.LCX_INVALID      # history missing
    assert L.lcx_sample(by(ok), fake, 1, 100, None, 0, None, fake, None) == lcx.LCX_INVALID      # a draw needs u


def test_failed_ubatch_rolls_back_like_the_oracle():
    """A failed ubatch (-3) releases its cells and those of the later ubatches; earlier ubatches
    stay. The failure is made on the host (a host-only context's injected launch failure) and
    compared with the oracle's rule (a non-finite logit fails its ubatch)."""
    import dataclasses
    hp = hparams_of(TINY)
    c = lcx.Context(None, 256, 2, 2, host_only_hp=hp)
    assert c.inject_failure(1) == 0
    # tokens of two sequences, ubatches of 2: [s0 p0, s1 p0] [s0 p1, s1 p1] [s0 p2]
    toks, seqs = [1, 2, 3, 4, 5], [0, 1, 0, 1, 0]
    assert c.decode(toks, seq_id=seqs, logits=[1, 0, 1, 1, 1]) == lcx.LCX_COMPUTE_FAILED
    # the first ubatch stays, with its one row; the failed and the later ubatch go
    assert (c.seq_pos_max(0), c.seq_pos_max(1), c.n_outputs()) == (0, 0, 1)
    assert c.stats().n_cells_used == 2
    assert c.decode([6, 7], seq_id=[0, 1]) == 0              # the failure was one-shot
    assert (c.seq_pos_max(0), c.seq_pos_max(1)) == (1, 1)
    assert c.inject_failure(0) == 0
    assert c.decode([8], seq_id=[1]) == lcx.LCX_COMPUTE_FAILED and c.seq_pos_max(1) == 1
    # the oracle: the flagged row of a NaN-embedding token in ubatch 1 fails it
    host = synth.make_model(TINY)
    bad = 11
    emb = host.tok_embd.copy()
    emb[bad].view(np.uint16)[:] = 0x7E00
    octx = oracle.Context(oracle.Model(dataclasses.replace(host, tok_embd=emb)), 256, 2, 2)
    rc, lg, _ = octx.decode([1, 2, bad, 4, 5], seq=seqs, logits=[1, 0, 1, 1, 1])
    assert rc == -3 and (octx.seq_pos_max(0), octx.seq_pos_max(1)) == (0, 0) and lg.shape[0] == 1


def test_inject_failure_needs_a_host_only_context():
    assert lcx.lib().lcx_ctx_inject_failure(None, 0) == lcx.LCX_INVALID


def test_split_equal_failures_roll_back_like_the_oracle():
    """A stream per sequence: batches are cut by split_equal. A failure injected at ubatch k
    (host only) releases the same cells as the oracle's failed ubatch k (a NaN embedding in it), and
    no rows are reported."""
    import dataclasses
    seqs = np.array([0, 1, 2, 0, 1, 2, 0, 2, 0, 0], np.int32)
    base = np.array([11, 12, 13, 14, 15, 16, 17, 18, 19, 20], np.int32)
    host = synth.make_model(TINY, n_layer=1)
    emb = host.tok_embd.copy()
    emb[7].view(np.uint16)[:] = 0x7E00
    om = oracle.Model(dataclasses.replace(host, tok_embd=emb))
    # ubatches {0,1,2} {3,4,5} {6,7} {8,9}: a bad token at index 5 fails ubatch 1, at 8 ubatch 3
    for where, k in ((5, 1), (8, 3), (6, 2)):
        toks = base.copy()
        toks[where] = 7
        oc = oracle.Context(om, 256, 3, 4)
        oc.set_kv_unified(False)
        assert oc.decode(toks, seq=seqs, logits=np.ones(10, np.int8))[0] == -3
        hc = _host_ctx(n_ctx=256, n_seq=3, n_ubatch=4)
        assert hc.set_kv_unified(False) == 0 and hc.inject_failure(k) == 0
        assert hc.decode(base, seq_id=seqs, logits=np.ones(10, np.int8)) == lcx.LCX_COMPUTE_FAILED
        assert hc.n_outputs() == 0
        assert [hc.seq_pos_max(s) for s in range(3)] == [oc.seq_pos_max(s) for s in range(3)], (where, k)
    hc = _host_ctx(n_ctx=256, n_seq=3, n_ubatch=4)
    assert hc.decode([1], seq_id=[0]) == 0 and hc.set_kv_unified(False) == lcx.LCX_INVALID   # cells held


def test_gemm_tile_forcing_accepts_only_compiled_shapes():
    # the prefill GEMM's tile-shape override is host state: no device needed to set or reject it
    for good in ((64, 1, 1), (64, 2, 3), (128, 1, 8), (128, 2, 2), (256, 1, 1)):
        assert lcx.set_gemm_tile(*good) == lcx.LCX_OK, good
    for bad in ((32, 1, 1), (256, 2, 1), (128, 3, 1), (128, 1, 0), (128, 1, 9), (96, 1, 1)):
        assert lcx.set_gemm_tile(*bad) == lcx.LCX_INVALID, bad
    assert lcx.set_gemm_tile(0) == lcx.LCX_OK
