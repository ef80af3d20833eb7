"""Pins of the CPU oracle against things other than itself.

Hand-computed blocks, closed forms, invariants, library routines for special cases, and brute
force on tiny inputs. A plausible slip anywhere in the oracle (a dropped term, a sign, an index,
a transposed operand, a missing RoPE) makes one of these fail.
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TYPES = {"Q8_0": synth.Q8_0, "Q4_0": synth.Q4_0, "F16": synth.F16}


def _golden_blocks():
    out = []
    with open(os.path.join(GOLDEN, "dequant_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split(":")
            parts = lhs.split()
            qtype = TYPES[parts[0]]
            raw = bytes.fromhex("".join(parts[1:]))
            exp = {int(a): float(b) for a, b in (kv.split("=") for kv in rhs.split())}
            out.append((parts[0], qtype, raw, exp))
    return out


@pytest.mark.parametrize("name,qtype,raw,exp", _golden_blocks(), ids=lambda v: v if isinstance(v, str) else "")
def test_dequant_hand_blocks(name, qtype, raw, exp):
    n = len(raw) // 2 if qtype == synth.F16 else 32
    vals = oracle.dequant_row(qtype, np.frombuffer(raw, dtype=np.uint8), n)
    for i, v in exp.items():
        assert vals[i] == v, (name, i, vals[i], v)


def test_half_decode_matches_numpy_everywhere():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits[::7]])
    r = ref[::7]
    fin = np.isfinite(r)
    assert np.array_equal(got[fin], r[fin])
    assert np.array_equal(np.isnan(got), np.isnan(r))


def test_round_to_half_hand_values_and_numpy():
    ulp1 = 2.0 ** -10
    cases = {1.0 + ulp1 / 2: 1.0,               # tie -> even
             1.0 + 1.5 * ulp1: 1.0 + 2 * ulp1,  # tie -> even
             65519.0: 65504.0, 65520.0: math.inf,
             2.0 ** -25: 0.0, 3 * 2.0 ** -25: 2.0 ** -23, -1.0 / 3.0: -0.333251953125}
    for x, y in cases.items():
        assert oracle.round_to_half(x) == y, x
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 1e-5, 1000), rng.normal(0, 3e4, 1000)])
    got = np.array([oracle.round_to_half(float(x)) for x in xs])
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).astype(np.float64)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("qtype", [synth.Q8_0, synth.Q4_0])
def test_quantize_dequant_roundtrip_bound(qtype):
    w = synth.normal(99, 7, 64 * 256, 0.0, 0.02).reshape(64, 256)
    w[3, :32] = 0.0                            # an all-zero block
    rows = synth.encode(w, qtype)
    for r in range(64):
        deq = oracle.dequant_row(qtype, rows[r], 256)
        for b in range(8):
            blk = rows[r, b * synth.BLOCK_BYTES[qtype]: (b + 1) * synth.BLOCK_BYTES[qtype]]
            d = abs(float(np.frombuffer(blk[:2].tobytes(), dtype=np.float16)[0]))
            err = np.abs(deq[b * 32:(b + 1) * 32] - w[r, b * 32:(b + 1) * 32])
            # half a step, plus the fp16 rounding of the scale itself; Q4_0's +8 end is clamped
            bound = d * (1.0 if qtype == synth.Q4_0 else 0.5) + 8 * d * 2.0 ** -11 + 1e-12
            assert np.all(err <= bound), (r, b, err.max(), d)
    assert np.all(oracle.dequant_row(qtype, rows[3], 32) == 0.0)


@pytest.mark.parametrize("qtype,K,N", [(synth.Q8_0, 32, 3), (synth.Q8_0, 64, 16), (synth.Q4_0, 704, 5),
                                       (synth.Q4_0, 64, 16), (synth.F16, 48, 4)])
def test_matvec_brute_force(qtype, K, N):
    w = synth.normal(5, K + N, N * K, 0.0, 0.05).reshape(N, K)
    rows = synth.encode(w, qtype)
    x = np.random.default_rng(K).normal(size=K)
    y = oracle.matvec(qtype, rows, N, K, x)
    Wd = oracle.dequant_matrix(qtype, rows, K)
    assert np.allclose(y, Wd @ x, rtol=1e-12, atol=1e-14)


def test_matvec_closed_form_single_weight():
    # one nonzero weight at (n=2, k=37): y = e_2 * w * x_37; w = 127/256 so d = 2^-8 and q = 127 exactly
    w = np.zeros((4, 64), dtype=np.float32)
    w[2, 37] = 127.0 / 256.0
    rows = synth.encode(w, synth.Q8_0)
    x = np.arange(64, dtype=np.float64)
    y = oracle.matvec(synth.Q8_0, rows, 4, 64, x)
    assert y.tolist() == [0.0, 0.0, 127.0 / 256.0 * 37, 0.0]


def test_rmsnorm_invariants():
    rng = np.random.default_rng(0)
    x = rng.normal(size=256)
    ones = np.ones(256, dtype=np.float32)
    y = oracle.rmsnorm(x, ones, 0.0)
    assert math.isclose(math.sqrt(np.mean(y * y)), 1.0, rel_tol=1e-14)
    assert np.allclose(oracle.rmsnorm(7.5 * x, ones, 0.0), y, rtol=1e-13)
    assert np.allclose(oracle.rmsnorm(np.array([3.0, 4.0]), np.array([1, 2], np.float32), 0.0),
                       [3 / math.sqrt(12.5), 8 / math.sqrt(12.5)], rtol=1e-15)
    # eps enters under the root: x = [1, 1], eps = 3 -> 1 / sqrt(4)
    assert np.allclose(oracle.rmsnorm(np.ones(2), np.ones(2, np.float32), 3.0), [0.5, 0.5], rtol=1e-15)
    g = rng.normal(1, 0.1, 256).astype(np.float32)
    assert np.allclose(oracle.rmsnorm(x, g, 0.0), y * g.astype(np.float64), rtol=1e-14)


def test_rope_pins():
    rng = np.random.default_rng(2)
    x = rng.normal(size=64)
    assert np.array_equal(oracle.rope(x, 0, 10000.0), x)                       # identity at pos 0
    for p in (1, 17, 32895):
        assert math.isclose(np.linalg.norm(oracle.rope(x, p, 5e5)), np.linalg.norm(x), rel_tol=1e-13)
    e0 = np.zeros(4); e0[0] = 1.0
    assert np.allclose(oracle.rope(e0, 1, 10000.0), [math.cos(1), math.sin(1), 0, 0], rtol=0, atol=1e-16)
    e2 = np.zeros(4); e2[2] = 1.0                                               # pair 1: angle 10000^(-2/4) = 0.01
    assert np.allclose(oracle.rope(e2, 1, 10000.0), [0, 0, math.cos(0.01), math.sin(0.01)], atol=1e-16)
    e3 = np.zeros(4); e3[3] = 1.0
    assert np.allclose(oracle.rope(e3, 3, 10000.0), [0, 0, -math.sin(0.03), math.cos(0.03)], atol=1e-16)
    q, k = rng.normal(size=64), rng.normal(size=64)
    d1 = oracle.rope(q, 10, 1e4) @ oracle.rope(k, 3, 1e4)
    d2 = oracle.rope(q, 107, 1e4) @ oracle.rope(k, 100, 1e4)                  # only p - p' matters
    assert math.isclose(d1, d2, rel_tol=1e-10)


def test_silu_pins():
    assert oracle.silu(0.0) == 0.0
    assert math.isclose(oracle.silu(1.0), 0.7310585786300049, rel_tol=1e-15)
    assert math.isclose(oracle.silu(-2.0), -2.0 / (1.0 + math.e ** 2), rel_tol=1e-15)
    assert math.isclose(oracle.silu(40.0), 40.0, rel_tol=1e-15)
    assert abs(oracle.silu(-40.0)) < 1e-15


def test_attention_pins():
    rng = np.random.default_rng(3)
    hd, H, KV = 8, 4, 2
    q = rng.normal(size=H * hd)
    K1, V1 = rng.normal(size=(1, KV * hd)), rng.normal(size=(1, KV * hd))
    o = oracle.attend_gqa(q, K1, V1, H, KV, hd)                   # one key returns its value
    assert np.allclose(o, np.concatenate([V1[0, :hd], V1[0, :hd], V1[0, hd:], V1[0, hd:]]), rtol=1e-15)
    K, V = rng.normal(size=(9, KV * hd)), rng.normal(size=(9, KV * hd))
    o = oracle.attend_gqa(np.zeros(H * hd), K, V, H, KV, hd)      # q = 0: mean of the values
    assert np.allclose(o[:hd], V[:, :hd].mean(0), rtol=1e-13) and np.allclose(o[3 * hd:], V[:, hd:].mean(0), rtol=1e-13)
    o = oracle.attend_gqa(q, K, np.ones_like(V), H, KV, hd)       # rows of the softmax sum to 1
    assert np.allclose(o, 1.0, rtol=1e-14)
    Vz = np.zeros_like(V); Vz[:, :hd] = V[:, :hd]                 # GQA map: kv head 0 feeds q heads 0, 1 only
    o = oracle.attend_gqa(q, K, Vz, H, KV, hd)
    assert np.all(o[2 * hd:] == 0.0) and np.all(np.abs(o[:2 * hd]) > 0)
    # brute force against an explicit score matrix
    for h in range(H):
        kv = h // (H // KV)
        s = K[:, kv * hd:(kv + 1) * hd] @ q[h * hd:(h + 1) * hd] / math.sqrt(hd)
        p = np.exp(s - s.max()); p /= p.sum()
        assert np.allclose(o[h * hd:(h + 1) * hd] if False else oracle.attend_gqa(q, K, V, H, KV, hd)[h * hd:(h + 1) * hd],
                           p @ V[:, kv * hd:(kv + 1) * hd], rtol=1e-12)


# ----------------------------------------------------------------------------- whole model
TINY = synth.CONFIGS["tiny"]


@pytest.fixture(scope="module")
def tiny_model():
    return synth.make_model(TINY)


def _ctx(m, n_ctx=128, n_seq=1):
    return oracle.Context(oracle.Model(m), n_ctx, n_seq, 512)


def test_prefill_equals_stepwise_decode(tiny_model):
    toks = synth.prompt_tokens(TINY, 12)
    a = _ctx(tiny_model)
    rc, la, ia = a.decode(toks, np.arange(12), np.zeros(12), np.ones(12))
    assert rc == 0 and la.shape == (12, TINY.n_vocab)
    b = _ctx(tiny_model)
    rows = []
    for i, t in enumerate(toks):
        rc, lb, ib = b.decode([t], [i], [0], [1])
        assert rc == 0
        rows.append(lb[0])
    assert np.array_equal(la, np.stack(rows))
    for l in range(TINY.n_layer):
        for p in (0, 5, 11):
            ka, va = a.kv_get(0, p, l)
            kb, vb = b.kv_get(0, p, l)
            assert np.array_equal(ka, kb) and np.array_equal(va, vb)


def test_kv_cells_are_f16_and_layer0_composition(tiny_model):
    c = _ctx(tiny_model)
    toks = synth.prompt_tokens(TINY, 5)
    assert c.decode(toks)[0] == 0
    m = tiny_model
    hd, KVh = TINY.head_dim, TINY.n_head_kv
    for p in range(5):
        k, v = c.kv_get(0, p, 0)
        assert np.array_equal(k, k.astype(np.float16).astype(np.float64))
        x = oracle.dequant_row(TINY.t_embd, m.tok_embd[toks[p]], TINY.n_embd)
        xn = oracle.rmsnorm(x, m.layers[0]["attn_norm"], TINY.rms_eps)
        kk = oracle.matvec(TINY.t_linear, m.layers[0]["wk"], KVh * hd, TINY.n_embd, xn)
        vv = oracle.matvec(TINY.t_linear, m.layers[0]["wv"], KVh * hd, TINY.n_embd, xn)
        kk = np.concatenate([oracle.rope(kk[h * hd:(h + 1) * hd], p, TINY.rope_theta) for h in range(KVh)])
        assert np.array_equal(k, kk.astype(np.float16).astype(np.float64))
        assert np.array_equal(v, vv.astype(np.float16).astype(np.float64))


def test_layer_trace_composition(tiny_model):
    """q is RoPE'd at the token's position and attends exactly the cells 0..pos of its sequence."""
    c = _ctx(tiny_model)
    c.set_trace(1)
    toks = synth.prompt_tokens(TINY, 7)
    assert c.decode(toks)[0] == 0
    m, hd, H, KVh, d = tiny_model, TINY.head_dim, TINY.n_head, TINY.n_head_kv, TINY.n_embd
    x, q, o, x1 = c.trace("x"), c.trace("q"), c.trace("o"), c.trace("x1")
    xn = oracle.rmsnorm(x, m.layers[1]["attn_norm"], TINY.rms_eps)
    q_ref = oracle.matvec(TINY.t_linear, m.layers[1]["wq"], H * hd, d, xn)
    q_ref = np.concatenate([oracle.rope(q_ref[h * hd:(h + 1) * hd], 6, TINY.rope_theta) for h in range(H)])
    assert np.allclose(q, q_ref, rtol=1e-13, atol=1e-15)
    K = np.stack([c.kv_get(0, p, 1)[0] for p in range(7)])
    V = np.stack([c.kv_get(0, p, 1)[1] for p in range(7)])
    assert np.allclose(o, oracle.attend_gqa(q, K, V, H, KVh, hd), rtol=1e-13, atol=1e-15)
    assert np.allclose(x1, x + oracle.matvec(TINY.t_linear, m.layers[1]["wo"], d, H * hd, o), rtol=1e-13)


def _rms(x, g, eps):
    return x / np.sqrt(np.mean(x * x) + eps) * g.astype(np.float64)


def test_zero_layers_closed_form():
    """All layer weights zero: x stays the embedding, logits = Wout rms(emb) g."""
    m = synth.make_model(TINY, zero=synth.LAYER_TENSORS)
    c = _ctx(m)
    toks = synth.prompt_tokens(TINY, 4)
    rc, lg, am = c.decode(toks, logits=np.ones(4))
    assert rc == 0
    E = oracle.dequant_matrix(TINY.t_embd, m.tok_embd, TINY.n_embd)
    Wout = oracle.dequant_matrix(TINY.t_out, m.output, TINY.n_embd)
    for i, t in enumerate(toks):
        ref = Wout @ _rms(E[t], m.output_norm, TINY.rms_eps)
        assert np.allclose(lg[i], ref, rtol=1e-12, atol=1e-14)
        assert am[i] == int(np.argmax(ref))


def test_tied_output_uses_embedding():
    m = synth.make_model(TINY, zero=synth.LAYER_TENSORS, tied=True)
    c = _ctx(m)
    rc, lg, _ = c.decode([7])
    E = oracle.dequant_matrix(TINY.t_embd, m.tok_embd, TINY.n_embd)
    assert rc == 0 and np.allclose(lg[0], E @ _rms(E[7], m.output_norm, TINY.rms_eps), rtol=1e-12)


def test_attention_only_closed_form():
    """wq = 0 makes every score 0, so attention is the plain mean of the f16 V cells 0..t of the
    sequence; with the FFN gate zero the layer is x + Wo mean(v)."""
    m = synth.make_model(TINY, zero=("wq", "w_gate"), n_layer=1)
    c = _ctx(m)
    toks = synth.prompt_tokens(TINY, 6)
    rc, lg, _ = c.decode(toks, logits=np.ones(6))
    assert rc == 0
    d, hd, H, KVh = TINY.n_embd, TINY.head_dim, TINY.n_head, TINY.n_head_kv
    L = m.layers[0]
    E = oracle.dequant_matrix(TINY.t_embd, m.tok_embd, d)
    Wv = oracle.dequant_matrix(TINY.t_linear, L["wv"], d)
    Wo = oracle.dequant_matrix(TINY.t_linear, L["wo"], H * hd)
    Wout = oracle.dequant_matrix(TINY.t_out, m.output, d)
    vs = [(Wv @ _rms(E[t], L["attn_norm"], TINY.rms_eps)).astype(np.float16).astype(np.float64) for t in toks]
    for i in range(6):
        mv = np.mean(vs[:i + 1], axis=0)                              # [KV*hd]
        o = np.concatenate([mv[(h // (H // KVh)) * hd:((h // (H // KVh)) + 1) * hd] for h in range(H)])
        x1 = E[toks[i]] + Wo @ o
        ref = Wout @ _rms(x1, m.output_norm, TINY.rms_eps)
        assert np.allclose(lg[i], ref, rtol=1e-11, atol=1e-13), i


def test_ffn_only_closed_form():
    """wv = 0 makes attention output 0; the layer is x + Wd (silu(Wg xn) * (Wu xn)), with the
    n_ff = 688 inputs of ffn_down padded to 704 by zeros."""
    m = synth.make_model(TINY, zero=("wv",), n_layer=1)
    c = _ctx(m)
    rc, lg, _ = c.decode([11, 300], logits=[1, 1])
    assert rc == 0
    d, F = TINY.n_embd, TINY.n_ff
    L = m.layers[0]
    E = oracle.dequant_matrix(TINY.t_embd, m.tok_embd, d)
    Wg = oracle.dequant_matrix(TINY.t_linear, L["w_gate"], d)
    Wu = oracle.dequant_matrix(TINY.t_linear, L["w_up"], d)
    Wd = oracle.dequant_matrix(TINY.t_linear, L["w_down"], 704)[:, :F]
    Wout = oracle.dequant_matrix(TINY.t_out, m.output, d)
    for i, t in enumerate([11, 300]):
        xn = _rms(E[t], L["ffn_norm"], TINY.rms_eps)
        a, u = Wg @ xn, Wu @ xn
        x1 = E[t] + Wd @ (a / (1 + np.exp(-a)) * u)
        assert np.allclose(lg[i], Wout @ _rms(x1, m.output_norm, TINY.rms_eps), rtol=1e-11, atol=1e-13)


def test_sequences_are_independent(tiny_model):
    ta, tb = synth.prompt_tokens(TINY, 5, 0), synth.prompt_tokens(TINY, 7, 1)
    both = _ctx(tiny_model, n_seq=2)
    toks = [ta[0], tb[0], tb[1], ta[1], ta[2], tb[2], tb[3], tb[4], ta[3], tb[5], ta[4], tb[6]]
    seqs = [0, 1, 1, 0, 0, 1, 1, 1, 0, 1, 0, 1]
    rc, lg, am = both.decode(toks, seq=seqs, logits=np.ones(12))
    assert rc == 0
    alone_a = _ctx(tiny_model).decode(ta, logits=np.ones(5))[1]
    alone_b = _ctx(tiny_model).decode(tb, logits=np.ones(7))[1]
    ia = [i for i, s in enumerate(seqs) if s == 0]
    ib = [i for i, s in enumerate(seqs) if s == 1]
    assert np.array_equal(lg[ia], alone_a) and np.array_equal(lg[ib], alone_b)


def test_batch_rules_and_return_codes(tiny_model):
    c = _ctx(tiny_model, n_ctx=100, n_seq=2)
    assert c.n_ctx == 256                                  # rounded up to a multiple of 256
    V = TINY.n_vocab
    assert c.decode([])[0] == -1
    assert c.decode([V])[0] == -1 and c.decode([-1])[0] == -1
    assert c.decode([1], seq=[2])[0] == -1
    assert c.decode([1, 2], pos=[0, 2])[0] == -1           # not consecutive
    assert c.decode([1], pos=[1])[0] == -1                 # does not continue from the last position
    assert c.seq_pos_max(0) == -1
    rc, lg, am = c.decode([1, 2, 3])                       # positions filled, last token flagged
    assert rc == 0 and lg.shape[0] == 1 and c.seq_pos_max(0) == 2
    rc, lg, _ = c.decode([4, 5], seq=[1, 1], logits=[1, 0])
    assert rc == 0 and lg.shape[0] == 1 and c.seq_pos_max(1) == 1
    rc, _, _ = c.decode([6], pos=[3])
    assert rc == 0 and c.seq_pos_max(0) == 3
    big = np.ones(256 - 6 + 1, dtype=np.int32)             # one more cell than is free
    assert c.decode(big)[0] == 1 and c.seq_pos_max(0) == 3  # nothing committed
    assert c.decode(big[:-1])[0] == 0 and c.seq_pos_max(0) == 3 + 250
    c.kv_clear()
    assert c.seq_pos_max(0) == -1 and c.seq_pos_max(1) == -1
    assert c.decode([9])[0] == 0 and c.seq_pos_max(0) == 0


def test_argmax_ties_take_lowest_index():
    m = synth.make_model(TINY, zero=synth.LAYER_TENSORS)
    m.output[:] = 0                                         # d = 0: every logit is exactly 0
    assert _ctx(m).decode([3])[2].tolist() == [0]
    # rows 9 and 5 equal and far above the rest: the tie goes to 5
    w = np.zeros((TINY.n_vocab, TINY.n_embd), dtype=np.float32)
    w[[5, 9]] = 0.25
    m.output = synth.encode(w, TINY.t_out)
    m.output_norm[:] = 1.0
    m.tok_embd = synth.encode(np.full((TINY.n_vocab, TINY.n_embd), 0.5, np.float32), TINY.t_embd)
    rc, lg, am = _ctx(m).decode([3])
    assert rc == 0 and lg[0, 5] == lg[0, 9] > 0 and am.tolist() == [5]


def test_default_flags_select_last_token(tiny_model):
    toks = synth.prompt_tokens(TINY, 6)
    all_rows = _ctx(tiny_model).decode(toks, logits=np.ones(6))[1]
    rc, lg, _ = _ctx(tiny_model).decode(toks)
    assert rc == 0 and lg.shape[0] == 1 and np.array_equal(lg[0], all_rows[-1])
    rc, lg, _ = _ctx(tiny_model).decode(toks, logits=[0, 1, 0, 0, 1, 0])
    assert np.array_equal(lg, all_rows[[1, 4]])            # flagged rows, in batch order


def test_non_finite_logits_fail_their_ubatch():
    """A flagged row whose logits are not finite is a failed compute (-3): the cells of its
    ubatch are removed again; earlier ubatches stay in the cache, and so do their logits rows,
    which the decode loop copied out before the failing ubatch ran (step 12: each ubatch's rows
    are copied into the output buffer inside the loop, and the failure returns from it)."""
    import dataclasses
    cfg = synth.CONFIGS["tiny"]
    host = synth.make_model(cfg)
    bad = 7
    emb = host.tok_embd.copy()
    emb[bad].view(np.uint16)[:] = 0x7E00                   # an f16 NaN embedding row
    om = oracle.Model(dataclasses.replace(host, tok_embd=emb))
    # the bad token itself flagged: its own ubatch (the first) fails, nothing stays
    octx = oracle.Context(om, cfg.n_ctx, 1, 2)
    rc, lg, am = octx.decode([1, bad], logits=[1, 1])
    assert rc == -3 and lg.shape[0] == 0 and octx.seq_pos_max(0) == -1
    # ubatches [1, 2] [3, bad] [5]: the bad token's K/V reach token 5, whose row fails; the
    # first two ubatches stay (positions 0..3) with the one row they flagged (token 2)
    octx = oracle.Context(om, cfg.n_ctx, 1, 2)
    rc, lg, am = octx.decode([1, 2, 3, bad, 5], logits=[0, 1, 0, 0, 1])
    assert rc == -3 and lg.shape[0] == 1 and am.shape[0] == 1
    assert octx.seq_pos_max(0) == 3
    good = oracle.Context(om, cfg.n_ctx, 1, 2)
    rc2, lg2, am2 = good.decode([1, 2], logits=[0, 1])    # that row alone, from a clean context
    assert rc2 == 0 and np.array_equal(lg, lg2) and np.array_equal(am, am2)
    rc, lg, am = octx.decode([9], logits=[1])             # the sequence goes on from position 4
    assert rc == -3 and lg.shape[0] == 0 and octx.seq_pos_max(0) == 3   # (its K/V still include the bad cell)


# ----------------------------------------------------------------------------- evaluation order
@pytest.mark.parametrize("T", [1, 3, 8, 13, 17])
def test_matmat_rows_equal_matvec_and_brute_force(T):
    """Every token of a block product is the same k-ordered sum as its own matrix-vector
    product (bit for bit), and both are the plain product of the dequantized matrix."""
    K, N = 704, 37
    w = synth.normal(11, T, N * K, 0.0, 0.05).reshape(N, K)
    rows = synth.encode(w, synth.Q4_0)
    X = np.random.default_rng(T).normal(size=(T, K))
    Y = oracle.matmat(synth.Q4_0, rows, N, K, X)
    for t in range(T):
        assert np.array_equal(Y[t], oracle.matvec(synth.Q4_0, rows, N, K, X[t])), t
    assert np.allclose(Y, X @ oracle.dequant_matrix(synth.Q4_0, rows, K).T, rtol=1e-12, atol=1e-14)


def test_blocks_of_a_long_ubatch_equal_stepwise_decode(tiny_model):
    """A 300-token ubatch runs as two blocks (256 + 44 tokens) layer by layer; it must equal 300
    single-token decodes bit for bit, rows and cells."""
    toks = synth.uniform_int(TINY.token_seed, 77, 300, 0, TINY.n_vocab)
    a = _ctx(tiny_model, n_ctx=512)
    flags = np.zeros(300, np.int8)
    flags[[0, 255, 256, 299]] = 1
    rc, la, ia = a.decode(toks, logits=flags)
    assert rc == 0 and la.shape[0] == 4
    b = _ctx(tiny_model, n_ctx=512)
    rows = []
    for i, t in enumerate(toks):
        rc, lb, _ = b.decode([t], logits=[flags[i]])
        assert rc == 0
        if flags[i]:
            rows.append(lb[0])
    assert np.array_equal(la, np.stack(rows))
    for l in range(TINY.n_layer):
        for p in (0, 100, 255, 256, 299):
            assert all(np.array_equal(u, v) for u, v in zip(a.kv_get(0, p, l), b.kv_get(0, p, l)))


def _elision_case(cfg, n_layer, n_tok, flags_at):
    host = synth.make_model(cfg, n_layer=n_layer)
    om = oracle.Model(host)
    toks = synth.prompt_tokens(cfg, n_tok)
    flags = np.zeros(n_tok, np.int8)
    flags[flags_at] = 1
    out = []
    for elide in (True, False):
        c = oracle.Context(om, 512, 1, 512)
        c.set_elide(elide)
        rc, lg, am = c.decode(toks, logits=flags)
        assert rc == 0 and lg.shape[0] == len(flags_at)
        rc2, lg2, am2 = c.decode([int(am[-1])])           # a step that attends the elided tokens' cells
        assert rc2 == 0
        cells = [c.kv_get(0, p, l) for l in range(n_layer) for p in range(n_tok + 1)]
        out.append((lg, am, lg2, am2, cells))
    (la, aa, la2, aa2, ca), (lb, ab, lb2, ab2, cb) = out
    assert np.array_equal(la, lb) and np.array_equal(aa, ab)
    assert np.array_equal(la2, lb2) and np.array_equal(aa2, ab2)
    assert all(np.array_equal(x[0], y[0]) and np.array_equal(x[1], y[1]) for x, y in zip(ca, cb))


def test_last_layer_elision_is_exact_tiny():
    """Unflagged tokens computing only K and V in the last layer changes no logit and no cell."""
    _elision_case(TINY, 2, 20, [0, 9, 19])


def test_last_layer_elision_is_exact_1b_shape():
    _elision_case(synth.CONFIGS["1b"], 16, 10, [3, 9])


@pytest.mark.parametrize("n_threads", [2, 8])
def test_thread_count_changes_nothing(tiny_model, n_threads):
    """The pool's chunking (rows of every product, query heads of attention) must not change a
    bit of the result: the same batch with 1 and with several threads."""
    toks = synth.uniform_int(TINY.token_seed, 78, 70, 0, TINY.n_vocab)
    seqs = np.arange(70) % 3
    res = []
    for n in (1, n_threads):
        oracle.set_threads(n)
        try:
            c = _ctx(tiny_model, n_ctx=256, n_seq=3)
            rc, lg, am = c.decode(toks, seq=seqs, logits=np.ones(70))
            assert rc == 0
            res.append((lg, am, [c.kv_get(s, p, l) for s in range(3) for p in (0, 11, 22) for l in (0, 1)]))
        finally:
            oracle.set_threads(1)
    (la, aa, ca), (lb, ab, cb) = res
    assert np.array_equal(la, lb) and np.array_equal(aa, ab)
    assert all(np.array_equal(x[0], y[0]) and np.array_equal(x[1], y[1]) for x, y in zip(ca, cb))


# ----------------------------------------------------------------------------- a stream per sequence
def test_stream_per_sequence_capacity_and_rows():
    """With a stream per sequence (step 10: the cache is divided by n_ctx_seq = n_ctx / n_seq_max),
    a batch that would give one sequence more than n_ctx_seq cells is refused with 1 and nothing is
    committed; the logits rows come back in batch order and equal those of one shared store (the
    split changes nothing but the order of evaluation)."""
    m = synth.make_model(TINY)
    om = oracle.Model(m)
    c = oracle.Context(om, 256, 2, 4)
    assert c.set_kv_unified(False) == 0
    assert c.decode(np.arange(129) % 50, seq=np.zeros(129, np.int32))[0] == 1    # 129 > 256 / 2
    assert c.seq_pos_max(0) == -1
    assert c.decode(np.arange(128) % 50, seq=np.zeros(128, np.int32))[0] == 0
    assert c.decode([3], seq=[0])[0] == 1 and c.decode([3], seq=[1])[0] == 0
    shared = oracle.Context(om, 256, 2, 4)
    assert shared.decode(np.arange(129) % 50, seq=np.zeros(129, np.int32))[0] == 0   # one store: fits
    # rows in batch order, equal to the shared store's
    toks = synth.prompt_tokens(TINY, 11, 3)
    seqs = np.array([0, 1, 2, 0, 0, 2, 1, 0, 2, 2, 0], np.int32)
    flags = np.array([1, 0, 1, 1, 0, 1, 1, 0, 0, 1, 1], np.int8)
    a = oracle.Context(om, 256, 3, 4)
    a.set_kv_unified(False)
    b = oracle.Context(om, 256, 3, 4)
    ra, rb = a.decode(toks, seq=seqs, logits=flags), b.decode(toks, seq=seqs, logits=flags)
    assert ra[0] == rb[0] == 0 and np.array_equal(ra[1], rb[1]) and np.array_equal(ra[2], rb[2])
    assert c.set_kv_unified(True) == -1                                            # cells held


def test_split_equal_ubatches_by_their_rollback():
    """split_equal with n_ubatch 4 over sequences 0 (5 tokens), 1 (2) and 2 (3): the ubatches are
    {s0p0, s1p0, s2p0}, {s0p1, s1p1, s2p1}, {s0p2, s2p2}, {s0p3, s0p4}. A NaN embedding at s2p1,
    flagged, fails the second ubatch: only the first stays (every sequence back to position 0), no
    rows are reported; a NaN at s0p3 fails the fourth: sequences 1 and 2 complete, 0 keeps 0..2."""
    import dataclasses
    host = synth.make_model(TINY)
    bad = 7
    emb = host.tok_embd.copy()
    emb[bad].view(np.uint16)[:] = 0x7E00
    om = oracle.Model(dataclasses.replace(host, tok_embd=emb))
    seqs = np.array([0, 1, 2, 0, 1, 2, 0, 2, 0, 0], np.int32)      # s0 at 0,3,6,8,9; s1 at 1,4; s2 at 2,5,7
    base = np.array([11, 12, 13, 14, 15, 16, 17, 18, 19, 20], np.int32)
    for where, keep in ((5, (0, 0, 0)), (8, (2, 1, 2))):
        toks = base.copy()
        toks[where] = bad
        c = oracle.Context(om, 256, 3, 4)
        c.set_kv_unified(False)
        rc, lg, _ = c.decode(toks, seq=seqs, logits=np.ones(10, np.int8))
        assert rc == -3 and lg.shape[0] == 0
        assert tuple(c.seq_pos_max(s) for s in range(3)) == keep, (where, keep)
    # the same batch in one shared store (consecutive chunks of 4): the bad token at index 5 fails
    # the second chunk (tokens 4..7); the first chunk's 4 rows stay
    toks = base.copy()
    toks[5] = bad
    c = oracle.Context(om, 256, 3, 4)
    rc, lg, _ = c.decode(toks, seq=seqs, logits=np.ones(10, np.int8))
    assert rc == -3 and lg.shape[0] == 4 and tuple(c.seq_pos_max(s) for s in range(3)) == (1, 0, 0)
