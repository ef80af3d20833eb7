"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle on the same seeded inputs.

Covers the tiny model end to end (prefill in one and in several ubatches, teacher-forced and
on-device greedy decode, several sequences, return codes), and prefixes of the 1B-shape and
8B-shape models in the launch configuration the benchmark uses.
"""
import numpy as np
import pytest

import oracle
import synth

from gpu_common import check_rows, gpu_decode, rel_l2

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_ubatch_forward_gb300 as lcx  # noqa: E402
from llama_ubatch_forward_gb300.torch_io import upload  # noqa: E402

TINY = synth.CONFIGS["tiny"]


@pytest.fixture(scope="module", autouse=True)
def setup():
    lcx.build()
    oracle.set_threads()


@pytest.fixture(scope="module")
def tiny():
    host = synth.make_model(TINY)
    return host, upload(host), oracle.Model(host)


# ------------------------------------------------------------------ dequant rows: bit exact
@pytest.mark.parametrize("qtype", [synth.F16, synth.Q8_0, synth.Q4_0])
def test_get_rows_bit_exact(qtype):
    n_rows, n_cols = 300, 4096
    w = synth.normal(77, qtype, n_rows * n_cols, 0.0, 0.02).reshape(n_rows, n_cols)
    w[5] *= 1e-3                                     # small scales, incl. subnormal f16 scales
    rows = synth.encode(w, qtype)
    ids = synth.uniform_int(78, qtype, 257, 0, n_rows)
    ids[:3] = [0, n_rows - 1, 5]
    out = torch.empty((ids.size, n_cols), dtype=torch.float32, device="cuda")
    rc = lcx.get_rows(qtype, torch.from_numpy(rows).cuda(), n_rows, n_cols, torch.from_numpy(ids).cuda(), out)
    torch.cuda.synchronize()
    assert rc == 0
    got = out.cpu().numpy().astype(np.float64)
    for i, r in enumerate(ids):
        assert np.array_equal(got[i], oracle.dequant_row(qtype, rows[r], n_cols)), i


# ------------------------------------------------------------------ tiny workload
def _oracle_greedy(octx, prompt, n_steps):
    rc, lg, am = octx.decode(prompt, logits=np.ones(len(prompt)))
    assert rc == 0
    toks, rows = [int(am[-1])], [lg]
    for _ in range(n_steps - 1):
        rc, l1, a1 = octx.decode([toks[-1]])
        assert rc == 0
        rows.append(l1)
        toks.append(int(a1[0]))
    return np.concatenate(rows), toks


@pytest.mark.parametrize("n_ubatch", [512, 5])
def test_tiny_prefill_and_decode(tiny, n_ubatch):
    host, gm, om = tiny
    prompt = synth.prompt_tokens(TINY, 16)
    octx = oracle.Context(om, TINY.n_ctx, 1, n_ubatch)
    ref, toks = _oracle_greedy(octx, prompt, 16)
    ctx = lcx.Context(gm, TINY.n_ctx, 1, n_ubatch)
    rc, lg, am = gpu_decode(ctx, TINY.n_vocab, prompt, flags=np.ones(16))
    assert rc == 0
    rows, ams = [lg], [am]
    for t in toks[:-1]:                                # teacher-forced with the oracle's tokens
        rc, l1, a1 = gpu_decode(ctx, TINY.n_vocab, [t])
        assert rc == 0
        rows.append(l1)
        ams.append(a1)
    check_rows(np.concatenate(rows), np.concatenate(ams), ref, np.argmax(ref, axis=1), f"tiny ub={n_ubatch}")
    assert ctx.seq_pos_max(0) == octx.seq_pos_max(0) == 16 + 15 - 1


def test_tiny_greedy_on_device(tiny):
    host, gm, om = tiny
    prompt = synth.prompt_tokens(TINY, 16)
    octx = oracle.Context(om, TINY.n_ctx, 1, 512)
    ref, toks = _oracle_greedy(octx, prompt, 17)
    ctx = lcx.Context(gm, TINY.n_ctx, 1, 512)
    rc, lg, am = gpu_decode(ctx, TINY.n_vocab, prompt)
    assert rc == 0
    out = torch.full((16,), -1, dtype=torch.int32, device="cuda")
    assert ctx.decode_greedy(0, int(am[0]), 16, out) == 0
    gen = out.cpu().numpy().tolist()
    # each generated token is the argmax of the previous step: compare while margins are clear
    srt = np.sort(ref[15:], axis=1)
    margins = srt[:, -1] - srt[:, -2]
    for i in range(16):
        if margins[i + 1] <= 1e-2:
            break
        assert gen[i] == toks[i + 1], (i, gen, toks)
    host_out = np.zeros(4, dtype=np.int32)             # host output buffer variant
    assert ctx.decode_greedy(0, gen[-1], 4, host_out) == 0
    assert ctx.seq_pos_max(0) == 16 + 16 + 4 - 1


def test_tiny_multi_sequence(tiny):
    host, gm, om = tiny
    p = [synth.prompt_tokens(TINY, n, s) for s, n in enumerate((5, 9, 3))]
    toks, seqs = [], []
    for i in range(9):
        for s in range(3):
            if i < len(p[s]):
                toks.append(int(p[s][i]))
                seqs.append(s)
    flags = np.ones(len(toks), np.int8)
    octx = oracle.Context(om, TINY.n_ctx, 3, 512)
    ctx = lcx.Context(gm, TINY.n_ctx, 3, 4)
    rc_o, ref, am_o = octx.decode(toks, seq=seqs, logits=flags)
    rc, lg, am = gpu_decode(ctx, TINY.n_vocab, toks, seq=seqs, flags=flags)
    assert rc == rc_o == 0
    check_rows(lg, am, ref, am_o, "multi-seq prefill")
    # one decode step for all three sequences in one ubatch
    nxt = [7, 11, 13]
    rc_o, ref, am_o = octx.decode(nxt, seq=[2, 0, 1], logits=np.ones(3))
    rc, lg, am = gpu_decode(ctx, TINY.n_vocab, nxt, seq=[2, 0, 1], flags=np.ones(3))
    assert rc == rc_o == 0
    check_rows(lg, am, ref, am_o, "multi-seq decode")


def test_tiny_return_codes(tiny):
    host, gm, om = tiny
    ctx = lcx.Context(gm, 128, 2, 64)
    assert gpu_decode(ctx, TINY.n_vocab, [TINY.n_vocab])[0] == -1
    assert gpu_decode(ctx, TINY.n_vocab, [1], seq=[2])[0] == -1
    assert gpu_decode(ctx, TINY.n_vocab, np.arange(257) % 7)[0] == 1      # n_ctx 128 -> 256 cells
    assert ctx.seq_pos_max(0) == -1
    assert gpu_decode(ctx, TINY.n_vocab, np.arange(256) % 7)[0] == 0
    assert gpu_decode(ctx, TINY.n_vocab, [1])[0] == 1
    ctx.kv_clear()
    rc, lg, am = gpu_decode(ctx, TINY.n_vocab, [3, 4])
    octx = oracle.Context(om, 128, 2, 64)
    rc_o, ref, am_o = octx.decode([3, 4])
    assert rc == rc_o == 0
    check_rows(lg, am, ref, am_o, "after clear")


def test_prefill_matches_stepwise_decode_on_gpu(tiny):
    host, gm, om = tiny
    prompt = synth.prompt_tokens(TINY, 12)
    a = lcx.Context(gm, 128, 1, 512)
    _, la, _ = gpu_decode(a, TINY.n_vocab, prompt, flags=np.ones(12))
    b = lcx.Context(gm, 128, 1, 512)
    rows = [gpu_decode(b, TINY.n_vocab, [t])[1][0] for t in prompt]
    assert rel_l2(la, np.stack(rows)).max() <= 2e-3


# ------------------------------------------------------------------ larger shapes
def _prefix_parity(cfg, n_prompt, n_decode, n_ubatch, n_ctx):
    host = synth.make_model(cfg)
    om = oracle.Model(host)
    gm = upload(host)
    prompt = synth.prompt_tokens(cfg, n_prompt)
    octx = oracle.Context(om, n_ctx, 1, n_ubatch)
    flags = np.zeros(n_prompt, np.int8)
    flags[[0, n_prompt // 2, n_prompt - 1]] = 1
    rc, ref0, am0 = octx.decode(prompt, logits=flags)
    assert rc == 0
    ctx = lcx.Context(gm, n_ctx, 1, n_ubatch)
    rc, lg, am = gpu_decode(ctx, cfg.n_vocab, prompt, flags=flags)
    assert rc == 0
    errs = [check_rows(lg, am, ref0, am0, f"{cfg.name} prefill")]
    tok = int(am0[-1])
    for i in range(n_decode):
        rc, ref1, am1 = octx.decode([tok])
        rc2, l1, a1 = gpu_decode(ctx, cfg.n_vocab, [tok])
        assert rc == rc2 == 0
        errs.append(check_rows(l1, a1, ref1, am1, f"{cfg.name} decode {i}"))
        tok = int(am1[0])
    return errs


def test_8b_prefix():
    errs = _prefix_parity(synth.CONFIGS["8b"], 12, 3, 512, 8192)
    print("8b rel errors", errs)


def test_tiny_stream_per_sequence(tiny):
    """A stream per sequence: split_equal ubatches whose flagged rows are not consecutive in the
    batch (written through the scratch and copied to their batch-order rows), host and device
    argmax, against the oracle run the same way."""
    host, gm, om = tiny
    toks = synth.uniform_int(TINY.token_seed, 555, 23, 0, TINY.n_vocab)
    seqs = np.array([0, 1, 2, 0, 0, 2, 1, 0, 2, 2, 0, 1, 1, 2, 0, 0, 1, 2, 2, 0, 1, 0, 2], np.int32)
    flags = (synth.uniform_int(TINY.token_seed, 556, 23, 0, 3) > 0).astype(np.int8)
    octx = oracle.Context(om, 384, 3, 4)
    assert octx.set_kv_unified(False) == 0
    ctx = lcx.Context(gm, 384, 3, 4)
    assert ctx.set_kv_unified(False) == 0
    rc_o, ref, am_o = octx.decode(toks, seq=seqs, logits=flags)
    rc, lg, am = gpu_decode(ctx, TINY.n_vocab, toks, seq=seqs, flags=flags)
    assert rc == rc_o == 0
    check_rows(lg, am, ref, am_o, "split_equal prefill")
    # one step for every sequence, device argmax
    nxt = np.array([5, 6, 7], np.int32)
    rc_o, ref, am_o = octx.decode(nxt, seq=[1, 2, 0], logits=np.ones(3))
    out = torch.full((3, TINY.n_vocab), float("nan"), dtype=torch.float32, device="cuda")
    amd = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    assert ctx.decode(nxt, seq_id=[1, 2, 0], logits=np.ones(3), logits_out=out, argmax_out=amd) == 0
    torch.cuda.synchronize()
    check_rows(out.cpu().numpy(), amd.cpu().numpy(), ref, am_o, "split_equal step")
    for s in range(3):
        assert ctx.seq_pos_max(s) == octx.seq_pos_max(s)
