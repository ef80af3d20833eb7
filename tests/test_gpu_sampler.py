"""lcx_sample (the sampler chain on the device) against the sampler oracle, through the C ABI.

Rows of synthetic logits with the shape of the model's output (128256 entries, a few strong
candidates over a wide normal background) and small vocabularies with a ragged length. For every
row the GPU token must be one the oracle returns when each floating-point decision (the top-p
target, the min-p threshold, the draw target) moves by at most 1e-4 of its size; away from those
boundaries that set is the single oracle token. Greedy and top-k = 1 are compared exactly, and the
draw's frequencies over a grid of random numbers are compared with the softmax probabilities."""
import math

import numpy as np
import pytest

import synth
from oracle import sampler as S

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_ubatch_forward_gb300 as lcx  # noqa: E402


def logits_rows(seed, n_rows, V, peak=8.0, n_peak=6, ties=False):
    x = synth.normal(seed, 1, n_rows * V, 0.0, 2.0).reshape(n_rows, V)
    ids = synth.uniform_int(seed, 2, n_rows * n_peak, 0, V).reshape(n_rows, n_peak)
    for r in range(n_rows):
        x[r, ids[r]] += peak * (1.0 + np.arange(n_peak) / n_peak)
    if ties:
        x = np.round(x)
    return x.astype(np.float32)


def uniforms(seed, n):
    return (synth.uniform_int(seed, 3, n, 0, 1 << 24) / float(1 << 24)).astype(np.float32)


def run(x, u=None, hist=None, **prm):
    lcx.build()
    dx = torch.from_numpy(x).cuda()
    du = None if u is None else torch.from_numpy(u).cuda()
    dh = None if hist is None else torch.from_numpy(np.ascontiguousarray(hist, dtype=np.int32)).cuda()
    rc, out = lcx.sample(dx, du, dh, **prm)
    torch.cuda.synchronize()
    assert rc == 0, lcx.lib().lcx_last_error()
    return out.cpu().numpy()


CHAINS = [
    dict(top_k=40, top_p=0.95, min_p=0.05, temp=0.8),   # a common console default
    dict(top_k=0, top_p=0.9, temp=1.0),                 # top-p over the whole vocabulary
    dict(min_p=0.1, temp=1.5),
    dict(temp=1.0),                                     # the plain softmax draw
    dict(top_k=1000, top_p=0.5, temp=0.7),
    dict(top_k=7, temp=2.0),
]


@pytest.mark.parametrize("ci", range(len(CHAINS)))
@pytest.mark.parametrize("V", [128256, 1000])
def test_chain_matches_oracle(ci, V):
    prm = CHAINS[ci]
    n = 8
    x = logits_rows(100 + ci, n, V)
    u = uniforms(200 + ci, n)
    got = run(x, u, **prm)
    exact = 0
    for r in range(n):
        ok = S.acceptable_tokens(x[r], u=float(u[r]), **prm)
        assert int(got[r]) in ok, (r, int(got[r]), sorted(ok)[:8])
        if len(ok) == 1:
            exact += 1
    assert exact >= n // 2   # most rows are far from every boundary


@pytest.mark.parametrize("V", [128256, 513])
def test_greedy_and_top1_are_argmax(V):
    x = logits_rows(7, 6, V, ties=True)   # integer logits: many ties, the lowest id must win
    want = x.argmax(axis=1)
    assert np.array_equal(run(x, None, temp=0.0), want)
    assert np.array_equal(run(x, uniforms(8, 6), top_k=1, temp=0.9), want)


def test_repeat_penalty_and_ties():
    V, n, nh = 128256, 6, 64
    x = logits_rows(11, n, V, ties=True)
    hist = synth.uniform_int(12, 4, n * nh, -5, V).reshape(n, nh)
    hist[:, :3] = x.argmax(axis=1)[:, None]            # the leader is in the history
    u = uniforms(13, n)
    for prm in (dict(penalty_repeat=1.3, top_k=50, temp=0.9), dict(penalty_repeat=1.3, temp=0.0),
                dict(penalty_repeat=0.7, top_k=20, top_p=0.8, temp=1.0)):
        got = run(x, u, hist, **prm)
        for r in range(n):
            ok = S.acceptable_tokens(x[r], hist[r], u=float(u[r]), **prm)
            assert int(got[r]) in ok, (prm, r, int(got[r]), sorted(ok)[:8])


def test_draw_frequencies_match_softmax():
    V, n = 16, 4096
    base = logits_rows(21, 1, V, peak=2.0, n_peak=3)[0]
    x = np.repeat(base[None, :], n, axis=0)
    u = ((np.arange(n) + 0.5) / n).astype(np.float32)
    for T in (1.0, 0.6):
        got = run(x, u, temp=T)
        f = np.bincount(got, minlength=V) / n
        p = np.exp((base.astype(np.float64) - base.max()) / T)
        p /= p.sum()
        assert np.all(np.abs(f - p) <= 2.0 / n), (T, np.abs(f - p).max())


def test_edges_and_invalid_arguments():
    one = np.array([[0.25]], np.float32)
    assert run(one, np.array([0.999], np.float32), top_k=5, top_p=0.1, min_p=0.5, temp=1.0)[0] == 0
    x = torch.zeros((2, 8), dtype=torch.float32, device="cuda")
    u = torch.zeros(2, dtype=torch.float32, device="cuda")
    assert lcx.sample(x, None, temp=1.0)[0] == lcx.LCX_INVALID             # a draw needs u
    assert lcx.sample(x, u, penalty_repeat=0.0)[0] == lcx.LCX_INVALID       # penalty must be > 0
    big = torch.zeros((1, (1 << 18) + 1), dtype=torch.float32, device="cuda")
    assert lcx.sample(big, u[:1], temp=0.0)[0] == lcx.LCX_INVALID           # vocabulary limit
    assert lcx.sample(x[:0], u[:0], temp=1.0)[0] == 0                       # no rows: nothing to do


def test_on_decode_logits_greedy_equals_forward_argmax():
    from llama_ubatch_forward_gb300.torch_io import upload
    cfg = synth.CONFIGS["tiny"]
    host = synth.make_model(cfg)
    gm = upload(host)
    ctx = lcx.Context(gm, cfg.n_ctx, 1, 512)
    prompt = synth.prompt_tokens(cfg, 12)
    logits = torch.empty((12, cfg.n_vocab), dtype=torch.float32, device="cuda")
    am = np.zeros(12, dtype=np.int32)
    assert ctx.decode(prompt, logits=np.ones(12), logits_out=logits, argmax_out=am) == 0
    rc, tok = lcx.sample(logits, None, temp=0.0)
    torch.cuda.synchronize()
    assert rc == 0 and np.array_equal(tok.cpu().numpy(), am)
    u = torch.from_numpy(uniforms(31, 12)).cuda()
    rc, tok = lcx.sample(logits, u, top_k=40, top_p=0.95, min_p=0.05, temp=0.8)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    for r in range(12):
        ok = S.acceptable_tokens(lg[r], u=float(u[r]), top_k=40, top_p=0.95, min_p=0.05, temp=0.8)
        assert int(tok[r]) in ok
    assert math.isfinite(float(lg.max()))
