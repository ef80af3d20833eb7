"""The persistent one-token decode step (one cooperative launch per token).

  * a one-token ubatch is exactly one launch, and the same decode as separate launches
    (LCX_DECODE_STEP=0, read when a context first runs a one-token ubatch) is 5 per layer + 3;
  * with the attention split over dozens of CTAs (tiny model, 1500 cached positions), the step
    matches the oracle;
  * at contexts of 700 and 3000 positions (1B and 8B shapes, several 16-cell groups per warp),
    the step and the separate launches agree: both split each activation block into int8
    hi / lo parts, so a last-bit difference from another summation order can flip a rounding
    and the two drift apart by about 1e-4 over the layers, far inside the 5e-3 oracle bar;
  * the step's in-kernel timeline (trace mode) has one slot per phase, in order.
"""
import os

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


def _ctx(gm, n_ctx, step: bool, n_ubatch=512):
    old = os.environ.get("LCX_DECODE_STEP")
    os.environ["LCX_DECODE_STEP"] = "1" if step else "0"
    try:
        ctx = lcx.Context(gm, n_ctx, 1, n_ubatch)
        # the choice is made at the context's first one-token ubatch: make it now
        assert ctx.decode([1], argmax_out=np.zeros(1, np.int32)) == 0
        ctx.kv_clear()
    finally:
        if old is None:
            del os.environ["LCX_DECODE_STEP"]
        else:
            os.environ["LCX_DECODE_STEP"] = old
    return ctx


def test_one_launch_per_token():
    host = synth.make_model(TINY)
    gm = upload(host)
    om = oracle.Model(host)
    prompt = synth.prompt_tokens(TINY, 16)
    octx = oracle.Context(om, TINY.n_ctx, 1, 512)
    rc, _, am_o = octx.decode(prompt)
    assert rc == 0
    rc, ref, am_ref = octx.decode([int(am_o[0])])
    assert rc == 0
    counts = {}
    for step in (True, False):
        ctx = _ctx(gm, TINY.n_ctx, step)
        assert gpu_decode(ctx, TINY.n_vocab, prompt)[0] == 0
        k0 = ctx.stats().n_kernels
        rc, lg, am = gpu_decode(ctx, TINY.n_vocab, [int(am_o[0])])
        assert rc == 0
        counts[step] = ctx.stats().n_kernels - k0
        check_rows(lg, am, ref, am_ref, f"tiny step={step}")
    assert counts[True] == 1
    assert counts[False] == 5 * TINY.n_layer + 3


def test_step_many_splits_matches_oracle():
    host = synth.make_model(TINY)
    gm = upload(host)
    om = oracle.Model(host)
    n = 1500
    prompt = synth.uniform_int(TINY.token_seed, 900, n, 0, TINY.n_vocab)
    octx = oracle.Context(om, 2048, 1, 512)
    rc, _, am_o = octx.decode(prompt)
    assert rc == 0
    ctx = _ctx(gm, 2048, True)
    assert gpu_decode(ctx, TINY.n_vocab, prompt)[0] == 0
    tok = int(am_o[0])
    for i in range(3):
        rc, ref, am_ref = octx.decode([tok])
        rc2, lg, am = gpu_decode(ctx, TINY.n_vocab, [tok])
        assert rc == rc2 == 0
        check_rows(lg, am, ref, am_ref, f"tiny ctx {n} step {i}")
        tok = int(am_ref[0])


def _step_vs_launches(cfg, n_prompt, n_steps, n_ctx, n_ubatch):
    host = synth.make_model(cfg)
    gm = upload(host)
    prompt = synth.prompt_tokens(cfg, n_prompt)
    out = {}
    for step in (True, False):
        ctx = _ctx(gm, n_ctx, step, n_ubatch)
        rc, lg, am = gpu_decode(ctx, cfg.n_vocab, prompt)
        assert rc == 0
        rows, toks = [], []
        tok = int(am[0])
        for _ in range(n_steps):
            rc, l1, a1 = gpu_decode(ctx, cfg.n_vocab, [tok])
            assert rc == 0
            rows.append(l1[0])
            tok = int(a1[0])
            toks.append(tok)
        # and the on-device greedy loop, which chains the steps' argmax on the device
        g = torch.full((4,), -1, dtype=torch.int32, device="cuda")
        assert ctx.decode_greedy(0, tok, 4, g) == 0
        out[step] = (np.stack(rows), toks, g.cpu().numpy().tolist())
        ctx.close()
    (ls, ts, gs), (ll, tl, gl) = out[True], out[False]
    err = rel_l2(ls, ll)
    assert err.max() <= 2e-3, err
    srt = np.sort(ll, axis=1)
    sure = (srt[:, -1] - srt[:, -2]) > 1e-2
    assert np.array_equal(np.array(ts)[sure], np.array(tl)[sure])
    if sure.all():
        assert gs == gl
    return float(err.max())


def test_step_matches_launches_1b_context_700():
    print("1b step vs launches", _step_vs_launches(synth.CONFIGS["1b"], 700, 4, 4096, 512))


def test_step_matches_launches_8b_context_3000():
    print("8b step vs launches", _step_vs_launches(synth.CONFIGS["8b"], 3000, 3, 8192, 512))


def test_step_timeline_slots():
    host = synth.make_model(TINY)
    gm = upload(host)
    ctx = _ctx(gm, TINY.n_ctx, True)
    assert gpu_decode(ctx, TINY.n_vocab, synth.prompt_tokens(TINY, 8))[0] == 0
    assert ctx.set_profiling(2) == 0
    assert gpu_decode(ctx, TINY.n_vocab, [5])[0] == 0
    tr = ctx.trace().astype(np.float64)
    assert tr.shape[0] == 5 * TINY.n_layer + 2
    # slot 0 (embedding) has no staging; every other phase: first in <= first staged <= last
    # staged <= last done, and each phase starts after the previous one started
    ph = tr[1:]
    assert np.all(ph[:, 0] <= ph[:, 1]) and np.all(ph[:, 1] <= ph[:, 2]) and np.all(ph[:, 2] <= ph[:, 3])
    assert tr[0, 0] <= tr[0, 3]
    assert np.all(np.diff(tr[:, 0]) >= 0)
    assert ctx.set_profiling(False) == 0
