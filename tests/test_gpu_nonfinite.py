"""A logits row holding a value that is not finite fails its ubatch on the GPU as in the oracle.

The input is made on the host: one token's f16 embedding row is all NaN. Its K and V carry the NaN
into the cache, and every later token of its sequence that attends them gets NaN logits. The
library must then do what the oracle does (the article's decode loop, step 12: a failed compute
returns -3 after the failed ubatch's positions are rolled back; the ubatches already run stay,
with the rows copied out before the failure): return LCX_COMPUTE_FAILED, release the cells of the
failed and later ubatches, and report only the rows of the earlier ones -- on every logits path
(the weight-streaming GEMV head, the persistent one-token step, the tensor-core GEMM head and the
on-device greedy loop).
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth

from gpu_common import check_rows, gpu_decode

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_ubatch_forward_gb300 as lcx  # noqa: E402
from llama_ubatch_forward_gb300.torch_io import upload  # noqa: E402

TINY = synth.CONFIGS["tiny"]
BAD = 7


@pytest.fixture(scope="module")
def models():
    lcx.build()
    host = synth.make_model(TINY)
    emb = host.tok_embd.copy()
    emb[BAD].view(np.uint16)[:] = 0x7E00                # an f16 NaN row
    bad = dataclasses.replace(host, tok_embd=emb)
    return upload(bad), oracle.Model(bad)


def _both(models, n_ubatch, n_ctx=TINY.n_ctx):
    gm, om = models
    return lcx.Context(gm, n_ctx, 1, n_ubatch), oracle.Context(om, n_ctx, 1, n_ubatch)


def _compare(ctx, octx, toks, flags):
    rc_o, ref, am_o = octx.decode(toks, logits=flags)
    rc, lg, am = gpu_decode(ctx, TINY.n_vocab, toks, flags=flags)
    assert rc == rc_o, (rc, rc_o)
    assert ctx.n_outputs() == ref.shape[0], (ctx.n_outputs(), ref.shape[0])
    assert ctx.seq_pos_max(0) == octx.seq_pos_max(0)
    if ref.shape[0]:
        check_rows(lg, am, ref, am_o, "rows kept")
    return rc


def test_own_ubatch_fails_gemv_head(models):
    ctx, octx = _both(models, 2)
    assert _compare(ctx, octx, [1, BAD], [1, 1]) == -3
    assert ctx.seq_pos_max(0) == -1


def test_later_ubatch_fails_on_the_persistent_step(models):
    # ubatches [1, 2] [3, bad] [5]: token 5 (a one-token ubatch: the persistent step) attends the
    # NaN cell; the first ubatch's row stays
    ctx, octx = _both(models, 2)
    assert _compare(ctx, octx, [1, 2, 3, BAD, 5], [0, 1, 0, 0, 1]) == -3
    assert ctx.n_outputs() == 1 and ctx.seq_pos_max(0) == 3
    assert _compare(ctx, octx, [9], [1]) == -3          # the NaN cell is still attended
    assert ctx.seq_pos_max(0) == 3


def test_tensor_core_head_rows_of_earlier_ubatch_stay(models):
    # ubatches of 16 tokens, every row flagged: the head runs as the tensor-core GEMM; the bad
    # token sits in the second ubatch
    toks = synth.uniform_int(TINY.token_seed, 901, 40, 0, TINY.n_vocab)
    toks[toks == BAD] = BAD + 1
    toks[21] = BAD
    ctx, octx = _both(models, 16)
    assert _compare(ctx, octx, toks, np.ones(40, np.int8)) == -3
    assert ctx.n_outputs() == 16 and ctx.seq_pos_max(0) == 15
    # the cache goes on from position 16, clean
    rc = _compare(ctx, octx, toks[22:30], np.ones(8, np.int8))
    assert rc == 0 and ctx.seq_pos_max(0) == 23


def test_greedy_loop_stops_at_the_failing_step(models):
    ctx, octx = _both(models, 512)
    assert _compare(ctx, octx, [1, BAD], [0, 0]) == 0   # no rows: nothing to check yet
    out = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    assert ctx.decode_greedy(0, 5, 4, out) == lcx.LCX_COMPUTE_FAILED
    assert ctx.n_outputs() == 0 and ctx.seq_pos_max(0) == 1
    assert octx.decode([5])[0] == -3 and octx.seq_pos_max(0) == 1
    # a clean sequence runs its steps to the end
    ctx2, octx2 = _both(models, 512)
    assert _compare(ctx2, octx2, [1, 2, 3], [0, 0, 1]) == 0
    host_out = np.full(3, -1, np.int32)
    assert ctx2.decode_greedy(0, 4, 3, host_out) == 0 and ctx2.n_outputs() == 3
