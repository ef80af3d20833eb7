"""Every compiled tile shape of the prefill tensor-core GEMM, checked against the oracle.

The GEMM's cost model picks one tile shape per launch (bn tokens x mt 128-row weight tiles, K
steps split over ks CTAs), so a shape that the named workloads never pick would go unchecked;
lcx_set_gemm_tile forces each shape in turn. The model has dimensions of its own -- d 512, FFN
1536, 8 query and 2 KV heads of 64, vocabulary 1024, 2 layers; K = 512 (8 K steps of 64) for the
Q/K/V, output, gate/up projections and the head, K = 1536 (24 steps) for the down projection --
with Q4_0 and with Q8_0 weights. A 300-token prompt runs as one ubatch (300 = 2 x 128 + 44: whole
token tiles and a ragged tail under every bn) with 40 rows flagged, so every epilogue (Q/K/V with
RoPE and the KV append, residual add, SwiGLU, logits with argmax) runs under every shape, and
rows past N (padding of the weight tiles) are read. Each forced shape must meet the acceptance
bar against the oracle and agree with the cost model's own choice up to summation order.
"""
import dataclasses

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

BASE = dataclasses.replace(synth.CONFIGS["tiny"], name="gemm-shapes", index=11, n_vocab=1024, n_embd=512,
                           n_head=8, n_head_kv=2, head_dim=64, n_ff=1536, n_ctx=512)
T = 300
FLAGGED = np.sort(np.random.default_rng(5).choice(T, 40, replace=False))
# (bn, mt, ks): the five compiled shapes, and splits of the K steps (ks 3 applies to the down
# projection's 24 steps only: 8 steps in 3 splits leave fewer than 4 a split, so those run whole);
# 64 x 2 runs with the operands swapped (the sums transposed through shared memory), also split;
# 6 splits of the down projection (and 3 with Q8_0 at 64 x 2) stage the other splits' partial
# sums in batches
SHAPES = [(64, 1, 1), (64, 2, 1), (128, 1, 1), (128, 2, 1), (256, 1, 1), (128, 2, 2), (64, 1, 3), (256, 1, 2),
          (64, 2, 2), (64, 2, 3), (128, 2, 6)]

_cache = {}


def _setup(qtype):
    if qtype not in _cache:
        lcx.build()
        oracle.set_threads()
        cfg = dataclasses.replace(BASE, t_linear=qtype, t_out=qtype)
        host = synth.make_model(cfg)
        prompt = synth.prompt_tokens(cfg, T)
        flags = np.zeros(T, np.int8)
        flags[FLAGGED] = 1
        om = oracle.Model(host)
        octx = oracle.Context(om, cfg.n_ctx, 1, 512)
        rc, ref, am = octx.decode(prompt, logits=flags)
        assert rc == 0
        gm = upload(host)
        ctx = lcx.Context(gm, cfg.n_ctx, 1, 512)
        assert lcx.set_gemm_tile(0) == 0
        rc, lg, am2 = gpu_decode(ctx, cfg.n_vocab, prompt, flags=flags)
        assert rc == 0
        check_rows(lg, am2, ref, am, "cost model's shapes")
        _cache[qtype] = (cfg, gm, prompt, flags, ref, am, lg)
    return _cache[qtype]


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0], ids=["q4_0", "q8_0"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"{b}x{m}k{k}" for b, m, k in SHAPES])
def test_forced_tile_shape(qtype, shape):
    cfg, gm, prompt, flags, ref, am, lg_default = _setup(qtype)
    ctx = lcx.Context(gm, cfg.n_ctx, 1, 512)
    assert lcx.set_gemm_tile(*shape) == 0
    try:
        k0 = ctx.stats().n_kernels
        rc, lg, am2 = gpu_decode(ctx, cfg.n_vocab, prompt, flags=flags)
        assert ctx.stats().n_kernels > k0
    finally:
        lcx.set_gemm_tile(0)
    assert rc == 0
    check_rows(lg, am2, ref, am, f"tile {shape}")
    # the same arithmetic as the cost model's shapes but for the order of the f32 sums
    assert rel_l2(lg, lg_default).max() <= 1e-4, shape
