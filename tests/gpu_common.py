"""Shared helpers of the GPU parity tests: device upload, oracle runs, tolerance checks."""
import numpy as np

# Acceptance: per-row relative L2 error of logits <= 5e-3; argmax ids equal wherever the
# oracle's top-1 / top-2 margin exceeds 1e-2.
LOGIT_RTOL = 5e-3
ARGMAX_MARGIN = 1e-2


def rel_l2(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.linalg.norm(gpu - ref, axis=-1) / np.linalg.norm(ref, axis=-1)


def check_rows(gpu_logits, gpu_argmax, ref_logits, ref_argmax, tag=""):
    assert gpu_logits.shape == ref_logits.shape, (tag, gpu_logits.shape, ref_logits.shape)
    err = rel_l2(gpu_logits, ref_logits)
    assert np.all(np.isfinite(gpu_logits)), tag
    assert err.max() <= LOGIT_RTOL, (tag, float(err.max()), int(err.argmax()))
    srt = np.sort(ref_logits, axis=1)
    margin = srt[:, -1] - srt[:, -2]
    sure = margin > ARGMAX_MARGIN
    assert np.array_equal(np.asarray(gpu_argmax)[sure], np.asarray(ref_argmax)[sure]), tag
    return float(err.max())


def gpu_decode(ctx, n_vocab, tokens, pos=None, seq=None, flags=None):
    """Runs lcx_decode with device logits and host argmax; returns (rc, logits, argmax)."""
    import torch
    n = len(tokens)
    n_out = n if flags is None else int(np.count_nonzero(flags))
    if flags is None:
        n_out = 1
    logits = torch.empty((max(n_out, 1), n_vocab), dtype=torch.float32, device="cuda")
    am = np.full(max(n_out, 1), -7, dtype=np.int32)
    rc = ctx.decode(tokens, pos, seq, flags, logits_out=logits, argmax_out=am)
    torch.cuda.synchronize()
    k = ctx.n_outputs()
    return rc, logits[:k].cpu().numpy(), am[:k]
