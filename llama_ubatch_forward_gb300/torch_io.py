"""Moves a host model in stored form (uint8 block rows, float32 gains) onto the device with
PyTorch and builds an lcx Model over it. Marshalling only: no arithmetic of the forward."""
from __future__ import annotations

import numpy as np

from . import Model, lcx_hparams

LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


def hparams_of(cfg, n_layer: int | None = None) -> lcx_hparams:
    return lcx_hparams(cfg.n_vocab, cfg.n_embd, cfg.n_layer if n_layer is None else n_layer, cfg.n_head,
                       cfg.n_head_kv, cfg.head_dim, cfg.n_ff, cfg.rms_eps, cfg.rope_theta, cfg.t_linear,
                       cfg.t_embd, cfg.t_out)


def to_device(a: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def upload(host, device="cuda") -> Model:
    """host: an object with cfg, tok_embd, output_norm, output (or None) and layers (dicts).

    Matrices are uploaded one layer at a time and released once the model holds its own
    re-laid-out copy; the embedding table and the norm gains stay referenced by the model."""
    import torch
    tok = to_device(host.tok_embd, device)
    on = to_device(host.output_norm, device)
    out = None if host.output is None else to_device(host.output, device)
    layers = [{k: to_device(L[k], device) for k in LAYER_KEYS} for L in host.layers]
    m = Model(hparams_of(host.cfg, len(host.layers)), tok, on, out, layers)
    torch.cuda.synchronize()
    # keep only what the model reads in place
    m._keep = (tok, on, None, [{"attn_norm": L["attn_norm"], "ffn_norm": L["ffn_norm"]} for L in layers])
    del layers, out
    return m
