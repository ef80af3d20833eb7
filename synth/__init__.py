"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

Holds no arithmetic of the forward itself: it draws normal weights, norm gains and token ids
from a counter-based generator and encodes weights into the stored block formats (Q8_0, Q4_0,
F16) that a model file would hold. The C source (``synth.c``) documents the generator and the
encodings; this module compiles it on first use and wraps it with numpy.

Model shapes follow the five workloads the forward is measured on: a tiny Llama-style decoder,
a 1B-shape and an 8B-shape Llama, long-context decode on the 8B shape and 64-sequence batched
decode on the 8B shape.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libsynth.so")
_lib = None

# block type ids (the same numbering the C ABI uses for lcx_type)
F16, Q4_0, Q8_0 = 1, 2, 8
BLOCK_BYTES = {Q8_0: 34, Q4_0: 18}


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        i64, u64, i32, f32, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
        L.synth_draw_u64.restype = u64
        L.synth_draw_u64.argtypes = [u64, u64, u64]
        L.synth_normal_f32.argtypes = [u64, u64, i64, f32, f32, vp, i32]
        L.synth_uniform_i32.argtypes = [u64, u64, i64, ctypes.c_int32, ctypes.c_int32, vp]
        L.synth_encode_q8_0.argtypes = [vp, i64, i64, i64, vp, i32]
        L.synth_encode_q4_0.argtypes = [vp, i64, i64, i64, vp, i32]
        L.synth_encode_f16.argtypes = [vp, i64, vp, i32]
        L.synth_f32_to_f16.restype = ctypes.c_uint16
        L.synth_f32_to_f16.argtypes = [f32]
        _lib = L
    return _lib


def _threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def normal(seed: int, tid: int, n: int, mean: float, std: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().synth_normal_f32(seed, tid, n, mean, std, _ptr(out), _threads())
    return out


def uniform_int(seed: int, tid: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    lib().synth_uniform_i32(seed, tid, n, lo, hi, _ptr(out))
    return out


def row_bytes(qtype: int, k: int) -> int:
    """Bytes of one stored row of k elements (block types pad k up to a multiple of 32)."""
    if qtype == F16:
        return 2 * k
    return ((k + 31) // 32) * BLOCK_BYTES[qtype]


def encode(w: np.ndarray, qtype: int) -> np.ndarray:
    """Encode a row-major f32 matrix [n_rows, k] into stored rows (uint8 [n_rows, row_bytes])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n_rows, k = w.shape
    if qtype == F16:
        out = np.empty((n_rows, k), dtype=np.uint16)
        lib().synth_encode_f16(_ptr(w), n_rows * k, _ptr(out), _threads())
        return out.view(np.uint8).reshape(n_rows, 2 * k)
    k_pad = ((k + 31) // 32) * 32
    out = np.empty((n_rows, row_bytes(qtype, k)), dtype=np.uint8)
    fn = lib().synth_encode_q8_0 if qtype == Q8_0 else lib().synth_encode_q4_0
    fn(_ptr(w), n_rows, k, k_pad, _ptr(out), _threads())
    return out


def f32_to_f16_bits(x: float) -> int:
    return int(lib().synth_f32_to_f16(float(x)))


# ------------------------------------------------------------------------------------ configs

@dataclass(frozen=True)
class Config:
    name: str
    index: int
    n_vocab: int
    n_embd: int
    n_layer: int
    n_head: int
    n_head_kv: int
    head_dim: int
    n_ff: int
    rope_theta: float
    n_ctx: int
    t_linear: int
    t_embd: int
    t_out: int
    rms_eps: float = 1e-5

    @property
    def weight_seed(self) -> int:
        return 0x1CC0 + self.index

    @property
    def token_seed(self) -> int:
        return 0x70C0 + self.index


CONFIGS = {
    "tiny": Config("tiny", 0, 512, 256, 2, 4, 2, 64, 688, 10000.0, 128, Q8_0, F16, Q8_0),
    "1b": Config("1b", 1, 128256, 2048, 16, 32, 8, 64, 8192, 500000.0, 4096, Q8_0, Q8_0, Q8_0),
    "8b": Config("8b", 2, 128256, 4096, 32, 32, 8, 128, 14336, 500000.0, 8192, Q4_0, Q8_0, Q8_0),
    "long": Config("long", 3, 128256, 4096, 32, 32, 8, 128, 14336, 500000.0, 32896, Q4_0, Q8_0, Q8_0),
    "multiseq": Config("multiseq", 4, 128256, 4096, 32, 32, 8, 128, 14336, 500000.0, 262144, Q4_0, Q8_0, Q8_0),
}

# tensor ids of the counter-based draw
TID_TOK_EMBD, TID_OUTPUT_NORM, TID_OUTPUT = 0, 1, 2
LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


def layer_tid(layer: int, name: str) -> int:
    return 16 + 16 * layer + LAYER_TENSORS.index(name)


def matrix_shape(cfg: Config, name: str) -> tuple[int, int]:
    """(rows N, row length K) of a layer matrix: row n holds the K input weights of output n."""
    d, hd = cfg.n_embd, cfg.head_dim
    return {
        "wq": (cfg.n_head * hd, d),
        "wk": (cfg.n_head_kv * hd, d),
        "wv": (cfg.n_head_kv * hd, d),
        "wo": (d, cfg.n_head * hd),
        "w_gate": (cfg.n_ff, d),
        "w_up": (cfg.n_ff, d),
        "w_down": (d, cfg.n_ff),
    }[name]


@dataclass
class Model:
    """A synthetic model as host arrays in stored form (the bytes the forward reads)."""
    cfg: Config
    tok_embd: np.ndarray            # uint8 [V, row_bytes(t_embd, d)]
    output_norm: np.ndarray         # float32 [d]
    output: np.ndarray | None       # uint8 [V, row_bytes(t_out, d)] or None (tied to tok_embd)
    layers: list = field(default_factory=list)   # dicts: norms float32 [d], matrices uint8 [N, row_bytes]

    def weight_bytes(self) -> int:
        n = self.tok_embd.nbytes + self.output_norm.nbytes + (self.output.nbytes if self.output is not None else 0)
        for L in self.layers:
            n += sum(v.nbytes for v in L.values())
        return n


def make_model(cfg: Config, zero: tuple[str, ...] = (), n_layer: int | None = None,
               tied: bool = False) -> Model:
    """Draw and encode every tensor of `cfg`.

    `zero` names layer tensors (as in LAYER_TENSORS) whose weights are set to exactly zero;
    `n_layer` overrides the layer count (a prefix of the same draws); `tied` drops `output`.
    """
    s = cfg.weight_seed
    d, V = cfg.n_embd, cfg.n_vocab
    emb = normal(s, TID_TOK_EMBD, V * d, 0.0, 0.02).reshape(V, d)
    tok_embd = encode(emb, cfg.t_embd)
    del emb
    out_norm = normal(s, TID_OUTPUT_NORM, d, 1.0, 0.02)
    output = None
    if not tied:
        w = normal(s, TID_OUTPUT, V * d, 0.0, 0.02).reshape(V, d)
        output = encode(w, cfg.t_out)
        del w
    layers = []
    for l in range(cfg.n_layer if n_layer is None else n_layer):
        L = {}
        for name in LAYER_TENSORS:
            tid = layer_tid(l, name)
            if name.endswith("norm"):
                g = normal(s, tid, d, 1.0, 0.02)
                if name in zero:
                    g[:] = 0.0
                L[name] = g
                continue
            N, K = matrix_shape(cfg, name)
            w = normal(s, tid, N * K, 0.0, 0.02).reshape(N, K)
            if name in zero:
                w[:] = 0.0
            L[name] = encode(w, cfg.t_linear)
            del w
        layers.append(L)
    return Model(cfg, tok_embd, out_norm, output, layers)


def prompt_tokens(cfg: Config, n: int, stream: int = 0) -> np.ndarray:
    """n uniform token ids in [0, n_vocab) for prompt stream `stream` (one per sequence)."""
    return uniform_int(cfg.token_seed, stream, n, 0, cfg.n_vocab)


def multiseq_prompt_lengths(cfg: Config, n_seq: int = 64, lo: int = 256, hi: int = 4096) -> np.ndarray:
    """Prompt lengths uniform in [lo, hi] for the batched-decode workload."""
    return uniform_int(cfg.token_seed, 1000, n_seq, lo, hi + 1)


def with_shape(cfg: Config, **kw) -> Config:
    return replace(cfg, **kw)
