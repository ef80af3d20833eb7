"""ORACLE -- test infrastructure only.

ctypes wrapper of ``oracle.cpp``, the plain fp64 CPU forward of a Llama-architecture decoder over
one batch. Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg use it;
the product library never loads it and shares no code with it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.cpp")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                               src, "-o", tmp])
        os.replace(tmp, _SO)
    return _SO


class Hparams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_vocab", "n_embd", "n_layer", "n_head", "n_head_kv",
                                               "head_dim", "n_ff")] + \
               [("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double)] + \
               [(n, ctypes.c_int32) for n in ("t_linear", "t_embd", "t_out")]


class Layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate",
                                                "w_up", "w_down")]


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        vp, i32, i64, u32, dp = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_double
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_get_threads.restype = ctypes.c_int
        L.orc_model_create.restype = vp
        L.orc_model_create.argtypes = [ctypes.POINTER(Hparams), vp, vp, vp, ctypes.POINTER(Layer)]
        L.orc_model_free.argtypes = [vp]
        L.orc_ctx_create.restype = vp
        L.orc_ctx_create.argtypes = [vp, u32, u32, u32]
        L.orc_ctx_free.argtypes = [vp]
        L.orc_n_ctx.restype = u32
        L.orc_n_ctx.argtypes = [vp]
        L.orc_kv_clear.argtypes = [vp]
        L.orc_seq_pos_max.restype = i32
        L.orc_seq_pos_max.argtypes = [vp, i32]
        L.orc_kv_get.restype = i32
        L.orc_kv_get.argtypes = [vp, i32, i32, i32, vp, vp]
        L.orc_decode.restype = i32
        L.orc_decode.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp]
        L.orc_set_trace.argtypes = [vp, i32]
        L.orc_get_trace.restype = i64
        L.orc_get_trace.argtypes = [vp, i32, vp]
        L.orc_row_bytes.restype = i64
        L.orc_row_bytes.argtypes = [i32, i64]
        L.orc_dequant_row.argtypes = [i32, vp, i64, vp]
        L.orc_half_to_double.restype = dp
        L.orc_half_to_double.argtypes = [ctypes.c_uint16]
        L.orc_round_to_half.restype = dp
        L.orc_round_to_half.argtypes = [dp]
        L.orc_matvec.argtypes = [i32, vp, i64, i64, vp, vp]
        L.orc_matmat.argtypes = [i32, vp, i64, i64, vp, i64, vp]
        L.orc_set_elide.argtypes = [vp, i32]
        L.orc_set_kv_unified.restype = i32
        L.orc_set_kv_unified.argtypes = [vp, i32]
        L.orc_rmsnorm.argtypes = [vp, i64, vp, dp, vp]
        L.orc_rope.argtypes = [vp, i32, i64, dp]
        L.orc_silu.restype = dp
        L.orc_silu.argtypes = [dp]
        L.orc_attend_gqa.argtypes = [vp, vp, vp, i64, i32, i32, i32, vp]
        _lib = L
    return _lib


def set_threads(n: int | None = None) -> int:
    n = n or os.cpu_count() or 1
    lib().orc_set_threads(int(n))
    return int(n)


def _p(a):
    return None if a is None else a.ctypes.data


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


# ------------------------------------------------------------------ single operations
def dequant_row(qtype: int, row: np.ndarray, n: int) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.uint8)
    assert row.nbytes >= lib().orc_row_bytes(qtype, n)
    out = np.empty(n, dtype=np.float64)
    lib().orc_dequant_row(qtype, _p(row), n, _p(out))
    return out


def dequant_matrix(qtype: int, rows: np.ndarray, k: int) -> np.ndarray:
    return np.stack([dequant_row(qtype, rows[i], k) for i in range(rows.shape[0])])


def half_to_double(h: int) -> float:
    return lib().orc_half_to_double(int(h))


def round_to_half(x: float) -> float:
    return lib().orc_round_to_half(float(x))


def matvec(qtype: int, W: np.ndarray, n: int, k: int, x) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = _f64(x)
    y = np.empty(n, dtype=np.float64)
    lib().orc_matvec(qtype, _p(W), n, k, _p(x), _p(y))
    return y


def matmat(qtype: int, W: np.ndarray, n: int, k: int, X) -> np.ndarray:
    """Y [T][n] = X [T][k] times the stored matrix W [n][k] transposed (every token as matvec)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.float64)
    Y = np.empty((X.shape[0], n), dtype=np.float64)
    lib().orc_matmat(qtype, _p(W), n, k, _p(X), X.shape[0], _p(Y))
    return Y


def rmsnorm(x, g, eps: float) -> np.ndarray:
    x = _f64(x)
    g = np.ascontiguousarray(g, dtype=np.float32)
    y = np.empty_like(x)
    lib().orc_rmsnorm(_p(x), x.size, _p(g), eps, _p(y))
    return y


def rope(x, pos: int, theta: float) -> np.ndarray:
    y = _f64(x).copy()
    lib().orc_rope(_p(y), y.size, pos, theta)
    return y


def silu(a: float) -> float:
    return lib().orc_silu(float(a))


def attend_gqa(q, K, V, n_head: int, n_head_kv: int, hd: int) -> np.ndarray:
    """q [n_head*hd]; K, V [n][n_head_kv*hd] -> o [n_head*hd]."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    n = K.shape[0]
    o = np.empty(n_head * hd, dtype=np.float64)
    lib().orc_attend_gqa(_p(q), _p(K), _p(V), n, n_head, n_head_kv, hd, _p(o))
    return o


# ------------------------------------------------------------------ model / context
class Model:
    def __init__(self, m):
        """m: a synth.Model (host arrays in stored form)."""
        cfg = m.cfg
        self.src = m
        self.cfg = cfg
        self.hp = Hparams(cfg.n_vocab, cfg.n_embd, len(m.layers), cfg.n_head, cfg.n_head_kv, cfg.head_dim,
                          cfg.n_ff, cfg.rms_eps, cfg.rope_theta, cfg.t_linear, cfg.t_embd, cfg.t_out)
        arr = (Layer * max(1, len(m.layers)))()
        for i, L in enumerate(m.layers):
            arr[i] = Layer(*[L[n].ctypes.data for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm",
                                                         "w_gate", "w_up", "w_down")])
        self._layers = arr
        self.h = lib().orc_model_create(ctypes.byref(self.hp), _p(m.tok_embd), _p(m.output_norm),
                                        _p(m.output), arr)
        if not self.h:
            raise ValueError("oracle rejected the model shape")

    def __del__(self):
        if getattr(self, "h", None):
            lib().orc_model_free(self.h)
            self.h = None


class Context:
    def __init__(self, model: Model, n_ctx: int, n_seq_max: int = 1, n_ubatch: int = 512):
        self.model = model
        self.h = lib().orc_ctx_create(model.h, n_ctx, n_seq_max, n_ubatch)
        if not self.h:
            raise ValueError("oracle rejected the context parameters")
        self.n_vocab = model.cfg.n_vocab

    def __del__(self):
        if getattr(self, "h", None):
            lib().orc_ctx_free(self.h)
            self.h = None

    @property
    def n_ctx(self) -> int:
        return lib().orc_n_ctx(self.h)

    def kv_clear(self):
        lib().orc_kv_clear(self.h)

    def seq_pos_max(self, seq: int) -> int:
        return lib().orc_seq_pos_max(self.h, seq)

    def kv_get(self, seq: int, pos: int, layer: int):
        w = self.model.cfg.n_head_kv * self.model.cfg.head_dim
        k = np.empty(w, dtype=np.float64)
        v = np.empty(w, dtype=np.float64)
        rc = lib().orc_kv_get(self.h, seq, pos, layer, _p(k), _p(v))
        if rc != 0:
            raise IndexError("no such cell")
        return k, v

    def set_elide(self, on: bool):
        """Last layer: tokens whose logits are not flagged compute only K and V (on, the default)."""
        lib().orc_set_elide(self.h, 1 if on else 0)

    def set_kv_unified(self, on: bool) -> int:
        """One KV store for all sequences (True, the default) or a stream per sequence (False)."""
        return lib().orc_set_kv_unified(self.h, 1 if on else 0)

    def set_trace(self, layer: int):
        lib().orc_set_trace(self.h, layer)

    def trace(self, which: str) -> np.ndarray:
        idx = {"x": 0, "q": 1, "o": 2, "x1": 3}[which]
        n = lib().orc_get_trace(self.h, idx, None)
        if n < 0:
            raise LookupError("no trace recorded")
        out = np.empty(n, dtype=np.float64)
        lib().orc_get_trace(self.h, idx, _p(out))
        return out

    def decode(self, tokens, pos=None, seq=None, logits=None):
        """Returns (rc, logits [n_out][V] float64, argmax [n_out] int32)."""
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        n = tok.size
        pos_a = None if pos is None else np.ascontiguousarray(pos, dtype=np.int32)
        seq_a = None if seq is None else np.ascontiguousarray(seq, dtype=np.int32)
        flg = None if logits is None else np.ascontiguousarray(logits, dtype=np.int8)
        n_flag = n if n > 0 else 0
        out = np.empty((max(n_flag, 1), self.n_vocab), dtype=np.float64)
        am = np.empty(max(n_flag, 1), dtype=np.int32)
        n_out = ctypes.c_int32(0)
        rc = lib().orc_decode(self.h, n, _p(tok), _p(pos_a), _p(seq_a), _p(flg), _p(out), _p(am),
                              ctypes.byref(n_out))
        k = n_out.value
        return rc, out[:k].copy(), am[:k].copy()
