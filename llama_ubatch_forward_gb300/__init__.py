"""Python binding of liblcx (include/lcx.h): argument marshalling only.

Every step of the forward runs in the library's CUDA kernels; this module loads the in-tree
shared library, mirrors the C structs with ctypes and wraps the calls under the same names.
PyTorch, when used by callers, only provides device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "liblcx.so")
_lib = None

LCX_F16, LCX_Q4_0, LCX_Q8_0 = 1, 2, 8
LCX_OK, LCX_NO_KV_SLOT, LCX_ABORTED = 0, 1, 2
LCX_INVALID, LCX_ALLOC_FAILED, LCX_COMPUTE_FAILED = -1, -2, -3
LCX_ATTENTION_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024   # as include/lcx.h

SYMBOLS = ("lcx_model_create", "lcx_model_free", "lcx_ctx_create", "lcx_ctx_free", "lcx_decode",
           "lcx_decode_greedy", "lcx_kv_clear", "lcx_seq_pos_max", "lcx_n_outputs", "lcx_set_abort",
           "lcx_get_stats", "lcx_ctx_create_host_only", "lcx_get_rows", "lcx_last_error", "lcx_set_profiling",
           "lcx_get_profile", "lcx_attention_workspace_size", "lcx_attention", "lcx_attention_noalloc",
           "lcx_kv_read", "lcx_get_trace", "lcx_sample", "lcx_ctx_inject_failure", "lcx_ctx_set_kv_unified",
           "lcx_set_gemm_tile")


def build(force: bool = False) -> str:
    from . import buildlib as _b
    return _b.build(force=force)


class lcx_hparams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_vocab", "n_embd", "n_layer", "n_head", "n_head_kv",
                                               "head_dim", "n_ff")] + \
               [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)] + \
               [(n, ctypes.c_int32) for n in ("t_linear", "t_embd", "t_out")]


class lcx_layer_w(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate",
                                                "w_up", "w_down")]


class lcx_weights(ctypes.Structure):
    _fields_ = [("tok_embd", ctypes.c_void_p), ("output_norm", ctypes.c_void_p), ("output", ctypes.c_void_p),
                ("layers", ctypes.POINTER(lcx_layer_w))]


class lcx_batch(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int32), ("token", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("seq_id", ctypes.c_void_p), ("logits", ctypes.c_void_p)]


class lcx_sampler(ctypes.Structure):
    _fields_ = [("penalty_repeat", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float),
                ("min_p", ctypes.c_float), ("temp", ctypes.c_float)]


class lcx_stats(ctypes.Structure):
    _fields_ = [("n_decode", ctypes.c_int64), ("n_ubatch", ctypes.c_int64), ("n_ubatch_last", ctypes.c_int32),
                ("n_outputs_last", ctypes.c_int32), ("n_kernels", ctypes.c_int64), ("n_cells_used", ctypes.c_int64),
                ("n_ctx", ctypes.c_uint32), ("n_pages", ctypes.c_uint32), ("n_gemm_wide", ctypes.c_int64)]


class lcx_kernel_profile(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64), ("ms", ctypes.c_double), ("bytes", ctypes.c_double),
                ("flops", ctypes.c_double)]


class lcx_profile(ctypes.Structure):
    _fields_ = [(n, lcx_kernel_profile) for n in ("gemv", "gemm", "attention", "other")]


ABORT_CB = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p)


def lib():
    """The loaded library; raises if the CUDA extension has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"liblcx is not built ({LIB_PATH} missing): call llama_ubatch_forward_gb300.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, u32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_int64
        L.lcx_model_create.restype = vp
        L.lcx_model_create.argtypes = [ctypes.POINTER(lcx_hparams), ctypes.POINTER(lcx_weights), ctypes.POINTER(i32)]
        L.lcx_model_free.argtypes = [vp]
        L.lcx_ctx_create.restype = vp
        L.lcx_ctx_create.argtypes = [vp, u32, u32, u32, vp]
        L.lcx_ctx_create_host_only.restype = vp
        L.lcx_ctx_create_host_only.argtypes = [ctypes.POINTER(lcx_hparams), u32, u32, u32]
        L.lcx_ctx_free.argtypes = [vp]
        L.lcx_decode.restype = i32
        L.lcx_decode.argtypes = [vp, lcx_batch, vp, vp]
        L.lcx_decode_greedy.restype = i32
        L.lcx_decode_greedy.argtypes = [vp, i32, i32, i32, vp]
        L.lcx_kv_clear.argtypes = [vp]
        L.lcx_ctx_set_kv_unified.restype = i32
        L.lcx_ctx_set_kv_unified.argtypes = [vp, i32]
        L.lcx_seq_pos_max.restype = i32
        L.lcx_seq_pos_max.argtypes = [vp, i32]
        L.lcx_n_outputs.restype = i32
        L.lcx_n_outputs.argtypes = [vp]
        L.lcx_set_abort.argtypes = [vp, ABORT_CB, vp]
        L.lcx_get_stats.argtypes = [vp, ctypes.POINTER(lcx_stats)]
        L.lcx_get_rows.restype = i32
        L.lcx_get_rows.argtypes = [i32, vp, i64, i64, vp, i32, vp, vp]
        L.lcx_last_error.restype = ctypes.c_char_p
        L.lcx_attention_workspace_size.restype = ctypes.c_size_t
        L.lcx_attention_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.lcx_attention.restype = i32
        L.lcx_attention.argtypes = [i32, i32, i32, i32, vp, vp, vp, i32, vp, i32, vp, vp, i32, vp, vp,
                                    ctypes.c_size_t, vp]
        L.lcx_attention_noalloc.restype = i32
        L.lcx_attention_noalloc.argtypes = [i32, i32, i32, i32, vp, vp, vp, i32, vp, i32, vp, vp, i32, vp, vp]
        L.lcx_ctx_inject_failure.restype = i32
        L.lcx_ctx_inject_failure.argtypes = [vp, i32]
        L.lcx_set_gemm_tile.restype = i32
        L.lcx_set_gemm_tile.argtypes = [i32, i32, i32]
        L.lcx_sample.restype = i32
        L.lcx_sample.argtypes = [ctypes.POINTER(lcx_sampler), vp, i32, i32, vp, i32, vp, vp, vp]
        L.lcx_get_trace.restype = i32
        L.lcx_get_trace.argtypes = [vp, vp, i32]
        L.lcx_kv_read.restype = i32
        L.lcx_kv_read.argtypes = [vp, i32, i32, i32, vp, vp]
        L.lcx_set_profiling.restype = i32
        L.lcx_set_profiling.argtypes = [vp, i32]
        L.lcx_get_profile.restype = i32
        L.lcx_get_profile.argtypes = [vp, ctypes.POINTER(lcx_profile)]
        _lib = L
    return _lib


def _ptr(a):
    """Data pointer of a numpy array / torch tensor / int / None."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    return a.ctypes.data


def make_batch(tokens, pos=None, seq_id=None, logits=None):
    """An lcx_batch over host numpy int32/int8 arrays (kept alive by the returned tuple)."""
    import numpy as np
    keep = [np.ascontiguousarray(tokens, dtype=np.int32)]
    b = lcx_batch(keep[0].size, keep[0].ctypes.data, None, None, None)
    if pos is not None:
        keep.append(np.ascontiguousarray(pos, dtype=np.int32)); b.pos = keep[-1].ctypes.data
    if seq_id is not None:
        keep.append(np.ascontiguousarray(seq_id, dtype=np.int32)); b.seq_id = keep[-1].ctypes.data
    if logits is not None:
        keep.append(np.ascontiguousarray(logits, dtype=np.int8)); b.logits = keep[-1].ctypes.data
    return b, keep


class Model:
    """lcx_model over device weights. `weights` maps names to objects with data_ptr() (device);
    they must outlive the model (the library borrows them)."""

    def __init__(self, hp: lcx_hparams, tok_embd, output_norm, output, layers: list[dict]):
        self.hp = hp
        self._keep = (tok_embd, output_norm, output, layers)
        arr = (lcx_layer_w * len(layers))()
        for i, L in enumerate(layers):
            arr[i] = lcx_layer_w(*[_ptr(L[n]) for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm",
                                                         "w_gate", "w_up", "w_down")])
        self._arr = arr
        w = lcx_weights(_ptr(tok_embd), _ptr(output_norm), _ptr(output), arr)
        err = ctypes.c_int32(0)
        self.h = lib().lcx_model_create(ctypes.byref(hp), ctypes.byref(w), ctypes.byref(err))
        if not self.h:
            raise RuntimeError(f"lcx_model_create failed ({err.value}): {lib().lcx_last_error().decode()}")

    def close(self):
        if getattr(self, "h", None):
            lib().lcx_model_free(self.h)
            self.h = None

    __del__ = close


class Context:
    def __init__(self, model: Model | None, n_ctx: int, n_seq_max: int = 1, n_ubatch: int = 512, stream=None,
                 host_only_hp: lcx_hparams | None = None):
        self.model = model
        if model is None:
            self.h = lib().lcx_ctx_create_host_only(ctypes.byref(host_only_hp), n_ctx, n_seq_max, n_ubatch)
            self.n_vocab = host_only_hp.n_vocab
        else:
            s = None if stream is None else (stream if isinstance(stream, int) else stream.cuda_stream)
            self.h = lib().lcx_ctx_create(model.h, n_ctx, n_seq_max, n_ubatch, s)
            self.n_vocab = model.hp.n_vocab
        if not self.h:
            raise RuntimeError(f"lcx_ctx_create failed: {lib().lcx_last_error().decode()}")
        self._abort = None

    def close(self):
        if getattr(self, "h", None):
            lib().lcx_ctx_free(self.h)
            self.h = None

    __del__ = close

    def decode(self, tokens, pos=None, seq_id=None, logits=None, logits_out=None, argmax_out=None) -> int:
        b, keep = make_batch(tokens, pos, seq_id, logits)
        return lib().lcx_decode(self.h, b, _ptr(logits_out), _ptr(argmax_out))

    def decode_greedy(self, seq: int, token: int, n_steps: int, tokens_out) -> int:
        return lib().lcx_decode_greedy(self.h, seq, token, n_steps, _ptr(tokens_out))

    def kv_clear(self):
        lib().lcx_kv_clear(self.h)

    def set_kv_unified(self, unified: bool) -> int:
        """One cell store for all sequences (True, the default) or a stream per sequence."""
        return lib().lcx_ctx_set_kv_unified(self.h, 1 if unified else 0)

    def inject_failure(self, ubatch: int) -> int:
        """Host-only contexts: ubatch `ubatch` of the next decode fails as a failed launch would."""
        return lib().lcx_ctx_inject_failure(self.h, ubatch)

    def seq_pos_max(self, seq: int) -> int:
        return lib().lcx_seq_pos_max(self.h, seq)

    def n_outputs(self) -> int:
        return lib().lcx_n_outputs(self.h)

    def set_abort(self, fn):
        """fn() -> bool, called before every ubatch after the first; None removes it."""
        if fn is None:
            self._abort = None
            lib().lcx_set_abort(self.h, ABORT_CB(0), None)
            return
        self._abort = ABORT_CB(lambda _ud: 1 if fn() else 0)
        lib().lcx_set_abort(self.h, self._abort, None)

    def set_profiling(self, on) -> int:
        """False: off; True: per-launch events; 2: in-kernel timeline (see trace())."""
        return lib().lcx_set_profiling(self.h, 2 if on == 2 else (1 if on else 0))

    def trace(self):
        """The recorded timeline as a numpy array [launches][4] (ns)."""
        import numpy as np
        n = lib().lcx_get_trace(self.h, None, 0)
        out = np.zeros((max(n, 0), 4), dtype=np.uint64)
        if n > 0:
            lib().lcx_get_trace(self.h, out.ctypes.data, n)
        return out

    def profile(self) -> dict:
        p = lcx_profile()
        lib().lcx_get_profile(self.h, ctypes.byref(p))
        return {n: {"launches": getattr(p, n).launches, "ms": getattr(p, n).ms, "bytes": getattr(p, n).bytes,
                    "flops": getattr(p, n).flops} for n in ("gemv", "gemm", "attention", "other")}

    def kv_read(self, layer: int, seq: int, pos: int):
        """(k, v) of one cell as float16 numpy arrays [n_head_kv * head_dim]."""
        import numpy as np
        hp = self.model.hp
        k = np.empty(hp.n_head_kv * hp.head_dim, dtype=np.uint16)
        v = np.empty_like(k)
        rc = lib().lcx_kv_read(self.h, layer, seq, pos, k.ctypes.data, v.ctypes.data)
        if rc != 0:
            raise IndexError(f"lcx_kv_read -> {rc}")
        return k.view(np.float16), v.view(np.float16)

    def stats(self) -> lcx_stats:
        s = lcx_stats()
        lib().lcx_get_stats(self.h, ctypes.byref(s))
        return s


def set_gemm_tile(bn: int = 0, mt: int = 1, ks: int = 1) -> int:
    """Force the prefill GEMM's tile shape for every later launch (bn = 0: the cost model's)."""
    return lib().lcx_set_gemm_tile(bn, mt, ks)


def get_rows(qtype: int, table, n_rows: int, n_cols: int, ids, out, stream=None) -> int:
    s = None if stream is None else (stream if isinstance(stream, int) else stream.cuda_stream)
    return lib().lcx_get_rows(qtype, _ptr(table), n_rows, n_cols, _ptr(ids), int(ids.numel()), _ptr(out), s)


def attention(q, k_cache, v_cache, page_table, pos, seq, max_pos: int, out, workspace=None, stream=None) -> int:
    """lcx_attention over torch device tensors: q [T][H*hd] f32, caches [n_pages][KV][64][hd] f16,
    page_table [n_seq][max_pages] i32, pos/seq [T] i32, out [T][H*hd] f32."""
    T = int(pos.numel())
    n_pages, n_kv, _, hd = (int(x) for x in k_cache.shape)
    H = int(q.shape[1]) // hd
    s = None if stream is None else (stream if isinstance(stream, int) else stream.cuda_stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return lib().lcx_attention(T, H, n_kv, hd, _ptr(q), _ptr(k_cache), _ptr(v_cache), n_pages, _ptr(page_table),
                               int(page_table.shape[1]), _ptr(pos), _ptr(seq), max_pos, _ptr(out), _ptr(workspace),
                               ws_bytes, s)


def attention_workspace_size(T: int, n_head: int, n_head_kv: int, head_dim: int, max_pos: int) -> int:
    return int(lib().lcx_attention_workspace_size(T, n_head, n_head_kv, head_dim, max_pos))


def attention_noalloc(q, k_cache, v_cache, page_table, pos, seq, max_pos: int, out, stream=None) -> int:
    """lcx_attention_noalloc (no workspace: the library's fixed device scratch is used)."""
    T = int(pos.numel())
    n_pages, n_kv, _, hd = (int(x) for x in k_cache.shape)
    H = int(q.shape[1]) // hd
    s = None if stream is None else (stream if isinstance(stream, int) else stream.cuda_stream)
    return lib().lcx_attention_noalloc(T, H, n_kv, hd, _ptr(q), _ptr(k_cache), _ptr(v_cache), n_pages,
                                       _ptr(page_table), int(page_table.shape[1]), _ptr(pos), _ptr(seq), max_pos,
                                       _ptr(out), s)


def sample(logits, u=None, history=None, penalty_repeat: float = 1.0, top_k: int = 0, top_p: float = 1.0,
           min_p: float = 0.0, temp: float = 1.0, tokens_out=None, stream=None):
    """lcx_sample over torch device tensors: logits [n_rows][n_vocab] f32, u [n_rows] f32,
    history [n_rows][n_history] i32 or None; returns (rc, tokens_out [n_rows] i32)."""
    import torch
    n_rows, n_vocab = (int(x) for x in logits.shape)
    if tokens_out is None:
        tokens_out = torch.empty(n_rows, dtype=torch.int32, device=logits.device)
    prm = lcx_sampler(penalty_repeat, top_k, top_p, min_p, temp)
    n_hist = 0 if history is None else int(history.shape[1])
    s = None if stream is None else (stream if isinstance(stream, int) else stream.cuda_stream)
    rc = lib().lcx_sample(ctypes.byref(prm), _ptr(logits), n_rows, n_vocab, _ptr(history), n_hist, _ptr(u),
                          _ptr(tokens_out), s)
    return rc, tokens_out
