"""CPU oracle for the batch-1 Llama decode forward pass.

TEST INFRASTRUCTURE.  A plain, slow, single-threaded C evaluation of the pass
("The Forward Pass in Java", Example 13, with the per-step passages cited in
llm_oracle.c), used only by tests/, by the package smoke check and by the
benchmark's CPU-baseline leg.  The product path never imports it.  It shares
no code with the CUDA library; both receive the same seeded inputs from the
separate ``synth`` module.

Parity status: every primitive and the whole pass are pinned by the
``-m "not gpu"`` tests (printed worked examples of the pages, closed forms,
invariants, and the pages' end-to-end self-test with its printed token ids).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, F16, Q8_0 = 0, 1, 8
_HERE = os.path.dirname(os.path.abspath(__file__))
_LOCK = threading.Lock()
_LIB = None
CFLAGS = ["-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp"]


def build(force: bool = False) -> str:
    """Compile llm_oracle.c into oracle/_build/liborc.so."""
    srcs = [os.path.join(_HERE, "llm_oracle.c"), os.path.join(_HERE, "llm_oracle.h")]
    out_dir = os.path.join(_HERE, "_build")
    out = os.path.join(out_dir, "liborc.so")
    if not force and os.path.exists(out) and all(os.path.getmtime(out) >= os.path.getmtime(s) for s in srcs):
        return out
    os.makedirs(out_dir, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, srcs[0], "-lm"])
    os.replace(tmp, out)
    return out


class _Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_layers", "dim", "n_heads", "n_kv_heads", "head_dim",
                                            "ffn_dim", "vocab", "max_seq", "rope_dims")] + \
               [("eps", ctypes.c_float), ("rope_base", ctypes.c_float), ("rope_neox", ctypes.c_int),
                ("wtype", ctypes.c_int), ("f16_cache", ctypes.c_int), ("llamacpp_rounding", ctypes.c_int)]


class _Layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("attn_norm", "ffn_norm", "bq", "bk", "bv", "wq", "wk", "wv",
                                               "wo", "w_gate", "w_up", "w_down")]


class _Weights(ctypes.Structure):
    _fields_ = [("tok_embd", ctypes.c_void_p), ("output_norm", ctypes.c_void_p), ("output", ctypes.c_void_p),
                ("rope_freqs", ctypes.c_void_p), ("layers", ctypes.POINTER(_Layer))]


_TRACE_FN = ctypes.CFUNCTYPE(None, ctypes.c_char_p, ctypes.c_int, ctypes.POINTER(ctypes.c_float),
                             ctypes.c_int, ctypes.c_void_p)


def load(path: str):
    """Load an oracle shared library and declare its C signatures."""
    L = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.orc_create.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Weights)]
    L.orc_create.restype = vp
    L.orc_destroy.argtypes = [vp]
    L.orc_set_trace.argtypes = [vp, _TRACE_FN, vp]
    L.orc_forward.argtypes = [vp, i, i, vp]
    L.orc_forward.restype = i
    L.orc_prefill.argtypes = [vp, vp, i, i, vp]
    L.orc_prefill.restype = i
    L.orc_kv.argtypes = [vp, i, i]
    L.orc_kv.restype = ctypes.POINTER(ctypes.c_float)
    L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_f16_to_f32.restype = f
    L.orc_f32_to_f16.argtypes = [f]
    L.orc_f32_to_f16.restype = ctypes.c_uint16
    L.orc_dequant_row.argtypes = [vp, i, ctypes.c_int64, i, vp]
    L.orc_quantize_q8_0.argtypes = [vp, ctypes.c_int64, vp]
    L.orc_rmsnorm.argtypes = [vp, vp, vp, i, f]
    L.orc_matvec.argtypes = [vp, vp, i, vp, i, i]
    L.orc_rope.argtypes = [vp, i, i, i, i, f, i, vp]
    L.orc_silu.argtypes = [f]
    L.orc_silu.restype = f
    L.orc_attention.argtypes = [vp, vp, vp, vp, i, i, i, i]
    L.orc_argmax.argtypes = [vp, i]
    L.orc_argmax.restype = i
    L.orc_matvec_llamacpp.argtypes = [vp, vp, i, vp, i, i]
    L.orc_set_threads.argtypes = [i]
    L.orc_attention_llamacpp.argtypes = [vp, vp, vp, vp, i, i, i, i]
    return L


def lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            try:
                _LIB = load(build())
            except OSError:                        # a binary built on another machine
                _LIB = load(build(force=True))
    return _LIB


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


# ------------------------------------------------------------- primitives --
def f16_to_f32(bits) -> np.ndarray:
    L = lib()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([L.orc_f16_to_f32(int(v)) for v in b], dtype=np.float32)


def f32_to_f16(x) -> np.ndarray:
    L = lib()
    a = _f32(x).ravel()
    return np.array([L.orc_f32_to_f16(float(v)) for v in a], dtype=np.uint16)


def set_threads(n: int) -> None:
    """1 (the default): the oracle runs on the calling thread.  n > 1: the
    rows of every matrix product and the heads of attention are split over n
    OpenMP threads (each output element still computed by one thread in the
    same order, so every result is bitwise the single-thread one)."""
    lib().orc_set_threads(int(n))


class threads:
    """Context manager: the oracle on n threads inside the block, 1 after."""

    def __init__(self, n: int | None = None):
        self.n = n or os.cpu_count() or 1

    def __enter__(self):
        set_threads(self.n)
        return self

    def __exit__(self, *exc):
        set_threads(1)
        return False


def dequant_row(w: np.ndarray, wtype: int, row: int, cols: int) -> np.ndarray:
    out = np.empty(cols, dtype=np.float32)
    lib().orc_dequant_row(_p(np.ascontiguousarray(w)), wtype, row, cols, _p(out))
    return out


def quantize_q8_0(x) -> np.ndarray:
    a = _f32(x)
    out = np.zeros((a.size // 32) * 34, dtype=np.uint8)
    lib().orc_quantize_q8_0(_p(a), a.size, _p(out))
    return out


def rmsnorm(x, g, eps: float) -> np.ndarray:
    x, g = _f32(x), _f32(g)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_p(out), _p(x), _p(g), x.size, eps)
    return out


def matvec(w, wtype: int, x, rows: int, cols: int, llamacpp: bool = False) -> np.ndarray:
    """W x; with ``llamacpp`` the activations are rounded as llama.cpp rounds
    them for the weight type (orc_matvec_llamacpp)."""
    x = _f32(x)
    out = np.empty(rows, dtype=np.float32)
    fn = lib().orc_matvec_llamacpp if llamacpp else lib().orc_matvec
    fn(_p(out), _p(np.ascontiguousarray(w)), wtype, _p(x), rows, cols)
    return out


def rope(vec, n_heads: int, head_dim: int, rope_dims: int, pos: int, base: float, neox: bool,
         freqs=None) -> np.ndarray:
    v = _f32(vec).copy()
    fr = None if freqs is None else _f32(freqs)
    lib().orc_rope(_p(v), n_heads, head_dim, rope_dims, pos, base, int(neox), _p(fr))
    return v


def silu(z: float) -> float:
    return lib().orc_silu(float(z))


def attention(q, kcache, vcache, n_heads: int, n_kv_heads: int, head_dim: int, pos: int,
              llamacpp: bool = False) -> np.ndarray:
    """Attention of one position; with ``llamacpp`` q and the probabilities are
    rounded to F16 (orc_attention_llamacpp)."""
    q, k, v = _f32(q), _f32(kcache), _f32(vcache)
    out = np.empty(n_heads * head_dim, dtype=np.float32)
    fn = lib().orc_attention_llamacpp if llamacpp else lib().orc_attention
    fn(_p(out), _p(q), _p(k), _p(v), n_heads, n_kv_heads, head_dim, pos)
    return out


def argmax(v) -> int:
    a = _f32(v)
    return lib().orc_argmax(_p(a), a.size)


# ------------------------------------------------------------------ model --
class OracleModel:
    """The whole pass over host weights in GGUF layout.

    ``cfg`` needs the attributes n_layers, dim, n_heads, n_kv_heads, head_dim,
    ffn_dim, vocab, max_seq, rope_dims, eps, rope_base, rope_neox, wtype.
    ``tensors`` needs tok_embd, output_norm, output (None: tied), rope_freqs
    (None: unit) and ``layers``: a list of dicts with attn_norm, ffn_norm, bq,
    bk, bv (None: no bias), wq, wk, wv, wo, w_gate, w_up, w_down.
    The arrays are referenced, not copied: keep them alive with this object.
    ``llamacpp_rounding`` adds llama.cpp's rounding points ("What a Llama
    model computes, and why" §8) to every matrix product and the attention.
    """

    def __init__(self, cfg, tensors, f16_cache: bool = True, max_seq: int | None = None,
                 llamacpp_rounding: bool = False):
        self._L = L = lib()
        self.cfg = cfg
        self.max_seq = int(max_seq if max_seq is not None else cfg.max_seq)
        c = _Config(n_layers=cfg.n_layers, dim=cfg.dim, n_heads=cfg.n_heads, n_kv_heads=cfg.n_kv_heads,
                    head_dim=cfg.head_dim, ffn_dim=cfg.ffn_dim, vocab=cfg.vocab, max_seq=self.max_seq,
                    rope_dims=cfg.rope_dims, eps=cfg.eps, rope_base=cfg.rope_base,
                    rope_neox=int(cfg.rope_neox), wtype=cfg.wtype, f16_cache=int(f16_cache),
                    llamacpp_rounding=int(llamacpp_rounding))
        self._keep = [tensors]
        layers = (_Layer * cfg.n_layers)()
        for l, T in enumerate(tensors.layers):
            for name in _Layer._fields_:
                n = name[0]
                a = T.get(n)
                if a is not None:
                    a = np.ascontiguousarray(a)
                    self._keep.append(a)
                setattr(layers[l], n, _p(a))
        def keep(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            self._keep.append(a)
            return _p(a)
        w = _Weights(tok_embd=keep(tensors.tok_embd), output_norm=keep(tensors.output_norm),
                     output=keep(tensors.output), rope_freqs=keep(tensors.rope_freqs), layers=layers)
        self._layers = layers
        self._h = L.orc_create(ctypes.byref(c), ctypes.byref(w))
        if not self._h:
            raise ValueError("oracle rejected the configuration")
        self._trace_cb = None

    def close(self):
        if getattr(self, "_h", None):
            self._L.orc_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def set_trace(self, fn):
        """fn(name: str, layer: int, values: np.ndarray) after each named step, or None."""
        if fn is None:
            self._trace_cb = _TRACE_FN(lambda *a: None)
        else:
            def cb(name, layer, ptr, n, user):
                fn(name.decode(), layer, np.ctypeslib.as_array(ptr, shape=(n,)).copy())
            self._trace_cb = _TRACE_FN(cb)
        self._L.orc_set_trace(self._h, self._trace_cb, None)

    def forward(self, token: int, pos: int) -> np.ndarray:
        logits = np.empty(self.cfg.vocab, dtype=np.float32)
        if self._L.orc_forward(self._h, int(token), int(pos), _p(logits)) != 0:
            raise IndexError(f"token {token} or pos {pos} out of range")
        return logits

    def prefill(self, tokens, pos0: int = 0) -> np.ndarray:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        logits = np.empty(self.cfg.vocab, dtype=np.float32)
        if self._L.orc_prefill(self._h, _p(t), t.size, int(pos0), _p(logits)) != 0:
            raise IndexError("prefill range out of bounds")
        return logits

    def kv(self, layer: int, which: int) -> np.ndarray:
        """Writable view [max_seq, n_kv_heads*head_dim] of one layer's K (0) or V (1) cache."""
        ptr = self._L.orc_kv(self._h, layer, which)
        kv_dim = self.cfg.n_kv_heads * self.cfg.head_dim
        return np.ctypeslib.as_array(ptr, shape=(self.max_seq, kv_dim))

    def set_kv_rows_f16(self, layer: int, which: int, rows_f16: np.ndarray):
        """Pre-fill cache rows 0..n-1 of one layer from FP16 bit patterns."""
        n = rows_f16.shape[0]
        self.kv(layer, which)[:n] = np.asarray(rows_f16, dtype=np.uint16).view(np.float16).astype(np.float32)
