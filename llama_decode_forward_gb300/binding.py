"""ctypes binding of libllmdecode with the names of include/llm.h.

Argument marshalling only: every step of the decode pass runs in the CUDA
library.  PyTorch is used for device memory and streams (``DeviceWeights``
uploads host arrays into CUDA tensors).  If the library cannot be built or
loaded, importing this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

LLM_F32, LLM_F16, LLM_Q8_0 = 0, 1, 8
LLM_OK = 0
LLM_ERR_INVALID_ARG, LLM_ERR_UNSUPPORTED, LLM_ERR_OUT_OF_RANGE = -1, -2, -3
LLM_ERR_CUDA, LLM_ERR_NO_MEMORY, LLM_ERR_DEVICE_TIMEOUT, LLM_ERR_STATE, LLM_ERR_NONFINITE = -4, -5, -6, -7, -8
LLM_ERR_CHECK = -9
LLM_NUMERICS_EXACT, LLM_NUMERICS_LLAMACPP = 0, 1
LLM_DEBUG_Q, LLM_DEBUG_K, LLM_DEBUG_V, LLM_DEBUG_ATTN_OUT, LLM_DEBUG_FFN_SWIGLU, LLM_DEBUG_FFN_OUT = range(6)


class llm_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_layers", "dim", "n_heads", "n_kv_heads", "head_dim", "ffn_dim",
                                            "vocab", "max_seq", "rope_dims")] + \
               [("eps", ctypes.c_float), ("rope_base", ctypes.c_float), ("rope_neox", ctypes.c_int),
                ("wtype", ctypes.c_int), ("numerics", ctypes.c_int)]


class llm_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("attn_norm", "ffn_norm", "bq", "bk", "bv", "wq", "wk", "wv", "wo",
                                               "w_gate", "w_up", "w_down")]


class llm_weights(ctypes.Structure):
    _fields_ = [("tok_embd", ctypes.c_void_p), ("output_norm", ctypes.c_void_p), ("output", ctypes.c_void_p),
                ("rope_freqs", ctypes.c_void_p), ("layers", ctypes.POINTER(llm_layer_weights))]


class llm_gguf_layout(ctypes.Structure):
    _fields_ = [("version", ctypes.c_uint32), ("n_tensors", ctypes.c_int64), ("n_kv", ctypes.c_int64),
                ("alignment", ctypes.c_uint64), ("infos_end", ctypes.c_uint64), ("data_start", ctypes.c_uint64),
                ("file_size", ctypes.c_uint64)]


class llm_gguf_tensor(ctypes.Structure):
    _fields_ = [("type", ctypes.c_int32), ("n_dims", ctypes.c_int32), ("dims", ctypes.c_int64 * 4),
                ("offset", ctypes.c_uint64), ("file_offset", ctypes.c_uint64), ("bytes", ctypes.c_uint64),
                ("data", ctypes.c_void_p)]


_vp, _i32, _int = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int
_SIGS = {
    "llm_create": ([ctypes.POINTER(llm_config), ctypes.POINTER(llm_weights), _vp, ctypes.POINTER(_vp)], _int),
    "llm_reset": ([_vp], _int),
    "llm_decode_step": ([_vp, _i32, _i32, _vp, _vp], _int),
    "llm_decode_step_async": ([_vp, _vp, _i32, _vp], _int),
    "llm_generate": ([_vp, _i32, _i32, _i32, _vp], _int),
    "llm_prefill": ([_vp, _vp, _i32, _i32, _vp, _vp], _int),
    "llm_sync": ([_vp], _int),
    "llm_logits_device": ([_vp], _vp),
    "llm_get_config": ([_vp, ctypes.POINTER(llm_config)], _int),
    "llm_kv_view": ([_vp, _int, ctypes.POINTER(_vp), ctypes.POINTER(_vp)], _int),
    "llm_test_kv_store": ([_vp, _int, _i32, _vp, _vp], _int),
    "llm_test_dequant_rows": ([_vp, _int, _int, _i32, _i32, _vp], _int),
    "llm_test_gemv": ([_vp, _int, _int, _vp, _vp], _int),
    "llm_column_groups": ([_vp], _int),
    "llm_trace_read": ([_vp, _vp, ctypes.POINTER(_i32)], _int),
    "llm_decode_step_noalloc": ([_vp, _vp, _i32, _vp, _vp], _int),
    "llm_launch_count": ([_vp], ctypes.c_int64),
    "llm_destroy": ([_vp], None),
    "llm_gguf_open": ([ctypes.c_char_p, ctypes.POINTER(_vp), ctypes.c_char_p, ctypes.c_size_t], _int),
    "llm_gguf_close": ([_vp], None),
    "llm_gguf_summary": ([_vp, ctypes.POINTER(llm_gguf_layout)], _int),
    "llm_gguf_find_tensor": ([_vp, ctypes.c_char_p, ctypes.POINTER(llm_gguf_tensor)], _int),
    "llm_gguf_tensor_at": ([_vp, ctypes.c_int64, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(llm_gguf_tensor)],
                           _int),
    "llm_gguf_meta_at": ([_vp, ctypes.c_int64, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(_i32)], _int),
    "llm_gguf_meta_type": ([_vp, ctypes.c_char_p, ctypes.POINTER(_i32), ctypes.POINTER(_i32),
                            ctypes.POINTER(ctypes.c_uint64)], _int),
    "llm_gguf_meta_int": ([_vp, ctypes.c_char_p, ctypes.POINTER(ctypes.c_int64)], _int),
    "llm_gguf_meta_float": ([_vp, ctypes.c_char_p, ctypes.POINTER(ctypes.c_double)], _int),
    "llm_gguf_meta_string": ([_vp, ctypes.c_char_p, ctypes.POINTER(_vp), ctypes.POINTER(ctypes.c_uint64)], _int),
    "llm_gguf_config": ([_vp, _i32, ctypes.POINTER(llm_config), ctypes.c_char_p, ctypes.c_size_t], _int),
    "llm_create_from_gguf": ([_vp, _i32, _vp, ctypes.POINTER(_vp), ctypes.c_char_p, ctypes.c_size_t], _int),
    "llm_status_string": ([_int], ctypes.c_char_p),
    "llm_last_error": ([_vp], ctypes.c_char_p),
    "llm_test_fail_alloc": ([_i32], _int),
    "llm_checked_build": ([], _int),
    "llm_debug_tensor": ([_vp, _int, _int, _vp, _i32], _int),
    "llm_test_logits_limit": ([_vp, _i32], _int),
    "llm_test_guards": ([_vp], ctypes.c_int64),
    "llm_test_poke_guard": ([_vp, _int], _int),
    "llm_prefill_f16_copy": ([_vp, _int], _int),
}


def declared_symbols(header: str | None = None) -> list[str]:
    """Names of the functions include/llm.h declares."""
    import re
    header = header or os.path.join(_build.ROOT, "include", "llm.h")
    with open(header) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(llm_\w+)\s*\(", text, re.M)))


def load_library(path: str | None = None):
    """The library at `path`, or the in-tree build: LLM_DECODE_VARIANT=checked
    (device-side index checks) or =trace (phase stamps) selects a variant."""
    if path is None:
        variant = os.environ.get("LLM_DECODE_VARIANT", "")
        if variant not in ("", "checked", "trace"):
            raise ValueError(f"LLM_DECODE_VARIANT={variant!r}: expected checked or trace")
        path = _build.build(checked=variant == "checked", trace=variant == "trace")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = load_library()
LIBRARY_PATH = _lib._name


class LlmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_lib.llm_status_string(status).decode()} ({status}): {message}")
        self.status = status


def _check(rc: int, h=None):
    if rc != LLM_OK:
        msg = _lib.llm_last_error(h).decode() if h else ""
        raise LlmError(rc, msg)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


# ------------------------------------------------------ the C functions --
def llm_create(cfg: llm_config, weights: llm_weights, stream=None):
    h = _vp()
    rc = _lib.llm_create(ctypes.byref(cfg), ctypes.byref(weights), stream, ctypes.byref(h))
    if rc != LLM_OK:
        raise LlmError(rc, _lib.llm_last_error(None).decode())     # this thread's failed create
    return h.value


def llm_reset(h):
    _check(_lib.llm_reset(h), h)


def llm_get_config(h) -> llm_config:
    c = llm_config()
    _check(_lib.llm_get_config(h, ctypes.byref(c)), h)
    return c


def _check_logits_buffer(h, logits_host):
    """The C call writes vocab floats to logits_host: refuse a buffer that
    cannot hold them instead of letting the library write past its end."""
    if logits_host is None:
        return
    if not isinstance(logits_host, np.ndarray) or logits_host.dtype != np.float32 or \
            not logits_host.flags.c_contiguous or not logits_host.flags.writeable:
        raise TypeError("logits_host must be a writable C-contiguous float32 numpy array")
    vocab = llm_get_config(h).vocab
    if logits_host.size < vocab:
        raise ValueError(f"logits_host holds {logits_host.size} floats; the model's vocab is {vocab}")


def llm_decode_step(h, token: int, pos: int, logits_host: np.ndarray | None = None) -> int:
    out = ctypes.c_int32(0)
    _check_logits_buffer(h, logits_host)
    _check(_lib.llm_decode_step(h, int(token), int(pos), _ptr(logits_host), ctypes.addressof(out)), h)
    return out.value


def llm_decode_step_async(h, token_dev, pos: int, argmax_dev):
    _check(_lib.llm_decode_step_async(h, _ptr(token_dev), int(pos), _ptr(argmax_dev)), h)


def llm_generate(h, token: int, pos: int, n_steps: int, tokens_dev):
    _check(_lib.llm_generate(h, int(token), int(pos), int(n_steps), _ptr(tokens_dev)), h)


def llm_prefill(h, tokens_host, pos0: int, logits_host: np.ndarray | None = None) -> int:
    t = np.ascontiguousarray(tokens_host, dtype=np.int32)
    out = ctypes.c_int32(0)
    _check_logits_buffer(h, logits_host)
    _check(_lib.llm_prefill(h, t.ctypes.data, t.size, int(pos0), _ptr(logits_host), ctypes.addressof(out)), h)
    return out.value


def llm_prefill_f16_copy(h, enable: bool = True) -> None:
    """Keep (or free) the F16 copy of a Q8_0 handle's layer matrices that the
    batched prefill's GEMMs then read."""
    _check(_lib.llm_prefill_f16_copy(h, 1 if enable else 0), h)


def llm_sync(h):
    _check(_lib.llm_sync(h), h)


def llm_logits_device(h) -> int:
    return _lib.llm_logits_device(h)


def llm_kv_view(h, layer: int):
    k, v = _vp(), _vp()
    _check(_lib.llm_kv_view(h, layer, ctypes.byref(k), ctypes.byref(v)), h)
    return k.value, v.value


def llm_test_kv_store(h, layer: int, pos: int, k_dev, v_dev):
    _check(_lib.llm_test_kv_store(h, layer, pos, _ptr(k_dev), _ptr(v_dev)), h)


def llm_test_dequant_rows(h, which: int, layer: int, row0: int, n_rows: int, out_dev):
    _check(_lib.llm_test_dequant_rows(h, which, layer, row0, n_rows, _ptr(out_dev)), h)


def llm_test_gemv(h, which: int, layer: int, x_dev, y_dev):
    _check(_lib.llm_test_gemv(h, which, layer, _ptr(x_dev), _ptr(y_dev)), h)


def llm_column_groups(h) -> int:
    return int(_lib.llm_column_groups(h))


def llm_debug_tensor(h, layer: int, which: int) -> np.ndarray:
    """One named intermediate of the last decode step (LLM_DEBUG_*)."""
    c = llm_get_config(h)
    q_dim, kv_dim = c.n_heads * c.head_dim, c.n_kv_heads * c.head_dim
    n = {LLM_DEBUG_Q: q_dim, LLM_DEBUG_K: kv_dim, LLM_DEBUG_V: kv_dim, LLM_DEBUG_ATTN_OUT: c.dim,
         LLM_DEBUG_FFN_SWIGLU: c.ffn_dim, LLM_DEBUG_FFN_OUT: c.dim}.get(which, 0)
    out = np.empty(max(n, 1), np.float32)
    _check(_lib.llm_debug_tensor(h, int(layer), int(which), out.ctypes.data, n), h)
    return out[:n]


def llm_checked_build() -> bool:
    return bool(_lib.llm_checked_build())


def llm_test_logits_limit(h, limit: int) -> None:
    _check(_lib.llm_test_logits_limit(h, int(limit)), h)


def llm_test_fail_alloc(nth: int) -> None:
    _check(_lib.llm_test_fail_alloc(int(nth)))


def llm_test_guards(h) -> int:
    """Changed guard-band bytes around the handle's KV cache, activations
    and prefill workspace (0 when intact)."""
    n = int(_lib.llm_test_guards(h))
    if n < 0:
        _check(n, h)
    return n


def llm_test_poke_guard(h, band: int) -> None:
    _check(_lib.llm_test_poke_guard(h, int(band)), h)


def llm_decode_step_noalloc(h, token_dev, pos: int, logits_dev, argmax_dev):
    """One decode step that allocates nothing: its working memory is a fixed
    device array of the library (for callers that may not allocate device
    memory while serving).  All three buffers are device tensors; synchronous."""
    _check(_lib.llm_decode_step_noalloc(h, _ptr(token_dev), int(pos), _ptr(logits_dev), _ptr(argmax_dev)), h)


def llm_trace_read(h) -> np.ndarray:
    """Phase stamps of the last step, [sms][1024] uint64 ns (LLM_TRACE builds only)."""
    n = _i32()
    buf = np.zeros(1024 * 1024, np.uint64)
    _check(_lib.llm_trace_read(h, buf.ctypes.data, ctypes.byref(n)), h)
    return buf[: n.value * 1024].reshape(n.value, 1024).copy()


def llm_launch_count(h) -> int:
    return _lib.llm_launch_count(h)


def llm_destroy(h):
    _lib.llm_destroy(h)


def llm_status_string(status: int) -> str:
    return _lib.llm_status_string(status).decode()


def llm_last_error(h) -> str:
    return _lib.llm_last_error(h).decode()


# ------------------------------------------------------- device plumbing --
def config_struct(cfg) -> llm_config:
    return llm_config(n_layers=cfg.n_layers, dim=cfg.dim, n_heads=cfg.n_heads, n_kv_heads=cfg.n_kv_heads,
                      head_dim=cfg.head_dim, ffn_dim=cfg.ffn_dim, vocab=cfg.vocab, max_seq=cfg.max_seq,
                      rope_dims=cfg.rope_dims, eps=cfg.eps, rope_base=cfg.rope_base, rope_neox=int(cfg.rope_neox),
                      wtype=int(cfg.wtype), numerics=int(getattr(cfg, "numerics", LLM_NUMERICS_EXACT)))


class DeviceWeights:
    """Host arrays (GGUF layout) copied into CUDA tensors, and the llm_weights
    record pointing at them.  ``host`` needs tok_embd, output_norm, output,
    rope_freqs and ``layers`` (dicts with the llm_layer_weights names)."""

    def __init__(self, host, device="cuda"):
        import torch
        self.tensors = []

        def up(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                a = a.view(np.int16)
            t = torch.from_numpy(a).to(device)
            self.tensors.append(t)
            return t.data_ptr()

        n = len(host.layers)
        self._layers = (llm_layer_weights * n)()
        for l, L in enumerate(host.layers):
            for name, _ in llm_layer_weights._fields_:
                setattr(self._layers[l], name, up(L.get(name)))
        self.struct = llm_weights(tok_embd=up(host.tok_embd), output_norm=up(host.output_norm),
                                  output=up(host.output), rope_freqs=up(host.rope_freqs), layers=self._layers)

    def free(self):
        self.tensors.clear()


class Decoder:
    """A handle plus its uploaded weights (the weights may be freed after
    creation: the library keeps its own copy)."""

    def __init__(self, cfg, host_weights, stream=None, keep_weights: bool = False):
        import torch
        self.cfg = cfg
        dw = DeviceWeights(host_weights)
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        self.stream = stream
        self.h = llm_create(config_struct(cfg), dw.struct, stream)
        torch.cuda.synchronize()
        if not keep_weights:
            dw.free()
        self.dw = dw

    def close(self):
        if getattr(self, "h", None):
            llm_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def kv_tensors(self, layer: int):
        """(K, V) of one layer as int16 CUDA tensors [max_seq, kv_dim] viewing the cache."""
        import torch
        k, v = llm_kv_view(self.h, layer)
        kv_dim = self.cfg.n_kv_heads * self.cfg.head_dim
        n = self.cfg.max_seq * kv_dim
        return (_wrap_device(k, n, torch.int16).view(self.cfg.max_seq, kv_dim),
                _wrap_device(v, n, torch.int16).view(self.cfg.max_seq, kv_dim))

    def logits_tensor(self):
        import torch
        return _wrap_device(llm_logits_device(self.h), self.cfg.vocab, torch.float32)


# ------------------------------------------------------------ GGUF --
class GgufFile:
    """A GGUF file opened by the library (llm_gguf_open): checked at open,
    memory-mapped until close().  Raises LlmError with the library's reason."""

    def __init__(self, path: str):
        err = ctypes.create_string_buffer(512)
        g = _vp()
        rc = _lib.llm_gguf_open(os.fsencode(path), ctypes.byref(g), err, len(err))
        if rc != LLM_OK:
            raise LlmError(rc, err.value.decode())
        self.g = g.value

    def close(self):
        if getattr(self, "g", None):
            _lib.llm_gguf_close(self.g)
            self.g = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def summary(self) -> dict:
        s = llm_gguf_layout()
        _check(_lib.llm_gguf_summary(self.g, ctypes.byref(s)))
        return {n: getattr(s, n) for n, _ in llm_gguf_layout._fields_}

    @staticmethod
    def _tensor_dict(t: llm_gguf_tensor) -> dict:
        return {"type": t.type, "dims": [t.dims[i] for i in range(t.n_dims)], "offset": t.offset,
                "file_offset": t.file_offset, "bytes": t.bytes, "data": t.data}

    def tensor(self, name: str) -> dict | None:
        t = llm_gguf_tensor()
        rc = _lib.llm_gguf_find_tensor(self.g, name.encode(), ctypes.byref(t))
        if rc == LLM_ERR_OUT_OF_RANGE:
            return None
        _check(rc)
        return self._tensor_dict(t)

    def tensors(self) -> list:
        out, i = [], 0
        while True:
            name, t = ctypes.c_char_p(), llm_gguf_tensor()
            rc = _lib.llm_gguf_tensor_at(self.g, i, ctypes.byref(name), ctypes.byref(t))
            if rc == LLM_ERR_OUT_OF_RANGE:
                return out
            _check(rc)
            out.append((name.value.decode(), self._tensor_dict(t)))
            i += 1

    def keys(self) -> list:
        out, i = [], 0
        while True:
            key, t = ctypes.c_char_p(), _i32()
            rc = _lib.llm_gguf_meta_at(self.g, i, ctypes.byref(key), ctypes.byref(t))
            if rc == LLM_ERR_OUT_OF_RANGE:
                return out
            _check(rc)
            out.append((key.value.decode(), t.value))
            i += 1

    def meta_type(self, key: str):
        t, et, n = _i32(), _i32(), ctypes.c_uint64()
        _check(_lib.llm_gguf_meta_type(self.g, key.encode(), ctypes.byref(t), ctypes.byref(et), ctypes.byref(n)))
        return t.value, et.value, n.value

    def meta_int(self, key: str) -> int:
        v = ctypes.c_int64()
        _check(_lib.llm_gguf_meta_int(self.g, key.encode(), ctypes.byref(v)))
        return v.value

    def meta_float(self, key: str) -> float:
        v = ctypes.c_double()
        _check(_lib.llm_gguf_meta_float(self.g, key.encode(), ctypes.byref(v)))
        return v.value

    def meta_string(self, key: str) -> str:
        p, n = _vp(), ctypes.c_uint64()
        _check(_lib.llm_gguf_meta_string(self.g, key.encode(), ctypes.byref(p), ctypes.byref(n)))
        return ctypes.string_at(p.value, n.value).decode("utf-8") if n.value else ""

    def config(self, max_seq: int = 0) -> llm_config:
        c, err = llm_config(), ctypes.create_string_buffer(512)
        rc = _lib.llm_gguf_config(self.g, int(max_seq), ctypes.byref(c), err, len(err))
        if rc != LLM_OK:
            raise LlmError(rc, err.value.decode())
        return c


def llm_create_from_gguf(gguf: GgufFile, max_seq: int = 0, stream=None):
    h, err = _vp(), ctypes.create_string_buffer(512)
    rc = _lib.llm_create_from_gguf(gguf.g, int(max_seq), stream, ctypes.byref(h), err, len(err))
    if rc != LLM_OK:
        raise LlmError(rc, err.value.decode())
    return h.value


class GgufDecoder(Decoder):
    """A handle created from a GGUF file (llm_create_from_gguf); ``cfg`` holds
    the shape the library derived from the file's metadata."""

    def __init__(self, path: str, max_seq: int = 0, stream=None):
        import torch
        from types import SimpleNamespace
        with GgufFile(path) as g:
            c = g.config(max_seq)
            self.cfg = SimpleNamespace(**{n: getattr(c, n) for n, _ in llm_config._fields_})
            if stream is None:
                stream = torch.cuda.current_stream().cuda_stream
            self.stream = stream
            self.h = llm_create_from_gguf(g, max_seq, stream)
        torch.cuda.synchronize()
        self.dw = None


def _wrap_device(ptr: int, n: int, dtype):
    """A torch view of library-owned device memory (no copy, no ownership)."""
    import torch
    itemsize = torch.tensor([], dtype=dtype).element_size()

    class _Holder:
        __cuda_array_interface__ = {
            "shape": (n,), "typestr": {torch.int16: "<i2", torch.float32: "<f4", torch.int32: "<i4"}[dtype],
            "data": (ptr, False), "version": 3, "strides": (itemsize,)}

    return torch.as_tensor(_Holder(), device="cuda")
