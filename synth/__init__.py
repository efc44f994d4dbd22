"""Seeded synthetic inputs: model shapes, random weights, prompts and KV rows.

Both the CPU oracle and the CUDA decode library are fed from here.  This
module draws random numbers and encodes them in the weight formats of the
GGUF files the pages read (F32, F16, 34-byte Q8_0 blocks); it computes
nothing of the forward pass.  The generator itself is ``synth.c`` (counter
based SplitMix64 + Box-Muller), built on first use with the host compiler.

Recipe (one per workload; shapes from the pages' models):
  * float weights ~ N(0, 0.02), stored F32 or F16 (round to nearest even);
  * norm gains ~ 1 + N(0, 0.1); Q/K/V biases (F32) ~ N(0, 0.02);
  * Q8_0 blocks: quants uniform over -127..127, scale f16(|N(0,0.02)| / 127);
  * prompts: token ids uniform over [0, vocab);
  * pre-filled KV rows: f16(N(0, 1)).
Seeds: weights 0xC0FFEE00 + n, prompt + 1, KV rows + 2 (n = workload number).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

F32, F16, Q8_0 = 0, 1, 8
_HERE = os.path.dirname(os.path.abspath(__file__))
_LOCK = threading.Lock()
_LIB = None


def build(force: bool = False) -> str:
    """Compile synth.c into synth/_build/libsynth.so (host compiler, OpenMP)."""
    src = os.path.join(_HERE, "synth.c")
    out_dir = os.path.join(_HERE, "_build")
    out = os.path.join(out_dir, "libsynth.so")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(out_dir, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-std=gnu11", "-O2", "-fPIC", "-shared", "-fopenmp",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = build()
            try:
                lib = ctypes.CDLL(path)
            except OSError:                       # stale binary from another machine
                lib = ctypes.CDLL(build(force=True))
            u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.syn_normal_f32.argtypes = [u64, u64, i64, dbl, dbl, vp]
            lib.syn_normal_f16.argtypes = [u64, u64, i64, dbl, dbl, vp]
            lib.syn_uniform_i32.argtypes = [u64, u64, i64, ctypes.c_int32, ctypes.c_int32, vp]
            lib.syn_q8_0.argtypes = [u64, u64, i64, dbl, vp]
            lib.syn_splitmix64_at.argtypes = [u64, u64]
            lib.syn_splitmix64_at.restype = u64
            lib.syn_draw.argtypes = [u64, u64, u64]
            lib.syn_draw.restype = u64
            lib.syn_normal_at.argtypes = [u64, u64, u64]
            lib.syn_normal_at.restype = dbl
            _LIB = lib
    return _LIB


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def normal_f32(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _lib().syn_normal_f32(seed, stream, n, mean, std, _p(out))
    return out


def normal_f16(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """FP16 bit patterns (uint16) of N(mean, std) samples."""
    out = np.empty(n, dtype=np.uint16)
    _lib().syn_normal_f16(seed, stream, n, mean, std, _p(out))
    return out


def uniform_i32(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _lib().syn_uniform_i32(seed, stream, n, lo, hi, _p(out))
    return out


def q8_0_blocks(seed: int, stream: int, n_elems: int, std: float = 0.02) -> np.ndarray:
    assert n_elems % 32 == 0
    out = np.empty((n_elems // 32) * 34, dtype=np.uint8)
    _lib().syn_q8_0(seed, stream, n_elems // 32, std, _p(out))
    return out


# ----------------------------------------------------------------- shapes --
@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    dim: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    max_seq: int
    eps: float
    rope_base: float
    rope_neox: int
    wtype: int
    tied: bool
    bias: bool = False
    rope_freqs: bool = False          # pass explicit (unit) frequency factors
    number: int = 0                   # workload number, picks the seeds
    numerics: int = 0                 # llm_numerics of the library handle (0 exact, 1 llama.cpp rounding)

    @property
    def rope_dims(self) -> int:
        return self.head_dim

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def scaled(self, **kw) -> "ModelConfig":
        d = dict(self.__dict__)
        d.update(kw)
        return ModelConfig(**d)


# The five workloads.  Shapes and distributions as stated for each; where a
# value is not stated the reading is recorded beside it.
TINY = ModelConfig("tiny-llama-f32", n_layers=4, dim=256, n_heads=8, n_kv_heads=2, head_dim=32,
                   ffn_dim=768, vocab=151936, max_seq=4096, eps=1e-5, rope_base=10000.0,
                   rope_neox=0, wtype=F32, tied=False, number=1)
STORIES15M = ModelConfig("stories15M-f32", n_layers=6, dim=288, n_heads=6, n_kv_heads=6, head_dim=48,
                         ffn_dim=768, vocab=32000, max_seq=256, eps=1e-5, rope_base=10000.0,
                         rope_neox=0, wtype=F32, tied=False, number=2)
LLAMA1B_Q8 = ModelConfig("llama-3.2-1b-q8_0", n_layers=16, dim=2048, n_heads=32, n_kv_heads=8, head_dim=64,
                         ffn_dim=8192, vocab=128256, max_seq=32768, eps=1e-5, rope_base=500000.0,
                         rope_neox=0, wtype=Q8_0, tied=True, rope_freqs=True, number=3)
QWEN2_F16 = ModelConfig("qwen2-1b-f16", n_layers=16, dim=2048, n_heads=32, n_kv_heads=8, head_dim=64,
                        ffn_dim=8192, vocab=128256, max_seq=640, eps=1e-5, rope_base=1000000.0,
                        rope_neox=1, wtype=F16, tied=True, bias=True, number=4)
LLAMA7B_Q8 = ModelConfig("llama-2-7b-q8_0", n_layers=32, dim=4096, n_heads=32, n_kv_heads=32, head_dim=128,
                         ffn_dim=11008, vocab=32000, max_seq=16384, eps=1e-5, rope_base=10000.0,
                         rope_neox=0, wtype=Q8_0, tied=False, number=5)
WORKLOADS = {c.number: c for c in (TINY, STORIES15M, LLAMA1B_Q8, QWEN2_F16, LLAMA7B_Q8)}


def weight_seed(cfg: ModelConfig) -> int:
    return 0xC0FFEE00 + cfg.number


def prompt_seed(cfg: ModelConfig) -> int:
    return weight_seed(cfg) + 1


def kv_seed(cfg: ModelConfig) -> int:
    return weight_seed(cfg) + 2


# stream ids: one per tensor
_S_EMBD, _S_OUT, _S_OUTNORM, _S_PROMPT = 1, 2, 3, 4
_LAYER_TENSORS = ("attn_norm", "ffn_norm", "bq", "bk", "bv", "wq", "wk", "wv", "wo",
                  "w_gate", "w_up", "w_down")


def _layer_stream(layer: int, name: str) -> int:
    return 64 * (layer + 1) + _LAYER_TENSORS.index(name)


def _kv_stream(layer: int, which: int) -> int:
    return (1 << 40) + 2 * layer + which


@dataclass
class Weights:
    """Host weights in GGUF layout: a [in -> out] matrix is `out` rows of `in`
    values (F32 float32, F16 uint16 bits) or of in/32 Q8_0 blocks (uint8)."""
    cfg: ModelConfig
    tok_embd: np.ndarray
    output_norm: np.ndarray
    output: np.ndarray | None
    rope_freqs: np.ndarray | None
    layers: list = field(default_factory=list)

    def nbytes(self) -> int:
        n = self.tok_embd.nbytes + self.output_norm.nbytes
        n += self.output.nbytes if self.output is not None else 0
        for L in self.layers:
            n += sum(v.nbytes for v in L.values() if v is not None)
        return n


def _matrix(cfg: ModelConfig, seed: int, stream: int, rows: int, cols: int) -> np.ndarray:
    n = rows * cols
    if cfg.wtype == F32:
        return normal_f32(seed, stream, n, 0.0, 0.02)
    if cfg.wtype == F16:
        return normal_f16(seed, stream, n, 0.0, 0.02)
    return q8_0_blocks(seed, stream, n, 0.02)


def make_weights(cfg: ModelConfig, seed: int | None = None) -> Weights:
    s = weight_seed(cfg) if seed is None else seed
    d, q, kv, f = cfg.dim, cfg.q_dim, cfg.kv_dim, cfg.ffn_dim
    w = Weights(cfg=cfg,
                tok_embd=_matrix(cfg, s, _S_EMBD, cfg.vocab, d),
                output_norm=normal_f32(s, _S_OUTNORM, d, 1.0, 0.1),
                output=None if cfg.tied else _matrix(cfg, s, _S_OUT, cfg.vocab, d),
                rope_freqs=np.ones(cfg.rope_dims // 2, dtype=np.float32) if cfg.rope_freqs else None)
    for l in range(cfg.n_layers):
        L = {
            "attn_norm": normal_f32(s, _layer_stream(l, "attn_norm"), d, 1.0, 0.1),
            "ffn_norm": normal_f32(s, _layer_stream(l, "ffn_norm"), d, 1.0, 0.1),
            "bq": normal_f32(s, _layer_stream(l, "bq"), q, 0.0, 0.02) if cfg.bias else None,
            "bk": normal_f32(s, _layer_stream(l, "bk"), kv, 0.0, 0.02) if cfg.bias else None,
            "bv": normal_f32(s, _layer_stream(l, "bv"), kv, 0.0, 0.02) if cfg.bias else None,
            "wq": _matrix(cfg, s, _layer_stream(l, "wq"), q, d),
            "wk": _matrix(cfg, s, _layer_stream(l, "wk"), kv, d),
            "wv": _matrix(cfg, s, _layer_stream(l, "wv"), kv, d),
            "wo": _matrix(cfg, s, _layer_stream(l, "wo"), d, q),
            "w_gate": _matrix(cfg, s, _layer_stream(l, "w_gate"), f, d),
            "w_up": _matrix(cfg, s, _layer_stream(l, "w_up"), f, d),
            "w_down": _matrix(cfg, s, _layer_stream(l, "w_down"), d, f),
        }
        w.layers.append(L)
    return w


def prompt(cfg: ModelConfig, n: int, seed: int | None = None) -> np.ndarray:
    s = prompt_seed(cfg) if seed is None else seed
    return uniform_i32(s, _S_PROMPT, n, 0, cfg.vocab - 1)


def kv_rows(cfg: ModelConfig, layer: int, which: int, n_rows: int, seed: int | None = None) -> np.ndarray:
    """FP16 bits of pre-filled cache rows 0..n_rows-1 of one layer, shape
    [n_rows, n_kv_heads * head_dim]; which: 0 = K, 1 = V."""
    s = kv_seed(cfg) if seed is None else seed
    return normal_f16(s, _kv_stream(layer, which), n_rows * cfg.kv_dim, 0.0, 1.0).reshape(n_rows, cfg.kv_dim)


def draw(seed: int, stream: int, i: int) -> int:
    return int(_lib().syn_draw(seed, stream, i))


def splitmix64_at(state: int, i: int) -> int:
    """Value i of the SplitMix64 sequence whose state starts at ``state``."""
    return int(_lib().syn_splitmix64_at(state, i))


def normal_at(seed: int, stream: int, i: int) -> float:
    """Normal i of a stream (float64, before any rounding to the stored type)."""
    return float(_lib().syn_normal_at(seed, stream, i))
