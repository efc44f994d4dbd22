"""Writes GGUF version 3 files for tests (the writer the loader page condenses
in its Example 13): header, metadata, tensor infos, padding to the
alignment, and the data section with each tensor padded to the alignment.

Also turns a seeded synthetic model (``synth.Weights``) into a file with the
tensor names and metadata keys of "The Forward Pass in Java" (Examples 1 and
13), so the library's GGUF path can be checked against the same weights.
"""
from __future__ import annotations

import struct

import numpy as np

UINT8, INT8, UINT16, INT16, UINT32, INT32, FLOAT32, BOOL, STRING, ARRAY, UINT64, INT64, FLOAT64 = range(13)
_FMT = {UINT8: "<B", INT8: "<b", UINT16: "<H", INT16: "<h", UINT32: "<I", INT32: "<i", FLOAT32: "<f",
        BOOL: "<B", UINT64: "<Q", INT64: "<q", FLOAT64: "<d"}


def le(v: int, n: int) -> bytes:
    return int(v).to_bytes(n, "little", signed=v < 0)


def gstr(s: str) -> bytes:
    b = s.encode("utf-8")
    return le(len(b), 8) + b


def value(t: int, v) -> bytes:
    if t == STRING:
        return gstr(v)
    if t == ARRAY:
        et, items = v
        return le(et, 4) + le(len(items), 8) + b"".join(value(et, x) for x in items)
    return struct.pack(_FMT[t], v)


def write(metadata, tensors, alignment=None, magic=b"GGUF", version=3, offsets=None) -> bytes:
    """metadata: [(key, type, value)]; tensors: [(name, ggml_type, dims, raw_bytes)].
    alignment None writes no general.alignment key (readers then use 32).
    offsets, when given, replace the computed tensor offsets (for broken files)."""
    al = 32 if alignment is None else alignment
    md = list(metadata)
    if alignment is not None:
        md.append(("general.alignment", UINT32, alignment))
    out = bytearray(magic + le(version, 4) + le(len(tensors), 8) + le(len(md), 8))
    for k, t, v in md:
        out += gstr(k) + le(t, 4) + value(t, v)
    off = 0
    offs = []
    for i, (name, t, dims, raw) in enumerate(tensors):
        o = off if offsets is None else offsets[i]
        offs.append(off)
        out += gstr(name) + le(len(dims), 4) + b"".join(le(d, 8) for d in dims) + le(t, 4) + le(o, 8)
        off += (len(raw) + al - 1) // al * al
    while len(out) % al:
        out.append(0)
    for (name, t, dims, raw), o in zip(tensors, offs):
        out += raw
        while (len(out)) % al:
            out.append(0)
    return bytes(out)


def _raw(a: np.ndarray) -> bytes:
    return np.ascontiguousarray(a).tobytes()


def model_file(cfg, W, arch: str | None = None, vocab_key: bool = True, alignment=None, extra_metadata=()) -> bytes:
    """A GGUF file of a synthetic model: llama or qwen2 keys by its RoPE layout,
    tensors named as llama.cpp names them (token_embd, output_norm, output,
    rope_freqs, blk.N.attn_norm / attn_q / attn_k / attn_v / attn_output /
    ffn_norm / ffn_gate / ffn_up / ffn_down weights, attn_q / attn_k / attn_v
    biases), dims innermost first."""
    a = arch or ("qwen2" if cfg.rope_neox else "llama")
    md = [("general.architecture", STRING, a),
          (f"{a}.context_length", UINT32, cfg.max_seq),
          (f"{a}.embedding_length", UINT32, cfg.dim),
          (f"{a}.block_count", UINT32, cfg.n_layers),
          (f"{a}.feed_forward_length", UINT32, cfg.ffn_dim),
          (f"{a}.attention.head_count", UINT32, cfg.n_heads),
          (f"{a}.attention.head_count_kv", UINT32, cfg.n_kv_heads),
          (f"{a}.attention.layer_norm_rms_epsilon", FLOAT32, cfg.eps),
          (f"{a}.rope.freq_base", FLOAT32, cfg.rope_base),
          (f"{a}.rope.dimension_count", UINT32, cfg.rope_dims)]
    if vocab_key:
        md.append((f"{a}.vocab_size", UINT32, cfg.vocab))
    md += list(extra_metadata)
    wt = cfg.wtype
    tens = [("token_embd.weight", wt, [cfg.dim, cfg.vocab], _raw(W.tok_embd))]
    if W.rope_freqs is not None:
        tens.append(("rope_freqs.weight", 0, [cfg.rope_dims // 2], _raw(W.rope_freqs)))
    for l, L in enumerate(W.layers):
        p = f"blk.{l}."
        tens.append((p + "attn_norm.weight", 0, [cfg.dim], _raw(L["attn_norm"])))
        tens.append((p + "attn_q.weight", wt, [cfg.dim, cfg.q_dim], _raw(L["wq"])))
        tens.append((p + "attn_k.weight", wt, [cfg.dim, cfg.kv_dim], _raw(L["wk"])))
        tens.append((p + "attn_v.weight", wt, [cfg.dim, cfg.kv_dim], _raw(L["wv"])))
        if L.get("bq") is not None:
            tens.append((p + "attn_q.bias", 0, [cfg.q_dim], _raw(L["bq"])))
            tens.append((p + "attn_k.bias", 0, [cfg.kv_dim], _raw(L["bk"])))
            tens.append((p + "attn_v.bias", 0, [cfg.kv_dim], _raw(L["bv"])))
        tens.append((p + "attn_output.weight", wt, [cfg.q_dim, cfg.dim], _raw(L["wo"])))
        tens.append((p + "ffn_norm.weight", 0, [cfg.dim], _raw(L["ffn_norm"])))
        tens.append((p + "ffn_gate.weight", wt, [cfg.dim, cfg.ffn_dim], _raw(L["w_gate"])))
        tens.append((p + "ffn_up.weight", wt, [cfg.dim, cfg.ffn_dim], _raw(L["w_up"])))
        tens.append((p + "ffn_down.weight", wt, [cfg.ffn_dim, cfg.dim], _raw(L["w_down"])))
    tens.append(("output_norm.weight", 0, [cfg.dim], _raw(W.output_norm)))
    if W.output is not None:
        tens.append(("output.weight", wt, [cfg.dim, cfg.vocab], _raw(W.output)))
    return write(md, tens, alignment=alignment)
