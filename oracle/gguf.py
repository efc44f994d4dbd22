"""CPU oracle for reading GGUF model files.

TEST INFRASTRUCTURE.  A plain Python reader of the GGUF version 3 layout as
"Loading GGUF with the FFM API" (codeloopback.dev, llm-gguf-loader-ffm)
describes it, and the model-shape rules of "The Forward Pass in Java"
(Example 1, Config record).  Used only by tests/ to check the library's
native reader on the same files; the product path never imports it, and it
shares no code with the library.

Parity status: pinned by the ``-m "not gpu"`` tests against the byte
positions, offsets and rejection messages the loader page prints for its
worked examples (Examples 3, 4, 5 and 11) and the two configurations "The
Forward Pass in Java" prints in Example 1.
"""
from __future__ import annotations

import struct

import numpy as np

MAGIC = 0x46554747                  # "GGUF" read as a little-endian uint32 (loader page, Example 1)
VERSION = 3                         # the version this reader accepts (Example 11)
DEFAULT_ALIGNMENT = 32              # when general.alignment is absent (Example 5)
F32, F16, Q8_0 = 0, 1, 8            # ggml tensor type ids (Example 13)

# Metadata value types (Example 13, Cursor.value)
UINT8, INT8, UINT16, INT16, UINT32, INT32, FLOAT32, BOOL, STRING, ARRAY, UINT64, INT64, FLOAT64 = range(13)
_SCALAR = {UINT8: ("<B", 1), INT8: ("<b", 1), UINT16: ("<H", 2), INT16: ("<h", 2), UINT32: ("<I", 4),
           INT32: ("<i", 4), FLOAT32: ("<f", 4), BOOL: ("<B", 1), UINT64: ("<Q", 8), INT64: ("<q", 8),
           FLOAT64: ("<d", 8)}


class GgufError(ValueError):
    """A file the reader rejects; the message says which check failed."""


class _Cursor:
    """Little-endian reads from a byte string, each one bounds-checked."""

    def __init__(self, data: bytes, pos: int = 0):
        self.data, self.pos = data, pos

    def take(self, n: int) -> bytes:
        if n < 0 or self.pos + n > len(self.data):
            raise GgufError(f"truncated: {n} bytes needed at {self.pos}, file has {len(self.data)}")
        b = self.data[self.pos:self.pos + n]
        self.pos += n
        return b

    def scalar(self, t: int):
        fmt, n = _SCALAR[t]
        v = struct.unpack(fmt, self.take(n))[0]
        return bool(v) if t == BOOL else v

    def u32(self) -> int:
        return self.scalar(UINT32)

    def u64(self) -> int:
        return self.scalar(UINT64)

    def string(self) -> str:
        n = self.u64()                              # byte length, then UTF-8 bytes, no terminator (Example 4)
        return self.take(n).decode("utf-8")

    def value(self, t: int):
        if t == STRING:
            return self.string()
        if t == ARRAY:                              # element type, element count, elements (Example 4)
            et = self.u32()
            n = self.u64()
            if et not in _SCALAR and et not in (STRING, ARRAY):
                raise GgufError(f"bad array element type {et} at {self.pos}")
            return (et, [self.value(et) for _ in range(n)])
        if t not in _SCALAR:
            raise GgufError(f"bad value type {t} at {self.pos}")
        return self.scalar(t)


def tensor_bytes(t: int, dims) -> int:
    """Bytes of a tensor of type t (Example 13, TensorInfo.byteSize)."""
    n = 1
    for d in dims:
        n *= d
    if t == F32:
        return 4 * n
    if t == F16:
        return 2 * n
    if t == Q8_0:
        if dims[0] % 32:
            raise GgufError(f"Q8_0 rows of {dims[0]} values are not whole 32-value blocks")
        return n // 32 * 34
    raise GgufError(f"unsupported ggml type {t}")


def pad(n: int, alignment: int) -> int:
    return (n + alignment - 1) // alignment * alignment


def read(data: bytes) -> dict:
    """Parse and check a whole GGUF file, in the loader page's order (Example
    11): size of the header, magic, version, then metadata and tensor infos,
    each tensor's offset against the padded sizes before it, and each
    tensor's end against the file size.  Returns the header counts, the
    metadata {key: (type, value)} in file order, the tensor infos in file
    order, the alignment, where the infos end and where the data starts."""
    if len(data) < 24:
        raise GgufError("shorter than the 24-byte header")
    c = _Cursor(data)
    magic = c.u32()
    if magic != MAGIC:
        raise GgufError(f"magic 0x{magic:08X} is not GGUF")
    version = c.u32()
    if version != VERSION:
        raise GgufError(f"version {version} (this loader reads {VERSION})")
    n_tensors, n_kv = c.u64(), c.u64()
    meta = {}
    for _ in range(n_kv):
        key = c.string()
        t = c.u32()
        meta[key] = (t, c.value(t))
    tensors = []
    for _ in range(n_tensors):
        name = c.string()
        nd = c.u32()
        dims = [c.u64() for _ in range(nd)]
        t = c.u32()
        off = c.u64()
        tensors.append({"name": name, "dims": dims, "type": t, "offset": off})
    infos_end = c.pos
    alignment = DEFAULT_ALIGNMENT
    if "general.alignment" in meta:
        t, v = meta["general.alignment"]
        if t != UINT32 or v == 0:
            raise GgufError("general.alignment must be a nonzero UINT32")
        alignment = v
    data_start = pad(infos_end, alignment)
    expect = 0
    for i, ti in enumerate(tensors):
        ti["bytes"] = tensor_bytes(ti["type"], ti["dims"])
        if ti["offset"] != expect:
            which = "first tensor" if i == 0 else f"tensor {ti['name']}"
            raise GgufError(f"{which} offset {ti['offset']}, expected {expect}")
        expect += pad(ti["bytes"], alignment)
    for ti in tensors:
        end = data_start + ti["offset"] + ti["bytes"]
        if end > len(data):
            raise GgufError(f"tensor needs bytes up to {end}, file has {len(data)}")
        ti["file_offset"] = data_start + ti["offset"]
    return {"version": version, "n_tensors": n_tensors, "n_kv": n_kv, "metadata": meta, "tensors": tensors,
            "alignment": alignment, "infos_end": infos_end, "data_start": data_start}


def tensor_floats(data: bytes, info: dict) -> np.ndarray:
    """A tensor's values as float32 (Example 13, floats(): F32 as stored, F16
    widened, Q8_0 as d * qs per 32-value block), in file order."""
    raw = np.frombuffer(data, dtype=np.uint8, count=info["bytes"], offset=info["file_offset"])
    if info["type"] == F32:
        return raw.view("<f4").astype(np.float32)
    if info["type"] == F16:
        return raw.view("<f2").astype(np.float32)
    blocks = raw.reshape(-1, 34)
    d = blocks[:, :2].copy().view("<f2").astype(np.float32)
    q = blocks[:, 2:].view(np.int8).astype(np.float32)
    return (d * q).reshape(-1)


def model_config(meta: dict) -> dict:
    """The model shape from the metadata ("The Forward Pass in Java", Example 1,
    Config.from): keys under the architecture's prefix, with the defaults the
    page gives for the optional ones (head_count_kv = head_count, freq_base
    10000, dimension_count = dim / heads, vocabulary = the tokenizer's token
    count), and the RoPE pair layout by architecture (llama normal, qwen2
    NEOX)."""
    def get(k, default=None):
        if k in meta:
            return meta[k][1]
        if default is None:
            raise GgufError(f"missing key {k}")
        return default

    a = get("general.architecture")
    if a not in ("llama", "qwen2"):
        raise GgufError(f"architecture not supported here: {a}")
    dim, heads = int(get(a + ".embedding_length")), int(get(a + ".attention.head_count"))
    kv_heads = int(get(a + ".attention.head_count_kv", heads))
    if a + ".vocab_size" in meta:
        vocab = int(meta[a + ".vocab_size"][1])
    else:
        vocab = len(get("tokenizer.ggml.tokens")[1])
    return {"arch": a, "dim": dim, "layers": int(get(a + ".block_count")), "heads": heads, "kv_heads": kv_heads,
            "head_dim": dim // heads, "ffn": int(get(a + ".feed_forward_length")), "vocab": vocab,
            "context_length": int(get(a + ".context_length")),
            "eps": float(np.float32(get(a + ".attention.layer_norm_rms_epsilon"))),
            "rope_base": float(np.float32(get(a + ".rope.freq_base", 10000.0))),
            "rope_dims": int(get(a + ".rope.dimension_count", dim // heads)), "neox": a == "qwen2"}
