"""Pins of the oracle's GGUF reader (and of the test writer) against the
worked examples the pages print.

"Loading GGUF with the FFM API": Example 3 (the 24-byte header), Example 4
(strings and arrays: byte positions), Example 5 (tensor infos, alignment 32
and 64, data offsets), Example 11 (the order of the checks and the reason
each broken file is rejected), Example 13 (F16 / Q8_0 decoding).
"The Forward Pass in Java": Example 1 (the model shape from metadata, with
its defaults, for the tiny model and for the qwen2 keys, and the weight
counts derived from it)."""
import numpy as np
import pytest

import oracle
from oracle import gguf as G
import synth
from gguf_writer import (ARRAY, FLOAT32, INT32, STRING, UINT32, UINT64, le, value, write)


def test_header_is_24_bytes():
    # Example 3: magic, version, tensor count, key-value count at 0, 4, 8, 16
    b = write([], [])
    assert b[:4] == b"GGUF" and int.from_bytes(b[:4], "little") == 0x46554747
    assert int.from_bytes(b[4:8], "little") == 3
    g = G.read(b)
    assert (g["n_tensors"], g["n_kv"], g["infos_end"], g["data_start"]) == (0, 0, 24, 32)


def test_strings_and_arrays_byte_positions():
    # Example 4: the string 世界 ends at byte 14, the 4-token string array at
    # 82, the INT32 array [3, 1, 1, 1] at 110
    tokens = ["<s>", "Ġworld", "Ċ", "ä¸ĸçķĮ"]
    s = value(STRING, "世界")
    a = value(ARRAY, (STRING, tokens))
    i = value(ARRAY, (INT32, [3, 1, 1, 1]))
    assert len(s) == 14 and len(s) + len(a) == 82 and len(s) + len(a) + len(i) == 110
    c = G._Cursor(s + a + i)
    assert c.string() == "世界" and c.pos == 14
    assert c.value(ARRAY) == (STRING, tokens) and c.pos == 82
    assert c.value(ARRAY) == (INT32, [3, 1, 1, 1]) and c.pos == 110


def _example5_file(alignment):
    embd = np.zeros(10 * 34, np.uint8)          # Q8_0 [64, 5]: 10 blocks, 340 bytes
    norm = np.ones(64, np.float32)
    return write([("general.architecture", STRING, "llama")],
                 [("token_embd.weight", G.Q8_0, [64, 5], embd.tobytes()),
                  ("output_norm.weight", G.F32, [64], norm.tobytes())], alignment=alignment)


@pytest.mark.parametrize("alignment,infos_end,data_start,norm_offset", [(None, 176, 192, 352), (64, 209, 256, 384)])
def test_tensor_infos_alignment_and_offsets(alignment, infos_end, data_start, norm_offset):
    # Example 5: infos end at 176 (209 with general.alignment = 64), the data
    # section starts at 192 (256); output_norm.weight sits at offset 352 (384),
    # file byte 544 (640)
    g = G.read(_example5_file(alignment))
    assert g["alignment"] == (32 if alignment is None else 64)
    assert (g["infos_end"], g["data_start"]) == (infos_end, data_start)
    e, n = g["tensors"]
    assert (e["name"], e["dims"], e["type"], e["offset"]) == ("token_embd.weight", [64, 5], 8, 0)
    assert (n["name"], n["dims"], n["type"], n["offset"]) == ("output_norm.weight", [64], 0, norm_offset)
    assert (e["file_offset"], n["file_offset"]) == (data_start, data_start + norm_offset)


def _example11_file(magic: str, version: int, offset: int, data_bytes: int) -> bytes:
    # the page's file(): no metadata, one F32 tensor "w" [8] at `offset`,
    # padding to 32 bytes, then data_bytes bytes of data
    o = bytearray(magic.encode("ascii") + le(version, 4) + le(1, 8) + le(0, 8))
    o += le(1, 8) + b"w" + le(1, 4) + le(8, 8) + le(0, 4) + le(offset, 8)
    while len(o) % 32:
        o.append(0)
    return bytes(o + bytes(data_bytes))


EXAMPLE11 = [
    ("good file", _example11_file("GGUF", 3, 0, 32), None),
    ("truncated data", _example11_file("GGUF", 3, 0, 16), "tensor needs bytes up to 96, file has 80"),
    ("wrong magic", _example11_file("GGML", 3, 0, 32), "magic 0x4C4D4747 is not GGUF"),
    ("version 2", _example11_file("GGUF", 2, 0, 32), "version 2 (this loader reads 3)"),
    ("wrong offset", _example11_file("GGUF", 3, 64, 32), "first tensor offset 64, expected 0"),
    ("20 bytes", _example11_file("GGUF", 3, 0, 32)[:20], "shorter than the 24-byte header"),
]


@pytest.mark.parametrize("label,data,reason", EXAMPLE11, ids=[e[0] for e in EXAMPLE11])
def test_checks_in_order(label, data, reason):
    # Example 11: "ok: tensor at 64, 32 bytes" for the good file, and the
    # first failing check's reason for each broken one
    if reason is None:
        g = G.read(data)
        t = g["tensors"][0]
        assert (t["file_offset"], t["bytes"]) == (64, 32)
    else:
        with pytest.raises(G.GgufError) as e:
            G.read(data)
        assert str(e.value) == reason


def test_tensor_sizes():
    # Example 7: a [4, 3] tensor is 12 values, 48 bytes in F32 and 24 in F16;
    # Example 8: 128 Q8_0 values make 4 blocks of 34 bytes, 136 bytes
    assert G.tensor_bytes(G.F32, [4, 3]) == 48 and G.tensor_bytes(G.F16, [4, 3]) == 24
    assert G.tensor_bytes(G.Q8_0, [128]) == 136


def test_header_shorter_than_24_bytes():
    # Example 11: a file shorter than the 24-byte header is rejected before
    # the counts are read, whatever its length
    good = _example11_file("GGUF", 3, 0, 32)
    for n in (0, 4, 8, 16, 20, 23):
        with pytest.raises(G.GgufError) as e:
            G.read(good[:n])
        assert str(e.value) == "shorter than the 24-byte header"


def test_decoding_f16_and_q8_0():
    # Example 13 floats(): F16 widened (Example 6's raw bits 0xB400 = -0.25),
    # Q8_0 as d * qs per block; checked against the C oracle's own decoding
    f16 = np.array([0xB400, 0x3C00, 0x7BFF, 0x0001], np.uint16)
    q8 = synth.q8_0_blocks(7, 3, 64, 0.02)
    data = write([], [("h", G.F16, [4], f16.tobytes()), ("q", G.Q8_0, [64], q8.tobytes())])
    g = G.read(data)
    h, q = g["tensors"]
    got = G.tensor_floats(data, h)
    assert h["bytes"] == 8 and got.size == 4 and G.tensor_floats(data, q).size == 64
    assert got[0] == -0.25 and got[1] == 1.0 and got[2] == 65504.0 and got[3] == np.float32(2.0 ** -24)
    np.testing.assert_array_equal(G.tensor_floats(data, q), oracle.dequant_row(q8, oracle.Q8_0, 0, 64))


TINY_MD = {"general.architecture": (STRING, "llama"), "llama.context_length": (UINT64, 4096),
           "llama.embedding_length": (UINT64, 256), "llama.block_count": (UINT64, 4),
           "llama.feed_forward_length": (UINT64, 704), "llama.attention.head_count": (UINT64, 8),
           "llama.attention.head_count_kv": (UINT64, 2), "llama.rope.dimension_count": (UINT64, 32),
           "llama.attention.layer_norm_rms_epsilon": (FLOAT32, 1e-5), "llama.rope.freq_base": (FLOAT32, 500000.0),
           "tokenizer.ggml.tokens": (ARRAY, (STRING, [""] * 151936))}
QWEN_MD = {"general.architecture": (STRING, "qwen2"), "qwen2.block_count": (UINT64, 32),
           "qwen2.context_length": (UINT64, 32768), "qwen2.embedding_length": (UINT64, 4096),
           "qwen2.feed_forward_length": (UINT64, 11008), "qwen2.attention.head_count": (UINT64, 32),
           "qwen2.attention.head_count_kv": (UINT64, 32), "qwen2.rope.freq_base": (FLOAT32, 1000000.0),
           "qwen2.attention.layer_norm_rms_epsilon": (FLOAT32, 1e-6),
           "tokenizer.ggml.tokens": (ARRAY, (STRING, [""] * 151936))}


@pytest.mark.parametrize("md,expect,per_layer,total", [
    (TINY_MD, dict(arch="llama", dim=256, layers=4, heads=8, kv_heads=2, head_dim=32, ffn=704, vocab=151936,
                   context_length=4096, rope_dims=32, neox=False), 705_024, 80_611_584),
    (QWEN_MD, dict(arch="qwen2", dim=4096, layers=32, heads=32, kv_heads=32, head_dim=128, ffn=11008,
                   vocab=151936, context_length=32768, rope_dims=128, neox=True), 202_383_360, 7_720_931_328)],
    ids=["tiny-llama", "qwen2-keys"])
def test_model_config_and_weight_counts(md, expect, per_layer, total):
    # "The Forward Pass in Java", Example 1: the two printed Config records and
    # the printed weight counts (per layer 2 dim^2 + 2 dim kv_dim + 3 dim ffn
    # + 2 dim; total layers * per layer + 2 vocab dim + dim)
    c = G.model_config(md)
    for k, v in expect.items():
        assert c[k] == v, k
    assert c["eps"] == float(np.float32(1e-5 if c["arch"] == "llama" else 1e-6))
    assert c["rope_base"] == (500000.0 if c["arch"] == "llama" else 1000000.0)
    kv_dim = c["kv_heads"] * c["head_dim"]
    pl = 2 * c["dim"] ** 2 + 2 * c["dim"] * kv_dim + 3 * c["dim"] * c["ffn"] + 2 * c["dim"]
    assert pl == per_layer and c["layers"] * pl + 2 * c["vocab"] * c["dim"] + c["dim"] == total


def test_model_config_defaults():
    # Example 1's defaults: no head_count_kv -> head_count, no freq_base ->
    # 10000, no dimension_count -> dim / heads, vocab from the token list
    md = {k: v for k, v in TINY_MD.items()
          if k not in ("llama.attention.head_count_kv", "llama.rope.freq_base", "llama.rope.dimension_count")}
    c = G.model_config(md)
    assert (c["kv_heads"], c["rope_base"], c["rope_dims"], c["vocab"]) == (8, 10000.0, 32, 151936)
    with pytest.raises(G.GgufError):
        G.model_config({**TINY_MD, "general.architecture": (STRING, "gpt2")})


def test_synthetic_model_round_trip():
    # a seeded model written as GGUF reads back with every tensor intact
    from gguf_writer import model_file
    cfg = synth.ModelConfig("rt", n_layers=2, dim=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96, vocab=50,
                            max_seq=32, eps=1e-5, rope_base=10000.0, rope_neox=1, wtype=synth.Q8_0, tied=False,
                            bias=True, rope_freqs=True, number=91)
    W = synth.make_weights(cfg)
    data = model_file(cfg, W, alignment=64)
    g = G.read(data)
    names = [t["name"] for t in g["tensors"]]
    assert names[0] == "token_embd.weight" and names[-1] == "output.weight" and "blk.1.attn_q.bias" in names
    c = G.model_config(g["metadata"])
    assert (c["arch"], c["dim"], c["layers"], c["heads"], c["kv_heads"], c["ffn"], c["vocab"]) == \
        ("qwen2", 64, 2, 4, 2, 96, 50)
    t = {x["name"]: x for x in g["tensors"]}
    raw = np.frombuffer(data, np.uint8, count=t["blk.1.ffn_down.weight"]["bytes"],
                        offset=t["blk.1.ffn_down.weight"]["file_offset"])
    np.testing.assert_array_equal(raw, W.layers[1]["w_down"].view(np.uint8).reshape(-1))
