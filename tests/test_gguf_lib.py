"""The library's native GGUF reader (llm_gguf_*, host code, no GPU) against
the oracle's reader on the same files: the loader page's example files, the
13 metadata value types, synthetic models of every weight type, the model
shape, and the checks that reject a file or a model before any device work."""
import numpy as np
import pytest

from oracle import gguf as G
import synth
import gguf_writer as W
from test_gguf_oracle import EXAMPLE11, _example5_file


@pytest.fixture(scope="module")
def lib():
    import llama_decode_forward_gb300 as L
    return L


def _save(tmp_path, name, data):
    p = tmp_path / name
    p.write_bytes(data)
    return str(p)


@pytest.mark.parametrize("label,data,reason", EXAMPLE11, ids=[e[0] for e in EXAMPLE11])
def test_example11_checks(lib, tmp_path, label, data, reason):
    path = _save(tmp_path, "f.gguf", data)
    if reason is None:
        with lib.GgufFile(path) as g:
            t = g.tensor("w")
            assert (t["file_offset"], t["bytes"], t["type"], t["dims"]) == (64, 32, 0, [8])
    else:
        with pytest.raises(lib.LlmError) as e:
            lib.GgufFile(path)
        assert str(e.value).endswith(": " + reason)


@pytest.mark.parametrize("alignment", [None, 64])
def test_example5_layout(lib, tmp_path, alignment):
    data = _example5_file(alignment)
    ref = G.read(data)
    with lib.GgufFile(_save(tmp_path, "f.gguf", data)) as g:
        s = g.summary()
        assert (s["version"], s["n_tensors"], s["n_kv"], s["alignment"], s["infos_end"], s["data_start"],
                s["file_size"]) == (3, 2, ref["n_kv"], ref["alignment"], ref["infos_end"], ref["data_start"], len(data))
        got = g.tensors()
        assert [n for n, _ in got] == [t["name"] for t in ref["tensors"]]
        for (n, t), r in zip(got, ref["tensors"]):
            assert (t["type"], t["dims"], t["offset"], t["file_offset"], t["bytes"]) == \
                (r["type"], r["dims"], r["offset"], r["file_offset"], r["bytes"])


def test_all_value_types(lib, tmp_path):
    md = [("u8", W.UINT8, 200), ("i8", W.INT8, -100), ("u16", W.UINT16, 60000), ("i16", W.INT16, -30000),
          ("u32", W.UINT32, 4000000000), ("i32", W.INT32, -2000000000), ("f32", W.FLOAT32, 1.5),
          ("b", W.BOOL, 1), ("s", W.STRING, "世界 ok"), ("a", W.ARRAY, (W.STRING, ["<s>", "Ġworld", "Ċ"])),
          ("ai", W.ARRAY, (W.INT32, [3, 1, 1, 1])), ("u64", W.UINT64, 2 ** 40 + 7), ("i64", W.INT64, -(2 ** 50)),
          ("f64", W.FLOAT64, 0.1), ("nested", W.ARRAY, (W.ARRAY, [(W.UINT8, [1, 2]), (W.STRING, ["x"])]))]
    data = W.write(md, [("t", G.F32, [4], np.arange(4, dtype=np.float32).tobytes())])
    ref = G.read(data)["metadata"]
    with lib.GgufFile(_save(tmp_path, "f.gguf", data)) as g:
        assert g.keys() == [(k, t) for k, t, _ in md]
        for k, t, v in md:
            if t in (W.FLOAT32, W.FLOAT64):
                assert g.meta_float(k) == ref[k][1]
            elif t == W.STRING:
                assert g.meta_string(k) == v
            elif t == W.ARRAY:
                assert g.meta_type(k) == (W.ARRAY, v[0], len(v[1]))
            else:
                assert g.meta_int(k) == int(v)
        with pytest.raises(lib.LlmError):
            g.meta_int("s")                      # a string is not an integer
        with pytest.raises(lib.LlmError):
            g.meta_int("missing")


SMALL = [
    synth.ModelConfig("g-f32", n_layers=2, dim=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96, vocab=50,
                      max_seq=64, eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=synth.F32, tied=False, number=81),
    synth.ModelConfig("g-f16", n_layers=2, dim=64, n_heads=4, n_kv_heads=4, head_dim=16, ffn_dim=96, vocab=50,
                      max_seq=64, eps=1e-6, rope_base=1e6, rope_neox=1, wtype=synth.F16, tied=True, bias=True,
                      number=82),
    synth.ModelConfig("g-q8", n_layers=3, dim=64, n_heads=8, n_kv_heads=2, head_dim=8, ffn_dim=128, vocab=70,
                      max_seq=64, eps=1e-5, rope_base=500000.0, rope_neox=0, wtype=synth.Q8_0, tied=True,
                      rope_freqs=True, number=83),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c.name for c in SMALL])
@pytest.mark.parametrize("alignment", [None, 64])
def test_synthetic_models_match_the_oracle(lib, tmp_path, cfg, alignment):
    Wt = synth.make_weights(cfg)
    data = W.model_file(cfg, Wt, alignment=alignment)
    ref = G.read(data)
    rc = G.model_config(ref["metadata"])
    with lib.GgufFile(_save(tmp_path, "m.gguf", data)) as g:
        s = g.summary()
        assert (s["n_tensors"], s["n_kv"], s["data_start"]) == (ref["n_tensors"], ref["n_kv"], ref["data_start"])
        for (n, t), r in zip(g.tensors(), ref["tensors"]):
            assert n == r["name"] and (t["type"], t["dims"], t["file_offset"], t["bytes"]) == \
                (r["type"], r["dims"], r["file_offset"], r["bytes"])
        c = g.config()
        assert (c.n_layers, c.dim, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn_dim, c.vocab, c.max_seq,
                c.rope_dims, c.rope_neox, c.wtype) == \
            (rc["layers"], rc["dim"], rc["heads"], rc["kv_heads"], rc["head_dim"], rc["ffn"], rc["vocab"],
             rc["context_length"], rc["rope_dims"], int(rc["neox"]), cfg.wtype)
        assert c.eps == np.float32(rc["eps"]) and c.rope_base == np.float32(rc["rope_base"])
        # and the shape is the synthetic model's own
        assert (c.n_layers, c.dim, c.n_heads, c.n_kv_heads, c.ffn_dim, c.vocab, c.rope_neox) == \
            (cfg.n_layers, cfg.dim, cfg.n_heads, cfg.n_kv_heads, cfg.ffn_dim, cfg.vocab, cfg.rope_neox)
        assert g.config(max_seq=17).max_seq == 17


def test_vocab_from_token_list_and_defaults(lib, tmp_path):
    cfg = SMALL[0]
    Wt = synth.make_weights(cfg)
    data = W.model_file(cfg, Wt, vocab_key=False,
                        extra_metadata=[("tokenizer.ggml.tokens", W.ARRAY, (W.STRING, [f"t{i}" for i in range(50)]))])
    with lib.GgufFile(_save(tmp_path, "m.gguf", data)) as g:
        assert g.config().vocab == 50 == G.model_config(G.read(data)["metadata"])["vocab"]


def test_rejected_models(lib, tmp_path):
    cfg = SMALL[2]
    Wt = synth.make_weights(cfg)
    # another architecture
    data = W.model_file(cfg, Wt, arch="gpt2")
    with lib.GgufFile(_save(tmp_path, "a.gguf", data)) as g:
        with pytest.raises(lib.LlmError) as e:
            g.config()
        assert e.value.status == lib.LLM_ERR_UNSUPPORTED and "gpt2" in str(e.value)
        with pytest.raises(lib.LlmError):
            lib.llm_create_from_gguf(g)
    # a Q8_0 row that is not whole blocks, and a tensor type this reader does not handle
    bad = W.write([], [("q", G.Q8_0, [40], bytes(34 * 2))])
    with pytest.raises(lib.LlmError) as e:
        lib.GgufFile(_save(tmp_path, "b.gguf", bad))
    assert "32-value blocks" in str(e.value)
    with pytest.raises(lib.LlmError) as e:
        lib.GgufFile(_save(tmp_path, "c.gguf", W.write([], [("k", 12, [256], bytes(210))])))
    assert e.value.status == lib.LLM_ERR_UNSUPPORTED
    # a matrix of another type than the embedding: rejected before any device work
    Wf = synth.make_weights(SMALL[0])
    data = bytearray(W.model_file(SMALL[0], Wf))
    g0 = G.read(bytes(data))
    info = next(t for t in g0["tensors"] if t["name"] == "blk.1.ffn_up.weight")
    md = [(k, t, v) for k, (t, v) in g0["metadata"].items()]
    tens = []
    for t in g0["tensors"]:
        raw = bytes(data[t["file_offset"]:t["file_offset"] + t["bytes"]])
        if t["name"] == "blk.1.ffn_up.weight":
            tens.append((t["name"], G.F16, t["dims"], bytes(t["bytes"] // 2)))
        else:
            tens.append((t["name"], t["type"], t["dims"], raw))
    with lib.GgufFile(_save(tmp_path, "e.gguf", W.write(md, tens))) as g:
        with pytest.raises(lib.LlmError) as e:
            lib.llm_create_from_gguf(g)
        assert e.value.status == lib.LLM_ERR_UNSUPPORTED and "blk.1.ffn_up.weight" in str(e.value)
    # a missing layer tensor
    tens2 = [x for x in tens if x[0] != "blk.0.attn_k.weight"]
    with lib.GgufFile(_save(tmp_path, "f.gguf", W.write(md, tens2))) as g:
        with pytest.raises(lib.LlmError) as e:
            lib.llm_create_from_gguf(g)
        assert "blk.0.attn_k.weight" in str(e.value)
    assert info["bytes"] > 0


def test_unsupported_shape_is_rejected_before_staging(lib, tmp_path):
    # a well-formed file whose shape the kernels cannot run (head_dim 320):
    # rejected with llm_create's reason before any tensor reaches the device,
    # so the same answer comes back on a machine without a GPU
    cfg = synth.ModelConfig("g-hd320", n_layers=1, dim=1280, n_heads=4, n_kv_heads=4, head_dim=320, ffn_dim=64,
                            vocab=40, max_seq=16, eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=synth.F32,
                            tied=True, number=84)
    data = W.model_file(cfg, synth.make_weights(cfg))
    with lib.GgufFile(_save(tmp_path, "m.gguf", data)) as g:
        assert g.config().head_dim == 320
        with pytest.raises(lib.LlmError) as e:
            lib.llm_create_from_gguf(g)
    assert e.value.status == lib.LLM_ERR_UNSUPPORTED
    assert "head_dim must be a multiple of 8, <= 256" in str(e.value)


def test_block_count_beyond_the_tensors_is_refused(lib, tmp_path):
    # a 2-block model whose metadata claims a million blocks: refused from the
    # tensor count, before any per-block work
    cfg = SMALL[0]
    data = W.model_file(cfg, synth.make_weights(cfg))
    g0 = G.read(data)
    md = [(k, t, 1_000_000 if k == "llama.block_count" else v) for k, (t, v) in g0["metadata"].items()]
    tens = [(t["name"], t["type"], t["dims"], data[t["file_offset"]:t["file_offset"] + t["bytes"]])
            for t in g0["tensors"]]
    with lib.GgufFile(_save(tmp_path, "m.gguf", W.write(md, tens))) as g:
        assert g.config().n_layers == 1_000_000
        with pytest.raises(lib.LlmError) as e:
            lib.llm_create_from_gguf(g)
    assert e.value.status == lib.LLM_ERR_INVALID_ARG and "block_count 1000000" in str(e.value)


def test_truncations_are_rejected_not_read(lib, tmp_path):
    # every prefix of a valid file is either rejected with a reason or (only
    # the whole file) accepted: no read past the end
    cfg = SMALL[1]
    data = W.model_file(cfg, synth.make_weights(cfg))
    cuts = sorted(set([0, 1, 23, 24, 25, 40, 100] + list(range(0, G.read(data)["data_start"] + 64, 37)) +
                      [len(data) - 1]))
    for n in cuts:
        with pytest.raises(lib.LlmError):
            lib.GgufFile(_save(tmp_path, "t.gguf", data[:n]))
    with lib.GgufFile(_save(tmp_path, "t.gguf", data)) as g:
        assert g.summary()["file_size"] == len(data)


def test_open_errors(lib, tmp_path):
    # a missing path and a directory are rejected with a reason, not mapped
    for path, words in ((tmp_path / "absent.gguf", "cannot open"), (tmp_path, "not a regular file")):
        with pytest.raises(lib.LlmError) as e:
            lib.GgufFile(str(path))
        assert e.value.status == lib.LLM_ERR_INVALID_ARG and words in str(e.value)
