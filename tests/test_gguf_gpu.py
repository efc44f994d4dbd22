"""A model loaded from a GGUF file (llm_create_from_gguf) against the same
weights handed to llm_create directly (bitwise: the same kernel on the same
bytes) and against the CPU oracle (within the logits tolerance)."""
import numpy as np
import pytest

import oracle
import synth
from gguf_writer import model_file
from harness import check_logits
from test_decode_gpu import SMALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import llama_decode_forward_gb300 as L
    return L


@pytest.mark.parametrize("name", ["f32", "f16_neox_bias_tied", "q8_0_tied_freqs"])
def test_model_from_gguf(lib, tmp_path, name):
    cfg = SMALL[name]
    W = synth.make_weights(cfg)
    path = tmp_path / "m.gguf"
    path.write_bytes(model_file(cfg, W, alignment=64))
    g = lib.GgufDecoder(str(path), max_seq=cfg.max_seq)
    d = lib.Decoder(cfg, W)
    ora = oracle.OracleModel(cfg, W)
    assert (g.cfg.n_layers, g.cfg.dim, g.cfg.vocab, g.cfg.wtype, g.cfg.rope_neox) == \
        (cfg.n_layers, cfg.dim, cfg.vocab, cfg.wtype, cfg.rope_neox)
    a = np.empty(cfg.vocab, np.float32)
    b = np.empty(cfg.vocab, np.float32)
    for pos, t in enumerate(synth.prompt(cfg, 6)):
        ref = ora.forward(int(t), pos)
        ia = lib.llm_decode_step(g.h, int(t), pos, a)
        ib = lib.llm_decode_step(d.h, int(t), pos, b)
        np.testing.assert_array_equal(a, b)
        assert ia == ib
        check_logits(a, ref, cfg.wtype, f"{name} from GGUF, pos {pos}")
    g.close()
    d.close()
