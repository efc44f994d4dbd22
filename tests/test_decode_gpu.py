"""Parity of the CUDA decode step (through the C ABI) with the CPU oracle."""
import numpy as np
import pytest

import oracle
import synth
from harness import TOL, check_logits, gpu_kv, margin, prefill_kv_both

pytestmark = pytest.mark.gpu


def small(wtype, **kw):
    """Small shapes spanning several CTAs per phase, with ragged row counts."""
    base = dict(n_layers=2, dim=256, n_heads=8, n_kv_heads=2, head_dim=32, ffn_dim=544, vocab=1000, max_seq=160,
                eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=wtype, tied=False, number=40 + wtype)
    base.update(kw)
    return synth.ModelConfig("small", **base)


SMALL = {
    "f32": small(synth.F32),
    "f16_neox_bias_tied": small(synth.F16, rope_neox=1, bias=True, tied=True, rope_base=1e6),
    "q8_0_tied_freqs": small(synth.Q8_0, tied=True, rope_freqs=True, rope_base=500000.0),
    "q8_0_mha_hd48": small(synth.Q8_0, dim=288, n_heads=6, n_kv_heads=6, head_dim=48, ffn_dim=768, vocab=777),
    "f32_hd128_gq4": small(synth.F32, dim=512, n_heads=4, n_kv_heads=1, head_dim=128, ffn_dim=320, vocab=513),
}


@pytest.fixture(scope="module")
def lib():
    import llama_decode_forward_gb300 as L
    return L


def make_pair(lib, cfg):
    W = synth.make_weights(cfg)
    ora = oracle.OracleModel(cfg, W)
    dec = lib.Decoder(cfg, W)
    return W, ora, dec


# ------------------------------------------------------------ bit-exact --
@pytest.mark.parametrize("name", ["f32", "f16_neox_bias_tied", "q8_0_tied_freqs"])
def test_weight_decode_bit_exact(lib, name):
    import torch
    cfg = SMALL[name]
    W, ora, dec = make_pair(lib, cfg)
    d, q, kv, f = cfg.dim, cfg.q_dim, cfg.kv_dim, cfg.ffn_dim
    tensors = [("wq", q, d), ("wk", kv, d), ("wv", kv, d), ("wo", d, q), ("w_gate", f, d), ("w_up", f, d),
               ("w_down", d, f)]
    for layer in range(cfg.n_layers):
        for which, (name_t, rows, cols) in enumerate(tensors):
            for r0 in (0, rows // 2, rows - 3):
                out = torch.empty(3 * cols, dtype=torch.float32, device="cuda")
                lib.llm_test_dequant_rows(dec.h, which, layer, r0, 3, out)
                got = out.cpu().numpy().reshape(3, cols)
                for k in range(3):
                    ref = oracle.dequant_row(W.layers[layer][name_t], cfg.wtype, r0 + k, cols)
                    assert np.array_equal(got[k].view(np.uint32), ref.view(np.uint32)), (name_t, r0 + k)
    for which, arr in ((7, W.tok_embd), (8, W.output if W.output is not None else W.tok_embd)):
        for r0 in (0, 517, cfg.vocab - 2):
            out = torch.empty(2 * d, dtype=torch.float32, device="cuda")
            lib.llm_test_dequant_rows(dec.h, which, 0, r0, 2, out)
            got = out.cpu().numpy().reshape(2, d)
            for k in range(2):
                assert np.array_equal(got[k].view(np.uint32), oracle.dequant_row(arr, cfg.wtype, r0 + k, d).view(np.uint32))


def test_q8_0_decode_edge_scales_bit_exact(lib):
    """Scales 0, FP16 subnormals, the largest FP16, and quants -128/127."""
    import torch
    cfg = small(synth.Q8_0, n_layers=1)
    W = synth.make_weights(cfg)
    blocks = W.layers[0]["wq"].reshape(-1, 34)
    for i, s in enumerate((0x0000, 0x0001, 0x03ff, 0x0400, 0x7bff, 0x8001, 0xfbff, 0x3c00)):
        blocks[i, 0], blocks[i, 1] = s & 0xff, s >> 8
        blocks[i, 2 + i] = 0x80
        blocks[i, 3 + i] = 0x7f
    dec = lib.Decoder(cfg, W)
    out = torch.empty(cfg.dim, dtype=torch.float32, device="cuda")
    lib.llm_test_dequant_rows(dec.h, 0, 0, 0, 1, out)
    ref = oracle.dequant_row(W.layers[0]["wq"], synth.Q8_0, 0, cfg.dim)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_kv_store_bit_exact_layout(lib):
    """F16 round-to-nearest-even and the [pos][kv_head][i] index map."""
    import torch
    cfg = small(synth.F32, n_layers=2)
    W = synth.make_weights(cfg)
    dec = lib.Decoder(cfg, W)
    rng = np.random.default_rng(11)
    kv = cfg.kv_dim
    h = rng.integers(0, 0x7bff, kv).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    specials = np.array([65504, 65520, 70000, -1e-7, 2 ** -25, 3 * 2 ** -26, 1e-6, 0.0], np.float32)
    k = ((lo + hi) / 2).astype(np.float32)                            # exact ties
    k[:specials.size] = specials
    v = (rng.standard_normal(kv) * np.exp(rng.uniform(-12, 10, kv))).astype(np.float32)
    for layer, pos in ((0, 0), (1, 37), (1, cfg.max_seq - 1)):
        lib.llm_test_kv_store(dec.h, layer, pos, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
        for which, src in ((0, k), (1, v)):
            got = gpu_kv(dec, layer, which, pos)
            assert np.array_equal(got, oracle.f32_to_f16(src)), (layer, pos, which)
        kk, _ = dec.kv_tensors(layer)
        flat = kk.view(-1).cpu().numpy().view(np.uint16)
        assert np.array_equal(flat[pos * kv:(pos + 1) * kv], oracle.f32_to_f16(k))


# ------------------------------------------------------------ one step --
@pytest.mark.parametrize("name", sorted(SMALL))
def test_decode_steps_match_oracle(lib, name):
    """Teacher-forced steps at positions that cross the attention split and
    chunk boundaries, after pre-filling the cache with seeded rows."""
    cfg = SMALL[name]
    W, ora, dec = make_pair(lib, cfg)
    prefill_kv_both(cfg, ora, dec, cfg.max_seq - 1)
    toks = synth.prompt(cfg, 12)
    logits = np.empty(cfg.vocab, np.float32)
    for i, pos in enumerate((0, 1, 15, 16, 17, 63, 64, 65, 100, 129, cfg.max_seq - 1)):
        tok = int(toks[i])
        ref = ora.forward(tok, pos)
        am = lib.llm_decode_step(dec.h, tok, pos, logits)
        check_logits(logits, ref, cfg.wtype, f"{name} pos {pos}")
        if am != oracle.argmax(ref):
            assert margin(ref) < TOL[cfg.wtype]
        assert am == int(np.argmax(logits)) or logits[am] == logits.max()
        # the row written at pos agrees with the oracle's stored row
        for l in range(cfg.n_layers):
            for which in (0, 1):
                g = gpu_kv(dec, l, which, pos).view(np.float16).astype(np.float32)
                r = ora.kv(l, which)[pos]
                assert np.max(np.abs(g - r)) <= TOL[cfg.wtype] * max(1.0, float(np.max(np.abs(r)))), (l, which)


def test_decode_step_edge_tokens_and_errors(lib):
    cfg = SMALL["q8_0_tied_freqs"]
    W, ora, dec = make_pair(lib, cfg)
    logits = np.empty(cfg.vocab, np.float32)
    for pos, tok in ((0, 0), (1, cfg.vocab - 1)):
        ref = ora.forward(tok, pos)
        lib.llm_decode_step(dec.h, tok, pos, logits)
        check_logits(logits, ref, cfg.wtype)
    for tok, pos in ((cfg.vocab, 2), (-1, 2), (3, cfg.max_seq), (3, -1)):
        with pytest.raises(lib.LlmError) as e:
            lib.llm_decode_step(dec.h, tok, pos)
        assert e.value.status == lib.LLM_ERR_OUT_OF_RANGE
    # the handle's shape; host buffers that cannot take vocab floats are refused before the call
    c = lib.llm_get_config(dec.h)
    assert (c.n_layers, c.dim, c.vocab, c.max_seq, c.wtype) == (cfg.n_layers, cfg.dim, cfg.vocab, cfg.max_seq,
                                                               cfg.wtype)
    with pytest.raises(ValueError):
        lib.llm_decode_step(dec.h, 3, 2, np.empty(cfg.vocab - 1, np.float32))
    with pytest.raises(TypeError):
        lib.llm_decode_step(dec.h, 3, 2, np.empty(cfg.vocab, np.float64))


def test_device_side_bad_token_is_reported(lib):
    import torch
    cfg = SMALL["f32"]
    W, ora, dec = make_pair(lib, cfg)
    tok = torch.tensor([cfg.vocab + 5], dtype=torch.int32, device="cuda")
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.llm_decode_step_async(dec.h, tok, 0, out)
    with pytest.raises(lib.LlmError) as e:
        lib.llm_sync(dec.h)
    assert e.value.status == lib.LLM_ERR_OUT_OF_RANGE
    with pytest.raises(lib.LlmError) as e:
        lib.llm_decode_step(dec.h, 1, 0)
    assert e.value.status == lib.LLM_ERR_STATE
    lib.llm_reset(dec.h)
    logits = np.empty(cfg.vocab, np.float32)
    lib.llm_decode_step(dec.h, 1, 0, logits)
    check_logits(logits, ora.forward(1, 0), cfg.wtype)


def test_repeated_step_is_deterministic(lib):
    """Same inputs twice: identical logits bits (no float atomics in reductions)."""
    cfg = SMALL["q8_0_tied_freqs"]
    W, ora, dec = make_pair(lib, cfg)
    prefill_kv_both(cfg, ora, dec, 90)
    a = np.empty(cfg.vocab, np.float32)
    b = np.empty(cfg.vocab, np.float32)
    lib.llm_decode_step(dec.h, 7, 90, a)
    lib.llm_decode_step(dec.h, 7, 90, b)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
