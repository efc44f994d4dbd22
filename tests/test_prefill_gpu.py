"""Batched prefill (F16 and Q8_0 weights, tensor-core GEMMs) against the
oracle and against the decode step run token by token ("What a Llama model
computes, and why" §4: prefill equals token-by-token).  The GEMM operands are
rounded to F16 (the reading of the prefill precision; a Q8_0 weight becomes
d * q rounded to F16), so the comparison is within the F16/Q8_0 logit
tolerance; the K/V rows it writes are compared element-wise within the same
tolerance."""
import numpy as np
import pytest

import oracle
import synth
from harness import TOL, check_logits, margin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import llama_decode_forward_gb300 as L
    return L


def f16cfg(**kw):
    base = dict(n_layers=2, dim=256, n_heads=8, n_kv_heads=2, head_dim=32, ffn_dim=576, vocab=1000, max_seq=300,
                eps=1e-5, rope_base=1e6, rope_neox=1, wtype=synth.F16, tied=True, bias=True, number=71)
    base.update(kw)
    return synth.ModelConfig("prefill_small", **base)


def kv_as_float(dec, layer, which, rows):
    k, v = dec.kv_tensors(layer)
    t = (k if which == 0 else v)[rows]
    return t.cpu().numpy().view(np.float16).astype(np.float64)


@pytest.mark.parametrize("kw", [{}, dict(rope_neox=0, bias=False, tied=False, number=72),
                                dict(wtype=synth.Q8_0, rope_neox=0, bias=False, number=73),
                                dict(wtype=synth.Q8_0, tied=False, rope_freqs=True, number=74)])
def test_prefill_matches_oracle_and_continues(lib, kw):
    cfg = f16cfg(**kw)
    W = synth.make_weights(cfg)
    ora = oracle.OracleModel(cfg, W)
    dec = lib.Decoder(cfg, W)
    toks = synth.prompt(cfg, 237)
    # 200 tokens from position 0: two 128-row GEMM tiles, the second ragged
    ref = ora.prefill(toks[:200], 0)
    got = np.empty(cfg.vocab, np.float32)
    am = lib.llm_prefill(dec.h, toks[:200], 0, got)
    check_logits(got, ref, cfg.wtype, "prefill 0..199")
    if am != oracle.argmax(ref):
        assert margin(ref) < TOL[cfg.wtype]
    for l in range(cfg.n_layers):
        for which in (0, 1):
            g = kv_as_float(dec, l, which, slice(0, 200))
            r = ora.kv(l, which)[:200].astype(np.float64)
            assert np.max(np.abs(g - r)) <= TOL[cfg.wtype], (l, which)
    # continuing the sequence: 37 more tokens attend to the 200 cached rows
    ref = ora.prefill(toks[200:], 200)
    am = lib.llm_prefill(dec.h, toks[200:], 200, got)
    check_logits(got, ref, cfg.wtype, "prefill 200..236")
    # and a decode step after the batched prefill
    nxt = oracle.argmax(ref)
    ref = ora.forward(nxt, 237)
    lib.llm_decode_step(dec.h, nxt, 237, got)
    check_logits(got, ref, cfg.wtype, "decode after prefill")
    dec.close()


@pytest.mark.parametrize("base", [synth.QWEN2_F16, synth.LLAMA1B_Q8], ids=["qwen2-1b-f16", "llama-3.2-1b-q8_0"])
def test_prefill_512_full_width_equals_token_by_token(lib, base):
    """The 1B-shaped models (Qwen2-style F16: NEOX, biases, tied; Llama 3.2
    Q8_0: normal pairs, frequency factors, tied): a 512-token batched prefill
    against 512 decode steps of the library's decode path."""
    cfg = base.scaled(max_seq=600)
    W = synth.make_weights(cfg)
    toks = synth.prompt(cfg, 512)
    a = lib.Decoder(cfg, W)
    b = lib.Decoder(cfg, W)
    la = np.empty(cfg.vocab, np.float32)
    lb = np.empty(cfg.vocab, np.float32)
    am_a = lib.llm_prefill(a.h, toks, 0, la)
    for p, t in enumerate(toks):
        am_b = lib.llm_decode_step(b.h, int(t), p, lb if p == len(toks) - 1 else None)
    check_logits(la, lb, cfg.wtype, "prefill vs token-by-token")
    if am_a != am_b:
        assert margin(lb) < TOL[cfg.wtype]
    for l in (0, cfg.n_layers - 1):
        for which in (0, 1):
            ga = kv_as_float(a, l, which, slice(0, 512))
            gb = kv_as_float(b, l, which, slice(0, 512))
            assert np.max(np.abs(ga - gb)) <= TOL[cfg.wtype], (l, which)
    a.close()
    b.close()
