"""Non-unit RoPE frequency factors ("What a Llama model computes, and why"
§2.4: pair i turns by p * base^(-2i/d) / f_i; §6: Llama 3's factors leave the
fast pairs alone and divide the slow ones by up to 8) on the decode step and
the batched prefill, against the oracle, which applies the same divisors
after its float angle chain (pinned in test_oracle_pins)."""
import numpy as np
import pytest

import oracle
import synth
from harness import TOL, check_logits, margin, prefill_kv_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import llama_decode_forward_gb300 as L
    return L


def llama3_style(n_pairs: int) -> np.ndarray:
    """1 for the fastest quarter of the pairs, a ramp 1.5 .. 4 over the next
    quarter, 8 for the slowest half."""
    q = n_pairs // 4
    f = np.concatenate([np.ones(q), np.linspace(1.5, 4.0, q), np.full(n_pairs - 2 * q, 8.0)])
    return f.astype(np.float32)


def cfg_of(wtype, neox, **kw):
    base = dict(n_layers=2, dim=256, n_heads=8, n_kv_heads=2, head_dim=32, ffn_dim=512, vocab=1000, max_seq=420,
                eps=1e-5, rope_base=500000.0, rope_neox=neox, wtype=wtype, tied=True, rope_freqs=True,
                number=120 + neox + 2 * wtype)
    base.update(kw)
    return synth.ModelConfig("rope_freqs", **base)


def with_factors(cfg):
    W = synth.make_weights(cfg)
    W.rope_freqs = llama3_style(cfg.rope_dims // 2)
    return W


@pytest.mark.parametrize("wtype,neox", [(synth.Q8_0, 0), (synth.Q8_0, 1), (synth.F16, 0)])
def test_decode_with_factors_matches_oracle(lib, wtype, neox):
    cfg = cfg_of(wtype, neox)
    W = with_factors(cfg)
    ora = oracle.OracleModel(cfg, W)
    dec = lib.Decoder(cfg, W)
    prefill_kv_both(cfg, ora, dec, 300)             # angles up to ~300 radians on the fast pairs
    logits = np.empty(cfg.vocab, np.float32)
    tok = int(synth.prompt(cfg, 1)[0])
    for pos in (300, 301, 302):
        ref = ora.forward(tok, pos)
        am = lib.llm_decode_step(dec.h, tok, pos, logits)
        check_logits(logits, ref, cfg.wtype, f"pos {pos}")
        if am != oracle.argmax(ref):
            assert margin(ref) < TOL[cfg.wtype]
        tok = oracle.argmax(ref)
    # the K rows the step wrote: within tolerance of the oracle's
    for l in range(cfg.n_layers):
        k, _ = dec.kv_tensors(l)
        g = k[300:303].cpu().numpy().view(np.float16).astype(np.float64)
        r = ora.kv(l, 0)[300:303].astype(np.float64)
        assert np.max(np.abs(g - r)) <= TOL[cfg.wtype]
    dec.close()


def test_factors_change_the_result(lib):
    """The divisors reach the kernel: unit and Llama 3-style factors give
    different K rows at a large position, and each matches its oracle."""
    cfg = cfg_of(synth.Q8_0, 0)
    W1 = synth.make_weights(cfg)                     # unit factors
    W8 = with_factors(cfg)
    rows = []
    for W in (W1, W8):
        dec = lib.Decoder(cfg, W)
        ora = oracle.OracleModel(cfg, W)
        prefill_kv_both(cfg, ora, dec, 400)
        logits = np.empty(cfg.vocab, np.float32)
        tok = int(synth.prompt(cfg, 1)[0])
        ref = ora.forward(tok, 400)
        lib.llm_decode_step(dec.h, tok, 400, logits)
        check_logits(logits, ref, cfg.wtype, "pos 400")
        k, _ = dec.kv_tensors(0)
        rows.append(k[400].cpu().numpy().view(np.float16).astype(np.float64))
        dec.close()
    assert np.max(np.abs(rows[0] - rows[1])) > 0.1


@pytest.mark.parametrize("wtype", [synth.F16, synth.Q8_0])
def test_prefill_with_factors_matches_oracle(lib, wtype):
    cfg = cfg_of(wtype, 1 if wtype == synth.F16 else 0, bias=wtype == synth.F16, number=130 + wtype)
    W = with_factors(cfg)
    ora = oracle.OracleModel(cfg, W)
    dec = lib.Decoder(cfg, W)
    toks = synth.prompt(cfg, 260)
    with oracle.threads():
        ref = ora.prefill(toks, 0)
    got = np.empty(cfg.vocab, np.float32)
    am = lib.llm_prefill(dec.h, toks, 0, got)
    check_logits(got, ref, cfg.wtype, "prefill 0..259")
    if am != oracle.argmax(ref):
        assert margin(ref) < TOL[cfg.wtype]
    for l in range(cfg.n_layers):
        for which in (0, 1):
            k, v = dec.kv_tensors(l)
            g = (k if which == 0 else v)[:260].cpu().numpy().view(np.float16).astype(np.float64)
            r = ora.kv(l, which)[:260].astype(np.float64)
            assert np.max(np.abs(g - r)) <= TOL[cfg.wtype], (l, which)
    dec.close()
