"""Layer-by-layer parity ("The Forward Pass in Java", Example 11: every named
intermediate checked, not only the final logits): the decode step's
intermediates read back with llm_debug_tensor against the oracle's trace of
the same step.

q and k are read before RoPE and rotated here by the oracle's RoPE before
the comparison with the oracle's Qcur / Kcur; v, attn_out, ffn_swiglu and
ffn_out are compared as they are.  Bound: max |gpu - oracle| <= 1e-3 of the
tensor's largest magnitude (at least 1), and the tensor sums (what
llama-eval-callback prints) within 1e-3 of the sum of magnitudes: far inside
the logits' acceptance tolerance, loose enough for float summation order and
the Q8_0 products' 24-bit activations."""
import numpy as np
import pytest

import oracle
import synth
from harness import prefill_kv_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import llama_decode_forward_gb300 as L
    return L


def small(wtype, **kw):
    base = dict(n_layers=3, dim=256, n_heads=8, n_kv_heads=2, head_dim=32, ffn_dim=544, vocab=1000, max_seq=160,
                eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=wtype, tied=False, number=100 + wtype)
    base.update(kw)
    return synth.ModelConfig("small_trace", **base)


MODELS = {
    "q8_0": small(synth.Q8_0, rope_freqs=True, rope_base=500000.0),
    "f16_neox_bias": small(synth.F16, rope_neox=1, bias=True),
    "f32_hd128": small(synth.F32, dim=512, n_heads=4, n_kv_heads=1, head_dim=128, ffn_dim=320, vocab=513),
}


def close(got, ref, what):
    got, ref = got.astype(np.float64), ref.astype(np.float64)
    scale = max(1.0, float(np.max(np.abs(ref))))
    d = float(np.max(np.abs(got - ref)))
    assert d <= 1e-3 * scale, f"{what}: max diff {d:.3g} (scale {scale:.3g})"
    assert abs(got.sum() - ref.sum()) <= 1e-3 * max(1.0, float(np.abs(ref).sum())), f"{what}: sums"


@pytest.mark.parametrize("name", sorted(MODELS))
def test_every_intermediate_matches_the_oracle_trace(lib, name):
    cfg = MODELS[name]
    W = synth.make_weights(cfg)
    ora = oracle.OracleModel(cfg, W)
    dec = lib.Decoder(cfg, W)
    with pytest.raises(lib.LlmError) as e:
        lib.llm_debug_tensor(dec.h, 0, lib.LLM_DEBUG_V)
    assert e.value.status == lib.LLM_ERR_STATE                # no step yet
    prefill_kv_both(cfg, ora, dec, cfg.max_seq - 1)
    trace = {}
    ora.set_trace(lambda nm, layer, v: trace.__setitem__((nm, layer), v))
    freqs = W.rope_freqs
    for pos, tok in ((0, 5), (17, 9), (cfg.max_seq - 1, 11)):
        trace.clear()
        ref_logits = ora.forward(tok, pos)
        logits = np.empty(cfg.vocab, np.float32)
        lib.llm_decode_step(dec.h, tok, pos, logits)
        assert np.max(np.abs(logits - ref_logits)) <= 2e-2
        for l in range(cfg.n_layers):
            q = lib.llm_debug_tensor(dec.h, l, lib.LLM_DEBUG_Q)
            k = lib.llm_debug_tensor(dec.h, l, lib.LLM_DEBUG_K)
            q = oracle.rope(q, cfg.n_heads, cfg.head_dim, cfg.rope_dims, pos, cfg.rope_base, cfg.rope_neox, freqs)
            k = oracle.rope(k, cfg.n_kv_heads, cfg.head_dim, cfg.rope_dims, pos, cfg.rope_base, cfg.rope_neox,
                            freqs)
            close(q, trace[("Qcur", l)], f"{name} pos {pos} layer {l} Qcur")
            close(k, trace[("Kcur", l)], f"{name} pos {pos} layer {l} Kcur")
            for which, nm in ((lib.LLM_DEBUG_V, "Vcur"), (lib.LLM_DEBUG_ATTN_OUT, "attn_out"),
                              (lib.LLM_DEBUG_FFN_SWIGLU, "ffn_swiglu"), (lib.LLM_DEBUG_FFN_OUT, "ffn_out")):
                close(lib.llm_debug_tensor(dec.h, l, which), trace[(nm, l)], f"{name} pos {pos} layer {l} {nm}")
    ora.set_trace(None)
    lib.llm_reset(dec.h)
    with pytest.raises(lib.LlmError) as e:
        lib.llm_debug_tensor(dec.h, 0, lib.LLM_DEBUG_FFN_OUT)
    assert e.value.status == lib.LLM_ERR_STATE                # cleared by the reset
    with pytest.raises(lib.LlmError) as e:
        lib.llm_debug_tensor(dec.h, cfg.n_layers, lib.LLM_DEBUG_V)
    assert e.value.status == lib.LLM_ERR_OUT_OF_RANGE
    dec.close()
