"""llm_prefill_f16_copy: a Q8_0 handle's batched prefill reading an F16 copy
of its layer matrices instead of expanding the quants inside each GEMM.
Both hold d * q rounded to nearest even ("What a Llama model computes, and
why" §4, the prefill's F16 operands), so the prefill's logits and the K/V
rows it writes must agree bit for bit with and without the copy; the decode
step does not read the copy."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import llama_decode_forward_gb300 as L
    return L


def q8cfg(**kw):
    base = dict(n_layers=2, dim=256, n_heads=8, n_kv_heads=2, head_dim=32, ffn_dim=576, vocab=1000, max_seq=300,
                eps=1e-5, rope_base=500000.0, rope_neox=0, wtype=synth.Q8_0, tied=False, rope_freqs=True, number=75)
    base.update(kw)
    return synth.ModelConfig("prefill_copy", **base)


def kv_bits(dec, n_layers, rows):
    out = []
    for l in range(n_layers):
        k, v = dec.kv_tensors(l)
        out.append(k[rows].cpu().numpy().copy())
        out.append(v[rows].cpu().numpy().copy())
    return out


def run(lib, dec, cfg, toks, cuts):
    """Prefill toks in the pieces given by cuts, then one decode step: every
    logits vector as bits, and the K/V rows written."""
    got, out = np.empty(cfg.vocab, np.float32), []
    for a, b in zip(cuts[:-1], cuts[1:]):
        lib.llm_prefill(dec.h, toks[a:b], a, got)
        out.append(got.view(np.uint32).copy())
    lib.llm_decode_step(dec.h, 7, cuts[-1], got)
    out.append(got.view(np.uint32).copy())
    return out, kv_bits(dec, cfg.n_layers, slice(0, cuts[-1] + 1))


def test_copy_gives_the_same_bits(lib):
    cfg = q8cfg()
    W = synth.make_weights(cfg)
    toks = synth.prompt(cfg, 237)
    cuts = [0, 200, 237]                       # two 128-row tiles (the second ragged), then a continuation
    a = lib.Decoder(cfg, W)
    b = lib.Decoder(cfg, W)
    lib.llm_prefill_f16_copy(b.h)
    lib.llm_prefill_f16_copy(b.h)              # a second enable keeps the one copy
    la, ka = run(lib, a, cfg, toks, cuts)
    lb, kb = run(lib, b, cfg, toks, cuts)
    for x, y in zip(la, lb):
        assert np.array_equal(x, y)
    for x, y in zip(ka, kb):
        assert np.array_equal(x, y)
    a.close()
    b.close()


def test_copy_full_width_1b(lib):
    """The 512-token prefill of the Llama 3.2 1B-shaped Q8_0 model, with and
    without the copy, on one handle."""
    cfg = synth.LLAMA1B_Q8.scaled(max_seq=600)
    W = synth.make_weights(cfg)
    toks = synth.prompt(cfg, 512)
    dec = lib.Decoder(cfg, W)
    la, ka = run(lib, dec, cfg, toks, [0, 512])
    lib.llm_reset(dec.h)
    lib.llm_prefill_f16_copy(dec.h)
    lb, kb = run(lib, dec, cfg, toks, [0, 512])
    for x, y in zip(la, lb):
        assert np.array_equal(x, y)
    for x, y in zip(ka, kb):
        assert np.array_equal(x, y)
    dec.close()


def test_copy_memory_is_freed(lib):
    cfg = q8cfg(n_layers=3, number=76)
    W = synth.make_weights(cfg)
    dec = lib.Decoder(cfg, W)
    lib.llm_prefill_f16_copy(dec.h)            # the expansion kernel's code is loaded once, not counted below
    lib.llm_prefill_f16_copy(dec.h, False)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    lib.llm_prefill_f16_copy(dec.h)
    torch.cuda.synchronize()
    layer_weights = cfg.n_layers * cfg.dim * (cfg.q_dim + 2 * cfg.kv_dim + 3 * cfg.ffn_dim) + \
        cfg.n_layers * cfg.q_dim * cfg.dim
    assert free0 - torch.cuda.mem_get_info()[0] >= 2 * layer_weights
    lib.llm_prefill_f16_copy(dec.h, False)
    lib.llm_prefill_f16_copy(dec.h, False)     # freeing twice does nothing
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    dec.close()


def test_copy_refusals(lib):
    for cfg in (q8cfg(wtype=synth.F16, number=77), q8cfg(wtype=synth.F32, number=78),
                q8cfg(ffn_dim=544, number=79)):      # 544: the prefill runs token by token
        dec = lib.Decoder(cfg, synth.make_weights(cfg))
        with pytest.raises(lib.LlmError) as e:
            lib.llm_prefill_f16_copy(dec.h)
        assert e.value.status == lib.LLM_ERR_UNSUPPORTED
        lib.llm_prefill_f16_copy(dec.h, False)        # nothing to free
        dec.close()


def test_copy_allocation_failure_keeps_the_expanding_path(lib):
    cfg = q8cfg(number=80)
    W = synth.make_weights(cfg)
    a = lib.Decoder(cfg, W)
    b = lib.Decoder(cfg, W)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    lib.llm_test_fail_alloc(1)
    with pytest.raises(lib.LlmError) as e:
        lib.llm_prefill_f16_copy(b.h)
    lib.llm_test_fail_alloc(0)
    assert e.value.status == lib.LLM_ERR_NO_MEMORY
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    toks = synth.prompt(cfg, 150)
    la, _ = run(lib, a, cfg, toks, [0, 150])
    lb, _ = run(lib, b, cfg, toks, [0, 150])
    for x, y in zip(la, lb):
        assert np.array_equal(x, y)
    a.close()
    b.close()
