"""Host-side failure handling and memory-safety checks of the library, made
without faulting the GPU: injected allocation failures (llm_test_fail_alloc),
calls on destroyed handles, guard bands around the KV cache, the activations
and the prefill workspace (llm_test_guards), and reuse after llm_reset."""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import check_logits, prefill_kv_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import llama_decode_forward_gb300 as L
    return L


def small(wtype, **kw):
    base = dict(n_layers=2, dim=256, n_heads=8, n_kv_heads=2, head_dim=32, ffn_dim=544, vocab=1000, max_seq=160,
                eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=wtype, tied=False, number=80 + wtype)
    base.update(kw)
    return synth.ModelConfig("small_robust", **base)


def test_each_create_allocation_failure_is_clean(lib):
    """Every allocation of llm_create fails in turn: NO_MEMORY, a reason, no
    device memory left behind; then a normal create works."""
    cfg = small(synth.Q8_0)
    W = synth.make_weights(cfg)
    dw = lib.DeviceWeights(W)
    stream = torch.cuda.current_stream().cuda_stream
    # one full create and step first: the kernels' code and the context's own
    # buffers are loaded once, not counted as a leak below
    h = lib.llm_create(lib.config_struct(cfg), dw.struct, stream)
    lib.llm_decode_step(h, 5, 0)
    lib.llm_destroy(h)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    failed = 0
    for n in range(1, 40):
        lib.llm_test_fail_alloc(n)
        try:
            h = lib.llm_create(lib.config_struct(cfg), dw.struct, stream)
        except lib.LlmError as e:
            assert e.status == lib.LLM_ERR_NO_MEMORY, (n, e)
            assert "alloc" in str(e).lower(), str(e)
            torch.cuda.synchronize()
            assert torch.cuda.mem_get_info()[0] == free0, n
            failed += 1
            continue
        lib.llm_test_fail_alloc(0)
        break
    assert failed >= 5                      # weights, KV cache, layer table, activations, pinned words, maps
    ora = oracle.OracleModel(cfg, W)
    logits = np.empty(cfg.vocab, np.float32)
    lib.llm_decode_step(h, 5, 0, logits)
    check_logits(logits, ora.forward(5, 0), cfg.wtype)
    lib.llm_destroy(h)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_prefill_workspace_allocation_failure(lib):
    cfg = small(synth.F16, max_seq=300, ffn_dim=512)        # batched prefill: widths a multiple of 64
    W = synth.make_weights(cfg)
    ora = oracle.OracleModel(cfg, W)
    dec = lib.Decoder(cfg, W)
    toks = synth.prompt(cfg, 40)
    lib.llm_test_fail_alloc(1)
    with pytest.raises(lib.LlmError) as e:
        lib.llm_prefill(dec.h, toks, 0)
    lib.llm_test_fail_alloc(0)
    assert e.value.status == lib.LLM_ERR_NO_MEMORY
    logits = np.empty(cfg.vocab, np.float32)
    lib.llm_prefill(dec.h, toks, 0, logits)
    for i, t in enumerate(toks[:-1]):
        ora.forward(int(t), i)
    check_logits(logits, ora.forward(int(toks[-1]), len(toks) - 1), cfg.wtype)
    assert lib.llm_test_guards(dec.h) == 0
    dec.close()


def test_destroyed_handle_is_refused(lib):
    cfg = small(synth.F32, n_layers=1)
    W = synth.make_weights(cfg)
    dw = lib.DeviceWeights(W)
    h = lib.llm_create(lib.config_struct(cfg), dw.struct, torch.cuda.current_stream().cuda_stream)
    lib.llm_decode_step(h, 1, 0)
    lib.llm_destroy(h)
    lib.llm_destroy(h)                        # a second destroy does nothing
    lib.llm_destroy(None)
    raw = lib.binding._lib
    assert raw.llm_decode_step(h, 1, 1, None, None) == lib.LLM_ERR_INVALID_ARG
    assert raw.llm_reset(h) == lib.LLM_ERR_INVALID_ARG
    assert raw.llm_sync(h) == lib.LLM_ERR_INVALID_ARG
    assert not raw.llm_logits_device(h)
    assert raw.llm_launch_count(h) == 0
    assert raw.llm_last_error(h).decode() == "not a live handle"


def test_guard_bands_intact_and_detect_a_planted_write(lib):
    """Steps at the first and last cache rows, a prefill and the no-alloc
    step leave every guard byte as written; a byte changed next to either end
    of each buffer is reported."""
    cfg = small(synth.F16, max_seq=200, ffn_dim=512)
    W = synth.make_weights(cfg)
    ora = oracle.OracleModel(cfg, W)
    dec = lib.Decoder(cfg, W)
    prefill_kv_both(cfg, ora, dec, cfg.max_seq - 1)
    logits = np.empty(cfg.vocab, np.float32)
    for pos in (0, 1, cfg.max_seq - 1):
        lib.llm_decode_step(dec.h, 3, pos, logits)
        check_logits(logits, ora.forward(3, pos), cfg.wtype)
    lib.llm_prefill(dec.h, synth.prompt(cfg, 70), cfg.max_seq - 70)
    tok = torch.tensor([4], dtype=torch.int32, device="cuda")
    out = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    lib.llm_decode_step_noalloc(dec.h, tok, 5, out, am)
    assert lib.llm_test_guards(dec.h) == 0
    for band in range(6):                     # KV cache, activations, prefill workspace: before and after
        lib.llm_test_poke_guard(dec.h, band)
        assert lib.llm_test_guards(dec.h) == band + 1
    with pytest.raises(lib.LlmError) as e:
        lib.llm_test_poke_guard(dec.h, 6)
    assert e.value.status == lib.LLM_ERR_OUT_OF_RANGE
    dec.close()


def test_reuse_after_reset_matches_a_fresh_handle(lib):
    cfg = small(synth.Q8_0)
    W = synth.make_weights(cfg)
    a = lib.Decoder(cfg, W)
    b = lib.Decoder(cfg, W)
    x = np.empty(cfg.vocab, np.float32)
    y = np.empty(cfg.vocab, np.float32)
    for pos, tok in enumerate(synth.prompt(cfg, 6)):
        lib.llm_decode_step(a.h, int(tok), pos, x)
    lib.llm_reset(a.h)
    for pos, tok in enumerate(synth.prompt(cfg, 3)[::-1]):
        lib.llm_decode_step(a.h, int(tok), pos, x)
        lib.llm_decode_step(b.h, int(tok), pos, y)
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32)), pos
    a.close()
    b.close()
