"""The decode step that allocates nothing (llm_decode_step_noalloc: working
memory in a fixed device array of the library, for callers that may not
allocate device memory while serving) against the regular decode step, on two
calls in a row.  Both launch the same kernel on the same inputs, so logits,
argmax and the K/V rows they write must be the same bits; the logits are also
checked against the oracle.  Kept in its own file, collected last, so that it
also runs after every other test has used the library in this process."""
import numpy as np
import pytest

import oracle
import synth
from harness import TOL, check_logits

pytestmark = pytest.mark.gpu


def _cfg():
    return synth.ModelConfig("noalloc", n_layers=2, dim=256, n_heads=8, n_kv_heads=2, head_dim=32, ffn_dim=544,
                             vocab=1000, max_seq=160, eps=1e-5, rope_base=500000.0, rope_neox=0, wtype=synth.Q8_0,
                             tied=True, rope_freqs=True, number=61)


def _fill_kv(cfg, dec, n_rows, ora=None):
    import torch
    for l in range(cfg.n_layers):
        k, v = dec.kv_tensors(l)
        for which, t in ((0, k), (1, v)):
            rows = synth.kv_rows(cfg, l, which, n_rows)
            t[:n_rows].copy_(torch.from_numpy(rows.view(np.int16)).to("cuda"))
            if ora is not None:
                ora.set_kv_rows_f16(l, which, rows)


def test_noalloc_step_matches_decode_step():
    import torch
    import llama_decode_forward_gb300 as L
    cfg = _cfg()
    W = synth.make_weights(cfg)
    ref = L.Decoder(cfg, W)
    new = L.Decoder(cfg, W)
    ora = oracle.OracleModel(cfg, W)
    _fill_kv(cfg, ref, 90)
    _fill_kv(cfg, new, 90, ora)
    torch.cuda.synchronize()
    toks = [int(t) for t in synth.prompt(cfg, 2)]
    ref_logits = np.empty(cfg.vocab, np.float32)
    tok_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits_dev = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
    am_dev = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    handle_logits_before = None
    for t, pos in zip(toks, (90, 91)):                 # two calls in a row; the second reads the first's KV row
        am_ref = L.llm_decode_step(ref.h, t, pos, ref_logits)
        tok_dev.fill_(t)
        torch.cuda.synchronize()
        L.llm_decode_step_noalloc(new.h, tok_dev, pos, logits_dev, am_dev)
        got = logits_dev.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref_logits.view(np.uint32)), f"pos {pos}: logits differ"
        assert int(am_dev.item()) == am_ref
        check_logits(got, ora.forward(t, pos), synth.Q8_0, f"pos {pos} against the oracle")
        for l in range(cfg.n_layers):
            for a, b in zip(ref.kv_tensors(l), new.kv_tensors(l)):
                assert torch.equal(a[pos], b[pos]), f"layer {l}: KV row {pos} differs"
    ref.close()
    new.close()
    ora.close()


def test_noalloc_rejects_null_arguments():
    import torch
    import llama_decode_forward_gb300 as L
    cfg = _cfg()
    dec = L.Decoder(cfg, synth.make_weights(cfg))
    logits_dev = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
    with pytest.raises(L.LlmError) as ei:
        L.llm_decode_step_noalloc(dec.h, None, 0, logits_dev, None)
    assert ei.value.status == L.LLM_ERR_INVALID_ARG
    dec.close()


def test_noalloc_refuses_a_model_larger_than_the_array():
    """A model whose step needs more than the fixed array (here 121 layers
    with a 16384-wide FFN: its tagged vectors alone pass 16 MiB) is refused
    with UNSUPPORTED before anything is launched.  Every tensor points at one
    zero-filled device buffer; the weights' values do not matter here."""
    import ctypes
    import torch
    import llama_decode_forward_gb300 as L
    n_layers, dim, ffn = 121, 256, 16384
    cfg = L.llm_config(n_layers=n_layers, dim=dim, n_heads=8, n_kv_heads=2, head_dim=32, ffn_dim=ffn, vocab=64,
                       max_seq=8, rope_dims=32, eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=L.LLM_Q8_0)
    zeros = torch.zeros(ffn * dim // 32 * 34 // 4 + 1024, dtype=torch.int32, device="cuda")
    p = zeros.data_ptr()
    layers = (L.llm_layer_weights * n_layers)()
    for l in range(n_layers):
        for name, _ in L.llm_layer_weights._fields_:
            setattr(layers[l], name, None if name in ("bq", "bk", "bv") else p)
    w = L.llm_weights(tok_embd=p, output_norm=p, output=None, rope_freqs=None, layers=layers)
    h = ctypes.c_void_p()
    rc = L.binding._lib.llm_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(h))
    assert rc == L.LLM_OK, L.binding._lib.llm_last_error(None)
    try:
        tok = torch.zeros(1, dtype=torch.int32, device="cuda")
        am = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.empty(64, dtype=torch.float32, device="cuda")
        launches = L.llm_launch_count(h)
        with pytest.raises(L.LlmError) as ei:
            L.llm_decode_step_noalloc(h, tok, 0, logits, am)
        assert ei.value.status == L.LLM_ERR_UNSUPPORTED
        assert "scratch" in str(ei.value)
        assert L.llm_launch_count(h) == launches
    finally:
        L.binding._lib.llm_destroy(h)
