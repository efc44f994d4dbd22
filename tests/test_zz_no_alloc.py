"""The decode step that allocates nothing (llm_decode_step_noalloc: working
memory in a fixed device array of the library, for callers that may not
allocate device memory while serving) against the regular decode step, on two
calls in a row.  Kept in its own file, collected last, so that it also runs
after every other test has used the library in this process."""
import numpy as np
import pytest

import synth
from harness import TOL

pytestmark = pytest.mark.gpu


def _cfg():
    return synth.ModelConfig("noalloc", n_layers=2, dim=256, n_heads=8, n_kv_heads=2, head_dim=32, ffn_dim=544,
                             vocab=1000, max_seq=160, eps=1e-5, rope_base=500000.0, rope_neox=0, wtype=synth.Q8_0,
                             tied=True, rope_freqs=True, number=61)


def _fill_kv(cfg, dec, n_rows):
    import torch
    for l in range(cfg.n_layers):
        k, v = dec.kv_tensors(l)
        for which, t in ((0, k), (1, v)):
            rows = synth.kv_rows(cfg, l, which, n_rows)
            t[:n_rows].copy_(torch.from_numpy(rows.view(np.int16)).to("cuda"))


def test_noalloc_step_matches_decode_step():
    import torch
    import llama_decode_forward_gb300 as L
    cfg = _cfg()
    W = synth.make_weights(cfg)
    ref = L.Decoder(cfg, W)
    new = L.Decoder(cfg, W)
    _fill_kv(cfg, ref, 90)
    _fill_kv(cfg, new, 90)
    torch.cuda.synchronize()
    toks = [int(t) for t in synth.prompt(cfg, 2)]
    ref_logits = np.empty(cfg.vocab, np.float32)
    tok_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits_dev = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
    am_dev = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for t, pos in zip(toks, (90, 91)):                 # two calls in a row; the second reads the first's KV row
        am_ref = L.llm_decode_step(ref.h, t, pos, ref_logits)
        tok_dev.fill_(t)
        torch.cuda.synchronize()
        L.llm_decode_step_noalloc(new.h, tok_dev, pos, logits_dev, am_dev)
        got = logits_dev.cpu().numpy()
        assert np.all(np.isfinite(got))
        d = float(np.max(np.abs(got.astype(np.float64) - ref_logits.astype(np.float64))))
        assert d <= TOL[synth.Q8_0], f"pos {pos}: max |dlogit| {d}"
        assert int(am_dev.item()) == am_ref
        for l in range(cfg.n_layers):
            for a, b in zip(ref.kv_tensors(l), new.kv_tensors(l)):
                assert torch.equal(a[pos], b[pos]), f"layer {l}: KV row {pos} differs"
    ref.close()
    new.close()


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
