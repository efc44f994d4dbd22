"""The five workloads at full size: greedy streams and logits against the oracle.

Teacher-forced runs feed the oracle's tokens to both sides and compare every
step's logits; free-running runs let the GPU feed its own argmax back on the
device (llm_generate) and require the same token stream, except after a step
whose oracle top-2 margin is below the tolerance (a near tie)."""
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


def oracle_stream(ora, prompt, n_gen):
    """Prompt forwards at 0..len-1, then greedy generation of n_gen tokens
    (the last generated token is not fed back).  Returns tokens, logits list."""
    logits = None
    for p, t in enumerate(prompt):
        logits = ora.forward(int(t), p)
    toks, all_logits = [], [logits]
    pos = len(prompt)
    for i in range(n_gen):
        toks.append(oracle.argmax(logits))
        if i == n_gen - 1:
            break
        logits = ora.forward(toks[-1], pos)
        all_logits.append(logits)
        pos += 1
    return toks, all_logits


def run_stream_workload(lib, cfg, prompt_len, n_gen):
    import torch
    W = synth.make_weights(cfg)
    prompt = synth.prompt(cfg, prompt_len)
    ora = oracle.OracleModel(cfg, W)
    ref_toks, ref_logits = oracle_stream(ora, prompt, n_gen)
    dec = lib.Decoder(cfg, W)
    # teacher-forced: every step's logits
    logits = np.empty(cfg.vocab, np.float32)
    lib.llm_prefill(dec.h, prompt, 0, logits)
    check_logits(logits, ref_logits[0], cfg.wtype, "prompt")
    worst = 0.0
    for i in range(1, n_gen):
        lib.llm_decode_step(dec.h, ref_toks[i - 1], prompt_len + i - 1, logits)
        worst = max(worst, check_logits(logits, ref_logits[i], cfg.wtype, f"step {i}"))
    # free-running with device-side feedback
    lib.llm_reset(dec.h)
    first = lib.llm_prefill(dec.h, prompt, 0)
    out = torch.zeros(n_gen - 1, dtype=torch.int32, device="cuda")
    lib.llm_generate(dec.h, first, prompt_len, n_gen - 1, out)
    lib.llm_sync(dec.h)
    got = [first] + out.cpu().tolist()
    for i, (g, r) in enumerate(zip(got, ref_toks)):
        if g != r:
            assert margin(ref_logits[i]) < TOL[cfg.wtype], f"stream diverged at {i}: {g} != {r}"
            break
    return worst


def test_tiny_llama_f32_stream(lib):
    """Tiny random Llama, F32: 8-token prompt, 32 greedy tokens."""
    run_stream_workload(lib, synth.TINY, 8, 32)


def test_stories15m_f32_stream(lib):
    """stories15M shape, F32: 1-token prompt, 256 greedy tokens (positions 0..255)."""
    run_stream_workload(lib, synth.STORIES15M, 1, 256)


@pytest.mark.parametrize("pos", [4095, 512, 32767])
def test_llama1b_q8_0_step_at_context(lib, pos):
    """Llama-3.2-1B shape, Q8_0: one step after pos seeded cache rows, the
    launch configuration the benchmark times."""
    cfg = synth.LLAMA1B_Q8
    W = synth.make_weights(cfg)
    ora = oracle.OracleModel(cfg, W, max_seq=pos + 1)
    dec = lib.Decoder(cfg, W)
    prefill_kv_both(cfg.scaled(max_seq=pos + 1), ora, dec, pos)
    tok = int(synth.prompt(cfg, 1)[0])
    with oracle.threads():
        ref = ora.forward(tok, pos)
    logits = np.empty(cfg.vocab, np.float32)
    am = lib.llm_decode_step(dec.h, tok, pos, logits)
    check_logits(logits, ref, cfg.wtype, f"pos {pos}")
    if am != oracle.argmax(ref):
        assert margin(ref) < TOL[cfg.wtype]


def test_qwen2_f16_prefill_512_and_128_greedy_steps(lib):
    """Qwen2-style F16 (NEOX, biases, tied), as the workload states: a
    512-token batched prefill (tensor-core GEMMs) from seeded uniform token
    ids, then 128 greedy decode steps; teacher-forced logits at every step and
    the free-running stream against the oracle (run on every host core, which
    gives the single-thread oracle's bits)."""
    with oracle.threads():
        run_stream_workload(lib, synth.QWEN2_F16.scaled(max_seq=640), 512, 128)


@pytest.mark.parametrize("ctx", [1, 1024, 4096, 16384])
def test_llama7b_q8_0_step_at_context(lib, ctx):
    """Llama-2-7B shape, Q8_0: one step at pos ctx-1 after ctx-1 seeded cache
    rows (the context sweep of the workload)."""
    cfg = synth.LLAMA7B_Q8
    pos = ctx - 1
    W = synth.make_weights(cfg)
    ora = oracle.OracleModel(cfg, W, max_seq=ctx)
    dec = lib.Decoder(cfg.scaled(max_seq=max(ctx, 16)), W)
    if pos:
        prefill_kv_both(cfg.scaled(max_seq=ctx), ora, dec, pos)
    tok = int(synth.prompt(cfg, 1)[0])
    with oracle.threads():
        ref = ora.forward(tok, pos)
    logits = np.empty(cfg.vocab, np.float32)
    am = lib.llm_decode_step(dec.h, tok, pos, logits)
    check_logits(logits, ref, cfg.wtype, f"ctx {ctx}")
    if am != oracle.argmax(ref):
        assert margin(ref) < TOL[cfg.wtype]
    # the K/V rows the step wrote at pos, against the oracle's (layer 0 and the last)
    for l in (0, cfg.n_layers - 1):
        k, v = dec.kv_tensors(l)
        for which, t in ((0, k), (1, v)):
            g = t[pos].cpu().numpy().view(np.float16).astype(np.float64)
            r = ora.kv(l, which)[pos].astype(np.float64)
            assert np.max(np.abs(g - r)) <= TOL[cfg.wtype], (l, which)
    ora.close()
    dec.close()
