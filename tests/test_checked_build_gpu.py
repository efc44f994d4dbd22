"""The LLM_CHECKED variant of the library (device-side index checks on the
decode step's global writes and weight-stream ranges, reporting
LLM_ERR_CHECK instead of trapping), run in a child process that loads it
(LLM_DECODE_VARIANT=checked):

- on valid models no check fires, and the logits are bitwise those of the
  regular build (the checks do not touch the arithmetic);
- a check made to fail (the logits bound narrowed through
  llm_test_logits_limit) is reported as LLM_ERR_CHECK with the writes past
  the bound skipped, and the handle works again after llm_reset."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import synth
from harness import prefill_kv_both

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
import numpy as np
sys.path[:0] = [sys.argv[1], sys.argv[1] + "/tests"]
import llama_decode_forward_gb300 as L
import synth, oracle
from harness import prefill_kv_both, check_logits
import test_checked_build_gpu as T
out = {"checked": L.llm_checked_build()}
for name, cfg in T.MODELS.items():
    W = synth.make_weights(cfg)
    ora = oracle.OracleModel(cfg, W, llamacpp_rounding=bool(cfg.numerics))
    dec = L.Decoder(cfg, W)
    prefill_kv_both(cfg, ora, dec, cfg.max_seq - 1)
    logits = np.empty(cfg.vocab, np.float32)
    rows = []
    for pos in T.POSITIONS:
        L.llm_decode_step(dec.h, 3, pos, logits)
        check_logits(logits, ora.forward(3, pos), cfg.wtype)
        rows.append(logits.view(np.uint32).tolist())
    out[name] = rows
    if cfg.wtype == synth.F16:
        L.llm_prefill(dec.h, synth.prompt(cfg, 40), 10, logits)
        out[name + "_prefill"] = logits.view(np.uint32).tolist()
    assert L.llm_test_guards(dec.h) == 0
    if name == "q8_0":
        half = cfg.vocab // 2
        prev = logits.copy()                  # the device buffer still holds these
        L.llm_test_logits_limit(dec.h, half)
        try:
            L.llm_decode_step(dec.h, 3, 5, logits)
            out["planted"] = "no error"
        except L.LlmError as e:
            out["planted"] = e.status
        ref = ora.forward(3, 5)
        out["planted_head_ok"] = bool(np.max(np.abs(logits[:half] - ref[:half])) <= 2e-2)
        out["planted_tail_untouched"] = bool(np.array_equal(logits[half:].view(np.uint32), prev[half:].view(np.uint32)))
        L.llm_test_logits_limit(dec.h, 0)
        L.llm_reset(dec.h)
        L.llm_decode_step(dec.h, 3, 5, logits)
        check_logits(logits, ora.forward(3, 5), cfg.wtype)
        out["after_reset"] = "ok"
    dec.close()
print("RESULT " + json.dumps(out))
"""


def small(wtype, **kw):
    base = dict(n_layers=2, dim=256, n_heads=8, n_kv_heads=2, head_dim=32, ffn_dim=544, vocab=1000, max_seq=160,
                eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=wtype, tied=False, number=90 + wtype)
    base.update(kw)
    return synth.ModelConfig("small_checked", **base)


MODELS = {
    "q8_0": small(synth.Q8_0, tied=True),
    "f16": small(synth.F16, rope_neox=1, bias=True, ffn_dim=512),
    "f32_hd128": small(synth.F32, dim=512, n_heads=4, n_kv_heads=1, head_dim=128, ffn_dim=320, vocab=513),
    "q8_0_llamacpp": small(synth.Q8_0, numerics=1),
}
POSITIONS = (0, 17, 100, 159)


@pytest.fixture(scope="module")
def child():
    env = dict(os.environ, LLM_DECODE_VARIANT="checked")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")][-1]
    return json.loads(line[len("RESULT "):])


def test_checked_build_is_loaded(child):
    assert child["checked"] == 1


@pytest.mark.parametrize("name", sorted(MODELS))
def test_checked_build_matches_regular_build_bitwise(child, name):
    import llama_decode_forward_gb300 as L
    assert not L.llm_checked_build()
    cfg = MODELS[name]
    W = synth.make_weights(cfg)
    import oracle
    ora = oracle.OracleModel(cfg, W, llamacpp_rounding=bool(cfg.numerics))
    dec = L.Decoder(cfg, W)
    prefill_kv_both(cfg, ora, dec, cfg.max_seq - 1)
    logits = np.empty(cfg.vocab, np.float32)
    for pos, want in zip(POSITIONS, child[name]):
        L.llm_decode_step(dec.h, 3, pos, logits)
        assert logits.view(np.uint32).tolist() == want, pos
    if cfg.wtype == synth.F16:
        L.llm_prefill(dec.h, synth.prompt(cfg, 40), 10, logits)
        assert logits.view(np.uint32).tolist() == child[name + "_prefill"]
    dec.close()


def test_failed_check_is_reported_and_skipped(child):
    import llama_decode_forward_gb300 as L
    assert child["planted"] == L.LLM_ERR_CHECK
    assert child["planted_head_ok"] and child["planted_tail_untouched"]
    assert child["after_reset"] == "ok"
