"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign or index, a transposed operand, an off-by-one, a wrong tie
rule), builds it on the CPU, swaps it in, and requires that at least one of
the pins in test_oracle_pins.py fails.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "llm_oracle.c")

MUTANTS = {
    "gqa_head_map": ("int kv_off = (h / group) * head_dim;", "int kv_off = (h % n_kv_heads) * head_dim;"),
    "rope_sign": ("vec[a] = p0 - p1;", "vec[a] = p0 + p1;"),
    "rope_k_skipped": ("orc_rope(k, c->n_kv_heads,", "if (0) orc_rope(k, c->n_kv_heads,"),
    "neox_pair": ("int b = neox ? a + rope_dims / 2 : a + 1;", "int b = neox ? a + 1 : a + rope_dims / 2;"),
    "attn_scale_dropped": ("att[t] = s / sq;", "att[t] = s;"),
    "causal_off_by_one": ("for (int t = 0; t <= pos; t++) {\n            const float *kt",
                          "for (int t = 0; t <= pos && t < pos + 1 - (pos > 0); t++) {\n            const float *kt"),
    "attn_residual_dropped": ("trace(m, \"attn_out\", l, xb, dim);\n        for (int i = 0; i < dim; i++) x[i] = x[i] + xb[i];",
                              "trace(m, \"attn_out\", l, xb, dim);\n        for (int i = 0; i < dim; i++) x[i] = xb[i];"),
    "gemv_column_reversed": ("float p = wr[i] * x[i]; s = s + p;", "float p = wr[i] * x[cols - 1 - i]; s = s + p;"),
    "rmsnorm_eps_dropped": ("sqrt(ss / (double)n + (double)eps)", "sqrt(ss / (double)n)"),
    "rmsnorm_gain_dropped": ("out[i] = t * g[i];", "out[i] = t;"),
    "silu_sign": ("float e = (float)exp((double)(-z));", "float e = (float)exp((double)(z));"),
    "swiglu_up_dropped": ("hb[i] = orc_silu(hb[i]) * hb2[i];", "hb[i] = orc_silu(hb[i]);"),
    "argmax_last_tie": ("if (v[i] > v[best]) best = i;", "if (v[i] >= v[best]) best = i;"),
    "q8_block_stride": ("const uint8_t *blk = p + (size_t)b * 34;", "const uint8_t *blk = p + (size_t)b * 32;"),
    "f16_no_ties_to_even": ("if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h++;", "if (rem >= 0x1000u) h++;"),
    "untied_output_ignored": ("m->w.output ? m->w.output : m->w.tok_embd", "m->w.tok_embd"),
    "kv_row_shift": ("kc[(int64_t)pos * kv_dim + i] = store(m, k[i]);",
                     "kc[(int64_t)(pos > 0 ? pos - 1 : 0) * kv_dim + i] = store(m, k[i]);"),
}

DETECTORS = [
    lambda: pins.test_whole_pass_printed_selftest_tokens("llama"),
    lambda: pins.test_whole_pass_printed_selftest_tokens("qwen2"),
    lambda: pins.test_whole_pass_against_dense_float64(oracle.F32, 0, False),
    lambda: pins.test_whole_pass_against_dense_float64(oracle.Q8_0, 0, True),
    pins.test_rmsnorm_printed_examples,
    pins.test_rope_printed_example_and_identities,
    pins.test_silu_and_swiglu_printed_example,
    pins.test_argmax_printed_example_and_ties,
    pins.test_attention_printed_gqa_example,
    pins.test_dequant_printed_example_ex2,
    pins.test_f16_matches_ieee_library_conversion,
    pins.test_matvec_printed_example,
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, source, monkeypatch):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation anchor for {name} not unique"
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "mutant.c")
        with open(src, "w") as f:
            f.write(source.replace(old, new))
        so = os.path.join(d, "libmutant.so")
        subprocess.check_call(["gcc", *oracle.CFLAGS, f"-I{os.path.dirname(SRC)}", "-o", so, src, "-lm"])
        monkeypatch.setattr(oracle, "_LIB", oracle.load(so))
        caught = []
        for det in DETECTORS:
            try:
                det()
            except AssertionError:
                caught.append(det)
                break
        assert caught, f"no pin detects mutant {name}"
