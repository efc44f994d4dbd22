"""The GGUF oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of oracle/gguf.py (a wrong default
alignment, padding rounded the wrong way, a dropped check, a check in the
wrong order, a wrong block size, a string length read as characters, a
wrong default in the model shape), loads the copy in place of the oracle,
and requires that at least one pin of test_gguf_oracle.py fails."""
import importlib.util
import os
import sys

import pytest

from oracle import gguf as G
import test_gguf_oracle as pins

SRC = G.__file__

MUTANTS = {
    "default_alignment_64": ("DEFAULT_ALIGNMENT = 32", "DEFAULT_ALIGNMENT = 64"),
    "pad_rounds_down": ("return (n + alignment - 1) // alignment * alignment",
                        "return n // alignment * alignment"),
    "offset_check_dropped": ("        if ti[\"offset\"] != expect:", "        if False:"),
    "end_check_dropped": ("        if end > len(data):", "        if False:"),
    "version_check_dropped": ("    if version != VERSION:", "    if False:"),
    "header_size_23": ("    if len(data) < 24:", "    if len(data) < 23:"),
    "q8_block_33": ("return n // 32 * 34", "return n // 32 * 33"),
    "f16_two_bytes_dropped": ("        return 2 * n", "        return 4 * n"),
    "string_length_in_chars": ("        return self.take(n).decode(\"utf-8\")",
                               "        return self.data[self.pos:].decode(\"utf-8\", \"ignore\")[:n] if "
                               "self.take(len(self.data[self.pos:].decode(\"utf-8\", \"ignore\")[:n].encode())) "
                               "is not None else ''"),
    "kv_heads_default_1": ("kv_heads = int(get(a + \".attention.head_count_kv\", heads))",
                           "kv_heads = int(get(a + \".attention.head_count_kv\", 1))"),
    "neox_for_llama": ("\"neox\": a == \"qwen2\"", "\"neox\": a == \"llama\""),
    "q8_scale_ignored": ("    return (d * q).reshape(-1)", "    return q.reshape(-1)"),
}

DETECTORS = [
    pins.test_header_is_24_bytes,
    pins.test_strings_and_arrays_byte_positions,
    lambda: pins.test_tensor_infos_alignment_and_offsets(None, 176, 192, 352),
    lambda: pins.test_tensor_infos_alignment_and_offsets(64, 209, 256, 384),
    *[(lambda e=e: pins.test_checks_in_order(*e)) for e in pins.EXAMPLE11],
    pins.test_decoding_f16_and_q8_0,
    pins.test_tensor_sizes,
    pins.test_header_shorter_than_24_bytes,
    lambda: pins.test_model_config_and_weight_counts(pins.TINY_MD, dict(arch="llama", dim=256, layers=4, heads=8,
                                                                        kv_heads=2, head_dim=32, ffn=704,
                                                                        vocab=151936, context_length=4096,
                                                                        rope_dims=32, neox=False),
                                                     705_024, 80_611_584),
    pins.test_model_config_defaults,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch, tmp_path):
    with open(SRC) as f:
        src = f.read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site of {name} not found exactly once"
    path = tmp_path / "gguf_mutant.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("gguf_mutant", path)
    mutant = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mutant)
    monkeypatch.setattr(pins, "G", mutant)
    caught = 0
    for d in DETECTORS:
        try:
            d()
        except (Exception, pytest.fail.Exception):      # a failed assert, a pytest.raises that did not raise
            caught += 1
    assert caught > 0, f"no pin catches the mutant {name}"
