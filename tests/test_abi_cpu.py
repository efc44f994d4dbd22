"""The C ABI without a GPU: the library builds, loads, exports every symbol
include/llm.h declares, and rejects bad arguments on the host."""
import ctypes
import os
import subprocess

import pytest

import llama_decode_forward_gb300 as L


def test_exports_every_declared_symbol():
    names = L.declared_symbols()
    assert len(names) >= 15
    lib = ctypes.CDLL(L.LIBRARY_PATH)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIBRARY_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported


def test_library_is_built_for_sm_103a():
    """Every compile and the link pass exactly one -gencode pair, sm_103a
    machine code from compute_103a (no other architecture, no PTX to JIT)."""
    from llama_decode_forward_gb300 import build as B
    want = ["-gencode", "arch=compute_103a,code=sm_103a"]
    for cmd in [B.compile_command(s, "x.o") for s in B.sources()] + [B.link_command(["x.o"], "lib.so")]:
        i = cmd.index("-gencode")
        assert cmd[i:i + 2] == want, cmd
        assert cmd.count("-gencode") == 1 and not any("-arch" in a for a in cmd), cmd
    assert B.compile_command("a.cu", "a.o", trace=True)[-4:-2] == ["-c", "a.cu"]
    assert "-DLLM_TRACE" in B.compile_command("a.cu", "a.o", trace=True)
    checked = B.compile_command("a.cu", "a.o", checked=True)
    assert "-DLLM_CHECKED" in checked and "-DLLM_TRACE" not in checked
    assert "-DLLM_CHECKED" not in B.compile_command("a.cu", "a.o")
    assert B.CHECKED_LIB != B.LIB and B.TRACE_LIB != B.LIB
    with pytest.raises(ValueError):
        B.build(trace=True, checked=True)


def test_status_strings():
    for s in range(0, -10, -1):
        assert L.llm_status_string(s) not in ("", "unknown status")
    assert L.llm_status_string(-99) == "unknown status"


def _cfg(**kw):
    base = dict(n_layers=2, dim=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96, vocab=50, max_seq=16,
                rope_dims=16, eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=L.LLM_Q8_0)
    base.update(kw)
    return L.llm_config(**base)


def _weights(n_layers=2, null_field=None):
    layers = (L.llm_layer_weights * n_layers)()
    for l in range(n_layers):
        for name, _ in L.llm_layer_weights._fields_:
            setattr(layers[l], name, None if name in ("bq", "bk", "bv") or name == null_field else 0x1000)
    return L.llm_weights(tok_embd=0x1000, output_norm=0x1000, output=None, rope_freqs=None, layers=layers)


@pytest.mark.parametrize("kw,status", [
    (dict(n_layers=0), L.LLM_ERR_INVALID_ARG),
    (dict(n_heads=3), L.LLM_ERR_INVALID_ARG),              # n_heads % n_kv_heads
    (dict(head_dim=8), L.LLM_ERR_INVALID_ARG),             # head_dim * n_heads != dim
    (dict(rope_dims=15), L.LLM_ERR_INVALID_ARG),           # odd
    (dict(rope_dims=32), L.LLM_ERR_INVALID_ARG),           # > head_dim
    (dict(ffn_dim=100), L.LLM_ERR_INVALID_ARG),            # Q8_0 needs multiples of 32
    (dict(wtype=2), L.LLM_ERR_UNSUPPORTED),
    (dict(wtype=L.LLM_F16, ffn_dim=100), L.LLM_ERR_UNSUPPORTED),
    (dict(dim=4 * 320, head_dim=320, ffn_dim=96), L.LLM_ERR_UNSUPPORTED),   # head_dim > 256
    (dict(max_seq=-1), L.LLM_ERR_INVALID_ARG),
    (dict(numerics=2), L.LLM_ERR_INVALID_ARG),
    (dict(numerics=-1), L.LLM_ERR_INVALID_ARG),
])
def test_create_rejects_bad_config(kw, status):
    with pytest.raises(L.LlmError) as e:
        L.llm_create(_cfg(**kw), _weights(n_layers=_cfg(**kw).n_layers if _cfg(**kw).n_layers > 0 else 1))
    assert e.value.status == status


def test_create_rejects_null_weight():
    with pytest.raises(L.LlmError) as e:
        L.llm_create(_cfg(), _weights(null_field="w_down"))
    assert e.value.status == L.LLM_ERR_INVALID_ARG


def test_create_failure_reason_without_a_handle():
    # no handle exists after a failed create: llm_last_error(NULL) holds the
    # calling thread's reason, and the Python error carries it
    with pytest.raises(L.LlmError) as e:
        L.llm_create(_cfg(rope_dims=15), _weights())
    assert "rope_dims must be even" in str(e.value)
    assert "rope_dims must be even" in L.llm_last_error(None)
    with pytest.raises(L.LlmError) as e:
        L.llm_create(_cfg(), _weights(null_field="wq"))
    assert L.llm_last_error(None) == "layer 0: a weight pointer is NULL"
    # another thread has its own reason
    import threading
    seen = []
    t = threading.Thread(target=lambda: seen.append(L.llm_last_error(None)))
    t.start()
    t.join()
    assert seen == [""]


def test_create_without_gpu_fails_loudly():
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except Exception:
        pass
    with pytest.raises(L.LlmError) as e:
        L.llm_create(_cfg(), _weights())
    assert e.value.status in (L.LLM_ERR_CUDA, L.LLM_ERR_UNSUPPORTED)


def test_null_handle_calls_are_rejected():
    assert L.binding._lib.llm_reset(None) == L.LLM_ERR_INVALID_ARG
    assert L.binding._lib.llm_sync(None) == L.LLM_ERR_INVALID_ARG
    assert L.binding._lib.llm_decode_step(None, 0, 0, None, None) == L.LLM_ERR_INVALID_ARG
    assert L.binding._lib.llm_launch_count(None) == 0
    assert L.binding._lib.llm_get_config(None, None) == L.LLM_ERR_INVALID_ARG
    assert L.binding._lib.llm_prefill_f16_copy(None, 1) == L.LLM_ERR_INVALID_ARG
    assert L.binding._lib.llm_prefill_f16_copy(None, 0) == L.LLM_ERR_INVALID_ARG
    L.binding._lib.llm_destroy(None)
