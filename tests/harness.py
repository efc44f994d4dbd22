"""Shared helpers of the parity tests: build a model on both sides from the
same seeded inputs and compare what the CUDA library returns with the oracle.

Tolerances (from the acceptance rules of the decode pass): max |logit
difference| <= 2e-3 for F32 weights and <= 2e-2 for F16 / Q8_0 weights;
argmax identical unless the oracle's top-2 margin is below that tolerance;
Q8_0 decoding and the F16 KV store bit-exact."""
from __future__ import annotations

import numpy as np

import synth

TOL = {synth.F32: 2e-3, synth.F16: 2e-2, synth.Q8_0: 2e-2}


def margin(logits: np.ndarray) -> float:
    top2 = np.partition(logits.astype(np.float64), -2)[-2:]
    return float(top2[1] - top2[0])


def check_logits(gpu: np.ndarray, ref: np.ndarray, wtype: int, what: str = "") -> float:
    tol = TOL[wtype]
    assert gpu.shape == ref.shape
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU logits"
    d = float(np.max(np.abs(gpu.astype(np.float64) - ref.astype(np.float64))))
    assert d <= tol, f"{what}: max |dlogit| {d:.3g} > {tol}"
    ga, ra = int(np.argmax(gpu)), int(np.argmax(ref))
    if ga != ra:
        assert margin(ref) < tol, f"{what}: argmax {ga} != oracle {ra} with margin {margin(ref):.3g}"
    return d


def prefill_kv_both(cfg, oracle_model, decoder, n_rows: int):
    """Fill rows 0..n_rows-1 of every layer's cache with the seeded F16 rows."""
    import torch
    for l in range(cfg.n_layers):
        for which in (0, 1):
            rows = synth.kv_rows(cfg, l, which, n_rows)
            oracle_model.set_kv_rows_f16(l, which, rows)
            k, v = decoder.kv_tensors(l)
            (k if which == 0 else v)[:n_rows].copy_(torch.from_numpy(rows.view(np.int16)).to("cuda"))
    torch.cuda.synchronize()


def gpu_kv(decoder, layer: int, which: int, rows) -> np.ndarray:
    k, v = decoder.kv_tensors(layer)
    t = (k if which == 0 else v)[rows]
    return t.cpu().numpy().view(np.uint16)
