"""The oracle's row-split variant (orc_set_threads): every output element is
still computed by one thread in the same order, so a forward pass on several
threads is bitwise the single-thread one (logits and every cached K/V value).
This is what lets the full-size parity tests and the all-core CPU baseline use
every host core."""
import os

import numpy as np

import oracle
import synth


def _run(cfg, W, toks, n_threads):
    with oracle.threads(n_threads):
        ora = oracle.OracleModel(cfg, W)
        logits = [ora.forward(int(t), p).copy() for p, t in enumerate(toks)]
        kv = [ora.kv(l, w).copy() for l in range(cfg.n_layers) for w in (0, 1)]
        ora.close()
    return logits, kv


def test_threads_are_bitwise_single_thread():
    for wtype, kw in ((synth.Q8_0, {}), (synth.F16, dict(rope_neox=1, bias=True)), (synth.F32, {})):
        cfg = synth.ModelConfig("threads", n_layers=2, dim=128, n_heads=4, n_kv_heads=2, head_dim=32, ffn_dim=320,
                                vocab=333, max_seq=24, eps=1e-5, rope_base=10000.0, rope_neox=kw.get("rope_neox", 0),
                                wtype=wtype, tied=False, bias=kw.get("bias", False), number=97)
        W = synth.make_weights(cfg)
        toks = synth.prompt(cfg, 9)
        a_logits, a_kv = _run(cfg, W, toks, 1)
        b_logits, b_kv = _run(cfg, W, toks, max(4, os.cpu_count() or 4))
        for x, y in zip(a_logits, b_logits):
            assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
        for x, y in zip(a_kv, b_kv):
            assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def test_default_is_one_thread():
    """The threads context restores the single-thread default on exit."""
    with oracle.threads(3):
        pass
    cfg = synth.ModelConfig("threads1", n_layers=1, dim=64, n_heads=2, n_kv_heads=1, head_dim=32, ffn_dim=96,
                            vocab=40, max_seq=4, eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=synth.F32,
                            tied=True, number=98)
    W = synth.make_weights(cfg)
    ora = oracle.OracleModel(cfg, W)
    assert np.all(np.isfinite(ora.forward(1, 0)))
    ora.close()
