"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks one oracle function against printed worked examples
(tests/golden/, each file citing its page and example), closed forms,
invariants, library routines, or brute force on tiny inputs.
"""
import json
import math
import os
import types

import numpy as np
import pytest

import oracle
from javarandom import JavaRandom, java_round

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def f32(x):
    return float(np.float32(x))


def fmt(values, decimals):
    return [f"{v:.{decimals}f}" for v in values]


# ------------------------------------------------------------------ F16 --
def test_f16_printed_example():
    g = golden("gguf_ffm_ex7_f16.json")
    v = np.array([np.float32(np.float32(0.1) * np.float32(i)) - np.float32(0.35) for i in range(12)], np.float32)
    bits = oracle.f32_to_f16(v)
    back = oracle.f16_to_f32(bits)
    assert fmt(back, 6) == fmt(g["f16_decoded"], 6)
    assert int(bits[1]) == int(g["element1_bits"], 16)


def test_f16_matches_ieee_library_conversion():
    # numpy's float16 cast is IEEE round-to-nearest-even, incl. subnormals and overflow
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-5).astype(np.float32),      # FP16 subnormal range
        (rng.standard_normal(5000) * 1e-8).astype(np.float32),       # underflow to zero
        (rng.standard_normal(5000) * 7e4).astype(np.float32),        # overflow to inf
        np.array([65504, 65519.99, 65520, -65520, 2 ** -24, 2 ** -25, 2 ** -25 * 1.0000001, 3 * 2 ** -26,
                  6.1035156e-05, 0.0, -0.0, np.inf, -np.inf], np.float32),
    ])
    # exact halfway cases: FP16 value + half an ULP
    h = rng.integers(0, 0x7bff, 3000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float32)
    hi = (h + 1).view(np.float16).astype(np.float32)
    x = np.concatenate([x, ((lo.astype(np.float64) + hi) / 2).astype(np.float32)])
    ours = oracle.f32_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    allbits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    allbits = allbits[(allbits & 0x7c00) != 0x7c00]                   # skip inf/NaN encodings
    assert np.array_equal(oracle.f16_to_f32(allbits), allbits.view(np.float16).astype(np.float32))


# ------------------------------------------------------- weight decoding --
def test_dequant_printed_example_ex2():
    g = golden("forward_pass_java_ex2_dequant.json")
    w = np.array([np.float32(math.cos(i * 0.7)) * np.float32(0.08) for i in range(64)], np.float32)
    f16 = oracle.f32_to_f16(w)
    q8 = oracle.quantize_q8_0(w)
    assert q8.size == g["Q8_0"]["bytes"]
    for name, data, wt in (("F32", w, oracle.F32), ("F16", f16, oracle.F16), ("Q8_0", q8, oracle.Q8_0)):
        x = oracle.dequant_row(data, wt, 0, 64)
        assert fmt(x[1:4], 7) == fmt(g[name]["x1_3"], 7), name
        err = np.max(np.abs(x.astype(np.float64) - w.astype(np.float64)))
        assert f"{err:.7f}" == f"{g[name]['max_error']:.7f}", name


def test_q8_0_blocks_printed_example():
    g = golden("gguf_ffm_ex8_q8_0.json")
    x = np.array([np.float32(math.sin(i * 0.3)) * np.float32(0.1 if i < 32 else 1.0) for i in range(128)],
                 np.float32)
    t = oracle.quantize_q8_0(x)
    assert t.size == g["tensor_bytes"]
    for b, blk in enumerate(g["blocks"]):
        at = blk["byte"]
        assert at == 34 * b
        d = oracle.f16_to_f32(np.array([int(t[at]) | (int(t[at + 1]) << 8)], np.uint16))[0]
        assert f"{d:.6f}" == f"{blk['d']:.6f}"
        assert [int(np.int8(v)) for v in t[at + 2:at + 6].view(np.int8)] == blk["qs0_3"]
    for r, row in enumerate(g["rows"]):
        vals = oracle.dequant_row(t, oracle.Q8_0, r, 64)
        assert f"{vals[5]:.6f}" == f"{row['element5']:.6f}"
        assert f"{x[r * 64 + 5]:.6f}" == f"{row['original5']:.6f}"
        err = np.max(np.abs(vals.astype(np.float64) - x[r * 64:(r + 1) * 64]))
        assert f"{err:.6f}" == f"{row['max_error']:.6f}"


def _brute_q8_decode(blocks, rows, cols):
    b = blocks.reshape(rows, cols // 32, 34)
    d = b[:, :, 0:2].copy().view(np.uint16).view(np.float16).astype(np.float32)   # [rows, nb, 1]
    qs = b[:, :, 2:].view(np.int8).astype(np.float32)
    return (d * qs).reshape(rows, cols)


def test_q8_0_decode_brute_force_including_edge_scales():
    rng = np.random.default_rng(1)
    rows, cols = 7, 96
    blocks = rng.integers(0, 256, rows * cols // 32 * 34).astype(np.uint8)
    scales = np.array([0x0000, 0x0001, 0x03ff, 0x0400, 0x7bff, 0x8001, 0x3c00], np.uint16)   # 0, subnormals, max
    bb = blocks.reshape(-1, 34)
    for i, s in enumerate(scales):
        bb[i, 0], bb[i, 1] = s & 0xff, s >> 8
    bb[0, 2], bb[1, 3] = 0x80, 0x7f                                     # quants -128 and 127
    ref = _brute_q8_decode(blocks, rows, cols)
    for r in range(rows):
        got = oracle.dequant_row(blocks, oracle.Q8_0, r, cols)
        assert np.array_equal(got.view(np.uint32), ref[r].view(np.uint32))


def test_f16_weight_decode_brute_force():
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 0x7c00, 3 * 40).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32).reshape(3, 40)
    for r in range(3):
        assert np.array_equal(oracle.dequant_row(bits, oracle.F16, r, 40), ref[r])


# -------------------------------------------------------------- RMSNorm --
def test_rmsnorm_printed_examples():
    g = golden("forward_pass_java_ex4_rmsnorm.json")
    for case in g["cases"]:
        y = oracle.rmsnorm(case["x"], case["w"], g["eps"])
        assert [repr(float(v)) for v in y] == [repr(float(np.float32(v))) for v in case["y"]]
    r = JavaRandom(g["random_256"]["seed"])
    h = np.array([np.float32(r.next_gaussian() * 0.02) for _ in range(256)], np.float32)
    rms = lambda v: math.sqrt(float(np.sum(v.astype(np.float64) ** 2)) / v.size)
    y = oracle.rmsnorm(h, np.ones(256), g["eps"])
    assert f"{rms(h):.5f}" == f"{g['random_256']['rms_before']:.5f}"
    assert f"{rms(y):.5f}" == f"{g['random_256']['rms_after']:.5f}"
    y = oracle.rmsnorm(np.full(256, 1e-4, np.float32), np.ones(256), g["eps"])
    assert f"{rms(y):.5f}" == f"{g['eps_dominated']['rms_after']:.5f}"


def test_rmsnorm_closed_forms():
    rng = np.random.default_rng(3)
    for n in (4, 256, 2048, 4096):
        x = rng.standard_normal(n).astype(np.float32) * 3
        eps = 1e-5
        m = float(np.mean(x.astype(np.float64) ** 2))
        y = oracle.rmsnorm(x, np.ones(n), eps)
        rms_y = math.sqrt(float(np.mean(y.astype(np.float64) ** 2)))
        assert abs(rms_y - math.sqrt(m / (m + eps))) < 2e-6
        g = (1 + 0.1 * rng.standard_normal(n)).astype(np.float32)
        y = oracle.rmsnorm(x, g, eps).astype(np.float64)
        ref = x.astype(np.float64) / math.sqrt(m + eps) * g
        assert np.max(np.abs(y - ref) / np.abs(ref).clip(1e-30)) < 4e-7


# ------------------------------------------------------------------ GEMV --
def test_matvec_printed_example():
    g = golden("forward_pass_java_ex5_matvec.json")
    cols, rows = g["dims"]
    out = oracle.matvec(np.array(g["w"], np.float32), oracle.F32, g["x"], rows, cols)
    assert list(out) == g["out"]
    assert list(out) != g["bytes_read_as_columns"]


@pytest.mark.parametrize("wtype", [oracle.F32, oracle.F16, oracle.Q8_0])
def test_matvec_against_float64_matmul(wtype):
    rng = np.random.default_rng(4 + wtype)
    rows, cols = 37, 256
    wf = (rng.standard_normal((rows, cols)) * 0.05).astype(np.float32)
    if wtype == oracle.F32:
        data, dense = wf, wf
    elif wtype == oracle.F16:
        data = wf.astype(np.float16).view(np.uint16)
        dense = data.view(np.float16).astype(np.float32)
    else:
        data = oracle.quantize_q8_0(wf.ravel())
        dense = _brute_q8_decode(data, rows, cols)
    x = rng.standard_normal(cols).astype(np.float32)
    out = oracle.matvec(data, wtype, x, rows, cols).astype(np.float64)
    ref = dense.astype(np.float64) @ x.astype(np.float64)
    bound = cols * 2.0 ** -23 * (np.abs(dense.astype(np.float64)) @ np.abs(x.astype(np.float64)))
    assert np.all(np.abs(out - ref) <= bound)


# ------------------------------------------------------------------ RoPE --
def test_rope_printed_example_and_identities():
    g = golden("forward_pass_java_ex6_rope.json")
    x = np.array(g["x"], np.float32)
    normal = oracle.rope(x, 1, 8, 8, 1, g["base"], False)
    neox = oracle.rope(x, 1, 8, 8, 1, g["base"], True)
    assert fmt(normal, 3) == fmt(g["normal"], 3)
    assert fmt(neox, 3) == fmt(g["neox"], 3)
    perm = np.array(g["interleave_permutation"])
    assert np.array_equal(oracle.rope(x[perm], 1, 8, 8, 1, g["base"], False).view(np.uint32),
                          neox[perm].view(np.uint32))
    assert np.array_equal(oracle.rope(x, 1, 8, 8, 0, g["base"], False).view(np.uint32), x.view(np.uint32))


def test_rope_invariants_random():
    rng = np.random.default_rng(6)
    for hd, base in ((64, 500000.0), (128, 10000.0), (48, 10000.0), (64, 1e6)):
        nh = 3
        x = rng.standard_normal(nh * hd).astype(np.float32)
        for pos in (0, 1, 7, 511, 4095, 32767):
            for neox in (False, True):
                y = oracle.rope(x, nh, hd, hd, pos, base, neox)
                if pos == 0:
                    assert np.array_equal(y.view(np.uint32), x.view(np.uint32))
                # each pair keeps its length
                for h in range(nh):
                    for i in range(hd // 2):
                        a = h * hd + (i if neox else 2 * i)
                        b = a + (hd // 2 if neox else 1)
                        n0 = math.hypot(x[a], x[b])
                        n1 = math.hypot(y[a], y[b])
                        assert abs(n1 - n0) <= 4e-7 * max(n0, 1e-30) + 1e-12
            # normal(permuted x) == permuted NEOX(x), bit for bit
            perm = np.concatenate([h * hd + np.stack([np.arange(hd // 2), np.arange(hd // 2) + hd // 2], 1).ravel()
                                   for h in range(nh)])
            assert np.array_equal(oracle.rope(x[perm], nh, hd, hd, pos, base, False).view(np.uint32),
                                  oracle.rope(x, nh, hd, hd, pos, base, True)[perm].view(np.uint32))


def test_rope_angles_against_float64_rotation():
    # theta_i = pos * base^(-2i/n); the float chain drifts by a few float ulps of theta
    rng = np.random.default_rng(7)
    hd, base, pos = 64, 500000.0, 1000
    x = rng.standard_normal(hd).astype(np.float32)
    y = oracle.rope(x, 1, hd, hd, pos, base, False).astype(np.float64)
    for i in range(hd // 2):
        th = pos * base ** (-2.0 * i / hd)
        a, b = float(x[2 * i]), float(x[2 * i + 1])
        ra, rb = a * math.cos(th) - b * math.sin(th), a * math.sin(th) + b * math.cos(th)
        tol = (abs(a) + abs(b)) * (abs(th) * 2 ** -23 * (i + 2) + 2 ** -22)
        assert abs(y[2 * i] - ra) <= tol and abs(y[2 * i + 1] - rb) <= tol


def test_rope_frequency_divisors():
    rng = np.random.default_rng(8)
    hd = 64
    x = rng.standard_normal(2 * hd).astype(np.float32)
    ones = np.ones(hd // 2, np.float32)
    twos = np.full(hd // 2, 2.0, np.float32)
    for pos in (2, 64, 4094):
        assert np.array_equal(oracle.rope(x, 2, hd, hd, pos, 500000.0, False, ones).view(np.uint32),
                              oracle.rope(x, 2, hd, hd, pos, 500000.0, False).view(np.uint32))
        # dividing every angle by 2 equals rotating at half the position (power-of-two scaling is exact)
        assert np.array_equal(oracle.rope(x, 2, hd, hd, pos, 500000.0, False, twos).view(np.uint32),
                              oracle.rope(x, 2, hd, hd, pos // 2, 500000.0, False).view(np.uint32))


# ----------------------------------------------------- SiLU and SwiGLU --
def test_silu_and_swiglu_printed_example():
    g = golden("forward_pass_java_ex8_swiglu.json")
    assert fmt([oracle.silu(z) for z in g["silu"]["z"]], 4) == fmt(g["silu"]["y"], 4)
    b = g["block"]
    gate = oracle.matvec(np.array(b["gate_w"], np.float32), oracle.F32, b["x"], b["ffn"], b["dim"])
    up = oracle.matvec(np.array(b["up_w"], np.float32), oracle.F32, b["x"], b["ffn"], b["dim"])
    h = np.array([np.float32(oracle.silu(gv)) * uv for gv, uv in zip(gate, up)], np.float32)
    down = oracle.matvec(np.array(b["down_w"], np.float32), oracle.F32, h, b["dim"], b["ffn"])
    assert fmt(gate, 3) == fmt(b["gate"], 3)
    assert fmt([oracle.silu(v) for v in gate], 3) == fmt(b["silu_gate"], 3)
    assert fmt(up, 3) == fmt(b["up"], 3)
    assert fmt(h, 3) == fmt(b["h"], 3)
    assert fmt(down, 3) == fmt(b["down"], 3)


def test_silu_closed_form():
    for z in np.linspace(-30, 30, 601, dtype=np.float32):
        ref = float(z) / (1.0 + math.exp(-float(z)))
        assert abs(oracle.silu(z) - ref) <= 3 * 2 ** -24 * abs(ref) + 1e-45


# ---------------------------------------------------------------- argmax --
def test_argmax_printed_example_and_ties():
    g = golden("forward_pass_java_ex9_logits.json")
    logits = oracle.matvec(np.array(g["output_w"], np.float32), oracle.F32, g["h"], g["vocab"], g["dim"])
    assert fmt(logits, 3) == fmt(g["logits"], 3)
    p = np.exp(logits.astype(np.float64) - logits.max())
    assert fmt(p / p.sum(), 3) == fmt(g["probabilities"], 3)
    assert oracle.argmax(logits) == g["greedy"] == int(np.argmax(p))
    assert oracle.argmax(g["tie"]["v"]) == g["tie"]["argmax"]
    rng = np.random.default_rng(9)
    for _ in range(50):
        v = rng.integers(-5, 6, 1000).astype(np.float32)               # many exact ties
        assert oracle.argmax(v) == int(np.argmax(v))                   # numpy: first occurrence


# ------------------------------------------------------------ attention --
def test_attention_printed_gqa_example():
    g = golden("forward_pass_java_ex7_gqa.json")
    heads, kvh, hd = g["heads"], g["kv_heads"], g["head_dim"]
    kv_dim, ctx, group = kvh * hd, 8, heads // kvh
    kc = np.zeros((ctx, kv_dim), np.float32)
    vc = np.zeros((ctx, kv_dim), np.float32)
    r = JavaRandom(g["seed"])
    for pos in range(3):
        q = np.array([np.float32(java_round(r.next_gaussian() * 10)) / np.float32(10) for _ in range(heads * hd)],
                     np.float32)
        for i in range(kv_dim):
            kc[pos, i] = np.float32(java_round(r.next_gaussian() * 10)) / np.float32(10)
            vc[pos, i] = np.float32(pos + 1) + np.float32(i) / np.float32(10)
        out = oracle.attention(q, kc, vc, heads, kvh, hd, pos)
        assert fmt(out[0:2], 3) == fmt(g["head0"][pos], 3)
        assert fmt(out[4:6], 3) == fmt(g["head2"][pos], 3)
        # the weights: attend over one-hot values so that the output is a_t itself
        for t in range(pos + 1):
            onehot = np.zeros_like(vc)
            onehot[t, :] = 1.0
            w = oracle.attention(q, kc, onehot, heads, kvh, hd, pos)
            got = [w[h * hd] for h in range(heads)]
            assert fmt(got, 2) == fmt([g["weights"][pos][h][t] for h in range(heads)], 2)
            for h in range(heads):                                      # head h reads KV head h // group
                assert h // group == h * kvh // heads


def test_attention_f16_cache_printed_differences():
    g = golden("forward_pass_java_ex10_f16cache.json")
    r = JavaRandom(g["seed"])
    hd = g["head_dim"]
    for case in g["cases"]:
        n = case["n"]
        q = np.array([np.float32(r.next_gaussian()) for _ in range(hd)], np.float32)
        k = np.zeros((n, hd), np.float32)
        v = np.zeros((n, hd), np.float32)
        for t in range(n):
            for i in range(hd):
                k[t, i] = np.float32(r.next_gaussian())
                v[t, i] = np.float32(r.next_gaussian())
        exact = oracle.attention(q, k, v, 1, 1, hd, n - 1)
        kr = oracle.f16_to_f32(oracle.f32_to_f16(k)).reshape(n, hd)
        vr = oracle.f16_to_f32(oracle.f32_to_f16(v)).reshape(n, hd)
        half = oracle.attention(q, kr, vr, 1, 1, hd, n - 1)
        assert f"{np.max(np.abs(exact)):.4f}" == f"{case['largest_output']:.4f}"
        assert f"{np.max(np.abs(exact - half)):.6f}" == f"{case['largest_diff']:.6f}"


def test_attention_structural_properties():
    rng = np.random.default_rng(10)
    nh, nkv, hd, pos = 8, 2, 16, 37
    q = rng.standard_normal(nh * hd).astype(np.float32)
    k = rng.standard_normal((pos + 1 + 5, nkv * hd)).astype(np.float32)
    v = rng.standard_normal((pos + 1 + 5, nkv * hd)).astype(np.float32)
    k[pos + 1:] = np.nan                                                # rows after pos are never read
    v[pos + 1:] = np.nan
    out = oracle.attention(q, k, v, nh, nkv, hd, pos)
    assert np.all(np.isfinite(out))
    # weights sum to one: attend over all-ones values
    ones = np.ones_like(v)
    assert np.max(np.abs(oracle.attention(q, k, ones, nh, nkv, hd, pos) - 1.0)) < 1e-6
    # position 0: the output is V of the head's KV group, bit for bit
    out0 = oracle.attention(q, k, v, nh, nkv, hd, 0)
    for h in range(nh):
        g = h // (nh // nkv)
        assert np.array_equal(out0[h * hd:(h + 1) * hd], v[0, g * hd:(g + 1) * hd])
    # brute force in float64 with a library softmax
    from scipy.special import softmax
    for h in range(nh):
        g = h // (nh // nkv)
        s = k[:pos + 1, g * hd:(g + 1) * hd].astype(np.float64) @ q[h * hd:(h + 1) * hd].astype(np.float64)
        a = softmax(s / math.sqrt(hd))
        ref = a @ v[:pos + 1, g * hd:(g + 1) * hd].astype(np.float64)
        assert np.max(np.abs(out[h * hd:(h + 1) * hd] - ref)) < 1e-5


# ----------------------------------------------------------- whole pass --
def _selftest_model(neox):
    g = golden("forward_pass_java_ex13_selftest.json")
    s = g["shape"]
    dim, nl, ffn, vocab = s["dim"], s["layers"], s["ffn"], s["vocab"]
    r = JavaRandom(g["seed"])

    def init(rows, cols):
        return np.array([np.float32(r.next_gaussian() / math.sqrt(cols)) for _ in range(rows * cols)], np.float32)

    ones = np.ones(dim, np.float32)
    T = types.SimpleNamespace(tok_embd=init(vocab, dim), output=init(vocab, dim), output_norm=ones,
                              rope_freqs=None, layers=[])
    for _ in range(nl):
        L = {"attn_norm": ones, "ffn_norm": ones, "bq": None, "bk": None, "bv": None}
        L["wq"] = init(dim, dim)
        L["wk"] = init(8, dim)
        L["wv"] = init(8, dim)
        L["wo"] = init(dim, dim)
        L["w_gate"] = init(ffn, dim)
        L["w_up"] = init(ffn, dim)
        L["w_down"] = init(dim, ffn)
        T.layers.append(L)
    cfg = types.SimpleNamespace(n_layers=nl, dim=dim, n_heads=s["heads"], n_kv_heads=s["kv_heads"],
                                head_dim=dim // s["heads"], ffn_dim=ffn, vocab=vocab, max_seq=s["context"],
                                rope_dims=dim // s["heads"], eps=s["eps"], rope_base=s["rope_base"],
                                rope_neox=int(neox), wtype=oracle.F32)
    return g, cfg, T


@pytest.mark.parametrize("arch", ["llama", "qwen2"])
def test_whole_pass_printed_selftest_tokens(arch):
    """The pages' self-test: greedy ids printed for both RoPE layouts, and the
    cached pass bit-identical to recomputation from position 0 at every step."""
    g, cfg, T = _selftest_model(arch == "qwen2")
    cached = oracle.OracleModel(cfg, T, f16_cache=False)
    seq = list(g["prompt"])
    logits = None
    for p in range(len(seq)):
        logits = cached.forward(seq[p], p)
    for _ in range(g["steps"]):
        uncached = oracle.OracleModel(cfg, T, f16_cache=False)
        for p in range(len(seq)):
            ref = uncached.forward(seq[p], p)
        assert np.array_equal(logits.view(np.uint32), ref.view(np.uint32))
        seq.append(oracle.argmax(logits))
        logits = cached.forward(seq[-1], len(seq) - 1)
    assert seq[len(g["prompt"]):] == g["generated"][arch]


def _dense_float64_logits(cfg, T, tokens, f16_cache):
    """Independent batched evaluation in float64: all positions at once with a
    causal mask, weights decoded by numpy (no oracle code involved)."""
    def dense(a, rows, cols):
        if cfg.wtype == oracle.F32:
            return a.reshape(rows, cols).astype(np.float64)
        if cfg.wtype == oracle.F16:
            return a.view(np.float16).astype(np.float64).reshape(rows, cols)
        return _brute_q8_decode(a, rows, cols).astype(np.float64)
    n, d, hd = len(tokens), cfg.dim, cfg.head_dim
    nh, nkv = cfg.n_heads, cfg.n_kv_heads
    def norm(x, g):
        return x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + cfg.eps) * g
    def rope(x, nheads):                                  # x [n, nheads*hd]
        x = x.reshape(n, nheads, hd).copy()
        i = np.arange(hd // 2)
        th = np.arange(n)[:, None] * cfg.rope_base ** (-2.0 * i / hd)[None, :]
        c, s = np.cos(th)[:, None, :], np.sin(th)[:, None, :]
        a_idx, b_idx = (i, i + hd // 2) if cfg.rope_neox else (2 * i, 2 * i + 1)
        a, b = x[:, :, a_idx].copy(), x[:, :, b_idx].copy()
        x[:, :, a_idx], x[:, :, b_idx] = a * c - b * s, a * s + b * c
        return x.reshape(n, nheads * hd)
    x = dense(T.tok_embd, cfg.vocab, d)[np.array(tokens)]
    for L in T.layers:
        h = norm(x, L["attn_norm"])
        q = h @ dense(L["wq"], nh * hd, d).T
        k = h @ dense(L["wk"], nkv * hd, d).T
        v = h @ dense(L["wv"], nkv * hd, d).T
        q, k = rope(q, nh), rope(k, nkv)
        if f16_cache:
            k = k.astype(np.float16).astype(np.float64)
            v = v.astype(np.float16).astype(np.float64)
        o = np.zeros((n, nh * hd))
        mask = np.tril(np.ones((n, n), bool))
        for hh in range(nh):
            gg = hh // (nh // nkv)
            s = q[:, hh * hd:(hh + 1) * hd] @ k[:, gg * hd:(gg + 1) * hd].T / math.sqrt(hd)
            s = np.where(mask, s, -np.inf)
            a = np.exp(s - s.max(axis=1, keepdims=True))
            a /= a.sum(axis=1, keepdims=True)
            o[:, hh * hd:(hh + 1) * hd] = a @ v[:, gg * hd:(gg + 1) * hd]
        x = x + o @ dense(L["wo"], d, nh * hd).T
        h = norm(x, L["ffn_norm"])
        gt = h @ dense(L["w_gate"], cfg.ffn_dim, d).T
        up = h @ dense(L["w_up"], cfg.ffn_dim, d).T
        x = x + (gt / (1 + np.exp(-gt)) * up) @ dense(L["w_down"], d, cfg.ffn_dim).T
    h = norm(x, T.output_norm)
    wout = T.output if T.output is not None else T.tok_embd
    return h @ dense(wout, cfg.vocab, d).T


@pytest.mark.parametrize("wtype,neox,tied", [(oracle.F32, 0, False), (oracle.F16, 1, True), (oracle.Q8_0, 0, True)])
def test_whole_pass_against_dense_float64(wtype, neox, tied):
    import synth
    cfg = synth.ModelConfig("tiny-check", n_layers=2, dim=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96,
                            vocab=50, max_seq=16, eps=1e-5, rope_base=10000.0, rope_neox=neox, wtype=wtype,
                            tied=tied, number=90 + wtype)
    T = synth.make_weights(cfg)
    tokens = [int(t) for t in synth.prompt(cfg, 9)]
    for f16_cache in (False, True):
        m = oracle.OracleModel(cfg, T, f16_cache=f16_cache)
        ref = _dense_float64_logits(cfg, T, tokens, f16_cache)
        for p, t in enumerate(tokens):
            logits = m.forward(t, p).astype(np.float64)
            scale = np.max(np.abs(ref[p]))
            # F16 cache: both sides round K/V to F16, but from slightly different values
            tol = (3e-3 if f16_cache else 2e-5) * scale
            assert np.max(np.abs(logits - ref[p])) < tol, (p, f16_cache)


def test_whole_pass_zero_blocks_closed_form():
    """With Wo = Wdown = 0 the residual stream stays the embedding row, so the
    logits are Wout . RMSNorm(embd) (tied and untied)."""
    import synth
    cfg = synth.ModelConfig("tiny-zero", n_layers=3, dim=32, n_heads=4, n_kv_heads=1, head_dim=8, ffn_dim=64,
                            vocab=40, max_seq=8, eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=oracle.F32,
                            tied=True, number=97)
    for tied in (True, False):
        T = synth.make_weights(cfg.scaled(tied=tied))
        for L in T.layers:
            L["wo"] = np.zeros_like(L["wo"])
            L["w_down"] = np.zeros_like(L["w_down"])
        m = oracle.OracleModel(cfg, T)
        for p, tok in enumerate((3, 17, 39)):
            x = T.tok_embd.reshape(cfg.vocab, cfg.dim)[tok].astype(np.float64)
            h = x / math.sqrt(np.mean(x * x) + cfg.eps) * T.output_norm
            W = (T.output if T.output is not None else T.tok_embd).reshape(cfg.vocab, cfg.dim).astype(np.float64)
            assert np.max(np.abs(m.forward(tok, p) - W @ h)) < 1e-5


def test_prefill_equals_token_by_token_bitwise():
    import synth
    cfg = synth.ModelConfig("tiny-prefill", n_layers=2, dim=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96,
                            vocab=50, max_seq=32, eps=1e-5, rope_base=1e6, rope_neox=1, wtype=oracle.F16,
                            tied=True, bias=True, number=98)
    T = synth.make_weights(cfg)
    toks = synth.prompt(cfg, 12)
    a, b = oracle.OracleModel(cfg, T), oracle.OracleModel(cfg, T)
    la = a.prefill(toks[:7], 0)
    la = a.prefill(toks[7:], 7)
    for p, t in enumerate(toks):
        lb = b.forward(int(t), p)
    assert np.array_equal(la.view(np.uint32), lb.view(np.uint32))
    for l in range(cfg.n_layers):
        for w in (0, 1):
            assert np.array_equal(a.kv(l, w)[:12], b.kv(l, w)[:12])


def test_embedding_lookup_printed_example_pins_java_random():
    g = golden("forward_pass_java_ex3_embedding.json")
    r = JavaRandom(g["seed"])
    emb = np.array([np.float32(java_round(r.next_gaussian() * 100)) / np.float32(100)
                    for _ in range(g["dim"] * g["vocab"])], np.float32)
    for tok, row in g["lookups"].items():
        got = oracle.dequant_row(emb, oracle.F32, int(tok), g["dim"])
        assert [repr(float(v)) for v in got] == [repr(float(np.float32(v))) for v in row]


def test_forward_rejects_out_of_range():
    import synth
    cfg = synth.ModelConfig("tiny-range", n_layers=1, dim=32, n_heads=2, n_kv_heads=1, head_dim=16, ffn_dim=32,
                            vocab=10, max_seq=4, eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=oracle.F32,
                            tied=True, number=99)
    m = oracle.OracleModel(cfg, synth.make_weights(cfg))
    with pytest.raises(IndexError):
        m.forward(10, 0)
    with pytest.raises(IndexError):
        m.forward(0, 4)
