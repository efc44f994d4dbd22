"""Pins of the oracle's llama.cpp rounding mode against what the page and the
mathematics fix.

"What a Llama model computes, and why" §8 ("Where llama.cpp rounds") lists
the points where llama.cpp's CPU path rounds and the Java engine does not:
- the activations of a Q8_0 product are quantized to Q8_0 before the integer
  dot;
- F16 weights get F16 activations, and F32 weights keep exact ones;
- q is rounded to F16 before the q.k dots;
- the softmax probabilities are rounded to F16 before they weight V.

The Q8_0 quantizer is the one "Loading GGUF with the FFM API" Example 8
prints. test_oracle_pins.py pins it, the dequantizer, the plain product and
the plain attention. The checks here use only those pinned primitives, exact
rational arithmetic, numpy's IEEE F16 conversion and float64 evaluation.
test_pins_catch_mutant plants mistakes in a copy of the oracle and requires
that one of these pins fails.
"""
import os
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

U = 2.0 ** -24            # unit roundoff of binary32
F32, F16, Q8 = oracle.F32, oracle.F16, oracle.Q8_0


def _bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def _q8_rows(rng, rows, cols, edge_scales=False):
    """Q8_0 weight rows: quants in [-127, 127] and F16 scales near 0.01
    (optionally also zero, subnormal and large scales)."""
    nb = cols // 32
    q = rng.integers(-127, 128, (rows, nb, 32)).astype(np.int8)
    d = (rng.standard_normal((rows, nb)) * 0.01).astype(np.float16)
    if edge_scales:
        flat = d.reshape(-1)
        special = np.array([0x0000, 0x0001, 0x03ff, 0x0400, 0x5bff, 0x8001, 0xbc00], np.uint16).view(np.float16)
        flat[:special.size] = special
    blk = np.zeros((rows, nb, 34), np.uint8)
    blk[:, :, 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    blk[:, :, 2:] = q.view(np.uint8)
    return blk.reshape(-1)


def _exact_block_terms(w, x, rows, cols):
    """Exact d_w*d_x*sum_j(qw_j*qx_j) per block and row, from the dequantized
    weight row and the dequantized Q8_0 activations.  Every dequantized value
    d*q is exact in float, so the sum of their exact products is the block's
    exact integer dot times both scales."""
    xd = oracle.dequant_row(oracle.quantize_q8_0(x), Q8, 0, cols)
    fx = [Fraction(float(v)) for v in xd]
    out = []
    for r in range(rows):
        wd = oracle.dequant_row(w, Q8, r, cols)
        out.append([sum(Fraction(float(wd[j])) * fx[j] for j in range(32 * b, 32 * b + 32))
                    for b in range(cols // 32)])
    return out


# ------------------------------------------------------------- Q8_0 product --
def test_q8_block_term_is_its_exact_value_rounded_once():
    """One block per row: no float sum, so the result is the exact integer dot
    times both scales rounded once to float (the value has at most 42
    significant bits, so float64 holds it exactly before that rounding)."""
    rng = np.random.default_rng(11)
    rows, cols = 96, 32
    w = _q8_rows(rng, rows, cols, edge_scales=True)
    for x in (rng.standard_normal(cols).astype(np.float32),
              (rng.standard_normal(cols) * 1e-3).astype(np.float32),
              np.zeros(cols, np.float32)):
        got = oracle.matvec(w, Q8, x, rows, cols, llamacpp=True)
        want = np.array([np.float32(float(t[0])) for t in _exact_block_terms(w, x, rows, cols)], np.float32)
        assert np.array_equal(_bits(got), _bits(want))


def test_q8_rows_sum_block_terms_within_the_float_bound():
    """Several blocks: the result is within the float summation bound of the
    exact sum of the block terms; the product with unquantized activations is
    far outside it, so the bound tells the two apart."""
    rng = np.random.default_rng(12)
    rows, cols = 16, 256
    nb = cols // 32
    w = _q8_rows(rng, rows, cols)
    x = rng.standard_normal(cols).astype(np.float32)
    got = oracle.matvec(w, Q8, x, rows, cols, llamacpp=True)
    plain = oracle.matvec(w, Q8, x, rows, cols)
    far = 0
    for r, terms in enumerate(_exact_block_terms(w, x, rows, cols)):
        exact = sum(terms)
        bound = Fraction((nb + 1) * U) * sum(abs(t) for t in terms)
        assert abs(Fraction(float(got[r])) - exact) <= bound, r
        far += abs(Fraction(float(plain[r])) - exact) > 10 * bound
    assert far == rows


def test_q8_activations_on_the_grid_are_not_changed():
    """Activations that are already k * 2^-5 with |k| <= 127 and a +-127 in
    every block quantize exactly (d = 2^-5), so the quantized product equals
    the exact product of the given values within the float bound."""
    rng = np.random.default_rng(13)
    rows, cols = 8, 128
    k = rng.integers(-127, 128, cols)
    k[::32] = 127
    x = (k * 2.0 ** -5).astype(np.float32)
    assert np.array_equal(oracle.dequant_row(oracle.quantize_q8_0(x), Q8, 0, cols), x)
    w = _q8_rows(rng, rows, cols)
    got = oracle.matvec(w, Q8, x, rows, cols, llamacpp=True)
    for r in range(rows):
        prods = [Fraction(float(a)) * Fraction(float(b)) for a, b in zip(oracle.dequant_row(w, Q8, r, cols), x)]
        bound = Fraction((cols // 32 + 1) * U) * sum(abs(p) for p in prods)
        assert abs(Fraction(float(got[r])) - sum(prods)) <= bound


# -------------------------------------------------------- F32 / F16 products --
def test_f32_weights_keep_exact_activations():
    rng = np.random.default_rng(14)
    rows, cols = 12, 80
    w = rng.standard_normal(rows * cols).astype(np.float32)
    x = rng.standard_normal(cols).astype(np.float32)
    assert np.array_equal(_bits(oracle.matvec(w, F32, x, rows, cols, llamacpp=True)),
                          _bits(oracle.matvec(w, F32, x, rows, cols)))


def test_f16_weights_get_f16_rounded_activations():
    """F16 weights: the product of the F16-rounded activations (numpy's IEEE
    conversion); activations that are already F16 values are unchanged."""
    rng = np.random.default_rng(15)
    rows, cols = 12, 80
    w = rng.standard_normal(rows * cols).astype(np.float16)
    x = rng.standard_normal(cols).astype(np.float32)
    xr = x.astype(np.float16).astype(np.float32)
    got = oracle.matvec(w, F16, x, rows, cols, llamacpp=True)
    assert np.array_equal(_bits(got), _bits(oracle.matvec(w, F16, xr, rows, cols)))
    assert not np.array_equal(_bits(got), _bits(oracle.matvec(w, F16, x, rows, cols)))
    assert np.array_equal(_bits(oracle.matvec(w, F16, xr, rows, cols, llamacpp=True)),
                          _bits(oracle.matvec(w, F16, xr, rows, cols)))
    # and within the float bound of the exact product of the rounded values
    for r in range(rows):
        prods = [Fraction(float(a)) * Fraction(float(b)) for a, b in zip(w[r * cols:(r + 1) * cols], xr)]
        bound = Fraction((cols + 1) * U) * sum(abs(p) for p in prods)
        assert abs(Fraction(float(got[r])) - sum(prods)) <= bound


# ---------------------------------------------------------------- attention --
def test_attention_one_position_returns_v():
    """pos 0: one probability, exactly 1 (an F16 value), so every head returns
    its KV head's V row whatever q is (grouped heads: h / (n_heads/n_kv))."""
    rng = np.random.default_rng(16)
    nh, nkv, hd = 8, 2, 16
    q = rng.standard_normal(nh * hd).astype(np.float32)
    k = rng.standard_normal(nkv * hd).astype(np.float16).astype(np.float32)
    v = rng.standard_normal(nkv * hd).astype(np.float16).astype(np.float32)
    out = oracle.attention(q, k, v, nh, nkv, hd, 0, llamacpp=True).reshape(nh, hd)
    for h in range(nh):
        g = h // (nh // nkv)
        assert np.array_equal(_bits(out[h]), _bits(v[g * hd:(g + 1) * hd]))


@pytest.mark.parametrize("n", [2, 3, 4, 5, 7])
def test_attention_uniform_probabilities_are_f16(n):
    """q = 0: every score is 0, every probability is 1/n computed in float and
    rounded to F16.  With small-integer V each product and sum is exact, so
    the output is that F16 probability times the column sums of V exactly.
    For n = 3, 5, 7 this differs from the unrounded 1/n."""
    rng = np.random.default_rng(20 + n)
    nh, nkv, hd = 2, 1, 8
    k = rng.standard_normal((n, hd)).astype(np.float16).astype(np.float32)
    v = rng.integers(-8, 9, (n, hd)).astype(np.float32)
    q = np.zeros(nh * hd, np.float32)
    p = np.float16(np.float32(1.0) / np.float32(n))
    got = oracle.attention(q, k, v, nh, nkv, hd, n - 1, llamacpp=True).reshape(nh, hd)
    want = np.array([np.float32(float(Fraction(float(p)) * int(c))) for c in v.sum(axis=0)], np.float32)
    for h in range(nh):
        assert np.array_equal(_bits(got[h]), _bits(want))
    plain = oracle.attention(q, k, v, nh, nkv, hd, n - 1).reshape(nh, hd)
    assert np.array_equal(_bits(plain[0]), _bits(want)) == (n in (2, 4))


def _two_position_probs(q0, q1, a):
    """float64 softmax of the scores (q0*a/2, q1*a/2) (head_dim 4, one-hot K
    rows with value a), each probability then rounded to F16; None when a
    probability lies too close to an F16 rounding midpoint for the float32
    route to be sure of the same rounding."""
    s = np.array([q0 * a / 2.0, q1 * a / 2.0])
    e = np.exp(s - s.max())
    p = e / e.sum()
    r = p.astype(np.float16)
    for pv in p:
        lo = np.float16(pv)
        ulp = float(np.spacing(lo))
        frac = (pv - float(lo)) / ulp
        if abs(abs(frac) - 0.5) < 1e-3:
            return None
    return r


def test_attention_rounds_q_to_f16():
    """One-hot K rows make each score q_t * a / 2 exactly and one-hot V rows
    return the two probabilities, so the output is f16(softmax(f16(q) a/2)).
    Cases are drawn until the F16 probabilities with rounded q differ from
    those with exact q, so that the pin tells the two apart."""
    rng = np.random.default_rng(17)
    hd, a = 4, np.float32(64.0)
    k = np.zeros((2, hd), np.float32)
    k[0, 0] = k[1, 1] = a
    v = np.zeros((2, hd), np.float32)
    v[0, 2] = v[1, 3] = 1.0
    checked = 0
    for _ in range(400):
        q0, q1 = np.float32(rng.uniform(-0.3, 0.3)), np.float32(rng.uniform(-0.3, 0.3))
        rq = _two_position_probs(float(np.float16(q0)), float(np.float16(q1)), float(a))
        raw = _two_position_probs(float(q0), float(q1), float(a))
        if rq is None or raw is None or np.array_equal(rq, raw):
            continue
        q = np.array([q0, q1, 0, 0], np.float32)
        got = oracle.attention(q, k, v, 1, 1, hd, 1, llamacpp=True)
        assert got[0] == 0 and got[1] == 0
        assert np.array_equal(_bits(got[2:]), _bits(rq.astype(np.float32)))
        checked += 1
        if checked == 8:
            break
    assert checked == 8


def test_attention_within_bound_of_float64_with_the_rounding_points():
    """Random GQA case: the output against a float64 evaluation with the same
    two rounding points (f16(q); f16 of each float64 probability), allowing
    for a probability that the float32 route rounds to the neighbouring F16
    value (one F16 ulp of that probability times |V|)."""
    rng = np.random.default_rng(18)
    nh, nkv, hd, pos = 8, 2, 32, 40
    q = rng.standard_normal(nh * hd).astype(np.float32)
    k = rng.standard_normal(((pos + 1), nkv * hd)).astype(np.float16).astype(np.float32)
    v = rng.standard_normal(((pos + 1), nkv * hd)).astype(np.float16).astype(np.float32)
    got = oracle.attention(q, k, v, nh, nkv, hd, pos, llamacpp=True).reshape(nh, hd)
    plain = oracle.attention(q, k, v, nh, nkv, hd, pos).reshape(nh, hd)
    qr = q.astype(np.float16).astype(np.float64).reshape(nh, hd)
    differs = 0
    for h in range(nh):
        g = h // (nh // nkv)
        kk, vv = k[:, g * hd:(g + 1) * hd].astype(np.float64), v[:, g * hd:(g + 1) * hd].astype(np.float64)
        s = kk @ qr[h] / np.sqrt(hd)
        e = np.exp(s - s.max())
        p = (e / e.sum()).astype(np.float16).astype(np.float64)
        want = p @ vv
        slack = np.abs(vv).T @ np.spacing(p.astype(np.float16)).astype(np.float64) + 1e-5 * np.abs(want) + 1e-7
        assert np.all(np.abs(got[h] - want) <= slack), h
        differs += not np.array_equal(_bits(got[h]), _bits(plain[h]))
    assert differs == nh


# -------------------------------------------------------------- whole pass --
def _cfg(wtype, number, **kw):
    base = dict(n_layers=2, dim=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96, vocab=50, max_seq=16,
                eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=wtype, tied=False)
    base.update(kw)
    return synth.ModelConfig(f"llamacpp-{wtype}", number=number, **base)


def test_f32_model_first_position_is_unchanged():
    """F32 weights keep exact activations and one position has probability 1,
    so at pos 0 every traced step of the pass equals the plain one bitwise;
    from pos 1 on, the attention rounding changes the logits."""
    cfg = _cfg(F32, 140)
    T = synth.make_weights(cfg)
    toks = [int(t) for t in synth.prompt(cfg, 4)]
    a = oracle.OracleModel(cfg, T)
    b = oracle.OracleModel(cfg, T, llamacpp_rounding=True)
    ta, tb = [], []
    a.set_trace(lambda n, l, v: ta.append((n, l, v)))
    b.set_trace(lambda n, l, v: tb.append((n, l, v)))
    la, lb = a.forward(toks[0], 0), b.forward(toks[0], 0)
    assert np.array_equal(_bits(la), _bits(lb))
    assert [(n, l) for n, l, _ in ta] == [(n, l) for n, l, _ in tb]
    assert all(np.array_equal(_bits(x), _bits(y)) for (_, _, x), (_, _, y) in zip(ta, tb))
    later = [not np.array_equal(_bits(a.forward(t, p)), _bits(b.forward(t, p))) for p, t in enumerate(toks[1:], 1)]
    assert all(later)


@pytest.mark.parametrize("wtype,bias", [(Q8, False), (F16, True)])
def test_every_product_of_the_pass_rounds(wtype, bias):
    """With the mode on, each traced product of the pass is the rounded
    product of its traced input, q/k are the rounded products after bias and
    RoPE, and the attention output is the rounded attention over the cache:
    the mode reaches every matrix product, including the logits, and the
    attention of every layer."""
    cfg = _cfg(wtype, 141 + wtype, bias=bias, tied=(wtype == Q8), rope_neox=int(wtype == F16))
    T = synth.make_weights(cfg)
    m = oracle.OracleModel(cfg, T, llamacpp_rounding=True)
    d, hd, nh, nkv, ff = cfg.dim, cfg.head_dim, cfg.n_heads, cfg.n_kv_heads, cfg.ffn_dim
    toks = [int(t) for t in synth.prompt(cfg, 5)]
    for p, t in enumerate(toks):
        tr = {}
        m.set_trace(lambda n, l, v: tr.__setitem__((n, l), v))
        logits = m.forward(t, p)
        mv = lambda w, x, rows, cols: oracle.matvec(w, wtype, x, rows, cols, llamacpp=True)
        for l, L in enumerate(T.layers):
            h = tr["attn_norm", l]
            def proj(w, b, rows):
                y = mv(w, h, rows, d)
                return y if b is None else (y + np.asarray(b, np.float32)).astype(np.float32)
            qv = oracle.rope(proj(L["wq"], L.get("bq"), nh * hd), nh, hd, cfg.rope_dims, p, cfg.rope_base,
                             cfg.rope_neox)
            kv = oracle.rope(proj(L["wk"], L.get("bk"), nkv * hd), nkv, hd, cfg.rope_dims, p, cfg.rope_base,
                             cfg.rope_neox)
            assert np.array_equal(_bits(tr["Qcur", l]), _bits(qv))
            assert np.array_equal(_bits(tr["Kcur", l]), _bits(kv))
            assert np.array_equal(_bits(tr["Vcur", l]), _bits(proj(L["wv"], L.get("bv"), nkv * hd)))
            att = oracle.attention(tr["Qcur", l], m.kv(l, 0)[:p + 1], m.kv(l, 1)[:p + 1], nh, nkv, hd, p,
                                   llamacpp=True)
            assert np.array_equal(_bits(tr["kqv_out", l]), _bits(att))
            assert np.array_equal(_bits(tr["attn_out", l]), _bits(mv(L["wo"], tr["kqv_out", l], d, nh * hd)))
            assert np.array_equal(_bits(tr["ffn_gate", l]), _bits(mv(L["w_gate"], tr["ffn_norm", l], ff, d)))
            assert np.array_equal(_bits(tr["ffn_up", l]), _bits(mv(L["w_up"], tr["ffn_norm", l], ff, d)))
            assert np.array_equal(_bits(tr["ffn_out", l]), _bits(mv(L["w_down"], tr["ffn_swiglu", l], d, ff)))
        wout = T.output if T.output is not None else T.tok_embd
        assert np.array_equal(_bits(logits), _bits(mv(wout, tr["result_norm", -1], cfg.vocab, d)))


# ---------------------------------------------------------------- mutations --
SRC = os.path.join(os.path.dirname(oracle.__file__), "llm_oracle.c")

MUTANTS = {
    "q8_x_scale_dropped": ("float dd = dw * dx;", "float dd = dw;"),
    "q8_two_roundings": ("float c = (float)sumi * dd;", "float c = ((float)sumi * dw) * dx;"),
    "q8_x_block_fixed": ("*xb = xq + (size_t)b * 34;", "*xb = xq;"),
    "q8_x_quants_unsigned": ("sumi += (int)(int8_t)wb[2 + j] * (int)(int8_t)xb[2 + j];",
                             "sumi += (int)(int8_t)wb[2 + j] * (int)xb[2 + j];"),
    "f16_x_not_rounded": ("for (int i = 0; i < cols; i++) xr[i] = round_f16(x[i]);",
                          "for (int i = 0; i < cols; i++) xr[i] = x[i];"),
    "q_not_rounded": ("qh[i] = llamacpp ? round_f16(q[h * head_dim + i]) : q[h * head_dim + i];",
                      "qh[i] = q[h * head_dim + i];"),
    "p_not_rounded": ("if (llamacpp) a = round_f16(a);", ""),
    "p_rounded_before_division": ("float a = att[t] / sum;\n            if (llamacpp) a = round_f16(a);",
                                  "float a = (llamacpp ? round_f16(att[t]) : att[t]) / sum;"),
    "model_products_plain": ("if (m->c.llamacpp_rounding) orc_matvec_llamacpp(", "if (0) orc_matvec_llamacpp("),
    "model_attention_plain": ("hd, pos, c->llamacpp_rounding);", "hd, pos, 0);"),
}

DETECTORS = [
    test_q8_block_term_is_its_exact_value_rounded_once,
    test_q8_rows_sum_block_terms_within_the_float_bound,
    test_f16_weights_get_f16_rounded_activations,
    test_attention_rounds_q_to_f16,
    lambda: test_attention_uniform_probabilities_are_f16(3),
    test_attention_within_bound_of_float64_with_the_rounding_points,
    test_f32_model_first_position_is_unchanged,
    lambda: test_every_product_of_the_pass_rounds(Q8, False),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    with open(SRC) as f:
        source = f.read()
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation anchor for {name} not unique"
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "mutant.c")
        with open(src, "w") as f:
            f.write(source.replace(old, new))
        so = os.path.join(d, "libmutant.so")
        subprocess.check_call(["gcc", *oracle.CFLAGS, f"-I{os.path.dirname(SRC)}", "-o", so, src, "-lm"])
        monkeypatch.setattr(oracle, "_LIB", oracle.load(so))
        caught = 0
        for det in DETECTORS:
            try:
                det()
            except AssertionError:
                caught += 1
        assert caught > 0, f"no pin catches the mutant {name}"
