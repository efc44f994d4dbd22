"""The decode step's matrix-vector products, run by the step's own device code
(llm_test_gemv: activation staging, Q8_0 digit records, the shared-memory
weight ring, the row reduction) on crafted input vectors, against float64
products element by element.

Q8_0 bound ("What a Llama model computes, and why" §8 names ggml's 8-bit
activations; this library's reading keeps far more): every 32-element block of
the input is taken as integers X = round(x * 2^e), e chosen from the block's
largest |x| (biased exponent be: e = 148 - be, clamped to [-126, 126], 126 for
zero or subnormal maxima), so each element is off by at most 2^-(e+1); the
block's dot with the int8 quants is then exact, and the float work after it
(the digit sums combined, the two scale products, the reduction over the row's
blocks) rounds a few times, each by at most 2^-24 of its operands.  F16 / F32
weights: plain float products and sums, bounded by the usual float dot
bound."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import llama_decode_forward_gb300 as L
    return L


def q8_blocks(raw: np.ndarray, rows: int, cols: int):
    b = raw.reshape(rows, cols // 32, 34)
    d = b[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    q = b[:, :, 2:].copy().view(np.int8).astype(np.float64)
    return d, q


def dense(raw, wtype, rows, cols) -> np.ndarray:
    if wtype == synth.Q8_0:
        d, q = q8_blocks(raw, rows, cols)
        return (d[:, :, None] * q).reshape(rows, cols)
    if wtype == synth.F16:
        return raw.view(np.float16).astype(np.float64).reshape(rows, cols)
    return raw.astype(np.float64).reshape(rows, cols)


def block_exponent(x: np.ndarray) -> np.ndarray:
    """The kernel's e per 32-element block (x float32, length % 32 == 0)."""
    m = np.abs(x.reshape(-1, 32)).max(axis=1).astype(np.float32)
    be = (m.view(np.uint32) >> 23) & 0xFF
    e = np.clip(148 - be.astype(np.int64), -126, 126)
    return np.where(be == 0, 126, e)


def bound(raw, wtype, rows, cols, x) -> np.ndarray:
    """Largest allowed |gpu - exact| per row."""
    x64 = x.astype(np.float64)
    if wtype == synth.Q8_0:
        d, q = q8_blocks(raw, rows, cols)
        delta = np.ldexp(1.0, -(block_exponent(x) + 1))                     # per block
        act = (np.abs(d) * (np.abs(q).sum(axis=2) * delta[None, :])).sum(axis=1)
        mag = (np.abs(d)[:, :, None] * np.abs(q) * np.abs(x64).reshape(1, -1, 32)).sum(axis=(1, 2))
        return act + 16 * 2.0 ** -24 * mag + 1e-30
    W = dense(raw, wtype, rows, cols)
    return 64 * 2.0 ** -24 * (np.abs(W) @ np.abs(x64)) + 1e-30


def crafted(n: int, seed: int) -> np.ndarray:
    """Blocks of 32: random normal, one large among tiny ones, all zero,
    float subnormals, mixed magnitudes; cycled over the vector."""
    rng = np.random.default_rng(seed)
    out = np.empty(n, np.float32)
    for b in range(n // 32):
        kind = b % 6
        if kind == 0:
            v = rng.standard_normal(32)
        elif kind == 1:
            v = rng.standard_normal(32) * 1e-6
            v[rng.integers(32)] = 900.0 * (1 if b % 2 else -1)
        elif kind == 2:
            v = np.zeros(32)
        elif kind == 3:
            v = rng.standard_normal(32) * 1e-40                            # float subnormals
        elif kind == 4:
            v = rng.standard_normal(32) * 10.0 ** rng.integers(-4, 4, 32)
        else:
            v = rng.standard_normal(32) * 1e-3
            v[::7] = 0.0
        out[32 * b:32 * b + 32] = v
    return out


def matrices(cfg, W):
    """(which, raw bytes, rows, cols, grouped) of the five products."""
    d, q, kv, f = cfg.dim, cfg.q_dim, cfg.kv_dim, cfg.ffn_dim
    L = W.layers[0]
    qkv = np.concatenate([L["wq"].ravel(), L["wk"].ravel(), L["wv"].ravel()])
    es = {synth.F32: 4, synth.F16: 2, synth.Q8_0: 34}[cfg.wtype]
    unit = 32 if cfg.wtype == synth.Q8_0 else 1
    g = L["w_gate"].ravel().view(np.uint8).reshape(f, d // unit * es)
    u = L["w_up"].ravel().view(np.uint8).reshape(f, d // unit * es)
    gu = np.stack([g, u], axis=1).reshape(-1).view(L["w_gate"].dtype)
    out = W.output if W.output is not None else W.tok_embd
    return [(0, qkv, q + 2 * kv, d, False), (1, L["wo"], d, q, True), (2, gu, 2 * f, d, False),
            (3, L["w_down"], d, f, True), (4, out, cfg.vocab, d, False)]


def run_products(lib, cfg, seed):
    import torch
    W = synth.make_weights(cfg)
    if cfg.wtype == synth.Q8_0:
        # a few scales set to FP16 subnormals and to zero
        blocks = W.layers[0]["wq"].reshape(-1, 34)
        for i, s in enumerate((0x0001, 0x0003, 0x03ff, 0x8002, 0x0000)):
            blocks[7 * i + 1, 0], blocks[7 * i + 1, 1] = s & 0xFF, s >> 8
    dec = lib.Decoder(cfg, W)
    G = lib.llm_column_groups(dec.h)
    assert G >= 1 and cfg.n_kv_heads % G == 0
    worst = 0.0
    for which, raw, rows, cols, grouped in matrices(cfg, W):
        x = crafted(cols, seed + which)
        xd = torch.from_numpy(x).cuda()
        yd = torch.full((G * rows if grouped else rows,), float("nan"), dtype=torch.float32, device="cuda")
        lib.llm_test_gemv(dec.h, which, 0, xd, yd)
        y = yd.cpu().numpy().astype(np.float64)
        if grouped:
            y = y.reshape(G, rows)
            c = cols // G
            for g in range(G):
                xs = x[g * c:(g + 1) * c]
                if cfg.wtype == synth.Q8_0:
                    sub = raw.reshape(rows, cols // 32, 34)[:, g * c // 32:(g + 1) * c // 32].reshape(-1)
                else:
                    sub = raw.reshape(rows, cols)[:, g * c:(g + 1) * c].reshape(-1)
                exact = dense(sub, cfg.wtype, rows, c) @ xs.astype(np.float64)
                lim = bound(sub, cfg.wtype, rows, c, xs)
                err = np.abs(y[g] - exact)
                assert np.all(np.isfinite(y[g])), (which, g)
                assert np.all(err <= lim), (which, g, int(np.argmax(err - lim)), float(np.max(err / lim)))
                worst = max(worst, float(np.max(err / lim)))
        else:
            exact = dense(raw, cfg.wtype, rows, cols) @ x.astype(np.float64)
            lim = bound(raw, cfg.wtype, rows, cols, x)
            err = np.abs(y - exact)
            assert np.all(np.isfinite(y)), which
            assert np.all(err <= lim), (which, int(np.argmax(err - lim)), float(np.max(err / lim)))
            worst = max(worst, float(np.max(err / lim)))
    dec.close()
    return worst


def test_q8_0_gemv_within_fixed_point_bound(lib):
    """The Llama-3.2-1B shape (one layer, 8 column groups) on Q8_0."""
    cfg = synth.LLAMA1B_Q8.scaled(n_layers=1, vocab=4000, max_seq=64)
    assert run_products(lib, cfg, 11) <= 1.0


def test_q8_0_gemv_far_finer_than_8bit_activations(lib):
    """The reading's point: the 24-bit block fixed point is not ggml's 8-bit
    activation quantization.  On random inputs the kernel's error is three
    orders of magnitude below that of the oracle's llama.cpp-style product
    (activations quantized to Q8_0 blocks), and of the order of a float dot."""
    import torch
    import oracle
    cfg = synth.LLAMA1B_Q8.scaled(n_layers=1, vocab=4000, max_seq=64)
    W = synth.make_weights(cfg)
    dec = lib.Decoder(cfg, W)
    rows, cols = cfg.q_dim + 2 * cfg.kv_dim, cfg.dim
    raw = np.concatenate([W.layers[0]["wq"].ravel(), W.layers[0]["wk"].ravel(), W.layers[0]["wv"].ravel()])
    x = np.random.default_rng(3).standard_normal(cols).astype(np.float32)
    yd = torch.empty(rows, dtype=torch.float32, device="cuda")
    lib.llm_test_gemv(dec.h, 0, 0, torch.from_numpy(x).cuda(), yd)
    exact = dense(raw, synth.Q8_0, rows, cols) @ x.astype(np.float64)
    gpu_err = np.abs(yd.cpu().numpy().astype(np.float64) - exact)
    q8_err = np.abs(oracle.matvec(raw, synth.Q8_0, x, rows, cols, llamacpp=True).astype(np.float64) - exact)
    f32_err = np.abs(oracle.matvec(raw, synth.Q8_0, x, rows, cols).astype(np.float64) - exact)
    assert np.median(gpu_err) * 1000 < np.median(q8_err)
    assert np.median(gpu_err) < 8 * np.median(f32_err) + 1e-12
    dec.close()


@pytest.mark.parametrize("wtype", [synth.F16, synth.F32])
def test_float_gemv_within_dot_bound(lib, wtype):
    cfg = synth.ModelConfig("gemv_float", n_layers=1, dim=512, n_heads=8, n_kv_heads=4, head_dim=64, ffn_dim=1536,
                            vocab=3000, max_seq=32, eps=1e-5, rope_base=10000.0, rope_neox=0, wtype=wtype, tied=False,
                            number=91)
    assert run_products(lib, cfg, 23) <= 1.0
