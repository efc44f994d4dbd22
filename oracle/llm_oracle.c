/*
 * CPU oracle for the batch-1 Llama decode forward pass (test infrastructure).
 * See llm_oracle.h for the scope, the sources and who may use it.
 *
 * Build: gcc -std=c11 -O2 -fno-fast-math -ffp-contract=off -fPIC -shared
 * (no fused multiply-add, no reassociation: every float operation below is one
 * IEEE-754 binary32 operation in program order).
 */
#include "llm_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <stdio.h>

/* ------------------------------------------------------------------ F16 --
 * "Loading GGUF with the FFM API", Example 7: FP16 has 1 sign bit, 5 exponent
 * bits (bias 15) and 10 fraction bits; conversion to FP16 rounds to the
 * nearest representable value, ties to even, as ggml does.  Subnormals are
 * kept; values at or beyond the overflow threshold become infinity. */
float orc_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    float v;
    if (e == 0) v = ldexpf((float)f, -24);                        /* zero / subnormal: f * 2^-24 */
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexpf((float)(1024 + f), e - 25);                   /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

uint16_t orc_f32_to_f16(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return sign | 0x7e00u;                   /* NaN */
    if (a >= 0x477ff000u) return sign | 0x7c00u;                  /* >= 65520 (halfway to 2^16): inf */
    if (a >= 0x38800000u) {                                       /* normal FP16 range, >= 2^-14 */
        uint32_t e = (a >> 23) - 127 + 15, mant = a & 0x7fffffu;
        uint32_t h = (e << 10) | (mant >> 13), rem = mant & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h++;  /* a carry into the exponent is right */
        return sign | (uint16_t)h;
    }
    if (a <= 0x33000000u) return sign;                            /* <= 2^-25: rounds to zero (tie to even) */
    /* FP16 subnormal: count units of 2^-24.  a = m * 2^(E-23) with E in [-25,-15]. */
    int E = (int)(a >> 23) - 127;
    uint32_t m = (a & 0x7fffffu) | 0x800000u;
    int s = -E - 1;                                               /* 14..24 */
    uint32_t q = m >> s, rem = m & ((1u << s) - 1u), half = 1u << (s - 1);
    if (rem > half || (rem == half && (q & 1u))) q++;
    return sign | (uint16_t)q;
}

/* --------------------------------------------------------- weight decode --
 * "The Forward Pass in Java", Example 2 and "Loading GGUF with the FFM API",
 * Examples 7-8: F32 is copied, F16 is widened per value, and a Q8_0 block of
 * 34 bytes (little-endian FP16 scale d, then 32 signed bytes qs) decodes to
 * d * qs[j] in float.  Element i of a row lies in block i/32 at quant i%32. */
void orc_dequant_row(const void *w, int wtype, int64_t row, int cols, float *out) {
    if (wtype == ORC_F32) {
        memcpy(out, (const float *)w + row * (int64_t)cols, sizeof(float) * (size_t)cols);
    } else if (wtype == ORC_F16) {
        const uint8_t *p = (const uint8_t *)w + row * (int64_t)cols * 2;
        for (int i = 0; i < cols; i++) out[i] = orc_f16_to_f32((uint16_t)(p[2 * i] | (p[2 * i + 1] << 8)));
    } else {                                                      /* Q8_0 */
        const uint8_t *p = (const uint8_t *)w + row * (int64_t)(cols / 32) * 34;
        for (int b = 0; b < cols / 32; b++) {
            const uint8_t *blk = p + (size_t)b * 34;
            float d = orc_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
            for (int j = 0; j < 32; j++) out[b * 32 + j] = d * (float)(int8_t)blk[2 + j];
        }
    }
}

/* The reference quantizer of "The Forward Pass in Java", Example 2 (and
 * "Loading GGUF with the FFM API", Example 8): per 32 values d = amax/127 is
 * stored as FP16 and qs = round-half-away-from-zero(x / d).  Test utility. */
void orc_quantize_q8_0(const float *x, int64_t n, uint8_t *out) {
    for (int64_t b = 0; b < n / 32; b++) {
        float amax = 0.0f;
        for (int j = 0; j < 32; j++) { float a = fabsf(x[b * 32 + j]); if (a > amax) amax = a; }
        float d = amax / 127.0f, id = d != 0.0f ? 1.0f / d : 0.0f;
        uint16_t dh = orc_f32_to_f16(d);
        uint8_t *blk = out + b * 34;
        blk[0] = (uint8_t)(dh & 0xff);
        blk[1] = (uint8_t)(dh >> 8);
        for (int j = 0; j < 32; j++) {
            float v = x[b * 32 + j] * id;
            double r = floor(fabs((double)v) + 0.5);
            blk[2 + j] = (uint8_t)(int8_t)(int)(v < 0 ? -r : r);
        }
    }
}

/* ------------------------------------------------------------- RMSNorm --
 * "The Forward Pass in Java", Example 4: y[i] = x[i] / sqrt(mean(x^2)+eps) *
 * g[i], the sum of squares accumulated in double as ggml does; the scale is
 * rounded to float, then x[i]*scale and *g[i] are float products. */
void orc_rmsnorm(float *out, const float *x, const float *g, int n, float eps) {
    double ss = 0.0;
    for (int i = 0; i < n; i++) ss += (double)x[i] * (double)x[i];
    float scale = (float)(1.0 / sqrt(ss / (double)n + (double)eps));
    for (int i = 0; i < n; i++) {
        float t = x[i] * scale;
        out[i] = t * g[i];
    }
}

/* ------------------------------------------------------------- threads --
 * Off by default (1).  With n > 1 the rows of each matrix product and the
 * heads of attention are split over n threads; every output element is still
 * computed by one thread in the same order, so results do not change. */
static int orc_threads_ = 1;

void orc_set_threads(int n) { orc_threads_ = n > 1 ? n : 1; }

/* ---------------------------------------------------------------- GEMV --
 * "The Forward Pass in Java", Example 5: out[r] = sum_i W[r*cols+i] * x[i],
 * a GGUF tensor with dims [cols, rows] storing row r at r*cols; the sum runs
 * in float from i = 0.  Rows are decoded one at a time (decoding is exact, so
 * this equals decoding the whole tensor first). */
void orc_matvec(float *out, const void *w, int wtype, const float *x, int rows, int cols) {
#pragma omp parallel num_threads(orc_threads_) if (orc_threads_ > 1)
    {
        float *row = (float *)malloc(sizeof(float) * (size_t)cols);
#pragma omp for schedule(static)
        for (int r = 0; r < rows; r++) {
            const float *wr;
            if (wtype == ORC_F32) wr = (const float *)w + (int64_t)r * cols;
            else { orc_dequant_row(w, wtype, r, cols, row); wr = row; }
            float s = 0.0f;
            for (int i = 0; i < cols; i++) { float p = wr[i] * x[i]; s = s + p; }
            out[r] = s;
        }
        free(row);
    }
}

/* ---------------------------------------------------------------- RoPE --
 * "The Forward Pass in Java", Example 6 with "What a Llama model computes,
 * and why" §2.4: pair i of each head turns by theta_i = pos * base^(-2i/n_rot)
 * / f_i.  As in ggml's rope cache, theta_scale = base^(-2/n_rot) is computed
 * once and theta is advanced by a float multiply per pair; the frequency
 * divisor is applied to the chain's value.  Normal layout pairs (2i, 2i+1),
 * NEOX pairs (i, i + n_rot/2).  Dims >= n_rot are left unchanged. */
void orc_rope(float *vec, int n_heads, int head_dim, int rope_dims, int pos, float base,
              int neox, const float *freqs) {
    float theta_scale = (float)pow((double)base, -2.0 / (double)rope_dims);
    for (int h = 0; h < n_heads; h++) {
        float theta = (float)pos;
        for (int i = 0; i < rope_dims / 2; i++) {
            float th = freqs ? theta / freqs[i] : theta;
            float c = (float)cos((double)th), s = (float)sin((double)th);
            int a = h * head_dim + (neox ? i : 2 * i);
            int b = neox ? a + rope_dims / 2 : a + 1;
            float x0 = vec[a], x1 = vec[b];
            float p0 = x0 * c, p1 = x1 * s, p2 = x0 * s, p3 = x1 * c;
            vec[a] = p0 - p1;
            vec[b] = p2 + p3;
            theta = theta * theta_scale;
        }
    }
}

/* ---------------------------------------------------------------- SiLU --
 * "The Forward Pass in Java", Example 8: silu(z) = z / (1 + e^-z), with the
 * exponential taken in double and rounded to float. */
float orc_silu(float z) {
    float e = (float)exp((double)(-z));
    float den = 1.0f + e;
    return z / den;
}

/* ----------------------------------------------------------- attention --
 * "The Forward Pass in Java", Example 7 and the Llama class: query head h
 * reads KV head h / (n_heads/n_kv_heads); s_t = (q . K_t) / sqrt(hd) for
 * t = 0..pos; softmax with the maximum subtracted (exp in double, rounded to
 * float; the sum in float); out = sum_t (e_t/sum) * V_t accumulated over t in
 * ascending order.  Rows after pos are never read (causality).
 * With `llamacpp` set, the two rounding points of "What a Llama model
 * computes, and why" §8 are added: ggml's F16 matrix products convert their
 * F32 operand, so q is rounded to F16 before the q.k dots (K is F16) and each
 * probability e_t/sum is rounded to F16 before it weights V (V is F16). */
static float round_f16(float v) { return orc_f16_to_f32(orc_f32_to_f16(v)); }

static void attention(float *out, const float *q, const float *kcache, const float *vcache,
                      int n_heads, int n_kv_heads, int head_dim, int pos, int llamacpp) {
    int kv_dim = n_kv_heads * head_dim, group = n_heads / n_kv_heads;
    float sq = (float)sqrt((double)head_dim);
    for (int i = 0; i < n_heads * head_dim; i++) out[i] = 0.0f;
#pragma omp parallel num_threads(orc_threads_) if (orc_threads_ > 1)
    {
    float *att = (float *)malloc(sizeof(float) * (size_t)(pos + 1));
    float *qh = (float *)malloc(sizeof(float) * (size_t)head_dim);
#pragma omp for schedule(static)
    for (int h = 0; h < n_heads; h++) {
        int kv_off = (h / group) * head_dim;
        for (int i = 0; i < head_dim; i++) qh[i] = llamacpp ? round_f16(q[h * head_dim + i]) : q[h * head_dim + i];
        float mx = -INFINITY;
        for (int t = 0; t <= pos; t++) {
            const float *kt = kcache + (int64_t)t * kv_dim + kv_off;
            float s = 0.0f;
            for (int i = 0; i < head_dim; i++) { float p = qh[i] * kt[i]; s = s + p; }
            att[t] = s / sq;
            if (att[t] > mx) mx = att[t];
        }
        float sum = 0.0f;
        for (int t = 0; t <= pos; t++) { att[t] = (float)exp((double)(att[t] - mx)); sum = sum + att[t]; }
        float *oh = out + h * head_dim;
        for (int t = 0; t <= pos; t++) {
            float a = att[t] / sum;
            if (llamacpp) a = round_f16(a);
            const float *vt = vcache + (int64_t)t * kv_dim + kv_off;
            for (int i = 0; i < head_dim; i++) { float p = a * vt[i]; oh[i] = oh[i] + p; }
        }
    }
    free(qh);
    free(att);
    }
}

void orc_attention(float *out, const float *q, const float *kcache, const float *vcache,
                   int n_heads, int n_kv_heads, int head_dim, int pos) {
    attention(out, q, kcache, vcache, n_heads, n_kv_heads, head_dim, pos, 0);
}

void orc_attention_llamacpp(float *out, const float *q, const float *kcache, const float *vcache,
                            int n_heads, int n_kv_heads, int head_dim, int pos) {
    attention(out, q, kcache, vcache, n_heads, n_kv_heads, head_dim, pos, 1);
}

/* ------------------------------------------- GEMV with llama.cpp rounding --
 * "What a Llama model computes, and why" §8: ggml converts the activations of
 * a matrix product to the weight's vector-dot format first.  F32 weights keep
 * F32 activations (the plain product).  F16 weights get F16-rounded
 * activations (round to nearest even); each product of two F16 values is
 * exact in float, and the sum runs in float from i = 0.  Q8_0 weights get the
 * activations quantized to Q8_0 blocks by the reference quantizer; block b of
 * row r then contributes its integer dot sumi = sum_j qw[j]*qx[j] (exact in
 * int) times d_w*d_x (a product of two F16 values, exact in float), so each
 * block's term is its exact value rounded once to float; the terms are summed
 * in float from block 0.  The pages fix the rounding points, not this order
 * of the float operations: it is the plainest reading of "the integer dot". */
void orc_matvec_llamacpp(float *out, const void *w, int wtype, const float *x, int rows, int cols) {
    if (wtype == ORC_F32) {
        orc_matvec(out, w, wtype, x, rows, cols);
        return;
    }
    if (wtype == ORC_F16) {
        float *xr = (float *)malloc(sizeof(float) * (size_t)cols);
        for (int i = 0; i < cols; i++) xr[i] = round_f16(x[i]);
        orc_matvec(out, w, wtype, xr, rows, cols);
        free(xr);
        return;
    }
    int nb = cols / 32;
    uint8_t *xq = (uint8_t *)malloc((size_t)nb * 34);
    orc_quantize_q8_0(x, cols, xq);
    for (int r = 0; r < rows; r++) {
        const uint8_t *wr = (const uint8_t *)w + (int64_t)r * nb * 34;
        float s = 0.0f;
        for (int b = 0; b < nb; b++) {
            const uint8_t *wb = wr + (size_t)b * 34, *xb = xq + (size_t)b * 34;
            int sumi = 0;
            for (int j = 0; j < 32; j++) sumi += (int)(int8_t)wb[2 + j] * (int)(int8_t)xb[2 + j];
            float dw = orc_f16_to_f32((uint16_t)(wb[0] | (wb[1] << 8)));
            float dx = orc_f16_to_f32((uint16_t)(xb[0] | (xb[1] << 8)));
            float dd = dw * dx;
            float c = (float)sumi * dd;
            s = s + c;
        }
        out[r] = s;
    }
    free(xq);
}

/* -------------------------------------------------------------- argmax --
 * "The Forward Pass in Java", Example 9: the first index whose value is
 * strictly greater than every value before it (llama.cpp's temp-0 rule). */
int orc_argmax(const float *v, int n) {
    int best = 0;
    for (int i = 1; i < n; i++) if (v[i] > v[best]) best = i;
    return best;
}

/* --------------------------------------------------------------- model -- */
struct orc_model {
    orc_config c;
    orc_weights w;
    orc_layer *layers;
    float **kcache, **vcache;            /* per layer: max_seq * kv_dim */
    orc_trace_fn trace;
    void *trace_user;
};

static size_t wbytes_per_row(int wtype, int cols) {
    if (wtype == ORC_F32) return (size_t)cols * 4;
    if (wtype == ORC_F16) return (size_t)cols * 2;
    return (size_t)(cols / 32) * 34;
}

orc_model *orc_create(const orc_config *cfg, const orc_weights *w) {
    if (!cfg || !w || !w->tok_embd || !w->output_norm || !w->layers) return NULL;
    const orc_config *c = cfg;
    if (c->n_layers <= 0 || c->dim <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
        c->ffn_dim <= 0 || c->vocab <= 0 || c->max_seq <= 0) return NULL;
    if (c->n_heads % c->n_kv_heads != 0 || c->n_heads * c->head_dim != c->dim) return NULL;
    if (c->rope_dims <= 0 || c->rope_dims % 2 || c->rope_dims > c->head_dim) return NULL;
    if (c->wtype != ORC_F32 && c->wtype != ORC_F16 && c->wtype != ORC_Q8_0) return NULL;
    if (c->wtype == ORC_Q8_0 && (c->dim % 32 || c->ffn_dim % 32)) return NULL;
    orc_model *m = (orc_model *)calloc(1, sizeof(orc_model));
    m->c = *c;
    m->w = *w;
    m->layers = (orc_layer *)malloc(sizeof(orc_layer) * (size_t)c->n_layers);
    memcpy(m->layers, w->layers, sizeof(orc_layer) * (size_t)c->n_layers);
    m->w.layers = m->layers;
    size_t kv = (size_t)c->max_seq * (size_t)(c->n_kv_heads * c->head_dim);
    m->kcache = (float **)calloc((size_t)c->n_layers, sizeof(float *));
    m->vcache = (float **)calloc((size_t)c->n_layers, sizeof(float *));
    for (int l = 0; l < c->n_layers; l++) {
        m->kcache[l] = (float *)calloc(kv, sizeof(float));
        m->vcache[l] = (float *)calloc(kv, sizeof(float));
        if (!m->kcache[l] || !m->vcache[l]) { orc_destroy(m); return NULL; }
    }
    (void)wbytes_per_row;
    return m;
}

void orc_destroy(orc_model *m) {
    if (!m) return;
    for (int l = 0; l < m->c.n_layers; l++) {
        if (m->kcache) free(m->kcache[l]);
        if (m->vcache) free(m->vcache[l]);
    }
    free(m->kcache);
    free(m->vcache);
    free(m->layers);
    free(m);
}

void orc_set_trace(orc_model *m, orc_trace_fn fn, void *user) { m->trace = fn; m->trace_user = user; }

float *orc_kv(orc_model *m, int layer, int which) {
    if (!m || layer < 0 || layer >= m->c.n_layers) return NULL;
    return which ? m->vcache[layer] : m->kcache[layer];
}

static void trace(orc_model *m, const char *name, int layer, const float *v, int n) {
    if (m->trace) m->trace(name, layer, v, n, m->trace_user);
}

/* Every matrix product of the pass, with or without the llama.cpp rounding. */
static void mv(const orc_model *m, float *out, const void *w, const float *x, int rows, int cols) {
    if (m->c.llamacpp_rounding) orc_matvec_llamacpp(out, w, m->c.wtype, x, rows, cols);
    else orc_matvec(out, w, m->c.wtype, x, rows, cols);
}

static void add_bias(float *x, const float *b, int n) {
    if (b) for (int i = 0; i < n; i++) x[i] = x[i] + b[i];
}

/* "The Forward Pass in Java", Example 10: the stored value is the F16
 * round trip of v when the cache is F16. */
static float store(const orc_model *m, float v) {
    return m->c.f16_cache ? orc_f16_to_f32(orc_f32_to_f16(v)) : v;
}

/* "The Forward Pass in Java", Example 13, Llama.forward: one token at
 * position pos.  Embedding lookup; per layer RMSNorm, Q/K/V (+ biases),
 * RoPE on q and k, K/V stored at row pos, attention, output projection and
 * residual, RMSNorm, SwiGLU and residual; final RMSNorm and the logits
 * (output.weight or, when absent, token_embd.weight: Example 9).  With
 * llamacpp_rounding every matrix product and the attention round as
 * llama.cpp does ("What a Llama model computes, and why" §8); the embedding
 * row is decoded exactly either way. */
int orc_forward(orc_model *m, int token, int pos, float *logits) {
    const orc_config *c = &m->c;
    if (token < 0 || token >= c->vocab || pos < 0 || pos >= c->max_seq) return -1;
    int dim = c->dim, hd = c->head_dim, qdim = c->n_heads * hd, kv_dim = c->n_kv_heads * hd;
    float *x = (float *)malloc(sizeof(float) * (size_t)dim);
    float *xb = (float *)malloc(sizeof(float) * (size_t)dim);
    float *q = (float *)malloc(sizeof(float) * (size_t)qdim);
    float *k = (float *)malloc(sizeof(float) * (size_t)kv_dim);
    float *v = (float *)malloc(sizeof(float) * (size_t)kv_dim);
    float *heads = (float *)malloc(sizeof(float) * (size_t)qdim);
    float *hb = (float *)malloc(sizeof(float) * (size_t)c->ffn_dim);
    float *hb2 = (float *)malloc(sizeof(float) * (size_t)c->ffn_dim);

    orc_dequant_row(m->w.tok_embd, c->wtype, token, dim, x);
    trace(m, "embd", -1, x, dim);
    for (int l = 0; l < c->n_layers; l++) {
        const orc_layer *L = &m->layers[l];
        orc_rmsnorm(xb, x, L->attn_norm, dim, c->eps);
        trace(m, "attn_norm", l, xb, dim);
        mv(m, q, L->wq, xb, qdim, dim);
        mv(m, k, L->wk, xb, kv_dim, dim);
        mv(m, v, L->wv, xb, kv_dim, dim);
        add_bias(q, L->bq, qdim);
        add_bias(k, L->bk, kv_dim);
        add_bias(v, L->bv, kv_dim);
        orc_rope(q, c->n_heads, hd, c->rope_dims, pos, c->rope_base, c->rope_neox, m->w.rope_freqs);
        orc_rope(k, c->n_kv_heads, hd, c->rope_dims, pos, c->rope_base, c->rope_neox, m->w.rope_freqs);
        trace(m, "Qcur", l, q, qdim);
        trace(m, "Kcur", l, k, kv_dim);
        trace(m, "Vcur", l, v, kv_dim);
        float *kc = m->kcache[l], *vc = m->vcache[l];
        for (int i = 0; i < kv_dim; i++) {
            kc[(int64_t)pos * kv_dim + i] = store(m, k[i]);
            vc[(int64_t)pos * kv_dim + i] = store(m, v[i]);
        }
        attention(heads, q, kc, vc, c->n_heads, c->n_kv_heads, hd, pos, c->llamacpp_rounding);
        trace(m, "kqv_out", l, heads, qdim);
        mv(m, xb, L->wo, heads, dim, qdim);
        trace(m, "attn_out", l, xb, dim);
        for (int i = 0; i < dim; i++) x[i] = x[i] + xb[i];
        trace(m, "ffn_inp", l, x, dim);
        orc_rmsnorm(xb, x, L->ffn_norm, dim, c->eps);
        trace(m, "ffn_norm", l, xb, dim);
        mv(m, hb, L->w_gate, xb, c->ffn_dim, dim);
        mv(m, hb2, L->w_up, xb, c->ffn_dim, dim);
        trace(m, "ffn_gate", l, hb, c->ffn_dim);
        trace(m, "ffn_up", l, hb2, c->ffn_dim);
        for (int i = 0; i < c->ffn_dim; i++) hb[i] = orc_silu(hb[i]) * hb2[i];
        trace(m, "ffn_swiglu", l, hb, c->ffn_dim);
        mv(m, xb, L->w_down, hb, dim, c->ffn_dim);
        trace(m, "ffn_out", l, xb, dim);
        for (int i = 0; i < dim; i++) x[i] = x[i] + xb[i];
        trace(m, "l_out", l, x, dim);
    }
    orc_rmsnorm(xb, x, m->w.output_norm, dim, c->eps);
    trace(m, "result_norm", -1, xb, dim);
    mv(m, logits, m->w.output ? m->w.output : m->w.tok_embd, xb, c->vocab, dim);
    trace(m, "result_output", -1, logits, c->vocab);

    free(x); free(xb); free(q); free(k); free(v); free(heads); free(hb); free(hb2);
    return 0;
}

/* "What a Llama model computes, and why" §4: token i of a prompt batch sits
 * at pos0+i and attends to rows 0..pos0+i; only the last token's logits are
 * returned.  Run token by token, which the page states gives the same logits
 * and cache by construction. */
int orc_prefill(orc_model *m, const int32_t *tokens, int n, int pos0, float *logits) {
    if (n <= 0 || pos0 < 0 || pos0 + n > m->c.max_seq) return -1;
    for (int i = 0; i < n; i++)
        if (orc_forward(m, tokens[i], pos0 + i, logits) != 0) return -1;
    return 0;
}
