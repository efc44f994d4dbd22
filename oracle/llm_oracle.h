/*
 * CPU oracle for the batch-1 Llama decode forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow C evaluation (single
 * threaded unless orc_set_threads says otherwise) of what the GPU library computes, written from the method's
 * definition so that the CUDA path can be checked against it.  Only the test
 * suite, the package smoke check and the benchmark's CPU-baseline leg may load
 * it.  It shares no code, header, table or helper with the CUDA library.
 *
 * Source of every step: "The Forward Pass in Java" (codeloopback.dev,
 * llm-forward-pass), Example 13 (the Llama class, method `forward`), with the
 * per-step specialisations cited beside each function in llm_oracle.c:
 *   - Example 2 / "Loading GGUF with the FFM API" Examples 7-8: weight decoding
 *   - Example 4: RMSNorm with a double-precision sum of squares
 *   - Example 5: matrix-vector product in GGUF dimension order
 *   - Example 6: RoPE, normal and NEOX pair layouts, float angle chain
 *   - Example 7: grouped-query attention over the KV cache
 *   - Example 8: SwiGLU; Example 9: logits, tied embeddings, argmax
 *   - Example 10: F16 KV cache (round to nearest even)
 *   - "What a Llama model computes, and why" §2.4: per-pair frequency factors
 *   - "What a Llama model computes, and why" §4: prefill equals token-by-token
 *   - "What a Llama model computes, and why" §8 ("Where llama.cpp rounds"):
 *     the optional llama.cpp rounding points (Q8_0 activations of a Q8_0
 *     product, F16 activations of an F16 product, q and the softmax
 *     probabilities rounded to F16 in attention)
 *
 * Arithmetic: F32 storage and F32 operations, left to right, no fused
 * multiply-add (compiled with -ffp-contract=off), double only where the pages
 * use it (RMSNorm sum, sqrt, exp, cos, sin, pow).
 *
 * Parity pins: every exported function is pinned by tests under tests/
 * (printed worked examples of the pages, closed forms, invariants, and the
 * pages' end-to-end self-test whose generated token ids are printed).
 */
#ifndef LLM_ORACLE_H
#define LLM_ORACLE_H

#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ggml type ids ("Loading GGUF with the FFM API", tensor-info types). */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_Q8_0 = 8 };

typedef struct {
    int n_layers, dim, n_heads, n_kv_heads, head_dim, ffn_dim, vocab, max_seq, rope_dims;
    float eps, rope_base;
    int rope_neox;   /* 0: pairs (2i, 2i+1); 1: pairs (i, i + rope_dims/2) */
    int wtype;       /* ORC_F32 / ORC_F16 / ORC_Q8_0 for every matrix incl. the embedding */
    int f16_cache;   /* 1: K/V rounded through F16 before storing (the pages' f16Cache flag) */
    int llamacpp_rounding;  /* 1: round where llama.cpp's CPU path rounds (orc_matvec_llamacpp,
                               orc_attention_llamacpp); 0: the Java engine's float arithmetic */
} orc_config;

/* Host pointers in GGUF layout: a [in -> out] matrix is `out` rows of `in`
 * values (or in/32 Q8_0 blocks of 34 bytes).  Norm gains and biases are F32.
 * Biases may be NULL.  The oracle never copies or frees them. */
typedef struct {
    const float *attn_norm, *ffn_norm, *bq, *bk, *bv;
    const void *wq, *wk, *wv, *wo, *w_gate, *w_up, *w_down;
} orc_layer;

typedef struct {
    const void *tok_embd;      /* [vocab][dim] */
    const float *output_norm;  /* [dim] */
    const void *output;        /* [vocab][dim] or NULL: tied to tok_embd */
    const float *rope_freqs;   /* [rope_dims/2] divisors or NULL: all 1 */
    const orc_layer *layers;   /* [n_layers] */
} orc_weights;

typedef struct orc_model orc_model;

/* Trace hook: called after each named step with llama.cpp's tensor names
 * (embd, attn_norm-l, Qcur-l, Kcur-l, Vcur-l, kqv_out-l, attn_out-l, ffn_inp-l,
 * ffn_norm-l, ffn_gate-l, ffn_up-l, ffn_swiglu-l, ffn_out-l, l_out-l,
 * result_norm, result_output).  `layer` is -1 outside the layer loop. */
typedef void (*orc_trace_fn)(const char *name, int layer, const float *v, int n, void *user);

/* ---- threads ----
 * 1 (the default): everything on the calling thread.  n > 1: the rows of
 * every matrix product and the heads of attention are split over n OpenMP
 * threads; each output element is still computed by one thread in the same
 * order, so every result is bitwise the single-thread one. */
void orc_set_threads(int n);

/* ---- model ---- */
orc_model *orc_create(const orc_config *cfg, const orc_weights *w);  /* NULL on bad config */
void orc_destroy(orc_model *m);
void orc_set_trace(orc_model *m, orc_trace_fn fn, void *user);
/* One token at `pos`: writes K/V row `pos` of every layer and the logits
 * (vocab floats).  Returns 0, or -1 when token/pos is out of range. */
int orc_forward(orc_model *m, int token, int pos, float *logits);
/* Token-by-token prefill of tokens[0..n) at pos0..pos0+n-1; logits of the last. */
int orc_prefill(orc_model *m, const int32_t *tokens, int n, int pos0, float *logits);
/* The KV cache of one layer: [max_seq][n_kv_heads][head_dim] floats holding the
 * stored values (F16-representable when f16_cache).  which: 0 = K, 1 = V. */
float *orc_kv(orc_model *m, int layer, int which);

/* ---- primitives (exported so that each can be pinned on its own) ---- */
float orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_f16(float f);
void orc_dequant_row(const void *w, int wtype, int64_t row, int cols, float *out);
void orc_quantize_q8_0(const float *x, int64_t n, uint8_t *out);   /* test utility */
void orc_rmsnorm(float *out, const float *x, const float *g, int n, float eps);
void orc_matvec(float *out, const void *w, int wtype, const float *x, int rows, int cols);
void orc_rope(float *vec, int n_heads, int head_dim, int rope_dims, int pos, float base,
              int neox, const float *freqs);
float orc_silu(float z);
/* All query heads of one position over cached rows 0..pos (K/V rows of
 * kv_dim = n_kv_heads*head_dim floats).  out: n_heads*head_dim floats. */
void orc_attention(float *out, const float *q, const float *kcache, const float *vcache,
                   int n_heads, int n_kv_heads, int head_dim, int pos);
int orc_argmax(const float *v, int n);

/* ---- llama.cpp rounding points ("What a Llama model computes, and why" §8) ----
 * orc_matvec_llamacpp: as orc_matvec, with the activations rounded as ggml
 * rounds them for the weight type: unchanged for F32, rounded to F16 for F16,
 * quantized to Q8_0 blocks (orc_quantize_q8_0) for Q8_0, whose product is
 * then the integer dot of the two blocks' quants times both scales.
 * orc_attention_llamacpp: as orc_attention, with q rounded to F16 before the
 * q.k dots and each probability e_t/sum rounded to F16 before it weights V. */
void orc_matvec_llamacpp(float *out, const void *w, int wtype, const float *x, int rows, int cols);
void orc_attention_llamacpp(float *out, const float *q, const float *kcache, const float *vcache,
                            int n_heads, int n_kv_heads, int head_dim, int pos);

#ifdef __cplusplus
}
#endif
#endif
