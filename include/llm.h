/*
 * llm.h — C ABI of libllmdecode: batch-1 decode forward pass of a Llama-family
 * model on one NVIDIA GB300 (sm_103a), plus a tensor-core batched prefill.
 *
 * What the calls compute is the forward pass of "The Forward Pass in Java"
 * (codeloopback.dev, llm-forward-pass), Example 13 (`Llama.forward`): embedding
 * lookup, per layer RMSNorm, Q/K/V projections (+ optional biases), RoPE on q
 * and k (normal or NEOX pairs), K/V appended to an F16 cache at row `pos`,
 * grouped-query attention over rows 0..pos, output projection + residual,
 * RMSNorm, SwiGLU feed-forward + residual; then the final RMSNorm, the logits
 * product (tied to the embedding when there is no output matrix) and the greedy
 * argmax of Example 9.  "What a Llama model computes, and why" (branes-ai
 * synapse) §2 gives the same steps with Llama-3.2-1B shapes, §2.4 the per-pair
 * frequency factors and §4 the batched prefill.
 *
 * Conventions for every call:
 *   - Return value: LLM_OK (0) or a negative llm_status.  On failure nothing is
 *     enqueued unless the status says so, and llm_last_error(h) holds a one-line
 *     reason.  No call aborts or prints.
 *   - Pointers documented as "device" must point to memory of the current CUDA
 *     device; "host" pointers to ordinary (pageable or pinned) host memory.
 *   - A handle is not thread-safe: one host thread drives a handle at a time.
 *   - All device work of a handle is enqueued on the stream given at creation.
 *     "Synchronous" calls wait for that stream before returning.
 */
#ifndef LLM_H
#define LLM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL means the legacy default stream. */
typedef struct CUstream_st *llm_stream_t;

/* Weight storage types, numbered as ggml's type ids ("Loading GGUF with the
 * FFM API", tensor types F32 = 0, F16 = 1, Q8_0 = 8). */
typedef enum { LLM_F32 = 0, LLM_F16 = 1, LLM_Q8_0 = 8 } llm_dtype;

typedef enum {
    LLM_OK = 0,
    LLM_ERR_INVALID_ARG = -1,     /* NULL pointer, inconsistent shape, bad config field */
    LLM_ERR_UNSUPPORTED = -2,     /* a valid model this build does not handle (dtype, head size, ...) */
    LLM_ERR_OUT_OF_RANGE = -3,    /* token not in [0, vocab), pos not in [0, max_seq), pos0+n > max_seq */
    LLM_ERR_CUDA = -4,            /* a CUDA runtime call failed; llm_last_error has its message */
    LLM_ERR_NO_MEMORY = -5,       /* device allocation failed */
    LLM_ERR_DEVICE_TIMEOUT = -6,  /* a bounded wait inside a kernel gave up; the step's outputs are invalid */
    LLM_ERR_STATE = -7,           /* call not valid in the handle's state (e.g. after a device error) */
    LLM_ERR_NONFINITE = -8,       /* a residual-stream update was NaN, infinite or not below 2^15 in
                                     magnitude (the decode step's fixed-point accumulators); the step's
                                     outputs are invalid and the handle needs llm_reset */
    LLM_ERR_CHECK = -9            /* libraries built with LLM_CHECKED only: a device-side index check of
                                     the decode step failed and the access it guarded was skipped; the
                                     step's outputs are invalid and the handle needs llm_reset */
} llm_status;

/* Rounding of the decode step ("What a Llama model computes, and why" §8).
 * LLM_NUMERICS_EXACT: every matrix product takes its F32 input vector as it
 * is (Q8_0 rows meet the activations as 24-bit block fixed point, about what
 * an F32 sum keeps), and attention's q and probabilities stay F32.
 * LLM_NUMERICS_LLAMACPP: llama.cpp's rounding points.  A Q8_0 product first
 * quantizes its input to Q8_0 blocks (d = amax/127 stored as F16, each
 * element x/d rounded half away from zero) and sums the blocks' integer dots
 * times d_w*d_x; an F16 product rounds its input to F16; attention rounds q
 * to F16 and each probability e_t/sum to F16 after the normaliser over all
 * positions (so the step streams the K rows twice).  RMSNorm's scale is
 * applied before the rounding ((x * scale) * g).  llm_prefill is not
 * affected by this field.  Slower than EXACT; meant for comparing with
 * llama.cpp's outputs. */
typedef enum { LLM_NUMERICS_EXACT = 0, LLM_NUMERICS_LLAMACPP = 1 } llm_numerics;

/* Model shape ("The Forward Pass in Java", Example 1, Config record).
 * head_dim * n_heads must equal dim; n_heads must be a multiple of n_kv_heads;
 * rope_dims is even and <= head_dim (dims beyond it are not rotated);
 * head_dim is a multiple of 8 and at most 256.  For LLM_Q8_0, dim and ffn_dim
 * are multiples of 32; for LLM_F16, multiples of 8; for LLM_F32, of 4.
 * max_seq is the number of KV-cache rows the handle allocates. */
typedef struct {
    int n_layers, dim, n_heads, n_kv_heads, head_dim, ffn_dim, vocab, max_seq, rope_dims;
    float eps;          /* RMSNorm epsilon */
    float rope_base;    /* RoPE frequency base */
    int rope_neox;      /* 0: pairs (2i, 2i+1) (llama); 1: pairs (i, i + rope_dims/2) (qwen2) */
    int wtype;          /* llm_dtype of every matrix, the embedding and the output */
    int numerics;       /* llm_numerics of the decode step (0, the zero-initialised default: exact) */
} llm_config;

/* One layer's tensors, all DEVICE pointers in GGUF layout ("The Forward Pass
 * in Java", Example 5): a [in -> out] matrix is `out` rows of `in` values
 * (F32/F16) or of in/32 Q8_0 blocks of 34 bytes (FP16 scale, 32 int8), row r
 * at r * row_bytes — the same bytes as a PyTorch [out, in] tensor.
 * attn_norm / ffn_norm: F32 [dim].  bq [n_heads*head_dim], bk / bv
 * [n_kv_heads*head_dim]: F32 or NULL (no bias).  wq [dim -> n_heads*head_dim],
 * wk / wv [dim -> n_kv_heads*head_dim], wo [n_heads*head_dim -> dim],
 * w_gate / w_up [dim -> ffn_dim], w_down [ffn_dim -> dim]. */
typedef struct {
    const float *attn_norm, *ffn_norm, *bq, *bk, *bv;
    const void *wq, *wk, *wv, *wo, *w_gate, *w_up, *w_down;
} llm_layer_weights;

/* tok_embd: [dim -> vocab] in wtype (DEVICE).  output_norm: F32 [dim] (DEVICE).
 * output: [dim -> vocab] in wtype, or NULL for tied embeddings ("The Forward
 * Pass in Java", Example 9).  rope_freqs: F32 [rope_dims/2] per-pair divisors
 * of the angle ("What a Llama model computes, and why" §2.4), or NULL for 1.
 * layers: HOST array of n_layers records. */
typedef struct {
    const void *tok_embd;
    const float *output_norm;
    const void *output;
    const float *rope_freqs;
    const llm_layer_weights *layers;
} llm_weights;

typedef struct llm_handle llm_handle;

/* Creates a handle: validates the config, copies every tensor once into the
 * library's own device layout (Q8_0 split into 16-byte aligned int8 quants and
 * FP16 scales; Q/K/V rows and gate/up rows fused), allocates the F16 KV cache
 * [n_layers][2][max_seq][n_kv_heads][head_dim] and the activations.  The
 * caller's weight buffers are only read during this call.  Synchronous.
 * Errors: INVALID_ARG, UNSUPPORTED, NO_MEMORY, CUDA; *out is set to NULL then,
 * and llm_last_error(NULL) gives the reason. */
int llm_create(const llm_config *cfg, const llm_weights *w, llm_stream_t stream, llm_handle **out);

/* Starts a new sequence (P4 "The Engine": Attention.reset).  Logical only: the
 * cache is not cleared; rows are overwritten as positions are decoded.  Also
 * clears a sticky device error.  Synchronous. */
int llm_reset(llm_handle *h);

/* One decode step, synchronous, HOST in/out: token at position `pos`.  Writes
 * K/V row `pos` of every layer, attends over rows 0..pos (rows 0..pos-1 must
 * hold this sequence's K/V, as in Llama.forward), and returns the logits
 * (vocab floats, copied to logits_host when not NULL) and the greedy argmax
 * (first index of the maximum, to argmax_host when not NULL).
 * Errors: OUT_OF_RANGE (token, pos), DEVICE_TIMEOUT, CUDA, STATE. */
int llm_decode_step(llm_handle *h, int32_t token, int32_t pos, float *logits_host, int32_t *argmax_host);

/* The same step enqueued without waiting.  The token is read on the device
 * from token_dev (so it can be the previous step's argmax); the argmax is
 * written to argmax_dev (DEVICE, may equal token_dev + 1 etc.); the logits stay
 * in the handle's buffer (llm_logits_device).  pos is range-checked on the
 * host; the token is clamped on the device and an out-of-range token sets the
 * handle's device error (reported by llm_sync as OUT_OF_RANGE). */
int llm_decode_step_async(llm_handle *h, const int32_t *token_dev, int32_t pos, int32_t *argmax_dev);

/* Greedy generation with device-side feedback ("The Forward Pass in Java",
 * Example 12 loop, without the end-of-generation check): n_steps steps at
 * positions pos..pos+n_steps-1; step 0 consumes `token`, step i > 0 consumes
 * tokens_dev[i-1]; step i writes its argmax to tokens_dev[i] (DEVICE, n_steps
 * int32).  Enqueued without waiting; no host round trip between steps. */
int llm_generate(llm_handle *h, int32_t token, int32_t pos, int32_t n_steps, int32_t *tokens_dev);

/* Batched prefill of tokens_host[0..n) at positions pos0..pos0+n-1 ("What a
 * Llama model computes, and why" §4): every K/V row is written and token i
 * attends to rows 0..pos0+i; only the last token's logits are produced (to
 * logits_host when not NULL; argmax to argmax_host when not NULL).  F16 and
 * Q8_0 weights run the projections as tensor-core GEMMs on F16 operands (a
 * Q8_0 matrix is expanded to F16, d*q rounded to nearest even, just before its
 * GEMM) when dim, n_heads*head_dim and ffn_dim are multiples of 64; otherwise,
 * and for F32 weights, the decode step runs token by token.  Synchronous.
 * Errors: OUT_OF_RANGE, INVALID_ARG, CUDA. */
int llm_prefill(llm_handle *h, const int32_t *tokens_host, int32_t n, int32_t pos0,
                float *logits_host, int32_t *argmax_host);

/* enable != 0: gives a Q8_0 handle an F16 copy of its layer matrices (QKV, O,
 * gate/up, down), each value d*q rounded to nearest even: the values the
 * batched prefill's GEMMs otherwise expand from the quants tile by tile.
 * Later llm_prefill calls read the copy instead, with the same results bit
 * for bit and the GEMMs at the speed of F16 weights; the decode step still
 * streams the Q8_0 matrices.  Costs 2 bytes of device memory per layer
 * weight (about 2 GB for a 1B model); enabling twice keeps one copy.
 * enable == 0 frees the copy (waiting for the handle's stream first).
 * Asynchronous on the handle's stream.  Errors: UNSUPPORTED for F16 or F32
 * weights or a model whose prefill runs token by token, NO_MEMORY (nothing
 * kept), CUDA. */
int llm_prefill_f16_copy(llm_handle *h, int enable);

/* Waits for the handle's stream and reports a device-side error of the
 * enqueued steps (DEVICE_TIMEOUT, OUT_OF_RANGE) or CUDA. */
int llm_sync(llm_handle *h);

/* DEVICE pointer to the handle's logits buffer (vocab floats): the logits of
 * the latest llm_decode_step / llm_decode_step_async / llm_generate /
 * llm_prefill on the handle; llm_decode_step_noalloc writes the caller's
 * buffer instead and leaves this one untouched.  Valid until the next step on
 * the handle and the handle's destruction. */
const float *llm_logits_device(const llm_handle *h);

/* The handle's model shape (the llm_config it was created with; for a handle
 * from llm_create_from_gguf, the shape read from the file), copied to *out.
 * Host only, no device work.  Errors: INVALID_ARG (NULL). */
int llm_get_config(const llm_handle *h, llm_config *out);

/* Test hook: DEVICE pointers to layer `layer`'s K and V cache,
 * [max_seq][n_kv_heads][head_dim] FP16 each ("The Forward Pass in Java",
 * Example 7: element pos*kv_dim + kv_head*head_dim + i).  Writable, so a
 * harness can pre-fill rows of a long context. */
int llm_kv_view(llm_handle *h, int layer, uint16_t **k_dev, uint16_t **v_dev);

/* Test hook: runs the device KV store on given values — k_dev / v_dev are
 * DEVICE F32 vectors of n_kv_heads*head_dim already rotated — writing row `pos`
 * of layer `layer` exactly as the decode step does (FP16, round to nearest
 * even; "The Forward Pass in Java", Example 10).  Synchronous. */
int llm_test_kv_store(llm_handle *h, int layer, int32_t pos, const float *k_dev, const float *v_dev);

/* Test hook: decodes rows [row0, row0+n_rows) of one weight matrix from the
 * library's own layout with the same device routine the matrix-vector kernels
 * use, into out_dev (DEVICE, n_rows*cols F32).  which: 0 wq, 1 wk, 2 wv, 3 wo,
 * 4 w_gate, 5 w_up, 6 w_down (of `layer`), 7 tok_embd, 8 output.  Synchronous. */
int llm_test_dequant_rows(llm_handle *h, int which, int layer, int32_t row0, int32_t n_rows, float *out_dev);

/* Test hook: one matrix-vector product of the decode step on a given input,
 * run by the step's own device code (activation staging — for Q8_0 the
 * per-32-element fixed-point digit records —, the shared-memory weight ring
 * and the row reduction), so that its arithmetic can be checked element by
 * element.  which: 0 [wq;wk;wv] of `layer` (x_dev: dim floats; y_dev:
 * n_heads*head_dim + 2*n_kv_heads*head_dim), 1 wo (x_dev: n_heads*head_dim;
 * y_dev: llm_column_groups(h) * dim floats, group g's partial product over
 * its columns [g*c, (g+1)*c), c = n_heads*head_dim/groups, at g*dim), 2 the
 * interleaved gate/up rows (x_dev: dim; y_dev: 2*ffn_dim, row 2i gate i,
 * row 2i+1 up i), 3 w_down (x_dev: ffn_dim; y_dev: groups * dim, as for wo),
 * 4 the logits matrix (x_dev: dim; y_dev: vocab).  DEVICE F32 buffers.
 * Synchronous.  Errors: INVALID_ARG, OUT_OF_RANGE (layer), STATE, CUDA. */
int llm_test_gemv(llm_handle *h, int which, int layer, const float *x_dev, float *y_dev);

/* Named intermediates of the handle's last llm_decode_step (or
 * llm_decode_step_async / llm_generate step), read back from the buffers the
 * step exchanges them through, for layer-by-layer checks like those of "The
 * Forward Pass in Java", Example 11 (llama.cpp's tensor names):
 *   LLM_DEBUG_Q / _K / _V   q, k, v after their biases, before RoPE
 *                           (n_heads*head_dim / n_kv_heads*head_dim values);
 *                           v is llama.cpp's Vcur
 *   LLM_DEBUG_ATTN_OUT      attn_out: the output projection's update of the
 *                           residual stream (dim values)
 *   LLM_DEBUG_FFN_SWIGLU    ffn_swiglu: silu(gate) * up (ffn_dim values)
 *   LLM_DEBUG_FFN_OUT       ffn_out: the down projection's update (dim)
 * The updates are the decode step's fixed-point sums (2^-32 steps) rounded to
 * float.  host: HOST float[n], n the tensor's length.  Synchronous.
 * Errors: INVALID_ARG (which, NULL, n), OUT_OF_RANGE (layer), STATE when no
 * step ran since create or llm_reset, or the values are not all from the
 * last decode step (llm_prefill and llm_decode_step_noalloc do not write these
 * buffers). */
enum {
    LLM_DEBUG_Q = 0, LLM_DEBUG_K = 1, LLM_DEBUG_V = 2,
    LLM_DEBUG_ATTN_OUT = 3, LLM_DEBUG_FFN_SWIGLU = 4, LLM_DEBUG_FFN_OUT = 5
};
int llm_debug_tensor(llm_handle *h, int layer, int which, float *host, int32_t n);

/* 1 if this library was built with LLM_CHECKED (device-side index checks on
 * the decode step's global writes and weight-stream ranges, reporting
 * LLM_ERR_CHECK instead of trapping), else 0. */
int llm_checked_build(void);

/* Test hook of LLM_CHECKED builds: the index check of the decode step's
 * logits writes accepts only indices below `limit` (0 restores vocab), so a
 * test can see a failing check reported as LLM_ERR_CHECK with the writes past
 * `limit` skipped.  Errors: UNSUPPORTED in other builds, OUT_OF_RANGE. */
int llm_test_logits_limit(llm_handle *h, int32_t limit);

/* Test hook: allocation failure.  The nth device or pinned-host allocation
 * the library makes from now on (in llm_create, llm_create_from_gguf or
 * llm_prefill's workspace) fails as if the device were out of memory, once;
 * 0 disarms.  The failing call returns LLM_ERR_NO_MEMORY and releases what it
 * had allocated.  Process-wide.  Errors: INVALID_ARG for nth < 0. */
int llm_test_fail_alloc(int32_t nth);

/* Test hook: guard bands.  The KV cache, the activation buffer and the
 * prefill workspace are allocated with 4096 bytes more on each side, filled
 * with 0xA5.  Returns how many of those bytes differ from 0xA5 (0: no kernel
 * wrote past either end of these buffers), or a negative status.
 * Synchronous. */
int64_t llm_test_guards(llm_handle *h);

/* Test hook: overwrites the guard byte adjacent to one end of a guarded
 * buffer (band 2b: before buffer b, 2b+1: after it; b = 0 KV cache,
 * 1 activations, 2 prefill workspace once allocated), so that a test can see
 * llm_test_guards report it.  Synchronous.  Errors: OUT_OF_RANGE. */
int llm_test_poke_guard(llm_handle *h, int band);

/* The number of column groups the decode step splits the output and down
 * projections into (a divisor of n_kv_heads), or INVALID_ARG for NULL. */
int llm_column_groups(const llm_handle *h);

/* Phase trace of the last decode step: copies sms * 1024 %globaltimer stamps
 * (nanoseconds, uint64, per CTA: the start and end of every phase of every
 * layer, as laid out in the library's trace table) to `host` (HOST, caller
 * owned).  `sms` receives the CTA count.  Only libraries compiled with
 * LLM_TRACE record stamps; others return LLM_ERR_UNSUPPORTED.  Synchronous. */
int llm_trace_read(llm_handle *h, uint64_t *host, int32_t *sms);

/* One decode step like llm_decode_step_async, but its working memory (the
 * tagged activation vectors and attention partials of every layer, the
 * residual accumulators, the grid counter, argmax and error words) lives in
 * a fixed 16 MiB device array inside the library rather than in buffers of
 * the handle, so the call allocates no memory of any kind.  The described decode pass has no counterpart of this
 * call: it exists for callers that may not allocate device memory while
 * serving (a process whose remaining device memory is owned by its own pool
 * and cannot grow after start-up).
 *   token_dev   DEVICE int32, the input token (read by the kernel).
 *   pos         position of the token, in [0, max_seq).
 *   logits_dev  DEVICE float[vocab], written with the step's logits (the
 *               handle's own logits buffer, llm_logits_device, is untouched).
 *   argmax_dev  DEVICE int32, written with the first index of the max logit.
 * The handle's KV cache row `pos` is written as by llm_decode_step, and the
 * step computes the same bits as llm_decode_step (the same kernel).
 * Synchronous: returns after the step has finished on the handle's stream.
 * Errors: LLM_ERR_INVALID_ARG for NULL pointers, LLM_ERR_OUT_OF_RANGE for a
 * bad pos (or a device-side token out of range, after which the handle needs
 * llm_reset), LLM_ERR_UNSUPPORTED when the model's step needs more than the
 * fixed array holds (the message gives both sizes), LLM_ERR_DEVICE_TIMEOUT
 * if a bounded device wait expired.
 * The first call on a device looks up the array's address; make it before
 * any stream capture starts.  The array is shared by every handle on the
 * device: calls that overlap in time race on it and must be serialised by
 * the caller. */
int llm_decode_step_noalloc(llm_handle *h, const int32_t *token_dev, int32_t pos, float *logits_dev,
                            int32_t *argmax_dev);

/* Number of kernel launches enqueued on the handle's stream so far (all calls). */
int64_t llm_launch_count(const llm_handle *h);

/* Releases every device buffer of the handle (after waiting for its stream).
 * The library keeps a set of the handles llm_create returned and that are
 * not yet destroyed: every call refuses any other pointer with
 * LLM_ERR_INVALID_ARG (llm_logits_device returns NULL, llm_launch_count 0),
 * and llm_destroy of such a pointer (a second destroy, NULL) does nothing.
 * A pointer that a later llm_create happens to return again names that new
 * handle. */
void llm_destroy(llm_handle *h);

const char *llm_status_string(int status);
/* The one-line reason of the handle's last failed call.  With h == NULL: the
 * reason of the calling thread's last failed llm_create, "" after one that
 * succeeded (llm_create_from_gguf reports through its `err` buffer).  The
 * string stays valid until the next call on the handle (with NULL: until this
 * thread's next llm_create). */
const char *llm_last_error(const llm_handle *h);

/* ------------------------------------------------------------ GGUF files --
 * A model file in the GGUF version 3 layout of "Loading GGUF with the FFM API"
 * (codeloopback.dev, llm-gguf-loader-ffm): a 24-byte header (magic "GGUF",
 * version, tensor count, key-value count; Example 3), key-value metadata
 * (Examples 4, 13), tensor infos (name, dims innermost first, ggml type,
 * offset into the data section; Example 5), padding to general.alignment
 * (UINT32, 32 when absent), then the data section with each tensor padded to
 * the alignment.  All numbers little-endian.  Host memory only; none of these
 * calls touches the GPU except llm_create_from_gguf. */
typedef struct llm_gguf llm_gguf;

/* Metadata value types ("Loading GGUF with the FFM API", Example 13). */
typedef enum {
    LLM_GGUF_UINT8 = 0, LLM_GGUF_INT8 = 1, LLM_GGUF_UINT16 = 2, LLM_GGUF_INT16 = 3, LLM_GGUF_UINT32 = 4,
    LLM_GGUF_INT32 = 5, LLM_GGUF_FLOAT32 = 6, LLM_GGUF_BOOL = 7, LLM_GGUF_STRING = 8, LLM_GGUF_ARRAY = 9,
    LLM_GGUF_UINT64 = 10, LLM_GGUF_INT64 = 11, LLM_GGUF_FLOAT64 = 12
} llm_gguf_type;

typedef struct {
    uint32_t version;
    int64_t n_tensors, n_kv;
    uint64_t alignment;      /* general.alignment, or 32 */
    uint64_t infos_end;      /* file byte where the tensor infos end */
    uint64_t data_start;     /* infos_end rounded up to the alignment */
    uint64_t file_size;
} llm_gguf_layout;

typedef struct {
    int32_t type;            /* ggml type: LLM_F32, LLM_F16 or LLM_Q8_0 */
    int32_t n_dims;          /* 1..4 */
    int64_t dims[4];         /* innermost first; unused ones are 1 */
    uint64_t offset;         /* from the start of the data section */
    uint64_t file_offset;    /* data_start + offset */
    uint64_t bytes;          /* F32 4, F16 2 per value, Q8_0 34 per 32-value block */
    const void *data;        /* HOST view into the mapped file, valid until llm_gguf_close */
} llm_gguf_tensor;

/* Opens and maps `path` read-only and checks it in the loader page's order
 * (Example 11): at least the 24-byte header, the magic, version 3, metadata
 * and tensor infos within the file, a nonzero UINT32 general.alignment when
 * present, every tensor of type F32 / F16 / Q8_0 (Q8_0 rows whole 32-value
 * blocks), each tensor's offset equal to the padded sizes of the tensors
 * before it, and each tensor's end within the file.  On success *out owns
 * the mapping (free with llm_gguf_close).  Errors: INVALID_ARG (missing file,
 * failed check; `err`, when not NULL, receives a one-line reason of at most
 * err_len bytes, e.g. "magic 0x4C4D4747 is not GGUF"), UNSUPPORTED (version,
 * tensor type), NO_MEMORY (mapping failed); *out is NULL then. */
int llm_gguf_open(const char *path, llm_gguf **out, char *err, size_t err_len);
void llm_gguf_close(llm_gguf *g);

/* The header counts and the layout of the file (Example 5). */
int llm_gguf_summary(const llm_gguf *g, llm_gguf_layout *s);

/* A tensor by name, or by index in file order (name: HOST string owned by g).
 * Errors: INVALID_ARG (NULL), OUT_OF_RANGE (no such tensor / index). */
int llm_gguf_find_tensor(const llm_gguf *g, const char *name, llm_gguf_tensor *t);
int llm_gguf_tensor_at(const llm_gguf *g, int64_t i, const char **name, llm_gguf_tensor *t);

/* Metadata: the i-th key in file order with its type; a key's type (element
 * type and count for arrays, byte count for strings, 1 otherwise); an integer
 * value (any of the integer types and BOOL; UINT64 above INT64_MAX is
 * OUT_OF_RANGE); a float value (FLOAT32 widened, FLOAT64); a string value (a
 * HOST pointer into the mapping, `len` bytes of UTF-8, not zero-terminated).
 * Errors: OUT_OF_RANGE (no such key / index), INVALID_ARG (NULL, other type). */
int llm_gguf_meta_at(const llm_gguf *g, int64_t i, const char **key, int32_t *type);
int llm_gguf_meta_type(const llm_gguf *g, const char *key, int32_t *type, int32_t *elem_type, uint64_t *count);
int llm_gguf_meta_int(const llm_gguf *g, const char *key, int64_t *out);
int llm_gguf_meta_float(const llm_gguf *g, const char *key, double *out);
int llm_gguf_meta_string(const llm_gguf *g, const char *key, const char **s, uint64_t *len);

/* The model shape from the metadata ("The Forward Pass in Java", Example 1):
 * general.architecture "llama" (RoPE pairs (2i, 2i+1)) or "qwen2" (NEOX
 * pairs); <arch>.embedding_length, block_count, attention.head_count,
 * feed_forward_length, context_length, attention.layer_norm_rms_epsilon;
 * optional attention.head_count_kv (default head_count), rope.freq_base
 * (10000), rope.dimension_count (dim / heads), vocab_size (the length of the
 * tokenizer.ggml.tokens array); wtype = the type of token_embd.weight.
 * max_seq > 0 sets the KV-cache rows, else <arch>.context_length is used.
 * Errors: INVALID_ARG (missing or mistyped key, no token_embd.weight),
 * UNSUPPORTED (other architecture); `err` as for llm_gguf_open. */
int llm_gguf_config(const llm_gguf *g, int32_t max_seq, llm_config *cfg, char *err, size_t err_len);

/* A handle for the model in the file: llm_gguf_config, then the tensors of
 * "The Forward Pass in Java", Example 13, by their llama.cpp names —
 * token_embd.weight, output_norm.weight, output.weight (absent: tied to the
 * embedding), rope_freqs.weight (optional), and for each layer N
 * blk.N.attn_norm, attn_q, attn_k, attn_v, attn_output, ffn_norm, ffn_gate,
 * ffn_up, ffn_down (.weight) and the optional blk.N.attn_q/k/v.bias — each
 * checked for its shape (matrices [in, out], vectors [n]) and type (every
 * matrix the embedding's type, vectors F32), copied once to a temporary
 * device buffer, given to llm_create on `stream`, and freed before return.
 * The file stays owned by the caller (the handle keeps no reference to it).
 * Synchronous.  Errors: those of llm_gguf_config and llm_create, INVALID_ARG
 * / UNSUPPORTED for a missing or mismatched tensor, NO_MEMORY / CUDA for the
 * staging buffer; *out is NULL then and `err` holds the reason. */
int llm_create_from_gguf(const llm_gguf *g, int32_t max_seq, llm_stream_t stream, llm_handle **out, char *err,
                         size_t err_len);

#ifdef __cplusplus
}
#endif
#endif /* LLM_H */
