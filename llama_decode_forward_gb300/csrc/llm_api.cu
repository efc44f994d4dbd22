// C ABI of libllmdecode (declared in include/llm.h): handle lifetime, weight
// repacking, argument validation and step launches.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>
#include <unordered_set>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "llm_internal.cuh"

namespace llm {
bool step_geometry(StepParams& p, int dim, int stage_floats, int n_heads, int n_kv, int hd, int rope_dims,
                   int rowp_floats, int rowp_logits, bool llamacpp, size_t* smem_bytes);
bool matrix_plan(DMat& m, int wtype, bool pair);
bool gview_plan(GView& v, int wtype, int rows, int cols, int ngrp, int max_rows);
const void* step_kernel_ptr(int wtype, bool llamacpp);
void launch_kv_store(cudaStream_t st, __half* kc, __half* vc, int pos, int kv_dim, const float* k, const float* v);
void launch_dequant_rows(cudaStream_t st, int wtype, const DMat& m, int row0, int n_rows, float* out);
cudaError_t launch_gemv_test(cudaStream_t st, int wtype, bool llamacpp, const StepParams& p, int which, int layer,
                             const float* x, float* y, int sms, size_t smem);
}  // namespace llm

using namespace llm;

// ------------------------------------------------------------ allocations --
// Every device and pinned-host allocation of the library goes through these
// two functions.  llm_test_fail_alloc(n) arms a countdown: the n-th
// allocation from then on fails with cudaErrorMemoryAllocation without
// calling CUDA (and disarms the countdown), so tests can make each allocation
// of llm_create or llm_prefill fail in turn.
static std::atomic<int> g_fail_countdown{0};

static bool injected_failure() {
    int n = g_fail_countdown.load();
    while (n > 0 && !g_fail_countdown.compare_exchange_weak(n, n - 1)) {}
    return n == 1;
}

namespace llm {
cudaError_t dev_alloc(void** p, size_t bytes) {
    if (injected_failure()) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(p, bytes);
}
}  // namespace llm

static cudaError_t host_alloc(void** p, size_t bytes) {
    if (injected_failure()) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMallocHost(p, bytes);
}

// Guard bands: the KV cache, the activations and the prefill workspace are
// allocated with kGuardBytes more on each side, filled with kGuardByte; the
// buffer proper starts kGuardBytes into the allocation (256-byte alignment
// kept).  llm_test_guards counts guard bytes that changed: a kernel that
// wrote past either end of one of these buffers shows up there.
constexpr size_t kGuardBytes = 4096;
constexpr int kGuardByte = 0xA5;

struct Guarded {
    uint8_t* raw = nullptr;   // the allocation (freed with cudaFree)
    size_t bytes = 0;         // the buffer proper
    uint8_t* ptr() const { return raw ? raw + kGuardBytes : nullptr; }
};

static cudaError_t guarded_alloc(Guarded& g, size_t bytes, cudaStream_t st) {
    void* raw = nullptr;
    cudaError_t e = dev_alloc(&raw, bytes + 2 * kGuardBytes);
    if (e != cudaSuccess) return e;
    g.raw = static_cast<uint8_t*>(raw);
    g.bytes = bytes;
    e = cudaMemsetAsync(g.raw, kGuardByte, kGuardBytes, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(g.raw + kGuardBytes + bytes, kGuardByte, kGuardBytes, st);
    return e;
}

static void guarded_free(Guarded& g) {
    cudaFree(g.raw);
    g = Guarded{};
}

struct HostPinned {
    int token_in;
    int argmax;
    int err;
};

struct llm_handle {
    llm_config cfg;
    cudaStream_t st = nullptr;
    int device = 0, sms = 0;
    int q_dim = 0, kv_dim = 0, max_splits = 1;
    int ngrp = 1;                    // column groups of the decode step's O and down products
    size_t smem = 0;
    const void* kernel = nullptr;
    StepParams geo{};                // shared-memory geometry of the step kernel
    CUtensorMap* kv_maps = nullptr;  // device array [kMapsPerLayer * n_layers]
    float theta_scale = 0.f, attn_div = 0.f;

    uint8_t* arena = nullptr;        // weights in the library layout
    size_t arena_bytes = 0;
    __half* kv = nullptr;            // [n_layers][2][max_seq][kv_dim]
    uint8_t* act = nullptr;          // activations, counters, partials
    Guarded kv_mem, act_mem, ws_mem; // the guarded allocations behind kv, act and prefill_ws
    std::vector<LayerDev> layers;
    LayerDev* d_layers = nullptr;
    DMat embd{}, out{};
    const float* out_norm = nullptr;
    const float* rope_freqs = nullptr;

    unsigned long long* tv = nullptr;  // tagged activation vectors of every layer
    size_t tv_words = 0;
    unsigned long long* part = nullptr;  // tagged attention partials of every layer
    size_t part_words = 0;
    unsigned long long* delta = nullptr; // residual accumulators, two parities
    size_t delta_words = 0;
    unsigned* epoch = nullptr;          // tag of the last completed step
    float* logits = nullptr;
    unsigned long long* best = nullptr;
    unsigned* counters = nullptr;
    int n_counters = 0;
    int* err = nullptr;
    int* tok_in = nullptr;
    int* tok_out = nullptr;
    HostPinned* pinned = nullptr;

    int64_t launches = 0;
    bool broken = false;             // a device error was seen; cleared by llm_reset
    std::string last_error;

    unsigned long long* trace = nullptr;   // LLM_TRACE builds: [sms][kTraceSlots]
    void* prefill_ws = nullptr;      // prefill workspace (lazily sized)
    size_t prefill_ws_bytes = 0;
    __half* f16_copy = nullptr;      // llm_prefill_f16_copy: F16 copy of the Q8_0 layer matrices
    size_t f16_copy_bytes = 0;
    int test_logits_limit = 0;       // llm_test_logits_limit: > 0 narrows the checked logits bound
};

// --------------------------------------------------------------- helpers --
static int fail(llm_handle* h, int status, const char* fmt, ...) {
    if (h) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        h->last_error = buf;
    }
    return status;
}

#define CK(h, call)                                                                                   \
    do {                                                                                              \
        cudaError_t e_ = (call);                                                                      \
        if (e_ != cudaSuccess) {                                                                      \
            cudaGetLastError();                                                                       \
            return fail((h), e_ == cudaErrorMemoryAllocation ? LLM_ERR_NO_MEMORY : LLM_ERR_CUDA,      \
                        "%s: %s", #call, cudaGetErrorString(e_));                                     \
        }                                                                                             \
    } while (0)

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

static int scale_stride(int cols) { return ((cols / 32) + 7) & ~7; }

static size_t mat_bytes(int wtype, long long rows, long long cols) {
    if (wtype == LLM_Q8_0) return (size_t)(rows * cols + rows * scale_stride((int)cols) * 2);
    return (size_t)(rows * cols * (wtype == LLM_F16 ? 2 : 4));
}

// Q8_0 blocks (34 bytes: FP16 scale, 32 int8) of `rows` rows -> the int8
// quants and the scales of the library layout (two planes); source row r goes
// to destination row dst0 + r*mul + phase.
__global__ void repack_q8_kernel(const uint8_t* __restrict__ src, int rows, int cols, uint8_t* dq, __half* dd,
                                 int dstride, int dst0, int mul, int phase) {
    const int nb = cols / 32;
    const long long total = (long long)rows * nb;
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < total;
         b += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(b / nb), j = (int)(b % nb);
        const uint8_t* s = src + b * 34;
        const long long dr = (long long)dst0 + (long long)r * mul + phase;
        dd[dr * dstride + j] = __ushort_as_half((unsigned short)(s[0] | (s[1] << 8)));
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; k++)
            w[k] = (uint32_t)s[2 + 4 * k] | ((uint32_t)s[3 + 4 * k] << 8) | ((uint32_t)s[4 + 4 * k] << 16) |
                   ((uint32_t)s[5 + 4 * k] << 24);
        uint4* d = reinterpret_cast<uint4*>(dq + dr * cols + (long long)j * 32);
        d[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

// Copy one matrix from the caller's GGUF layout into destination rows.
static int put_matrix(llm_handle* h, const void* src, int rows, int cols, const DMat& dst, int dst0, int mul,
                      int phase) {
    const int wt = h->cfg.wtype;
    if (!src) return fail(h, LLM_ERR_INVALID_ARG, "a weight pointer is NULL");
    if (wt == LLM_Q8_0) {
        const long long total = (long long)rows * (cols / 32);
        const int blocks = (int)((total + 255) / 256 < 65535 * 8 ? (total + 255) / 256 : 65535 * 8);
        repack_q8_kernel<<<blocks, 256, 0, h->st>>>((const uint8_t*)src, rows, cols, (uint8_t*)dst.q,
                                                    (__half*)dst.d, dst.dstride, dst0, mul, phase);
        h->launches++;
        CK(h, cudaGetLastError());
    } else {
        const size_t rb = (size_t)cols * (wt == LLM_F16 ? 2 : 4);
        CK(h, cudaMemcpy2DAsync((uint8_t*)dst.q + ((size_t)dst0 + phase) * rb, rb * mul, src, rb, rb, rows,
                                cudaMemcpyDeviceToDevice, h->st));
    }
    return LLM_OK;
}

// A matrix of `rows` rows in the arena.  pair: rows 2i and 2i+1 are one
// super-row of the streaming plan (m.rows then counts super-rows).
static DMat carve_mat(llm_handle* h, size_t& off, int rows, int cols, bool pair = false) {
    DMat m{};
    m.rows = rows;
    m.cols = cols;
    if (h->cfg.wtype == LLM_Q8_0) {
        m.q = h->arena + off;
        off += align256((size_t)rows * cols);
        m.dstride = scale_stride(cols);
        m.d = reinterpret_cast<const __half*>(h->arena + off);
        off += align256((size_t)rows * m.dstride * 2);
    } else {
        m.q = h->arena + off;
        off += align256(mat_bytes(h->cfg.wtype, rows, cols));
        m.d = nullptr;
    }
    if (pair) m.rows = rows / 2;
    if (!matrix_plan(m, h->cfg.wtype, pair)) m.rpc = 0;
    return m;
}

// The model shape alone: what the kernels support (no weight pointers).
static int validate_config(const llm_config* c, llm_handle* h) {
    if (!c) return fail(h, LLM_ERR_INVALID_ARG, "config is NULL");
    if (c->n_layers <= 0 || c->dim <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
        c->ffn_dim <= 0 || c->vocab <= 0 || c->max_seq <= 0)
        return fail(h, LLM_ERR_INVALID_ARG, "every size must be positive");
    if (c->n_heads % c->n_kv_heads) return fail(h, LLM_ERR_INVALID_ARG, "n_heads %% n_kv_heads != 0");
    if (c->head_dim * c->n_heads != c->dim) return fail(h, LLM_ERR_INVALID_ARG, "head_dim * n_heads != dim");
    if (c->rope_dims <= 0 || c->rope_dims % 2 || c->rope_dims > c->head_dim)
        return fail(h, LLM_ERR_INVALID_ARG, "rope_dims must be even and in (0, head_dim]");
    if (!(c->eps >= 0.f) || !(c->rope_base > 0.f)) return fail(h, LLM_ERR_INVALID_ARG, "bad eps or rope_base");
    if (c->numerics != LLM_NUMERICS_EXACT && c->numerics != LLM_NUMERICS_LLAMACPP)
        return fail(h, LLM_ERR_INVALID_ARG, "numerics must be LLM_NUMERICS_EXACT or LLM_NUMERICS_LLAMACPP");
    if (c->wtype != LLM_F32 && c->wtype != LLM_F16 && c->wtype != LLM_Q8_0)
        return fail(h, LLM_ERR_UNSUPPORTED, "weight type %d not supported", c->wtype);
    const int mult = c->wtype == LLM_Q8_0 ? 32 : (c->wtype == LLM_F16 ? 8 : 4);
    if (c->dim % mult || c->ffn_dim % mult)
        return fail(h, c->wtype == LLM_Q8_0 ? LLM_ERR_INVALID_ARG : LLM_ERR_UNSUPPORTED,
                    "dim and ffn_dim must be multiples of %d for this weight type", mult);
    if (c->head_dim % 8 || c->head_dim > 256) return fail(h, LLM_ERR_UNSUPPORTED, "head_dim must be a multiple of 8, <= 256");
    const int gq = c->n_heads / c->n_kv_heads;
    if (gq > kConsumerWarps || gq * c->head_dim > kMaxGroupDim)
        return fail(h, LLM_ERR_UNSUPPORTED, "query heads per kv head too large");
    // the step kernel keeps a phase's activation vector in shared memory and
    // each lane 64 of its elements in registers; rows must fit a ring slot
    const int q_dim = c->n_heads * c->head_dim;
    if (c->dim > 5760 || c->ffn_dim > 16384 || q_dim > 5760)
        return fail(h, LLM_ERR_UNSUPPORTED, "dim must be at most 5760 and ffn_dim at most 16384");
    if ((long long)slot_row_bytes(c->wtype, c->ffn_dim, scale_stride(c->ffn_dim)) > kSlotBytes ||
        (long long)slot_row_bytes(c->wtype, c->dim, scale_stride(c->dim)) > kSlotBytes)
        return fail(h, LLM_ERR_UNSUPPORTED, "matrix rows too long for the streaming ring");
    return LLM_OK;
}

static int validate(const llm_config* c, const llm_weights* w, llm_handle* h) {
    if (!c || !w) return fail(h, LLM_ERR_INVALID_ARG, "config or weights is NULL");
    const int rc = validate_config(c, h);
    if (rc) return rc;
    if (!w->tok_embd || !w->output_norm || !w->layers) return fail(h, LLM_ERR_INVALID_ARG, "a weight pointer is NULL");
    for (int l = 0; l < c->n_layers; l++) {
        const llm_layer_weights& L = w->layers[l];
        if (!L.attn_norm || !L.ffn_norm || !L.wq || !L.wk || !L.wv || !L.wo || !L.w_gate || !L.w_up || !L.w_down)
            return fail(h, LLM_ERR_INVALID_ARG, "layer %d: a weight pointer is NULL", l);
    }
    return LLM_OK;
}

static void free_handle(llm_handle* h) {
    if (!h) return;
    if (h->st) cudaStreamSynchronize(h->st);
    cudaFree(h->arena);
    guarded_free(h->kv_mem);
    guarded_free(h->act_mem);
    cudaFree(h->d_layers);
    cudaFree(h->kv_maps);
    guarded_free(h->ws_mem);
    cudaFree(h->f16_copy);
    cudaFree(h->trace);
    if (h->pinned) cudaFreeHost(h->pinned);
    cudaGetLastError();
    delete h;
}

// ----------------------------------------------------------- live handles --
// Every handle llm_create returned that llm_destroy has not freed.  The entry
// points refuse any other pointer with LLM_ERR_INVALID_ARG before touching
// it, so a second llm_destroy or a call on a destroyed handle does nothing
// (a pointer that a later llm_create happens to receive again names that new
// handle).
static std::mutex g_live_mu;
static std::unordered_set<const llm_handle*>& live_set() {
    static std::unordered_set<const llm_handle*> s;
    return s;
}
static bool alive(const llm_handle* h) {
    if (!h) return false;
    std::lock_guard<std::mutex> g(g_live_mu);
    return live_set().count(h) != 0;
}
#define LIVE_OR_RETURN(h)                           \
    do {                                            \
        if (!alive(h)) return LLM_ERR_INVALID_ARG;  \
    } while (0)

namespace llm {
// The shape checks of llm_create, for callers that want them before moving
// any weights (llm_create_from_gguf): LLM_OK, or a status and *why.
int check_shape(const llm_config* c, std::string* why) {
    llm_handle tmp;
    const int rc = validate_config(c, &tmp);
    if (why) *why = tmp.last_error;
    return rc;
}
}  // namespace llm

// Reason of the calling thread's last failed llm_create: there is no handle
// to hold it then, so llm_last_error(NULL) returns it.
static thread_local std::string t_create_error;

// A failed llm_create: keep the handle's reason for llm_last_error(NULL) and
// release what was allocated so far.
static int create_failed(llm_handle* h, int rc) {
    t_create_error = h->last_error.empty() ? llm_status_string(rc) : h->last_error;
    free_handle(h);
    return rc;
}

// ------------------------------------------------------------------ ABI --
extern "C" int llm_create(const llm_config* cfg, const llm_weights* w, llm_stream_t stream, llm_handle** out) {
    if (!out) return LLM_ERR_INVALID_ARG;
    *out = nullptr;
    llm_handle* h = new llm_handle();
    int rc = validate(cfg, w, h);
    if (rc) {
        t_create_error = h->last_error;
        delete h;                          // nothing allocated yet: no CUDA call
        return rc;
    }
    const llm_config& c = *cfg;
    h->cfg = c;
    h->st = (cudaStream_t)stream;
    h->q_dim = c.n_heads * c.head_dim;
    h->kv_dim = c.n_kv_heads * c.head_dim;
#define CKC(call)                                                                                      \
    do {                                                                                               \
        cudaError_t e_ = (call);                                                                       \
        if (e_ != cudaSuccess) {                                                                       \
            cudaGetLastError();                                                                        \
            return create_failed(h, fail(h, e_ == cudaErrorMemoryAllocation ? LLM_ERR_NO_MEMORY : LLM_ERR_CUDA, \
                                         "%s: %s", #call, cudaGetErrorString(e_)));                    \
        }                                                                                              \
    } while (0)
    CKC(cudaGetDevice(&h->device));
    CKC(cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, h->device));
    int coop = 0;
    CKC(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device));
    if (!coop) return create_failed(h, fail(h, LLM_ERR_UNSUPPORTED, "the device has no cooperative launch"));

    // ---- weight arena
    const int L = c.n_layers, d = c.dim, q = h->q_dim, kv = h->kv_dim, f = c.ffn_dim;
    size_t bytes = 0;
    for (int l = 0; l < L; l++) {
        bytes += align256(mat_bytes(c.wtype, q + 2 * kv, d)) + 256 * 2;
        bytes += align256(mat_bytes(c.wtype, d, q)) + 256 * 2;
        bytes += align256(mat_bytes(c.wtype, 2 * f, d)) + 256 * 2;
        bytes += align256(mat_bytes(c.wtype, d, f)) + 256 * 2;
        bytes += 2 * align256((size_t)d * 4) + align256((size_t)(q + 2 * kv) * 4);
    }
    bytes += align256(mat_bytes(c.wtype, c.vocab, d)) + 512;
    if (w->output) bytes += align256(mat_bytes(c.wtype, c.vocab, d)) + 512;
    bytes += align256((size_t)d * 4) + align256((size_t)c.rope_dims * 2 + 4);
    h->arena_bytes = bytes;
    CKC(dev_alloc((void**)&h->arena, bytes));

    size_t off = 0;
    h->layers.resize(L);
    for (int l = 0; l < L; l++) {
        const llm_layer_weights& W = w->layers[l];
        LayerDev& D = h->layers[l];
        D.qkv = carve_mat(h, off, q + 2 * kv, d);
        D.o = carve_mat(h, off, d, q);
        D.gu = carve_mat(h, off, 2 * f, d, true);
        D.down = carve_mat(h, off, d, f);
        float* an = (float*)(h->arena + off); off += align256((size_t)d * 4);
        float* fn = (float*)(h->arena + off); off += align256((size_t)d * 4);
        float* bias = (float*)(h->arena + off); off += align256((size_t)(q + 2 * kv) * 4);
        D.attn_norm = an;
        D.ffn_norm = fn;
        D.qkv_bias = (W.bq || W.bk || W.bv) ? bias : nullptr;
        if ((rc = put_matrix(h, W.wq, q, d, D.qkv, 0, 1, 0)) ||
            (rc = put_matrix(h, W.wk, kv, d, D.qkv, q, 1, 0)) ||
            (rc = put_matrix(h, W.wv, kv, d, D.qkv, q + kv, 1, 0)) ||
            (rc = put_matrix(h, W.wo, d, q, D.o, 0, 1, 0)) ||
            (rc = put_matrix(h, W.w_gate, f, d, D.gu, 0, 2, 0)) ||
            (rc = put_matrix(h, W.w_up, f, d, D.gu, 0, 2, 1)) ||
            (rc = put_matrix(h, W.w_down, d, f, D.down, 0, 1, 0)))
            return create_failed(h, rc);
        CKC(cudaMemcpyAsync(an, W.attn_norm, (size_t)d * 4, cudaMemcpyDeviceToDevice, h->st));
        CKC(cudaMemcpyAsync(fn, W.ffn_norm, (size_t)d * 4, cudaMemcpyDeviceToDevice, h->st));
        if (D.qkv_bias) {
            CKC(cudaMemsetAsync(bias, 0, (size_t)(q + 2 * kv) * 4, h->st));
            if (W.bq) CKC(cudaMemcpyAsync(bias, W.bq, (size_t)q * 4, cudaMemcpyDeviceToDevice, h->st));
            if (W.bk) CKC(cudaMemcpyAsync(bias + q, W.bk, (size_t)kv * 4, cudaMemcpyDeviceToDevice, h->st));
            if (W.bv) CKC(cudaMemcpyAsync(bias + q + kv, W.bv, (size_t)kv * 4, cudaMemcpyDeviceToDevice, h->st));
        }
    }
    h->embd = carve_mat(h, off, c.vocab, d);
    if ((rc = put_matrix(h, w->tok_embd, c.vocab, d, h->embd, 0, 1, 0))) return create_failed(h, rc);
    if (w->output) {
        h->out = carve_mat(h, off, c.vocab, d);
        if ((rc = put_matrix(h, w->output, c.vocab, d, h->out, 0, 1, 0))) return create_failed(h, rc);
    } else {
        h->out = h->embd;                                      // tied embeddings
    }
    float* onorm = (float*)(h->arena + off); off += align256((size_t)d * 4);
    CKC(cudaMemcpyAsync(onorm, w->output_norm, (size_t)d * 4, cudaMemcpyDeviceToDevice, h->st));
    h->out_norm = onorm;
    if (w->rope_freqs) {
        float* fr = (float*)(h->arena + off); off += align256((size_t)c.rope_dims * 2 + 4);
        CKC(cudaMemcpyAsync(fr, w->rope_freqs, (size_t)(c.rope_dims / 2) * 4, cudaMemcpyDeviceToDevice, h->st));
        h->rope_freqs = fr;
    }

    // ---- KV cache
    const size_t kv_bytes = (size_t)L * 2 * c.max_seq * kv * sizeof(__half);
    CKC(guarded_alloc(h->kv_mem, kv_bytes, h->st));
    h->kv = reinterpret_cast<__half*>(h->kv_mem.ptr());
    CKC(cudaMemsetAsync(h->kv, 0, kv_bytes, h->st));
    for (int l = 0; l < L; l++) {
        h->layers[l].kc = h->kv + (size_t)(2 * l) * c.max_seq * kv;
        h->layers[l].vc = h->layers[l].kc + (size_t)c.max_seq * kv;
    }
    CKC(dev_alloc((void**)&h->d_layers, sizeof(LayerDev) * L));
    CKC(cudaMemcpyAsync(h->d_layers, h->layers.data(), sizeof(LayerDev) * L, cudaMemcpyHostToDevice, h->st));

    // ---- column groups of the decode step: the largest divisor of n_kv up
    // to 8 (else the smallest above) whose Wo and Wdown column blocks have
    // whole Q8_0 blocks (rows of 16-byte words for F16/F32) and whose merged
    // attention output fits the kernel's pairs of consumer threads
    {
        const int unit = c.wtype == LLM_Q8_0 ? 32 : (c.wtype == LLM_F16 ? 8 : 4);
        auto fits = [&](int n) {
            return c.n_kv_heads % n == 0 && q % n == 0 && f % n == 0 && (q / n) % unit == 0 && (f / n) % unit == 0 &&
                   q / n <= 2 * kConsumers && n <= h->sms;
        };
        int ng = 0;
        for (int n = 1; n <= c.n_kv_heads && n <= 8; n++)
            if (fits(n)) ng = n;
        for (int n = 9; !ng && n <= c.n_kv_heads; n++)
            if (fits(n)) ng = n;
        if (!ng)
            return create_failed(h, fail(h, LLM_ERR_UNSUPPORTED,
                                         "no column grouping of the output and down projections fits this shape"));
        h->ngrp = ng;
    }
    const int gdg = q / h->ngrp, fdg = f / h->ngrp;
    const int min_gsz = h->sms / h->ngrp;                      // CTAs in the smallest group
    const int view_rows = (d + min_gsz - 1) / min_gsz;         // most rows a CTA takes of a group's columns
    if (!gview_plan(h->geo.ov, c.wtype, d, q, h->ngrp, view_rows) ||
        !gview_plan(h->geo.dv, c.wtype, d, f, h->ngrp, view_rows))
        return create_failed(h, fail(h, LLM_ERR_UNSUPPORTED, "no streaming plan for the output or down projection"));

    // ---- activations
    // position splits per kv head: enough units to cover every SM, at most 32
    // (the merge takes one split per lane) and at most 256 weights per group
    {
        int ms = h->sms / c.n_kv_heads;
        if (ms > 32) ms = 32;
        const int hg = c.n_heads / h->ngrp;
        if (ms > kOwnFloats / hg) ms = kOwnFloats / hg;
        h->max_splits = ms > 1 ? ms : 1;
    }
    h->n_counters = 1;
    size_t a = 0;
    auto take = [&](size_t b) { size_t o = a; a += align256(b); return o; };
    h->tv_words = (size_t)L * (size_t)tv_layout(d, q, kv, f).stride;
    h->part_words = (size_t)L * (size_t)part_words_per_layer(c.n_heads, h->max_splits, c.head_dim);
    h->delta_words = (size_t)2 * L * 2 * d;
    const size_t o_tv = take(h->tv_words * 8), o_part = take(h->part_words * 8), o_delta = take(h->delta_words * 8),
                 o_epoch = take(4), o_logits = take((size_t)c.vocab * 4), o_best = take(8),
                 o_ctr = take((size_t)h->n_counters * 4), o_err = take(4), o_tin = take(4), o_tout = take(4);
    CKC(guarded_alloc(h->act_mem, a, h->st));
    h->act = h->act_mem.ptr();
    CKC(cudaMemsetAsync(h->act, 0, a, h->st));
    h->tv = (unsigned long long*)(h->act + o_tv);
    h->part = (unsigned long long*)(h->act + o_part);
    h->delta = (unsigned long long*)(h->act + o_delta);
    h->epoch = (unsigned*)(h->act + o_epoch);
    h->logits = (float*)(h->act + o_logits);
    h->best = (unsigned long long*)(h->act + o_best);
    h->counters = (unsigned*)(h->act + o_ctr);
    h->err = (int*)(h->act + o_err);
    h->tok_in = (int*)(h->act + o_tin);
    h->tok_out = (int*)(h->act + o_tout);
    CKC(host_alloc((void**)&h->pinned, sizeof(HostPinned)));
#ifdef LLM_TRACE
    CKC(dev_alloc((void**)&h->trace, (size_t)h->sms * kTraceSlots * 8));
    CKC(cudaMemsetAsync(h->trace, 0, (size_t)h->sms * kTraceSlots * 8, h->st));
#endif

    h->theta_scale = (float)pow((double)c.rope_base, -2.0 / (double)c.rope_dims);
    h->attn_div = (float)sqrt((double)c.head_dim);
    h->kernel = step_kernel_ptr(c.wtype, c.numerics == LLM_NUMERICS_LLAMACPP);
    // row partials a CTA keeps for one GEMV phase (multi-warp teams): its rows
    // times the warps of a team; the logits phase's are kept apart
    int rowp_floats = 0, rowp_logits = 0;
    {
        auto parts = [](const DMat& m) { return m.tw > 32 ? m.tw / 32 : 0; };
        const DMat& Q = h->layers[0].qkv;
        const DMat& GU = h->layers[0].gu;
        rowp_floats = std::max(rowp_floats, (Q.rows + h->sms - 1) / h->sms * parts(Q));
        rowp_floats = std::max(rowp_floats, 2 * ((fdg + min_gsz - 1) / min_gsz) * parts(GU));
        rowp_floats = std::max(rowp_floats, view_rows * parts(h->geo.ov.m));
        rowp_floats = std::max(rowp_floats, view_rows * parts(h->geo.dv.m));
        rowp_logits = (h->out.rows + h->sms - 1) / h->sms * parts(h->out);
    }
    if (!step_geometry(h->geo, d, std::max(gdg, fdg), c.n_heads, c.n_kv_heads, c.head_dim, c.rope_dims, rowp_floats,
                       rowp_logits, c.numerics == LLM_NUMERICS_LLAMACPP, &h->smem))
        return create_failed(h, fail(h, LLM_ERR_UNSUPPORTED, "the step's shared-memory layout does not fit"));
    // per-CTA shares that live in shared memory, and every matrix's plan
    if ((q + 2 * kv + h->sms - 1) / h->sms > kOwnFloats || 2 * ((fdg + min_gsz - 1) / min_gsz) > kOwnFloats)
        return create_failed(h, fail(h, LLM_ERR_UNSUPPORTED, "a CTA's share of a vector exceeds %d floats", kOwnFloats));
    for (int l = 0; l < L; l++) {
        const LayerDev& D = h->layers[l];
        if (!D.qkv.rpc || !D.gu.rpc)
            return create_failed(h, fail(h, LLM_ERR_UNSUPPORTED, "layer %d: no streaming plan for a matrix", l));
    }
    if (!h->embd.rpc || !h->out.rpc)
        return create_failed(h, fail(h, LLM_ERR_UNSUPPORTED, "no streaming plan for the vocabulary matrix"));
    CKC(cudaFuncSetAttribute(h->kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h->smem));
    int per_sm = 0;
    CKC(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, h->kernel, kBlock, h->smem));
    if (per_sm < 1) return create_failed(h, fail(h, LLM_ERR_UNSUPPORTED, "the step kernel cannot be resident"));

    // Tensor maps of every layer: the K and V cache ([max_seq][kv_dim] F16,
    // box [attn_rows][attn_w], read by the step kernel's TMA tile loads; the
    // tensor-core attention reads its tiles with ldmatrix, so they are
    // swizzled by their row width: 128, 64 or 32 bytes), then the column-group
    // views of Wo and Wdown (values as a 3-D view {U, cols/U, rows}, Q8_0
    // scales as a 2-D view {dstride, rows}; rows past the end read as zero).
    {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q_res;
        CKC(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q_res));
        if (!fn || q_res != cudaDriverEntryPointSuccess)
            return create_failed(h, fail(h, LLM_ERR_CUDA, "cuTensorMapEncodeTiled is not available"));
        auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        std::vector<CUtensorMap> maps((size_t)kMapsPerLayer * L);
        memset(maps.data(), 0, sizeof(CUtensorMap) * maps.size());
        const int es = c.wtype == LLM_Q8_0 ? 1 : (c.wtype == LLM_F16 ? 2 : 4);
        const CUtensorMapDataType vdt = c.wtype == LLM_Q8_0 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                        : c.wtype == LLM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        auto value_view = [&](CUtensorMap* m, const DMat& w, const GView& v) {
            cuuint64_t gdim[3] = {(cuuint64_t)v.U, (cuuint64_t)(w.cols / v.U), (cuuint64_t)w.rows};
            cuuint64_t gstride[2] = {(cuuint64_t)v.U * es, (cuuint64_t)w.cols * es};
            cuuint32_t box[3] = {(cuuint32_t)v.U, (cuuint32_t)(v.m.cols / v.U), (cuuint32_t)v.R};
            cuuint32_t estride[3] = {1, 1, 1};
            return encode(m, vdt, 3, (void*)w.q, gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        };
        auto scale_view = [&](CUtensorMap* m, const DMat& w, const GView& v) {
            cuuint64_t gdim[2] = {(cuuint64_t)w.dstride, (cuuint64_t)w.rows};
            cuuint64_t gstride[1] = {(cuuint64_t)w.dstride * 2};
            cuuint32_t box[2] = {(cuuint32_t)(v.rowd / 2), (cuuint32_t)v.R};
            cuuint32_t estride[2] = {1, 1};
            return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (void*)w.d, gdim, gstride, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        };
        for (int l = 0; l < L; l++) {
            CUtensorMap* lm = &maps[(size_t)kMapsPerLayer * l];
            for (int which = 0; which < 2; which++) {
                void* base = which ? (void*)h->layers[l].vc : (void*)h->layers[l].kc;
                cuuint64_t gdim[2] = {(cuuint64_t)kv, (cuuint64_t)c.max_seq};
                cuuint64_t gstride[1] = {(cuuint64_t)kv * 2};
                cuuint32_t box[2] = {(cuuint32_t)h->geo.attn_w, (cuuint32_t)h->geo.attn_rows};
                cuuint32_t estride[2] = {1, 1};
                const int row_bytes = h->geo.attn_w * 2;
                const CUtensorMapSwizzle swz = !h->geo.attn_mma ? CU_TENSOR_MAP_SWIZZLE_NONE
                                               : row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                               : row_bytes == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : row_bytes == 32  ? CU_TENSOR_MAP_SWIZZLE_32B
                                                                  : CU_TENSOR_MAP_SWIZZLE_NONE;
                CUresult r = encode(&lm[which], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, gdim, gstride, box, estride,
                                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
                if (r != CUDA_SUCCESS)
                    return create_failed(h, fail(h, LLM_ERR_CUDA, "cuTensorMapEncodeTiled (KV) of layer %d: error %d", l,
                                                 (int)r));
            }
            CUresult r = value_view(&lm[2], h->layers[l].o, h->geo.ov);
            if (r == CUDA_SUCCESS) r = value_view(&lm[4], h->layers[l].down, h->geo.dv);
            if (r == CUDA_SUCCESS && c.wtype == LLM_Q8_0) r = scale_view(&lm[3], h->layers[l].o, h->geo.ov);
            if (r == CUDA_SUCCESS && c.wtype == LLM_Q8_0) r = scale_view(&lm[5], h->layers[l].down, h->geo.dv);
            if (r != CUDA_SUCCESS)
                return create_failed(h, fail(h, LLM_ERR_CUDA, "cuTensorMapEncodeTiled (Wo / Wdown) of layer %d: error %d",
                                             l, (int)r));
        }
        CKC(dev_alloc((void**)&h->kv_maps, sizeof(CUtensorMap) * maps.size()));
        CKC(cudaMemcpyAsync(h->kv_maps, maps.data(), sizeof(CUtensorMap) * maps.size(), cudaMemcpyHostToDevice,
                            h->st));
    }
    CKC(cudaStreamSynchronize(h->st));
    t_create_error.clear();
    {
        std::lock_guard<std::mutex> g(g_live_mu);
        live_set().insert(h);
    }
    *out = h;
    return LLM_OK;
#undef CKC
}

// The step's parameters: the handle's model, layout and buffers (the
// no-alloc step then points the working memory elsewhere).
static StepParams step_params(const llm_handle* h, const int* token_dev, int pos, int* argmax_dev) {
    const llm_config& c = h->cfg;
    StepParams p = h->geo;
    p.layers = h->d_layers;
    p.kv_maps = h->kv_maps;
    p.trace = h->trace;
    p.embd = h->embd;
    p.out = h->out;
    p.out_norm = h->out_norm;
    p.rope_freqs = h->rope_freqs;
    p.n_layers = c.n_layers; p.dim = c.dim; p.n_heads = c.n_heads; p.n_kv = c.n_kv_heads; p.hd = c.head_dim;
    p.ffn = c.ffn_dim; p.vocab = c.vocab; p.max_seq = c.max_seq; p.rope_dims = c.rope_dims; p.neox = c.rope_neox;
    p.q_dim = h->q_dim; p.kv_dim = h->kv_dim; p.ngrp = h->ngrp;
    p.eps = c.eps; p.theta_scale = h->theta_scale; p.attn_div = h->attn_div;
    p.tv = h->tv; p.part = h->part; p.delta = h->delta; p.epoch = h->epoch; p.logits = h->logits;
    p.max_splits = h->max_splits; p.best = h->best; p.counters = h->counters; p.err = h->err;
    p.token_in = token_dev; p.token_out = argmax_dev; p.pos = pos;
    const int s = (pos + 1 + 15) / 16;
    p.splits = s < 1 ? 1 : (s > h->max_splits ? h->max_splits : s);
    p.tv_words = (long long)h->tv_words;
    p.part_words = (long long)h->part_words;
    p.delta_words = (long long)h->delta_words;
    p.logits_limit = h->test_logits_limit > 0 ? h->test_logits_limit : c.vocab;
    return p;
}

static int launch_step(llm_handle* h, const int* token_dev, int pos, int* argmax_dev) {
    StepParams p = step_params(h, token_dev, pos, argmax_dev);
    void* args[] = {&p};
    CK(h, cudaLaunchCooperativeKernel(h->kernel, dim3(h->sms), dim3(kBlock), args, h->smem, h->st));
    h->launches++;
    return LLM_OK;
}

// The status of a device error word: the first of timeout, token, range,
// check that is set, with every set condition named in the message.
static int device_error_status(llm_handle* h, int e) {
    if (!e) return LLM_OK;
    h->broken = true;
    std::string why;
    auto add = [&](int bit, const char* text) {
        if (!(e & bit)) return;
        if (!why.empty()) why += "; ";
        why += text;
    };
    add(kErrTimeout, "a bounded device wait expired");
    add(kErrToken, "a device-side token was out of range");
    add(kErrRange, "a residual update was not finite or not below 2^15 in magnitude");
    add(kErrCheck, "a device-side index check failed and its access was skipped");
    const int status = e & kErrTimeout ? LLM_ERR_DEVICE_TIMEOUT
                       : e & kErrToken ? LLM_ERR_OUT_OF_RANGE
                       : e & kErrRange ? LLM_ERR_NONFINITE
                       : e & kErrCheck ? LLM_ERR_CHECK
                                       : LLM_ERR_CUDA;
    return fail(h, status, "%s", why.c_str());
}

static int read_device_error(llm_handle* h) {
    CK(h, cudaMemcpyAsync(&h->pinned->err, h->err, 4, cudaMemcpyDeviceToHost, h->st));
    CK(h, cudaStreamSynchronize(h->st));
    return device_error_status(h, h->pinned->err);
}

extern "C" int llm_reset(llm_handle* h) {
    LIVE_OR_RETURN(h);
    CK(h, cudaStreamSynchronize(h->st));
    CK(h, cudaMemsetAsync(h->err, 0, 4, h->st));
    CK(h, cudaMemsetAsync(h->counters, 0, (size_t)h->n_counters * 4, h->st));
    CK(h, cudaMemsetAsync(h->best, 0, 8, h->st));
    // a step that stopped early may have left words with the next step's tag
    // and accumulator words half added
    CK(h, cudaMemsetAsync(h->tv, 0, h->tv_words * 8, h->st));
    CK(h, cudaMemsetAsync(h->part, 0, h->part_words * 8, h->st));
    CK(h, cudaMemsetAsync(h->delta, 0, h->delta_words * 8, h->st));
    CK(h, cudaMemsetAsync(h->epoch, 0, 4, h->st));
    CK(h, cudaStreamSynchronize(h->st));
    h->broken = false;
    return LLM_OK;
}

extern "C" int llm_decode_step(llm_handle* h, int32_t token, int32_t pos, float* logits_host, int32_t* argmax_host) {
    LIVE_OR_RETURN(h);
    if (h->broken) return fail(h, LLM_ERR_STATE, "handle has a device error; call llm_reset");
    if (token < 0 || token >= h->cfg.vocab) return fail(h, LLM_ERR_OUT_OF_RANGE, "token %d not in [0, %d)", token, h->cfg.vocab);
    if (pos < 0 || pos >= h->cfg.max_seq) return fail(h, LLM_ERR_OUT_OF_RANGE, "pos %d not in [0, %d)", pos, h->cfg.max_seq);
    h->pinned->token_in = token;
    CK(h, cudaMemcpyAsync(h->tok_in, &h->pinned->token_in, 4, cudaMemcpyHostToDevice, h->st));
    int rc = launch_step(h, h->tok_in, pos, h->tok_out);
    if (rc) return rc;
    CK(h, cudaMemcpyAsync(&h->pinned->argmax, h->tok_out, 4, cudaMemcpyDeviceToHost, h->st));
    if (logits_host)
        CK(h, cudaMemcpyAsync(logits_host, h->logits, (size_t)h->cfg.vocab * 4, cudaMemcpyDeviceToHost, h->st));
    if ((rc = read_device_error(h))) return rc;
    if (argmax_host) *argmax_host = h->pinned->argmax;
    return LLM_OK;
}

extern "C" int llm_decode_step_async(llm_handle* h, const int32_t* token_dev, int32_t pos, int32_t* argmax_dev) {
    LIVE_OR_RETURN(h);
    if (!token_dev || !argmax_dev) return fail(h, LLM_ERR_INVALID_ARG, "NULL argument");
    if (h->broken) return fail(h, LLM_ERR_STATE, "handle has a device error; call llm_reset");
    if (pos < 0 || pos >= h->cfg.max_seq) return fail(h, LLM_ERR_OUT_OF_RANGE, "pos %d not in [0, %d)", pos, h->cfg.max_seq);
    return launch_step(h, token_dev, pos, argmax_dev);
}

extern "C" int llm_generate(llm_handle* h, int32_t token, int32_t pos, int32_t n_steps, int32_t* tokens_dev) {
    LIVE_OR_RETURN(h);
    if (!tokens_dev || n_steps < 0) return fail(h, LLM_ERR_INVALID_ARG, "bad argument");
    if (h->broken) return fail(h, LLM_ERR_STATE, "handle has a device error; call llm_reset");
    if (token < 0 || token >= h->cfg.vocab) return fail(h, LLM_ERR_OUT_OF_RANGE, "token %d not in [0, %d)", token, h->cfg.vocab);
    if (pos < 0 || (long long)pos + n_steps > h->cfg.max_seq)
        return fail(h, LLM_ERR_OUT_OF_RANGE, "positions %d..%d exceed max_seq %d", pos, pos + n_steps - 1, h->cfg.max_seq);
    if (n_steps == 0) return LLM_OK;
    h->pinned->token_in = token;
    CK(h, cudaMemcpyAsync(h->tok_in, &h->pinned->token_in, 4, cudaMemcpyHostToDevice, h->st));
    for (int i = 0; i < n_steps; i++) {
        int rc = launch_step(h, i == 0 ? h->tok_in : tokens_dev + i - 1, pos + i, tokens_dev + i);
        if (rc) return rc;
    }
    return LLM_OK;
}

static PrefillCtx prefill_ctx(const llm_handle* h) {
    PrefillCtx pc{};
    pc.st = h->st; pc.sms = h->sms; pc.wtype = h->cfg.wtype;
    pc.n_layers = h->cfg.n_layers; pc.dim = h->cfg.dim; pc.n_heads = h->cfg.n_heads; pc.n_kv = h->cfg.n_kv_heads;
    pc.hd = h->cfg.head_dim; pc.ffn = h->cfg.ffn_dim; pc.vocab = h->cfg.vocab; pc.rope_dims = h->cfg.rope_dims;
    pc.neox = h->cfg.rope_neox; pc.q_dim = h->q_dim; pc.kv_dim = h->kv_dim;
    pc.eps = h->cfg.eps; pc.theta_scale = h->theta_scale; pc.attn_div = h->attn_div;
    pc.layers = h->layers.data(); pc.embd = h->embd; pc.out = h->out; pc.out_norm = h->out_norm;
    pc.rope_freqs = h->rope_freqs; pc.logits = h->logits; pc.argmax_dev = h->tok_out; pc.best = h->best; pc.err = h->err;
    pc.f16_copy = h->f16_copy;
    return pc;
}

extern "C" int llm_prefill_f16_copy(llm_handle* h, int enable) {
    LIVE_OR_RETURN(h);
    if (!enable) {
        if (h->f16_copy) {
            CK(h, cudaStreamSynchronize(h->st));
            CK(h, cudaFree(h->f16_copy));
            h->f16_copy = nullptr;
            h->f16_copy_bytes = 0;
        }
        return LLM_OK;
    }
    if (h->f16_copy) return LLM_OK;
    PrefillCtx pc = prefill_ctx(h);
    if (h->cfg.wtype != LLM_Q8_0)
        return fail(h, LLM_ERR_UNSUPPORTED, "an F16 prefill copy is for Q8_0 weights only");
    if (!prefill_supported(pc))
        return fail(h, LLM_ERR_UNSUPPORTED, "this model's prefill runs the decode step token by token");
    const size_t bytes = prefill_f16_copy_bytes(pc);
    void* p = nullptr;
    if (dev_alloc(&p, bytes) != cudaSuccess) {
        cudaGetLastError();
        return fail(h, LLM_ERR_NO_MEMORY, "allocating the %zu-byte F16 prefill copy", bytes);
    }
    int launches = 0;
    const cudaError_t e = prefill_make_f16_copy(pc, static_cast<__half*>(p), &launches);
    h->launches += launches;
    if (e == cudaSuccess) {
        h->f16_copy = static_cast<__half*>(p);
        h->f16_copy_bytes = bytes;
        return LLM_OK;
    }
    cudaStreamSynchronize(h->st);
    cudaFree(p);
    cudaGetLastError();
    return fail(h, LLM_ERR_CUDA, "F16 prefill copy: %s", cudaGetErrorString(e));
}

extern "C" int llm_prefill(llm_handle* h, const int32_t* tokens_host, int32_t n, int32_t pos0, float* logits_host,
                           int32_t* argmax_host) {
    LIVE_OR_RETURN(h);
    if (!tokens_host || n <= 0) return fail(h, LLM_ERR_INVALID_ARG, "bad argument");
    if (h->broken) return fail(h, LLM_ERR_STATE, "handle has a device error; call llm_reset");
    if (pos0 < 0 || (long long)pos0 + n > h->cfg.max_seq)
        return fail(h, LLM_ERR_OUT_OF_RANGE, "positions %d..%d exceed max_seq %d", pos0, pos0 + n - 1, h->cfg.max_seq);
    for (int i = 0; i < n; i++)
        if (tokens_host[i] < 0 || tokens_host[i] >= h->cfg.vocab)
            return fail(h, LLM_ERR_OUT_OF_RANGE, "token %d not in [0, %d)", tokens_host[i], h->cfg.vocab);
    int rc;
    const PrefillCtx pc = prefill_ctx(h);
    if (prefill_supported(pc)) {
        // F16 weights: tensor-core batches of up to kPrefillRows tokens
        const size_t need = prefill_workspace_bytes(pc);
        if (h->prefill_ws_bytes < need) {
            CK(h, cudaStreamSynchronize(h->st));
            guarded_free(h->ws_mem);
            h->prefill_ws = nullptr;
            h->prefill_ws_bytes = 0;
            CK(h, guarded_alloc(h->ws_mem, need, h->st));
            h->prefill_ws = h->ws_mem.ptr();
            h->prefill_ws_bytes = need;
        }
        const char* what = "";
        const cudaError_t e = prefill_f16(pc, h->prefill_ws, tokens_host, n, pos0, &what);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(h, LLM_ERR_CUDA, "prefill (%s): %s", what, cudaGetErrorString(e));
        }
        h->launches += 1 + (int64_t)h->cfg.n_layers * 8 + 3;
        CK(h, cudaMemcpyAsync(&h->pinned->argmax, h->tok_out, 4, cudaMemcpyDeviceToHost, h->st));
        if (logits_host)
            CK(h, cudaMemcpyAsync(logits_host, h->logits, (size_t)h->cfg.vocab * 4, cudaMemcpyDeviceToHost, h->st));
        if ((rc = read_device_error(h))) return rc;
        if (argmax_host) *argmax_host = h->pinned->argmax;
        return LLM_OK;
    }
    for (int i = 0; i < n - 1; i++) {
        h->pinned->token_in = tokens_host[i];
        CK(h, cudaMemcpyAsync(h->tok_in, &h->pinned->token_in, 4, cudaMemcpyHostToDevice, h->st));
        if ((rc = launch_step(h, h->tok_in, pos0 + i, h->tok_out))) return rc;
        CK(h, cudaStreamSynchronize(h->st));    // the pinned token slot is reused
    }
    return llm_decode_step(h, tokens_host[n - 1], pos0 + n - 1, logits_host, argmax_host);
}

extern "C" int llm_sync(llm_handle* h) {
    LIVE_OR_RETURN(h);
    CK(h, cudaStreamSynchronize(h->st));
    return read_device_error(h);
}

extern "C" const float* llm_logits_device(const llm_handle* h) { return alive(h) ? h->logits : nullptr; }

extern "C" int llm_get_config(const llm_handle* h, llm_config* out) {
    if (!alive(h) || !out) return LLM_ERR_INVALID_ARG;
    *out = h->cfg;
    return LLM_OK;
}

extern "C" int llm_kv_view(llm_handle* h, int layer, uint16_t** k_dev, uint16_t** v_dev) {
    if (!alive(h) || !k_dev || !v_dev) return LLM_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return fail(h, LLM_ERR_OUT_OF_RANGE, "layer %d", layer);
    *k_dev = reinterpret_cast<uint16_t*>(h->layers[layer].kc);
    *v_dev = reinterpret_cast<uint16_t*>(h->layers[layer].vc);
    return LLM_OK;
}

extern "C" int llm_test_kv_store(llm_handle* h, int layer, int32_t pos, const float* k_dev, const float* v_dev) {
    if (!alive(h) || !k_dev || !v_dev) return LLM_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers || pos < 0 || pos >= h->cfg.max_seq)
        return fail(h, LLM_ERR_OUT_OF_RANGE, "layer %d / pos %d", layer, pos);
    launch_kv_store(h->st, h->layers[layer].kc, h->layers[layer].vc, pos, h->kv_dim, k_dev, v_dev);
    h->launches++;
    CK(h, cudaGetLastError());
    CK(h, cudaStreamSynchronize(h->st));
    return LLM_OK;
}

extern "C" int llm_test_dequant_rows(llm_handle* h, int which, int layer, int32_t row0, int32_t n_rows, float* out_dev) {
    if (!alive(h) || !out_dev || n_rows < 0) return LLM_ERR_INVALID_ARG;
    if (which < 7 && (layer < 0 || layer >= h->cfg.n_layers)) return fail(h, LLM_ERR_OUT_OF_RANGE, "layer %d", layer);
    const llm_config& c = h->cfg;
    DMat m{};
    int first = 0, mul = 1, phase = 0, rows = 0;
    switch (which) {
        case 0: m = h->layers[layer].qkv; first = 0; rows = h->q_dim; break;
        case 1: m = h->layers[layer].qkv; first = h->q_dim; rows = h->kv_dim; break;
        case 2: m = h->layers[layer].qkv; first = h->q_dim + h->kv_dim; rows = h->kv_dim; break;
        case 3: m = h->layers[layer].o; rows = c.dim; break;
        case 4: m = h->layers[layer].gu; mul = 2; phase = 0; rows = c.ffn_dim; break;
        case 5: m = h->layers[layer].gu; mul = 2; phase = 1; rows = c.ffn_dim; break;
        case 6: m = h->layers[layer].down; rows = c.dim; break;
        case 7: m = h->embd; rows = c.vocab; break;
        case 8: m = h->out; rows = c.vocab; break;
        default: return fail(h, LLM_ERR_INVALID_ARG, "which = %d", which);
    }
    if (row0 < 0 || (long long)row0 + n_rows > rows) return fail(h, LLM_ERR_OUT_OF_RANGE, "rows %d..%d", row0, row0 + n_rows);
    for (int r = 0; r < n_rows; r++) {
        launch_dequant_rows(h->st, c.wtype, m, first + (row0 + r) * mul + phase, 1, out_dev + (size_t)r * m.cols);
        h->launches++;
    }
    CK(h, cudaGetLastError());
    CK(h, cudaStreamSynchronize(h->st));
    return LLM_OK;
}

extern "C" int llm_test_gemv(llm_handle* h, int which, int layer, const float* x_dev, float* y_dev) {
    if (!alive(h) || !x_dev || !y_dev) return LLM_ERR_INVALID_ARG;
    if (which < 0 || which > 4) return fail(h, LLM_ERR_INVALID_ARG, "which = %d", which);
    if (layer < 0 || layer >= h->cfg.n_layers) return fail(h, LLM_ERR_OUT_OF_RANGE, "layer %d", layer);
    if (h->broken) return fail(h, LLM_ERR_STATE, "handle has a device error; call llm_reset");
    StepParams p = step_params(h, h->tok_in, 0, h->tok_out);
    p.trace = nullptr;
    CK(h, launch_gemv_test(h->st, h->cfg.wtype, h->cfg.numerics == LLM_NUMERICS_LLAMACPP, p, which, layer, x_dev,
                           y_dev, h->sms, h->smem));
    h->launches++;
    CK(h, cudaStreamSynchronize(h->st));
    return read_device_error(h);
}

// Named intermediates of the last decode step, read back from the buffers the
// step kernel exchanges them through: the tagged Q/K/V and SwiGLU vectors,
// and the residual accumulator words of the attention and FFN updates.
extern "C" int llm_debug_tensor(llm_handle* h, int layer, int which, float* host, int32_t n) {
    LIVE_OR_RETURN(h);
    if (!host) return fail(h, LLM_ERR_INVALID_ARG, "NULL host buffer");
    if (layer < 0 || layer >= h->cfg.n_layers) return fail(h, LLM_ERR_OUT_OF_RANGE, "layer %d", layer);
    const llm_config& c = h->cfg;
    const TvLayout tl = tv_layout(c.dim, h->q_dim, h->kv_dim, c.ffn_dim);
    long long off;
    int len;
    bool tagged = true;
    switch (which) {
        case LLM_DEBUG_Q: off = tl.qkv; len = h->q_dim; break;
        case LLM_DEBUG_K: off = tl.qkv + h->q_dim; len = h->kv_dim; break;
        case LLM_DEBUG_V: off = tl.qkv + h->q_dim + h->kv_dim; len = h->kv_dim; break;
        case LLM_DEBUG_FFN_SWIGLU: off = tl.u; len = c.ffn_dim; break;
        case LLM_DEBUG_ATTN_OUT: off = 0; len = c.dim; tagged = false; break;
        case LLM_DEBUG_FFN_OUT: off = 1; len = c.dim; tagged = false; break;
        default: return fail(h, LLM_ERR_INVALID_ARG, "which %d", which);
    }
    if (n != len) return fail(h, LLM_ERR_INVALID_ARG, "tensor %d has %d values, buffer %d", which, len, n);
    CK(h, cudaStreamSynchronize(h->st));
    unsigned epoch = 0;
    CK(h, cudaMemcpy(&epoch, h->epoch, 4, cudaMemcpyDeviceToHost));
    if (epoch == 0) return fail(h, LLM_ERR_STATE, "no decode step has run on this handle since its reset");
    std::vector<unsigned long long> w(len);
    const unsigned long long* src;
    if (tagged) {
        src = h->tv + (long long)layer * tl.stride + off;
    } else {
        // the step's parity of [2][n_layers][2][dim]; word (layer, off)
        src = h->delta + (size_t)(epoch & 1u) * c.n_layers * 2 * c.dim + ((size_t)layer * 2 + off) * c.dim;
    }
    CK(h, cudaMemcpy(w.data(), src, (size_t)len * 8, cudaMemcpyDeviceToHost));
    for (int i = 0; i < len; i++) {
        if (tagged) {
            if ((unsigned)(w[i] >> 32) != epoch)
                return fail(h, LLM_ERR_STATE, "value %d of tensor %d is not from the last decode step", i, which);
            const uint32_t bits = (uint32_t)w[i];
            memcpy(&host[i], &bits, 4);
        } else {
            // (count << 56) + round(v * 2^32): the count rounds to the nearest multiple of 2^56
            const unsigned long long cnt = (w[i] + (1ull << 55)) >> 56;
            if (cnt != (unsigned long long)h->ngrp)
                return fail(h, LLM_ERR_STATE, "accumulator %d of tensor %d holds %llu of %d parts", i, which, cnt, h->ngrp);
            const long long v = (long long)(w[i] - (cnt << 56));
            host[i] = (float)ldexp((double)v, -32);
        }
    }
    return LLM_OK;
}

extern "C" int llm_test_logits_limit(llm_handle* h, int32_t limit) {
    LIVE_OR_RETURN(h);
#ifdef LLM_CHECKED
    if (limit < 0 || limit > h->cfg.vocab) return fail(h, LLM_ERR_OUT_OF_RANGE, "limit %d", limit);
    h->test_logits_limit = limit;
    return LLM_OK;
#else
    (void)limit;
    return fail(h, LLM_ERR_UNSUPPORTED, "not an LLM_CHECKED build");
#endif
}

extern "C" int llm_checked_build(void) {
#ifdef LLM_CHECKED
    return 1;
#else
    return 0;
#endif
}

extern "C" int llm_test_fail_alloc(int32_t nth) {
    if (nth < 0) return LLM_ERR_INVALID_ARG;
    g_fail_countdown.store(nth);
    return LLM_OK;
}

// The guarded buffers of a handle, in the order llm_test_poke_guard numbers
// their bands: KV cache, activations, prefill workspace (when allocated).
static int guarded_buffers(const llm_handle* h, const Guarded** out) {
    int n = 0;
    out[n++] = &h->kv_mem;
    out[n++] = &h->act_mem;
    if (h->ws_mem.raw) out[n++] = &h->ws_mem;
    return n;
}

extern "C" int64_t llm_test_guards(llm_handle* h) {
    LIVE_OR_RETURN(h);
    const Guarded* g[3];
    const int n = guarded_buffers(h, g);
    std::vector<uint8_t> band(kGuardBytes);
    int64_t changed = 0;
    CK(h, cudaStreamSynchronize(h->st));
    for (int i = 0; i < n; i++)
        for (int side = 0; side < 2; side++) {
            const uint8_t* src = g[i]->raw + (side ? kGuardBytes + g[i]->bytes : 0);
            CK(h, cudaMemcpy(band.data(), src, kGuardBytes, cudaMemcpyDeviceToHost));
            for (size_t k = 0; k < kGuardBytes; k++) changed += band[k] != (uint8_t)kGuardByte;
        }
    return changed;
}

extern "C" int llm_test_poke_guard(llm_handle* h, int band) {
    LIVE_OR_RETURN(h);
    const Guarded* g[3];
    const int n = guarded_buffers(h, g);
    if (band < 0 || band >= 2 * n) return fail(h, LLM_ERR_OUT_OF_RANGE, "guard band %d of %d", band, 2 * n);
    const Guarded& b = *g[band / 2];
    // the byte next to the buffer: the one an off-by-one write would hit
    uint8_t* at = band % 2 ? b.raw + kGuardBytes + b.bytes : b.raw + kGuardBytes - 1;
    CK(h, cudaStreamSynchronize(h->st));
    CK(h, cudaMemset(at, 0x5A, 1));
    return LLM_OK;
}

extern "C" int llm_column_groups(const llm_handle* h) { return alive(h) ? h->ngrp : LLM_ERR_INVALID_ARG; }

extern "C" int llm_trace_read(llm_handle* h, uint64_t* host, int32_t* sms) {
    if (!alive(h) || !host || !sms) return LLM_ERR_INVALID_ARG;
    if (!h->trace) return LLM_ERR_UNSUPPORTED;
    *sms = h->sms;
    CK(h, cudaMemcpyAsync(host, h->trace, (size_t)h->sms * kTraceSlots * 8, cudaMemcpyDeviceToHost, h->st));
    CK(h, cudaStreamSynchronize(h->st));
    return LLM_OK;
}

extern "C" int64_t llm_launch_count(const llm_handle* h) { return alive(h) ? h->launches : 0; }

extern "C" void llm_destroy(llm_handle* h) {
    {
        std::lock_guard<std::mutex> g(g_live_mu);
        if (!h || !live_set().erase(h)) return;   // NULL, already destroyed, or never created
    }
    free_handle(h);
}

extern "C" const char* llm_status_string(int s) {
    switch (s) {
        case LLM_OK: return "ok";
        case LLM_ERR_INVALID_ARG: return "invalid argument";
        case LLM_ERR_UNSUPPORTED: return "unsupported configuration";
        case LLM_ERR_OUT_OF_RANGE: return "token or position out of range";
        case LLM_ERR_CUDA: return "CUDA error";
        case LLM_ERR_NO_MEMORY: return "device allocation failed";
        case LLM_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case LLM_ERR_STATE: return "invalid handle state";
        case LLM_ERR_NONFINITE: return "a non-finite or out-of-range value in the residual stream";
        case LLM_ERR_CHECK: return "a device-side index check failed (LLM_CHECKED build)";
        default: return "unknown status";
    }
}

extern "C" const char* llm_last_error(const llm_handle* h) {
    if (!h) return t_create_error.c_str();
    return alive(h) ? h->last_error.c_str() : "not a live handle";
}

// ------------------------------------------------------- no-alloc step --
// A decode step whose working memory (residual stream, q/k/v, attention
// output and split partials, FFN activations, grid counters, argmax and error
// words) comes from one fixed device array of this library instead of
// buffers of the handle.  It is for callers that must not allocate device
// memory while serving: a process that has handed the rest of the device to
// its own pool (KV pages, other models) and runs out of room or is not
// allowed to grow after start-up.  The call itself allocates nothing (no
// cudaMalloc, no cudaFree, no allocating library routine); the handle's
// weights, KV cache and pinned host words were set up by llm_create.
//
// The array is shared by every handle on a device, so calls that overlap in
// time (other threads, other streams, other handles on the same device) race
// on it and must be serialised by the caller.  The first call on a device
// looks up the array's address (cudaGetSymbolAddress, with that device
// current); make that first call before any stream capture begins.
constexpr size_t kStaticScratchBytes = (size_t)16 << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_step_scratch[kStaticScratchBytes];

namespace {
std::mutex g_scratch_mu;
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};

size_t scratch_align(size_t b) { return (b + 255) & ~(size_t)255; }

// Scratch layout of a handle's step: offsets in bytes, total in *bytes.
struct ScratchLayout {
    size_t epoch, tv, tv_bytes, part, part_bytes, delta, delta_bytes, best, counters, err, total;
};

ScratchLayout scratch_layout(const llm_handle* h) {
    ScratchLayout s{};
    size_t o = 0;
    auto take = [&](size_t b) { size_t at = o; o += scratch_align(b); return at; };
    s.epoch = take(4);                                  // shared by every handle: tags only grow
    s.tv_bytes = h->tv_words * 8;
    s.tv = take(s.tv_bytes);
    s.part_bytes = h->part_words * 8;
    s.part = take(s.part_bytes);
    s.delta_bytes = h->delta_words * 8;
    s.delta = take(s.delta_bytes);                      // cleared before every call
    s.best = take(8);                                   // these three must start at zero
    s.counters = take((size_t)h->n_counters * 4);
    s.err = take(4);
    s.total = o;
    return s;
}
}  // namespace

extern "C" int llm_decode_step_noalloc(llm_handle* h, const int32_t* token_dev, int32_t pos, float* logits_dev,
                                       int32_t* argmax_dev) {
    LIVE_OR_RETURN(h);
    if (!token_dev || !logits_dev || !argmax_dev) return fail(h, LLM_ERR_INVALID_ARG, "NULL argument");
    if (h->broken) return fail(h, LLM_ERR_STATE, "handle has a device error; call llm_reset");
    if (pos < 0 || pos >= h->cfg.max_seq) return fail(h, LLM_ERR_OUT_OF_RANGE, "pos %d not in [0, %d)", pos, h->cfg.max_seq);
    if (h->device < 0 || h->device >= kMaxDevices) return fail(h, LLM_ERR_UNSUPPORTED, "device %d", h->device);
    const ScratchLayout sl = scratch_layout(h);
    if (sl.total > kStaticScratchBytes)
        return fail(h, LLM_ERR_UNSUPPORTED, "this model's step needs %zu bytes of scratch; the static scratch holds %zu",
                    sl.total, kStaticScratchBytes);
    unsigned char* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_addr[h->device]) {
            int prev = -1;
            CK(h, cudaGetDevice(&prev));
            if (prev != h->device) CK(h, cudaSetDevice(h->device));
            void* a = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&a, g_step_scratch);
            if (prev != h->device) cudaSetDevice(prev);
            if (e != cudaSuccess || !a)
                return fail(h, LLM_ERR_CUDA, "cudaGetSymbolAddress of the step scratch: %s", cudaGetErrorString(e));
            g_scratch_addr[h->device] = a;
        }
        base = static_cast<unsigned char*>(g_scratch_addr[h->device]);
    }
    // argmax key, grid counter and error word start at zero (contiguous); the
    // residual accumulators too (another handle's steps cleared only their
    // own layout's words)
    CK(h, cudaMemsetAsync(base + sl.best, 0, sl.err + 4 - sl.best, h->st));
    CK(h, cudaMemsetAsync(base + sl.delta, 0, sl.delta_bytes, h->st));

    StepParams p = step_params(h, token_dev, pos, argmax_dev);
    p.trace = nullptr;
    p.tv = reinterpret_cast<unsigned long long*>(base + sl.tv);
    p.part = reinterpret_cast<unsigned long long*>(base + sl.part);
    p.delta = reinterpret_cast<unsigned long long*>(base + sl.delta);
    p.epoch = reinterpret_cast<unsigned*>(base + sl.epoch);
    p.logits = logits_dev;
    p.best = reinterpret_cast<unsigned long long*>(base + sl.best);
    p.counters = reinterpret_cast<unsigned*>(base + sl.counters);
    p.err = reinterpret_cast<int*>(base + sl.err);
    void* args[] = {&p};
    CK(h, cudaLaunchCooperativeKernel(h->kernel, dim3(h->sms), dim3(kBlock), args, h->smem, h->st));
    h->launches++;
    CK(h, cudaMemcpyAsync(&h->pinned->err, base + sl.err, 4, cudaMemcpyDeviceToHost, h->st));
    CK(h, cudaStreamSynchronize(h->st));
    const int e = h->pinned->err;
    if (e) {
        // a step that stopped early may have left words with the next step's tag
        CK(h, cudaMemsetAsync(base + sl.tv, 0, sl.tv_bytes, h->st));
        CK(h, cudaMemsetAsync(base + sl.part, 0, sl.part_bytes, h->st));
        CK(h, cudaStreamSynchronize(h->st));
    }
    return device_error_status(h, e);
}
