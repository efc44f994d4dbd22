// GGUF model files: a native reader of the version-3 layout described in
// "Loading GGUF with the FFM API" (codeloopback.dev, llm-gguf-loader-ffm) and
// the model shape and tensor names of "The Forward Pass in Java" (Examples 1
// and 13).  Host code only: the file is memory-mapped read-only, parsed and
// checked once at open; tensors are handed out as views into the mapping, and
// llm_create_from_gguf stages the ones a handle needs on the device.
#include <errno.h>
#include <fcntl.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/llm.h"

namespace llm {
int check_shape(const llm_config* c, std::string* why);   // llm_api.cu: llm_create's shape checks
cudaError_t dev_alloc(void** p, size_t bytes);             // llm_api.cu: the library's device allocations
}

namespace {

constexpr uint32_t kMagic = 0x46554747;        // "GGUF" read as a little-endian uint32 (Example 1)
constexpr uint32_t kVersion = 3;               // the version this reader accepts (Example 11)
constexpr uint64_t kDefaultAlignment = 32;     // when general.alignment is absent (Example 5)
constexpr int kMaxDims = 4;                    // ggml tensors have at most four dimensions

void put_err(char* err, size_t len, const char* fmt, ...) {
    if (!err || !len) return;
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(err, len, fmt, ap);
    va_end(ap);
}

// Little-endian reads from the mapping, each one bounds-checked.  A failed
// read sets `bad` and returns zeros; the caller checks `bad` once per item.
struct Cursor {
    const uint8_t* base;
    uint64_t size, pos = 0;
    bool bad = false;
    bool need(uint64_t n) {
        if (bad || n > size || pos > size - n) { bad = true; return false; }
        return true;
    }
    template <class T>
    T get() {
        T v{};
        if (need(sizeof(T))) { memcpy(&v, base + pos, sizeof(T)); pos += sizeof(T); }
        return v;
    }
    // A string: uint64 byte length, then that many UTF-8 bytes (Example 4).
    void str(uint64_t& at, uint64_t& len) {
        len = get<uint64_t>();
        at = pos;
        if (need(len)) pos += len;
    }
};

uint64_t scalar_size(int32_t t) {
    switch (t) {
        case LLM_GGUF_UINT8: case LLM_GGUF_INT8: case LLM_GGUF_BOOL: return 1;
        case LLM_GGUF_UINT16: case LLM_GGUF_INT16: return 2;
        case LLM_GGUF_UINT32: case LLM_GGUF_INT32: case LLM_GGUF_FLOAT32: return 4;
        case LLM_GGUF_UINT64: case LLM_GGUF_INT64: case LLM_GGUF_FLOAT64: return 8;
        default: return 0;
    }
}

struct Meta {
    std::string key;
    int32_t type = 0;
    int32_t elem_type = -1;     // arrays
    uint64_t count = 0;         // arrays: elements; strings: bytes
    uint64_t at = 0;            // file offset of the value (strings: of the bytes; arrays: of the first element)
};

struct Tensor {
    std::string name;
    int32_t type = 0, n_dims = 0;
    int64_t dims[kMaxDims] = {1, 1, 1, 1};
    uint64_t offset = 0, bytes = 0;
};

// Skips one value of type t (arrays recursively).
bool skip_value(Cursor& c, int32_t t, int depth) {
    if (t == LLM_GGUF_STRING) {
        uint64_t at, len;
        c.str(at, len);
        return !c.bad;
    }
    if (t == LLM_GGUF_ARRAY) {
        if (depth > 8) return false;
        const int32_t et = (int32_t)c.get<uint32_t>();
        const uint64_t n = c.get<uint64_t>();
        if (c.bad) return false;
        const uint64_t es = scalar_size(et);
        if (es) {
            if (n > c.size / es || !c.need(n * es)) {
                c.bad = true;
                return false;
            }
            c.pos += n * es;
            return true;
        }
        if (et != LLM_GGUF_STRING && et != LLM_GGUF_ARRAY) return false;
        for (uint64_t i = 0; i < n; i++)
            if (!skip_value(c, et, depth + 1)) return false;
        return true;
    }
    const uint64_t s = scalar_size(t);
    if (!s) return false;
    c.need(s);
    if (!c.bad) c.pos += s;
    return !c.bad;
}

// Bytes of a tensor (Example 13, TensorInfo.byteSize): F32 4 per value, F16
// 2, Q8_0 34 per 32-value block; 0 for a type this reader does not handle.
uint64_t tensor_bytes(const Tensor& t, bool& overflow) {
    uint64_t n = 1;
    for (int d = 0; d < t.n_dims; d++) {
        if (t.dims[d] < 0 || (t.dims[d] && n > UINT64_MAX / 64 / (uint64_t)t.dims[d])) overflow = true;
        n *= (uint64_t)t.dims[d];
    }
    switch (t.type) {
        case LLM_F32: return 4 * n;
        case LLM_F16: return 2 * n;
        case LLM_Q8_0: return n / 32 * 34;
        default: return 0;
    }
}

uint64_t pad(uint64_t n, uint64_t a) { return (n + a - 1) / a * a; }

}  // namespace

struct llm_gguf {
    int fd = -1;
    const uint8_t* map = nullptr;
    uint64_t size = 0;
    uint32_t version = 0;
    uint64_t alignment = kDefaultAlignment, infos_end = 0, data_start = 0;
    std::vector<Meta> meta;
    std::vector<Tensor> tensors;

    const Meta* find_meta(const char* key) const {
        for (const Meta& m : meta)
            if (m.key == key) return &m;
        return nullptr;
    }
    const Tensor* find_tensor(const char* name) const {
        for (const Tensor& t : tensors)
            if (t.name == name) return &t;
        return nullptr;
    }
};

namespace {

// Parse and check the mapped file in the loader page's order (Example 11):
// the 24-byte header, the magic, the version, then the metadata and tensor
// infos, the alignment, each tensor's type and offset (the padded sizes of
// the tensors before it) and each tensor's end against the file size.
int parse(llm_gguf* g, char* err, size_t err_len) {
    if (g->size < 24) {
        put_err(err, err_len, "shorter than the 24-byte header");
        return LLM_ERR_INVALID_ARG;
    }
    Cursor c{g->map, g->size};
    const uint32_t magic = c.get<uint32_t>();
    if (magic != kMagic) {
        put_err(err, err_len, "magic 0x%08X is not GGUF", magic);
        return LLM_ERR_INVALID_ARG;
    }
    g->version = c.get<uint32_t>();
    if (g->version != kVersion) {
        put_err(err, err_len, "version %u (this loader reads %u)", g->version, kVersion);
        return LLM_ERR_UNSUPPORTED;
    }
    const uint64_t n_tensors = c.get<uint64_t>(), n_kv = c.get<uint64_t>();
    // every key-value pair and tensor info takes at least 12 / 24 bytes
    if (n_kv > g->size / 12 || n_tensors > g->size / 24) {
        put_err(err, err_len, "counts larger than the file (%llu tensors, %llu keys)",
                (unsigned long long)n_tensors, (unsigned long long)n_kv);
        return LLM_ERR_INVALID_ARG;
    }
    g->meta.reserve(n_kv);
    for (uint64_t i = 0; i < n_kv; i++) {
        Meta m;
        uint64_t at, len;
        c.str(at, len);
        if (c.bad) break;
        m.key.assign(reinterpret_cast<const char*>(g->map + at), len);
        m.type = (int32_t)c.get<uint32_t>();
        if (c.bad) break;
        if (m.type == LLM_GGUF_STRING) {
            c.str(m.at, m.count);
        } else if (m.type == LLM_GGUF_ARRAY) {
            const uint64_t p = c.pos;
            m.elem_type = (int32_t)c.get<uint32_t>();
            m.count = c.get<uint64_t>();
            m.at = c.pos;
            c.pos = p;
            if (!c.bad && !skip_value(c, LLM_GGUF_ARRAY, 0)) {
                if (!c.bad) {
                    put_err(err, err_len, "bad array element type %d for key %s", m.elem_type, m.key.c_str());
                    return LLM_ERR_INVALID_ARG;
                }
            }
        } else {
            if (!scalar_size(m.type)) {
                put_err(err, err_len, "bad value type %d for key %s", m.type, m.key.c_str());
                return LLM_ERR_INVALID_ARG;
            }
            m.at = c.pos;
            skip_value(c, m.type, 0);
        }
        if (c.bad) break;
        g->meta.push_back(std::move(m));
    }
    if (c.bad) {
        put_err(err, err_len, "metadata runs past the end of the file");
        return LLM_ERR_INVALID_ARG;
    }
    g->tensors.reserve(n_tensors);
    for (uint64_t i = 0; i < n_tensors; i++) {
        Tensor t;
        uint64_t at, len;
        c.str(at, len);
        if (c.bad) break;
        t.name.assign(reinterpret_cast<const char*>(g->map + at), len);
        const uint32_t nd = c.get<uint32_t>();
        if (c.bad) break;
        if (nd < 1 || nd > (uint32_t)kMaxDims) {
            put_err(err, err_len, "tensor %s has %u dimensions", t.name.c_str(), nd);
            return LLM_ERR_INVALID_ARG;
        }
        t.n_dims = (int32_t)nd;
        for (uint32_t d = 0; d < nd; d++) t.dims[d] = (int64_t)c.get<uint64_t>();
        t.type = (int32_t)c.get<uint32_t>();
        t.offset = c.get<uint64_t>();
        if (c.bad) break;
        g->tensors.push_back(std::move(t));
    }
    if (c.bad) {
        put_err(err, err_len, "tensor infos run past the end of the file");
        return LLM_ERR_INVALID_ARG;
    }
    g->infos_end = c.pos;
    if (const Meta* a = g->find_meta("general.alignment")) {
        uint32_t v = 0;
        if (a->type == LLM_GGUF_UINT32) memcpy(&v, g->map + a->at, 4);
        if (a->type != LLM_GGUF_UINT32 || v == 0) {
            put_err(err, err_len, "general.alignment must be a nonzero UINT32");
            return LLM_ERR_INVALID_ARG;
        }
        g->alignment = v;
    }
    g->data_start = pad(g->infos_end, g->alignment);
    uint64_t expect = 0;
    for (size_t i = 0; i < g->tensors.size(); i++) {
        Tensor& t = g->tensors[i];
        bool overflow = false;
        t.bytes = tensor_bytes(t, overflow);
        if (overflow) {
            put_err(err, err_len, "tensor %s is larger than the file", t.name.c_str());
            return LLM_ERR_INVALID_ARG;
        }
        if (t.type != LLM_F32 && t.type != LLM_F16 && t.type != LLM_Q8_0) {
            put_err(err, err_len, "unsupported ggml type %d for %s", t.type, t.name.c_str());
            return LLM_ERR_UNSUPPORTED;
        }
        if (t.type == LLM_Q8_0 && t.dims[0] % 32) {
            put_err(err, err_len, "Q8_0 rows of %lld values are not whole 32-value blocks", (long long)t.dims[0]);
            return LLM_ERR_INVALID_ARG;
        }
        if (t.offset != expect) {
            if (i == 0)
                put_err(err, err_len, "first tensor offset %llu, expected %llu", (unsigned long long)t.offset,
                        (unsigned long long)expect);
            else
                put_err(err, err_len, "tensor %s offset %llu, expected %llu", t.name.c_str(),
                        (unsigned long long)t.offset, (unsigned long long)expect);
            return LLM_ERR_INVALID_ARG;
        }
        expect += pad(t.bytes, g->alignment);
    }
    for (const Tensor& t : g->tensors) {
        const uint64_t end = g->data_start + t.offset + t.bytes;
        if (end > g->size || end < t.bytes) {
            put_err(err, err_len, "tensor needs bytes up to %llu, file has %llu", (unsigned long long)end,
                    (unsigned long long)g->size);
            return LLM_ERR_INVALID_ARG;
        }
    }
    return LLM_OK;
}

bool meta_int(const llm_gguf* g, const std::string& key, int64_t& v) {
    const Meta* m = g->find_meta(key.c_str());
    return m && llm_gguf_meta_int(g, key.c_str(), &v) == LLM_OK;
}

bool meta_float(const llm_gguf* g, const std::string& key, double& v) {
    const Meta* m = g->find_meta(key.c_str());
    return m && llm_gguf_meta_float(g, key.c_str(), &v) == LLM_OK;
}

}  // namespace

extern "C" int llm_gguf_open(const char* path, llm_gguf** out, char* err, size_t err_len) {
    if (out) *out = nullptr;
    if (!path || !out) {
        put_err(err, err_len, "path or out is NULL");
        return LLM_ERR_INVALID_ARG;
    }
    const int fd = open(path, O_RDONLY | O_CLOEXEC);
    if (fd < 0) {
        put_err(err, err_len, "cannot open %s: %s", path, strerror(errno));
        return LLM_ERR_INVALID_ARG;
    }
    struct stat st;
    if (fstat(fd, &st) != 0) {
        put_err(err, err_len, "cannot stat %s: %s", path, strerror(errno));
        close(fd);
        return LLM_ERR_INVALID_ARG;
    }
    if (!S_ISREG(st.st_mode)) {
        put_err(err, err_len, "%s is not a regular file", path);
        close(fd);
        return LLM_ERR_INVALID_ARG;
    }
    llm_gguf* g = new llm_gguf();
    g->fd = fd;
    g->size = (uint64_t)st.st_size;
    if (g->size) {
        void* p = mmap(nullptr, g->size, PROT_READ, MAP_PRIVATE, fd, 0);
        if (p == MAP_FAILED) {
            put_err(err, err_len, "cannot map %s: %s", path, strerror(errno));
            llm_gguf_close(g);
            return LLM_ERR_NO_MEMORY;
        }
        g->map = static_cast<const uint8_t*>(p);
    }
    const int rc = parse(g, err, err_len);
    if (rc != LLM_OK) {
        llm_gguf_close(g);
        return rc;
    }
    *out = g;
    return LLM_OK;
}

extern "C" void llm_gguf_close(llm_gguf* g) {
    if (!g) return;
    if (g->map) munmap(const_cast<uint8_t*>(g->map), g->size);
    if (g->fd >= 0) close(g->fd);
    delete g;
}

extern "C" int llm_gguf_summary(const llm_gguf* g, llm_gguf_layout* s) {
    if (!g || !s) return LLM_ERR_INVALID_ARG;
    s->version = g->version;
    s->n_tensors = (int64_t)g->tensors.size();
    s->n_kv = (int64_t)g->meta.size();
    s->alignment = g->alignment;
    s->infos_end = g->infos_end;
    s->data_start = g->data_start;
    s->file_size = g->size;
    return LLM_OK;
}

static void fill_tensor(const llm_gguf* g, const Tensor& t, llm_gguf_tensor* o) {
    o->type = t.type;
    o->n_dims = t.n_dims;
    for (int d = 0; d < kMaxDims; d++) o->dims[d] = t.dims[d];
    o->offset = t.offset;
    o->file_offset = g->data_start + t.offset;
    o->bytes = t.bytes;
    o->data = g->map + g->data_start + t.offset;
}

extern "C" int llm_gguf_find_tensor(const llm_gguf* g, const char* name, llm_gguf_tensor* t) {
    if (!g || !name || !t) return LLM_ERR_INVALID_ARG;
    const Tensor* x = g->find_tensor(name);
    if (!x) return LLM_ERR_OUT_OF_RANGE;
    fill_tensor(g, *x, t);
    return LLM_OK;
}

extern "C" int llm_gguf_tensor_at(const llm_gguf* g, int64_t i, const char** name, llm_gguf_tensor* t) {
    if (!g || !name || !t) return LLM_ERR_INVALID_ARG;
    if (i < 0 || i >= (int64_t)g->tensors.size()) return LLM_ERR_OUT_OF_RANGE;
    *name = g->tensors[(size_t)i].name.c_str();
    fill_tensor(g, g->tensors[(size_t)i], t);
    return LLM_OK;
}

extern "C" int llm_gguf_meta_at(const llm_gguf* g, int64_t i, const char** key, int32_t* type) {
    if (!g || !key || !type) return LLM_ERR_INVALID_ARG;
    if (i < 0 || i >= (int64_t)g->meta.size()) return LLM_ERR_OUT_OF_RANGE;
    *key = g->meta[(size_t)i].key.c_str();
    *type = g->meta[(size_t)i].type;
    return LLM_OK;
}

extern "C" int llm_gguf_meta_type(const llm_gguf* g, const char* key, int32_t* type, int32_t* elem_type,
                                  uint64_t* count) {
    if (!g || !key) return LLM_ERR_INVALID_ARG;
    const Meta* m = g->find_meta(key);
    if (!m) return LLM_ERR_OUT_OF_RANGE;
    if (type) *type = m->type;
    if (elem_type) *elem_type = m->elem_type;
    if (count) *count = m->type == LLM_GGUF_ARRAY || m->type == LLM_GGUF_STRING ? m->count : 1;
    return LLM_OK;
}

extern "C" int llm_gguf_meta_int(const llm_gguf* g, const char* key, int64_t* out) {
    if (!g || !key || !out) return LLM_ERR_INVALID_ARG;
    const Meta* m = g->find_meta(key);
    if (!m) return LLM_ERR_OUT_OF_RANGE;
    const uint8_t* p = g->map + m->at;
    switch (m->type) {
        case LLM_GGUF_UINT8: case LLM_GGUF_BOOL: *out = p[0]; break;
        case LLM_GGUF_INT8: *out = (int8_t)p[0]; break;
        case LLM_GGUF_UINT16: { uint16_t v; memcpy(&v, p, 2); *out = v; break; }
        case LLM_GGUF_INT16: { int16_t v; memcpy(&v, p, 2); *out = v; break; }
        case LLM_GGUF_UINT32: { uint32_t v; memcpy(&v, p, 4); *out = v; break; }
        case LLM_GGUF_INT32: { int32_t v; memcpy(&v, p, 4); *out = v; break; }
        case LLM_GGUF_UINT64: {
            uint64_t v;
            memcpy(&v, p, 8);
            if (v > (uint64_t)INT64_MAX) return LLM_ERR_OUT_OF_RANGE;
            *out = (int64_t)v;
            break;
        }
        case LLM_GGUF_INT64: { int64_t v; memcpy(&v, p, 8); *out = v; break; }
        default: return LLM_ERR_INVALID_ARG;
    }
    return LLM_OK;
}

extern "C" int llm_gguf_meta_float(const llm_gguf* g, const char* key, double* out) {
    if (!g || !key || !out) return LLM_ERR_INVALID_ARG;
    const Meta* m = g->find_meta(key);
    if (!m) return LLM_ERR_OUT_OF_RANGE;
    const uint8_t* p = g->map + m->at;
    if (m->type == LLM_GGUF_FLOAT32) {
        float v;
        memcpy(&v, p, 4);
        *out = v;
    } else if (m->type == LLM_GGUF_FLOAT64) {
        memcpy(out, p, 8);
    } else {
        return LLM_ERR_INVALID_ARG;
    }
    return LLM_OK;
}

extern "C" int llm_gguf_meta_string(const llm_gguf* g, const char* key, const char** s, uint64_t* len) {
    if (!g || !key || !s || !len) return LLM_ERR_INVALID_ARG;
    const Meta* m = g->find_meta(key);
    if (!m) return LLM_ERR_OUT_OF_RANGE;
    if (m->type != LLM_GGUF_STRING) return LLM_ERR_INVALID_ARG;
    *s = reinterpret_cast<const char*>(g->map + m->at);
    *len = m->count;
    return LLM_OK;
}

// The model shape from the metadata ("The Forward Pass in Java", Example 1):
// keys under general.architecture's prefix, the page's defaults for the
// optional ones, the RoPE pair layout by architecture (llama normal, qwen2
// NEOX), the weight type of token_embd.weight.
extern "C" int llm_gguf_config(const llm_gguf* g, int32_t max_seq, llm_config* cfg, char* err, size_t err_len) {
    if (!g || !cfg) {
        put_err(err, err_len, "gguf or cfg is NULL");
        return LLM_ERR_INVALID_ARG;
    }
    const char* as;
    uint64_t alen;
    if (llm_gguf_meta_string(g, "general.architecture", &as, &alen) != LLM_OK) {
        put_err(err, err_len, "no general.architecture string");
        return LLM_ERR_INVALID_ARG;
    }
    const std::string a(as, alen);
    if (a != "llama" && a != "qwen2") {
        put_err(err, err_len, "architecture not supported here: %s", a.c_str());
        return LLM_ERR_UNSUPPORTED;
    }
    int64_t dim, layers, heads, kv_heads, ffn, ctx, vocab, rope_dims;
    double eps, base = 10000.0;
    const char* missing = nullptr;
    if (!meta_int(g, a + ".embedding_length", dim)) missing = "embedding_length";
    else if (!meta_int(g, a + ".block_count", layers)) missing = "block_count";
    else if (!meta_int(g, a + ".attention.head_count", heads)) missing = "attention.head_count";
    else if (!meta_int(g, a + ".feed_forward_length", ffn)) missing = "feed_forward_length";
    else if (!meta_int(g, a + ".context_length", ctx)) missing = "context_length";
    else if (!meta_float(g, a + ".attention.layer_norm_rms_epsilon", eps)) missing = "attention.layer_norm_rms_epsilon";
    if (missing) {
        put_err(err, err_len, "missing or mistyped key %s.%s", a.c_str(), missing);
        return LLM_ERR_INVALID_ARG;
    }
    if (heads <= 0 || dim <= 0) {
        put_err(err, err_len, "head_count and embedding_length must be positive");
        return LLM_ERR_INVALID_ARG;
    }
    if (!meta_int(g, a + ".attention.head_count_kv", kv_heads)) kv_heads = heads;
    if (g->find_meta((a + ".rope.freq_base").c_str()) && !meta_float(g, a + ".rope.freq_base", base)) {
        put_err(err, err_len, "%s.rope.freq_base is not a float", a.c_str());
        return LLM_ERR_INVALID_ARG;
    }
    if (!meta_int(g, a + ".rope.dimension_count", rope_dims)) rope_dims = dim / heads;
    if (!meta_int(g, a + ".vocab_size", vocab)) {
        int32_t t, et;
        uint64_t n;
        if (llm_gguf_meta_type(g, "tokenizer.ggml.tokens", &t, &et, &n) != LLM_OK || t != LLM_GGUF_ARRAY) {
            put_err(err, err_len, "no %s.vocab_size and no tokenizer.ggml.tokens array", a.c_str());
            return LLM_ERR_INVALID_ARG;
        }
        vocab = (int64_t)n;
    }
    const Tensor* embd = g->find_tensor("token_embd.weight");
    if (!embd) {
        put_err(err, err_len, "no token_embd.weight tensor");
        return LLM_ERR_INVALID_ARG;
    }
    const int64_t lim = INT32_MAX;
    if (dim > lim || layers > lim || heads > lim || kv_heads > lim || ffn > lim || ctx > lim || vocab > lim ||
        rope_dims > lim || layers < 0 || kv_heads < 0 || ffn < 0 || ctx < 0 || vocab < 0 || rope_dims < 0) {
        put_err(err, err_len, "a shape key is out of range");
        return LLM_ERR_INVALID_ARG;
    }
    cfg->n_layers = (int)layers;
    cfg->dim = (int)dim;
    cfg->n_heads = (int)heads;
    cfg->n_kv_heads = (int)kv_heads;
    cfg->head_dim = (int)(dim / heads);
    cfg->ffn_dim = (int)ffn;
    cfg->vocab = (int)vocab;
    cfg->max_seq = max_seq > 0 ? max_seq : (int)ctx;
    cfg->rope_dims = (int)rope_dims;
    cfg->eps = (float)eps;
    cfg->rope_base = (float)base;
    cfg->rope_neox = a == "qwen2";
    cfg->wtype = embd->type;
    cfg->numerics = LLM_NUMERICS_EXACT;
    return LLM_OK;
}

// The handle of a GGUF model: the tensors of "The Forward Pass in Java",
// Example 13 (token_embd, output_norm, optional output (tied otherwise),
// optional rope_freqs, and per layer blk.N.attn_norm, attn_q/k/v (+ optional
// biases), attn_output, ffn_norm, ffn_gate, ffn_up, ffn_down), each checked
// for its type and shape, staged on the device and handed to llm_create.
extern "C" int llm_create_from_gguf(const llm_gguf* g, int32_t max_seq, llm_stream_t stream, llm_handle** out,
                                    char* err, size_t err_len) {
    if (out) *out = nullptr;
    if (!g || !out) {
        put_err(err, err_len, "gguf or out is NULL");
        return LLM_ERR_INVALID_ARG;
    }
    llm_config cfg;
    int rc = llm_gguf_config(g, max_seq, &cfg, err, err_len);
    if (rc != LLM_OK) return rc;
    {
        // a shape the kernels cannot run is rejected before any tensor is staged on the device
        std::string why;
        rc = llm::check_shape(&cfg, &why);
        if (rc != LLM_OK) {
            put_err(err, err_len, "llm_create: %s", why.c_str());
            return rc;
        }
    }
    // every block needs 9 tensors (norms, q/k/v/o, gate/up/down) and the model
    // 2 more: a block count the file's tensors cannot back is refused before
    // the list of wanted tensors is built
    if ((int64_t)cfg.n_layers * 9 + 2 > (int64_t)g->tensors.size()) {
        put_err(err, err_len, "block_count %d needs at least %lld tensors; the file has %zu", cfg.n_layers,
                (long long)cfg.n_layers * 9 + 2, g->tensors.size());
        return LLM_ERR_INVALID_ARG;
    }
    const int wt = cfg.wtype;
    const int64_t q_dim = (int64_t)cfg.n_heads * cfg.head_dim, kv_dim = (int64_t)cfg.n_kv_heads * cfg.head_dim;
    struct Need {
        std::string name;
        bool matrix, optional;
        int64_t d0, d1;             // dims: [d0] for vectors, [d0, d1] for matrices
        const Tensor* t = nullptr;
        size_t at = 0;              // offset in the staging buffer
    };
    std::vector<Need> need;
    auto add = [&](const std::string& n, bool matrix, bool optional, int64_t d0, int64_t d1) {
        need.push_back(Need{n, matrix, optional, d0, d1});
    };
    add("token_embd.weight", true, false, cfg.dim, cfg.vocab);
    add("output_norm.weight", false, false, cfg.dim, 0);
    add("output.weight", true, true, cfg.dim, cfg.vocab);
    add("rope_freqs.weight", false, true, cfg.rope_dims / 2, 0);
    for (int l = 0; l < cfg.n_layers; l++) {
        const std::string p = "blk." + std::to_string(l) + ".";
        add(p + "attn_norm.weight", false, false, cfg.dim, 0);
        add(p + "attn_q.weight", true, false, cfg.dim, q_dim);
        add(p + "attn_k.weight", true, false, cfg.dim, kv_dim);
        add(p + "attn_v.weight", true, false, cfg.dim, kv_dim);
        add(p + "attn_q.bias", false, true, q_dim, 0);
        add(p + "attn_k.bias", false, true, kv_dim, 0);
        add(p + "attn_v.bias", false, true, kv_dim, 0);
        add(p + "attn_output.weight", true, false, q_dim, cfg.dim);
        add(p + "ffn_norm.weight", false, false, cfg.dim, 0);
        add(p + "ffn_gate.weight", true, false, cfg.dim, cfg.ffn_dim);
        add(p + "ffn_up.weight", true, false, cfg.dim, cfg.ffn_dim);
        add(p + "ffn_down.weight", true, false, cfg.ffn_dim, cfg.dim);
    }
    size_t total = 0;
    for (Need& n : need) {
        n.t = g->find_tensor(n.name.c_str());
        if (!n.t) {
            if (n.optional) continue;
            put_err(err, err_len, "no %s tensor", n.name.c_str());
            return LLM_ERR_INVALID_ARG;
        }
        const Tensor& t = *n.t;
        const bool shape_ok = n.matrix ? (t.n_dims == 2 && t.dims[0] == n.d0 && t.dims[1] == n.d1)
                                       : (t.n_dims == 1 && t.dims[0] == n.d0);
        if (!shape_ok) {
            put_err(err, err_len, "%s has dims [%lld, %lld], expected [%lld%s%lld]", n.name.c_str(),
                    (long long)t.dims[0], (long long)(t.n_dims > 1 ? t.dims[1] : 0), (long long)n.d0,
                    n.matrix ? ", " : "", (long long)(n.matrix ? n.d1 : 0));
            return LLM_ERR_INVALID_ARG;
        }
        if (n.matrix ? t.type != wt : t.type != LLM_F32) {
            put_err(err, err_len, "%s has ggml type %d, expected %d", n.name.c_str(), t.type,
                    n.matrix ? wt : (int)LLM_F32);
            return LLM_ERR_UNSUPPORTED;
        }
        n.at = total;
        total += (t.bytes + 255) & ~(size_t)255;
    }
    uint8_t* stage = nullptr;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t ce = llm::dev_alloc(reinterpret_cast<void**>(&stage), total ? total : 256);
    if (ce != cudaSuccess) {
        put_err(err, err_len, "staging %zu bytes: %s", total, cudaGetErrorString(ce));
        return ce == cudaErrorMemoryAllocation ? LLM_ERR_NO_MEMORY : LLM_ERR_CUDA;
    }
    for (const Need& n : need) {
        if (!n.t) continue;
        ce = cudaMemcpyAsync(stage + n.at, g->map + g->data_start + n.t->offset, n.t->bytes, cudaMemcpyHostToDevice,
                             st);
        if (ce != cudaSuccess) break;
    }
    if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
    if (ce != cudaSuccess) {
        put_err(err, err_len, "staging the tensors: %s", cudaGetErrorString(ce));
        cudaFree(stage);
        return LLM_ERR_CUDA;
    }
    auto dev = [&](const std::string& name) -> const void* {
        for (const Need& n : need)
            if (n.name == name) return n.t ? stage + n.at : nullptr;
        return nullptr;
    };
    std::vector<llm_layer_weights> lw((size_t)cfg.n_layers);
    for (int l = 0; l < cfg.n_layers; l++) {
        const std::string p = "blk." + std::to_string(l) + ".";
        llm_layer_weights& L = lw[(size_t)l];
        L.attn_norm = static_cast<const float*>(dev(p + "attn_norm.weight"));
        L.ffn_norm = static_cast<const float*>(dev(p + "ffn_norm.weight"));
        L.bq = static_cast<const float*>(dev(p + "attn_q.bias"));
        L.bk = static_cast<const float*>(dev(p + "attn_k.bias"));
        L.bv = static_cast<const float*>(dev(p + "attn_v.bias"));
        L.wq = dev(p + "attn_q.weight");
        L.wk = dev(p + "attn_k.weight");
        L.wv = dev(p + "attn_v.weight");
        L.wo = dev(p + "attn_output.weight");
        L.w_gate = dev(p + "ffn_gate.weight");
        L.w_up = dev(p + "ffn_up.weight");
        L.w_down = dev(p + "ffn_down.weight");
    }
    llm_weights w;
    w.tok_embd = dev("token_embd.weight");
    w.output_norm = static_cast<const float*>(dev("output_norm.weight"));
    w.output = dev("output.weight");
    w.rope_freqs = static_cast<const float*>(dev("rope_freqs.weight"));
    w.layers = lw.data();
    rc = llm_create(&cfg, &w, stream, out);
    if (rc != LLM_OK) put_err(err, err_len, "llm_create: %s", llm_last_error(nullptr));
    // llm_create copies every tensor into the handle's own layout before it returns
    cudaStreamSynchronize(st);
    cudaFree(stage);
    return rc;
}
