// Internal device layouts and helpers of libllmdecode (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/llm.h"

namespace llm {

constexpr int kThreads = 512;          // threads per CTA of the decode step kernel
constexpr int kWarps = kThreads / 32;
constexpr int kAttnChunk = 64;         // KV positions staged in shared memory at a time
constexpr int kMaxGroupDim = 1024;     // (n_heads / n_kv_heads) * head_dim handled per attention unit

// Device error word values (sticky until llm_reset).
enum : int { kErrNone = 0, kErrTimeout = 1, kErrToken = 2 };

// A weight matrix in the library's layout.  Row r of a Q8_0 matrix is `cols`
// int8 quants at q + r*cols and cols/32 FP16 scales at d + r*(cols/32); F16 and
// F32 matrices are `rows` rows of `cols` values at q (d unused).
struct DMat {
    const uint8_t* q;
    const __half* d;
    int rows, cols;
};

struct LayerDev {
    DMat qkv;                 // rows: q (n_heads*hd), k (kv_dim), v (kv_dim)
    DMat o;                   // [q_dim -> dim]
    DMat gu;                  // interleaved: row 2i = gate row i, row 2i+1 = up row i
    DMat down;                // [ffn -> dim]
    const float* attn_norm;
    const float* ffn_norm;
    const float* qkv_bias;    // [q_dim + 2 kv_dim] or nullptr
    __half* kc;               // [max_seq][kv_dim]
    __half* vc;
};

// Counters of one step: 5 phases per layer + the logits phase, then one merge
// counter per (layer, kv head).  All zero between steps.
struct StepParams {
    const LayerDev* layers;
    DMat embd;
    DMat out;
    const float* out_norm;
    const float* rope_freqs;  // [rope_dims/2] or nullptr
    int wtype;
    int n_layers, dim, n_heads, n_kv, hd, ffn, vocab, max_seq, rope_dims, neox, q_dim, kv_dim;
    float eps, theta_scale, attn_div;

    float* x;                 // residual stream [dim]
    float* qkv;               // [q_dim + 2 kv_dim]
    float* attn;              // attention output [q_dim]
    float* u;                 // SwiGLU output [ffn]
    float* logits;            // [vocab]
    float* attn_part;         // [n_heads][max_splits][hd + 2]
    int max_splits;
    unsigned long long* best; // packed argmax of the step
    unsigned* counters;
    int* err;

    const int* token_in;
    int* token_out;
    int pos;
    int splits;               // attention splits per kv head for this pos
};

__host__ __device__ inline int n_phase_counters(int n_layers) { return 5 * n_layers + 1; }

// ---------------------------------------------------------------- loads --
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ unsigned short ld_stream_u16(const void* p) {
    unsigned short r;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// int8 (as a byte of w) -> exact float: the byte, offset by 128, is placed in
// the low mantissa bits of 2^23 and the offset float 2^23 + 128 subtracted.
__device__ __forceinline__ float i8_to_f32(uint32_t w_xor80, int k) {
    const uint32_t sel = 0x7540u | (uint32_t)k;
    return __uint_as_float(__byte_perm(w_xor80, 0x4B000000u, sel)) - 8388736.0f;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Argmax key: larger value first, then smaller index.  NaN never wins.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    if (v != v) return 0ull;
    uint32_t b = __float_as_uint(v);
    uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
    return k == 0ull ? 0 : (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
}

}  // namespace llm
