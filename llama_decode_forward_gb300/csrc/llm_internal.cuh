// Internal device layouts and helpers of libllmdecode (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/llm.h"

namespace llm {

// Decode step kernel: one CTA per SM, 15 consumer warps + 1 producer warp
// (16 warps: 4 per SM sub-partition, so up to 128 registers per thread).
constexpr int kConsumerWarps = 15;
constexpr int kConsumers = kConsumerWarps * 32;   // 480
constexpr int kBlock = kConsumers + 32;           // 512
constexpr int kSlotBytes = 65536;                 // one ring slot (a chunk of weight rows or KV rows)
constexpr int kRedFloats = 1024;                  // row partials of one chunk
constexpr int kMaxGroupDim = 2 * kConsumers;      // (n_heads / n_kv_heads) * head_dim per attention unit
// 32-byte column blocks of a row one consumer thread owns: 2 for F16, else 1.
__host__ __device__ inline int max_blocks_per_thread(int wtype) { return wtype == LLM_F16 ? 2 : 1; }
constexpr int kMaxSmem = 232448;                  // 227 KB opt-in dynamic shared memory per CTA

// Device error word bits (sticky until llm_reset).
enum : int { kErrNone = 0, kErrTimeout = 1, kErrToken = 2, kErrRange = 4, kErrCheck = 8 };

// Index checks of LLM_CHECKED builds: a check that fails records kErrCheck in
// the error word and the access it guards is skipped (no trap).  Other builds
// compile the checks away.
#ifdef LLM_CHECKED
#define LLM_IN_BOUNDS(err, cond) ((cond) ? true : (atomicOr((err), kErrCheck), false))
#else
#define LLM_IN_BOUNDS(err, cond) true
#endif

// A weight matrix in the library's layout.  Q8_0: row r is `cols` int8 quants
// at q + r*cols, and cols/32
// FP16 scales at d + r*dstride (dstride = cols/32 rounded up to a multiple of
// 8, so every row of scales is 16-byte aligned).
// F16 / F32: `rows` rows of `cols` values at q.
// Streaming plan (set at creation): a ring slot carries `rpc` rows; a row is
// reduced by a team of `tw` lanes (32 elements per lane; tw <= 32 is a part
// of one warp, tw > 32 is tw/32 whole warps) and `teams` teams work side by side.
// pair = 2 (gate/up): rows 2i and 2i+1 form one "super-row"; `rows` counts
// super-rows (CTAs split the matrix by super-rows, so a gate row and its up
// row stay in one CTA) while the plan (tw, teams, rpc) counts single rows.
struct DMat {
    const uint8_t* q;
    const __half* d;
    int rows, cols, dstride;
    int rpc, tw, teams, pair;
};

// A column-group view of a row-major matrix (Wo, Wdown in the decode step):
// the grid is split into `ngrp` groups of CTAs and group g multiplies columns
// [g*m.cols, (g+1)*m.cols) of the matrix (m.cols = the group's width) by its
// own part of the input vector.  A CTA streams rows of its group's column block
// with TMA: the values as a 3-D tensor view {U, cols/U, rows} (one box of
// {U, m.cols/U, R} per chunk) and, for Q8_0, the scales as a 2-D view
// {dstride, rows} (a box of {SB, R} starting at the group's first scale
// rounded down to a multiple of 8, so the box starts on a 16-byte boundary).
struct GView {
    DMat m;          // streaming plan for m.cols columns (rows = the matrix's rows)
    int R;           // rows per chunk (the boxes' height)
    int U;           // elements in the innermost dimension of the value view
    int rowq;        // bytes of one row of the value box (m.cols * element size)
    int rowd;        // bytes of one row of the scale box (SB * 2), Q8_0
    int sboff;       // byte offset of the scale box in a ring slot
    int box_bytes;   // bytes one chunk delivers (both boxes)
};

struct LayerDev {
    DMat qkv;                 // rows: q (n_heads*hd), k (kv_dim), v (kv_dim)
    DMat o;                   // [q_dim -> dim], row-major (prefill, test hooks)
    DMat gu;                  // interleaved: row 2i = gate row i, row 2i+1 = up row i
    DMat down;                // [ffn -> dim], row-major (prefill, test hooks)
    const float* attn_norm;
    const float* ffn_norm;
    const float* qkv_bias;    // [q_dim + 2 kv_dim] or nullptr
    __half* kc;               // [max_seq][kv_dim]
    __half* vc;
};

// Counters of one step: the end-of-step count only (zero between steps).
//
// Activation vectors that cross the grid are tagged: each element is one
// 64-bit word, the float's bits in the low half and the step's tag in the high
// half, written with one store.  A reader waits until the words it needs carry
// the current tag, so the data is its own ready flag (no separate counter, no
// release/acquire round trip).  Each layer has its own set, each written
// exactly once per step: qkv [q_dim + 2 kv_dim], u [ffn] (silu(gate) * up),
// and the attention partials of every (head, split).
//
// The residual stream is updated through accumulator words: the O and down
// projections of column group g add their partial sums as
// (1 << 56) + round(v * 2^32) with red.add.u64, so a word holds the number of
// groups that have added (top 8 bits) and the exact fixed-point sum of their
// parts (integer addition: the same bits whatever the arrival order).  A
// reader waits until the count equals the number of groups, then adds the sum
// to the residual it keeps in shared memory.  Two parities (the step's tag
// parity) of [n_layers][2][dim] words; each step clears the other parity.
struct StepParams {
    const LayerDev* layers;
    const void* kv_maps;      // CUtensorMap[kMapsPerLayer * n_layers]: K, V, O values, O scales, down values, down scales
    GView ov, dv;             // column-group views of Wo and Wdown (same geometry in every layer)
    DMat embd;
    DMat out;
    const float* out_norm;
    const float* rope_freqs;  // [rope_dims/2] or nullptr
    int n_layers, dim, n_heads, n_kv, hd, ffn, vocab, max_seq, rope_dims, neox, q_dim, kv_dim;
    int ngrp;                 // column groups (divides n_kv)
    float eps, theta_scale, attn_div;

    unsigned long long* tv;   // tagged vectors, n_layers sets (tv_elems_per_layer words each)
    unsigned long long* part; // tagged attention partials, n_layers sets (part_words_per_layer each)
    unsigned long long* delta;// residual accumulators [2][n_layers][2][dim]
    unsigned* epoch;          // tag of the last completed step; this step writes epoch + 1
    float* logits;            // [vocab]
    int max_splits;
    unsigned long long* best; // packed argmax of the step
    unsigned* counters;
    int* err;

    const int* token_in;
    int* token_out;
    int pos;
    int splits;               // attention splits per kv head for this pos
    // sizes the index checks of LLM_CHECKED builds hold the step's accesses to
    long long tv_words, part_words, delta_words;
    int logits_limit;         // logits the step may write (vocab)

    // shared-memory geometry (bytes from the dynamic smem base)
    int ns;                   // ring slots
    int attn_rows;            // KV rows per ring slot
    int attn_mma;             // attention on tensor cores (mma.sync): head_dim in {32, 48, 64}, gq <= 4
    int attn_w;               // KV tile sub-tile width (elements): 64 when head_dim % 64 == 0 on the mma path, else head_dim
    int off_xs, off_red, off_res, off_rope, off_comb, off_bar, off_misc, off_own, off_gain;
    int scratch_floats;       // floats of the staging / attention scratch region (xs)

    unsigned long long* trace;  // [gridDim.x][kTraceSlots] phase stamps, or nullptr (LLM_TRACE builds)
};
constexpr int kMapsPerLayer = 6;

// Attention partials of one layer: acc [n_heads][max_splits][hd], then (m, l)
// [n_heads][max_splits][2], then the score statistics the llama.cpp-rounding
// step exchanges before its second pass [n_heads][max_splits][2] (tagged
// words).
__host__ __device__ inline long long part_words_per_layer(int n_heads, int max_splits, int hd) {
    long long w = (long long)n_heads * max_splits * (hd + 4);
    return w + (w & 1);
}

// Phase trace (compiled in with -DLLM_TRACE): per CTA, %globaltimer stamps (ns).
//   consumer  10*l + {0..9}: start/end of QKV, ATTN, O, GU, DOWN of layer l
//             160 + 4*l + {0..3}: first chunk of QKV, O, GU, DOWN landed
//             240, 241, 242: LOGITS start, end, argmax published
//   producer  256 + 8*l + {0..4}: first issue of QKV, ATTN, O, GU, DOWN; 256 + 8*l + 5: layer issued
//             448, 449: LOGITS first issue, all issued
//   consumer  512 + 4*l + {0..3}: activation lanes loaded in QKV, O, GU, DOWN
//   consumer  576 + 4*l + {0..3}: attention unit: q/k/v read and rotated, partial stored,
//             chosen to merge (merging unit only), merged output stored (merging unit only)
//   producer  640 + 4*l + {0..3}: first copy of QKV, O, GU, DOWN issued
//   consumer  768 + 4*l + {0..3}: SM cycles thread 0 waited for full slots in QKV, O, GU, DOWN
//   producer  896 + 4*l + {0..3}: SM cycles the producer waited for free slots while issuing them
constexpr int kTraceSlots = 1024;

__host__ __device__ inline int n_phase_counters(int) { return 1; }

// Tagged-vector set of one layer: element offsets of its vectors.
struct TvLayout {
    long long qkv, u, stride;
};
__host__ __device__ inline TvLayout tv_layout(int dim, int q_dim, int kv_dim, int ffn) {
    (void)dim;
    TvLayout t;
    t.qkv = 0;
    t.u = t.qkv + q_dim + 2LL * kv_dim;
    t.u += t.u & 1;                    // 16-byte aligned vectors
    t.stride = t.u + ffn;
    t.stride += t.stride & 1;
    return t;
}

// Batched prefill (F16 weights): what it needs of a handle.
constexpr int kPrefillRows = 512;            // tokens per tensor-core batch
struct PrefillCtx {
    cudaStream_t st;
    int sms, wtype;
    int n_layers, dim, n_heads, n_kv, hd, ffn, vocab, rope_dims, neox, q_dim, kv_dim;
    float eps, theta_scale, attn_div;
    const LayerDev* layers;                  // host array [n_layers] of device layouts
    DMat embd, out;
    const float* out_norm;
    const float* rope_freqs;
    float* logits;                           // [vocab]: the last token's logits
    int* argmax_dev;                         // the last token's argmax
    unsigned long long* best;                // argmax key, zero before and after
    int* err;                                // device error word
    const __half* f16_copy;                  // Q8_0: the F16 copy of the layer matrices, or nullptr
};
bool prefill_supported(const PrefillCtx& c);
size_t prefill_workspace_bytes(const PrefillCtx& c);
// The F16 copy of a Q8_0 model's layer matrices for the prefill GEMMs: its
// size, and its expansion (asynchronous on c.st; *launches counts kernels).
size_t prefill_f16_copy_bytes(const PrefillCtx& c);
cudaError_t prefill_make_f16_copy(const PrefillCtx& c, __half* dst, int* launches);
cudaError_t prefill_f16(const PrefillCtx& c, void* ws, const int32_t* tokens_host, int n, int pos0, const char** msg);

__host__ __device__ inline int dtype_bytes_x16(int wtype) {   // bytes per element, times 16
    return wtype == LLM_Q8_0 ? 16 : (wtype == LLM_F16 ? 32 : 64);
}

constexpr int kLaneElems = 32;                     // matrix columns one lane covers per row
constexpr int kMaxTeams = 7;                       // multi-warp teams of one GEMV phase
constexpr int kOwnFloats = 256;                    // residual rows a CTA owns, and its QKV bias rows

// Bytes of one row in a ring slot (quants/values plus Q8_0 scales).
__host__ __device__ inline int slot_row_bytes(int wtype, int cols, int dstride) {
    return wtype == LLM_Q8_0 ? cols + 2 * dstride : cols * (wtype == LLM_F16 ? 2 : 4);
}

// ---------------------------------------------------------------- PTX --
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// One tagged element: the float's bits and the tag in a single 64-bit store.
__device__ __forceinline__ void st_tagged(unsigned long long* a, float v, unsigned tag) {
    const unsigned long long w = ((unsigned long long)tag << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(a), "l"(w) : "memory");
}

// Two tagged elements (16-byte aligned); each 64-bit word is read whole.
__device__ __forceinline__ ulonglong2 ld_tagged2(const unsigned long long* a) {
    ulonglong2 r;
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(r.x), "=l"(r.y) : "l"(a) : "memory");
    return r;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Atomic add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for a phase with the thread suspended (up to about 1 us per call) until
// the phase completes: a waiting warp then takes no issue slots from the
// warps that share its SM sub-partition.
__device__ __forceinline__ bool mbar_sleep_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(1000u)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of a phase: never suspends the thread, so a spin on it
// sees the phase complete as soon as it does.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// 16-byte asynchronous copy global -> shared (completes at cp_async_wait_all).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// 1-D bulk copy global -> shared, completing `bytes` on the mbarrier.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Orders this thread's generic-proxy writes to shared memory before later
// async-proxy (TMA) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Four 8x8 b16 matrices from shared memory (lanes 8i..8i+7 give the row
// addresses of matrix i); .trans delivers each matrix transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}

// D = A * B + C for one m16n8k16 tile, F16 operands, F32 accumulation, with
// A's rows 8..15 zero: only the accumulator rows 0..7 (d0 = column 2t, d1 =
// column 2t + 1 of row lane/4) are carried.
__device__ __forceinline__ void mma_rows8(float& d0, float& d1, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    float x2, x3;                 // rows 8..15 of D, not used
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %12, %12};"
        : "=f"(d0), "=f"(d1), "=f"(x2), "=f"(x3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(d0), "f"(d1), "f"(0.f));
    asm volatile("" ::"f"(x2), "f"(x3));
}

// 2-D tiled tensor copy global -> shared (box of the tensor map at (x, y)).
__device__ __forceinline__ void tma_2d_g2s(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// 3-D tiled tensor copy global -> shared (box of the tensor map at (x, y, z)).
__device__ __forceinline__ void tma_3d_g2s(void* dst, const void* tmap, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// Residual accumulator words: (contributions << 56) + fixed-point sum (scale
// 2^32).  A contribution must stay below 2^15 in magnitude so that the sum of
// up to 255 of them never reaches the count bits.
constexpr float kAccScale = 4294967296.0f;       // 2^32
constexpr float kAccLimit = 32768.0f;             // 2^15
// round(v * 2^32) as a 64-bit integer for |v| < 2^15, in 32-bit operations
// (64-bit conversions run on the FP64 pipe, which is slow on this part): the
// scaled value is an exact float; below 2^31 it rounds to an int32, above it
// is already an integer and splits exactly into 2^16 * q + rem.
__device__ __forceinline__ long long acc_fixed(float v) {
    const float t = v * kAccScale;
    if (fabsf(t) < 2147483648.0f) return (long long)__float2int_rn(t);
    const int q = __float2int_rz(t * 1.52587890625e-05f);         // t / 2^16, truncated
    const float rem = fmaf(-(float)q, 65536.0f, t);                // exact
    return (long long)q * 65536 + (long long)__float2int_rn(rem);
}
__device__ __forceinline__ void acc_add(unsigned long long* a, float v, int* err) {
    long long fx = 0;
    if (fabsf(v) < kAccLimit) fx = acc_fixed(v);
    else atomicOr(err, kErrRange);                 // also NaN
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(a), "l"((1ull << 56) + (unsigned long long)fx)
                 : "memory");
}
__device__ __forceinline__ unsigned acc_count(unsigned long long w) { return (unsigned)((w + (1ull << 55)) >> 56); }
// The word's sum times 2^-32 as a float: magnitude split into 32-bit halves
// (each converted exactly or rounded once, then one fused multiply-add).
__device__ __forceinline__ float acc_value(unsigned long long w) {
    const unsigned long long c = (w + (1ull << 55)) >> 56;
    const long long v = (long long)(w - (c << 56));
    const unsigned long long a = v < 0 ? (unsigned long long)(-v) : (unsigned long long)v;
    const float f = __fadd_rn(__uint2float_rn((unsigned)(a >> 32)), __uint2float_rn((unsigned)a) * 2.3283064365386963e-10f);
    return v < 0 ? -f : f;
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }
__device__ __forceinline__ void block_join() { asm volatile("bar.sync 2, %0;" ::"n"(kBlock) : "memory"); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ double warp_sum(double v) {
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
