// The batch-1 decode step as one persistent, warp-specialised kernel.
//
// One CTA per SM (cooperative launch, so all CTAs are resident).  Warps 0-14
// compute ("consumers"); warp 15 ("producer") streams everything the CTA will
// read from HBM (its rows of every weight matrix and its KV-cache tiles) in a
// fixed order through a ring of 64 KB shared-memory slots, with cp.async.bulk
// (whole weight rows) and TMA tensor tiles (KV tiles, column blocks of Wo and
// Wdown), completing on mbarriers.  The producer never waits on other CTAs:
// nothing it loads depends on this step's results (KV row `pos`, which does,
// is patched in by the consumers), so HBM keeps streaming while the consumers
// wait for their inputs.
//
// The grid is split into `ngrp` column groups of CTAs (group g holds the kv
// heads [g*n_kv/ngrp, (g+1)*n_kv/ngrp) and the matching columns of Wo, and
// one ngrp-th of the FFN columns):
//
//   per layer l:  QKV   rows of [Wq;Wk;Wv] . RMSNorm(x)        -> qkv (+ bias)
//                 ATTN  (kv head, position split) units: RoPE(q), RoPE(k),
//                       K/V row `pos` stored as F16, partial softmax (m, l, acc)
//                 O     every CTA of group g merges the partials of its heads
//                       and multiplies them by its rows of g's columns of Wo
//                       -> adds to the residual accumulator (one word per row)
//                 GU    rows of [Wgate|Wup] . RMSNorm(x)        -> u = silu(gate) * up
//                       (group g computes its ffn/ngrp columns of u)
//                 DOWN  every CTA of group g multiplies g's part of u by its
//                       rows of g's columns of Wdown -> adds to the residual
//   LOGITS  rows of Wout . RMSNorm(x) -> logits, argmax (first index of the max)
//
// Steps follow "The Forward Pass in Java", Example 13 (Llama.forward).  The
// attention split and merge is the flash-decoding rearrangement of the same
// softmax (max-subtracted partial sums combined with exp(m_s - M) weights);
// splitting the O and down products by column groups only regroups their sums.
//
// A matrix row is reduced by a "team" of lanes, each holding 32 elements of
// the activation vector in registers; rows up to 1024 elements are part of a
// warp, longer rows whole warps that take four rows per pass.  Every CTA keeps
// the whole residual stream in shared memory and adds each layer's two
// accumulated updates to it in the same order, so all CTAs hold the same bits.
//
// Every wait is bounded; on expiry the error word is set, the producer drains
// its copies in flight, and the CTA exits.
#include <algorithm>
#include <type_traits>

#include "llm_internal.cuh"

namespace llm {

#ifdef LLM_TRACE
__device__ __forceinline__ void trace_mark(const StepParams& p, int k) {
    if (p.trace) p.trace[(size_t)blockIdx.x * kTraceSlots + k] = global_timer_ns();
}
#else
__device__ __forceinline__ void trace_mark(const StepParams&, int) {}
#endif
// Fine-grained marks inside the phases of one layer (trace builds): thread
// 0's time at step i of a phase, at slot c.fine + i (c.fine < 0: off).
#ifdef LLM_TRACE
#define FMARK(c, i) \
    do { if ((c).fine >= 0 && (c).tid == 0) trace_mark((c).p, (c).fine + (i)); } while (0)
#else
#define FMARK(c, i) do { } while (0)
#endif

// Spin until ready() holds.  The deadline (SM cycle counter) and the error
// word (a global load) are checked only every 256 polls, so a wait that ends
// reacts within a few hundred cycles.  Returns false on expiry (after setting
// the error word) or when another CTA has already reported a timeout.  (A
// failed index check of LLM_CHECKED builds does not end waits: data it kept
// from being written makes its readers time out, and writes nobody waits
// for, such as the logits, leave the rest of the step intact.)
constexpr long long kWaitLimitCycles = 4000000000ll;   // about 2 s at 2 GHz

template <class Ready>
__device__ __forceinline__ bool bounded_wait(Ready ready, int* err) {
    if (ready()) return true;
    const long long t0 = clock64();
    for (unsigned i = 1;; i++) {
        if (ready()) return true;
        if ((i & 255u) == 0) {
            if (*(volatile int*)err & kErrTimeout) return false;
            if (clock64() - t0 > kWaitLimitCycles) {
                atomicOr(err, kErrTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool tagged2_ready(const ulonglong2& w, unsigned tag) {
    return ((unsigned)(w.x >> 32) == tag) & ((unsigned)(w.y >> 32) == tag);
}

// Tagged elements once they carry `tag` (the step's): four consecutive ones
// (16-byte aligned), two, or one.  After a timeout (the error word is set)
// the values read as zero; every later wait of the step then gives up at once.
__device__ __forceinline__ float4 poll4(const unsigned long long* a, unsigned tag, int* err) {
    ulonglong2 w0, w1;
    const auto ready = [&] {
        w0 = ld_tagged2(a);
        w1 = ld_tagged2(a + 2);
        return tagged2_ready(w0, tag) & tagged2_ready(w1, tag);
    };
    if (!bounded_wait(ready, err)) return make_float4(0.f, 0.f, 0.f, 0.f);
    return make_float4(__uint_as_float((unsigned)w0.x), __uint_as_float((unsigned)w0.y),
                       __uint_as_float((unsigned)w1.x), __uint_as_float((unsigned)w1.y));
}
__device__ __forceinline__ float2 poll2(const unsigned long long* a, unsigned tag, int* err) {
    ulonglong2 w;
    const auto ready = [&] {
        w = ld_tagged2(a);
        return tagged2_ready(w, tag);
    };
    if (!bounded_wait(ready, err)) return make_float2(0.f, 0.f);
    return make_float2(__uint_as_float((unsigned)w.x), __uint_as_float((unsigned)w.y));
}
__device__ __forceinline__ float poll1(const unsigned long long* a, unsigned tag, int* err) {
    unsigned long long w;
    const auto ready = [&] {
        asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(a) : "memory");
        return (unsigned)(w >> 32) == tag;
    };
    if (!bounded_wait(ready, err)) return 0.f;
    return __uint_as_float((unsigned)w);
}

// Four residual-accumulator words (16-byte aligned) once `n` groups have
// added to each: their sums, as floats.
__device__ __forceinline__ float4 poll_acc4(const unsigned long long* a, unsigned n, int* err) {
    ulonglong2 w0, w1;
    const auto ready = [&] {
        w0 = ld_tagged2(a);
        w1 = ld_tagged2(a + 2);
        return (acc_count(w0.x) == n) & (acc_count(w0.y) == n) & (acc_count(w1.x) == n) & (acc_count(w1.y) == n);
    };
    if (!bounded_wait(ready, err)) return make_float4(0.f, 0.f, 0.f, 0.f);
    return make_float4(acc_value(w0.x), acc_value(w0.y), acc_value(w1.x), acc_value(w1.y));
}

// Shared-memory regions, addressed from the dynamic smem base with the
// offsets in the (constant-bank) parameters, so no region pointer stays live.
struct Smem {
    unsigned char* base;
    const StepParams& p;
    __device__ Smem(unsigned char* b, const StepParams& p_) : base(b), p(p_) {}
    __device__ __forceinline__ uint8_t* ring() const { return base; }
    // attention scratch, and the staged activation vector of a GEMV phase (scratch_floats floats)
    __device__ __forceinline__ float* xs() const { return reinterpret_cast<float*>(base + p.off_xs); }
    // [rows of this CTA][warps of a team] partial dots of multi-warp teams
    __device__ __forceinline__ float* rowp() const { return reinterpret_cast<float*>(base + p.off_red); }
    // the residual stream [dim]; in the logits phase, that phase's row partials
    __device__ __forceinline__ float* res() const { return reinterpret_cast<float*>(base + p.off_res); }
    __device__ __forceinline__ float* rope_c() const { return reinterpret_cast<float*>(base + p.off_rope); }
    __device__ __forceinline__ float* rope_s() const { return rope_c() + 128; }
    // [2 * kConsumers] attention split combine, merge partial sums
    __device__ __forceinline__ float* comb() const { return reinterpret_cast<float*>(base + p.off_comb); }
    // [kOwnFloats] the CTA's QKV bias rows / (gate, up) sums; then [kOwnFloats] merge weights
    __device__ __forceinline__ float* bias() const { return reinterpret_cast<float*>(base + p.off_own); }
    __device__ __forceinline__ float* aux() const { return bias() + kOwnFloats; }
    // the next RMSNorm's gains, fetched ahead of their phase (swizzled like the staged vector)
    __device__ __forceinline__ float* gains() const { return reinterpret_cast<float*>(base + p.off_gain); }
    __device__ __forceinline__ uint64_t* full() const { return reinterpret_cast<uint64_t*>(base + p.off_bar); }
    __device__ __forceinline__ uint64_t* empty() const { return full() + p.ns; }
    __device__ __forceinline__ int* misc() const { return reinterpret_cast<int*>(base + p.off_misc); }   // [0] abort, [1] flag
    __device__ __forceinline__ float* fred() const { return reinterpret_cast<float*>(base + p.off_misc + 64); }
    __device__ __forceinline__ double* fred_d() const { return reinterpret_cast<double*>(base + p.off_misc + 64); }
    __device__ __forceinline__ unsigned long long* best() const {
        return reinterpret_cast<unsigned long long*>(base + p.off_misc + 64 + 8 * (kConsumerWarps + 2));
    }
};

// ------------------------------------------------------------ schedule --
// Both roles walk the same sequence of chunks; these helpers define it.
__device__ __forceinline__ void share(int n, int j, int parts, int& a, int& b) {
    a = (int)((long long)n * j / parts);
    b = (int)((long long)n * (j + 1) / parts);
}
__device__ __forceinline__ void cta_rows(int rows, int& r0, int& r1) { share(rows, blockIdx.x, gridDim.x, r0, r1); }

// This CTA's column group: group g is CTAs [g*G/ngrp, (g+1)*G/ngrp); j is the
// CTA's index in it and n its size.
struct Part {
    int g, j, n;
};
__device__ __forceinline__ Part cta_part(int ngrp) {
    const long long G = gridDim.x, b = blockIdx.x;
    const int g = (int)((ngrp * (b + 1) - 1) / G);
    const int f0 = (int)(g * G / ngrp), f1 = (int)((g + 1) * G / ngrp);
    return Part{g, (int)b - f0, f1 - f0};
}

__device__ __forceinline__ void unit_range(const StepParams& p, int unit, int S, int& g, int& s, int& t0, int& t1) {
    g = unit / S;
    s = unit % S;
    const int n_pos = p.pos + 1, chunk = (n_pos + S - 1) / S;
    t0 = min(n_pos, s * chunk);
    t1 = min(n_pos, t0 + chunk);
}

__device__ __forceinline__ int row_qbytes(const DMat& m, int wtype) {
    return wtype == LLM_Q8_0 ? m.cols : m.cols * (wtype == LLM_F16 ? 2 : 4);
}

// Position in the ring: slot index and the parity of its current use.
struct RingPos {
    int slot = 0;
    uint32_t phase = 0;      // flips each time the slot index wraps
    int count = 0;           // chunks passed (saturates at ns: "ring filled once")
    __device__ __forceinline__ void advance(int ns) {
        if (++slot == ns) { slot = 0; phase ^= 1u; }
        if (count < ns) count++;
    }
};

__device__ __forceinline__ const char* layer_map(const StepParams& p, int layer, int which) {
    return reinterpret_cast<const char*>(p.kv_maps) + ((size_t)kMapsPerLayer * layer + which) * 128;
}

// First scale column of group g's scale box (the group's first scale rounded
// down to a multiple of 8, a 16-byte boundary).
__device__ __forceinline__ int gview_scale_x(const GView& v, int g) { return (g * (v.m.cols / 32)) & ~7; }

// ------------------------------------------------------------ producer --
struct Producer {
    const StepParams& p;
    Smem& sm;
    RingPos rp;
    long long it = 0;
    bool dead = false;
    long long waited = 0;  // trace builds: SM cycles spent waiting for free slots

    __device__ Producer(const StepParams& p_, Smem& s_) : p(p_), sm(s_) {}

    // Next free slot, or nullptr after an error.  A slot's first fill needs no
    // wait; later fills wait for the consumers' release of the previous use.
    __device__ uint8_t* acquire(int& slot) {
        slot = rp.slot;
        if (rp.count >= p.ns) {
            const uint32_t par = rp.phase ^ 1u;
            uint64_t* bar = &sm.empty()[slot];
#ifdef LLM_TRACE
            const long long tw0 = clock64();
#endif
            if (!bounded_wait([&] { return mbar_sleep_wait(bar, par); }, p.err)) {
                dead = true;
                return nullptr;
            }
#ifdef LLM_TRACE
            waited += clock64() - tw0;
#endif
        }
        return sm.ring() + (size_t)slot * kSlotBytes;
    }

    __device__ __forceinline__ void issued() {
        rp.advance(p.ns);
        it++;
    }

    // trace builds: the cycles waited for free slots during the phase with
    // producer trace slot tk (256 + 8 l + {0, 2, 3, 4}), at 896 + 4 l + j
    __device__ __forceinline__ void note_wait(int tk) {
#ifdef LLM_TRACE
        if (p.trace && tk >= 256 && tk < 448) {
            const int l = (tk - 256) / 8, k = (tk - 256) % 8;
            const int j = k == 0 ? 0 : k - 1;
            p.trace[(size_t)blockIdx.x * kTraceSlots + 896 + 4 * l + j] = waited;
        }
        waited = 0;
#endif
    }

    // Rows [r0, r1) of m (single rows) as whole rows, m.rpc per chunk.
    __device__ void rows(const DMat& m, int wtype, int r0, int r1, int tk) {
        if (dead) return;
        // a pair matrix counts super-rows and streams single rows
        if (!LLM_IN_BOUNDS(p.err, r0 >= 0 && r1 <= m.rows * (m.pair ? 2 : 1))) {
            dead = true;                      // the consumers' waits for these chunks time out
            return;
        }
        trace_mark(p, tk);
        const size_t rowq = (size_t)row_qbytes(m, wtype);
        const int rowd = wtype == LLM_Q8_0 ? 2 * m.dstride : 0;
        for (int r = r0; r < r1; r += m.rpc) {
            const int n = min(m.rpc, r1 - r);
            int slot;
            uint8_t* dst = acquire(slot);
            if (!dst) return;
            const uint32_t bq = (uint32_t)(n * rowq), bd = (uint32_t)(n * rowd);
            mbar_arrive_expect_tx(&sm.full()[slot], bq + bd);
            bulk_g2s(dst, m.q + (size_t)r * rowq, bq, &sm.full()[slot]);
            if (bd) bulk_g2s(dst + bq, reinterpret_cast<const uint8_t*>(m.d) + (size_t)r * rowd, bd, &sm.full()[slot]);
            issued();
        }
        note_wait(tk);
    }

    // Rows [r0, r1) of group g's column block of a matrix, v.R rows per chunk
    // (TMA boxes; rows past the matrix's end read as zero).
    __device__ void view(const GView& v, const char* mq, const char* md, int g, int r0, int r1, int tk) {
        if (dead) return;
        if (!LLM_IN_BOUNDS(p.err, r0 >= 0 && r1 <= v.m.rows && g >= 0 && g < p.ngrp)) {
            dead = true;
            return;
        }
        trace_mark(p, tk);
        const int y = g * (v.m.cols / v.U), sx = gview_scale_x(v, g);
        for (int r = r0; r < r1; r += v.R) {
            int slot;
            uint8_t* dst = acquire(slot);
            if (!dst) return;
            mbar_arrive_expect_tx(&sm.full()[slot], (uint32_t)v.box_bytes);
            tma_3d_g2s(dst, mq, 0, y, r, &sm.full()[slot]);
            if (v.rowd) tma_2d_g2s(dst + v.sboff, md, sx, r, &sm.full()[slot]);
            issued();
        }
        note_wait(tk);
    }

    // The K and V tiles of this CTA's attention units, chunk by chunk; with
    // two_pass (llama.cpp rounding) each unit's K tiles alone first, then its
    // K and V tiles again.
    __device__ void attention(int layer, bool two_pass) {
        if (dead) return;
        trace_mark(p, 256 + 8 * layer + 1);
        const int S = p.splits, units = p.n_kv * S, P = p.attn_rows;
        const void* kmap = layer_map(p, layer, 0);
        const void* vmap = layer_map(p, layer, 1);
        const uint32_t half_bytes = (uint32_t)(P * p.hd * 2);
        const int W = p.attn_w, nsub = p.hd / W;                   // sub-tiles of [P][W] per tile
        for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
            int g, s, t0, t1;
            unit_range(p, unit, S, g, s, t0, t1);
            for (int pass = two_pass ? 0 : 1; pass < 2; pass++) {
                const bool with_v = pass == 1;
                for (int c0 = t0; c0 < t1; c0 += P) {
                    int slot;
                    uint8_t* dst = acquire(slot);
                    if (!dst) return;
                    mbar_arrive_expect_tx(&sm.full()[slot], with_v ? 2 * half_bytes : half_bytes);
                    for (int j = 0; j < nsub; j++) {
                        tma_2d_g2s(dst + (size_t)j * P * W * 2, kmap, g * p.hd + j * W, c0, &sm.full()[slot]);
                        if (with_v)
                            tma_2d_g2s(dst + half_bytes + (size_t)j * P * W * 2, vmap, g * p.hd + j * W, c0,
                                       &sm.full()[slot]);
                    }
                    issued();
                }
            }
        }
        note_wait(-1);
    }

    __device__ void drain() {
        // the last min(it, ns) copies: slots rp.slot-1, rp.slot-2, ... backwards
        const int n = it < p.ns ? (int)it : p.ns;
        int slot = rp.slot;
        uint32_t phase = rp.phase;
        for (int k = 0; k < n; k++) {
            if (slot == 0) { slot = p.ns; phase ^= 1u; }
            slot--;
            uint64_t* bar = &sm.full()[slot];
            const long long t0 = clock64();
            while (!mbar_try_wait(bar, phase))
                if (clock64() - t0 > kWaitLimitCycles) break;
        }
    }
};

// ------------------------------------------------------------ consumers --
struct Consumer {
    const StepParams& p;
    Smem& sm;
    RingPos rp;            // next slot to consume
    int tid, warp, lane;
    unsigned tag;          // this step's tag of the tagged vectors
    unsigned long long* delta;   // this step's parity of the residual accumulators
    long long waited = 0;        // trace builds: SM cycles spent waiting for full ring slots
    int fine = -1;               // trace builds: first slot of this phase's fine marks, or -1

    __device__ Consumer(const StepParams& p_, Smem& s_) : p(p_), sm(s_) {
        tid = threadIdx.x;
        warp = tid >> 5;
        lane = tid & 31;
        tag = __ldcg(p.epoch) + 1u;
        delta = p.delta + (size_t)(tag & 1u) * p.n_layers * 2 * p.dim;
    }

    // element offsets of the tagged vectors within a layer's set
    __device__ __forceinline__ TvLayout tl() const { return tv_layout(p.dim, p.q_dim, p.kv_dim, p.ffn); }

    // layer l's tagged vector at element offset `off` of its set
    __device__ __forceinline__ unsigned long long* tv(int l, long long off) const {
        return p.tv + (long long)l * tl().stride + off;
    }
    // layer l's attention partials
    __device__ __forceinline__ unsigned long long* part(int l) const {
        return p.part + (long long)l * part_words_per_layer(p.n_heads, p.max_splits, p.hd);
    }
    // a tagged attention partial or statistic of this step (index-checked in
    // LLM_CHECKED builds)
    __device__ __forceinline__ void st_part(unsigned long long* a, float v) const {
        if (LLM_IN_BOUNDS(p.err, a >= p.part && a < p.part + p.part_words)) st_tagged(a, v, tag);
    }
    // layer l's residual accumulator after the attention block (0) or the FFN (1)
    __device__ __forceinline__ unsigned long long* acc(int l, int which) const {
        return delta + ((size_t)l * 2 + which) * p.dim;
    }

    __device__ bool aborted() const { return *(volatile int*)&sm.misc()[0] != 0; }

    // Wait for the next slot.  A timeout is recorded in the abort flag; the
    // caller checks it only at a point all consumer threads reach together.
    __device__ uint8_t* next_slot(int& slot) {
        slot = rp.slot;
        const uint32_t par = rp.phase;
        uint64_t* bar = &sm.full()[slot];
#ifdef LLM_TRACE
        const long long tw0 = clock64();
#endif
        if (!bounded_wait([&] { return mbar_sleep_wait(bar, par); }, p.err)) sm.misc()[0] = 1;
#ifdef LLM_TRACE
        waited += clock64() - tw0;
#endif
        return sm.ring() + (size_t)slot * kSlotBytes;
    }

    __device__ void release(int slot) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty()[slot]);
        rp.advance(p.ns);
    }

    // Start copying a norm's gains (n floats, n % 4 == 0) into shared memory;
    // stage_residual waits for them.  Each 16-byte word w lands at the swizzled
    // word (w & ~7) + ((w & 7) ^ ((w >> 3) & 7)), as the staged vectors do.
    __device__ void prefetch_gains(const float* g, int n) {
        float4* dst = reinterpret_cast<float4*>(sm.gains());
        for (int i = tid; i < n / 4; i += kConsumers)
            cp_async16(dst + (i & ~7) + ((i & 7) ^ ((i >> 3) & 7)), reinterpret_cast<const float4*>(g) + i);
        cp_async_commit();
    }

    // Sum of one value per warp (warps may pass 0), identical in every thread.
    __device__ float warps_total(float v) {
        v = warp_sum(v);
        if (lane == 0) sm.fred()[warp] = v;
        consumer_sync();
        float s = 0.f;
        for (int w = 0; w < kConsumerWarps; w++) s += sm.fred()[w];
        return s;
    }
};

// --------------------------------------------------------- weight decode --
// Element i of row r, decoded exactly as the format defines it: Q8_0
// d * qs (an exact float product), F16 widened, F32 as stored.
template <int DT>
__device__ __forceinline__ float weight_at(const DMat& m, int r, int i) {
    if constexpr (DT == LLM_Q8_0) {
        const float d = __half2float(m.d[(size_t)r * m.dstride + i / 32]);
        return __fmul_rn(d, (float)(int)(int8_t)m.q[(size_t)r * m.cols + i]);
    } else if constexpr (DT == LLM_F16) {
        return __half2float(reinterpret_cast<const __half*>(m.q)[(size_t)r * m.cols + i]);
    } else {
        return reinterpret_cast<const float*>(m.q)[(size_t)r * m.cols + i];
    }
}

// ------------------------------------------------------------ lane dots --
// A lane's 32 elements of one row (in the slot) against its 32 activations.
//
// F16 / F32: the activations are floats in registers (x2) and each product is
// an F32 FMA.
//
// Q8_0: the row's block is 32 int8 quants qs and one F16 scale d.  The lane's
// activations are held as fixed-point integers X_j = round(x_j * 2^e), e
// chosen from the largest |x_j| of the block so that |X_j| <= 2^22 (a
// resolution of 2^-22 of the block maximum, about what an F32 sum of the
// block's products keeps), as three base-256 digits X_j = D0_j + 256 D1_j +
// 65536 D2_j (D0, D1 unsigned bytes, D2 a signed byte).  The block's dot
// product is then exact integer arithmetic, four products per dp4a:
//   sum_j qs_j X_j = sum_k 256^k sum_j qs_j Dk_j,
// and the row's part is d * 2^-e times that sum, taken in float.  The digits
// of each 32-element block are made once per CTA while the phase's vector is
// staged (convert_group), and each lane loads its block's record.
template <int DT>
struct XReg {
    float2 x2[16];
};

template <>
struct XReg<LLM_Q8_0> {
    uint32_t d[3][8];   // digit k of elements 4i..4i+3 (byte b = element 4i + b)
    float inv;          // 2^-e
};

// d = a . b + c over four byte lanes: a signed, b unsigned / signed.
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// An int below 2^22 in magnitude as a float, exactly: placed in the mantissa
// of 1.5 * 2^23 by an integer add and taken out by a float subtraction (two
// full-rate operations instead of a conversion).
__device__ __forceinline__ float small_i2f(int a) { return __int_as_float(a + 0x4B400000) - 12582912.0f; }

// sum_j qs_j X_j of one block (two 16-byte words of quants), in float: each
// digit's sum is an exact integer below 2^21 in magnitude.
__device__ __forceinline__ float q8_block_sum(const uint4 (&w)[2], const XReg<LLM_Q8_0>& xr) {
    const uint32_t u[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
    int a0 = 0, a1 = 0, a2 = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        a0 = dp4a_su(u[i], xr.d[0][i], a0);
        a1 = dp4a_su(u[i], xr.d[1][i], a1);
        a2 = dp4a_ss(u[i], xr.d[2][i], a2);
    }
    return fmaf(fmaf(small_i2f(a2), 256.f, small_i2f(a1)), 256.f, small_i2f(a0));
}

// One staged group (four floats, word w of 32-element block b of the staging
// region xv) becomes its share of the block's digit record, in place: the
// record is 16-byte units u = 0..6 at unit u ^ (b & 7) of the block's 128
// bytes (the same swizzle as the staged words): units 0-1 digit 0 of the
// block's 32 elements, 2-3 digit 1, 4-5 digit 2, unit 6 {2^-e, 0, 0, 0}.
// The 8 groups of a block are held by lanes 8j..8j+7 of one warp, which meet
// in the shuffles for the block maximum after reading their words and before
// writing; every lane of the warp calls this (valid or not).
__device__ __forceinline__ void convert_group(float4* xv, int b, int w, bool valid, float4 v) {
    float m = valid ? fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))) : 0.f;
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    // m < 2^(be - 126) for the biased exponent be of m, so e = 148 - be keeps
    // |x| * 2^e below 2^22; zero and subnormal blocks take the largest e
    const int be = (int)((__float_as_uint(m) >> 23) & 0xFFu);
    const int e = be == 0 ? 126 : max(-126, min(126, 148 - be));
    const float sc = __uint_as_float((uint32_t)(127 + e) << 23);
    const int X0 = __float2int_rn(__fmul_rn(v.x, sc)), X1 = __float2int_rn(__fmul_rn(v.y, sc));
    const int X2 = __float2int_rn(__fmul_rn(v.z, sc)), X3 = __float2int_rn(__fmul_rn(v.w, sc));
    const uint32_t lo = __byte_perm((uint32_t)X0, (uint32_t)X1, 0x5140u);   // bytes 0,1 of X0 and X1
    const uint32_t hi = __byte_perm((uint32_t)X2, (uint32_t)X3, 0x5140u);
    const uint32_t b2 = __byte_perm(__byte_perm((uint32_t)X0, (uint32_t)X1, 0x0062u),
                                    __byte_perm((uint32_t)X2, (uint32_t)X3, 0x0062u), 0x5410u);
    if (valid) {
        uint32_t* blk = reinterpret_cast<uint32_t*>(xv + 8 * b);
        const int r = b & 7;
        blk[4 * ((0 + (w >> 2)) ^ r) + (w & 3)] = __byte_perm(lo, hi, 0x5410u);   // byte 0 of X0..X3
        blk[4 * ((2 + (w >> 2)) ^ r) + (w & 3)] = __byte_perm(lo, hi, 0x7632u);   // byte 1
        blk[4 * ((4 + (w >> 2)) ^ r) + (w & 3)] = b2;                             // byte 2 (signed)
        if (w == 0) reinterpret_cast<uint4*>(blk)[6 ^ r] = make_uint4((uint32_t)(127 - e) << 23, 0u, 0u, 0u);
    }
}

// The llama.cpp reading of a Q8_0 product ("What a Llama model computes, and
// why" §8): the block's activations are themselves quantized to Q8_0 first,
// d = amax / 127 kept as F16 and q_j = x_j * (1/d) rounded half away from
// zero (|q_j| <= 127; d = 0 gives q = 0).  The same digit record carries it:
// q_j as the signed top digit with the two low digits zero, and
// d_F16 * 2^-16 in place of 2^-e, so the three-digit dot returns
// d_F16 * sum_j qs_j q_j (the integer dot scaled by the block's F16 d).
__device__ __forceinline__ void convert_group_q8(float4* xv, int b, int w, bool valid, float4 v) {
    float m = valid ? fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))) : 0.f;
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    const float d = __fdiv_rn(m, 127.0f);
    const float id = d != 0.f ? __frcp_rn(d) : 0.f;
    auto q = [&](float x) { return (uint32_t)(int)roundf(__fmul_rn(x, id)) & 0xFFu; };
    const uint32_t b2 = q(v.x) | (q(v.y) << 8) | (q(v.z) << 16) | (q(v.w) << 24);
    if (valid) {
        uint32_t* blk = reinterpret_cast<uint32_t*>(xv + 8 * b);
        const int r = b & 7;
        blk[4 * ((0 + (w >> 2)) ^ r) + (w & 3)] = 0u;
        blk[4 * ((2 + (w >> 2)) ^ r) + (w & 3)] = 0u;
        blk[4 * ((4 + (w >> 2)) ^ r) + (w & 3)] = b2;
        if (w == 0) {
            const float dx = __half2float(__float2half_rn(d));
            reinterpret_cast<uint4*>(blk)[6 ^ r] = make_uint4(__float_as_uint(dx * (1.0f / 65536.0f)), 0u, 0u, 0u);
        }
    }
}

// x rounded to F16 (to nearest even) and widened back.
__device__ __forceinline__ float f16_round(float x) { return __half2float(__float2half_rn(x)); }

template <int DT>
struct LaneDot;

template <>
struct LaneDot<LLM_Q8_0> {
    static constexpr int kSeg = 2;           // 16-byte words per lane and row
};

template <>
struct LaneDot<LLM_F16> {
    static constexpr int kSeg = 4;
    __device__ __forceinline__ static float2 h2f(uint32_t v) {
        return __half22float2(__halves2half2(__ushort_as_half((unsigned short)(v & 0xffffu)),
                                             __ushort_as_half((unsigned short)(v >> 16))));
    }
    __device__ __forceinline__ static void acc(const uint4* w, const float2 (&x2)[16], float2& c0, float2& c1) {
#pragma unroll
        for (int s = 0; s < 4; s++) {
            c0 = __ffma2_rn(h2f(w[s].x), x2[4 * s], c0);
            c1 = __ffma2_rn(h2f(w[s].y), x2[4 * s + 1], c1);
            c0 = __ffma2_rn(h2f(w[s].z), x2[4 * s + 2], c0);
            c1 = __ffma2_rn(h2f(w[s].w), x2[4 * s + 3], c1);
        }
    }
};

template <>
struct LaneDot<LLM_F32> {
    static constexpr int kSeg = 8;
    __device__ __forceinline__ static void acc(const uint4* w, const float2 (&x2)[16], float2& c0, float2& c1) {
#pragma unroll
        for (int s = 0; s < 8; s++) {
            c0 = __ffma2_rn(make_float2(__uint_as_float(w[s].x), __uint_as_float(w[s].y)), x2[2 * s], c0);
            c1 = __ffma2_rn(make_float2(__uint_as_float(w[s].z), __uint_as_float(w[s].w)), x2[2 * s + 1], c1);
        }
    }
};

// One row: words of the lane (nseg of them valid, the rest read as zero).
template <int DT>
__device__ __forceinline__ float lane_row(const uint8_t* w, const uint8_t* scale, const XReg<DT>& xr, int nseg) {
    constexpr int NS = LaneDot<DT>::kSeg;
    uint4 v[NS];
#pragma unroll
    for (int s = 0; s < NS; s++) v[s] = s < nseg ? reinterpret_cast<const uint4*>(w)[s] : make_uint4(0u, 0u, 0u, 0u);
    if constexpr (DT == LLM_Q8_0) {
        if (!nseg) return 0.f;
        return __half2float(*reinterpret_cast<const __half*>(scale)) * (q8_block_sum(v, xr) * xr.inv);
    } else {
        float2 c0 = make_float2(0.f, 0.f), c1 = c0;
        LaneDot<DT>::acc(v, xr.x2, c0, c1);
        return (c0.x + c0.y) + (c1.x + c1.y);
    }
}

// Rows a multi-warp team reduces per pass: four for Q8_0 (two 16-byte words
// per lane and row), two for the wider F16 and F32 rows (register budget).
template <int DT>
struct RowsPerPass {
    static constexpr int value = DT == LLM_Q8_0 ? 4 : 2;
};

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ float lds_half(uint32_t a) {
    unsigned short h;
    asm volatile("ld.shared.b16 %0, [%1];" : "=h"(h) : "r"(a));
    return __half2float(__ushort_as_half(h));
}

// N rows at once: every shared-memory word of the N rows is loaded before the
// arithmetic starts, so the load latency is paid once.  Rows are given by
// their shared-memory addresses (quants or values w, Q8_0 scale sc).
// Q8_0: a lane reads its block's two 16-byte words in the order (sw, 1 - sw)
// with sw = bit 2 of the lane, so that the eight lanes of a quarter warp,
// whose blocks lie 32 bytes apart, touch all 32 banks once (the lane's digit
// words are permuted the same way when they are loaded, see lanes_prep).
template <int DT, int N>
__device__ __forceinline__ void lane_rows(const uint32_t (&w)[N], const uint32_t (&sc)[N], const XReg<DT>& xr,
                                          int nseg, int sw, float (&v)[N]) {
    constexpr int NS = LaneDot<DT>::kSeg;
    uint4 a[N][NS];
#pragma unroll
    for (int r = 0; r < N; r++)
#pragma unroll
        for (int s = 0; s < NS; s++)
            a[r][s] = s < nseg ? lds128(w[r] + 16 * (DT == LLM_Q8_0 ? (s ^ sw) : s)) : make_uint4(0u, 0u, 0u, 0u);
    if constexpr (DT == LLM_Q8_0) {
        float dq[N];
#pragma unroll
        for (int r = 0; r < N; r++) dq[r] = nseg ? lds_half(sc[r]) : 0.f;
#pragma unroll
        for (int r = 0; r < N; r++) v[r] = dq[r] * (q8_block_sum(a[r], xr) * xr.inv);
    } else {
#pragma unroll
        for (int r = 0; r < N; r++) {
            float2 c0 = make_float2(0.f, 0.f), c1 = c0;
            LaneDot<DT>::acc(a[r], xr.x2, c0, c1);
            v[r] = (c0.x + c0.y) + (c1.x + c1.y);
        }
    }
}

// ------------------------------------------------------------------ GEMV --
// The epilogue of a GEMV phase, chosen at run time (all phases share one
// copy of the GEMV code):
//   kStore   out[r] = v (+ bias of this CTA's row r), tagged
//   kSwiGLU  u[i] = silu(gate_i) * up_i ("The Forward Pass in Java",
//            Example 8): the (gate, up) sums of interleaved rows 2i, 2i+1
//            are parked in shared memory and the nonlinearity is applied to
//            all of the CTA's rows at once when the phase finishes
//   kLogits  logits[r] = v, keeping this thread's best (value, first index)
//   kAccum   v added to row r's residual accumulator word (fixed point)
struct Epi {
    enum : int { kStore, kSwiGLU, kLogits, kAccum };
    int kind;
    unsigned long long* out;      // tagged output vector (store, swiglu) or accumulator words (accum)
    const float* bias;            // store: smem bias indexed from `base`, or nullptr
    float* sm;                    // swiglu: (gate, up) sums
    int base;                     // first row (store), first super-row (swiglu)
    int end;                      // swiglu: end super-row
    unsigned tag;
    float* logits;
    int* err;
    unsigned long long best;
    float scale;                  // the RMSNorm scale of a normed phase (its vector is x * g), else 1
    const unsigned long long* lo; // LLM_CHECKED builds: out + r must lie in [lo, lo + n);
    long long n;                  // logits: r < n
    __device__ void row(int r, float v) {
        v *= scale;
        if (kind == kStore) {
            if (LLM_IN_BOUNDS(err, out + r >= lo && out + r < lo + n))
                st_tagged(out + r, bias ? v + bias[r - base] : v, tag);
        } else if (kind == kSwiGLU) {
            sm[r - 2 * base] = v;                 // row r: gate (even) or up (odd) of super-row r / 2
        } else if (kind == kAccum) {
            if (LLM_IN_BOUNDS(err, out + r >= lo && out + r < lo + n)) acc_add(out + r, v, err);
        } else {
            if (LLM_IN_BOUNDS(err, r >= 0 && r < n)) __stcg(logits + r, v);
            const unsigned long long k = argmax_key(v, r);
            best = k > best ? k : best;
        }
    }
    // LC (llama.cpp rounding): e^-g taken in double and rounded to float, as
    // the oracle takes it, so the product's input rounds from the same value
    template <bool LC>
    __device__ void finish(Consumer& c) {
        if (kind != kSwiGLU) return;
        consumer_sync();
        for (int k = c.tid; k < end - base; k += kConsumers) {
            const float g = sm[2 * k], up = sm[2 * k + 1];
            const float e = LC ? (float)exp(-(double)g) : expf(-g);
            if (LLM_IN_BOUNDS(err, out + base + k >= lo && out + base + k < lo + n))
                st_tagged(out + base + k, __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, e)), up), c.tag);
        }
    }
};

// Lane layout of a plan: team, lane index within the team (= the lane's
// 32-column block of the row), first column, 16-byte words of the row.
struct Lanes {
    int team, lit, col0, nseg;
    bool active;
};

template <int DT>
__device__ __forceinline__ Lanes lane_layout(const Consumer& c, const DMat& m) {
    constexpr int ES = DT == LLM_Q8_0 ? 1 : (DT == LLM_F16 ? 2 : 4);
    Lanes L;
    const int tw = m.tw;
    if (tw <= 32) {
        L.team = c.warp * (32 / tw) + c.lane / tw;
        L.lit = c.lane % tw;
    } else {
        const int wpr = tw / 32;
        L.team = c.warp / wpr;
        L.lit = (c.warp % wpr) * 32 + c.lane;
    }
    L.active = L.team < m.teams;
    L.col0 = L.lit * kLaneElems;
    L.nseg = L.active && L.col0 < m.cols ? min(kLaneElems, m.cols - L.col0) * ES / 16 : 0;
    return L;
}

// The lane's 32 activations (zero past the vector's end) from 8 float4 words
// w(k) = elements 4k..4k+3.
template <int DT, class Word>
__device__ __forceinline__ void xreg_from_words(Word w, XReg<DT>& xr) {
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const float4 v = w(k);
        xr.x2[2 * k] = make_float2(v.x, v.y);
        xr.x2[2 * k + 1] = make_float2(v.z, v.w);
    }
}

// The staging region holds a phase's activation vector as 16-byte words;
// word i of the 128-byte slice s = i / 8 sits at word s*8 + ((i & 7) ^ (s & 7)),
// so that the lanes' reads of their own slices fall in distinct banks.
__device__ __forceinline__ int swz(int i) { return (i & ~7) + ((i & 7) ^ ((i >> 3) & 7)); }

// One staged 4-element group (group i of the vector, valid when i < the
// vector's groups): Q8_0 phases turn it straight into its share of its
// 32-element block's digit record (convert_group, or convert_group_q8 under
// llama.cpp rounding, LC; the block's 8 groups are lanes 8j..8j+7 of one
// warp, so every lane of the warp calls this), the others store the floats
// (F16 phases under LC rounded to F16 first).
template <int DT, bool LC>
__device__ __forceinline__ void stage_group(float4* xv, int i, bool valid, float4 v) {
    if constexpr (DT == LLM_Q8_0) {
        if constexpr (LC) convert_group_q8(xv, i >> 3, i & 7, valid, v);
        else convert_group(xv, i >> 3, i & 7, valid, v);
    } else {
        if constexpr (LC && DT == LLM_F16) v = make_float4(f16_round(v.x), f16_round(v.y), f16_round(v.z), f16_round(v.w));
        if (valid) xv[swz(i)] = v;
    }
}

// Staging sources.  Each thread stages the 4-element groups i = tid, tid +
// kConsumers, ... (the same set in every phase, so a thread finds the
// residual values it keeps where it left them); the loops run warp by warp.
//
// The residual stream: x = x + (the update the block before added to the
// accumulator words d, once all ngrp groups have added), or at layer 0 the
// embedding row of `token` ("The Forward Pass in Java", Example 3: a copy of
// that row).  Kept in the residual region.  A normed phase stages x * g (the
// norm's gains, fetched ahead) and leaves the norm's scale to the rows'
// epilogue ("The Forward Pass in Java", Example 4: y = (x * scale) * g, and
// W y = scale * W (x * g)); returns the thread's sum of squares of x.  Under
// llama.cpp rounding (LC) a normed phase stages nothing here: its input is
// rounded after the scale is applied, so lanes_prep stages (x * scale) * g.
// The sum of squares of a norm: float, or double under llama.cpp rounding
// (LC), where the norm's scale is formed as the oracle forms it, in double.
template <bool LC>
using NormSum = std::conditional_t<LC, double, float>;

template <int DT, bool LC>
__device__ NormSum<LC> stage_residual(Consumer& c, const unsigned long long* d, int token, bool norm, float4* xv) {
    const StepParams& p = c.p;
    float4* res = reinterpret_cast<float4*>(c.sm.res());
    const float4* g4 = reinterpret_cast<const float4*>(c.sm.gains());
    const int ngr = p.dim / 4;
    NormSum<LC> ss = 0;
    if (norm) cp_async_wait_all();                     // this thread's part of the gains
    for (int i0 = c.tid - c.lane; i0 < ngr; i0 += kConsumers) {
        const int i = i0 + c.lane;
        const bool valid = i < ngr;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid) {
            if (d) {
                const float4 u = poll_acc4(d + 4 * i, (unsigned)p.ngrp, p.err);
                const float4 r = res[i];
                x = make_float4(__fadd_rn(r.x, u.x), __fadd_rn(r.y, u.y), __fadd_rn(r.z, u.z), __fadd_rn(r.w, u.w));
            } else {
                const int e = 4 * i;
                x = make_float4(weight_at<DT>(p.embd, token, e), weight_at<DT>(p.embd, token, e + 1),
                                weight_at<DT>(p.embd, token, e + 2), weight_at<DT>(p.embd, token, e + 3));
            }
            res[i] = x;
            if constexpr (LC)
                ss += ((double)x.x * x.x + (double)x.y * x.y) + ((double)x.z * x.z + (double)x.w * x.w);
            else
                ss += (x.x * x.x + x.y * x.y) + (x.z * x.z + x.w * x.w);
            if (norm && !LC) {
                const float4 g = g4[swz(i)];
                x = make_float4(__fmul_rn(x.x, g.x), __fmul_rn(x.y, g.y), __fmul_rn(x.z, g.z), __fmul_rn(x.w, g.w));
            }
        }
        if (!LC || !norm) stage_group<DT, LC>(xv, i, valid, x);
    }
    return ss;
}

// n elements (n % 4 == 0) of a tagged vector of this step.
template <int DT, bool LC>
__device__ void stage_tagged(Consumer& c, const unsigned long long* src, int n, float4* xv) {
    const int ngr = n / 4;
    for (int i0 = c.tid - c.lane; i0 < ngr; i0 += kConsumers) {
        const int i = i0 + c.lane;
        const bool valid = i < ngr;
        const float4 v = valid ? poll4(src + 4 * i, c.tag, c.p.err) : make_float4(0.f, 0.f, 0.f, 0.f);
        stage_group<DT, LC>(xv, i, valid, v);
    }
}

// The attention output of group g's heads, merged from the position splits'
// partials (m_s, l_s, acc_s): per head M = max_s m_s, w_s = e^(m_s - M) /
// sum_s' e^(m_s' - M) l_s', o = sum_s w_s acc_s.  Weights: one warp per head,
// one lane per split.  Weighted sums: thread (pair e2 of the group's outputs,
// split class sg) takes the splits s = sg, sg + NSG, ... in ascending order;
// the classes' sums are then added in class order (the same bits on every
// CTA of the group and in every run).  A thread issues its first eight loads
// before it waits on any of them.  Under llama.cpp rounding (LC) the splits'
// partials are already normalised by the head's global sum (each probability
// was rounded to F16 after it), so every weight w_s is 1.
template <int DT, bool LC>
__device__ void stage_merged(Consumer& c, int layer, int g, float4* xv) {
    const StepParams& p = c.p;
    const int HG = p.n_heads / p.ngrp, hd = p.hd, S = p.splits, MS = p.max_splits;
    const int h0 = g * HG, GDG = HG * hd;
    const unsigned long long* pacc = c.part(layer);
    const unsigned long long* pml = pacc + (size_t)p.n_heads * MS * hd;
    float* wgt = c.sm.aux();                                       // [HG][S]
    float* comb = c.sm.comb();                                     // [NSG][GDG]
    const int NP = GDG / 2, NSG = kConsumers / NP;
    const int e2 = c.tid % NP, sg = c.tid / NP;
    const bool act = sg < NSG;
    const int hh = (2 * e2) / hd, ii = (2 * e2) % hd;
    const unsigned long long* src = pacc + (size_t)(h0 + hh) * MS * hd + ii;
    constexpr int kB = 8;
    ulonglong2 w[kB];
#pragma unroll
    for (int k = 0; k < kB; k++) {
        const int s = sg + k * NSG;
        if (act && s < S) w[k] = ld_tagged2(src + (size_t)s * hd);
    }
    for (int h = c.warp; h < HG; h += kConsumerWarps) {
        const bool has = c.lane < S;
        if constexpr (LC) {
            if (has) wgt[h * S + c.lane] = 1.0f;
            continue;
        }
        const float2 ml = has ? poll2(pml + 2 * ((size_t)(h0 + h) * MS + c.lane), c.tag, p.err)
                              : make_float2(-INFINITY, 0.f);
        const float M = warp_max(ml.x);
        const float wv = has && ml.x != -INFINITY ? expf(ml.x - M) : 0.f;
        const float Ls = warp_sum(wv * ml.y);
        if (has) wgt[h * S + c.lane] = wv / Ls;
    }
#pragma unroll
    for (int k = 0; k < kB; k++) {
        const int s = sg + k * NSG;
        if (act && s < S && !tagged2_ready(w[k], c.tag)) {
            const float2 v = poll2(src + (size_t)s * hd, c.tag, p.err);
            w[k].x = __float_as_uint(v.x);
            w[k].y = __float_as_uint(v.y);
        }
    }
    consumer_sync();                                               // weights
    if (c.tid == 0) trace_mark(p, 576 + 4 * layer + 2);
    float ox = 0.f, oy = 0.f;
    if (act) {
        const float* wh = wgt + hh * S;
#pragma unroll
        for (int k = 0; k < kB; k++) {
            const int s = sg + k * NSG;
            if (s < S) {
                ox = fmaf(wh[s], __uint_as_float((unsigned)w[k].x), ox);
                oy = fmaf(wh[s], __uint_as_float((unsigned)w[k].y), oy);
            }
        }
        for (int s = sg + kB * NSG; s < S; s += NSG) {
            const float2 v = poll2(src + (size_t)s * hd, c.tag, p.err);
            ox = fmaf(wh[s], v.x, ox);
            oy = fmaf(wh[s], v.y, oy);
        }
        comb[sg * GDG + 2 * e2] = ox;
        comb[sg * GDG + 2 * e2 + 1] = oy;
    }
    consumer_sync();
    const int ngr = GDG / 4;
    for (int q0 = c.tid - c.lane; q0 < ngr; q0 += kConsumers) {
        const int q = q0 + c.lane;
        const bool valid = q < ngr;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid) {
            for (int k = 0; k < NSG; k++) {
                const float4 v = reinterpret_cast<const float4*>(comb + k * GDG)[q];
                o.x += v.x;
                o.y += v.y;
                o.z += v.z;
                o.w += v.w;
            }
        }
        stage_group<DT, LC>(xv, q, valid, o);
    }
}

// xr <- the lane's 32 activations of the staged vector (n elements; Q8_0: its
// block's digit record).  A normed phase's warps first pool their sums of
// squares (pass norm and the thread's sum ss); returns the norm's scale
// 1/sqrt(mean(x^2) + eps) ("The Forward Pass in Java", Example 4; the sum of
// squares a float tree sum), or 1.  Under llama.cpp rounding (LC) a normed
// phase's input y = (x * scale) * g is formed and staged here (from the
// residual and the gains each thread left in shared memory; the same groups
// as stage_residual) and 1 is returned.  Every consumer thread must call this
// (it synchronises).
template <int DT, bool LC>
__device__ float lanes_prep(Consumer& c, const Lanes& L, int n, bool norm, NormSum<LC> ss, XReg<DT>& xr) {
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    float4* xv = reinterpret_cast<float4*>(c.sm.xs());
    FMARK(c, 1);
    if (norm) {
        const NormSum<LC> w = warp_sum(ss);
        if (c.lane == 0) {
            if constexpr (LC) c.sm.fred_d()[c.warp] = w;
            else c.sm.fred()[c.warp] = w;
        }
    }
    consumer_sync();
    FMARK(c, 4);
    float scale = 1.0f;
    if (norm) {
        if constexpr (LC) {
            double tot = 0.0;
            for (int w = 0; w < kConsumerWarps; w++) tot += c.sm.fred_d()[w];
            scale = (float)(1.0 / sqrt(tot / (double)n + (double)c.p.eps));
        } else {
            float tot = 0.f;
            for (int w = 0; w < kConsumerWarps; w++) tot += c.sm.fred()[w];
            scale = 1.0f / sqrtf(tot / (float)n + c.p.eps);
        }
    }
    if constexpr (LC) {
        if (norm) {
            const float4* res = reinterpret_cast<const float4*>(c.sm.res());
            const float4* g4 = reinterpret_cast<const float4*>(c.sm.gains());
            const int ngr = n / 4;
            for (int i0 = c.tid - c.lane; i0 < ngr; i0 += kConsumers) {
                const int i = i0 + c.lane;
                const bool valid = i < ngr;
                float4 y = zero;
                if (valid) {
                    const float4 x = res[i], g = g4[swz(i)];
                    y = make_float4(__fmul_rn(__fmul_rn(x.x, scale), g.x), __fmul_rn(__fmul_rn(x.y, scale), g.y),
                                    __fmul_rn(__fmul_rn(x.z, scale), g.z), __fmul_rn(__fmul_rn(x.w, scale), g.w));
                }
                stage_group<DT, LC>(xv, i, valid, y);
            }
            consumer_sync();
            scale = 1.0f;
        }
    }
    const int col0 = L.col0;
    const bool have = L.active && col0 < n;
    const int sl = col0 >> 5;
    if constexpr (DT == LLM_Q8_0) {
        if (have) {
            const uint4* rec = reinterpret_cast<const uint4*>(xv + sl * 8);
            const int rot = sl & 7;
#pragma unroll
            for (int k = 0; k < 3; k++) {
                const uint4 a = rec[(2 * k) ^ rot], b = rec[(2 * k + 1) ^ rot];
                xr.d[k][0] = a.x; xr.d[k][1] = a.y; xr.d[k][2] = a.z; xr.d[k][3] = a.w;
                xr.d[k][4] = b.x; xr.d[k][5] = b.y; xr.d[k][6] = b.z; xr.d[k][7] = b.w;
            }
            xr.inv = __uint_as_float(rec[6 ^ rot].x);
            if ((c.lane >> 2) & 1) {               // the order lane_rows reads this lane's quant words in
#pragma unroll
                for (int k = 0; k < 3; k++)
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const uint32_t t = xr.d[k][i];
                        xr.d[k][i] = xr.d[k][i + 4];
                        xr.d[k][i + 4] = t;
                    }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; k++) xr.d[0][k] = xr.d[1][k] = xr.d[2][k] = 0u;
            xr.inv = 0.f;
        }
    } else {
        const float4* x4 = xv + sl * 8;
        const int rot = sl & 7;
        xreg_from_words<DT>([&](int k) { return have && col0 + 4 * k < n ? x4[k ^ rot] : zero; }, xr);
    }
    return scale;
}

// Where a chunk's rows sit in its ring slot.
struct ChunkGeo {
    int rowq, rowd;   // bytes per row of values, of Q8_0 scales
    int sfix;         // >= 0: the scales start at this byte offset; < 0: right after the chunk's values
    int soff;         // byte offset of the row's first scale within a scale row
    int rpc;          // rows per chunk
};

__device__ __forceinline__ ChunkGeo rows_geo(const DMat& m, int wtype) {
    return ChunkGeo{row_qbytes(m, wtype), wtype == LLM_Q8_0 ? 2 * m.dstride : 0, -1, 0, m.rpc};
}
__device__ __forceinline__ ChunkGeo view_geo(const GView& v, int g) {
    return ChunkGeo{v.rowq, v.rowd, v.sboff, v.rowd ? (g * (v.m.cols / 32) - gview_scale_x(v, g)) * 2 : 0, v.R};
}

// Rows [r0, r1) of m, chunk by chunk from the ring (the plan in m, the chunk
// layout in ck).  Multi-warp teams take four (Q8_0) or two rows per pass:
// their partial dots are reduced with one transposed butterfly and each warp
// parks its part of the rows in `rowp`; after the last chunk the consumers
// finish all rows at once (parts added in warp order, so the result does not
// depend on timing) and apply the phase's epilogue.
template <int DT, bool LC>
__device__ __forceinline__ void gemv_consume(Consumer& c, const DMat& m, const ChunkGeo& ck, int r0, int r1,
                                             const Lanes& L, const XReg<DT>& xr, float* rowp, Epi& epi, int tk) {
    constexpr int ES = DT == LLM_Q8_0 ? 1 : (DT == LLM_F16 ? 2 : 4);
    constexpr int RPP = RowsPerPass<DT>::value;
    const int tw = m.tw, teams = m.teams;
    const int xoff = L.col0 * ES, soff = ck.soff + L.lit * 2;
    const int sw = DT == LLM_Q8_0 ? (c.lane >> 2) & 1 : 0;
    const int wl = tw < 32 ? tw : 32;                 // lanes of a team within one warp
    const int wpr = tw > 32 ? tw / 32 : 1;            // warps of a team
    // the warp's first team decides how many passes the warp makes (every lane
    // of a warp takes part in the shuffles of every pass)
    const int wteam = tw <= 32 ? c.warp * (32 / tw) : c.warp / wpr;
    for (int r = r0; r < r1; r += ck.rpc) {
        const int n = min(ck.rpc, r1 - r);
        int slot;
        const uint8_t* buf = c.next_slot(slot);
        if (r == r0 && tk >= 0 && c.tid == 0) trace_mark(c.p, tk);
        FMARK(c, 6 + 2 * min((r - r0) / ck.rpc, 3));
        const uint8_t* sbase = buf + (ck.sfix >= 0 ? ck.sfix : n * ck.rowq);
        const uint32_t sbuf = smem_addr(buf), ssc = smem_addr(sbase);
        if (wl < RPP) {
            // teams narrower than the rows of a pass: one row per team and pass
            for (int j = 0; wteam + j * teams < n; j++) {
                const int rr = L.team + j * teams;
                const bool real = L.active && rr < n;
                const int mrow = real ? rr : 0;
                float v = real ? lane_row<DT>(buf + (size_t)mrow * ck.rowq + xoff, sbase + mrow * ck.rowd + soff, xr,
                                              L.nseg)
                               : 0.f;
                for (int o = wl >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (real && L.lit == 0) epi.row(r + rr, v);
            }
        } else {
            // RPP consecutive rows per team and pass.  A transposed butterfly
            // over the team's wl lanes reduces the RPP values at once: the
            // first step (distance wl/2) halves the values a lane carries, the
            // second (RPP 4, distance wl/4) halves them again, the rest are
            // plain; lane t of the team ends with row k = its bits at wl/2
            // (and wl/4).  Whole-warp teams of several warps park each warp's
            // part and finish the rows after the last chunk.
            const int h = wl >> 1, q = wl >> 2;
            float* rp = rowp + (size_t)(r - r0) * wpr + (tw > 32 ? c.warp % wpr : 0);
            for (int j = 0;; j++) {
                if ((wteam + j * teams) * RPP >= n) break;
                const int rbase = (L.team + j * teams) * RPP;
                uint32_t wq[RPP], ws[RPP];
#pragma unroll
                for (int k = 0; k < RPP; k++) {
                    const int mr = min(rbase + k, n - 1);
                    wq[k] = sbuf + (uint32_t)(mr * ck.rowq + xoff);
                    ws[k] = ssc + (uint32_t)(mr * ck.rowd + soff);
                }
                float v[RPP];
                lane_rows<DT, RPP>(wq, ws, xr, L.active && rbase < n ? L.nseg : 0, sw, v);
                float keep;
                int k, lo;
                if constexpr (RPP == 4) {
                    const bool u1 = (c.lane & h) != 0;
                    const float a0 = (u1 ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, u1 ? v[0] : v[2], h);
                    const float a1 = (u1 ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, u1 ? v[1] : v[3], h);
                    const bool u2 = (c.lane & q) != 0;
                    keep = (u2 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, u2 ? a0 : a1, q);
                    for (int o = q >> 1; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
                    k = (u1 ? 2 : 0) + (u2 ? 1 : 0);
                    lo = q;
                } else {
                    const bool u1 = (c.lane & h) != 0;
                    keep = (u1 ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, u1 ? v[0] : v[1], h);
                    for (int o = h >> 1; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
                    k = u1 ? 1 : 0;
                    lo = h;
                }
                if ((c.lane & (lo - 1)) == 0 && L.active && rbase + k < n) {
                    if (tw > 32) rp[(rbase + k) * wpr] = keep;
                    else epi.row(r + rbase + k, keep);
                }
            }
        }
        c.release(slot);
        FMARK(c, 7 + 2 * min((r - r0) / ck.rpc, 3));
    }
    if (tw > 32) {
        // finish every row: the warps' parts added in warp order
        consumer_sync();
        FMARK(c, 14);
        for (int i = c.tid; i < r1 - r0; i += kConsumers) {
            float t = 0.f;
            for (int k = 0; k < wpr; k++) t += rowp[i * wpr + k];
            epi.row(r0 + i, t);
        }
    }
    epi.template finish<LC>(c);
    // the next phase's staging must not overwrite what a warp still reads
    // (the gains, the (gate, up) sums, the row partials)
    consumer_sync();
    FMARK(c, 15);
#ifdef LLM_TRACE
    if (c.tid == 0 && tk >= 0 && c.p.trace) c.p.trace[(size_t)blockIdx.x * kTraceSlots + tk - 160 + 768] = c.waited;
    c.waited = 0;
#endif
}

// ------------------------------------------------------------------ RoPE --
// "The Forward Pass in Java", Example 6 and "What a Llama model computes, and
// why" §2.4: pair i turns by theta_i, where theta starts at pos and is
// multiplied by theta_scale once per pair in float (the same chain as ggml's
// rope cache), then divided by the pair's frequency factor.  cos/sin are taken
// in double and rounded to float.  One table per step, shared by q and k.
__device__ void rope_table(const StepParams& p, Smem& sm, int tid) {
    for (int i = tid; i < p.rope_dims / 2; i += kConsumers) {
        float th = (float)p.pos;
        for (int j = 0; j < i; j++) th = __fmul_rn(th, p.theta_scale);
        if (p.rope_freqs) th = __fdiv_rn(th, __ldg(p.rope_freqs + i));
        double s, c;
        sincos((double)th, &s, &c);
        sm.rope_c()[i] = (float)c;
        sm.rope_s()[i] = (float)s;
    }
}

__device__ __forceinline__ void rope_apply(const StepParams& p, const Smem& sm, float* v, int i) {
    const float c = sm.rope_c()[i], s = sm.rope_s()[i];
    const int a = p.neox ? i : 2 * i, b = p.neox ? i + p.rope_dims / 2 : 2 * i + 1;
    const float x0 = v[a], x1 = v[b];
    v[a] = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
    v[b] = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
}

// K/V row `pos` of one kv head, rounded to F16 to nearest even ("The Forward
// Pass in Java", Example 10), at element pos*kv_dim + off + i (Example 7).
__device__ __forceinline__ void store_kv(__half* kc, __half* vc, int pos, int kv_dim, int off, int i, __half k,
                                         __half v) {
    const size_t e = (size_t)pos * kv_dim + off + i;
    kc[e] = k;
    vc[e] = v;
}
__device__ __forceinline__ void store_kv_checked(const StepParams& p, __half* kc, __half* vc, int g, int i, __half k,
                                                 __half v) {
    if (LLM_IN_BOUNDS(p.err, p.pos >= 0 && p.pos < p.max_seq && g * p.hd + i < p.kv_dim))
        store_kv(kc, vc, p.pos, p.kv_dim, g * p.hd, i, k, v);
}

// score / sqrt(head_dim) ("The Forward Pass in Java", Example 11): a
// power-of-two divisor (head_dim 64, 256, ...) divides exactly as a multiply
// by its reciprocal, the same bits as the IEEE division at a fraction of the
// instructions.
__device__ __forceinline__ float attn_scale(float x, float div) {
    return (__float_as_uint(div) & 0x007FFFFFu) == 0u ? __fmul_rn(x, __frcp_rn(div)) : __fdiv_rn(x, div);
}

// ------------------------------------------------------------- attention --
// One unit = the positions [t0, t1) of kv head g, for its gq query heads
// ("The Forward Pass in Java", Example 11: scores q.k / sqrt(hd), softmax over
// the positions, weighted sum of the V rows).  The unit keeps a running max m
// and sum l per head across its chunks (online softmax) and writes its partial
// (m, l, acc): acc[h][d] at part[(h*max_splits + s)*hd + d], (m, l) at
// part[n_heads*max_splits*hd + 2*(h*max_splits + s)].  The O phase merges the
// splits (stage_merged): per head M = max_s m_s,
// w_s = e^(m_s - M) / sum_s' e^(m_s' - M) l_s', attn = sum_s w_s acc_s.
//
// Scratch shared by both forms of the unit: q_s [gq][hd] (rotated q, F32),
// kf [hd] (this position's k, F32), kp and vp [hd] each (its K and V rows,
// F16); the scalar form's score buffers follow.

// q of the unit's heads, rotated, into q_s (under llama.cpp rounding, LC,
// then rounded to F16: the q.k products take an F16 q); the writer (the unit
// that holds this step's position) rotates k, rounds K and V to F16 into
// kp/vp and stores them in the cache.  Ends with the scratch visible to all
// consumers.
template <bool LC>
__device__ void attention_prologue(Consumer& c, const LayerDev& L, int layer, int g, bool writer) {
    const StepParams& p = c.p;
    Smem& sm = c.sm;
    const int tid = c.tid, hd = p.hd, gq = p.n_heads / p.n_kv, h0 = g * gq, GD = gq * hd;
    float* q_s = sm.xs();
    float* kf = q_s + GD;
    __half* kp = reinterpret_cast<__half*>(kf + hd);
    __half* vp = kp + hd;
    const unsigned long long* qkv = c.tv(layer, c.tl().qkv);
    {
        float qv[2], kv = 0.f, vv = 0.f;
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const int i = tid + k * kConsumers;
            qv[k] = i < GD ? poll1(qkv + h0 * hd + i, c.tag, p.err) : 0.f;
        }
        if (writer && tid < hd) {
            kv = poll1(qkv + p.q_dim + g * hd + tid, c.tag, p.err);
            vv = poll1(qkv + p.q_dim + p.kv_dim + g * hd + tid, c.tag, p.err);
        }
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const int i = tid + k * kConsumers;
            if (i < GD) q_s[i] = qv[k];
        }
        if (writer && tid < hd) {
            kf[tid] = kv;
            vp[tid] = __float2half_rn(vv);
        }
    }
    consumer_sync();
    for (int i = tid; i < gq * (p.rope_dims / 2); i += kConsumers)
        rope_apply(p, sm, q_s + (i / (p.rope_dims / 2)) * hd, i % (p.rope_dims / 2));
    if (writer)
        for (int i = tid; i < p.rope_dims / 2; i += kConsumers) rope_apply(p, sm, kf, i);
    consumer_sync();
    if constexpr (LC)
        for (int i = tid; i < GD; i += kConsumers) q_s[i] = f16_round(q_s[i]);
    if (writer && tid < hd) {
        const __half kh = __float2half_rn(kf[tid]);
        kp[tid] = kh;
        store_kv_checked(p, L.kc, L.vc, g, tid, kh, vp[tid]);
    }
    consumer_sync();                                               // kp, vp visible
}

// Scalar form (any head size).  Under llama.cpp rounding (LC) the unit makes
// two passes over its positions ("What a Llama model computes, and why" §8:
// each probability is rounded to F16 after division by the softmax sum over
// all positions, so that sum must be known first).  Pass 0 reads only the K
// tiles and finds the unit's (m, l); the units of a kv head exchange them
// (tagged words after the (m, l) partials; every unit runs on its own CTA, all
// resident, and each reaches the exchange without waiting on another unit),
// and each forms the head's M = max_s m_s and L = sum_s e^(m_s - M) l_s from
// the same values in the same order.  Pass 1 recomputes the scores, takes
// p_t = f16(e^(s_t - M) / L) and accumulates p_t V_t with no rescaling.
template <bool LC>
__device__ bool attention_unit(Consumer& c, const LayerDev& L, int layer, int unit) {
    const StepParams& p = c.p;
    Smem& sm = c.sm;
    const int tid = c.tid, warp = c.warp, lane = c.lane;
    const int hd = p.hd, gq = p.n_heads / p.n_kv, P = p.attn_rows, S = p.splits;
    int g, s, t0, t1;
    unit_range(p, unit, S, g, s, t0, t1);
    const int h0 = g * gq, GD = gq * hd;
    float* q_s = sm.xs();                                          // [gq][hd]
    __half* kp = reinterpret_cast<__half*>(q_s + GD + hd);         // [hd] this position's K row (F16)
    __half* vp = kp + hd;                                          // [hd] this position's V row (F16)
    float* sc = q_s + GD + 2 * hd;                                 // [2][gq][P] scores, then probabilities
    float* ml = sc + 2 * gq * P;                                   // [2][gq] running max m, sum l (LC pass 1: M, L)
    float* corr = ml + 2 * gq;                                     // [2][gq] rescale of the chunk's old sums

    const bool writer = t0 <= p.pos && p.pos < t1;
    attention_prologue<LC>(c, L, layer, g, writer);
    if (tid < gq) { ml[tid] = -INFINITY; ml[gq + tid] = 0.f; }     // read after the first chunk's scores sync
    // PV work split: thread t accumulates the output pair o2 = t % (GD/2)
    // (elements 2*o2, 2*o2+1) over positions with index % NSPLIT == t / (GD/2).
    const int GD2 = GD / 2;
    const int NSPLIT = kConsumers / GD2;
    const int o2 = tid % GD2, sp = tid / GD2;
    const bool pv_active = sp < NSPLIT;
    const int oh = (2 * o2) / hd, oi = (2 * o2) % hd;
    const int nh2 = hd / 2;
    const int prow = p.pos - t0;                                   // this step's position within the unit
    float2 acc = make_float2(0.f, 0.f);
    unsigned long long* part_acc = c.part(layer);
    unsigned long long* part_ml = part_acc + (size_t)p.n_heads * p.max_splits * hd;

    int ci = 0;
    for (int pass = 0; pass < (LC ? 2 : 1); pass++) {
        const bool pv = !LC || pass == 1;                          // this pass accumulates P.V
        if (LC && pass == 1) {
            // exchange the splits' (m, l) and form each head's (M, L)
            consumer_sync();                                       // ml (also when the unit has no positions)
            unsigned long long* stats = part_ml + 2 * (size_t)p.n_heads * p.max_splits;
            for (int h = warp; h < gq; h += kConsumerWarps) {
                const size_t hb = (size_t)(h0 + h) * p.max_splits;
                const float mo = ml[h], lo = ml[gq + h];
                if (lane == 0) {
                    c.st_part(stats + 2 * (hb + s), mo);
                    c.st_part(stats + 2 * (hb + s) + 1, lo);
                }
                float2 v = make_float2(-INFINITY, 0.f);
                if (lane < S) v = lane == s ? make_float2(mo, lo) : poll2(stats + 2 * (hb + lane), c.tag, p.err);
                const float M = warp_max(v.x);
                const float Ls = warp_sum(v.x == -INFINITY ? 0.f : expf(v.x - M) * v.y);
                __syncwarp();
                if (lane == 0) { ml[h] = M; ml[gq + h] = Ls; }
            }
            consumer_sync();
            if (c.aborted()) return false;
        }
        for (int c0 = t0; c0 < t1; c0 += P, ci++) {
            const int np = min(P, t1 - c0);
            int slot;
            const uint8_t* buf = c.next_slot(slot);
            const __half* ks = reinterpret_cast<const __half*>(buf);
            const __half* vs = ks + (size_t)P * hd;
            float* scb = sc + (ci & 1) * gq * P;
            float* corrb = corr + (ci & 1) * gq;
            // scores: thread (h, position); the K row of this step's position is
            // the one just computed, not the copy the tile load may have read.
            // Four partial sums; the start column rotates with the lane so that a
            // warp's reads fall in different banks.
            for (int idx = tid; idx < gq * np; idx += kConsumers) {
                const int h = idx / np, pp = idx % np;
                const float2* q2 = reinterpret_cast<const float2*>(q_s + h * hd);
                const __half2* k2 = reinterpret_cast<const __half2*>(
                    writer && c0 + pp - t0 == prow ? kp : ks + (size_t)pp * hd);
                float2 a0 = make_float2(0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
                int j = lane % nh2;
                int k = 0;
                for (; k + 4 <= nh2; k += 4) {
                    const int j1 = j + 1 == nh2 ? 0 : j + 1;
                    const int j2 = j1 + 1 == nh2 ? 0 : j1 + 1;
                    const int j3 = j2 + 1 == nh2 ? 0 : j2 + 1;
                    a0 = __ffma2_rn(__half22float2(k2[j]), q2[j], a0);
                    a1 = __ffma2_rn(__half22float2(k2[j1]), q2[j1], a1);
                    a2 = __ffma2_rn(__half22float2(k2[j2]), q2[j2], a2);
                    a3 = __ffma2_rn(__half22float2(k2[j3]), q2[j3], a3);
                    j = j3 + 1 == nh2 ? 0 : j3 + 1;
                }
                for (; k < nh2; k++) {
                    a0 = __ffma2_rn(__half22float2(k2[j]), q2[j], a0);
                    j = j + 1 == nh2 ? 0 : j + 1;
                }
                const float2 a = make_float2((a0.x + a1.x) + (a2.x + a3.x), (a0.y + a1.y) + (a2.y + a3.y));
                scb[h * P + pp] = attn_scale(a.x + a.y, p.attn_div);
            }
            consumer_sync();
            if (c.aborted()) return false;
            if (warp < gq) {
                const int h = warp;
                if (LC && pv) {
                    // the head's global (M, L): p_t = f16(e^(s_t - M) / L), no rescaling
                    const float M = ml[h], Ls = ml[gq + h];
                    for (int pp = lane; pp < np; pp += 32)
                        scb[h * P + pp] = f16_round(__fdiv_rn(expf(__fsub_rn(scb[h * P + pp], M)), Ls));
                    if (lane == 0) corrb[h] = 1.0f;
                } else {
                    float mloc = -INFINITY;
                    for (int pp = lane; pp < np; pp += 32) mloc = fmaxf(mloc, scb[h * P + pp]);
                    mloc = warp_max(mloc);
                    const float mold = ml[h], mnew = fmaxf(mold, mloc);
                    float sum = 0.f;
                    for (int pp = lane; pp < np; pp += 32) {
                        const float e = expf(scb[h * P + pp] - mnew);
                        scb[h * P + pp] = e;
                        sum += e;
                    }
                    sum = warp_sum(sum);
                    if (lane == 0) {
                        const float cr = expf(mold - mnew);       // 0 on the first chunk (mold = -inf)
                        ml[h] = mnew;
                        ml[gq + h] = ml[gq + h] * cr + sum;
                        corrb[h] = cr;
                    }
                }
            }
            consumer_sync();
            if (pv && pv_active) {
                const float cr = corrb[oh];
                float2 v0 = make_float2(acc.x * cr, acc.y * cr), v1 = make_float2(0.f, 0.f), v2 = v1, v3 = v1;
                const float* e = scb + oh * P;
                auto vrow = [&](int pp) {
                    const __half* r = writer && c0 + pp - t0 == prow ? vp : vs + (size_t)pp * hd;
                    return __half22float2(*reinterpret_cast<const __half2*>(r + oi));
                };
                int pp = sp;
                for (; pp + 3 * NSPLIT < np; pp += 4 * NSPLIT) {
                    v0 = __ffma2_rn(make_float2(e[pp], e[pp]), vrow(pp), v0);
                    v1 = __ffma2_rn(make_float2(e[pp + NSPLIT], e[pp + NSPLIT]), vrow(pp + NSPLIT), v1);
                    v2 = __ffma2_rn(make_float2(e[pp + 2 * NSPLIT], e[pp + 2 * NSPLIT]), vrow(pp + 2 * NSPLIT), v2);
                    v3 = __ffma2_rn(make_float2(e[pp + 3 * NSPLIT], e[pp + 3 * NSPLIT]), vrow(pp + 3 * NSPLIT), v3);
                }
                for (; pp < np; pp += NSPLIT) v0 = __ffma2_rn(make_float2(e[pp], e[pp]), vrow(pp), v0);
                acc = make_float2((v0.x + v1.x) + (v2.x + v3.x), (v0.y + v1.y) + (v2.y + v3.y));
            }
            c.release(slot);
        }
    }
    // combine the PV position splits and write this unit's partial
    if (pv_active) {
        sm.comb()[sp * GD + 2 * o2] = acc.x;
        sm.comb()[sp * GD + 2 * o2 + 1] = acc.y;
    }
    consumer_sync();
    for (int oo = tid; oo < GD; oo += kConsumers) {
        float v = 0.f;
        for (int k = 0; k < NSPLIT; k++) v += sm.comb()[k * GD + oo];
        const int hh = oo / hd, ii = oo % hd;
        const size_t hs = (size_t)(h0 + hh) * p.max_splits + s;
        c.st_part(part_acc + hs * hd + ii, v);
        if (ii == 0) {
            c.st_part(part_ml + 2 * hs, ml[hh]);
            c.st_part(part_ml + 2 * hs + 1, ml[gq + hh]);
        }
    }
    consumer_sync();                                               // comb, scratch free
    return true;
}

// Shared-memory address of 16-byte chunk `ch` of row r of a K or V tile: the
// tile is hd / W sub-tiles of [P][W] F16 (W = 64 when hd is a multiple of
// 64, else hd), each written by TMA with the swizzle of its row width (128,
// 64 or 32 bytes: address bits 7.. XORed into the chunk bits 4..; none for
// other widths).  The ring is 1024-byte aligned, so the pattern computed on
template <int HD>
__device__ __forceinline__ uint32_t kv_chunk(uint32_t tile, int P, int r, int ch) {
    constexpr int W = HD % 64 == 0 ? 64 : HD;
    constexpr uint32_t SWZ = W * 2 == 128 ? 7u : W * 2 == 64 ? 3u : W * 2 == 32 ? 1u : 0u;
    constexpr int CPR = W / 8;
    const int sub = ch / CPR, cc = ch - sub * CPR;
    const uint32_t a = tile + (uint32_t)(sub * P + r) * (uint32_t)(W * 2) + (uint32_t)cc * 16u;
    return a ^ (((a >> 7) & SWZ) << 4);
}

// The two F16 parts of x: hi = x rounded to F16, lo = the rest rounded to
// F16, so that hi + lo carries about 22 bits of x and every product of a part
// with an F16 value is exact in F32.
__device__ __forceinline__ __half f16_part(float x, int part) {
    const __half hi = __float2half_rn(x);
    return part ? __float2half_rn(x - __half2float(hi)) : hi;
}
__device__ __forceinline__ uint32_t pack_h2(__half a, __half b) {
    return (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
}

// Tensor-core form (head_dim HD in {32, 48, 64}, gq <= 4): each warp
// takes 16-position tiles of the chunk.  Scores are one m16n8k16 product per
// 8 positions and 16 dimensions: A rows 2h and 2h+1 hold the F16 hi and lo
// parts of head h's q, B the K rows (ldmatrix from the swizzled tile), so the
// two rows of a head add up to q.k with F32 accumulation.  The warp keeps its
// own online softmax (m, l per head) over its tiles; the probabilities, again
// split into hi and lo rows, multiply the V rows (ldmatrix.trans) into the
// warp's accumulators.  At the end the warps' (m, l, acc) are merged in
// shared memory into the unit's partial.
template <int HD>
__device__ bool attention_unit_mma(Consumer& c, const LayerDev& L, int layer, int unit) {
    const StepParams& p = c.p;
    Smem& sm = c.sm;
    const int tid = c.tid, warp = c.warp, lane = c.lane;
    const int gq = p.n_heads / p.n_kv, P = p.attn_rows, S = p.splits;
    int g, s, t0, t1;
    unit_range(p, unit, S, g, s, t0, t1);
    const int h0 = g * gq, GD = gq * HD;
    const float* q_s = sm.xs();
    const __half* kp = reinterpret_cast<const __half*>(q_s + GD + HD);
    const __half* vp = kp + HD;
    const bool writer = t0 <= p.pos && p.pos < t1;
    attention_prologue<false>(c, L, layer, g, writer);
    if (tid == 0) trace_mark(p, 576 + 4 * layer);

    // A fragments of q: row r = lane / 4 is part (r & 1) of head r / 2
    const int r = lane >> 2, t = lane & 3, hq = r >> 1, part = r & 1;
    uint32_t aq[HD / 16][2];
#pragma unroll
    for (int ks = 0; ks < HD / 16; ks++)
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const int d = ks * 16 + 8 * j + 2 * t;
            const float x0 = hq < gq ? q_s[hq * HD + d] : 0.f, x1 = hq < gq ? q_s[hq * HD + d + 1] : 0.f;
            aq[ks][j] = pack_h2(f16_part(x0, part), f16_part(x1, part));
        }
    float m_run = -INFINITY, l_run = 0.f;
    float acc[HD / 8][2];
#pragma unroll
    for (int n = 0; n < HD / 8; n++) acc[n][0] = acc[n][1] = 0.f;

    int slot = 0;
    const uint8_t* buf = nullptr;
    for (int c0 = t0; c0 < t1; c0 += P) {
        if (buf) c.release(slot);
        const int np = min(P, t1 - c0);
        buf = c.next_slot(slot);
        const uint32_t kt = smem_addr(buf), vt = kt + (uint32_t)(P * HD * 2);
        if (writer && c0 <= p.pos && p.pos < c0 + np) {
            // this step's K and V rows replace the copies the tile load read
            const int row = p.pos - c0;
            if (tid < HD / 8) {
                const uint4 kv = reinterpret_cast<const uint4*>(kp)[tid];
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(kv_chunk<HD>(kt, P, row, tid)),
                             "r"(kv.x), "r"(kv.y), "r"(kv.z), "r"(kv.w) : "memory");
            } else if (tid < HD / 4) {
                const uint4 vv = reinterpret_cast<const uint4*>(vp)[tid - HD / 8];
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(kv_chunk<HD>(vt, P, row, tid - HD / 8)),
                             "r"(vv.x), "r"(vv.y), "r"(vv.z), "r"(vv.w) : "memory");
            }
            fence_proxy_async_smem();
        }
        consumer_sync();
        if (c.aborted()) return false;
        const int nt = (np + 15) >> 4;
        for (int tile = warp; tile < nt; tile += kConsumerWarps) {
            const int pj = tile * 16;
            // scores of positions pj + 8 * ns + 2t + {0, 1}, rows r (parts of head hq)
            float sc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
            {
                int kr = pj + ((lane >> 4) & 1) * 8 + (lane & 7);
                if (kr >= np) kr = 0;                                  // masked below
#pragma unroll
                for (int ks = 0; ks < HD / 16; ks++) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kv_chunk<HD>(kt, P, kr, 2 * ks + ((lane >> 3) & 1)), b0, b1, b2, b3);
                    mma_rows8(sc[0][0], sc[0][1], aq[ks][0], aq[ks][1], b0, b1);
                    mma_rows8(sc[1][0], sc[1][1], aq[ks][0], aq[ks][1], b2, b3);
                }
            }
            float e[2][2], mt = -INFINITY;
#pragma unroll
            for (int ns = 0; ns < 2; ns++)
#pragma unroll
                for (int k = 0; k < 2; k++) {
                    const float v = sc[ns][k] + __shfl_xor_sync(0xffffffffu, sc[ns][k], 4);   // hi + lo
                    const int pos = pj + 8 * ns + 2 * t + k;
                    e[ns][k] = pos < np ? attn_scale(v, p.attn_div) : -INFINITY;
                    mt = fmaxf(mt, e[ns][k]);
                }
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
            const float m_new = fmaxf(m_run, mt);
            const float cr = expf(m_run - m_new);                      // 0 on the warp's first tile
            float ls = 0.f;
#pragma unroll
            for (int ns = 0; ns < 2; ns++)
#pragma unroll
                for (int k = 0; k < 2; k++) {
                    e[ns][k] = expf(e[ns][k] - m_new);
                    ls += e[ns][k];
                }
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            l_run = l_run * cr + ls;
            m_run = m_new;
#pragma unroll
            for (int n = 0; n < HD / 8; n++) {
                acc[n][0] *= cr;
                acc[n][1] *= cr;
            }
            // probabilities as A: columns 2t, 2t+1 (positions of n-subtile 0) and 2t+8, 2t+9 (subtile 1)
            const uint32_t pa0 = pack_h2(f16_part(e[0][0], part), f16_part(e[0][1], part));
            const uint32_t pa2 = pack_h2(f16_part(e[1][0], part), f16_part(e[1][1], part));
            int vr = pj + ((lane >> 3) & 1) * 8 + (lane & 7);
            if (vr >= np) vr = 0;                                      // probability 0
#pragma unroll
            for (int n = 0; n < HD / 8; n += 2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(kv_chunk<HD>(vt, P, vr, n + (lane >> 4)), b0, b1, b2, b3);
                mma_rows8(acc[n][0], acc[n][1], pa0, pa2, b0, b1);
                mma_rows8(acc[n + 1][0], acc[n + 1][1], pa0, pa2, b2, b3);
            }
        }
    }
    unsigned long long* part_acc = c.part(layer);
    unsigned long long* part_ml = part_acc + (size_t)p.n_heads * p.max_splits * HD;
    if (!buf) {                                                    // no positions: an empty partial
        for (int oo = tid; oo < GD; oo += kConsumers) {
            const size_t hs = (size_t)(h0 + oo / HD) * p.max_splits + s;
            c.st_part(part_acc + hs * HD + oo % HD, 0.f);
            if (oo % HD == 0) {
                c.st_part(part_ml + 2 * hs, -INFINITY);
                c.st_part(part_ml + 2 * hs + 1, 0.f);
            }
        }
        consumer_sync();
        return true;
    }
    // the warps' partials, in the last slot (its tile is no longer read)
    consumer_sync();
    float* wpart = reinterpret_cast<float*>(const_cast<uint8_t*>(buf));   // [warp][gq][HD + 2]
    const int WS = gq * (HD + 2);
#pragma unroll
    for (int n = 0; n < HD / 8; n++)
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const float o = acc[n][k] + __shfl_xor_sync(0xffffffffu, acc[n][k], 4);
            if (part == 0 && hq < gq) wpart[warp * WS + hq * (HD + 2) + n * 8 + 2 * t + k] = o;
        }
    if (part == 0 && hq < gq && t == 0) {
        wpart[warp * WS + hq * (HD + 2) + HD] = m_run;
        wpart[warp * WS + hq * (HD + 2) + HD + 1] = l_run;
    }
    consumer_sync();
    // the warps' rescale factors, once per (head, warp): warp hh takes head hh,
    // lane w warp w's running max; M = the head's max, f_w = e^(m_w - M), and
    // the head's sum l = sum_w f_w l_w (warp order) with its (m, l) stored
    float* fw = sm.comb();                                         // [gq][kConsumerWarps]
    if (warp < gq) {
        const int hh = warp;
        const float mw = lane < kConsumerWarps ? wpart[lane * WS + hh * (HD + 2) + HD] : -INFINITY;
        const float M = warp_max(mw);
        const float f = mw == -INFINITY ? 0.f : expf(mw - M);
        if (lane < kConsumerWarps) fw[hh * kConsumerWarps + lane] = f;
        __syncwarp();
        if (lane == 0) {
            float l = 0.f;
            for (int w = 0; w < kConsumerWarps; w++) l = fmaf(fw[hh * kConsumerWarps + w], wpart[w * WS + hh * (HD + 2) + HD + 1], l);
            const size_t hs = (size_t)(h0 + hh) * p.max_splits + s;
            c.st_part(part_ml + 2 * hs, M);
            c.st_part(part_ml + 2 * hs + 1, l);
        }
    }
    consumer_sync();
    for (int oo = tid; oo < GD; oo += kConsumers) {
        const int hh = oo / HD, ii = oo % HD;
        float v = 0.f;
#pragma unroll 5
        for (int w = 0; w < kConsumerWarps; w++) v = fmaf(fw[hh * kConsumerWarps + w], wpart[w * WS + hh * (HD + 2) + ii], v);
        const size_t hs = (size_t)(h0 + hh) * p.max_splits + s;
        c.st_part(part_acc + hs * HD + ii, v);
    }
    fence_proxy_async_smem();                                      // the slot's next fill is a TMA write
    consumer_sync();
    c.release(slot);
    if (tid == 0) trace_mark(p, 576 + 4 * layer + 1);
    return true;
}

template <bool LC>
__device__ bool attention_any(Consumer& c, const LayerDev& L, int layer, int unit) {
    if constexpr (LC) return attention_unit<true>(c, L, layer, unit);   // the two-pass scalar form
    if (c.p.attn_mma) {
        switch (c.p.hd) {
            case 32: return attention_unit_mma<32>(c, L, layer, unit);
            case 48: return attention_unit_mma<48>(c, L, layer, unit);
            case 64: return attention_unit_mma<64>(c, L, layer, unit);
            default: break;
        }
    }
    return attention_unit<false>(c, L, layer, unit);
}
// ----------------------------------------------------------------- kernel --
template <int DT, bool LC>
__device__ bool consumer_main(const StepParams& p, Smem& sm) {
    Consumer c(p, sm);
    const int tid = c.tid, G = gridDim.x;
    int token = __ldcg(p.token_in);
    if (token < 0 || token >= p.vocab) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, kErrToken);
        token = 0;
    }
    // this CTA's share of the other parity's accumulators (the next step's)
    {
        unsigned long long* other = p.delta + (size_t)((c.tag & 1u) ^ 1u) * p.n_layers * 2 * p.dim;
        int z0, z1;
        cta_rows(p.n_layers * 2 * p.dim, z0, z1);
        for (int i = z0 + tid; i < z1; i += kConsumers) other[i] = 0ull;
    }
    c.prefetch_gains(p.layers[0].attn_norm, p.dim);
    rope_table(p, sm, tid);
    const Part pt = cta_part(p.ngrp);
    const int fdg = p.dv.m.cols;
    int rg0, rg1;            // this CTA's rows of its group's Wo and Wdown column blocks
    share(p.dim, pt.j, pt.n, rg0, rg1);
    int u0, u1;              // this CTA's FFN columns (gate/up super-rows)
    share(fdg, pt.j, pt.n, u0, u1);
    u0 += pt.g * fdg;
    u1 += pt.g * fdg;
    float4* xv = reinterpret_cast<float4*>(sm.xs());
    // Every GEMV phase (QKV, O, GU, DOWN of each layer, then the logits) goes
    // through the one call site below, so the kernel holds one copy of the
    // GEMV code.
    enum { kSrcResidual, kSrcTagged, kSrcMerged };
    const int nph = 4 * p.n_layers + 1;
    unsigned long long best = 0ull;
    for (int ph = 0; ph < nph; ph++) {
        const int l = ph >> 2, k = ph & 3;
        const bool last = ph == nph - 1;
        const LayerDev& L = p.layers[last ? p.n_layers - 1 : l];
        DMat m;
        ChunkGeo ck;
        int r0, r1, n, src;
        const unsigned long long* sv = nullptr;   // residual: accumulator words (nullptr: embedding); tagged: vector
        const float* gains = nullptr;
        float* rowp = sm.rowp();
        Epi e{};
        e.tag = c.tag;
        e.err = p.err;
        if (last) {
            // ---- LOGITS + argmax
            if (tid == 0) trace_mark(p, 240);
            m = p.out;
            cta_rows(m.rows, r0, r1);
            ck = rows_geo(m, DT);
            src = kSrcResidual;
            sv = c.acc(p.n_layers - 1, 1);
            n = p.dim;
            gains = sm.gains();
            rowp = sm.res();                       // the residual is dead once staged
            e.kind = Epi::kLogits;
            e.logits = p.logits;
        } else if (k == 0) {
            // ---- QKV
            if (tid == 0) trace_mark(p, 10 * l);
            m = L.qkv;
            cta_rows(m.rows, r0, r1);
            ck = rows_geo(m, DT);
            if (L.qkv_bias)
                for (int i = tid; i < r1 - r0; i += kConsumers) sm.bias()[i] = __ldg(L.qkv_bias + r0 + i);
            src = kSrcResidual;
            sv = l == 0 ? nullptr : c.acc(l - 1, 1);
            n = p.dim;
            gains = sm.gains();
            e.kind = Epi::kStore;
            e.out = c.tv(l, c.tl().qkv);
            e.bias = L.qkv_bias ? sm.bias() : nullptr;
            e.base = r0;
        } else if (k == 1) {
            // ---- ATTN, then O (this CTA's rows of its group's columns of Wo)
            if (tid == 0) trace_mark(p, 10 * l + 2);
            const int units = p.n_kv * p.splits;
            for (int unit = blockIdx.x; unit < units; unit += G)
                if (!attention_any<LC>(c, L, l, unit)) return false;
            if (tid == 0) trace_mark(p, 10 * l + 3);
            m = p.ov.m;
            r0 = rg0;
            r1 = rg1;
            ck = view_geo(p.ov, pt.g);
            src = kSrcMerged;
            n = m.cols;
            e.kind = Epi::kAccum;
            e.out = c.acc(l, 0);
        } else if (k == 2) {
            // ---- GU (this CTA's FFN columns)
            if (tid == 0) trace_mark(p, 10 * l + 6);
            m = L.gu;
            r0 = 2 * u0;
            r1 = 2 * u1;
            ck = rows_geo(m, DT);
            src = kSrcResidual;
            sv = c.acc(l, 0);
            n = p.dim;
            gains = sm.gains();
            e.kind = Epi::kSwiGLU;
            e.out = c.tv(l, c.tl().u);
            e.sm = sm.bias();
            e.base = u0;
            e.end = u1;
        } else {
            // ---- DOWN (this CTA's rows of its group's columns of Wdown)
            if (tid == 0) trace_mark(p, 10 * l + 8);
            m = p.dv.m;
            r0 = rg0;
            r1 = rg1;
            ck = view_geo(p.dv, pt.g);
            src = kSrcTagged;
            sv = c.tv(l, c.tl().u) + (size_t)pt.g * fdg;
            n = fdg;
            e.kind = Epi::kAccum;
            e.out = c.acc(l, 1);
        }
        if (e.kind == Epi::kAccum) {
            e.lo = p.delta;
            e.n = p.delta_words;
        } else if (e.kind == Epi::kLogits) {
            e.n = p.logits_limit;
        } else {
            e.lo = p.tv;
            e.n = p.tv_words;
        }
#ifdef LLM_TRACE
        c.fine = !last && l == 8 ? 960 + 16 * k : -1;
#endif
        FMARK(c, 0);
        NormSum<LC> ss = 0;
        if (src == kSrcResidual) ss = stage_residual<DT, LC>(c, sv, token, gains != nullptr, xv);
        else if (src == kSrcTagged) stage_tagged<DT, LC>(c, sv, n, xv);
        else stage_merged<DT, LC>(c, l, pt.g, xv);
        const Lanes Ln = lane_layout<DT>(c, m);
        XReg<DT> xr;
        e.scale = lanes_prep<DT, LC>(c, Ln, n, gains != nullptr, ss, xr);
        FMARK(c, 5);
        const int jt = last ? -1 : k;                               // trace: QKV 0, O 1, GU 2, DOWN 3
        if (tid == 0 && jt >= 0) trace_mark(p, 512 + 4 * l + jt);
        gemv_consume<DT, LC>(c, m, ck, r0, r1, Ln, xr, rowp, e, jt >= 0 ? 160 + 4 * l + jt : -1);
        if (last) {
            best = e.best;
        } else {
            if (tid == 0) trace_mark(p, 10 * l + 2 * k + 1 + (k > 0 ? 2 : 0));
            if (k == 0) c.prefetch_gains(L.ffn_norm, p.dim);       // QKV has read its gains
            if (k == 2) c.prefetch_gains(l + 1 < p.n_layers ? p.layers[l + 1].attn_norm : p.out_norm, p.dim);
        }
    }
    unsigned* fin = p.counters;
    if (tid == 0) trace_mark(p, 241);
    unsigned long long b = best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, b, o);
        b = other > b ? other : b;
    }
    if (c.lane == 0) sm.best()[c.warp] = b;
    consumer_sync();
    if (tid == 0) {
        unsigned long long bb = 0ull;
        for (int w = 0; w < kConsumerWarps; w++) bb = sm.best()[w] > bb ? sm.best()[w] : bb;
        atomicMax(p.best, bb);
        __threadfence();
        const unsigned old = atomicAdd(fin, 1u);
        sm.misc()[1] = (old == (unsigned)(G - 1));
    }
    consumer_sync();
    if (sm.misc()[1] && tid == 0) {
        // every CTA has passed its last wait: publish the argmax, re-arm the
        // counter, and make this step's tag the last completed one
        __threadfence();
        *p.token_out = argmax_key_index(atomicExch(p.best, 0ull));
        *p.epoch = c.tag;
        *fin = 0u;
        trace_mark(p, 242);
    }
    return true;
}

template <int DT, bool LC>
__device__ void producer_main(const StepParams& p, Smem& sm) {
    Producer pr(p, sm);
    const Part pt = cta_part(p.ngrp);
    const int fdg = p.dv.m.cols;
    int rg0, rg1, u0, u1;
    share(p.dim, pt.j, pt.n, rg0, rg1);
    share(fdg, pt.j, pt.n, u0, u1);
    u0 += pt.g * fdg;
    u1 += pt.g * fdg;
    for (int l = 0; l < p.n_layers && !pr.dead; l++) {
        const LayerDev& L = p.layers[l];
        int q0, q1;
        cta_rows(L.qkv.rows, q0, q1);
        pr.rows(L.qkv, DT, q0, q1, 256 + 8 * l);
        pr.attention(l, LC);
        pr.view(p.ov, layer_map(p, l, 2), layer_map(p, l, 3), pt.g, rg0, rg1, 256 + 8 * l + 2);
        pr.rows(L.gu, DT, 2 * u0, 2 * u1, 256 + 8 * l + 3);
        pr.view(p.dv, layer_map(p, l, 4), layer_map(p, l, 5), pt.g, rg0, rg1, 256 + 8 * l + 4);
        trace_mark(p, 256 + 8 * l + 5);
    }
    int o0, o1;
    cta_rows(p.out.rows, o0, o1);
    pr.rows(p.out, DT, o0, o1, 448);
    trace_mark(p, 449);
    pr.drain();   // on success every chunk was consumed and the waits return at once
}

template <int DT, bool LC>
__global__ void __launch_bounds__(kBlock, 1) decode_step_kernel(const __grid_constant__ StepParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the ring starts on a 1024-byte boundary (the swizzled KV tiles rely on it)
    Smem sm(reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023), p);
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.ns; i++) {
            mbar_init(&sm.full()[i], 1);
            mbar_init(&sm.empty()[i], kConsumerWarps);
        }
        sm.misc()[0] = 0;
        sm.misc()[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x >= kConsumers) {
        if (threadIdx.x == kConsumers) producer_main<DT, LC>(p, sm);
        __syncwarp();
    } else {
        consumer_main<DT, LC>(p, sm);
    }
    block_join();
}

// ------------------------------------------------------ host-side helpers --
// Streaming plan of one matrix (rows per slot, team width, team count).  Rows
// per chunk are a multiple of the rows all teams take in one pass.  A pair
// matrix (interleaved gate/up rows) is split across CTAs by super-rows, so a
// gate row and its up row stay in one CTA, and is streamed and reduced as
// single rows (pair = 2); the rows are paired when the phase finishes.
bool matrix_plan(DMat& m, int wtype, bool pair) {
    const int lpr = (m.cols + kLaneElems - 1) / kLaneElems;
    int half = 1;
    if (lpr <= 32) {
        while (half < lpr) half *= 2;
    } else {
        half = 32 * ((lpr + 31) / 32);
    }
    const int tw = half;
    int teams, rows_per_pass;
    if (tw <= 32) {
        teams = kConsumerWarps * (32 / tw);
        const int rpp = wtype == LLM_Q8_0 ? RowsPerPass<LLM_Q8_0>::value : 2;
        rows_per_pass = tw >= rpp ? teams * rpp : teams;
    } else {
        if (tw / 32 > kConsumerWarps) return false;
        teams = kConsumerWarps / (tw / 32);
        if (teams > kMaxTeams) teams = kMaxTeams;
        rows_per_pass = (wtype == LLM_Q8_0 ? RowsPerPass<LLM_Q8_0>::value : 2) * teams;
    }
    const int slot_rows = kSlotBytes / slot_row_bytes(wtype, m.cols, m.dstride);
    if (slot_rows < 1) return false;
    m.pair = pair ? 2 : 0;
    m.tw = tw;
    m.teams = teams;
    m.rpc = slot_rows >= rows_per_pass ? (slot_rows / rows_per_pass) * rows_per_pass
                                       : (slot_rows >= teams ? (slot_rows / teams) * teams : slot_rows);
    return true;
}

// Column-group view of a [rows x cols] matrix split into ngrp groups of
// cols/ngrp columns, each CTA taking at most max_rows rows of its group.
// Returns false if the groups do not fit the kernel's limits.
bool gview_plan(GView& v, int wtype, int rows, int cols, int ngrp, int max_rows) {
    if (cols % ngrp) return false;
    const int gc = cols / ngrp;
    const int es = wtype == LLM_Q8_0 ? 1 : (wtype == LLM_F16 ? 2 : 4);
    v = GView{};
    v.m.rows = rows;
    v.m.cols = gc;
    v.m.dstride = 0;
    if (!matrix_plan(v.m, wtype, false)) return false;
    v.U = gc % 32 == 0 ? 32 : 16 / es;
    if (wtype == LLM_Q8_0 && gc % 32) return false;
    if (gc % v.U || cols % v.U || gc / v.U > 256) return false;
    v.rowq = gc * es;
    v.rowd = 0;
    if (wtype == LLM_Q8_0) {
        const int cb = gc / 32;
        int extra = 0;
        for (int g = 0; g < ngrp; g++) extra = std::max(extra, (g * cb) % 8);
        const int sb = (cb + extra + 7) & ~7;
        if (sb > 256) return false;
        v.rowd = sb * 2;
    }
    const int per = v.rowq + v.rowd;
    if (max_rows < 1) max_rows = 1;
    const int chunks = (int)(((long long)max_rows * per + (kSlotBytes - 1024) - 1) / (kSlotBytes - 1024));
    int R = (max_rows + chunks - 1) / chunks;
    if (R > 256) R = 256;
    auto al128 = [](int b) { return (b + 127) & ~127; };
    while (R > 1 && al128(R * v.rowq) + R * v.rowd > kSlotBytes) R--;
    if (al128(R * v.rowq) + R * v.rowd > kSlotBytes) return false;
    v.R = R;
    v.m.rpc = R;
    v.sboff = al128(R * v.rowq);
    v.box_bytes = R * v.rowq + R * v.rowd;
    return true;
}

// Shared-memory geometry of the step kernel for a model.  stage_floats: the
// longest vector a GEMV phase stages (dim, or a group's Wo / Wdown columns);
// rowp_floats / rowp_logits: row partials of multi-warp teams (the logits
// phase keeps them in the residual region).  Returns false if the model does
// not fit the kernel's limits.
bool step_geometry(StepParams& p, int dim, int stage_floats, int n_heads, int n_kv, int hd, int rope_dims,
                   int rowp_floats, int rowp_logits, bool llamacpp, size_t* smem_bytes) {
    const int gq = n_heads / n_kv;
    // KV rows per slot: K and V tiles of P rows fill a slot, at most 256 (a TMA
    // box side), and the unit's scores (2 * gq * P floats) stay within 8 KB
    int P = kSlotBytes / (4 * hd);
    if (P > 256) P = 256;
    if (P > 1024 / gq) P = 1024 / gq;
    P &= ~7;
    if (P < 8) return false;
    const int GD = gq * hd;
    // tensor-core attention for the head sizes it is instantiated for
    // (head_dim 128 would need more registers than the kernel has to spare);
    // llama.cpp rounding takes the two-pass scalar form
    p.attn_mma = !llamacpp && (hd == 32 || hd == 48 || hd == 64) && gq <= 4;
    p.attn_w = p.attn_mma && hd % 64 == 0 ? 64 : hd;
    // q_s, kf, kp/vp; the scalar form adds its score buffers
    const size_t attn_scratch =
        sizeof(float) * (size_t)(GD + 2 * hd) + (p.attn_mma ? 0 : sizeof(float) * (size_t)(2 * gq * P + 4 * gq));
    auto slices = [](int n) { return (size_t)((n + 31) & ~31) * sizeof(float); };
    size_t xs = attn_scratch;
    xs = std::max(xs, slices(std::max(dim, stage_floats)));
    auto al = [](size_t b) { return (b + 127) & ~(size_t)127; };
    const size_t tpart = sizeof(float) * (size_t)std::max(rowp_floats, 1);
    const size_t res = sizeof(float) * (size_t)std::max(dim, rowp_logits);
    const size_t gain_bytes = slices(dim);
    if (rope_dims / 2 > 128 || GD > 2 * kConsumers || GD % 2) return false;
    const size_t fixed = al(xs) + al(tpart) + al(res) + al(2 * 128 * 4) + al(2 * kConsumers * 4) +
                         al(2 * kOwnFloats * 4) + al(gain_bytes) + 2048;   // barriers and flags; the ring's alignment
    long long ns = ((long long)kMaxSmem - (long long)fixed) / kSlotBytes;
    if (ns > 8) ns = 8;
    if (ns < 2) return false;
    size_t off = (size_t)ns * kSlotBytes;
    p.ns = (int)ns;
    p.attn_rows = P;
    p.scratch_floats = (int)(xs / sizeof(float));
    p.off_xs = (int)off; off += al(xs);
    p.off_red = (int)off; off += al(tpart);
    p.off_res = (int)off; off += al(res);
    p.off_rope = (int)off; off += al(2 * 128 * 4);
    p.off_comb = (int)off; off += al(2 * kConsumers * 4);
    p.off_own = (int)off; off += al(2 * kOwnFloats * 4);
    p.off_gain = (int)off; off += al(gain_bytes);
    p.off_bar = (int)off; off += al(2 * ns * 8);
    p.off_misc = (int)off; off += 64 + 8 * (kConsumerWarps + 2) + 8 * kConsumerWarps;
    *smem_bytes = al(off) + 1024;                               // room to align the ring to 1024 bytes
    return *smem_bytes <= (size_t)kMaxSmem;
}

const void* step_kernel_ptr(int wtype, bool llamacpp) {
    if (llamacpp) {
        switch (wtype) {
            case LLM_Q8_0: return (const void*)decode_step_kernel<LLM_Q8_0, true>;
            case LLM_F16: return (const void*)decode_step_kernel<LLM_F16, true>;
            default: return (const void*)decode_step_kernel<LLM_F32, true>;
        }
    }
    switch (wtype) {
        case LLM_Q8_0: return (const void*)decode_step_kernel<LLM_Q8_0, false>;
        case LLM_F16: return (const void*)decode_step_kernel<LLM_F16, false>;
        default: return (const void*)decode_step_kernel<LLM_F32, false>;
    }
}

// ------------------------------------------------------------ test hooks --
__global__ void kv_store_kernel(__half* kc, __half* vc, int pos, int kv_dim, const float* k, const float* v) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < kv_dim; i += gridDim.x * blockDim.x)
        store_kv(kc, vc, pos, kv_dim, 0, i, __float2half_rn(k[i]), __float2half_rn(v[i]));
}

template <int DT>
__global__ void dequant_rows_kernel(DMat m, int row0, int n_rows, float* out) {
    const long long n = (long long)n_rows * m.cols;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x)
        out[e] = weight_at<DT>(m, row0 + (int)(e / m.cols), (int)(e % m.cols));
}

// The decode step's GEMV on a given vector: the same staging (digit records
// for Q8_0), lane registers, ring and gemv_consume as the step, with the
// matrix chosen by `which` (0 QKV, 1 Wo by column groups, 2 gate/up, 3 Wdown
// by column groups, 4 the logits matrix).  x: the product's input vector (F32);
// y: its rows, or for 1 and 3 [ngrp][dim] the column groups' partial
// products.  LC: the staging of llama.cpp rounding (x quantized to Q8_0
// blocks, or rounded to F16).  No grid-wide dependency: every CTA computes
// its own rows.
template <int DT, bool LC>
__global__ void __launch_bounds__(kBlock, 1) gemv_test_kernel(const __grid_constant__ StepParams p, int which,
                                                              int layer, const float* x, float* y) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    Smem sm(reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023), p);
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.ns; i++) {
            mbar_init(&sm.full()[i], 1);
            mbar_init(&sm.empty()[i], kConsumerWarps);
        }
        sm.misc()[0] = 0;
        sm.misc()[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const LayerDev& L = p.layers[layer];
    const Part pt = cta_part(p.ngrp);
    const GView* v = which == 1 ? &p.ov : which == 3 ? &p.dv : nullptr;
    const DMat& m = v ? v->m : which == 0 ? L.qkv : which == 2 ? L.gu : p.out;
    int r0, r1, n;
    const float* xs = x;
    float* ys = y;
    if (v) {
        share(p.dim, pt.j, pt.n, r0, r1);
        n = m.cols;
        xs = x + (size_t)pt.g * n;
        ys = y + (size_t)pt.g * p.dim;
    } else {
        cta_rows(m.rows, r0, r1);
        if (which == 2) { r0 *= 2; r1 *= 2; }   // gate/up: super-rows, streamed as single rows
        n = p.dim;
    }
    if (threadIdx.x >= kConsumers) {
        if (threadIdx.x == kConsumers) {
            Producer pr(p, sm);
            if (v) pr.view(*v, layer_map(p, layer, which == 1 ? 2 : 4), layer_map(p, layer, which == 1 ? 3 : 5), pt.g, r0,
                           r1, -1);
            else pr.rows(m, DT, r0, r1, -1);
            pr.drain();
        }
        __syncwarp();
    } else {
        Consumer c(p, sm);
        float4* xv = reinterpret_cast<float4*>(sm.xs());
        const int ngr = n / 4;
        for (int i0 = c.tid - c.lane; i0 < ngr; i0 += kConsumers) {
            const int i = i0 + c.lane;
            const bool valid = i < ngr;
            stage_group<DT, LC>(xv, i, valid,
                                valid ? reinterpret_cast<const float4*>(xs)[i] : make_float4(0.f, 0.f, 0.f, 0.f));
        }
        const Lanes Ln = lane_layout<DT>(c, m);
        XReg<DT> xr;
        Epi e{};
        e.kind = Epi::kLogits;
        e.logits = ys;
        e.n = v ? p.dim : m.rows;
        e.err = p.err;
        e.scale = lanes_prep<DT, LC>(c, Ln, n, false, 0.f, xr);
        const ChunkGeo ck = v ? view_geo(*v, pt.g) : rows_geo(m, DT);
        gemv_consume<DT, LC>(c, m, ck, r0, r1, Ln, xr, which == 4 ? sm.res() : sm.rowp(), e, -1);
    }
    block_join();
}

cudaError_t launch_gemv_test(cudaStream_t st, int wtype, bool llamacpp, const StepParams& p, int which, int layer,
                             const float* x, float* y, int sms, size_t smem) {
    const void* fn = llamacpp ? (wtype == LLM_Q8_0 ? (const void*)gemv_test_kernel<LLM_Q8_0, true>
                                 : wtype == LLM_F16 ? (const void*)gemv_test_kernel<LLM_F16, true>
                                                    : (const void*)gemv_test_kernel<LLM_F32, true>)
                              : (wtype == LLM_Q8_0 ? (const void*)gemv_test_kernel<LLM_Q8_0, false>
                                 : wtype == LLM_F16 ? (const void*)gemv_test_kernel<LLM_F16, false>
                                                    : (const void*)gemv_test_kernel<LLM_F32, false>);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    StepParams q = p;
    void* args[] = {&q, &which, &layer, &x, &y};
    return cudaLaunchKernel(fn, dim3(sms), dim3(kBlock), args, smem, st);
}

void launch_kv_store(cudaStream_t st, __half* kc, __half* vc, int pos, int kv_dim, const float* k, const float* v) {
    kv_store_kernel<<<(kv_dim + 255) / 256, 256, 0, st>>>(kc, vc, pos, kv_dim, k, v);
}

void launch_dequant_rows(cudaStream_t st, int wtype, const DMat& m, int row0, int n_rows, float* out) {
    const long long n = (long long)n_rows * m.cols;
    const long long nb = (n + 255) / 256;
    const int blocks = (int)(nb < 4096 ? nb : 4096);
    if (wtype == LLM_Q8_0) dequant_rows_kernel<LLM_Q8_0><<<blocks, 256, 0, st>>>(m, row0, n_rows, out);
    else if (wtype == LLM_F16) dequant_rows_kernel<LLM_F16><<<blocks, 256, 0, st>>>(m, row0, n_rows, out);
    else dequant_rows_kernel<LLM_F32><<<blocks, 256, 0, st>>>(m, row0, n_rows, out);
}

}  // namespace llm
