// The batch-1 decode step as one persistent kernel.
//
// One CTA per SM (cooperative launch, so all CTAs are resident).  The step is
// a chain of phases; every phase reads the whole activation vector produced by
// the previous one, so phases are separated by grid-wide counters:
//
//   per layer l:  QKV   rows of [Wq;Wk;Wv] . RMSNorm(x)        -> qkv (+ bias)
//                 ATTN  (kv head, position split) units: RoPE(q), RoPE(k),
//                       K/V row `pos` stored as F16, partial softmax;
//                       the last split of a kv head merges the partials -> attn
//                 O     rows of Wo . attn                       -> x += ...
//                 GU    rows of [Wgate|Wup] . RMSNorm(x)        -> u = silu(g) * up
//                 DOWN  rows of Wdown . u                       -> x += ...
//   LOGITS  rows of Wout . RMSNorm(x) -> logits, argmax (first index of the max)
//
// Steps follow "The Forward Pass in Java", Example 13 (Llama.forward); the
// attention split and merge is the flash-decoding rearrangement of the same
// softmax (max-subtracted partial sums combined with exp(m_s - M) weights).
// Every wait is bounded: on expiry the CTA records kErrTimeout and returns.
#include "llm_internal.cuh"

namespace llm {

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

// ------------------------------------------------------------ grid sync --
__device__ __forceinline__ bool wait_counter(const StepParams& p, const unsigned* c, unsigned target,
                                             volatile int* s_flag) {
    if (threadIdx.x == 0) {
        int ok = 1;
        if (ld_acquire(c) < target) {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire(c) < target) {
                __nanosleep(32);
                if (*(volatile int*)p.err & kErrTimeout) { ok = 0; break; }
                if (global_timer_ns() - t0 > kWaitLimitNs) { atomicOr(p.err, kErrTimeout); ok = 0; break; }
            }
        }
        *s_flag = ok;
    }
    __syncthreads();
    return *s_flag != 0;
}

__device__ __forceinline__ void signal_counter(unsigned* c) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(c, 1u);
    }
}

// ------------------------------------------------------- block reductions --
__device__ double block_sum_double(double v, double* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
        for (int w = 0; w < kWarps; w++) s += red[w];
        red[kWarps] = s;
    }
    __syncthreads();
    double r = red[kWarps];
    __syncthreads();
    return r;
}

// xs <- RMSNorm(src) * g ("The Forward Pass in Java", Example 4): the sum of
// squares in double, scale = (float)(1/sqrt(ss/n + eps)), y = (x*scale)*g.
__device__ void load_normed(float* xs, const float* src, const float* g, int n, float eps, double* red) {
    double ss = 0.0;
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const float v = __ldcg(src + i);
        xs[i] = v;
        ss += (double)v * (double)v;
    }
    const double tot = block_sum_double(ss, red);
    const float scale = (float)(1.0 / sqrt(tot / (double)n + (double)eps));
    for (int i = threadIdx.x; i < n; i += kThreads) xs[i] = __fmul_rn(__fmul_rn(xs[i], scale), __ldg(g + i));
    __syncthreads();
}

__device__ void load_plain(float* xs, const float* src, int n) {
    for (int i = threadIdx.x; i < n; i += kThreads) xs[i] = __ldcg(src + i);
    __syncthreads();
}

// --------------------------------------------------------- weight decode --
// Element i of row r, decoded exactly as the format defines it: Q8_0
// d * qs (an exact float product), F16 widened, F32 as stored.
template <int DT>
__device__ __forceinline__ float weight_at(const DMat& m, int r, int i) {
    if (DT == LLM_Q8_0) {
        const float d = __half2float(m.d[(size_t)r * (m.cols / 32) + i / 32]);
        return __fmul_rn(d, (float)(int8_t)m.q[(size_t)r * m.cols + i]);
    } else if (DT == LLM_F16) {
        return __half2float(reinterpret_cast<const __half*>(m.q)[(size_t)r * m.cols + i]);
    } else {
        return reinterpret_cast<const float*>(m.q)[(size_t)r * m.cols + i];
    }
}

// ------------------------------------------------------------------ GEMV --
// Elements per 16-byte segment.
template <int DT> struct Seg { static constexpr int n = DT == LLM_Q8_0 ? 16 : (DT == LLM_F16 ? 8 : 4); };

// Dot of one 16-byte weight segment with the matching x values (from smem).
template <int DT>
__device__ __forceinline__ float seg_dot(const uint4 w, const float* xs) {
    if (DT == LLM_Q8_0) {
        const float4* xp = reinterpret_cast<const float4*>(xs);
        const uint32_t ws[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const float4 xv = xp[k];
            s0 = fmaf(i8_to_f32(ws[k], 0), xv.x, s0);
            s1 = fmaf(i8_to_f32(ws[k], 1), xv.y, s1);
            s0 = fmaf(i8_to_f32(ws[k], 2), xv.z, s0);
            s1 = fmaf(i8_to_f32(ws[k], 3), xv.w, s1);
        }
        return s0 + s1;
    } else if (DT == LLM_F16) {
        const float4* xp = reinterpret_cast<const float4*>(xs);
        const float4 xa = xp[0], xb = xp[1];
        const __half2* h = reinterpret_cast<const __half2*>(&w);
        const float2 a = __half22float2(h[0]), b = __half22float2(h[1]), c = __half22float2(h[2]),
                     d = __half22float2(h[3]);
        float s0 = a.x * xa.x, s1 = a.y * xa.y;
        s0 = fmaf(b.x, xa.z, s0); s1 = fmaf(b.y, xa.w, s1);
        s0 = fmaf(c.x, xb.x, s0); s1 = fmaf(c.y, xb.y, s1);
        s0 = fmaf(d.x, xb.z, s0); s1 = fmaf(d.y, xb.w, s1);
        return s0 + s1;
    } else {
        const float4 xv = *reinterpret_cast<const float4*>(xs);
        float s0 = __uint_as_float(w.x) * xv.x, s1 = __uint_as_float(w.y) * xv.y;
        s0 = fmaf(__uint_as_float(w.z), xv.z, s0);
        s1 = fmaf(__uint_as_float(w.w), xv.w, s1);
        return s0 + s1;
    }
}

// Lane-partial dots of NR consecutive rows starting at r0 (lane strides over
// 16-byte segments; loads issued four segments ahead per row).
template <int DT, int NR>
__device__ __forceinline__ void rows_dot(const DMat& m, int r0, const float* xs, float acc[NR]) {
    constexpr int E = Seg<DT>::n;
    constexpr int ES = DT == LLM_Q8_0 ? 1 : (DT == LLM_F16 ? 2 : 4);   // bytes per element
    const int lane = threadIdx.x & 31;
    const int nseg = m.cols / E;
    const size_t row_bytes = (size_t)m.cols * ES;
    const uint8_t* rowp[NR];
    const __half* drow[NR];
#pragma unroll
    for (int r = 0; r < NR; r++) {
        acc[r] = 0.f;
        rowp[r] = m.q + (size_t)(r0 + r) * row_bytes;
        drow[r] = DT == LLM_Q8_0 ? m.d + (size_t)(r0 + r) * (m.cols / 32) : nullptr;
    }
    int seg = lane;
    for (; seg + 96 < nseg; seg += 128) {
        uint4 w[NR][4];
        unsigned short dd[NR][4];
#pragma unroll
        for (int r = 0; r < NR; r++)
#pragma unroll
            for (int u = 0; u < 4; u++) {
                w[r][u] = ld_stream(rowp[r] + (size_t)(seg + 32 * u) * 16);
                if (DT == LLM_Q8_0) dd[r][u] = ld_stream_u16(drow[r] + (seg + 32 * u) / 2);
            }
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const float* xp = xs + (seg + 32 * u) * E;
#pragma unroll
            for (int r = 0; r < NR; r++) {
                const float s = seg_dot<DT>(w[r][u], xp);
                if (DT == LLM_Q8_0) acc[r] = fmaf(__half2float(__ushort_as_half(dd[r][u])), s, acc[r]);
                else acc[r] += s;
            }
        }
    }
    for (; seg < nseg; seg += 32) {
        uint4 w[NR];
        unsigned short dd[NR];
#pragma unroll
        for (int r = 0; r < NR; r++) {
            w[r] = ld_stream(rowp[r] + (size_t)seg * 16);
            if (DT == LLM_Q8_0) dd[r] = ld_stream_u16(drow[r] + seg / 2);
        }
#pragma unroll
        for (int r = 0; r < NR; r++) {
            const float s = seg_dot<DT>(w[r], xs + seg * E);
            if (DT == LLM_Q8_0) acc[r] = fmaf(__half2float(__ushort_as_half(dd[r])), s, acc[r]);
            else acc[r] += s;
        }
    }
#pragma unroll
    for (int r = 0; r < NR; r++) acc[r] = warp_sum(acc[r]);
}

// Rows of m split evenly over every warp of the grid; epi.row(r, v) is called
// by lane 0 with the full dot of row r.  pair=true: rows come in (2i, 2i+1)
// pairs and epi.pair(i, v0, v1) is called instead.
template <int DT, bool PAIR, class Epi>
__device__ __forceinline__ void gemv_phase(const DMat& m, const float* xs, Epi& epi) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * kWarps + warp, GW = (long long)gridDim.x * kWarps;
    const int units = PAIR ? m.rows / 2 : m.rows;
    const int u0 = (int)(units * gw / GW), u1 = (int)(units * (gw + 1) / GW);
    if constexpr (PAIR) {
        for (int u = u0; u < u1; u++) {
            float a[2];
            rows_dot<DT, 2>(m, 2 * u, xs, a);
            if (lane == 0) epi.pair(u, a[0], a[1]);
        }
    } else {
        int r = u0;
        for (; r + 1 < u1; r += 2) {
            float a[2];
            rows_dot<DT, 2>(m, r, xs, a);
            if (lane == 0) { epi.row(r, a[0]); epi.row(r + 1, a[1]); }
        }
        if (r < u1) {
            float a[1];
            rows_dot<DT, 1>(m, r, xs, a);
            if (lane == 0) epi.row(r, a[0]);
        }
    }
}

struct EpiStore {                 // out[r] = v (+ bias[r])
    float* out;
    const float* bias;
    __device__ void row(int r, float v) { __stcg(out + r, bias ? v + __ldg(bias + r) : v); }
};
struct EpiResidual {              // x[r] += v
    float* x;
    __device__ void row(int r, float v) { __stcg(x + r, __ldcg(x + r) + v); }
};
struct EpiSwiGLU {                // u[i] = silu(gate) * up ("The Forward Pass in Java", Example 8)
    float* u;
    __device__ void pair(int i, float g, float up) {
        const float e = expf(-g);
        __stcg(u + i, __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, e)), up));
    }
};
struct EpiLogits {                // logits[r] = v, keep this lane's best (value, first index)
    float* logits;
    unsigned long long best;
    __device__ void row(int r, float v) {
        __stcg(logits + r, v);
        const unsigned long long k = argmax_key(v, r);
        best = k > best ? k : best;
    }
};

// ------------------------------------------------------------------ RoPE --
// "The Forward Pass in Java", Example 6 and "What a Llama model computes, and
// why" §2.4: pair i turns by theta_i, where theta starts at pos and is
// multiplied by theta_scale once per pair in float (the same chain as ggml's
// rope cache), then divided by the pair's frequency factor.
__device__ __forceinline__ void rope_pair(float* v, int head_dim, int rope_dims, int neox, int i, int pos,
                                          float theta_scale, const float* freqs) {
    float th = (float)pos;
    for (int j = 0; j < i; j++) th = __fmul_rn(th, theta_scale);
    if (freqs) th = __fdiv_rn(th, __ldg(freqs + i));
    const float c = (float)cos((double)th), s = (float)sin((double)th);
    const int a = neox ? i : 2 * i, b = neox ? i + rope_dims / 2 : 2 * i + 1;
    const float x0 = v[a], x1 = v[b];
    v[a] = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
    v[b] = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
    (void)head_dim;
}

// K/V row `pos` of one kv head, rounded to F16 to nearest even ("The Forward
// Pass in Java", Example 10), at element pos*kv_dim + off + i (Example 7).
__device__ __forceinline__ void store_kv(__half* kc, __half* vc, int pos, int kv_dim, int off, int i, float k,
                                         float v) {
    const size_t e = (size_t)pos * kv_dim + off + i;
    kc[e] = __float2half_rn(k);
    vc[e] = __float2half_rn(v);
}

// ------------------------------------------------------------- attention --
struct AttnSmem {
    float* q;      // [gq][hd] rotated queries of the group
    float* kpos;   // [hd] rotated k of this position (writer split only)
    float* sc;     // [gq][kAttnChunk] scores, then exp weights
    float* mlc;    // [3][gq]: running max, running sum, correction
    __half* ks;    // [kAttnChunk][hd]
    __half* vs;    // [kAttnChunk][hd]
};

__device__ void attention_unit(const StepParams& p, const LayerDev& L, int layer, int g, int s, int S,
                               const AttnSmem& sm, volatile int* s_flag) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hd = p.hd, gq = p.n_heads / p.n_kv, h0 = g * gq, n_pos = p.pos + 1;
    const int chunk = (n_pos + S - 1) / S;
    const int t0 = min(n_pos, s * chunk), t1 = min(n_pos, t0 + chunk);

    // queries of the group, rotated
    for (int i = tid; i < gq * hd; i += kThreads) sm.q[i] = __ldcg(p.qkv + h0 * hd + i);
    __syncthreads();
    for (int i = tid; i < gq * (p.rope_dims / 2); i += kThreads) {
        const int h = i / (p.rope_dims / 2), pr = i % (p.rope_dims / 2);
        rope_pair(sm.q + h * hd, hd, p.rope_dims, p.neox, pr, p.pos, p.theta_scale, p.rope_freqs);
    }
    // the split holding `pos` rotates this token's k and stores K/V row pos
    const bool writer = t0 <= p.pos && p.pos < t1;
    if (writer) {
        for (int i = tid; i < hd; i += kThreads) sm.kpos[i] = __ldcg(p.qkv + p.q_dim + g * hd + i);
        __syncthreads();
        for (int i = tid; i < p.rope_dims / 2; i += kThreads)
            rope_pair(sm.kpos, hd, p.rope_dims, p.neox, i, p.pos, p.theta_scale, p.rope_freqs);
        __syncthreads();
        for (int i = tid; i < hd; i += kThreads)
            store_kv(L.kc, L.vc, p.pos, p.kv_dim, g * hd, i, sm.kpos[i],
                     __ldcg(p.qkv + p.q_dim + p.kv_dim + g * hd + i));
        __threadfence_block();
    }
    if (tid < gq) { sm.mlc[tid] = -INFINITY; sm.mlc[gq + tid] = 0.f; }
    __syncthreads();

    // online softmax over [t0, t1) in chunks staged in shared memory
    constexpr int kAcc = kMaxGroupDim / kThreads;
    float acc[kAcc];
#pragma unroll
    for (int a = 0; a < kAcc; a++) acc[a] = 0.f;
    const int per_row = hd / 8;
    for (int c0 = t0; c0 < t1; c0 += kAttnChunk) {
        const int np = min(kAttnChunk, t1 - c0);
        for (int idx = tid; idx < np * per_row; idx += kThreads) {
            const int row = idx / per_row, w = idx % per_row;
            const size_t e = (size_t)(c0 + row) * p.kv_dim + g * hd + w * 8;
            reinterpret_cast<uint4*>(sm.ks)[row * per_row + w] = __ldcg(reinterpret_cast<const uint4*>(L.kc + e));
            reinterpret_cast<uint4*>(sm.vs)[row * per_row + w] = __ldcg(reinterpret_cast<const uint4*>(L.vc + e));
        }
        __syncthreads();
        for (int idx = tid; idx < gq * np; idx += kThreads) {
            const int h = idx / np, pp = idx % np;
            const float* qh = sm.q + h * hd;
            const __half2* kr = reinterpret_cast<const __half2*>(sm.ks + pp * hd);
            float s0 = 0.f, s1 = 0.f;
            for (int i = 0; i < hd / 2; i++) {
                const float2 kv = __half22float2(kr[i]);
                s0 = fmaf(qh[2 * i], kv.x, s0);
                s1 = fmaf(qh[2 * i + 1], kv.y, s1);
            }
            sm.sc[h * kAttnChunk + pp] = __fdiv_rn(s0 + s1, p.attn_div);
        }
        __syncthreads();
        if (warp < gq) {
            const int h = warp;
            float mloc = -INFINITY;
            for (int pp = lane; pp < np; pp += 32) mloc = fmaxf(mloc, sm.sc[h * kAttnChunk + pp]);
            mloc = warp_max(mloc);
            const float mold = sm.mlc[h], mnew = fmaxf(mold, mloc);
            float sum = 0.f;
            for (int pp = lane; pp < np; pp += 32) {
                const float e = expf(sm.sc[h * kAttnChunk + pp] - mnew);
                sm.sc[h * kAttnChunk + pp] = e;
                sum += e;
            }
            sum = warp_sum(sum);
            if (lane == 0) {
                const float corr = expf(mold - mnew);     // 0 on the first chunk (mold = -inf)
                sm.mlc[h] = mnew;
                sm.mlc[gq + h] = sm.mlc[gq + h] * corr + sum;
                sm.mlc[2 * gq + h] = corr;
            }
        }
        __syncthreads();
#pragma unroll
        for (int a = 0; a < kAcc; a++) {
            const int o = tid + a * kThreads;
            if (o < gq * hd) {
                const int h = o / hd, i = o % hd;
                float v = acc[a] * sm.mlc[2 * gq + h];
                const float* e = sm.sc + h * kAttnChunk;
                for (int pp = 0; pp < np; pp++) v = fmaf(e[pp], __half2float(sm.vs[pp * hd + i]), v);
                acc[a] = v;
            }
        }
        __syncthreads();
    }
    // partial of this split: (m, l, acc) per head
    const int stride = hd + 2;
#pragma unroll
    for (int a = 0; a < kAcc; a++) {
        const int o = tid + a * kThreads;
        if (o < gq * hd) {
            const int h = o / hd, i = o % hd;
            float* part = p.attn_part + ((size_t)(h0 + h) * p.max_splits + s) * stride;
            __stcg(part + 2 + i, acc[a]);
            if (i == 0) { __stcg(part, sm.mlc[h]); __stcg(part + 1, sm.mlc[gq + h]); }
        }
    }
    // the last split to finish merges: M = max m_s, L = sum e^(m_s-M) l_s,
    // out = sum e^(m_s-M) acc_s / L
    unsigned* mc = p.counters + n_phase_counters(p.n_layers) + layer * p.n_kv + g;
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned old = atomicAdd(mc, 1u);
        *s_flag = (old == (unsigned)(S - 1));
    }
    __syncthreads();
    if (*s_flag) {
        __threadfence();
        for (int o = tid; o < gq * hd; o += kThreads) {
            const int h = o / hd, i = o % hd;
            const float* base = p.attn_part + (size_t)(h0 + h) * p.max_splits * stride;
            float M = -INFINITY;
            for (int ss = 0; ss < S; ss++) M = fmaxf(M, __ldcg(base + ss * stride));
            float Lsum = 0.f, v = 0.f;
            for (int ss = 0; ss < S; ss++) {
                const float ms = __ldcg(base + ss * stride);
                const float w = ms == -INFINITY ? 0.f : expf(ms - M);
                Lsum = fmaf(w, __ldcg(base + ss * stride + 1), Lsum);
                v = fmaf(w, __ldcg(base + ss * stride + 2 + i), v);
            }
            __stcg(p.attn + (h0 + h) * hd + i, v / Lsum);
        }
        signal_counter(p.counters + 5 * layer + 1);
    }
    __syncthreads();
}

// ----------------------------------------------------------------- kernel --
template <int DT>
__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(const StepParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ double red[kWarps + 1];
    __shared__ int s_flag;
    __shared__ unsigned long long s_best[kWarps];
    float* xs = reinterpret_cast<float*>(smem_raw);
    const int G = gridDim.x, tid = threadIdx.x;
    volatile int* flag = &s_flag;

    int token = __ldcg(p.token_in);
    if (token < 0 || token >= p.vocab) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, kErrToken);
        token = 0;
    }

    // attention scratch aliases the x buffer (phases never overlap)
    const int gq = p.n_heads / p.n_kv;
    AttnSmem am;
    am.q = xs;
    am.kpos = am.q + gq * p.hd;
    am.sc = am.kpos + p.hd;
    am.mlc = am.sc + gq * kAttnChunk;
    am.ks = reinterpret_cast<__half*>(am.mlc + ((3 * gq + 3) / 4) * 4);
    am.vs = am.ks + kAttnChunk * p.hd;

    for (int l = 0; l < p.n_layers; l++) {
        const LayerDev& L = p.layers[l];
        unsigned* ctr = p.counters + 5 * l;
        // ---- QKV
        if (l == 0) {
            double ss = 0.0;
            for (int i = tid; i < p.dim; i += kThreads) {
                const float v = weight_at<DT>(p.embd, token, i);
                xs[i] = v;
                ss += (double)v * (double)v;
                if (blockIdx.x == 0) __stcg(p.x + i, v);
            }
            const double tot = block_sum_double(ss, red);
            const float scale = (float)(1.0 / sqrt(tot / (double)p.dim + (double)p.eps));
            for (int i = tid; i < p.dim; i += kThreads) xs[i] = __fmul_rn(__fmul_rn(xs[i], scale), __ldg(L.attn_norm + i));
            __syncthreads();
        } else {
            if (!wait_counter(p, ctr - 1, G, flag)) return;
            load_normed(xs, p.x, L.attn_norm, p.dim, p.eps, red);
        }
        { EpiStore e{p.qkv, L.qkv_bias}; gemv_phase<DT, false>(L.qkv, xs, e); }
        signal_counter(ctr + 0);
        // ---- ATTN
        if (!wait_counter(p, ctr + 0, G, flag)) return;
        {
            const int S = p.splits, units = p.n_kv * S;
            for (int unit = blockIdx.x; unit < units; unit += G)
                attention_unit(p, L, l, unit / S, unit % S, S, am, flag);
        }
        // ---- O
        if (!wait_counter(p, ctr + 1, p.n_kv, flag)) return;
        load_plain(xs, p.attn, p.q_dim);
        { EpiResidual e{p.x}; gemv_phase<DT, false>(L.o, xs, e); }
        signal_counter(ctr + 2);
        // ---- GU
        if (!wait_counter(p, ctr + 2, G, flag)) return;
        load_normed(xs, p.x, L.ffn_norm, p.dim, p.eps, red);
        { EpiSwiGLU e{p.u}; gemv_phase<DT, true>(L.gu, xs, e); }
        signal_counter(ctr + 3);
        // ---- DOWN
        if (!wait_counter(p, ctr + 3, G, flag)) return;
        load_plain(xs, p.u, p.ffn);
        { EpiResidual e{p.x}; gemv_phase<DT, false>(L.down, xs, e); }
        signal_counter(ctr + 4);
    }
    // ---- LOGITS + argmax
    unsigned* fin = p.counters + 5 * p.n_layers;
    if (!wait_counter(p, fin - 1, G, flag)) return;
    load_normed(xs, p.x, p.out_norm, p.dim, p.eps, red);
    EpiLogits e{p.logits, 0ull};
    gemv_phase<DT, false>(p.out, xs, e);
    if ((tid & 31) == 0) s_best[tid >> 5] = e.best;
    __syncthreads();
    if (tid == 0) {
        unsigned long long b = 0ull;
        for (int w = 0; w < kWarps; w++) b = s_best[w] > b ? s_best[w] : b;
        atomicMax(p.best, b);
        __threadfence();
        const unsigned old = atomicAdd(fin, 1u);
        s_flag = (old == (unsigned)(G - 1));
    }
    __syncthreads();
    if (s_flag) {
        // every CTA has passed its last wait: publish the argmax, re-arm the counters
        __threadfence();
        if (tid == 0) {
            const unsigned long long b = atomicExch(p.best, 0ull);
            *p.token_out = argmax_key_index(b);
        }
        const int nc = n_phase_counters(p.n_layers) + p.n_layers * p.n_kv;
        for (int i = tid; i < nc; i += kThreads) p.counters[i] = 0u;
    }
}

// Shared memory of the step kernel for a model (bytes).
size_t step_smem_bytes(int dim, int q_dim, int ffn, int n_heads, int n_kv, int hd) {
    const int gq = n_heads / n_kv;
    size_t xbytes = sizeof(float) * (size_t)max(max(dim, q_dim), ffn);
    size_t abytes = sizeof(float) * (size_t)(gq * hd + hd + gq * kAttnChunk + ((3 * gq + 3) / 4) * 4) +
                    2 * sizeof(__half) * (size_t)kAttnChunk * hd;
    size_t b = xbytes > abytes ? xbytes : abytes;
    return (b + 15) & ~(size_t)15;
}

const void* step_kernel_ptr(int wtype) {
    switch (wtype) {
        case LLM_Q8_0: return (const void*)decode_step_kernel<LLM_Q8_0>;
        case LLM_F16: return (const void*)decode_step_kernel<LLM_F16>;
        default: return (const void*)decode_step_kernel<LLM_F32>;
    }
}

// ------------------------------------------------------------ test hooks --
__global__ void kv_store_kernel(__half* kc, __half* vc, int pos, int kv_dim, const float* k, const float* v) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < kv_dim; i += gridDim.x * blockDim.x)
        store_kv(kc, vc, pos, kv_dim, 0, i, k[i], v[i]);
}

template <int DT>
__global__ void dequant_rows_kernel(DMat m, int row0, int n_rows, float* out) {
    const long long n = (long long)n_rows * m.cols;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x)
        out[e] = weight_at<DT>(m, row0 + (int)(e / m.cols), (int)(e % m.cols));
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
