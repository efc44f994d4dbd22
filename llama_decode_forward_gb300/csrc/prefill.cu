// Batched prefill for F16 and Q8_0 weights ("What a Llama model computes, and why",
// §4: the same pass as the decode step, applied to n tokens at once; every
// K/V row is written, token i attends to rows 0..pos0+i, and only the last
// token's logits are produced).
//
// The projections are tensor-core GEMMs on the 5th-generation tensor cores:
// C[M][N] = A[M][K] . W[N][K]^T with A the token rows (F16, rounded to
// nearest even from the F32 activations) and W a weight matrix in the
// library's row layout (F16, K contiguous; Q8_0 tiles are expanded to F16,
// d * qs rounded to nearest even, in shared memory, or read from the
// handle's F16 copy of the matrices made by q8_expand_kernel), F32
// accumulation in tensor memory.  The GEMM kernel is persistent and
// warp-specialised (one CTA per SM; gemm_kernel below): a TMA producer warp,
// an MMA-issuing warp with two TMEM accumulators, four epilogue warps (bias,
// residual add, or SwiGLU over the interleaved gate/up columns, written
// through a shared-memory transpose), and for Q8_0 four or eight warps that
// expand the quants.
//
// Causal attention over the cache runs on mma.sync tensor-core tiles
// (attention_mma_kernel, two query tiles per block); the per-row steps
// (embedding, RMSNorm, the batch's RoPE table, RoPE + KV append, the last
// row's logits and argmax) are plain CUDA kernels.  Every kernel of a batch
// is a programmatic dependent launch (launch_dep, griddep_entry).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <type_traits>
#include <string>
#include <vector>

#include "llm_internal.cuh"

namespace llm {

namespace {

constexpr int kGBM = 128, kGBK = 64;
constexpr int kGABytes = kGBM * kGBK * 2;
// GEMM tile widths (multiples of 16, the MMA's N step), measured on a
// 512-token batch of the 1B shape: Q/K/V (3072 rows: 96 tiles of 128; 96-wide
// tiles were 7 % faster with F16 weights but slower with Q8_0, whose
// expansion then has half the converter warps), the dim-wide outputs O and
// down (2048: 128 tiles of 64), gate/up (16384: 256 tiles of 256; 296 tiles
// of 224 were slower)
constexpr int kBnQkv = 128, kBnNarrow = 64, kBnWide = 256;
constexpr long long kSpinLimit = 200000000ll;   // mbarrier polls before a wait gives up

// Programmatic dependent launch.  Every kernel of the batched prefill is
// launched with programmatic stream serialization (launch_dep) and lets the
// next kernel be scheduled as soon as all its own CTAs are running
// (griddep_launch); each waits for the whole previous kernel to complete, its
// memory visible (griddep_wait), before it touches activations.  So a
// kernel's launch and setup overlap the tail of the one before, and nothing
// else changes.  (Without the launch attribute both are no-ops.)
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_entry() {
    griddep_launch();
    griddep_wait();
}

// A launch with programmatic stream serialization (see griddep_entry).
template <class... KArgs, class... Args>
cudaError_t launch_dep(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ bool wait_parity(uint64_t* bar, uint32_t par, int* err) {
    for (long long i = 0; i < kSpinLimit; i++)
        if (mbar_test_wait(bar, par)) return true;
    atomicOr(err, kErrTimeout);
    return false;
}

// The same wait with the threads suspended between probes (about 1 us at
// most per probe): for warps that wait through a whole main loop, whose
// polling would otherwise take shared-memory bandwidth from the tensor cores.
constexpr long long kSleepLimit = 4000000ll;    // suspended probes before a wait gives up (a few seconds)
__device__ __forceinline__ bool sleep_parity(uint64_t* bar, uint32_t par, int* err) {
    for (long long i = 0; i < kSleepLimit; i++) {
        if (mbar_sleep_wait(bar, par)) return true;
        if ((i & 63) == 63 && (*(volatile int*)err & kErrTimeout)) return false;   // another wait gave up
    }
    atomicOr(err, kErrTimeout);
    return false;
}

// Shared-memory matrix descriptor of a K-major tile of rows x 64 F16 values
// stored with the 128-byte swizzle (8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t umma_desc_sw128(const void* p) {
    const uint64_t addr = smem_addr(p);
    uint64_t d = (addr >> 4) & 0x3FFFull;       // start address
    d |= (uint64_t)1 << 16;                      // leading-dimension offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;            // stride-dimension offset: 8 rows x 128 bytes
    d |= (uint64_t)1 << 46;                      // descriptor version
    d |= (uint64_t)2 << 61;                      // 128-byte swizzle
    return d;
}

enum { kEpiBias = 0, kEpiResidual = 1, kEpiSwiGLU = 2 };

struct GemmOut {
    float* out;          // kEpiBias: [M][N] f32
    const float* bias;   // kEpiBias: [N] or nullptr
    float* resid;        // kEpiResidual: [M][N] f32, += acc
    __half* hout;        // kEpiSwiGLU: [M][N/2] f16, silu(acc[2i]) * acc[2i+1]
};

// Q8_0 weights of a GEMM: the FP16 scales of the library layout (row r's
// block b at d[r * dstride + b]; d 16-byte aligned, dstride the block count
// rounded up to a multiple of 8); the int8 quants come through a tensor map.
struct GemmScales {
    const __half* d;
    int dstride;
};

// Shared-memory plan of the GEMM: a ring of kStages stages (A tile, W tile
// as F16, and for Q8_0 weights the W tile's int8 quants), then the
// epilogue's transpose buffers and the barriers.
//
// F16 weights: a stage is the A tile and the F16 W tile.  Q8_0 weights: a
// stage is the A tile and the W tile's int8 quants; the converters expand the
// quants into one of kWBufs F16 W buffers outside the ring (so the ring keeps
// more stages, and the expansions run ahead of the MMAs).
template <int BN, bool Q8>
struct GemmPlan {
    static constexpr int kBBytes = BN * kGBK * 2;                 // one F16 W tile
    static constexpr int kQBytes = Q8 ? BN * kGBK : 0;
    static constexpr int kStageBytes = kGABytes + (Q8 ? kQBytes : kBBytes);
    static constexpr int kEpiWarps = 4;
    // Q8_0 converter warps: 8, or 4 when the tile's BN x 4 work items do not
    // split evenly over 256 threads
    static constexpr int kConvWarps = !Q8 ? 0 : (BN * 4) % 256 == 0 ? 8 : 4;
    static constexpr int kWBufs = 2;                               // F16 W buffers (Q8_0)
    static constexpr int kWBufBytes = Q8 ? kWBufs * kBBytes : 0;
    static constexpr int kStages =
        (200 * 1024 - kWBufBytes) / kStageBytes > 8 ? 8 : (200 * 1024 - kWBufBytes) / kStageBytes;
    // TMEM columns of the two accumulators (a power of two of at least 32)
    static constexpr int kTmemCols = 2 * BN <= 32 ? 32 : 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128
                                     : 2 * BN <= 256 ? 256 : 512;
    static constexpr int kThreads = 32 * (2 + kEpiWarps + kConvWarps);
    static constexpr int kTransBytes = kEpiWarps * 32 * 33 * 4;
    static constexpr int kBarBytes = 8 * (2 * kStages + 2 * kWBufs + 4 + 1) + 16;
    static constexpr int kSmem = kStages * kStageBytes + kWBufBytes + kTransBytes + kBarBytes + 1024;
};

// One F16 value of the W tile in the 128-byte-swizzled K-major layout the
// MMA descriptors describe: row r's 64 values fill 128 bytes at r * 128, its
// 16-byte chunk c at chunk position c ^ (r & 7).
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t tile, int r, int c) {
    return tile + (uint32_t)r * 128u + (uint32_t)((c ^ (r & 7)) * 16);
}

// Byte offset of 16-byte chunk c (0..3) of row r in a tile of 64-byte rows
// loaded with the 64-byte TMA swizzle (address bits 4-5 XOR bits 7-8): eight
// consecutive rows' chunk c then fall in eight different bank groups.
__device__ __forceinline__ int sw64_chunk(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }

// Four int8 quants (one word) times the scale pair d2, as two F16 pairs: the
// quant q becomes the F16 value 1152 + q exactly (bytes 0x64, q ^ 0x80: 1024
// + (q + 128)), 1152 is subtracted exactly, and the product d * q is rounded
// once to nearest even by the F16 multiply.
__device__ __forceinline__ void q4_to_f16(uint32_t w, __half2 d2, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = w ^ 0x80808080u;
    const __half2 off = __half2half2(__ushort_as_half((unsigned short)0x6480));   // 1152
    const uint32_t ua = __byte_perm(x, 0x64646464u, 0x4140u), ub = __byte_perm(x, 0x64646464u, 0x4342u);
    __half2 a = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&ua), off), d2);
    __half2 b = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&ub), off), d2);
    lo = *reinterpret_cast<const uint32_t*>(&a);
    hi = *reinterpret_cast<const uint32_t*>(&b);
}

// C[M][N] = A[M][K] . W[N][K]^T, persistent and warp-specialised, one CTA per
// SM:
//   warp 0     TMA producer (one lane): per k-step the 128 x 64 A tile and
//              the BN x 64 W tile (F16; for Q8_0 weights its int8 quants)
//              into the ring stage;
//   warp 1     allocates 2 * BN TMEM columns (two accumulators) and issues
//              tcgen05.mma (M 128, N BN, K 16) from one lane, committing each
//              stage back to the producer and each finished tile to the
//              epilogue;
//   warps 2-5  epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 of the
//              finished accumulator (tcgen05.ld) while the next tile's MMAs
//              run in the other one, transposes each 32 x 32 block through
//              shared memory and writes rows with the lanes along the columns;
//   warps 6-9  (Q8_0) expand each stage's quants to F16 (d * q rounded to
//              nearest even, as an F16 matrix of the weights would hold)
//              into the stage's W tile.
// Tile t (t = blockIdx.x, + gridDim.x, ...) is row block t % Mt of column
// block t / Mt, so CTAs working at the same time share W tiles through L2.
// Every wait is bounded (kErrTimeout, then the role stops).
template <int BN, int EPI, bool Q8>
__global__ void __launch_bounds__(GemmPlan<BN, Q8>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb, GemmScales ws,
                GemmOut o, int M, int N, int K, int* err) {
    using G = GemmPlan<BN, Q8>;
    constexpr int S = G::kStages;
    griddep_launch();
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
    constexpr int WB = G::kWBufs;
    uint8_t* wbuf = sm + S * G::kStageBytes;                       // Q8_0: [WB] F16 W tiles
    float* trans = reinterpret_cast<float*>(wbuf + G::kWBufBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(wbuf + G::kWBufBytes + G::kTransBytes);
    uint64_t* empty = full + S;
    uint64_t* wfull = empty + S;         // [WB] Q8_0: W buffer b holds an expanded tile
    uint64_t* wempty = wfull + WB;       // [WB] Q8_0: the MMAs reading W buffer b are done
    uint64_t* accf = wempty + WB;        // [2] accumulator b holds a finished tile
    uint64_t* acce = accf + 2;           // [2] accumulator b has been read
    uint64_t* fin = acce + 2;            // every MMA issued has completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Mt = (M + kGBM - 1) / kGBM, Nt = (N + BN - 1) / BN, nk = K / kGBK;
    const int t_first = (int)blockIdx.x, t_step = (int)gridDim.x, t_count = Mt * Nt;
    auto tile_m0 = [&](int t) { return (t % Mt) * kGBM; };
    auto tile_n0 = [&](int t) { return (t / Mt) * BN; };
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < WB; b++) {
            mbar_init(&wfull[b], G::kConvWarps > 0 ? G::kConvWarps : 1);
            mbar_init(&wempty[b], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], G::kEpiWarps);
        }
        mbar_init(fin, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(G::kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = *tmem_slot;
    griddep_wait();                      // the barriers and TMEM were set up while the previous kernel finished

    if (warp == 0) {
        // ---- producer
        if (lane == 0) {
            long long it = 0;
            bool ok = true;
            for (int t = t_first; t < t_count && ok; t += t_step) {
                const int m0 = tile_m0(t), n0 = tile_n0(t);
                for (int kt = 0; kt < nk && ok; kt++, it++) {
                    const int s = (int)(it % S);
                    if (!(ok = wait_parity(&empty[s], (uint32_t)(((it / S) & 1) ^ 1), err))) break;
                    uint8_t* st = sm + s * G::kStageBytes;
                    mbar_arrive_expect_tx(&full[s], (uint32_t)(kGABytes + (Q8 ? G::kQBytes : G::kBBytes)));
                    tma_2d_g2s(st, &ma, kt * kGBK, m0, &full[s]);
                    tma_2d_g2s(st + kGABytes, &mb, kt * kGBK, n0, &full[s]);   // the W tile (F16 or quants)
                }
            }
            // the last copies have landed before the CTA can exit (at once when
            // the MMAs consumed them)
            for (long long k = it - 1; k >= 0 && k >= it - S; k--)
                wait_parity(&full[(int)(k % S)], (uint32_t)((k / S) & 1), err);
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            // F32 accumulator, F16 A and B, both K-major, N = BN, M = 128
            const uint32_t idesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kGBM >> 4) << 24);
            long long it = 0;
            bool ok = true;
            int j = 0;
            for (int t = t_first; t < t_count && ok; t += t_step, j++) {
                const int b = j & 1;
                if (!(ok = wait_parity(&acce[b], (uint32_t)(((j >> 1) & 1) ^ 1), err))) break;
                asm volatile("tcgen05.fence::after_thread_sync;");
                const uint32_t dacc = tmem + (uint32_t)(b * BN);
                for (int kt = 0; kt < nk; kt++, it++) {
                    const int s = (int)(it % S);
                    const uint32_t par = (uint32_t)((it / S) & 1);
                    const int wb = (int)(it % WB);
                    if (!(ok = wait_parity(&full[s], par, err))) break;
                    if (Q8 && !(ok = wait_parity(&wfull[wb], (uint32_t)((it / WB) & 1), err))) break;
                    asm volatile("tcgen05.fence::after_thread_sync;");
                    uint8_t* st = sm + s * G::kStageBytes;
                    const uint64_t da = umma_desc_sw128(st),
                                   db = umma_desc_sw128(Q8 ? wbuf + wb * G::kBBytes : st + kGABytes);
#pragma unroll
                    for (int kk = 0; kk < kGBK / 16; kk++) {
                        const uint32_t accumulate = (kt > 0 || kk > 0) ? 1u : 0u;
                        asm volatile(
                            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dacc),
                            "l"(da + 2 * kk), "l"(db + 2 * kk), "r"(idesc), "r"(accumulate));
                    }
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     smem_addr(&empty[s]))
                                 : "memory");
                    if (Q8)
                        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                         smem_addr(&wempty[wb]))
                                     : "memory");
                }
                if (!ok) break;
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 smem_addr(&accf[b]))
                             : "memory");
            }
            // every MMA issued has completed before the accumulators are freed
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_addr(fin))
                         : "memory");
            wait_parity(fin, 0, err);
        }
    } else if (warp < 2 + G::kEpiWarps) {
        // ---- epilogue
        const int q = warp & 3;                                   // TMEM lanes 32q .. 32q+31
        float* tb = trans + (warp - 2) * 32 * 33;
        int j = 0;
        for (int t = t_first; t < t_count; t += t_step, j++) {
            const int b = j & 1;
            const int m0 = tile_m0(t), n0 = tile_n0(t);
            if (!sleep_parity(&accf[b], (uint32_t)((j >> 1) & 1), err)) break;
            asm volatile("tcgen05.fence::after_thread_sync;");
            const int rbase = m0 + q * 32;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + c0);
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                    "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                    : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                      "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                      "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]),
                      "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]),
                      "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                    : "r"(taddr));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                // row `lane` of this 32 x 32 block, transposed through shared memory
                if constexpr (EPI == kEpiSwiGLU) {
                    // columns 2i (gate) and 2i+1 (up) of the interleaved matrix
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        const float g = __uint_as_float(v[2 * i]), up = __uint_as_float(v[2 * i + 1]);
                        const float e = expf(-g);
                        tb[lane * 33 + i] = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, e)), up);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; i++) tb[lane * 33 + i] = __uint_as_float(v[i]);
                }
                __syncwarp();
                if constexpr (EPI == kEpiSwiGLU) {
                    // two rows of 16 F16 outputs per pass
                    const int oc = (n0 + c0) / 2 + (lane & 15);
#pragma unroll 4
                    for (int r2 = 0; r2 < 32; r2 += 2) {
                        const int r = r2 + (lane >> 4), row = rbase + r;
                        if (row < M && 2 * oc + 1 < N)
                            o.hout[(size_t)row * (N / 2) + oc] = __float2half_rn(tb[r * 33 + (lane & 15)]);
                    }
                } else if constexpr (EPI == kEpiBias) {
                    const int col = n0 + c0 + lane;
                    const float bias = o.bias && col < N ? o.bias[col] : 0.f;
#pragma unroll 4
                    for (int r = 0; r < 32; r++) {
                        const int row = rbase + r;
                        if (row < M && col < N) o.out[(size_t)row * N + col] = tb[r * 33 + lane] + bias;
                    }
                } else {
                    // 16 residual values are loaded before any is stored (one
                    // memory latency per 16 rows, not one per row)
                    const int col = n0 + c0 + lane;
#pragma unroll 1
                    for (int h = 0; h < 32; h += 16) {
                        float old[16];
#pragma unroll
                        for (int r = 0; r < 16; r++) {
                            const int row = rbase + h + r;
                            old[r] = row < M && col < N ? __ldcg(o.resid + (size_t)row * N + col) : 0.f;
                        }
#pragma unroll
                        for (int r = 0; r < 16; r++) {
                            const int row = rbase + h + r;
                            if (row < M && col < N) o.resid[(size_t)row * N + col] = old[r] + tb[(h + r) * 33 + lane];
                        }
                    }
                }
                __syncwarp();
            }
            asm volatile("tcgen05.fence::before_thread_sync;");
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);
        }
    } else if constexpr (Q8) {
        // ---- Q8_0 expansion: the W tile's BN rows x 4 pairs of 16-byte
        // output chunks are items i = c + kCT k of the kCT converter threads
        // (row i % BN, pair i / BN): 16 quants in, 16 F16 values out.  Each
        // item's row has its two block scales of a k-step in one 4-byte
        // word; the words of four k-steps are one 16-byte load (a row's
        // scales start 16-byte aligned and are padded to a multiple of 8
        // blocks), issued four k-steps before the first of them is used.
        constexpr int kCT = 32 * G::kConvWarps;
        const int c = threadIdx.x - 32 * (2 + G::kEpiWarps);
        constexpr int kItems = BN * 4 / kCT;
        // one scale word per distinct row: all items of a thread share row
        // c % BN when kCT is a multiple of BN, else each item has its own
        constexpr bool kSameRow = kCT % BN == 0;
        constexpr int kRows = kSameRow ? 1 : kItems;
        static_assert(kItems >= 1 && (BN * 4) % kCT == 0, "converter items");
        long long it = 0;
        bool ok = true;
        for (int t = t_first; t < t_count && ok; t += t_step) {
            const int n0 = tile_n0(t);
            const uint32_t* drow[kRows];
#pragma unroll
            for (int j = 0; j < kRows; j++) {
                const int wrow = n0 + (c + kCT * j) % BN;           // item j's row
                drow[j] = wrow < N ? reinterpret_cast<const uint32_t*>(ws.d + (size_t)wrow * ws.dstride) : nullptr;
            }
            uint4 dq[kRows], dqn[kRows];
            const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int j = 0; j < kRows; j++) {
                dqn[j] = drow[j] ? __ldg(reinterpret_cast<const uint4*>(drow[j])) : zero4;
                dq[j] = zero4;
            }
            for (int kt = 0; kt < nk; kt++, it++) {
                if ((kt & 3) == 0) {
#pragma unroll
                    for (int j = 0; j < kRows; j++) {
                        dq[j] = dqn[j];
                        dqn[j] = drow[j] && kt + 4 < nk ? __ldg(reinterpret_cast<const uint4*>(drow[j] + kt + 4)) : zero4;
                    }
                }
                uint32_t dcur[kRows];
#pragma unroll
                for (int j = 0; j < kRows; j++) {
                    const uint4 v = dq[j];
                    dcur[j] = (kt & 2) ? ((kt & 1) ? v.w : v.z) : ((kt & 1) ? v.y : v.x);
                }
                const int s = (int)(it % S), wb = (int)(it % WB);
                if (!(ok = sleep_parity(&full[s], (uint32_t)((it / S) & 1), err))) break;
                if (!(ok = sleep_parity(&wempty[wb], (uint32_t)(((it / WB) & 1) ^ 1), err))) break;
                uint8_t* st = sm + s * G::kStageBytes;
                const uint32_t btile = smem_addr(wbuf + wb * G::kBBytes);
                const uint8_t* qtile = st + kGABytes;
#pragma unroll
                for (int k = 0; k < kItems; k++) {
                    const int i = c + kCT * k, r = i % BN, pair = i / BN;
                    const uint32_t dw = dcur[kSameRow ? 0 : k];
                    const __half d = __ushort_as_half((unsigned short)(pair < 2 ? dw & 0xFFFFu : dw >> 16));
                    const __half2 d2 = __half2half2(d);
                    const uint4 qv = *reinterpret_cast<const uint4*>(qtile + sw64_chunk(r, pair));
                    uint32_t h[8];
                    q4_to_f16(qv.x, d2, h[0], h[1]);
                    q4_to_f16(qv.y, d2, h[2], h[3]);
                    q4_to_f16(qv.z, d2, h[4], h[5]);
                    q4_to_f16(qv.w, d2, h[6], h[7]);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sw128_chunk(btile, r, 2 * pair)),
                                 "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]) : "memory");
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sw128_chunk(btile, r, 2 * pair + 1)),
                                 "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7]) : "memory");
                }
                fence_proxy_async_smem();                               // the MMA reads the tile
                __syncwarp();
                if (lane == 0) mbar_arrive(&wfull[wb]);
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(G::kTmemCols));
}

// Embedding rows of the batch: F16 widened, or Q8_0 decoded as d * qs (both
// exact in F32; Q8_0 quants are stored as int8).
__global__ void embed_rows_kernel(const int* tok, int n, DMat embd, int wtype, int dim, float* X) {
    griddep_entry();
    const int i = blockIdx.x;
    if (i >= n) return;
    const size_t r = (size_t)tok[i];
    for (int d = threadIdx.x; d < dim; d += blockDim.x) {
        float v;
        if (wtype == LLM_Q8_0)
            v = __fmul_rn(__half2float(embd.d[r * embd.dstride + d / 32]), (float)(int)(int8_t)embd.q[r * embd.cols + d]);
        else
            v = __half2float(reinterpret_cast<const __half*>(embd.q)[r * embd.cols + d]);
        X[(size_t)i * dim + d] = v;
    }
}

// A Q8_0 matrix (library layout) expanded to F16 for the tensor-core GEMMs:
// RMSNorm of every row ("The Forward Pass in Java", Example 4: y = (x*scale)*g,
// scale = 1/sqrt(mean(x^2) + eps)); the GEMM operand is y rounded to F16.
// One warp per row, 8 values per 16-byte step (dim % 8 == 0).
__global__ void rmsnorm_rows_f16_kernel(const float* X, int n, int dim, const float* g, float eps, __half* Y) {
    griddep_entry();
    const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (i >= n) return;
    const float4* x4 = reinterpret_cast<const float4*>(X + (size_t)i * dim);
    const float4* g4 = reinterpret_cast<const float4*>(g);
    const int n8 = dim / 8;
    float ss = 0.f;
    // unrolled so that a lane's loads are in flight together (one memory
    // latency per eight groups, not one per group)
#pragma unroll 8
    for (int k = lane; k < n8; k += 32) {
        const float4 a = x4[2 * k], b = x4[2 * k + 1];
        ss += (a.x * a.x + a.y * a.y) + (a.z * a.z + a.w * a.w) + ((b.x * b.x + b.y * b.y) + (b.z * b.z + b.w * b.w));
    }
    ss = warp_sum(ss);
    const float scale = 1.0f / sqrtf(ss / (float)dim + eps);
    uint4* y4 = reinterpret_cast<uint4*>(Y + (size_t)i * dim);
#pragma unroll 8
    for (int k = lane; k < n8; k += 32) {
        const float4 a = x4[2 * k], b = x4[2 * k + 1], ga = g4[2 * k], gb = g4[2 * k + 1];
        auto y = [&](float x, float gg) { return __float2half_rn(__fmul_rn(__fmul_rn(x, scale), gg)); };
        const __half2 h0 = __halves2half2(y(a.x, ga.x), y(a.y, ga.y)), h1 = __halves2half2(y(a.z, ga.z), y(a.w, ga.w));
        const __half2 h2 = __halves2half2(y(b.x, gb.x), y(b.y, gb.y)), h3 = __halves2half2(y(b.z, gb.z), y(b.w, gb.w));
        y4[k] = make_uint4(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1),
                           *reinterpret_cast<const uint32_t*>(&h2), *reinterpret_cast<const uint32_t*>(&h3));
    }
}

// cos and sin of every (row, pair) of the batch, tab[(i * half + j) * 2 + {0,
// 1}]: the decode step's float angle chain ("The Forward Pass in Java",
// Example 6: theta starts at the position and is multiplied by theta_scale
// once per pair; frequency factors per "What a Llama model computes, and
// why" §2.4), cos/sin taken in double.  The angles depend only on the
// position, so one table serves every layer of the batch.
__global__ void rope_table_kernel(float* tab, int n, int pos0, int half, float theta_scale, const float* freqs) {
    griddep_entry();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= n * half) return;
    const int i = e / half, j = e % half;
    float th = (float)(pos0 + i);
    for (int k = 0; k < j; k++) th = __fmul_rn(th, theta_scale);
    if (freqs) th = __fdiv_rn(th, freqs[j]);
    double sv, cv;
    sincos((double)th, &sv, &cv);
    tab[2 * e] = (float)cv;
    tab[2 * e + 1] = (float)sv;
}

// RoPE of q and k of row i at position pos0+i with the batch's angle table,
// then the F16 K and V rows of that position ("The Forward Pass in Java",
// Examples 7 and 10).
__global__ void rope_kv_rows_kernel(float* QKV, int n, int pos0, int n_heads, int n_kv, int hd, int rope_dims, int neox,
                                    const float* tab, __half* kc, __half* vc) {
    griddep_entry();
    const int i = blockIdx.x;
    if (i >= n) return;
    const int pos = pos0 + i;
    const int q_dim = n_heads * hd, kv_dim = n_kv * hd, half = rope_dims / 2;
    float* row = QKV + (size_t)i * (q_dim + 2 * kv_dim);
    const float2* cs = reinterpret_cast<const float2*>(tab) + (size_t)i * half;
#pragma unroll 4
    for (int t = threadIdx.x; t < (n_heads + n_kv) * half; t += blockDim.x) {
        const int head = t / half, j = t % half;
        float* v = head < n_heads ? row + head * hd : row + q_dim + (head - n_heads) * hd;
        const int a = neox ? j : 2 * j, b = neox ? j + half : 2 * j + 1;
        const float2 r = cs[j];
        const float x0 = v[a], x1 = v[b];
        v[a] = __fsub_rn(__fmul_rn(x0, r.x), __fmul_rn(x1, r.y));
        v[b] = __fadd_rn(__fmul_rn(x0, r.y), __fmul_rn(x1, r.x));
    }
    __syncthreads();
#pragma unroll 4
    for (int e = threadIdx.x; e < kv_dim; e += blockDim.x) {
        kc[(size_t)pos * kv_dim + e] = __float2half_rn(row[q_dim + e]);
        vc[(size_t)pos * kv_dim + e] = __float2half_rn(row[q_dim + kv_dim + e]);
    }
}

// Attention of row i (query position pos0+i) for the query heads of kv head g
// over cache rows 0..pos0+i ("The Forward Pass in Java", Example 7), in tiles
// of 128 positions with a running max and sum per head; output rounded to F16
// for the O projection.  Each tile's K and V rows are staged in shared memory
// with 16-byte loads; a thread's score loop starts at a column that rotates
// with its position so that the K reads fall in different banks.
constexpr int kAttnTile = 128;
__global__ void __launch_bounds__(128) attention_rows_kernel(const float* QKV, int n, int pos0, int n_heads, int n_kv,
                                                             int hd, float attn_div, const __half* kc,
                                                             const __half* vc, __half* A) {
    griddep_entry();
    const int i = blockIdx.x, g = blockIdx.y;
    if (i >= n) return;
    const int gq = n_heads / n_kv, q_dim = n_heads * hd, kv_dim = n_kv * hd, GD = gq * hd;
    const int n_pos = pos0 + i + 1;
    extern __shared__ __align__(16) float asm_[];
    __half* ks = reinterpret_cast<__half*>(asm_);      // [tile][hd]
    __half* vs = ks + kAttnTile * hd;                  // [tile][hd]
    float* q = reinterpret_cast<float*>(vs + kAttnTile * hd);   // [gq][hd]
    float* sc = q + GD;                                // [gq][tile]
    float* ml = sc + gq * kAttnTile;                   // [3][gq]: m, l, corr
    const float* qrow = QKV + (size_t)i * (q_dim + 2 * kv_dim) + g * gq * hd;
    for (int e = threadIdx.x; e < GD; e += blockDim.x) q[e] = qrow[e];
    if (threadIdx.x < gq) { ml[threadIdx.x] = -INFINITY; ml[gq + threadIdx.x] = 0.f; }
    float acc[8];                                      // GD <= 960 -> at most 8 elements per thread
#pragma unroll
    for (int k = 0; k < 8; k++) acc[k] = 0.f;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w16 = hd / 8;                            // 16-byte words per row
    for (int t0 = 0; t0 < n_pos; t0 += kAttnTile) {
        const int nt = min(kAttnTile, n_pos - t0);
        __syncthreads();                               // previous tile fully used
        for (int e = threadIdx.x; e < nt * w16; e += blockDim.x) {
            const int t = e / w16, w = e % w16;
            const size_t src = (size_t)(t0 + t) * kv_dim + g * hd + w * 8;
            reinterpret_cast<uint4*>(ks)[e] = *reinterpret_cast<const uint4*>(kc + src);
            reinterpret_cast<uint4*>(vs)[e] = *reinterpret_cast<const uint4*>(vc + src);
        }
        __syncthreads();
        if ((int)threadIdx.x < nt) {
            const int t = threadIdx.x, nh2 = hd / 2;
            const __half2* k2 = reinterpret_cast<const __half2*>(ks + t * hd);
            for (int h = 0; h < gq; h++) {
                const float2* q2 = reinterpret_cast<const float2*>(q + h * hd);
                float2 a = make_float2(0.f, 0.f);
                int j = t % nh2;
                for (int k = 0; k < nh2; k++) {
                    a = __ffma2_rn(__half22float2(k2[j]), q2[j], a);
                    j = j + 1 == nh2 ? 0 : j + 1;
                }
                sc[h * kAttnTile + t] = __fdiv_rn(a.x + a.y, attn_div);
            }
        }
        __syncthreads();
        for (int h = warp; h < gq; h += (int)(blockDim.x >> 5)) {
            float mloc = -INFINITY;
            for (int t = lane; t < nt; t += 32) mloc = fmaxf(mloc, sc[h * kAttnTile + t]);
            mloc = warp_max(mloc);
            const float mold = ml[h], mnew = fmaxf(mold, mloc);
            float sum = 0.f;
            for (int t = lane; t < nt; t += 32) {
                const float e = expf(sc[h * kAttnTile + t] - mnew);
                sc[h * kAttnTile + t] = e;
                sum += e;
            }
            sum = warp_sum(sum);
            if (lane == 0) {
                const float corr = expf(mold - mnew);
                ml[h] = mnew;
                ml[gq + h] = ml[gq + h] * corr + sum;
                ml[2 * gq + h] = corr;
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const int e = threadIdx.x + k * 128;
            if (e < GD) {
                const int h = e / hd, d = e % hd;
                float a = acc[k] * ml[2 * gq + h];
                const float* p = sc + h * kAttnTile;
                for (int t = 0; t < nt; t++) a = fmaf(p[t], __half2float(vs[t * hd + d]), a);
                acc[k] = a;
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const int e = threadIdx.x + k * 128;
        if (e < GD) A[(size_t)i * q_dim + g * gq * hd + e] = __float2half_rn(acc[k] / ml[gq + e / hd]);
    }
}

// The last row: RMSNorm in F32 (as the decode step), logits of every vocabulary
// row (F16 output matrix), argmax key of each warp's rows.
__global__ void final_norm_kernel(const float* x, int dim, const float* g, float eps, float* y) {
    griddep_entry();
    float ss = 0.f;
    for (int d = threadIdx.x; d < dim; d += blockDim.x) ss += x[d] * x[d];
    __shared__ float red[32];
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) tot += red[w];
    const float scale = 1.0f / sqrtf(tot / (float)dim + eps);
    for (int d = threadIdx.x; d < dim; d += blockDim.x) y[d] = __fmul_rn(__fmul_rn(x[d], scale), g[d]);
}

__global__ void logits_kernel(DMat out, int wtype, const float* y, int dim, int vocab, float* logits,
                              unsigned long long* best) {
    griddep_entry();
    extern __shared__ float ys[];
    // Q8_0: y[e] for e = 512 it + 16 l + 4 k + c sits at float4 (4 it + k) * 32 + l,
    // component c, so the 32 lanes' float4 reads of one k are 512 contiguous
    // bytes (the plain layout put lanes 16 floats apart: 16-way bank
    // conflicts on every read); F16: the plain layout
    for (int e = threadIdx.x; e < dim; e += blockDim.x)
        ys[wtype == LLM_Q8_0 ? (((e >> 9) * 4 + ((e >> 2) & 3)) * 32 + ((e >> 4) & 31)) * 4 + (e & 3) : e] = y[e];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
    unsigned long long key = 0ull;
    for (int r = blockIdx.x * wpb + warp; r < vocab; r += gridDim.x * wpb) {
        float s = 0.f;
        if (wtype == LLM_Q8_0) {
            // 16 quants per lane and step, the warp's 512 bytes contiguous:
            // half a 32-element block times that block's scale (rows are
            // multiples of 32 elements, the quant rows 16-byte aligned)
            const uint8_t* q = out.q + (size_t)r * out.cols;
            const __half* d = out.d + (size_t)r * out.dstride;
#pragma unroll 4
            for (int e = 16 * lane; e < dim; e += 512) {
                const uint4 w = *reinterpret_cast<const uint4*>(q + e);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                const float4* y4 = reinterpret_cast<const float4*>(ys) + (size_t)(e >> 9) * 128 + lane;
                float t = 0.f;
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const float4 v = y4[32 * k];
                    const float yv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int c = 0; c < 4; c++)
                        t = fmaf((float)(int)(int8_t)((ws[k] >> (8 * c)) & 0xFFu), yv[c], t);
                }
                s = fmaf(__half2float(d[e >> 5]), t, s);
            }
        } else {
            // 8 F16 values per lane and step (16 bytes), 512 bytes per warp
            const __half* w = reinterpret_cast<const __half*>(out.q) + (size_t)r * out.cols;
#pragma unroll 4
            for (int e = 8 * lane; e < dim; e += 256) {
                const uint4 v = *reinterpret_cast<const uint4*>(w + e);
                const uint32_t vs[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&vs[j]));
                    s = fmaf(f.x, ys[e + 2 * j], s);
                    s = fmaf(f.y, ys[e + 2 * j + 1], s);
                }
            }
        }
        s = warp_sum(s);
        if (lane == 0) {
            logits[r] = s;
            const unsigned long long k = argmax_key(s, r);
            key = k > key ? k : key;
        }
    }
    if (lane == 0 && key) atomicMax(best, key);
}

// The F16 copy of a Q8_0 matrix (rows x cols, cols a multiple of 64): each
// thread expands one 16-value chunk with q4_to_f16, the routine the GEMM's
// converter warps use, so the copy holds the very values those warps write
// into shared memory (d * q rounded to nearest even).
__global__ void q8_expand_kernel(const uint8_t* __restrict__ q, const __half* __restrict__ d, int dstride, int rows,
                                 int cols, __half* __restrict__ y) {
    const int chunks = cols / 16;
    const long long total = (long long)rows * chunks;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long r = e / chunks;
        const int c = (int)(e % chunks);
        const __half2 d2 = __half2half2(d[r * dstride + c / 2]);
        const uint4 qv = *reinterpret_cast<const uint4*>(q + r * cols + c * 16);
        uint4 a, b;
        q4_to_f16(qv.x, d2, a.x, a.y);
        q4_to_f16(qv.y, d2, a.z, a.w);
        q4_to_f16(qv.z, d2, b.x, b.y);
        q4_to_f16(qv.w, d2, b.z, b.w);
        uint4* out = reinterpret_cast<uint4*>(y + r * cols + c * 16);
        out[0] = a;
        out[1] = b;
    }
}

__global__ void argmax_publish_kernel(unsigned long long* best, int* out) {
    griddep_entry();
    *out = argmax_key_index(*best);
    *best = 0ull;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D map of a [rows][K] F16 matrix, box 64 x box_rows, 128-byte swizzle.
// ------------------------------------------------ attention on tensor cores --
// Causal attention of 16 prompt rows of one kv head over the cache ("The
// Forward Pass in Java", Example 11; "What a Llama model computes, and why"
// §4: row i attends to positions 0..pos0+i), one warp per query head of the
// kv head.  Scores and the weighted V sum are mma.sync m16n8k16 products on
// F16 parts: q and the probabilities are split into hi = their F16 rounding
// and lo = the rest rounded to F16, so each product of a part with an F16 K
// or V element is exact and the two parts add up in the F32 accumulator
// (the same arithmetic as the decode step's attention).  The online softmax
// (running max and sum per row, rescaled accumulators) runs on the
// accumulator fragments; K and V arrive in 64-position tiles, double
// buffered with cp.async, in rows padded to HD + 8 halves so that ldmatrix
// reads them without bank conflicts.  Each head has `split` warps: warp
// (head, sp) takes the 16-position sub-tiles whose index is sp modulo split,
// and at the end warp sp = 0 folds the others' (max, sum, accumulators) into
// its own in the order sp = 1, 2, ... (the same bits in every run).  The
// output row is divided by its sum and rounded to F16 (the O projection's
// operand).
// (not volatile: a pure function of its operands, so the compiler may
// interleave independent accumulation chains)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_bits(__half a, __half b) {
    return (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
}

constexpr int kAttnKT = 128;                     // cache positions per K/V tile

template <int HD>
__global__ void __launch_bounds__(HD == 128 ? 256 : 512) attention_mma_kernel(const float* QKV, int n, int pos0,
                                                                              int n_heads, int n_kv,
                                                            float attn_div, const __half* kc, const __half* vc,
                                                            __half* A, int split) {
    griddep_entry();
    constexpr int PITCH = HD + 8;                // halves per shared-memory row
    extern __shared__ __align__(16) __half kvs[];   // [2 buffers][K, V][kAttnKT][PITCH]; then the warps' partials
    const int gq = n_heads / n_kv, q_dim = n_heads * HD, kv_dim = n_kv * HD, row_w = q_dim + 2 * kv_dim;
    const int ntile = (n + 15) / 16;
    // two query tiles per block, the longest with the shortest (tiles
    // ntile-1-i and i): equal work in every block, one wave of blocks
    const int bx = (int)blockIdx.x;
    for (int pass = 0; pass < 2; pass++) {
        const int qt = pass == 0 ? ntile - 1 - bx : bx;
        if (pass == 1) {
            if (qt >= ntile - 1 - bx) break;
            __syncthreads();                         // the fold's reads of the reused K/V buffer are done
        }
        const int g = blockIdx.y;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int hq = warp % gq, sp = warp / gq;
        const int h = g * gq + hq;
        const int t0 = qt * 16;
        const int r = lane >> 2, t = lane & 3;
        const int n_pos = pos0 + min(t0 + 16, n);    // positions the tile's last row attends to
        // this thread's two rows; rows past the batch take the last row's causal limit (never stored)
        const int R0 = min(t0 + r, n - 1), R1 = min(t0 + r + 8, n - 1);
        // q fragments: element (row t0 + r + 8 (j & 1), column ks*16 + 8 (j >> 1) + 2t + {0, 1})
        uint32_t qhi[HD / 16][4], qlo[HD / 16][4];
    #pragma unroll
        for (int ks = 0; ks < HD / 16; ks++)
    #pragma unroll
            for (int j = 0; j < 4; j++) {
                const int row = (j & 1) ? R1 : R0, col = ks * 16 + (j >> 1) * 8 + 2 * t;
                const float2 x = *reinterpret_cast<const float2*>(QKV + (size_t)row * row_w + h * HD + col);
                const __half hx = __float2half_rn(x.x), hy = __float2half_rn(x.y);
                qhi[ks][j] = h2_bits(hx, hy);
                qlo[ks][j] = h2_bits(__float2half_rn(x.x - __half2float(hx)), __float2half_rn(x.y - __half2float(hy)));
            }
        float o[HD / 8][4];
    #pragma unroll
        for (int nt = 0; nt < HD / 8; nt++) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

        const int ntiles = (n_pos + kAttnKT - 1) / kAttnKT;
        // score / sqrt(head_dim): a power-of-two divisor (head_dim 64, 256, ...)
        // divides exactly as a multiply by its reciprocal (the same bits)
        const bool div_pow2 = (__float_as_uint(attn_div) & 0x007FFFFFu) == 0u;
        const float inv_div = __frcp_rn(attn_div);
        auto scale_score = [&](float x) { return div_pow2 ? __fmul_rn(x, inv_div) : __fdiv_rn(x, attn_div); };
        auto load_tile = [&](int c, int buf) {
            __half* ks_ = kvs + (size_t)(buf * 2) * kAttnKT * PITCH;
            __half* vs_ = ks_ + kAttnKT * PITCH;
            constexpr int W = HD / 8;                // 16-byte words per row
            for (int e = threadIdx.x; e < kAttnKT * W; e += blockDim.x) {
                const int pr = e / W, w = e % W;
                const int pos = min(c * kAttnKT + pr, n_pos - 1);   // rows past n_pos repeat a valid row (masked)
                const size_t src = (size_t)pos * kv_dim + (size_t)g * HD + w * 8;
                cp_async16(ks_ + pr * PITCH + w * 8, kc + src);
                cp_async16(vs_ + pr * PITCH + w * 8, vc + src);
            }
            cp_async_commit();
        };
        load_tile(0, 0);
        for (int c = 0; c < ntiles; c++) {
            if (c + 1 < ntiles) {
                load_tile(c + 1, (c + 1) & 1);
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            } else {
                cp_async_wait_all();
            }
            __syncthreads();
            const __half* ks_ = kvs + (size_t)((c & 1) * 2) * kAttnKT * PITCH;
            const __half* vs_ = ks_ + kAttnKT * PITCH;
            const uint32_t kbase = smem_addr(ks_), vbase = smem_addr(vs_);
            // this warp's sub-tiles of the tile: global index = sp modulo split
            const int sub0 = ((sp - c * (kAttnKT / 16)) % split + split) % split;
            for (int sub = sub0; sub < kAttnKT / 16; sub += split) {
                const int p0 = c * kAttnKT + sub * 16;
                if (p0 >= n_pos) break;
                // scores of positions p0 + 8 nt + 2t + {0, 1}, rows r and r + 8
                float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                {
                    const int mi = lane >> 3, ri = lane & 7;
                    const uint32_t krow = kbase + (uint32_t)((sub * 16 + ri + (mi >= 2 ? 8 : 0)) * PITCH * 2);
    #pragma unroll
                    for (int ks = 0; ks < HD / 16; ks++) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(krow + (uint32_t)((ks * 16 + (mi & 1) * 8) * 2), b0, b1, b2, b3);
                        mma16816(s[0], qhi[ks], b0, b1);
                        mma16816(s[1], qhi[ks], b2, b3);
                        mma16816(s[0], qlo[ks], b0, b1);
                        mma16816(s[1], qlo[ks], b2, b3);
                    }
                }
                float mt0 = -INFINITY, mt1 = -INFINITY;
    #pragma unroll
                for (int nt = 0; nt < 2; nt++)
    #pragma unroll
                    for (int k = 0; k < 2; k++) {
                        const int P = p0 + nt * 8 + 2 * t + k;
                        s[nt][k] = P <= pos0 + R0 ? scale_score(s[nt][k]) : -INFINITY;
                        s[nt][2 + k] = P <= pos0 + R1 ? scale_score(s[nt][2 + k]) : -INFINITY;
                        mt0 = fmaxf(mt0, s[nt][k]);
                        mt1 = fmaxf(mt1, s[nt][2 + k]);
                    }
                mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, 1));
                mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, 2));
                mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, 1));
                mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, 2));
                const float mn0 = fmaxf(m0, mt0), mn1 = fmaxf(m1, mt1);
                const float c0 = expf(m0 - mn0), c1 = expf(m1 - mn1);   // 0 on the first tile (m = -inf)
                float ls0 = 0.f, ls1 = 0.f;
    #pragma unroll
                for (int nt = 0; nt < 2; nt++)
    #pragma unroll
                    for (int k = 0; k < 2; k++) {
                        s[nt][k] = expf(s[nt][k] - mn0);
                        s[nt][2 + k] = expf(s[nt][2 + k] - mn1);
                        ls0 += s[nt][k];
                        ls1 += s[nt][2 + k];
                    }
                ls0 += __shfl_xor_sync(0xffffffffu, ls0, 1);
                ls0 += __shfl_xor_sync(0xffffffffu, ls0, 2);
                ls1 += __shfl_xor_sync(0xffffffffu, ls1, 1);
                ls1 += __shfl_xor_sync(0xffffffffu, ls1, 2);
                l0 = l0 * c0 + ls0;
                l1 = l1 * c1 + ls1;
                m0 = mn0;
                m1 = mn1;
    #pragma unroll
                for (int nt = 0; nt < HD / 8; nt++) {
                    o[nt][0] *= c0;
                    o[nt][1] *= c0;
                    o[nt][2] *= c1;
                    o[nt][3] *= c1;
                }
                // probabilities as A fragments (the accumulator layout is the A layout): hi and lo parts
                uint32_t phi[4], plo[4];
    #pragma unroll
                for (int j = 0; j < 4; j++) {
                    const float x = s[j >> 1][(j & 1) * 2], y = s[j >> 1][(j & 1) * 2 + 1];
                    const __half hx = __float2half_rn(x), hy = __float2half_rn(y);
                    phi[j] = h2_bits(hx, hy);
                    plo[j] = h2_bits(__float2half_rn(x - __half2float(hx)), __float2half_rn(y - __half2float(hy)));
                }
                {
                    const int mi = lane >> 3, ri = lane & 7;
                    const uint32_t vrow = vbase + (uint32_t)((sub * 16 + ri + (mi & 1) * 8) * PITCH * 2);
    #pragma unroll
                    for (int nt = 0; nt < HD / 8; nt += 2) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(vrow + (uint32_t)(((nt + (mi >> 1)) * 8) * 2), b0, b1, b2, b3);
                        mma16816(o[nt], phi, b0, b1);
                        mma16816(o[nt + 1], phi, b2, b3);
                        mma16816(o[nt], plo, b0, b1);
                        mma16816(o[nt + 1], plo, b2, b3);
                    }
                }
            }
            __syncthreads();                         // the buffer is reloaded two tiles later
        }
        // fold the head's other warps into warp sp = 0, in the order sp = 1, 2, ...
        if (split > 1) {
            constexpr int NV = HD / 2 + 4;           // a lane's accumulators, then m0, m1, l0, l1
            float* part = reinterpret_cast<float*>(kvs);   // the K/V tiles are no longer read
            if (sp > 0) {
                float* pw = part + (size_t)((sp - 1) * gq + hq) * NV * 32 + lane;
    #pragma unroll
                for (int nt = 0; nt < HD / 8; nt++)
    #pragma unroll
                    for (int k = 0; k < 4; k++) pw[(nt * 4 + k) * 32] = o[nt][k];
                pw[(HD / 2) * 32] = m0;
                pw[(HD / 2 + 1) * 32] = m1;
                pw[(HD / 2 + 2) * 32] = l0;
                pw[(HD / 2 + 3) * 32] = l1;
            }
            __syncthreads();
            if (sp > 0) continue;                    // warp 0 of the head folds and stores
            for (int k2 = 1; k2 < split; k2++) {
                const float* pw = part + (size_t)((k2 - 1) * gq + hq) * NV * 32 + lane;
                const float om0 = pw[(HD / 2) * 32], om1 = pw[(HD / 2 + 1) * 32];
                const float M0 = fmaxf(m0, om0), M1 = fmaxf(m1, om1);
                const float a0 = m0 == -INFINITY ? 0.f : expf(m0 - M0), b0 = om0 == -INFINITY ? 0.f : expf(om0 - M0);
                const float a1 = m1 == -INFINITY ? 0.f : expf(m1 - M1), b1 = om1 == -INFINITY ? 0.f : expf(om1 - M1);
                l0 = l0 * a0 + pw[(HD / 2 + 2) * 32] * b0;
                l1 = l1 * a1 + pw[(HD / 2 + 3) * 32] * b1;
                m0 = M0;
                m1 = M1;
    #pragma unroll
                for (int nt = 0; nt < HD / 8; nt++) {
                    o[nt][0] = o[nt][0] * a0 + pw[(nt * 4 + 0) * 32] * b0;
                    o[nt][1] = o[nt][1] * a0 + pw[(nt * 4 + 1) * 32] * b0;
                    o[nt][2] = o[nt][2] * a1 + pw[(nt * 4 + 2) * 32] * b1;
                    o[nt][3] = o[nt][3] * a1 + pw[(nt * 4 + 3) * 32] * b1;
                }
            }
        }
        const float i0 = 1.0f / l0, i1 = 1.0f / l1;
        const int row0 = t0 + r, row1 = t0 + r + 8;
    #pragma unroll
        for (int nt = 0; nt < HD / 8; nt++) {
            const int col = h * HD + nt * 8 + 2 * t;
            if (row0 < n)
                *reinterpret_cast<__half2*>(A + (size_t)row0 * q_dim + col) =
                    __floats2half2_rn(o[nt][0] * i0, o[nt][1] * i0);
            if (row1 < n)
                *reinterpret_cast<__half2*>(A + (size_t)row1 * q_dim + col) =
                    __floats2half2_rn(o[nt][2] * i1, o[nt][3] * i1);
        }
    }
}

// The tensor-core attention for the head sizes it is instantiated for and up
// to 8 query heads per kv head; other shapes keep attention_rows_kernel.
bool attention_mma_launch(cudaStream_t st, const float* QKV, int n, int pos0, int n_heads, int n_kv, int hd,
                          float attn_div, const __half* kc, const __half* vc, __half* A, cudaError_t* e) {
    const int gq = n_heads / n_kv;
    if (gq > 8 || !(hd == 32 || hd == 64 || hd == 128)) return false;
    // warps per head: up to 4, at most 16 warps a block (8 for head_dim 128,
    // whose accumulators need twice the registers)
    const int split = std::max(1, std::min(4, (hd == 128 ? 8 : 16) / gq));
    const dim3 grid(((n + 15) / 16 + 1) / 2, n_kv), block(32 * gq * split);   // two query tiles per block
    const size_t kv_bytes = (size_t)2 * 2 * kAttnKT * (hd + 8) * sizeof(__half);
    const size_t part_bytes = (size_t)(split - 1) * gq * (hd / 2 + 4) * 32 * sizeof(float);
    const size_t smem = std::max(kv_bytes, part_bytes);
    const void* fn = hd == 32 ? (const void*)attention_mma_kernel<32>
                     : hd == 64 ? (const void*)attention_mma_kernel<64>
                                : (const void*)attention_mma_kernel<128>;
    if (smem > 48 * 1024) {
        *e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (*e != cudaSuccess) return true;
    }
    auto k = hd == 32 ? attention_mma_kernel<32> : hd == 64 ? attention_mma_kernel<64> : attention_mma_kernel<128>;
    *e = launch_dep(k, grid, block, smem, st, QKV, n, pos0, n_heads, n_kv, attn_div, kc, vc, A, split);
    return true;
}

bool gemm_map(CUtensorMap* m, const void* base, int K, int rows, int box_rows = 128) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kGBK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The int8 quants of a Q8_0 matrix in the library layout ([rows][K], K
// contiguous) as BN x 64 boxes, 64-byte swizzle (sw64_chunk).
bool q8_map(CUtensorMap* m, const void* base, int K, int rows, int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)K};
    cuuint32_t box[2] = {(cuuint32_t)kGBK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One GEMM: min(tiles, SMs) persistent CTAs.  mb: the F16 weight tiles, or
// for Q8 the quant tiles (scales in ws).
template <int BN, int EPI, bool Q8>
cudaError_t gemm(cudaStream_t st, int sms, const CUtensorMap& ma, const CUtensorMap& mb, GemmScales ws,
                 const GemmOut& o, int M, int N, int K, int* err) {
    using G = GemmPlan<BN, Q8>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel<BN, EPI, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             G::kSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int tiles = ((M + kGBM - 1) / kGBM) * ((N + BN - 1) / BN);
    return launch_dep(gemm_kernel<BN, EPI, Q8>, dim3(tiles < sms ? tiles : sms), dim3(G::kThreads), (size_t)G::kSmem, st,
                      ma, mb, ws, o, M, N, K, err);
}

}  // namespace

bool prefill_supported(const PrefillCtx& c) {
    return (c.wtype == LLM_F16 || c.wtype == LLM_Q8_0) && c.dim % kGBK == 0 && c.q_dim % kGBK == 0 && c.ffn % kGBK == 0 &&
           c.n_heads / c.n_kv * c.hd <= 8 * 128 && c.rope_dims / 2 <= 128;
}

// The four GEMM weight matrices of layer l (QKV, O, gate/up as single rows,
// down): their rows and columns, and their element offsets in the F16 copy
// (each matrix starts 256-byte aligned).
static void copy_shape(const PrefillCtx& c, int l, int k, int* rows, int* cols) {
    const LayerDev& L = c.layers[l];
    switch (k) {
        case 0: *rows = L.qkv.rows; *cols = c.dim; break;
        case 1: *rows = L.o.rows; *cols = c.q_dim; break;
        case 2: *rows = 2 * L.gu.rows; *cols = c.dim; break;
        default: *rows = L.down.rows; *cols = c.ffn; break;
    }
}

static size_t copy_offset(const PrefillCtx& c, int l, int k) {
    size_t off = 0;
    for (int i = 0; i < 4 * l + k; i++) {
        int rows, cols;
        copy_shape(c, i / 4, i % 4, &rows, &cols);
        off += ((size_t)rows * cols + 127) & ~(size_t)127;
    }
    return off;
}

size_t prefill_f16_copy_bytes(const PrefillCtx& c) { return copy_offset(c, c.n_layers, 0) * sizeof(__half); }

cudaError_t prefill_make_f16_copy(const PrefillCtx& c, __half* dst, int* launches) {
    *launches = 0;
    if (c.wtype != LLM_Q8_0) return cudaErrorInvalidValue;
    for (int l = 0; l < c.n_layers; l++) {
        const LayerDev& L = c.layers[l];
        const DMat* m[4] = {&L.qkv, &L.o, &L.gu, &L.down};
        for (int k = 0; k < 4; k++) {
            int rows, cols;
            copy_shape(c, l, k, &rows, &cols);
            const long long chunks = (long long)rows * (cols / 16);
            const int blocks = (int)((chunks + 255) / 256 < 65535 ? (chunks + 255) / 256 : 65535);
            q8_expand_kernel<<<blocks, 256, 0, c.st>>>(static_cast<const uint8_t*>(m[k]->q), m[k]->d, m[k]->dstride,
                                                      rows, cols, dst + copy_offset(c, l, k));
            ++*launches;
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

size_t prefill_workspace_bytes(const PrefillCtx& c) {
    const size_t M = kPrefillRows;
    auto al = [](size_t b) { return (b + 255) & ~(size_t)255; };
    return al(M * 4) + al(M * c.dim * 4) + al(M * c.dim * 2) + al(M * (c.q_dim + 2 * c.kv_dim) * 4) +
           al(M * c.q_dim * 2) + al(M * c.ffn * 2) + al((size_t)c.dim * 4) + al(M * (c.rope_dims / 2) * 8);
}

// Runs the batch; `ws` holds prefill_workspace_bytes(c).  Returns a CUDA error
// or cudaSuccess; *msg names the failing step.
cudaError_t prefill_f16(const PrefillCtx& c, void* ws, const int32_t* tokens_host, int n, int pos0, const char** msg) {
    auto al = [](size_t b) { return (b + 255) & ~(size_t)255; };
    const size_t M = kPrefillRows;
    uint8_t* w = static_cast<uint8_t*>(ws);
    int* tok = reinterpret_cast<int*>(w); w += al(M * 4);
    float* X = reinterpret_cast<float*>(w); w += al(M * c.dim * 4);
    __half* Xh = reinterpret_cast<__half*>(w); w += al(M * c.dim * 2);
    float* QKV = reinterpret_cast<float*>(w); w += al(M * (c.q_dim + 2 * c.kv_dim) * 4);
    __half* Ah = reinterpret_cast<__half*>(w); w += al(M * c.q_dim * 2);
    __half* Hh = reinterpret_cast<__half*>(w); w += al(M * c.ffn * 2);
    float* ylast = reinterpret_cast<float*>(w); w += al((size_t)c.dim * 4);
    float* rtab = reinterpret_cast<float*>(w); w += al(M * (c.rope_dims / 2) * 8);   // the batch's cos/sin table
    cudaError_t e;
#define PF_CK(call, what)                 \
    do {                                  \
        if ((e = (call)) != cudaSuccess) { \
            *msg = what;                  \
            return e;                     \
        }                                 \
    } while (0)
    CUtensorMap mXh, mAh, mHh;
    if (!gemm_map(&mXh, Xh, c.dim, (int)M) || !gemm_map(&mAh, Ah, c.q_dim, (int)M) || !gemm_map(&mHh, Hh, c.ffn, (int)M)) {
        *msg = "tensor map of an activation operand";
        return cudaErrorInvalidValue;
    }
    // weight operands: the F16 matrices, the F16 copy of the Q8_0 ones, or
    // the int8 quants of the Q8_0 ones (expanded to F16 tile by tile inside
    // the GEMM), per layer: QKV, O, gate/up (single rows), down; box heights =
    // the GEMMs' tile widths
    const bool q8 = c.wtype == LLM_Q8_0 && !c.f16_copy;
    std::vector<CUtensorMap> mw((size_t)4 * c.n_layers);
    static constexpr int kBox[4] = {kBnQkv, kBnNarrow, kBnWide, kBnNarrow};
    for (int l = 0; l < c.n_layers; l++) {
        const LayerDev& L = c.layers[l];
        const DMat* dm[4] = {&L.qkv, &L.o, &L.gu, &L.down};
        for (int k = 0; k < 4; k++) {
            int rows, cols;
            copy_shape(c, l, k, &rows, &cols);
            const void* base = c.f16_copy ? static_cast<const void*>(c.f16_copy + copy_offset(c, l, k)) : dm[k]->q;
            if (!(q8 ? q8_map(&mw[4 * l + k], base, cols, rows, kBox[k])
                     : gemm_map(&mw[4 * l + k], base, cols, rows, kBox[k]))) {
                *msg = "tensor map of a weight matrix";
                return cudaErrorInvalidValue;
            }
        }
    }
    auto run = [&](auto bn, auto epi, const CUtensorMap& ma, const CUtensorMap& mb, const DMat& wm, const GemmOut& o,
                   int M, int N, int K) -> cudaError_t {
        constexpr int BN = decltype(bn)::value, EPI = decltype(epi)::value;
        const GemmScales sc{wm.d, wm.dstride};
        return q8 ? gemm<BN, EPI, true>(c.st, c.sms, ma, mb, sc, o, M, N, K, c.err)
                  : gemm<BN, EPI, false>(c.st, c.sms, ma, mb, sc, o, M, N, K, c.err);
    };
    using Qkv = std::integral_constant<int, kBnQkv>;
    using Narrow = std::integral_constant<int, kBnNarrow>;
    using Wide = std::integral_constant<int, kBnWide>;
    using EBias = std::integral_constant<int, kEpiBias>;
    using EResid = std::integral_constant<int, kEpiResidual>;
    using ESwi = std::integral_constant<int, kEpiSwiGLU>;
    const int gq = c.n_heads / c.n_kv;
    const int attn_smem = (int)(2 * sizeof(__half) * kAttnTile * c.hd +
                                sizeof(float) * ((size_t)gq * c.hd + (size_t)gq * kAttnTile + 3 * gq));
    if (attn_smem > 48 * 1024)
        PF_CK(cudaFuncSetAttribute(attention_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, attn_smem),
              "attention shared memory");
    for (int b0 = 0; b0 < n; b0 += kPrefillRows) {
        const int nb = n - b0 < kPrefillRows ? n - b0 : kPrefillRows;
        const int p0 = pos0 + b0;
        PF_CK(cudaMemcpyAsync(tok, tokens_host + b0, (size_t)nb * 4, cudaMemcpyHostToDevice, c.st), "token upload");
        PF_CK(launch_dep(embed_rows_kernel, dim3(nb), dim3(256), 0, c.st, tok, nb, c.embd, c.wtype, c.dim, X),
              "embedding");
        {
            const int cells = nb * (c.rope_dims / 2);
            PF_CK(launch_dep(rope_table_kernel, dim3((cells + 255) / 256), dim3(256), 0, c.st, rtab, nb, p0,
                             c.rope_dims / 2, c.theta_scale, c.rope_freqs),
                  "RoPE table");
        }
        // RMSNorm: one warp per row, two rows per block, so a batch's rows
        // spread over every SM (the row stream is bound by each SM's intake)
        constexpr int kNormRows = 2;
        const int norm_blocks = (nb + kNormRows - 1) / kNormRows;
        for (int l = 0; l < c.n_layers; l++) {
            const LayerDev& L = c.layers[l];
            PF_CK(launch_dep(rmsnorm_rows_f16_kernel, dim3(norm_blocks), dim3(32 * kNormRows), 0, c.st, X, nb, c.dim,
                             L.attn_norm, c.eps, Xh),
                  "attention RMSNorm");
            GemmOut oq{QKV, L.qkv_bias, nullptr, nullptr};
            PF_CK(run(Qkv{}, EBias{}, mXh, mw[4 * l + 0], L.qkv, oq, nb, L.qkv.rows, c.dim), "QKV GEMM");
            PF_CK(launch_dep(rope_kv_rows_kernel, dim3(nb), dim3(128), 0, c.st, QKV, nb, p0, c.n_heads, c.n_kv, c.hd,
                             c.rope_dims, c.neox, rtab, L.kc, L.vc),
                  "RoPE and KV append");
            {
                cudaError_t ea = cudaSuccess;
                if (!attention_mma_launch(c.st, QKV, nb, p0, c.n_heads, c.n_kv, c.hd, c.attn_div, L.kc, L.vc, Ah, &ea)) {
                    ea = launch_dep(attention_rows_kernel, dim3(nb, c.n_kv), dim3(128), (size_t)attn_smem, c.st, QKV,
                                    nb, p0, c.n_heads, c.n_kv, c.hd, c.attn_div, L.kc, L.vc, Ah);
                }
                PF_CK(ea, "attention");
            }
            GemmOut oo{nullptr, nullptr, X, nullptr};
            PF_CK(run(Narrow{}, EResid{}, mAh, mw[4 * l + 1], L.o, oo, nb, c.dim, c.q_dim), "O GEMM");
            PF_CK(launch_dep(rmsnorm_rows_f16_kernel, dim3(norm_blocks), dim3(32 * kNormRows), 0, c.st, X, nb, c.dim,
                             L.ffn_norm, c.eps, Xh),
                  "FFN RMSNorm");
            GemmOut og{nullptr, nullptr, nullptr, Hh};
            PF_CK(run(Wide{}, ESwi{}, mXh, mw[4 * l + 2], L.gu, og, nb, 2 * L.gu.rows, c.dim), "gate/up GEMM");
            GemmOut od{nullptr, nullptr, X, nullptr};
            PF_CK(run(Narrow{}, EResid{}, mHh, mw[4 * l + 3], L.down, od, nb, c.dim, c.ffn), "down GEMM");
        }
        if (b0 + nb == n) {
            PF_CK(launch_dep(final_norm_kernel, dim3(1), dim3(256), 0, c.st, (const float*)(X + (size_t)(nb - 1) * c.dim),
                             c.dim, c.out_norm, c.eps, ylast),
                  "final RMSNorm");
            PF_CK(launch_dep(logits_kernel, dim3(c.sms * 4), dim3(256), (size_t)((c.dim + 511) & ~511) * 4, c.st,
                             c.out, c.wtype, (const float*)ylast, c.dim, c.vocab, c.logits, c.best),
                  "logits");
            PF_CK(launch_dep(argmax_publish_kernel, dim3(1), dim3(1), 0, c.st, c.best, c.argmax_dev), "argmax");
        }
    }
#undef PF_CK
    return cudaSuccess;
}

}  // namespace llm
