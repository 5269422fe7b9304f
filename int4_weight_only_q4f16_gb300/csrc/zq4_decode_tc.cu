// zq4_decode_tc.cu -- the decode GEMV for M = 1..16 on GB300: weight tiles
// streamed by TMA into shared memory, multiply-accumulate on the tensor
// cores.
//
// What it computes: y = x * W^T with W in q4f16_1 ("Zero TVM Documentation",
// section "Q4F16 quantization format" and card 5 "int4 Matmul"), or the fused
// gate_up + SiLU*mul epilogue (card 6 "Fused FFN") when rows are interleaved
// gate/up pairs.
//
// How:
//  * CTA = 8 compute warps + 1 producer warp; the CTA owns 16-row tiles of W
//    (grid-stride). The producer streams a tile in stages of 16 rows x 1024
//    columns through a 4-stage shared-memory ring: four 2D tensor-map TMA
//    boxes of [16 rows x 128 B] of codes (128-byte swizzle) and one box of
//    [16 rows x 32] scales per stage, completion on an mbarrier. Rows past N
//    and columns past K are zero-filled by the TMA unit. The producer starts
//    before griddepcontrol.wait: weights never depend on the previous kernel,
//    so the next kernel's weight stream overlaps this one's tail. Beyond the
//    ring it keeps a window of 16 stages requested into L2 with tensor-map
//    prefetches (loaded DRAM latency on GB300 is ~3 us; ring refills then hit
//    L2).
//  * Each compute warp takes an eighth of a stage's 32-column groups. Per
//    group, lane (r, t) (r = lane/4, t = lane%4) unpacks word t of rows r and
//    r+8 into four f16 pairs that are the A fragments of two chained
//    m16n8k16 MMAs; the B fragment is the matching pair-permuted x chunk of
//    token r (x staged once per CTA in shared memory). The k order inside a
//    group is permuted identically on both operands, which leaves the dot
//    product unchanged. The group's fp32 MMA result is scaled by the fp32
//    group scale into a running fp32 accumulator.
//  * Unpack forms (ZQ4_TC_UNPACK): 0 (default) gives exact (q - 7) pairs
//    (0,4),(1,5),(2,6),(3,7) with one shift, four LOP3 and four f16x2 ops per
//    word. 1 and 2 give exact q/8 pairs (0,2),(1,3),(4,6),(5,7) with one
//    shift, two masks and four e2m3->f16x2 conversions (a code alone in a
//    byte read as e2m3 is q/8), two fewer half-rate instructions per word;
//    the zero-point term sum (7/8) x then comes from the same MMA chain with
//    every A element 7/8 (inline in form 1, once per CTA in form 2), so a row
//    of all-7 codes still gives exactly 0. The exact form is the default: in
//    the latency-bound regime measured here the zero-point work costs more
//    than the saved instructions.
//  * Tiles are reduced across the 8 warps through shared memory; the epilogue
//    writes f16 y (or silu(g)*u for interleaved gate/up rows).
//  * Every mbarrier wait is bounded in time; on expiry the kernel records
//    ZQ4_DEVERR_WAIT_TIMEOUT, drains the copies it issued, and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <type_traits>
#include <cstring>
#include <atomic>

#include "zq4_async.cuh"
#include "zq4_common.cuh"
#include "zq4_internal.h"
#include "zq4_rope.cuh"

namespace zq4 {

__device__ unsigned g_device_error = 0;

namespace tc {

// 4D tensor-map TMA load / L2 prefetch of one box at (c0, c1, c2, c3)
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            uint32_t mbar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(mbar)
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap *map, int c0, int c1, int c2, int c3)
{
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// Tile parameters (compile-time; the defaults are the tuned values).
#ifndef ZQ4_TC_WARPS
#define ZQ4_TC_WARPS 8
#endif
#ifndef ZQ4_TC_STAGES
#define ZQ4_TC_STAGES 4
#endif
#ifndef ZQ4_TC_OCC
#define ZQ4_TC_OCC 2
#endif
#ifndef ZQ4_TC_UNROLL
#define ZQ4_TC_UNROLL 4
#endif
// Unpack form: 0 = exact (q - 7) (no zero-point term), 1 = q/8 via e2m3 with
// the zero-point MMA chain inline, 2 = q/8 via e2m3 with the zero-point term
// computed once per CTA.
#ifndef ZQ4_TC_UNPACK
#define ZQ4_TC_UNPACK 0
#endif
#ifndef ZQ4_TC_KC
#define ZQ4_TC_KC 1024
#endif
// Stages of L2 look-ahead beyond the shared-memory ring.
#ifndef ZQ4_TC_PREFETCH
#define ZQ4_TC_PREFETCH 16
#endif

constexpr int kWarps = ZQ4_TC_WARPS;              // compute warps
constexpr int kThreads = (kWarps + 1) * 32;       // + producer warp
constexpr int kKC = ZQ4_TC_KC;                    // columns per stage
constexpr int kSegs = kKC / 256;                  // 128-byte code segments per row per stage
constexpr int kSegBytes = 16 * 128;               // one swizzled [16 rows x 128 B] box
constexpr int kScaleCols = kKC / 32;              // scales per row per stage
constexpr int kScaleBytes = 16 * kScaleCols * 2;  // [16 rows x kScaleCols scales]
constexpr int kStageBytes = kSegs * kSegBytes + kScaleBytes;   // 9 KB, a multiple of 1 KB
constexpr int kStages = ZQ4_TC_STAGES;
constexpr int kUnrollG = ZQ4_TC_UNROLL;           // groups unrolled per loop trip
constexpr int kGpw = (kKC / 32 + kWarps - 1) / kWarps;   // groups of a stage per warp
constexpr uint32_t kSevenEighths = 0x3B003B00u;   // f16x2 (7/8, 7/8)
constexpr int kUnpack = ZQ4_TC_UNPACK;
constexpr int kPrefetch = ZQ4_TC_PREFETCH;
constexpr int kPartLoads = 16;                    // add + RMSNorm: at most 32 x 16 CTAs per launch
__device__ __forceinline__ float lo_f32(uint32_t w) { return f16_bits_to_float(uint16_t(w)); }
__device__ __forceinline__ float hi_f32(uint32_t w) { return f16_bits_to_float(uint16_t(w >> 16)); }

static_assert(kStageBytes % 1024 == 0, "stages must keep the 1 KB swizzle alignment");

__device__ __forceinline__ void named_barrier_compute()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
}

// ---------------------------------------------------------------------------
// Shared-memory layout (offsets from a 1 KB aligned base)
// ---------------------------------------------------------------------------
__host__ __device__ inline size_t xs_row_bytes(int K) { return size_t(K) * 2 + 64; }
constexpr size_t kRingBytes = size_t(kStages) * kStageBytes;
constexpr size_t kMbarBytes = (16 * kStages + 127) / 128 * 128;   // full + empty per stage
template <int NB>
__host__ __device__ inline size_t red_bytes() { return size_t(kWarps) * NB * 16 * 8 * 4; }
__host__ __device__ inline size_t scale_bytes() { return size_t(kWarps) * kGpw * 8 * 8; }
// zero-point term of every (group, token): E[g][m] = sum_k in g (7/8) x[m,k]
template <int NB>
__host__ __device__ inline size_t zp_bytes(int K) { return kUnpack == 2 ? size_t(K / 32) * 8 * NB * 4 : 0; }

template <int NB>
__host__ __device__ inline size_t smem_bytes(int M, int K)
{
    return 1024 /* alignment slack */ + kRingBytes + kMbarBytes + red_bytes<NB>() + scale_bytes() +
           zp_bytes<NB>(K) + size_t(M) * xs_row_bytes(K);
}

// Argmax key of logit v at row n: the float's bits made order-preserving as
// an unsigned integer in the high word, ~n in the low word, so that the
// largest key is the largest logit and, among equal logits, the lowest row.
// -0 is taken as +0 (equal values tie), and every NaN gets the top value
// (a NaN counts as the largest; the first one wins).
__device__ __forceinline__ unsigned long long argmax_key(float v, int n)
{
    unsigned ord;
    if (v != v) {
        ord = 0xffffffffu;
    } else {
        const unsigned b = v == 0.f ? 0u : __float_as_uint(v);
        ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    }
    return (static_cast<unsigned long long>(ord) << 32) | static_cast<unsigned>(~unsigned(n));
}

// The QKV + RoPE mode's arguments: TcArgs and base^(-2i/D) for i < D/2, in
// fp64, computed on the host (the kernel reads them from parameter space).
struct TcRopeArgs : TcArgs {
    double freq[256];
};
// The MLX affine format's arguments: TcArgs and the biases' tensor map (the
// scales' map then holds one scale per 64 weights too).
struct TcAffArgs : TcArgs {
    CUtensorMap tm_bias;
};
template <int RU, bool AFF>
using TcArgsFor = typename std::conditional<AFF, TcAffArgs,
                                            typename std::conditional<RU == 5, TcRopeArgs, TcArgs>::type>::type;

// Affine unpack: four f16x2 values holding q exactly (no zero point), the
// element pairs of unpack_word_f16x2 (magic-number OR, then the bias removed).
__device__ __forceinline__ void unpack_word_q_f16x2(uint32_t w, uint32_t p[4])
{
    const uint32_t kMagic = 0x64006400u;       // (1024, 1024)
    const uint32_t kSixteenth = 0x2C002C00u;   // (1/16, 1/16)
    const uint32_t kNeg64 = 0xD400D400u;       // (-64, -64): 1024/16
    uint32_t w8 = w >> 8;
    p[0] = hsub2(and_or<0x000F000Fu>(w, kMagic), kMagic);
    p[1] = hfma2(and_or<0x00F000F0u>(w, kMagic), kSixteenth, kNeg64);
    p[2] = hsub2(and_or<0x000F000Fu>(w8, kMagic), kMagic);
    p[3] = hfma2(and_or<0x00F000F0u>(w8, kMagic), kSixteenth, kNeg64);
}
// affine: per-warp bias scratch and the x sums of every 64-column group ([K/64][16] floats)
__host__ __device__ inline size_t aff_bytes(int K) { return scale_bytes() + size_t(K / 64) * 16 * 4; }

template <int NB, int RU, bool AFF = false>
__global__ void __launch_bounds__(kThreads) k_decode_tc(const __grid_constant__ CUtensorMap tm_codes,
                                                        const __grid_constant__ CUtensorMap tm_scales,
                                                        const __grid_constant__ TcArgsFor<RU, AFF> a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const uint32_t ring = smem_addr(smem);
    const uint32_t full0 = ring + uint32_t(kRingBytes), empty0 = full0 + 8 * kStages;
    float *red = reinterpret_cast<float *>(smem + kRingBytes + kMbarBytes);
    float2 *sscr = reinterpret_cast<float2 *>(smem + kRingBytes + kMbarBytes + red_bytes<NB>());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = a.K, N = a.N;
    float *zp = reinterpret_cast<float *>(smem + kRingBytes + kMbarBytes + red_bytes<NB>() + scale_bytes());
    uint8_t *xs = smem + kRingBytes + kMbarBytes + red_bytes<NB>() + scale_bytes() + zp_bytes<NB>(K);
    // affine: per-warp bias scratch (as sscr) and the x sums of the 32-column groups, after x
    float2 *sbias = reinterpret_cast<float2 *>(xs + size_t(a.M) * xs_row_bytes(K));
    float *xsum = reinterpret_cast<float *>(xs + size_t(a.M) * xs_row_bytes(K) + scale_bytes());
    const int chunks = (K + kKC - 1) / kKC;
    // add + RMSNorm epilogue: squares of a tile's rows, the CTA's running sums per token
    __shared__ float s_sq[RU == 4 ? 16 : 1][16];
    __shared__ float s_ss[RU == 4 ? 16 : 1];
    if (RU == 4 && threadIdx.x < 16) s_ss[threadIdx.x] = 0.f;
    // QKV + RoPE epilogue: the tokens' positions and slots
    __shared__ int s_pos[RU == 5 ? 16 : 1], s_slot[RU == 5 ? 16 : 1];

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kWarps) {
        // ---------------- producer warp ----------------
        // Stage j of this CTA is chunk j % chunks of tile blockIdx + (j / chunks) * grid.
        const int nstage = ((a.tiles - int(blockIdx.x) + int(gridDim.x) - 1) / int(gridDim.x)) * chunks;
        const int tpp = RU == 5 ? a.D >> 4 : 1;          // RoPE: tiles per head
        auto prefetch_stage = [&](int j) {
            if (j >= nstage) return;
            const int tile = blockIdx.x + (j / chunks) * gridDim.x, k0 = (j % chunks) * kKC;
            const int nseg = min(kKC, K - k0) / 256;
            if (RU == 5) {
                const int hb = tile / tpp, i0 = (tile - hb * tpp) * 8;
                for (int g = 0; g < nseg; ++g) tma_prefetch_4d(&tm_codes, (k0 >> 3) + 32 * g, i0, 0, hb);
                tma_prefetch_4d(&tm_scales, k0 >> 5, i0, 0, hb);
                return;
            }
            for (int g = 0; g < nseg; ++g) tma_prefetch_2d(&tm_codes, (k0 >> 3) + 32 * g, tile * 16);
            if (AFF) {
                tma_prefetch_2d(&tm_scales, k0 >> 6, tile * 16);
                if constexpr (AFF) tma_prefetch_2d(&a.tm_bias, k0 >> 6, tile * 16);
            } else {
                tma_prefetch_2d(&tm_scales, k0 >> 5, tile * 16);
            }
        };
        // L2 look-ahead: the stages after the ring's first fill are requested
        // from DRAM now (before the grid-dependency wait), so ring refills
        // later hit L2 instead of paying the DRAM latency.
        if (lane == 0)
            for (int j = kStages; j < kStages + kPrefetch; ++j) prefetch_stage(j);
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < a.tiles && ok; tile += gridDim.x) {
            for (int c = 0; c < chunks; ++c, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                // The first kStages fills need no wait and run before the
                // previous grid completes; from then on the consumers must be
                // past their own wait on the previous grid for a stage to free.
                if (it == kStages) griddep_wait();
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const int k0 = c * kKC, nseg = min(kKC, K - k0) / 256;
                    const uint32_t full = full0 + 8 * s, st = ring + s * kStageBytes;
                    mbar_arrive_expect_tx(full, uint32_t(nseg * kSegBytes + kScaleBytes));
                    if (RU == 5) {
                        const int hb = tile / tpp, i0 = (tile - hb * tpp) * 8;
                        for (int g = 0; g < nseg; ++g)
                            tma_load_4d(st + g * kSegBytes, &tm_codes, (k0 >> 3) + 32 * g, i0, 0, hb, full);
                        tma_load_4d(st + kSegs * kSegBytes, &tm_scales, k0 >> 5, i0, 0, hb, full);
                    } else {
                        for (int g = 0; g < nseg; ++g)
                            tma_load_2d(st + g * kSegBytes, &tm_codes, (k0 >> 3) + 32 * g, tile * 16, full);
                        if (AFF) {                        // scales, then biases: one per 64 columns, 512 B each
                            tma_load_2d(st + kSegs * kSegBytes, &tm_scales, k0 >> 6, tile * 16, full);
                            if constexpr (AFF)
                                tma_load_2d(st + kSegs * kSegBytes + kScaleBytes / 2, &a.tm_bias, k0 >> 6, tile * 16, full);
                        } else {
                            tma_load_2d(st + kSegs * kSegBytes, &tm_scales, k0 >> 5, tile * 16, full);
                        }
                    }
                    if (it >= kStages) prefetch_stage(it + kPrefetch);   // keep the window moving
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) atomicOr(&g_device_error, ZQ4_DEVERR_WAIT_TIMEOUT);
        // Drain: never leave the CTA with copies in flight into its smem.
        for (int j = max(0, it - kStages); j < it; ++j) {
            if (!mbar_wait(full0 + 8 * (j % kStages), (j / kStages) & 1)) {
                if (lane == 0) atomicOr(&g_device_error, ZQ4_DEVERR_WAIT_TIMEOUT);
                break;
            }
        }
        return;
    }

    // ---------------- compute warps ----------------
    griddep_wait();
    if (RU == 5 && threadIdx.x < a.M) {                  // positions and slots of the launch's tokens
        s_pos[threadIdx.x] = a.pos[threadIdx.x];
        s_slot[threadIdx.x] = a.slot[threadIdx.x];
    }
    const uint32_t xrow = uint32_t(xs_row_bytes(K));
    {
        // Stage x[0..M): the 8 values of word chunk cw of token m are stored
        // as the pairs (x0,x2),(x1,x3),(x4,x6),(x5,x7) the unpack produces.
        // Loads are issued kBatch at a time so their latencies overlap.
        constexpr int kBatch = 8;
        const int words = K >> 3, total = a.M * words;
        for (int i0 = threadIdx.x; i0 < total; i0 += kBatch * kWarps * 32) {
            uint4 v[kBatch];
            // exact unpack pairs elements (i, i+4); the e2m3 unpack (0,2),(1,3),(4,6),(5,7)
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int i = i0 + b * kWarps * 32;
                if (i < total) {
                    const int m = i / words, cw = i - m * words;
                    v[b] = *reinterpret_cast<const uint4 *>(a.x + size_t(m) * K + size_t(cw) * 8);
                }
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int i = i0 + b * kWarps * 32;
                if (i < total) {
                    const int m = i / words, cw = i - m * words;
                    uint4 o;
                    if (kUnpack == 0) {
                        o.x = __byte_perm(v[b].x, v[b].z, 0x5410);
                        o.y = __byte_perm(v[b].x, v[b].z, 0x7632);
                        o.z = __byte_perm(v[b].y, v[b].w, 0x5410);
                        o.w = __byte_perm(v[b].y, v[b].w, 0x7632);
                    } else {
                        o.x = __byte_perm(v[b].x, v[b].y, 0x5410);
                        o.y = __byte_perm(v[b].x, v[b].y, 0x7632);
                        o.z = __byte_perm(v[b].z, v[b].w, 0x5410);
                        o.w = __byte_perm(v[b].z, v[b].w, 0x7632);
                    }
                    *reinterpret_cast<uint4 *>(xs + size_t(m) * xrow + size_t(cw) * 16) = o;
                }
            }
        }
    }
    named_barrier_compute();
    if (AFF) {
        // the x sums of every 64-column group (one scale and bias) and token (tokens past
        // M: 0), fp32, from the staged x (a 32-column chunk's values are 64 consecutive
        // bytes in the staging's pair order); groups spread over the threads
        const int G = K >> 6;
        for (int i = threadIdx.x; i < a.M * G; i += kWarps * 32) {
            const int m = i / G, g = i - m * G;
            const uint4 *xp = reinterpret_cast<const uint4 *>(xs + size_t(m) * xrow + size_t(g) * 128);
            float sum = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint4 v = xp[q];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) sum += lo_f32(w[h]) + hi_f32(w[h]);
            }
            xsum[size_t(g) * 16 + m] = sum;
        }
        for (int i = threadIdx.x; i < (16 - a.M) * G; i += kWarps * 32) {
            const int m = a.M + i / G, g = i % G;
            xsum[size_t(g) * 16 + m] = 0.f;
        }
        named_barrier_compute();
    }
    griddep_launch_dependents();
    const int r = lane >> 2, t = lane & 3;
    {
        // Zero-point term of every (group, token): the main loop's MMA chain
        // on the same B fragments with every A element 7/8, so that a row of
        // all-7 codes gives bit-identical D and E. Four groups are kept in
        // flight per warp; lanes of row 0 store.
        const uint32_t a7[4] = {kSevenEighths, kSevenEighths, kSevenEighths, kSevenEighths};
        const int G = kUnpack == 2 ? K >> 5 : 0;
        for (int g0 = warp; g0 < G; g0 += 4 * kWarps) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int g = g0 + u * kWarps;
                if (g < G) {
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        const int m = r + 8 * nb;
                        uint4 xv = make_uint4(0, 0, 0, 0);
                        if (m < a.M)
                            xv = *reinterpret_cast<const uint4 *>(xs + size_t(m) * xrow + size_t(g) * 64 + 16 * t);
                        const float z[4] = {0.f, 0.f, 0.f, 0.f};
                        float e[4];
                        mma16816(e, a7, xv.x, xv.y, z);
                        mma16816(e, a7, xv.z, xv.w, e);
                        if (r == 0) *reinterpret_cast<float2 *>(zp + (g * NB + nb) * 8 + 2 * t) = make_float2(e[0], e[1]);
                    }
                }
            }
        }
    }
    if (kUnpack == 2) named_barrier_compute();
    const uint32_t a7[4] = {kSevenEighths, kSevenEighths, kSevenEighths, kSevenEighths};

    float2 *sp = sscr + warp * kGpw * 8;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < a.tiles; tile += gridDim.x) {
        // add + RMSNorm: this thread's residual value of the tile, fetched
        // now so that its latency hides behind the tile's compute
        float rres = 0.f;
        if (RU == 4 && threadIdx.x < 16 * a.M && tile * 16 + (threadIdx.x & 15) < N)
            rres = f16_bits_to_float(a.resid[size_t(threadIdx.x >> 4) * N + tile * 16 + (threadIdx.x & 15)]);
        float acc[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[nb][j] = 0.f;
        for (int c = 0; c < chunks; ++c, ++it) {
            const int s = it % kStages;
            const uint32_t ph = (it / kStages) & 1;
            if (ok && !mbar_wait(full0 + 8 * s, ph)) ok = false;
            if (ok) {
                const int k0 = c * kKC, gc = min(kKC, K - k0) >> 5;
                const int gpw = (gc + kWarps - 1) / kWarps;
                const int g_lo = warp * gpw, ng = min(gc, g_lo + gpw) - g_lo;
                const uint8_t *st = smem + s * kStageBytes;
                // this warp's scales of the stage, as fp32 pairs 8*(s[r], s[r+8])
                const uint16_t *scl = reinterpret_cast<const uint16_t *>(st + kSegs * kSegBytes);
                if (AFF) {
                    // a scale and a bias per 64 columns (a pair of 32-column chunks; the
                    // warp's share starts on a pair and holds whole pairs): rows of kScaleCols / 2
                    const uint16_t *bia = scl + 16 * (kScaleCols / 2);
                    for (int i = lane; i < (ng >> 1) * 8; i += 32) {
                        const int gi = i >> 3, rp = i & 7, col = (g_lo >> 1) + gi;
                        sp[gi * 8 + rp] = make_float2(f16_bits_to_float(scl[rp * (kScaleCols / 2) + col]),
                                                      f16_bits_to_float(scl[(rp + 8) * (kScaleCols / 2) + col]));
                        sbias[warp * kGpw * 8 + gi * 8 + rp] =
                            make_float2(f16_bits_to_float(bia[rp * (kScaleCols / 2) + col]),
                                        f16_bits_to_float(bia[(rp + 8) * (kScaleCols / 2) + col]));
                    }
                } else {
                    for (int i = lane; i < ng * 8; i += 32) {
                        const int gi = i >> 3, rp = i & 7;
                        const float s0 = f16_bits_to_float(scl[rp * kScaleCols + g_lo + gi]);
                        const float s1 = f16_bits_to_float(scl[(rp + 8) * kScaleCols + g_lo + gi]);
                        const float f = kUnpack == 0 ? 1.f : 8.f;
                        sp[gi * 8 + rp] = make_float2(f * s0, f * s1);
                    }
                }
                __syncwarp();
                const int kg0 = (k0 >> 5) + g_lo;           // global index of the warp's first group
                const uint8_t *xg = xs + size_t(kg0) * 64 + 16 * t;
                const float *zg = zp + size_t(kg0) * NB * 8 + 2 * t;
                const uint8_t *rowr = st + r * 128 + 4 * t;  // row r; row r+8 is 1 KB further
                if constexpr (AFF) {
                    // one 64-column group per trip: the MMA chain sums both chunks' x.q, then
                    // s * sum(x q) + b * sum(x) once per group
                    static_assert(!AFF || 16 % (2 * kWarps) == 0, "a warp's share of 16 or 32 chunks is whole pairs");
                    const float2 *sbw = sbias + warp * kGpw * 8;
                    const float *xsg = xsum + size_t(kg0 >> 1) * 16 + 2 * t;
#pragma unroll(kUnrollG / 2)
                    for (int gp = 0; gp < (ng >> 1); ++gp) {
                        const int gl = g_lo + 2 * gp;        // first chunk of the pair, within the stage
                        const uint8_t *p0 = rowr + (gl >> 3) * kSegBytes + (((gl & 7) ^ r) << 4);
                        const uint8_t *p1 = rowr + ((gl + 1) >> 3) * kSegBytes + ((((gl + 1) & 7) ^ r) << 4);
                        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(p0);
                        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(p0 + 8 * 128);
                        const uint32_t w2 = *reinterpret_cast<const uint32_t *>(p1);
                        const uint32_t w3 = *reinterpret_cast<const uint32_t *>(p1 + 8 * 128);
                        const float2 sc = sp[gp * 8 + r];
                        const float2 bv = sbw[gp * 8 + r];
                        uint32_t pa[4], pb[4], pc[4], pd[4];
                        unpack_word_q_f16x2(w0, pa);
                        unpack_word_q_f16x2(w1, pb);
                        unpack_word_q_f16x2(w2, pc);
                        unpack_word_q_f16x2(w3, pd);
                        const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
                        const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
                        const uint32_t a2[4] = {pc[0], pd[0], pc[1], pd[1]};
                        const uint32_t a3[4] = {pc[2], pd[2], pc[3], pd[3]};
#pragma unroll
                        for (int nb = 0; nb < NB; ++nb) {
                            const int m = r + 8 * nb;
                            uint4 xv = make_uint4(0, 0, 0, 0), xw = make_uint4(0, 0, 0, 0);
                            if (m < a.M) {
                                const uint8_t *xq = xg + size_t(m) * xrow + 128 * gp;
                                xv = *reinterpret_cast<const uint4 *>(xq);
                                xw = *reinterpret_cast<const uint4 *>(xq + 64);
                            }
                            const float z[4] = {0.f, 0.f, 0.f, 0.f};
                            float d[4];
                            mma16816(d, a0, xv.x, xv.y, z);
                            mma16816(d, a1, xv.z, xv.w, d);
                            mma16816(d, a2, xw.x, xw.y, d);
                            mma16816(d, a3, xw.z, xw.w, d);
                            const float2 xs2 = *reinterpret_cast<const float2 *>(xsg + size_t(gp) * 16 + 8 * nb);
                            acc[nb][0] = fmaf(bv.x, xs2.x, fmaf(sc.x, d[0], acc[nb][0]));
                            acc[nb][1] = fmaf(bv.x, xs2.y, fmaf(sc.x, d[1], acc[nb][1]));
                            acc[nb][2] = fmaf(bv.y, xs2.x, fmaf(sc.y, d[2], acc[nb][2]));
                            acc[nb][3] = fmaf(bv.y, xs2.y, fmaf(sc.y, d[3], acc[nb][3]));
                        }
                    }
                } else {
#pragma unroll(kUnrollG)
                for (int gi = 0; gi < ng; ++gi) {
                    const int gl = g_lo + gi;                // group within the stage
                    const uint8_t *p = rowr + (gl >> 3) * kSegBytes + (((gl & 7) ^ r) << 4);
                    const uint32_t w0 = *reinterpret_cast<const uint32_t *>(p);
                    const uint32_t w1 = *reinterpret_cast<const uint32_t *>(p + 8 * 128);
                    const float2 sc = sp[gi * 8 + r];
                    uint32_t pa[4], pb[4];
                    if (kUnpack == 0) {
                        unpack_word_f16x2(w0, pa);
                        unpack_word_f16x2(w1, pb);
                    } else {
                        unpack_word_q8_f16x2(w0, pa);
                        unpack_word_q8_f16x2(w1, pb);
                    }
                    const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
                    const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        const int m = r + 8 * nb;
                        uint4 xv = make_uint4(0, 0, 0, 0);
                        if (m < a.M) xv = *reinterpret_cast<const uint4 *>(xg + size_t(m) * xrow + 64 * gi);
                        const float z[4] = {0.f, 0.f, 0.f, 0.f};
                        float d[4];
                        mma16816(d, a0, xv.x, xv.y, z);
                        mma16816(d, a1, xv.z, xv.w, d);
                        float e[4] = {0.f, 0.f, 0.f, 0.f};
                        if (kUnpack == 1) {
                            mma16816(e, a7, xv.x, xv.y, z);
                            mma16816(e, a7, xv.z, xv.w, e);
                        } else if (kUnpack == 2) {
                            const float2 ev = *reinterpret_cast<const float2 *>(zg + (gi * NB + nb) * 8);
                            e[0] = e[2] = ev.x;
                            e[1] = e[3] = ev.y;
                        }
                        acc[nb][0] = fmaf(sc.x, d[0] - e[0], acc[nb][0]);
                        acc[nb][1] = fmaf(sc.x, d[1] - e[1], acc[nb][1]);
                        acc[nb][2] = fmaf(sc.y, d[2] - e[2], acc[nb][2]);
                        acc[nb][3] = fmaf(sc.y, d[3] - e[3], acc[nb][3]);
                    }
                }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
        }
        // cross-warp reduction of the tile: red[w][nb][row][col]
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            float *rw = red + ((warp * NB + nb) * 16) * 8;
            rw[r * 8 + 2 * t] = acc[nb][0];
            rw[r * 8 + 2 * t + 1] = acc[nb][1];
            rw[(r + 8) * 8 + 2 * t] = acc[nb][2];
            rw[(r + 8) * 8 + 2 * t + 1] = acc[nb][3];
        }
        named_barrier_compute();
        const int row0 = tile * 16;
        if (RU == 1) {
            for (int o = threadIdx.x; o < 16 * a.M; o += kWarps * 32) {
                const int m = o >> 4, i = o & 15;
                if (row0 + i < N) {
                    float v = 0.f;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) v += red[((w * NB + (m >> 3)) * 16 + i) * 8 + (m & 7)];
                    a.y[size_t(m) * a.y_stride + row0 + i] = float_to_f16_bits(v);
                }
            }
        } else if (RU == 3) {
            // fp32 logits, and the tile's largest logit of every token folded
            // into the token's argmax key: the 16 rows of a token are 16
            // consecutive lanes of one warp (16 * M <= 256 outputs, one pass)
            const int o = threadIdx.x, m = o >> 4, i = o & 15;
            unsigned long long key = 0ull;
            if (o < 16 * a.M && row0 + i < N) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) v += red[((w * NB + (m >> 3)) * 16 + i) * 8 + (m & 7)];
                if (a.y32) a.y32[size_t(m) * a.y_stride + row0 + i] = v;
                key = argmax_key(v, row0 + i);
            }
            if (o < ((16 * a.M + 31) & ~31)) {
#pragma unroll
                for (int d = 8; d >= 1; d >>= 1) {
                    const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, d);
                    key = other > key ? other : key;
                }
                if (i == 0 && o < 16 * a.M) atomicMax(a.amax + m, key);
            }
        } else if (RU == 5) {
            // QKV + RoPE + KV append: tile row i < 8 is pair index i0 + i of head
            // hb (first half), row i + 8 its partner i0 + i + D/2; Q and K heads
            // rotated, Q to q_out, K and V to the cache rows of the token's slot
            const int tpp = a.D >> 4, hb = tile / tpp, i0 = (tile - hb * tpp) * 8, half = a.D >> 1;
            const bool rot = hb < a.H + a.Hkv;
            for (int o = threadIdx.x; o < 8 * a.M; o += kWarps * 32) {
                const int m = o >> 3, i = o & 7;
                float va = 0.f, vb = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    va += red[((w * NB + (m >> 3)) * 16 + i) * 8 + (m & 7)];
                    vb += red[((w * NB + (m >> 3)) * 16 + i + 8) * 8 + (m & 7)];
                }
                float oa = va, ob = vb;
                if constexpr (RU == 5)
                    if (rot) rope_rotate(s_pos[m], a.freq[i0 + i], va, vb, &oa, &ob);
                uint16_t *dst;
                if (hb < a.H) {
                    dst = a.q_out + size_t(m) * a.H * a.D + size_t(hb) * a.D;
                } else {
                    const int sl = s_slot[m];
                    if (sl < 0 || sl >= a.n_slots) {
                        if (a.dev_status) atomicOr(reinterpret_cast<unsigned *>(a.dev_status), ZQ4_DEV_BAD_SLOT);
                        continue;
                    }
                    dst = (rot ? a.k_cache : a.v_cache) + size_t(sl) * a.Hkv * a.D +
                          size_t(rot ? hb - a.H : hb - a.H - a.Hkv) * a.D;
                }
                dst[i0 + i] = float_to_f16_bits(oa);
                dst[i0 + i + half] = float_to_f16_bits(ob);
            }
        } else if (RU == 4) {
            // r = resid + x W^T: the new residual (f16 and fp32), and the
            // CTA's running sum of r^2 per token (rows in order, tiles in order)
            if (threadIdx.x < 16 * a.M) {                    // 16 M <= 256 outputs: one per thread
                const int o = threadIdx.x, m = o >> 4, i = o & 15;
                float v = 0.f;
                if (row0 + i < N) {
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) v += red[((w * NB + (m >> 3)) * 16 + i) * 8 + (m & 7)];
                    const size_t at = size_t(m) * N + row0 + i;
                    v += rres;
                    a.y[at] = float_to_f16_bits(v);
                    a.r32[at] = v;
                }
                s_sq[m][i] = v * v;
            }
            named_barrier_compute();
            if (threadIdx.x < a.M) {
                float t = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) t += s_sq[threadIdx.x][i];
                s_ss[threadIdx.x] += t;
            }
        } else {
            for (int o = threadIdx.x; o < 8 * a.M; o += kWarps * 32) {
                const int m = o >> 3, j = o & 7;
                if (row0 + 2 * j + 1 < N) {
                    float gv = 0.f, uv = 0.f;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) {
                        const float *rw = red + ((w * NB + (m >> 3)) * 16) * 8 + (m & 7);
                        gv += rw[(2 * j) * 8];
                        uv += rw[(2 * j + 1) * 8];
                    }
                    a.y[size_t(m) * a.y_stride + (row0 >> 1) + j] = float_to_f16_bits(silu_f32(gv) * uv);
                }
            }
        }
        named_barrier_compute();
    }
    if (!ok && lane == 0) atomicOr(&g_device_error, ZQ4_DEVERR_WAIT_TIMEOUT);
    if (RU == 4) {
        // The last CTA to finish adds the CTAs' sums of squares (CTA order,
        // in a fixed pattern: lane l takes CTAs l, l + 32, ..) and writes
        // every token's normalised rows; it leaves the counter at zero.
        __shared__ int s_last;
        __shared__ float s_inv[16];
        named_barrier_compute();
        if (threadIdx.x < a.M) a.part[size_t(blockIdx.x) * 16 + threadIdx.x] = s_ss[threadIdx.x];
        named_barrier_compute();
        if (threadIdx.x == 0) {
            __threadfence();
            s_last = atomicAdd(a.counter, 1u) == gridDim.x - 1;
        }
        named_barrier_compute();
        if (s_last) {
            __threadfence();
            // (grid <= 32 kPartLoads CTAs: the launcher caps it; all loads in flight at once)
            for (int m = warp; m < a.M; m += kWarps) {
                float v[kPartLoads];
#pragma unroll
                for (int j = 0; j < kPartLoads; ++j) {
                    const int c = lane + 32 * j;
                    v[j] = c < int(gridDim.x) ? __ldcg(a.part + size_t(c) * 16 + m) : 0.f;
                }
                float t = 0.f;
#pragma unroll
                for (int j = 0; j < kPartLoads; ++j) t += v[j];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                if (lane == 0) s_inv[m] = 1.0f / sqrtf(t / float(N) + a.eps);
            }
            named_barrier_compute();
            // every token's rows: four at a time where N allows (16-byte fp32
            // loads), the loads of a pass issued before its stores
            for (int m = 0; m < a.M; ++m) {
                const float inv = s_inv[m];
                const float *rr = a.r32 + size_t(m) * N;
                uint16_t *oo = a.out + size_t(m) * N;
                // (8-byte gamma and out rows: N % 4 == 0 keeps every row at the base's alignment)
                if ((N & 3) == 0 && ((reinterpret_cast<uintptr_t>(a.gamma) | reinterpret_cast<uintptr_t>(a.out)) & 7) == 0) {
                    const int n4 = N >> 2;
                    for (int q0 = threadIdx.x; q0 < n4; q0 += 4 * kWarps * 32) {
                        float4 rv[4];
                        uint2 gv[4];
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            const int q = q0 + b * kWarps * 32;
                            if (q < n4) {
                                rv[b] = __ldcg(reinterpret_cast<const float4 *>(rr) + q);
                                gv[b] = *reinterpret_cast<const uint2 *>(a.gamma + 4 * q);
                            }
                        }
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            const int q = q0 + b * kWarps * 32;
                            if (q < n4) {
                                const uint32_t lo = uint32_t(float_to_f16_bits(rv[b].x * inv * lo_f32(gv[b].x))) |
                                                    (uint32_t(float_to_f16_bits(rv[b].y * inv * hi_f32(gv[b].x))) << 16);
                                const uint32_t hi = uint32_t(float_to_f16_bits(rv[b].z * inv * lo_f32(gv[b].y))) |
                                                    (uint32_t(float_to_f16_bits(rv[b].w * inv * hi_f32(gv[b].y))) << 16);
                                *reinterpret_cast<uint2 *>(oo + 4 * q) = make_uint2(lo, hi);
                            }
                        }
                    }
                } else {
                    for (int n = threadIdx.x; n < N; n += kWarps * 32)
                        oo[n] = float_to_f16_bits(__ldcg(rr + n) * inv * f16_bits_to_float(a.gamma[n]));
                }
            }
            if (threadIdx.x == 0) *a.counter = 0u;
        }
    }
    if (RU == 3) {
        // The last CTA to finish turns the keys into rows and logits and
        // leaves keys and counter at zero for the next call (every CTA
        // counts itself, also after a timeout, so the count stays exact).
        __shared__ int s_last;
        named_barrier_compute();
        if (threadIdx.x == 0) {
            __threadfence();
            s_last = atomicAdd(a.done, 1ull) == gridDim.x - 1;
        }
        named_barrier_compute();
        if (s_last) {
            __threadfence();
            for (int m = threadIdx.x; m < a.M; m += kWarps * 32) {
                const unsigned long long key = __ldcg(a.amax + m);
                const unsigned ord = unsigned(key >> 32);
                a.idx[m] = int32_t(~unsigned(key & 0xffffffffu));
                if (a.maxval) a.maxval[m] = __uint_as_float((ord & 0x80000000u) ? (ord & 0x7fffffffu) : ~ord);
                a.amax[m] = 0ull;
            }
            if (threadIdx.x == 0) *a.done = 0ull;
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
    if (!f) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

// Tensor maps of one q4f16_1 matrix: codes as uint32 [N][K/8] read in boxes
// of [16 rows x 32 words] with the 128-byte swizzle, scales as uint16
// [N][K/32] in boxes of [16 rows x kScaleCols].
cudaError_t make_maps(const uint32_t *wq, const uint16_t *scales, int N, int K, CUtensorMap *codes,
                      CUtensorMap *sc)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint32_t estr[2] = {1, 1};
    {
        const cuuint64_t dim[2] = {cuuint64_t(K / 8), cuuint64_t(N)};
        const cuuint64_t stride[1] = {cuuint64_t(K / 2)};
        const cuuint32_t box[2] = {32, 16};
        if (enc(codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t *>(wq), dim, stride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dim[2] = {cuuint64_t(K / 32), cuuint64_t(N)};
        const cuuint64_t stride[1] = {cuuint64_t(K / 16)};
        const cuuint32_t box[2] = {cuuint32_t(kScaleCols), 16};
        if (enc(sc, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t *>(scales), dim, stride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

template <int NB, int RU, bool AFF = false>
cudaError_t launch_t(const CUtensorMap &mc, const CUtensorMap &ms, const TcArgsFor<RU, AFF> &a, cudaStream_t s)
{
    static int smem_set[kMaxDevices] = {};
    auto kern = k_decode_tc<NB, RU, AFF>;
    const size_t smem = smem_bytes<NB>(a.M, a.K) + (AFF ? aff_bytes(a.K) : 0);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(kern), smem, smem_set);
    if (e != cudaSuccess) return e;
    // CTAs per SM by shared memory (1 KB per CTA is reserved), at most ZQ4_TC_OCC.
    const int occ = std::max(1, std::min(ZQ4_TC_OCC, int(smem_per_sm() / (smem + 1024))));
    int grid = std::max(1, std::min(a.tiles, occ * sm_count()));
    if (RU == 4) grid = std::min(grid, 32 * kPartLoads);   // the last CTA reads one sum per CTA
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, mc, ms, a);
}

}  // namespace tc

bool decode_tc_supported(int M, int K)
{
    // Scale rows must be 16-byte multiples for the tensor map (K % 256 == 0);
    // activations are staged whole, in blocks of up to 8 rows.
    return K % 256 == 0 && tc::smem_bytes<1>(std::min(M, 8), K) <= 220 * 1024 && tc::encode_fn() != nullptr;
}

cudaError_t launch_decode_tc(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, uint16_t *y,
                             int M, int N, int K, bool gate_up, cudaStream_t s)
{
    CUtensorMap mc, ms;
    cudaError_t e = tc::make_maps(wq, scales, N, K, &mc, &ms);
    if (e != cudaSuccess) return e;
    const int out_cols = gate_up ? N / 2 : N;
    TcArgs a;
    a.wq = wq;
    a.scales = scales;
    a.N = N;
    a.K = K;
    a.tiles = (N + 15) / 16;
    a.y_stride = out_cols;
    const bool fit16 = tc::smem_bytes<2>(16, K) <= 220 * 1024;
    for (int m0 = 0; m0 < M;) {
        const int rem = M - m0;
        const int nb = (rem > 8 && fit16) ? 2 : 1;
        const int mt = std::min(rem, 8 * nb);
        a.x = x + size_t(m0) * K;
        a.y = y + size_t(m0) * out_cols;
        a.M = mt;
        if (nb == 2)
            e = gate_up ? tc::launch_t<2, 2>(mc, ms, a, s) : tc::launch_t<2, 1>(mc, ms, a, s);
        else
            e = gate_up ? tc::launch_t<1, 2>(mc, ms, a, s) : tc::launch_t<1, 1>(mc, ms, a, s);
        if (e != cudaSuccess) return e;
        m0 += mt;
    }
    return cudaSuccess;
}

cudaError_t launch_decode_tc_argmax(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, float *y32,
                                    int32_t *idx, float *maxval, unsigned long long *work, int M, int N, int K,
                                    cudaStream_t s)
{
    CUtensorMap mc, ms;
    cudaError_t e = tc::make_maps(wq, scales, N, K, &mc, &ms);
    if (e != cudaSuccess) return e;
    TcArgs a;
    a.wq = wq;
    a.scales = scales;
    a.y = nullptr;
    a.N = N;
    a.K = K;
    a.tiles = (N + 15) / 16;
    a.y_stride = N;
    const bool fit16 = tc::smem_bytes<2>(16, K) <= 220 * 1024;
    for (int m0 = 0, blk = 0; m0 < M; ++blk) {
        const int rem = M - m0;
        const int nb = (rem > 8 && fit16) ? 2 : 1;
        const int mt = std::min(rem, 8 * nb);
        a.x = x + size_t(m0) * K;
        a.y32 = y32 ? y32 + size_t(m0) * N : nullptr;
        a.amax = work + m0;
        a.done = work + M + blk;                 // one counter per block of tokens (at most 8 blocks)
        a.idx = idx + m0;
        a.maxval = maxval ? maxval + m0 : nullptr;
        a.M = mt;
        e = nb == 2 ? tc::launch_t<2, 3>(mc, ms, a, s) : tc::launch_t<1, 3>(mc, ms, a, s);
        if (e != cudaSuccess) return e;
        m0 += mt;
    }
    return cudaSuccess;
}

cudaError_t launch_decode_tc_addnorm(const uint32_t *wq, const uint16_t *scales, const uint16_t *x,
                                     const uint16_t *resid, const uint16_t *gamma, float eps, uint16_t *res_out,
                                     uint16_t *out, void *work, int M, int N, int K, cudaStream_t s)
{
    CUtensorMap mc, ms;
    cudaError_t e = tc::make_maps(wq, scales, N, K, &mc, &ms);
    if (e != cudaSuccess) return e;
    TcArgs a;
    memset(&a, 0, sizeof(a));
    a.wq = wq;
    a.scales = scales;
    a.N = N;
    a.K = K;
    a.tiles = (N + 15) / 16;
    a.y_stride = N;
    a.gamma = gamma;
    a.eps = eps;
    a.counter = static_cast<unsigned *>(work);
    float *r32 = reinterpret_cast<float *>(static_cast<uint8_t *>(work) + 16);
    a.part = r32 + size_t(M) * N;
    const bool fit16 = tc::smem_bytes<2>(16, K) <= 220 * 1024;
    for (int m0 = 0; m0 < M;) {
        const int rem = M - m0;
        const int nb = (rem > 8 && fit16) ? 2 : 1;
        const int mt = std::min(rem, 8 * nb);
        const size_t o = size_t(m0) * N;
        a.x = x + size_t(m0) * K;
        a.resid = resid + o;
        a.y = res_out + o;
        a.out = out + o;
        a.r32 = r32 + o;
        a.M = mt;
        e = nb == 2 ? tc::launch_t<2, 4>(mc, ms, a, s) : tc::launch_t<1, 4>(mc, ms, a, s);
        if (e != cudaSuccess) return e;
        m0 += mt;
    }
    return cudaSuccess;
}

bool decode_tc_affine_supported(int M, int K)
{
    // scale rows of K/64 f16 must be 16-byte multiples for their tensor maps
    return K % 512 == 0 && decode_tc_supported(std::min(M, 16), K) &&
           tc::smem_bytes<2>(std::min(M, 16), K) + tc::aff_bytes(K) <= 220 * 1024;
}

cudaError_t launch_decode_tc_affine(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                                    const uint16_t *x, uint16_t *y, int M, int N, int K, bool gate_up, cudaStream_t s)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tc::encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap mc, ms;
    cudaError_t e = tc::make_maps(wq, scales, N, K, &mc, &ms);    // codes (the scales map is replaced)
    if (e != cudaSuccess) return e;
    tc::TcAffArgs a;
    memset(&a, 0, sizeof(a));
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dim[2] = {cuuint64_t(K / 64), cuuint64_t(N)};
    const cuuint64_t stride[1] = {cuuint64_t(K / 32)};
    const cuuint32_t box[2] = {cuuint32_t(tc::kScaleCols / 2), 16};
    if (enc(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t *>(scales), dim, stride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&a.tm_bias, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t *>(biases), dim, stride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int out_cols = gate_up ? N / 2 : N;
    a.wq = wq;
    a.scales = scales;
    a.N = N;
    a.K = K;
    a.tiles = (N + 15) / 16;
    a.y_stride = out_cols;
    for (int m0 = 0; m0 < M;) {
        const int rem = M - m0;
        const int nb = rem > 8 ? 2 : 1;
        const int mt = std::min(rem, 8 * nb);
        a.x = x + size_t(m0) * K;
        a.y = y + size_t(m0) * out_cols;
        a.M = mt;
        if (nb == 2)
            e = gate_up ? tc::launch_t<2, 2, true>(mc, ms, a, s) : tc::launch_t<2, 1, true>(mc, ms, a, s);
        else
            e = gate_up ? tc::launch_t<1, 2, true>(mc, ms, a, s) : tc::launch_t<1, 1, true>(mc, ms, a, s);
        if (e != cudaSuccess) return e;
        m0 += mt;
    }
    return cudaSuccess;
}

bool decode_tc_rope_supported(int M, int K, int D)
{
    return decode_tc_supported(std::min(M, 16), K) && D > 0 && D % 16 == 0 && D / 2 <= 256;
}

cudaError_t launch_decode_tc_rope(const QkvArgs &q, cudaStream_t s)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tc::encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int K = q.K, D = q.D, heads = q.H + 2 * q.Hkv;
    // W viewed as [heads][2 halves][D/2 rows][K]: one box = pair rows i0..i0+7 of both halves
    CUtensorMap mc, ms;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    {
        const cuuint64_t dim[4] = {cuuint64_t(K / 8), cuuint64_t(D / 2), 2, cuuint64_t(heads)};
        const cuuint64_t stride[3] = {cuuint64_t(K / 2), cuuint64_t(D / 2) * (K / 2), cuuint64_t(D) * (K / 2)};
        const cuuint32_t box[4] = {32, 8, 2, 1};
        if (enc(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<uint32_t *>(q.wq), dim, stride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dim[4] = {cuuint64_t(K / 32), cuuint64_t(D / 2), 2, cuuint64_t(heads)};
        const cuuint64_t stride[3] = {cuuint64_t(K / 16), cuuint64_t(D / 2) * (K / 16), cuuint64_t(D) * (K / 16)};
        const cuuint32_t box[4] = {cuuint32_t(tc::kScaleCols), 8, 2, 1};
        if (enc(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<uint16_t *>(q.scales), dim, stride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    tc::TcRopeArgs a;
    memset(&a, 0, sizeof(a));
    for (int i = 0; i < D / 2; ++i) a.freq[i] = std::pow(q.base, -2.0 * double(i) / double(D));
    a.wq = q.wq;
    a.scales = q.scales;
    a.N = heads * D;
    a.K = K;
    a.tiles = heads * (D / 16);
    a.k_cache = q.k_cache;
    a.v_cache = q.v_cache;
    a.dev_status = q.dev_status;
    a.base = q.base;
    a.H = q.H;
    a.Hkv = q.Hkv;
    a.D = D;
    a.n_slots = q.n_slots;
    const bool fit16 = tc::smem_bytes<2>(16, K) <= 220 * 1024;
    cudaError_t e = cudaSuccess;
    for (int m0 = 0; m0 < q.M;) {
        const int rem = q.M - m0;
        const int nb = (rem > 8 && fit16) ? 2 : 1;
        const int mt = std::min(rem, 8 * nb);
        a.x = q.x + size_t(m0) * K;
        a.pos = q.pos + m0;
        a.slot = q.slot + m0;
        a.q_out = q.q_out + size_t(m0) * q.H * D;
        a.M = mt;
        e = nb == 2 ? tc::launch_t<2, 5>(mc, ms, a, s) : tc::launch_t<1, 5>(mc, ms, a, s);
        if (e != cudaSuccess) return e;
        m0 += mt;
    }
    return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() { return tc::encode_fn(); }

cudaError_t read_device_error(unsigned *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_device_error, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned));
}

}  // namespace zq4
