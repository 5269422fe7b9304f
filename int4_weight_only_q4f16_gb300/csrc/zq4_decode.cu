// zq4_decode.cu -- memory-bound q4f16_1 GEMV kernels for small M (decode),
// the gate_up + SiLU*mul epilogue, the MoE expert-gather variants, and the
// dequantize / layout helpers.
//
// What they compute: "Zero TVM Documentation", section "WGSL Kernel Roles",
// cards 5 ("int4 Matmul") and 6 ("Fused FFN"); "RESEARCH.md" (Zero-TVM),
// section "Matmul Shader Analysis"; "Zero-TVM benchmarks" (BENCH.md), section
// "MoE chunked prefill". How they compute it is a GB300 design of its own:
//
//  * one 16-byte load = the 4 words of one 32-weight scale group, so a warp
//    reads 512 contiguous bytes of a row per load instruction, never
//    allocating in L1;
//  * the activations x are staged once per CTA in shared memory, with each
//    word's 8 values stored as the pairs (0,4),(1,5),(2,6),(3,7) that the
//    unpack produces, and the four 16-byte chunks of a group rotated by
//    (group/2) mod 4 so that a quarter-warp's 16-byte reads hit 8 distinct
//    bank groups;
//  * codes become exact f16 (q - 7) with one LOP3 and one f16x2 op per two
//    weights; products are f16 x f16 -> fp32 fused multiply-adds, and each
//    group's sum is scaled once by its fp32 scale;
//  * lanes of a row (8, 16 or 32) reduce with warp shuffles;
//  * before waiting on the previous kernel (programmatic dependent launch)
//    each CTA asks L2 to prefetch the weight rows it owns: weights never
//    depend on the previous kernel, so the stream of weights continues
//    across kernel boundaries.
//
// The dense kernel also reads the MLX affine format (AFF): value = scale *
// code + bias, one scale and one bias per 64 weights ("Zero TVM
// Documentation", section "Qwen3.6-35B-A3B MoE"; "Zero-TVM benchmarks",
// "Affine wide loads"). Per 32-weight chunk it adds
// b * sum(x) + s * sum(x * q): the codes become exact f16 q (no zero point),
// the products are exact, and sum(x) of every chunk is taken once per CTA
// when x is staged.
#include <cuda_fp16.h>

#include <algorithm>

#include "zq4_common.cuh"
#include "zq4_internal.h"
#include "zq4_rope.cuh"

namespace zq4 {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;          // groups in flight per lane
constexpr int kMoeSlotChunk = 8;    // expert slots loaded together in DOWN_COMBINE

// ---------------------------------------------------------------------------
// Activation staging
// ---------------------------------------------------------------------------

// Shared-memory byte offset of chunk c (word c of the group, 0..3) of group g.
__device__ __forceinline__ uint32_t xs_offset(int g, int c)
{
    return uint32_t(g) * 64u + 16u * uint32_t(c ^ ((g >> 1) & 3));
}

// Stage rows [0, rows) of src (row stride K elements) into xs (row stride
// 2K bytes) in the paired/rotated layout; rows [rows, rows_alloc) are zeroed.
__device__ __forceinline__ void stage_rows(uint8_t *xs, const uint16_t *src, int rows,
                                           int rows_alloc, int K)
{
    const int words = K >> 3;                 // 8 values per chunk
    const int total = rows_alloc * words;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        int r = i / words, cw = i - r * words;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < rows) v = *reinterpret_cast<const uint4 *>(src + size_t(r) * K + size_t(cw) * 8);
        uint4 o;
        o.x = __byte_perm(v.x, v.z, 0x5410);  // (x0, x4)
        o.y = __byte_perm(v.x, v.z, 0x7632);  // (x1, x5)
        o.z = __byte_perm(v.y, v.w, 0x5410);  // (x2, x6)
        o.w = __byte_perm(v.y, v.w, 0x7632);  // (x3, x7)
        int g = cw >> 2, c = cw & 3;
        *reinterpret_cast<uint4 *>(xs + size_t(r) * K * 2 + xs_offset(g, c)) = o;
    }
}

// Codes of one word to exact f16 q (no zero point), in the pair order of
// unpack_word_f16x2: 1024 + q (or 1024 + 16 q) minus the magic.
__device__ __forceinline__ void unpack_word_f16x2_q(uint32_t w, uint32_t p[4])
{
    const uint32_t kMagic = 0x64006400u;       // (1024, 1024)
    const uint32_t kSixteenth = 0x2C002C00u;   // (1/16, 1/16)
    const uint32_t kNeg64 = 0xD400D400u;       // (-64, -64): 1024/16
    uint32_t w8 = w >> 8;
    p[0] = hsub2(and_or<0x000F000Fu>(w, kMagic), kMagic);                  // elements 0, 4
    p[1] = hfma2(and_or<0x00F000F0u>(w, kMagic), kSixteenth, kNeg64);      // elements 1, 5
    p[2] = hsub2(and_or<0x000F000Fu>(w8, kMagic), kMagic);                 // elements 2, 6
    p[3] = hfma2(and_or<0x00F000F0u>(w8, kMagic), kSixteenth, kNeg64);     // elements 3, 7
}

// sum(x) of every 32-weight chunk of rows [0, rows) of src (fp32, ascending
// k), rows [rows, rows_alloc) zero: xsum[r * (K/32) + g].
__device__ __forceinline__ void chunk_sums(float *xsum, const uint16_t *src, int rows, int rows_alloc, int K)
{
    const int G = K >> 5, total = rows_alloc * G;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int r = i / G, g = i - r * G;
        float acc = 0.f;
        if (r < rows) {
            const uint16_t *p = src + size_t(r) * K + size_t(g) * 32;
            for (int k = 0; k < 32; ++k) acc += f16_bits_to_float(p[k]);
        }
        xsum[i] = acc;
    }
}

// ---------------------------------------------------------------------------
// One 32-weight group of one row against MT staged activation rows.
// part[m] += s * sum_{k in group} x[m,k] * (q[k] - 7)
// ---------------------------------------------------------------------------
// AFF: part[m] += b * xsum[m][g] + s * sum_{k in group} x[m,k] * q[k].
template <int MT, bool AFF>
__device__ __forceinline__ void group_dot(const uint4 wv, float s, float b, uint32_t xs_base, int g,
                                          uint32_t row_bytes, const float *xsum, int G, float (&part)[MT])
{
    uint32_t p[4][4];
    if (AFF) {
        unpack_word_f16x2_q(wv.x, p[0]);
        unpack_word_f16x2_q(wv.y, p[1]);
        unpack_word_f16x2_q(wv.z, p[2]);
        unpack_word_f16x2_q(wv.w, p[3]);
    } else {
        unpack_word_f16x2(wv.x, p[0]);
        unpack_word_f16x2(wv.y, p[1]);
        unpack_word_f16x2(wv.z, p[2]);
        unpack_word_f16x2(wv.w, p[3]);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint4 xv = lds_v4(xs_base + uint32_t(m) * row_bytes + xs_offset(g, c));
            fma2_f16_f32(p[c][0], xv.x, a0, a1);
            fma2_f16_f32(p[c][1], xv.y, a0, a1);
            fma2_f16_f32(p[c][2], xv.z, a0, a1);
            fma2_f16_f32(p[c][3], xv.w, a0, a1);
        }
        if (AFF) part[m] = fmaf(b, xsum[m * G + g], part[m]);
        part[m] = fmaf(s, a0 + a1, part[m]);
    }
}

// Sum of v over the LPR lanes of a row segment (all lanes end with the sum).
template <int LPR>
__device__ __forceinline__ float segment_sum(float v, unsigned mask)
{
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(mask, v, o, LPR);
    return v;
}

template <int LPR>
__device__ __forceinline__ unsigned segment_mask()
{
    if (LPR == 32) return 0xFFFFFFFFu;
    unsigned lane = threadIdx.x & 31;
    return ((1u << (LPR & 31)) - 1u) << (lane & ~unsigned(LPR - 1));
}

// Accumulate RU consecutive rows (starting at row0) of a matrix against MT
// staged activation rows: part[r][m] holds this lane's partial sums.
// AFF: scales and biases [rows][K/64]; xsum = the staged chunk sums of x.
// The RU rows are row0, row0 + row_step, ..
template <int MT, int LPR, int RU, bool AFF>
__device__ __forceinline__ void rows_dot(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases, int K,
                                         int row0, uint32_t xs_base, const float *xsum, int lane,
                                         float (&part)[RU][MT], int row_step = 1)
{
    const int G = K >> 5, KW = K >> 3, GS = AFF ? K >> 6 : G;
    const uint32_t row_bytes = uint32_t(K) * 2;
    const uint32_t *wrow[RU];
    const uint16_t *srow[RU];
    const uint16_t *brow[RU];
#pragma unroll
    for (int r = 0; r < RU; ++r) {
        const size_t row = size_t(row0) + size_t(r) * row_step;
        wrow[r] = wq + row * KW;
        srow[r] = scales + row * GS;
        brow[r] = AFF ? biases + row * GS : nullptr;
#pragma unroll
        for (int m = 0; m < MT; ++m) part[r][m] = 0.f;
    }
    for (int g0 = lane; g0 < G; g0 += kUnroll * LPR) {
        uint4 wv[RU][kUnroll];
        uint16_t sv[RU][kUnroll], bv[RU][kUnroll];
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            int g = g0 + i * LPR;
#pragma unroll
            for (int r = 0; r < RU; ++r) {
                if (g < G) {
                    wv[r][i] = ldg_stream_v4(wrow[r] + 4 * g);
                    sv[r][i] = ldg_u16(srow[r] + (AFF ? g >> 1 : g));
                    bv[r][i] = AFF ? ldg_u16(brow[r] + (g >> 1)) : uint16_t(0);
                } else {
                    wv[r][i] = make_uint4(0, 0, 0, 0);
                    sv[r][i] = 0;
                    bv[r][i] = 0;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            int g = g0 + i * LPR;
            if (g < G) {
#pragma unroll
                for (int r = 0; r < RU; ++r)
                    group_dot<MT, AFF>(wv[r][i], f16_bits_to_float(sv[r][i]), f16_bits_to_float(bv[r][i]), xs_base,
                                       g, row_bytes, xsum, G, part[r]);
            }
        }
    }
}

// L2 prefetch of rows [row_lo, row_hi) of a q4f16_1 matrix by warp 0.
// (gs = scales per row: K/32, or K/64 for the affine format, whose biases
// are prefetched too when given)
__device__ __forceinline__ void prefetch_rows(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                                              int K, int gs, size_t row_lo, size_t row_hi)
{
    if (threadIdx.x < 32) {
        const size_t KW = size_t(K) >> 3, G = size_t(gs);
        prefetch_l2_range(wq + row_lo * KW, wq + row_hi * KW, threadIdx.x, 32);
        prefetch_l2_range(scales + row_lo * G, scales + row_hi * G, threadIdx.x, 32);
        if (biases) prefetch_l2_range(biases + row_lo * G, biases + row_hi * G, threadIdx.x, 32);
    }
}

// ---------------------------------------------------------------------------
// Dense GEMV (RU = 1) and gate_up + SiLU*mul (RU = 2, interleaved rows).
// A "unit" is RU consecutive rows; CTA b owns units [b*upc, (b+1)*upc).
// ---------------------------------------------------------------------------
// AFF: the MLX affine format (a.biases; scales and biases per 64 weights).
template <int MT, int LPR, int RU, bool AFF>
__global__ void __launch_bounds__(kThreads) k_dense(DenseArgs a)
{
    extern __shared__ __align__(16) uint8_t xs[];
    float *xsum = reinterpret_cast<float *>(xs + size_t(MT) * a.K * 2);   // AFF: [MT][K/32]
    const int u0 = blockIdx.x * a.units_per_cta;
    const int u1 = min(u0 + a.units_per_cta, a.units);
    prefetch_rows(a.wq, a.scales, AFF ? a.biases : nullptr, a.K, AFF ? a.K >> 6 : a.K >> 5, size_t(u0) * RU,
                  size_t(u1) * RU);
    griddep_wait();
    stage_rows(xs, a.x, a.M, MT, a.K);
    if (AFF) chunk_sums(xsum, a.x, a.M, MT, a.K);
    __syncthreads();
    griddep_launch_dependents();

    const int sub = threadIdx.x / LPR, lane = threadIdx.x % LPR;
    const unsigned mask = segment_mask<LPR>();
    const uint32_t xs_base = smem_addr(xs);
    for (int u = u0 + sub; u < u1; u += kThreads / LPR) {
        float part[RU][MT];
        rows_dot<MT, LPR, RU, AFF>(a.wq, a.scales, a.biases, a.K, u * RU, xs_base, xsum, lane, part);
#pragma unroll
        for (int r = 0; r < RU; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) part[r][m] = segment_sum<LPR>(part[r][m], mask);
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < a.M) {
                    float v = (RU == 1) ? part[0][m] : silu_f32(part[0][m]) * part[RU - 1][m];
                    a.y[size_t(m) * a.y_stride + u] = float_to_f16_bits(v);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// GEMV + residual add + RMSNorm ("Zero TVM Documentation", card 7 "Fused
// Add + RMSNorm", folded into the matmul that produces its input as a tail
// reduction): every CTA writes r = resid + x W^T for its rows (fp32 to the
// scratch, f16 as the new residual); the last CTA to finish (a counter)
// reduces sum(r^2) of each token in a fixed order, and writes
// f16(r * (1 / sqrt(mean + eps)) * gamma) for every row, then resets the
// counter. Deterministic: no floating-point atomics.
// ---------------------------------------------------------------------------
template <int MT, int LPR>
__global__ void __launch_bounds__(kThreads) k_dense_rms(RmsArgs a)
{
    extern __shared__ __align__(16) uint8_t xs[];
    __shared__ float s_red[kThreads / 32];
    __shared__ float s_inv[MT];
    __shared__ int s_last;
    const int u0 = blockIdx.x * a.units_per_cta;
    const int u1 = min(u0 + a.units_per_cta, a.N);
    prefetch_rows(a.wq, a.scales, nullptr, a.K, a.K >> 5, size_t(u0), size_t(u1));
    griddep_wait();
    stage_rows(xs, a.x, a.M, MT, a.K);
    __syncthreads();
    griddep_launch_dependents();

    const int sub = threadIdx.x / LPR, lane = threadIdx.x % LPR;
    const unsigned mask = segment_mask<LPR>();
    const uint32_t xs_base = smem_addr(xs);
    for (int u = u0 + sub; u < u1; u += kThreads / LPR) {
        float part[1][MT];
        rows_dot<MT, LPR, 1, false>(a.wq, a.scales, nullptr, a.K, u, xs_base, nullptr, lane, part);
#pragma unroll
        for (int m = 0; m < MT; ++m) part[0][m] = segment_sum<LPR>(part[0][m], mask);
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < a.M) {
                    const size_t o = size_t(m) * a.N + u;
                    const float v = part[0][m] + f16_bits_to_float(a.resid[o]);
                    a.res_out[o] = float_to_f16_bits(v);
                    a.r32[o] = v;
                }
            }
        }
    }
    // the last CTA normalises every row of every token
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(a.counter, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int warp = threadIdx.x >> 5, wl = threadIdx.x & 31;
    for (int m = 0; m < a.M; ++m) {
        float acc = 0.f;
        for (int n = threadIdx.x; n < a.N; n += kThreads) {
            const float v = __ldcg(a.r32 + size_t(m) * a.N + n);
            acc = fmaf(v, v, acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (wl == 0) s_red[warp] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            float t = 0.f;
            for (int w = 0; w < kThreads / 32; ++w) t += s_red[w];
            s_inv[m] = 1.0f / sqrtf(t / float(a.N) + a.eps);
        }
        __syncthreads();
    }
    const int total = a.M * a.N;
    for (int i = threadIdx.x; i < total; i += kThreads) {
        const int m = i / a.N, n = i - m * a.N;
        a.out[i] = float_to_f16_bits(__ldcg(a.r32 + i) * s_inv[m] * f16_bits_to_float(a.gamma[n]));
    }
    if (threadIdx.x == 0) *a.counter = 0u;
}

// ---------------------------------------------------------------------------
// QKV projection + RoPE + KV append ("Zero TVM Documentation", card 3 "QKV +
// RoPE + KV-append (fused, decode)"): a unit is one RoPE pair, rows
// (hb D + i, hb D + i + D/2) of head block hb (Q heads, then K, then V), so
// the pair is rotated in registers. Angle pos * base^(-2i/D) in fp64 (a few
// thousand per call). Q goes to q_out, rotated K and plain V to the cache
// rows of the token's slot; a slot outside [0, n_slots) writes nothing and
// sets ZQ4_DEV_BAD_SLOT.
// Angles: base^(-2i/D) once per CTA in fp64 (shared memory); the rotation
// itself is rope_rotate (zq4_rope.cuh).
// ---------------------------------------------------------------------------
constexpr int kMaxRopeHalf = 256;                 // D <= 512
template <int MT, int LPR>
__global__ void __launch_bounds__(kThreads) k_qkv_rope(QkvArgs a)
{
    extern __shared__ __align__(16) uint8_t xs[];
    __shared__ double s_freq[kMaxRopeHalf];
    __shared__ int s_pos[MT], s_slot[MT];
    const int half = a.D >> 1;
    for (int i = threadIdx.x; i < half; i += kThreads) s_freq[i] = pow(a.base, -2.0 * double(i) / double(a.D));
    const int u0 = blockIdx.x * a.units_per_cta;
    const int u1 = min(u0 + a.units_per_cta, a.units);
    if (u0 < u1) {
        const int r0 = (u0 / half) * a.D, r1 = ((u1 - 1) / half + 1) * a.D;
        prefetch_rows(a.wq, a.scales, nullptr, a.K, a.K >> 5, size_t(r0), size_t(r1));
    }
    griddep_wait();
    stage_rows(xs, a.x, a.M, MT, a.K);
    if (threadIdx.x < MT) {                     // positions and slots of the block's tokens, read once
        s_pos[threadIdx.x] = threadIdx.x < a.M ? a.pos[threadIdx.x] : 0;
        s_slot[threadIdx.x] = threadIdx.x < a.M ? a.slot[threadIdx.x] : -1;
    }
    __syncthreads();
    griddep_launch_dependents();

    const int sub = threadIdx.x / LPR, lane = threadIdx.x % LPR;
    const unsigned mask = segment_mask<LPR>();
    const uint32_t xs_base = smem_addr(xs);
    const int kv_row = a.Hkv * a.D;
    for (int u = u0 + sub; u < u1; u += kThreads / LPR) {
        const int hb = u / half, i = u - hb * half;
        float part[2][MT];
        rows_dot<MT, LPR, 2, false>(a.wq, a.scales, nullptr, a.K, hb * a.D + i, xs_base, nullptr, lane, part,
                                    half);
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) part[r][m] = segment_sum<LPR>(part[r][m], mask);
        if (lane != 0) continue;
        const bool rot = hb < a.H + a.Hkv;
        const double inv_freq = rot ? s_freq[i] : 0.0;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m >= a.M) continue;
            float oa = part[0][m], ob = part[1][m];
            if (rot) rope_rotate(s_pos[m], inv_freq, part[0][m], part[1][m], &oa, &ob);
            uint16_t *dst;
            if (hb < a.H) {
                dst = a.q_out + size_t(m) * a.H * a.D + size_t(hb) * a.D;
            } else {
                const int sl = s_slot[m];
                if (sl < 0 || sl >= a.n_slots) {
                    if (a.dev_status) atomicOr(reinterpret_cast<unsigned *>(a.dev_status), ZQ4_DEV_BAD_SLOT);
                    continue;
                }
                dst = (rot ? a.k_cache : a.v_cache) + size_t(sl) * kv_row + size_t(rot ? hb - a.H : hb - a.H - a.Hkv) * a.D;
            }
            dst[i] = float_to_f16_bits(oa);
            dst[i + half] = float_to_f16_bits(ob);
        }
    }
}

// ---------------------------------------------------------------------------
// MoE, mode GATE_UP_SILU: blockIdx.y = slot (t*top_k + j); the slot's expert
// is read after the wait (the ids may come from the previous kernel).
// ---------------------------------------------------------------------------
// AFF: affine banks (a.biases; scales and biases per 64 weights).
template <int LPR, bool AFF>
__global__ void __launch_bounds__(kThreads) k_moe_gate_up(MoeArgs a)
{
    extern __shared__ __align__(16) uint8_t xs[];
    float *xsum = reinterpret_cast<float *>(xs + size_t(a.K) * 2);     // AFF: [K/32]
    const int slot = blockIdx.y, t = slot / a.top_k;
    const int units = a.N >> 1;
    const int u0 = blockIdx.x * a.units_per_cta;
    const int u1 = min(u0 + a.units_per_cta, units);
    griddep_wait();
    const int e = a.ids[slot];
    const bool valid = e >= 0 && e < a.num_experts;
    uint16_t *yo = a.y + size_t(slot) * units;
    if (!valid) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && a.dev_status)
            atomicOr(reinterpret_cast<unsigned *>(a.dev_status), ZQ4_DEV_BAD_EXPERT_ID);
        for (int u = u0 + threadIdx.x; u < u1; u += blockDim.x) yo[u] = 0;
        griddep_launch_dependents();
        return;
    }
    const int gs = AFF ? a.K >> 6 : a.K >> 5;                          // scales per row
    const uint32_t *wq = a.wq + size_t(e) * a.N * (a.K >> 3);
    const uint16_t *sc = a.scales + size_t(e) * a.N * gs;
    const uint16_t *bi = AFF ? a.biases + size_t(e) * a.N * gs : nullptr;
    stage_rows(xs, a.x + size_t(t) * a.K, 1, 1, a.K);
    if (AFF) chunk_sums(xsum, a.x + size_t(t) * a.K, 1, 1, a.K);
    __syncthreads();
    griddep_launch_dependents();

    const int sub = threadIdx.x / LPR, lane = threadIdx.x % LPR;
    const unsigned mask = segment_mask<LPR>();
    const uint32_t xs_base = smem_addr(xs);
    for (int u = u0 + sub; u < u1; u += kThreads / LPR) {
        float part[2][1];
        rows_dot<1, LPR, 2, AFF>(wq, sc, bi, a.K, 2 * u, xs_base, xsum, lane, part);
        float g = segment_sum<LPR>(part[0][0], mask);
        float v = segment_sum<LPR>(part[1][0], mask);
        if (lane == 0) yo[u] = float_to_f16_bits(silu_f32(g) * v);
    }
}

// ---------------------------------------------------------------------------
// MoE, mode DOWN_COMBINE: blockIdx.y = token t; each unit is one output row
// n; y[t,n] = sum_j r[t,j] * (x[t,j,:] . w_{e_j}[n,:]).
// ---------------------------------------------------------------------------
template <int LPR, bool AFF>
__global__ void __launch_bounds__(kThreads) k_moe_down(MoeArgs a)
{
    extern __shared__ __align__(16) uint8_t xs[];
    float *xsum = reinterpret_cast<float *>(xs + size_t(a.top_k) * a.K * 2);   // AFF: [top_k][K/32]
    __shared__ int s_ids[32];
    __shared__ float s_r[32];
    const int t = blockIdx.y;
    const int u0 = blockIdx.x * a.units_per_cta;
    const int u1 = min(u0 + a.units_per_cta, a.N);
    griddep_wait();
    if (threadIdx.x < a.top_k) {
        int e = a.ids[t * a.top_k + threadIdx.x];
        bool valid = e >= 0 && e < a.num_experts;
        if (!valid && blockIdx.x == 0 && a.dev_status)
            atomicOr(reinterpret_cast<unsigned *>(a.dev_status), ZQ4_DEV_BAD_EXPERT_ID);
        s_ids[threadIdx.x] = valid ? e : -1;
        s_r[threadIdx.x] = a.route_w[t * a.top_k + threadIdx.x];
    }
    stage_rows(xs, a.x + size_t(t) * a.top_k * a.K, a.top_k, a.top_k, a.K);
    if (AFF) chunk_sums(xsum, a.x + size_t(t) * a.top_k * a.K, a.top_k, a.top_k, a.K);
    __syncthreads();
    griddep_launch_dependents();

    const int G = a.K >> 5, KW = a.K >> 3, GS = AFF ? a.K >> 6 : G;
    const uint32_t row_bytes = uint32_t(a.K) * 2;
    const size_t expert_words = size_t(a.N) * KW, expert_scales = size_t(a.N) * GS;
    const int sub = threadIdx.x / LPR, lane = threadIdx.x % LPR;
    const unsigned mask = segment_mask<LPR>();
    const uint32_t xs_base = smem_addr(xs);
    for (int n = u0 + sub; n < u1; n += kThreads / LPR) {
        float acc = 0.f;
        for (int g = lane; g < G; g += LPR) {
            for (int j0 = 0; j0 < a.top_k; j0 += kMoeSlotChunk) {
                uint4 wv[kMoeSlotChunk];
                uint16_t sv[kMoeSlotChunk], bv[kMoeSlotChunk];
#pragma unroll
                for (int i = 0; i < kMoeSlotChunk; ++i) {
                    int j = j0 + i, e = j < a.top_k ? s_ids[j] : -1;
                    if (e >= 0) {
                        const size_t so = size_t(e) * expert_scales + size_t(n) * GS + (AFF ? g >> 1 : g);
                        wv[i] = ldg_stream_v4(a.wq + size_t(e) * expert_words + size_t(n) * KW + 4 * g);
                        sv[i] = ldg_u16(a.scales + so);
                        bv[i] = AFF ? ldg_u16(a.biases + so) : uint16_t(0);
                    } else {
                        wv[i] = make_uint4(0, 0, 0, 0);
                        sv[i] = 0;
                        bv[i] = 0;
                    }
                }
#pragma unroll
                for (int i = 0; i < kMoeSlotChunk; ++i) {
                    int j = j0 + i;
                    if (j < a.top_k && s_ids[j] >= 0) {
                        float part[1] = {0.f};
                        group_dot<1, AFF>(wv[i], f16_bits_to_float(sv[i]), f16_bits_to_float(bv[i]),
                                          xs_base + uint32_t(j) * row_bytes, g, row_bytes,
                                          AFF ? xsum + j * G : nullptr, G, part);
                        acc = fmaf(s_r[j], part[0], acc);
                    }
                }
            }
        }
        acc = segment_sum<LPR>(acc, mask);
        if (lane == 0) a.y[size_t(t) * a.N + n] = float_to_f16_bits(acc);
    }
}

// ---------------------------------------------------------------------------
// Dequantize (one thread per packed word) and row-order rewrite.
// ---------------------------------------------------------------------------
__global__ void k_dequant_f32(const uint32_t *wq, const uint16_t *scales, float *w, int N, int K)
{
    const size_t words = size_t(N) * (K >> 3);
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < words;
         i += size_t(gridDim.x) * blockDim.x) {
        uint32_t v = wq[i];
        size_t n = i / (K >> 3), kw = i - n * (K >> 3);
        float s = f16_bits_to_float(scales[n * (K >> 5) + (kw >> 2)]);
        float *o = w + n * K + kw * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = float(int((v >> (4 * e)) & 0xF) - 7) * s;
    }
}

// f16((q - 7) * s): the exact f16 (q - 7) pairs times the f16 scale pair,
// rounded once to nearest even; the same operation the tensor-core GEMM
// applies when it dequantizes tiles.
__global__ void k_dequant_f16(const uint32_t *wq, const uint16_t *scales, uint16_t *w, int N, int K)
{
    const size_t words = size_t(N) * (K >> 3);
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < words;
         i += size_t(gridDim.x) * blockDim.x) {
        size_t n = i / (K >> 3), kw = i - n * (K >> 3);
        uint32_t s = scales[n * (K >> 5) + (kw >> 2)];
        uint32_t s2 = s | (s << 16);
        uint32_t p[4];
        unpack_word_f16x2(wq[i], p);
        uint16_t *o = w + n * K + kw * 8;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t d = hmul2(p[j], s2);     // elements j (low) and j + 4 (high)
            o[j] = uint16_t(d & 0xFFFF);
            o[j + 4] = uint16_t(d >> 16);
        }
    }
}

// dst row 2j <- src row j, dst row 2j+1 <- src row N/2 + j (or a plain copy).
__global__ void k_prepare(const uint32_t *wq_src, const uint16_t *sc_src, uint32_t *wq_dst,
                          uint16_t *sc_dst, int N, int K, int interleave)
{
    const int KW = K >> 3, G = K >> 5, half = N >> 1;
    const int dst_row = blockIdx.x;
    const int src_row = interleave ? ((dst_row & 1) ? half + (dst_row >> 1) : (dst_row >> 1)) : dst_row;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(wq_src + size_t(src_row) * KW);
    uint4 *d4 = reinterpret_cast<uint4 *>(wq_dst + size_t(dst_row) * KW);
    for (int i = threadIdx.x; i < KW / 4; i += blockDim.x) d4[i] = s4[i];
    for (int i = threadIdx.x; i < G; i += blockDim.x)
        sc_dst[size_t(dst_row) * G + i] = sc_src[size_t(src_row) * G + i];
}

// Segmented layout: segment (tile t, column block s) of 16 rows x 256
// columns is 2304 contiguous bytes, one 144-byte record per row: the row's
// 32 code words of the block, then its 8 group scales (16 bytes). Within a
// record, word 8q + g (q = 0..3, g = 0..7) holds word q of group g (column
// word 32 s + 4 g + q), so a decode lane that takes word q of every group
// reads 32 contiguous bytes; within a word, nibble slot i holds element
// (0, 2, 4, 6, 1, 3, 5, 7)[i], so that the unpack's four f16 pairs are the
// consecutive element pairs (0,1), (2,3), (4,5), (6,7) and x needs no
// reordering. The 144-byte row stride staggers the rows over the shared
// memory banks (no conflicts for the fragment loads). Segments are stored
// tile-major; rows past N are zero. Source row = dst row, or the gate/up
// interleave of the concatenated [gate; up] matrix. One CTA (144 threads)
// per segment: thread 36 i + c writes 4-byte word c of row record i.
__device__ __forceinline__ uint32_t seg_nibble_order(uint32_t w)
{
    uint32_t o = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = (i < 4) ? 2 * i : 2 * (i - 4) + 1;    // element in nibble slot i
        o |= ((w >> (4 * e)) & 0xFu) << (4 * i);
    }
    return o;
}

__global__ void k_prepare_segmented(const uint32_t *wq_src, const uint16_t *sc_src, uint8_t *dst, int N, int K,
                                    int interleave)
{
    const int KW = K >> 3, G = K >> 5, S = K >> 8, half = N >> 1;
    const int tile = blockIdx.x / S, seg = blockIdx.x - tile * S;
    uint32_t *base = reinterpret_cast<uint32_t *>(dst + size_t(blockIdx.x) * 2304);
    for (int i = threadIdx.x; i < 16 * 36; i += blockDim.x) {
        const int row = i / 36, c = i - row * 36, n = tile * 16 + row;
        uint32_t v = 0;
        if (n < N) {
            const int src = interleave ? ((n & 1) ? half + (n >> 1) : (n >> 1)) : n;
            if (c < 32) {
                const int q = c >> 3, g = c & 7;
                v = seg_nibble_order(wq_src[size_t(src) * KW + seg * 32 + 4 * g + q]);
            } else {
                v = *reinterpret_cast<const uint32_t *>(sc_src + size_t(src) * G + seg * 8 + 2 * (c - 32));
            }
        }
        base[i] = v;
    }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
namespace {

int pick_lpr(int K)
{
    int G = K >> 5;
    return G >= 32 ? 32 : (G >= 16 ? 16 : 8);
}

// Units per CTA: one unit per row segment of the CTA, doubled while the grid
// would still cover every SM twice (fewer, fuller CTAs stage x less often).
int units_per_cta(int units, int lpr)
{
    int subs = kThreads / lpr;
    int upc = subs;
    int sms = sm_count();
    while (units / (2 * upc) >= 2 * sms && upc < 8 * subs) upc *= 2;
    return upc;
}

// Shared memory of a dense launch: x rows, and for the affine format the
// chunk sums of x.
size_t dense_smem(int MT, int K, bool aff) { return size_t(MT) * K * 2 + (aff ? size_t(MT) * (K >> 5) * 4 : 0); }

template <int MT, int LPR, int RU, bool AFF>
cudaError_t launch_dense_t(const DenseArgs &a, cudaStream_t s)
{
    static int smem_set[kMaxDevices] = {};
    auto kern = k_dense<MT, LPR, RU, AFF>;
    size_t smem = dense_smem(MT, a.K, AFF);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(kern), smem, smem_set);
    if (e != cudaSuccess) return e;
    int grid = (a.units + a.units_per_cta - 1) / a.units_per_cta;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a);
}

template <int MT, int RU, bool AFF>
cudaError_t launch_dense_lpr(const DenseArgs &a, cudaStream_t s)
{
    switch (pick_lpr(a.K)) {
    case 32: return launch_dense_t<MT, 32, RU, AFF>(a, s);
    case 16: return launch_dense_t<MT, 16, RU, AFF>(a, s);
    default: return launch_dense_t<MT, 8, RU, AFF>(a, s);
    }
}

template <int RU, bool AFF>
cudaError_t launch_dense_mt(int MT, const DenseArgs &a, cudaStream_t s)
{
    switch (MT) {
    case 8: return launch_dense_lpr<8, RU, AFF>(a, s);
    case 4: return launch_dense_lpr<4, RU, AFF>(a, s);
    case 2: return launch_dense_lpr<2, RU, AFF>(a, s);
    default: return launch_dense_lpr<1, RU, AFF>(a, s);
    }
}

}  // namespace

size_t decode_max_smem() { return 227 * 1024; }

int decode_tokens_per_launch(int M, int K, bool aff)
{
    int mt = 8;
    while (mt > 1 && (mt > M || dense_smem(mt, K, aff) > decode_max_smem())) mt >>= 1;
    return mt;
}

int decode_tokens_per_launch(int M, int K) { return decode_tokens_per_launch(M, K, false); }

// biases != nullptr: the MLX affine format (scales and biases per 64 weights).
namespace {

template <int MT, int LPR>
cudaError_t launch_rms_t(const RmsArgs &a, cudaStream_t s)
{
    static int smem_set[kMaxDevices] = {};
    auto kern = k_dense_rms<MT, LPR>;
    const size_t smem = dense_smem(MT, a.K, false);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(kern), smem, smem_set);
    if (e != cudaSuccess) return e;
    const int grid = (a.N + a.units_per_cta - 1) / a.units_per_cta;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a);
}

template <int MT>
cudaError_t launch_rms_lpr(const RmsArgs &a, cudaStream_t s)
{
    switch (pick_lpr(a.K)) {
    case 32: return launch_rms_t<MT, 32>(a, s);
    case 16: return launch_rms_t<MT, 16>(a, s);
    default: return launch_rms_t<MT, 8>(a, s);
    }
}

}  // namespace

namespace {

template <int MT, int LPR>
cudaError_t launch_qkv_t(const QkvArgs &a, cudaStream_t s)
{
    static int smem_set[kMaxDevices] = {};
    auto kern = k_qkv_rope<MT, LPR>;
    const size_t smem = dense_smem(MT, a.K, false);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(kern), smem, smem_set);
    if (e != cudaSuccess) return e;
    const int grid = (a.units + a.units_per_cta - 1) / a.units_per_cta;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a);
}

template <int MT>
cudaError_t launch_qkv_lpr(const QkvArgs &a, cudaStream_t s)
{
    switch (pick_lpr(a.K)) {
    case 32: return launch_qkv_t<MT, 32>(a, s);
    case 16: return launch_qkv_t<MT, 16>(a, s);
    default: return launch_qkv_t<MT, 8>(a, s);
    }
}

}  // namespace

cudaError_t launch_qkv_rope(const QkvArgs &a0, cudaStream_t s)
{
    QkvArgs a = a0;
    a.units = (a.H + 2 * a.Hkv) * (a.D >> 1);
    a.units_per_cta = units_per_cta(a.units, pick_lpr(a.K));
    const uint16_t *x = a0.x;
    uint16_t *q = a0.q_out;
    for (int m0 = 0; m0 < a0.M;) {
        // tokens per launch: x in dynamic shared memory next to the static
        // frequency table
        int mt = 8;
        while (mt > 1 && (mt > a0.M - m0 || dense_smem(mt, a0.K, false) + sizeof(double) * kMaxRopeHalf >
                                                  decode_max_smem()))
            mt >>= 1;
        a.x = x + size_t(m0) * a.K;
        a.q_out = q + size_t(m0) * a.H * a.D;
        a.pos = a0.pos + m0;
        a.slot = a0.slot + m0;
        a.M = std::min(mt, a0.M - m0);
        cudaError_t e;
        switch (mt) {
        case 8: e = launch_qkv_lpr<8>(a, s); break;
        case 4: e = launch_qkv_lpr<4>(a, s); break;
        case 2: e = launch_qkv_lpr<2>(a, s); break;
        default: e = launch_qkv_lpr<1>(a, s); break;
        }
        if (e != cudaSuccess) return e;
        m0 += a.M;
    }
    return cudaSuccess;
}

// work: 16 bytes of counter (zero before the first call, left zero), then
// the fp32 r of M x N.
cudaError_t launch_add_rmsnorm(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, const uint16_t *resid,
                               const uint16_t *gamma, float eps, uint16_t *res_out, uint16_t *out, void *work, int M,
                               int N, int K, cudaStream_t s)
{
    RmsArgs a;
    a.wq = wq;
    a.scales = scales;
    a.gamma = gamma;
    a.eps = eps;
    a.N = N;
    a.K = K;
    a.counter = static_cast<unsigned *>(work);
    a.units_per_cta = units_per_cta(N, pick_lpr(K));
    float *r32 = reinterpret_cast<float *>(static_cast<uint8_t *>(work) + 16);
    for (int m0 = 0; m0 < M;) {
        const int mt = decode_tokens_per_launch(M - m0, K, false);
        const size_t o = size_t(m0) * N;
        a.x = x + size_t(m0) * K;
        a.resid = resid + o;
        a.res_out = res_out + o;
        a.out = out + o;
        a.r32 = r32 + o;
        a.M = std::min(mt, M - m0);
        cudaError_t e;
        switch (mt) {
        case 8: e = launch_rms_lpr<8>(a, s); break;
        case 4: e = launch_rms_lpr<4>(a, s); break;
        case 2: e = launch_rms_lpr<2>(a, s); break;
        default: e = launch_rms_lpr<1>(a, s); break;
        }
        if (e != cudaSuccess) return e;
        m0 += a.M;
    }
    return cudaSuccess;
}

cudaError_t launch_decode(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases, const uint16_t *x,
                          uint16_t *y, int M, int N, int K, bool gate_up, cudaStream_t s)
{
    const int RU = gate_up ? 2 : 1;
    const int out_cols = N / RU;
    const bool aff = biases != nullptr;
    DenseArgs a;
    a.wq = wq;
    a.scales = scales;
    a.biases = biases;
    a.K = K;
    a.units = out_cols;
    a.units_per_cta = units_per_cta(a.units, pick_lpr(K));
    a.y_stride = out_cols;
    for (int m0 = 0; m0 < M;) {
        int mt = decode_tokens_per_launch(M - m0, K, aff);
        a.x = x + size_t(m0) * K;
        a.y = y + size_t(m0) * out_cols;
        a.M = std::min(mt, M - m0);
        cudaError_t e = aff ? (gate_up ? launch_dense_mt<2, true>(mt, a, s) : launch_dense_mt<1, true>(mt, a, s))
                            : (gate_up ? launch_dense_mt<2, false>(mt, a, s) : launch_dense_mt<1, false>(mt, a, s));
        if (e != cudaSuccess) return e;
        m0 += a.M;
    }
    return cudaSuccess;
}

namespace {

template <int LPR, bool AFF>
cudaError_t launch_moe_t(const MoeArgs &a, int mode, dim3 grid, size_t smem, cudaStream_t s)
{
    static int set_gu[kMaxDevices] = {}, set_dn[kMaxDevices] = {};
    if (mode == ZQ4_MOE_GATE_UP_SILU) {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_moe_gate_up<LPR, AFF>), smem, set_gu);
        return e != cudaSuccess ? e : launch_pdl(k_moe_gate_up<LPR, AFF>, grid, dim3(kThreads), smem, s, a);
    }
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_moe_down<LPR, AFF>), smem, set_dn);
    return e != cudaSuccess ? e : launch_pdl(k_moe_down<LPR, AFF>, grid, dim3(kThreads), smem, s, a);
}

template <bool AFF>
cudaError_t launch_moe_lpr(int lpr, const MoeArgs &a, int mode, dim3 grid, size_t smem, cudaStream_t s)
{
    switch (lpr) {
    case 32: return launch_moe_t<32, AFF>(a, mode, grid, smem, s);
    case 16: return launch_moe_t<16, AFF>(a, mode, grid, smem, s);
    default: return launch_moe_t<8, AFF>(a, mode, grid, smem, s);
    }
}

}  // namespace

// Shared memory of a MoE launch: the staged x rows (1 for gate_up, top_k for
// down) and, for affine banks, their chunk sums.
size_t moe_smem(int mode, int K, int top_k, bool aff)
{
    const size_t rows = mode == ZQ4_MOE_GATE_UP_SILU ? 1 : size_t(top_k);
    return rows * K * 2 + (aff ? rows * (K >> 5) * 4 : 0);
}

// a.biases != nullptr: affine banks.
cudaError_t launch_moe(const MoeArgs &a0, int mode, cudaStream_t s)
{
    MoeArgs a = a0;
    const bool aff = a.biases != nullptr;
    const int lpr = pick_lpr(a.K);
    const size_t smem = moe_smem(mode, a.K, a.top_k, aff);
    dim3 grid;
    if (mode == ZQ4_MOE_GATE_UP_SILU) {
        a.units_per_cta = units_per_cta(a.N >> 1, lpr);
        grid = dim3(((a.N >> 1) + a.units_per_cta - 1) / a.units_per_cta, a.T * a.top_k);
    } else {
        a.units_per_cta = units_per_cta(a.N, lpr);
        grid = dim3((a.N + a.units_per_cta - 1) / a.units_per_cta, a.T);
    }
    return aff ? launch_moe_lpr<true>(lpr, a, mode, grid, smem, s) : launch_moe_lpr<false>(lpr, a, mode, grid, smem, s);
}

static int elementwise_grid(size_t items)
{
    size_t blocks = (items + 255) / 256;
    size_t cap = size_t(sm_count()) * 8;
    return int(std::max<size_t>(1, std::min(blocks, cap)));
}

cudaError_t launch_dequant_f32(const uint32_t *wq, const uint16_t *scales, float *w, int N, int K,
                               cudaStream_t s)
{
    k_dequant_f32<<<elementwise_grid(size_t(N) * (K >> 3)), 256, 0, s>>>(wq, scales, w, N, K);
    return cudaGetLastError();
}

cudaError_t launch_dequant_f16(const uint32_t *wq, const uint16_t *scales, uint16_t *w, int N,
                               int K, cudaStream_t s)
{
    k_dequant_f16<<<elementwise_grid(size_t(N) * (K >> 3)), 256, 0, s>>>(wq, scales, w, N, K);
    return cudaGetLastError();
}

cudaError_t launch_prepare(const uint32_t *wq_src, const uint16_t *sc_src, uint32_t *wq_dst,
                           uint16_t *sc_dst, int N, int K, int interleave, cudaStream_t s)
{
    k_prepare<<<N, 128, 0, s>>>(wq_src, sc_src, wq_dst, sc_dst, N, K, interleave);
    return cudaGetLastError();
}

cudaError_t launch_prepare_segmented(const uint32_t *wq_src, const uint16_t *sc_src, uint8_t *dst, int N, int K,
                                     int interleave, cudaStream_t s)
{
    const long long segs = (long long)((N + 15) / 16) * (K / 256);
    if (segs > 0x7fffffff) return cudaErrorInvalidValue;
    k_prepare_segmented<<<unsigned(segs), 144, 0, s>>>(wq_src, sc_src, dst, N, K, interleave);
    return cudaGetLastError();
}

}  // namespace zq4
