// zq4_segment.cuh -- the work unit of the decode kernels that stream the
// segmented weight layout (zq4_prepare_weight with ZQ4_PREP_SEGMENTED): one
// segment = 16 weight rows x 256 columns = 2304 contiguous bytes, one
// 144-byte record per row (32 code words, then the row's 8 group scales).
// Record word 8q + g holds word q of group g, its nibbles ordered so that the
// exact unpack yields the element pairs (0,1), (2,3), (4,5), (6,7).
//
// Per 32-column group, lane (r, t) (r = lane/4, t = lane%4) takes word t of
// rows r and r+8 -- the 32 contiguous bytes 144 r + 32 t .. of the segment
// hold word t of all eight groups, so four 16-byte shared loads fetch the
// lane's words of the whole segment, without bank conflicts (the 144-byte
// row stride staggers the rows over the banks) -- and unpacks them into
// exact f16 (q - 7) pairs: the A fragments of two chained m16n8k16 MMAs
// against x of token r at columns 32 g + 8 t .. 32 g + 8 t + 7 (B, read as
// it is stored), fp32 accumulation; the group result times the fp32 group
// scale goes into the lane's accumulator (rows r, r+8 x tokens 2t, 2t+1).
// q4f16_1 itself is the format of "Zero TVM Documentation", section "Q4F16
// quantization format".
#pragma once

#include <stdint.h>

#include "zq4_async.cuh"
#include "zq4_common.cuh"

namespace zq4 {
namespace segk {

constexpr int kSegCols = 256;
constexpr int kCodeBytes = 16 * 128;
constexpr int kSegBytes = kCodeBytes + 16 * 8 * 2;   // 2304
constexpr int kTokCols = 8;                          // MMA columns = tokens (M <= 8)

__host__ __device__ inline size_t xs_row_bytes(int K) { return size_t(K) * 2 + 64; }

// Part i of n of [lo, hi): [b, e), sizes equal to within one (32-bit math;
// callers keep (hi - lo) * n below 2^31).
__device__ __forceinline__ void split(int lo, int hi, int i, int n, int &b, int &e)
{
    const unsigned len = unsigned(hi - lo);
    b = lo + int(len * unsigned(i) / unsigned(n));
    e = lo + int(len * unsigned(i + 1) / unsigned(n));
}

__device__ __forceinline__ int part_begin(int lo, int hi, int i, int n)
{
    return lo + int(unsigned(hi - lo) * unsigned(i) / unsigned(n));
}

// Stage x [M][K] into shared memory rows of `xrow` bytes, as stored. Loads
// go through L2 only (x may have been written by other SMs) and are issued
// kBatch at a time per thread, so one memory latency covers up to kBatch *
// nthreads chunks (x is usually cold in L2 in a decode step: the weights
// stream through it).
template <int kBatch>
__device__ __forceinline__ void stage_x(uint8_t *xs, uint32_t xrow, const uint16_t *x, int M, int K, int tid,
                                        int nthreads)
{
    const int words = K >> 3, total = M * words;
    for (int i0 = tid; i0 < total; i0 += kBatch * nthreads) {
        uint4 v[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int i = i0 + b * nthreads;
            if (i < total) {
                const int m = i / words, cw = i - m * words;
                v[b] = __ldcg(reinterpret_cast<const uint4 *>(x + size_t(m) * K + size_t(cw) * 8));
            }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int i = i0 + b * nthreads;
            if (i < total) {
                const int m = i / words, cw = i - m * words;
                *reinterpret_cast<uint4 *>(xs + size_t(m) * xrow + size_t(cw) * 16) = v[b];
            }
        }
    }
}

// Byte offset of lane (r, t)'s code words of row r within a segment.
__device__ __forceinline__ uint32_t lane_code_offset(int lane)
{
    return uint32_t((lane >> 2) * 144 + 32 * (lane & 3));
}

// The lane's word of group g (0..7) from its two 16-byte loads of one row.
__device__ __forceinline__ uint32_t group_word(const uint4 &lo, const uint4 &hi, int g)
{
    const uint4 &v = g < 4 ? lo : hi;
    const int i = g & 3;
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// acc += one segment held in shared memory at `cb`; `aoff` =
// lane_code_offset(lane); `xg` = the staged x row of this lane's token at the
// segment's first column (+16 t).
__device__ __forceinline__ void accumulate(uint32_t cb, uint32_t aoff, const uint8_t *xg, int r, float (&acc)[4])
{
    const uint4 c0 = lds_v4(cb + aoff), c1 = lds_v4(cb + aoff + 16);               // row r, groups 0-3, 4-7
    const uint4 c8 = lds_v4(cb + aoff + 1152), c9 = lds_v4(cb + aoff + 1168);      // row r+8
    const uint4 sr = lds_v4(cb + r * 144 + 128);                                    // row r, scales 0..7
    const uint4 sr8 = lds_v4(cb + (r + 8) * 144 + 128);
    const uint32_t srw[4] = {sr.x, sr.y, sr.z, sr.w}, sr8w[4] = {sr8.x, sr8.y, sr8.z, sr8.w};
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        uint32_t pa[4], pb[4];
        unpack_word_f16x2(group_word(c0, c1, g), pa);
        unpack_word_f16x2(group_word(c8, c9, g), pb);
        const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
        const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
        const float s_r = f16_bits_to_float(uint16_t((g & 1) ? srw[g >> 1] >> 16 : srw[g >> 1]));
        const float s_r8 = f16_bits_to_float(uint16_t((g & 1) ? sr8w[g >> 1] >> 16 : sr8w[g >> 1]));
        const uint4 xv = *reinterpret_cast<const uint4 *>(xg + g * 64);
        const float z[4] = {0.f, 0.f, 0.f, 0.f};
        float d[4];
        mma16816(d, a0, xv.x, xv.y, z);
        mma16816(d, a1, xv.z, xv.w, d);
        acc[0] = fmaf(s_r, d[0], acc[0]);
        acc[1] = fmaf(s_r, d[1], acc[1]);
        acc[2] = fmaf(s_r8, d[2], acc[2]);
        acc[3] = fmaf(s_r8, d[3], acc[3]);
    }
}

// Write a whole tile (rows row0 .. row0+15) from the warp's accumulators:
// f16(acc), or f16(silu(g) * u) for interleaved gate/up rows (up sits in the
// lane 4 higher).
__device__ __forceinline__ void write_tile(const float (&acc)[4], int row0, int lane, int gate_up, int M, int N,
                                           int y_stride, uint16_t *y)
{
    const int r = lane >> 2, t = lane & 3;
    if (!gate_up) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = row0 + r + 8 * h;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int m = 2 * t + c;
                if (n < N && m < M) y[size_t(m) * y_stride + n] = float_to_f16_bits(acc[2 * h + c]);
            }
        }
    } else {
        float up[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) up[i] = __shfl_down_sync(0xffffffffu, acc[i], 4);
        if ((r & 1) == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = row0 + r + 8 * h;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int m = 2 * t + c;
                    if (n + 1 < N && m < M)
                        y[size_t(m) * y_stride + (n >> 1)] = float_to_f16_bits(silu_f32(acc[2 * h + c]) * up[2 * h + c]);
                }
            }
        }
    }
}

// Park this warp's part of a tile shared with other warps: slot 0 for the
// warp's first tile, 1 for its last ([kWarps*2][16][kTokCols] floats).
__device__ __forceinline__ void park(const float (&acc)[4], float *wpark, int warp, int slot, int lane)
{
    const int r = lane >> 2, t = lane & 3;
    float *pk = wpark + ((warp * 2 + slot) * 16) * kTokCols;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 2; ++c) pk[(r + 8 * h) * kTokCols + 2 * t + c] = acc[2 * h + c];
}

// After a CTA barrier: every thread takes (tile, output) items of the tiles
// [tb, te) that were split between warps and sums the parked parts of the
// contributing warps in warp order (bit-reproducible), then writes the
// output. `wtab` holds the warp range starts (segments, W + 1 entries)
// followed by each warp's first tile.
template <int W, int NT>
__device__ __forceinline__ void finalize_split(int tb, int te, int S, int gate_up, int M, int N, int y_stride,
                                               uint16_t *y, const float *wpark, const int *wtab)
{
    const int *wb = wtab, *wft = wtab + W + 1;
    const int per_tok = gate_up ? 8 : 16;
    const int items = (te - tb) * per_tok * M;
    for (int it = threadIdx.x; it < items; it += NT) {
        const int tt = tb + it / (per_tok * M);
        const int o = it - (tt - tb) * (per_tok * M);
        const int lo = tt * S, hi = lo + S;
        unsigned mask = 0;
#pragma unroll
        for (int w = 0; w < W; ++w)
            if (wb[w] < wb[w + 1] && wb[w] < hi && wb[w + 1] > lo) mask |= 1u << w;
        if (__popc(mask) < 2) continue;                  // one warp held the whole tile
        const int m = o / per_tok, i = o - m * per_tok;
        const int ra = gate_up ? 2 * i : i;
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            if (!((mask >> w) & 1)) continue;
            const float *qk = wpark + ((w * 2 + (tt == wft[w] ? 0 : 1)) * 16) * kTokCols;
            v0 += qk[ra * kTokCols + m];
            if (gate_up) v1 += qk[(ra + 1) * kTokCols + m];
        }
        const int row0 = tt * 16;
        if (!gate_up) {
            if (row0 + i < N) y[size_t(m) * y_stride + row0 + i] = float_to_f16_bits(v0);
        } else if (row0 + 2 * i + 1 < N) {
            y[size_t(m) * y_stride + (row0 >> 1) + i] = float_to_f16_bits(silu_f32(v0) * v1);
        }
    }
}

}  // namespace segk
}  // namespace zq4
