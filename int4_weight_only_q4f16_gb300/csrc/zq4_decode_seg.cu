// zq4_decode_seg.cu -- the decode GEMV / gate_up for M = 1..8 on weights in
// the segmented layout, one launch per projection.
//
// What it computes: y = x * W^T with W in q4f16_1 ("Zero TVM Documentation",
// section "Q4F16 quantization format" and card 5 "int4 Matmul"), or the fused
// gate_up + SiLU*mul output (card 6 "Fused FFN") for interleaved gate/up
// rows; fp32 accumulation, f16 output.
//
// How (sized so that two consecutive launches share every SM):
//  * Grid = one CTA of 8 warps per SM; CTA c takes the whole 16-row tiles
//    [c*T/G, (c+1)*T/G) and splits their 256-column segments evenly over its
//    warps. Each warp streams its segments through its own ring of 4
//    shared-memory slots, one contiguous bulk copy (2304 bytes) per segment,
//    with a look-ahead of L2 prefetches, and computes each with the segment
//    routine of zq4_segment.cuh (16-byte shared loads of the row records,
//    exact (q - 7) unpack, two chained m16n8k16 MMAs per group, fp32
//    scale-and-accumulate).
//  * The weights never depend on the previous kernel, so each warp requests
//    its first segments before griddepcontrol.wait; with about 100 KB of
//    shared memory and at most 128 registers per thread, a CTA of the next
//    launch fits beside one of this launch, so its weights are in flight (or
//    landed) while this launch finishes.
//  * Tiles held by one warp are written by it; parts of tiles shared between
//    warps are parked in shared memory and summed by all threads in warp
//    order after one CTA barrier (bit-reproducible).
//  * Every mbarrier wait is bounded; on expiry the kernel records
//    ZQ4_DEVERR_WAIT_TIMEOUT, lets its issued copies land and returns.
#include <cuda_fp16.h>

#include <algorithm>

#include "zq4_async.cuh"
#include "zq4_common.cuh"
#include "zq4_internal.h"
#include "zq4_segment.cuh"

namespace zq4 {

// Set (OR) by this file's kernel when an internal wait gives up; read and
// cleared by read_seg_error().
__device__ unsigned g_seg_error = 0;

namespace sgc {

using namespace segk;

#ifndef ZQ4_SEG_PREFETCH
#define ZQ4_SEG_PREFETCH 4
#endif

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 4;
constexpr int kPrefetch = ZQ4_SEG_PREFETCH;

struct Args {
    const uint8_t *seg;   // the matrix in the segmented layout
    const uint16_t *x;    // [M][K]
    uint16_t *y;          // [M][y_stride]
    int M, N, K, T, S, y_stride, gate_up;
};

constexpr size_t kRingOff = 0;
constexpr size_t kBarOff = kRingOff + size_t(kWarps) * kSlots * kSegBytes;
constexpr size_t kParkOff = kBarOff + size_t(kWarps) * kSlots * 8;
constexpr size_t kTabOff = kParkOff + size_t(kWarps) * 2 * 16 * kTokCols * 4;
constexpr size_t kXsOff = kTabOff + 128;
inline size_t smem_bytes(int M, int K) { return 1024 + kXsOff + size_t(M) * xs_row_bytes(K); }

__global__ void __launch_bounds__(kThreads, 2) k_gemv_seg(Args a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_addr(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, r = lane >> 2, t = lane & 3;
    const uint32_t ring0 = sbase + uint32_t(kRingOff) + uint32_t(warp * kSlots * kSegBytes);
    const uint32_t bar0 = sbase + uint32_t(kBarOff) + uint32_t(warp * kSlots * 8);
    float *wpark = reinterpret_cast<float *>(smem + kParkOff);
    int *wtab = reinterpret_cast<int *>(smem + kTabOff);
    uint8_t *xs = smem + kXsOff;
    const uint32_t xrow = uint32_t(xs_row_bytes(a.K));
    const int S = a.S;
    int tb, te, ub, ue;
    split(0, a.T, blockIdx.x, gridDim.x, tb, te);
    const int cb = tb * S, ce = te * S;
    split(cb, ce, warp, kWarps, ub, ue);
    const int n = ue - ub;

    // ---- before the grid-dependency wait: barriers, first copies, look-ahead
    if (lane == 0) {
        for (int j = 0; j < kSlots; ++j) mbar_init(bar0 + 8 * j, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    auto issue = [&](int i) {                    // lane 0: segment ub + i into slot i % kSlots
        const uint32_t bar = bar0 + 8 * (i % kSlots);
        mbar_arrive_expect_tx(bar, kSegBytes);
        bulk_load(ring0 + (i % kSlots) * kSegBytes, a.seg + size_t(ub + i) * kSegBytes, kSegBytes, bar);
    };
    if (lane == 0) {
        for (int i = 0; i < kSlots && i < n; ++i) issue(i);
        for (int i = kSlots; i < kSlots + kPrefetch && i < n; ++i)
            prefetch_l2_bulk(a.seg + size_t(ub + i) * kSegBytes, kSegBytes);
    }
    if (threadIdx.x <= kWarps) {
        const int b = part_begin(cb, ce, threadIdx.x, kWarps);
        wtab[threadIdx.x] = b;
        wtab[kWarps + 1 + threadIdx.x] = b / S;
    }

    // ---- x, once the previous kernel's writes are visible
    griddep_wait();
    stage_x<8>(xs, xrow, a.x, a.M, a.K, threadIdx.x, kThreads);
    __syncthreads();
    griddep_launch_dependents();

    const uint32_t aoff = lane_code_offset(lane);
    const uint8_t *xr = xs + size_t(min(r, a.M - 1)) * xrow + 16 * t;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int cur_tile = -1;
    const int first_tile = ub / S;
    auto flush = [&](int tt) {
        if (tt * S >= ub && (tt + 1) * S <= ue)
            write_tile(acc, tt * 16, lane, a.gate_up, a.M, a.N, a.y_stride, a.y);
        else
            park(acc, wpark, warp, tt == first_tile ? 0 : 1, lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = 0.f;
    };

    bool ok = true;
    int i = 0;
    for (; i < n; ++i) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (i % kSlots), (i / kSlots) & 1))) {
            ok = false;
            break;
        }
        const int u = ub + i, tt = u / S, seg = u - tt * S;
        if (tt != cur_tile) {
            if (cur_tile >= 0) flush(cur_tile);
            cur_tile = tt;
        }
        accumulate(ring0 + (i % kSlots) * kSegBytes, aoff, xr + seg * 32 * 16, r, acc);
        // every lane's reads of the slot are done before the refill overwrites it
        __syncwarp();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (lane == 0 && i + kSlots < n) {
            issue(i + kSlots);
            if (i + kSlots + kPrefetch < n)
                prefetch_l2_bulk(a.seg + size_t(ub + i + kSlots + kPrefetch) * kSegBytes, kSegBytes);
        }
    }
    if (ok) {
        if (cur_tile >= 0) flush(cur_tile);
    } else {
        if (lane == 0) atomicOr(&g_seg_error, ZQ4_DEVERR_WAIT_TIMEOUT);
        for (int c = i; c < n && c < i + kSlots; ++c)        // copies still in flight
            if (!mbar_wait(bar0 + 8 * (c % kSlots), (c / kSlots) & 1)) break;
    }
    __syncthreads();
    finalize_split<kWarps, kThreads>(tb, te, S, a.gate_up, a.M, a.N, a.y_stride, a.y, wpark, wtab);
}

}  // namespace sgc

bool seg_gemv_supported(int M, int K)
{
    return M >= 1 && M <= segk::kTokCols && K % segk::kSegCols == 0 &&
           sgc::smem_bytes(M, K) <= size_t(227) * 1024;
}

cudaError_t launch_gemv_seg(const uint8_t *wseg, const uint16_t *x, uint16_t *y, int M, int N, int K,
                            bool gate_up, cudaStream_t s)
{
    sgc::Args a;
    a.seg = wseg;
    a.x = x;
    a.y = y;
    a.M = M;
    a.N = N;
    a.K = K;
    a.T = (N + 15) / 16;
    a.S = K / segk::kSegCols;
    a.gate_up = gate_up ? 1 : 0;
    a.y_stride = gate_up ? N / 2 : N;
    static int smem_set[kMaxDevices] = {};
    const size_t smem = sgc::smem_bytes(M, K);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(sgc::k_gemv_seg), smem, smem_set);
    if (e != cudaSuccess) return e;
    const int grid = std::max(1, std::min(a.T, sm_count()));
    return launch_pdl(sgc::k_gemv_seg, dim3(grid), dim3(sgc::kThreads), smem, s, a);
}

cudaError_t read_seg_error(unsigned *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_seg_error, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_seg_error, &zero, sizeof(unsigned));
}

}  // namespace zq4
