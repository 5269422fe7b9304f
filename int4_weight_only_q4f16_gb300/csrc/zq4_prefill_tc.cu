// zq4_prefill_tc.cu -- the prefill-chunk GEMM (M >= 64) on the 5th-generation
// tensor cores: y[M,N] = x[M,K] * W^T with W in q4f16_1, fp32 accumulation
// in tensor memory.
//
// What it computes: the same fused dequantize + NT matmul as the decode path
// ("Zero TVM Documentation", section "Q4F16 quantization format" and card 5
// "int4 Matmul"; the gate_up + SiLU*mul epilogue of card 6 "Fused FFN"), for
// a chunk of many tokens, where the work is a dense contraction ("Zero-TVM
// benchmarks", the matrix-unit GEMM sections: weights dequantized into shared
// memory and fed to the matrix units with f32 accumulation).
//
// How, per CTA (one output tile of 128 tokens x 256 weight rows; K in steps
// of 64 through a 3-stage shared-memory ring):
//  * warp 0 (one lane): TMA producer. The x tile [128 x 64] f16 arrives with
//    the 128-byte swizzle, which is exactly the K-major SW128 operand layout
//    the tensor core reads; the packed weight tile [256 rows x 8 words] lands
//    dense next to it.
//  * warps 2..5 (128 threads): dequantize. Each thread takes two weight rows:
//    exact f16 (q - 7) from the packed words, one f16x2 multiply by the group
//    scale (the single rounding of the pages' f16 dequantization formula,
//    bit-identical to zq4_dequant_f16), reorder into natural k order and store
//    16-byte chunks into the SW128-swizzled B tile; then fence the generic
//    writes to the async proxy and arrive on the stage's barrier.
//  * warp 1: allocates 256 TMEM columns (the 128 x 256 fp32 accumulator); one
//    lane issues four tcgen05.mma.cta_group::1.kind::f16 (M=128, N=256, K=16)
//    per stage and commits them to the stage's "empty" barrier, which frees
//    the stage for the producer when the tensor core is done with it.
//  * epilogue: warps 2..5 read their 32-lane quarter of the accumulator with
//    tcgen05.ld, convert to f16 (or silu(g)*u for interleaved gate/up rows)
//    and store.
// Every mbarrier wait is bounded; on expiry the kernel records
// ZQ4_DEVERR_WAIT_TIMEOUT, lets its issued copies and MMAs complete, frees
// its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "zq4_common.cuh"
#include "zq4_internal.h"

namespace zq4 {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Set (OR) by this file's kernels when an internal wait gives up; read and
// cleared by read_prefill_error().
__device__ unsigned g_prefill_error = 0;

namespace pf {

constexpr int kBM = 128;                          // tokens per tile (MMA M)
constexpr int kBN = 256;                          // weight rows per tile (MMA N)
constexpr int kBK = 64;                           // K per stage (one 128-byte swizzle row of f16)
constexpr int kStages = 3;
constexpr int kABytes = kBM * kBK * 2;            // 16 KB
constexpr int kBBytes = kBN * kBK * 2;            // 32 KB
constexpr int kWBytes = kBN * kBK / 2;            // 8 KB packed
constexpr int kStageBytes = kABytes + kBBytes + kWBytes;
constexpr int kDqWarps = 8;                     // dequant / epilogue warps
constexpr int kThreads = 64 + 32 * kDqWarps;
constexpr int kTmemCols = 256;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

static_assert(kStageBytes % 1024 == 0, "stages keep the 1 KB swizzle alignment");
static_assert(32 * kDqWarps == kBN, "one dequant thread per weight row of the tile");

__device__ __forceinline__ unsigned long long globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t addr, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t addr)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(addr) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t addr, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(addr), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity)
{
    const unsigned long long t0 = globaltimer();
    for (unsigned i = 0;; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 255u) == 255u && globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t mbar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar)
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile with the
// 128-byte swizzle: rows of 128 B, 8-row atoms 1024 B apart (stride byte
// offset), leading byte offset unused for this layout, descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFFu) >> 4);          // start address
    d |= uint64_t(1) << 16;                          // leading byte offset (16 B, unused)
    d |= uint64_t(1024 >> 4) << 32;                  // stride byte offset: 1024 B
    d |= uint64_t(1) << 46;                          // descriptor version
    d |= uint64_t(2) << 61;                          // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: D f32, A and B f16, both K-major,
// N = kBN, M = kBM.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | (uint32_t(kBN >> 3) << 17) |
                            (uint32_t(kBM >> 4) << 24);

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

struct PrefillArgs {
    const uint16_t *scales;
    uint16_t *y;
    int M, N, K;
    int m_tiles;
    int y_stride;       // elements between output rows
    int gate_up;        // 1: rows interleaved gate/up, output silu(g)*u
    int vec_ok;         // 1: y and y_stride allow 16-byte stores
};

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    return uint32_t(float_to_f16_bits(lo)) | (uint32_t(float_to_f16_bits(hi)) << 16);
}

// Shared layout: [ring: kStages x (A | B | Wp)] [mbarriers] [tmem address]
constexpr int kBarOff = kStages * kStageBytes;

__global__ void __launch_bounds__(kThreads, 1) k_prefill(const __grid_constant__ CUtensorMap tm_x,
                                                         const __grid_constant__ CUtensorMap tm_w,
                                                         PrefillArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t full_tma0 = sbase + kBarOff;           // producer -> dequant
    const uint32_t full_b0 = full_tma0 + 8 * kStages;     // dequant -> MMA
    const uint32_t empty0 = full_b0 + 8 * kStages;        // MMA -> producer
    const uint32_t accum_bar = empty0 + 8 * kStages;      // MMA -> epilogue
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kBarOff + 8 * (3 * kStages + 1));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tile = blockIdx.x % a.m_tiles, n_tile = blockIdx.x / a.m_tiles;
    const int m0 = m_tile * kBM, n0 = n_tile * kBN;
    const int ksteps = (a.K + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_tma0 + 8 * s, 1);
            mbar_init(full_b0 + 8 * s, kDqWarps);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(accum_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        int issued = 0;
        if (lane == 0) {
            for (int ks = 0; ks < ksteps; ++ks, ++issued) {
                const int s = ks % kStages;
                if (!mbar_wait(empty0 + 8 * s, ((ks / kStages) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                const uint32_t st = sbase + s * kStageBytes;
                mbar_arrive_expect_tx(full_tma0 + 8 * s, kABytes + kWBytes);
                tma_load_2d(st + kABytes + kBBytes, &tm_w, ks * (kBK / 8), n0, full_tma0 + 8 * s);
                // the weights are constant; x may be the previous kernel's output
                if (ks < kStages) griddep_wait();
                tma_load_2d(st, &tm_x, ks * kBK, m0, full_tma0 + 8 * s);
            }
            if (!ok) atomicOr(&g_prefill_error, ZQ4_DEVERR_WAIT_TIMEOUT);
            // drain: every issued fill lands before this CTA tears down
            for (int j = std::max(0, issued - kStages); j < issued; ++j)
                if (!mbar_wait(full_tma0 + 8 * (j % kStages), (j / kStages) & 1)) {
                    atomicOr(&g_prefill_error, ZQ4_DEVERR_WAIT_TIMEOUT);
                    break;
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            for (int ks = 0; ks < ksteps; ++ks) {
                const int s = ks % kStages;
                if (!mbar_wait(full_b0 + 8 * s, (ks / kStages) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t st = sbase + s * kStageBytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    // K = 16 is 32 bytes along the 128-byte swizzled row
                    const uint64_t ad = smem_desc_sw128(st + kk * 32);
                    const uint64_t bd = smem_desc_sw128(st + kABytes + kk * 32);
                    umma_f16(tmem, ad, bd, (ks | kk) != 0);
                }
                umma_commit(empty0 + 8 * s);         // stage free once these MMAs are done
            }
            if (!ok) atomicOr(&g_prefill_error, ZQ4_DEVERR_WAIT_TIMEOUT);
            umma_commit(accum_bar);                  // all issued MMAs done -> epilogue
        }
        __syncwarp();
    } else {
        // ---------------- dequant, then epilogue (warps 2 .. 2+kDqWarps) ----------------
        const int nl = threadIdx.x - 64;             // weight row of the tile owned by this thread
        const int n = n0 + nl;
        const int G = a.K >> 5;
        const uint16_t *srow = a.scales + size_t(n < a.N ? n : 0) * G;
        griddep_wait();
        griddep_launch_dependents();
        uint32_t scn[2] = {0, 0};                    // scales of the next stage's two groups
        if (n < a.N) {
            scn[0] = ldg_u16(srow);
            if (G > 1) scn[1] = ldg_u16(srow + 1);
        }
        for (int ks = 0; ks < ksteps; ++ks) {
            const int s = ks % kStages;
            uint32_t sc2[2] = {scn[0] | (scn[0] << 16), scn[1] | (scn[1] << 16)};
            if (n < a.N) {                           // prefetch the following stage's scales
                const int g0 = 2 * ks + 2;
                scn[0] = g0 < G ? ldg_u16(srow + g0) : 0;
                scn[1] = g0 + 1 < G ? ldg_u16(srow + g0 + 1) : 0;
            }
            if (!mbar_wait(full_tma0 + 8 * s, (ks / kStages) & 1)) {
                ok = false;
                break;
            }
            const uint8_t *wp = smem + s * kStageBytes + kABytes + kBBytes;
            uint8_t *bt = smem + s * kStageBytes + kABytes;
            const uint4 w03 = *reinterpret_cast<const uint4 *>(wp + nl * 32);
            const uint4 w47 = *reinterpret_cast<const uint4 *>(wp + nl * 32 + 16);
            const uint32_t words[8] = {w03.x, w03.y, w03.z, w03.w, w47.x, w47.y, w47.z, w47.w};
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                uint32_t p[4];
                unpack_word_f16x2(words[w], p);          // (q-7) pairs (0,4),(1,5),(2,6),(3,7)
#pragma unroll
                for (int j = 0; j < 4; ++j) p[j] = hmul2(p[j], sc2[w >> 2]);
                uint4 o;                                  // natural order e0..e7
                o.x = __byte_perm(p[0], p[1], 0x5410);
                o.y = __byte_perm(p[2], p[3], 0x5410);
                o.z = __byte_perm(p[0], p[1], 0x7632);
                o.w = __byte_perm(p[2], p[3], 0x7632);
                *reinterpret_cast<uint4 *>(bt + nl * 128 + ((w ^ (nl & 7)) << 4)) = o;
            }
            // make the generic-proxy stores visible to the tensor core, then hand over
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(full_b0 + 8 * s);
        }
        if (!ok && lane == 0) atomicOr(&g_prefill_error, ZQ4_DEVERR_WAIT_TIMEOUT);

        // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 (its 32 tokens) and
        // the column half (w-2)/4 of the tile
        // (tcgen05.ld is warp-collective: the decision to read must be warp-uniform)
        const bool got = mbar_wait(accum_bar, 0);
        const bool acc_ready = __all_sync(0xffffffffu, got && ok);
        if (!acc_ready && lane == 0) atomicOr(&g_prefill_error, ZQ4_DEVERR_WAIT_TIMEOUT);
        tc_fence_after();
        const int q = warp & 3;
        const int cbase = ((warp - 2) >> 2) * (kBN / 2);
        const int m = m0 + 32 * q + lane;
        if (acc_ready) {
#pragma unroll 1
            for (int c0 = cbase; c0 < cbase + kBN / 2; c0 += 32) {
                float v[32];
                tmem_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(c0), v);
                if (m >= a.M || n0 + c0 >= a.N) continue;
                const bool full = n0 + c0 + 32 <= a.N && a.vec_ok;
                if (!a.gate_up) {
                    uint16_t *yo = a.y + size_t(m) * a.y_stride + n0 + c0;
                    if (full) {
#pragma unroll
                        for (int i = 0; i < 32; i += 8) {
                            uint4 o;
                            o.x = pack_f16x2(v[i], v[i + 1]);
                            o.y = pack_f16x2(v[i + 2], v[i + 3]);
                            o.z = pack_f16x2(v[i + 4], v[i + 5]);
                            o.w = pack_f16x2(v[i + 6], v[i + 7]);
                            *reinterpret_cast<uint4 *>(yo + i) = o;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (n0 + c0 + i < a.N) yo[i] = float_to_f16_bits(v[i]);
                    }
                } else {
                    float hv[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) hv[i] = silu_f32(v[2 * i]) * v[2 * i + 1];
                    uint16_t *yo = a.y + size_t(m) * a.y_stride + ((n0 + c0) >> 1);
                    if (full) {
#pragma unroll
                        for (int i = 0; i < 16; i += 8) {
                            uint4 o;
                            o.x = pack_f16x2(hv[i], hv[i + 1]);
                            o.y = pack_f16x2(hv[i + 2], hv[i + 3]);
                            o.z = pack_f16x2(hv[i + 4], hv[i + 5]);
                            o.w = pack_f16x2(hv[i + 6], hv[i + 7]);
                            *reinterpret_cast<uint4 *>(yo + i) = o;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (n0 + c0 + 2 * i + 1 < a.N) yo[i] = float_to_f16_bits(hv[i]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace pf

bool prefill_supported(int M, int K)
{
    return M >= kPrefillMinRows && K % 32 == 0 && tensor_map_encoder() != nullptr;
}

cudaError_t read_prefill_error(unsigned *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_prefill_error, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(unsigned));
}

cudaError_t launch_prefill(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, uint16_t *y,
                           int M, int N, int K, bool gate_up, cudaStream_t s)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap tmx, tmw;
    const cuuint32_t estr[2] = {1, 1};
    {
        const cuuint64_t dim[2] = {cuuint64_t(K), cuuint64_t(M)};
        const cuuint64_t stride[1] = {cuuint64_t(K) * 2};
        const cuuint32_t box[2] = {pf::kBK, pf::kBM};
        if (enc(&tmx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(x), dim, stride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dim[2] = {cuuint64_t(K / 8), cuuint64_t(N)};
        const cuuint64_t stride[1] = {cuuint64_t(K / 2)};
        const cuuint32_t box[2] = {pf::kBK / 8, pf::kBN};
        if (enc(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t *>(wq), dim, stride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    pf::PrefillArgs a;
    a.scales = scales;
    a.y = y;
    a.M = M;
    a.N = N;
    a.K = K;
    a.m_tiles = (M + pf::kBM - 1) / pf::kBM;
    a.gate_up = gate_up ? 1 : 0;
    a.y_stride = gate_up ? N / 2 : N;
    a.vec_ok = (reinterpret_cast<uintptr_t>(y) & 15) == 0 && a.y_stride % 8 == 0;
    const int n_tiles = (N + pf::kBN - 1) / pf::kBN;
    const size_t smem = 1024 + pf::kBarOff + 8 * (3 * pf::kStages + 1) + 16;
    static int smem_set[kMaxDevices] = {};
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(pf::k_prefill), smem, smem_set);
    if (e != cudaSuccess) return e;
    return launch_pdl(pf::k_prefill, dim3(a.m_tiles * n_tiles), dim3(pf::kThreads), smem, s, tmx, tmw, a);
}

}  // namespace zq4
