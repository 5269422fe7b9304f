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
// How, per CTA (one output tile of 128*MB tokens x 256 weight rows, MB = 1
// or 2; K in steps of 64):
//  * warp 0 (one lane): TMA producer into a deep ring of raw stages. Each
//    stage holds the x tile [128*MB x 64] f16, landed with the 128-byte
//    swizzle that is exactly the K-major SW128 operand layout the tensor core
//    reads, and the packed weight tile [256 rows x 8 words].
//  * warps 2..9 (256 threads, one weight row each): dequantize. Exact f16
//    (q - 7) from the packed words, one f16x2 multiply by the group scale
//    (the single rounding of the pages' f16 dequantization, bit-identical to
//    zq4_dequant_f16), reorder into natural k order and store 16-byte chunks
//    into a 2-slot ring of SW128-swizzled B tiles; then fence the generic
//    writes to the async proxy and arrive on the slot's barrier. Scales come
//    as one 16-byte load per row every four stages, a group ahead.
//  * warp 1: allocates 256*MB TMEM columns (MB fp32 accumulators of
//    128 x 256); one lane issues, per K = 16 step, MB tcgen05.mma.cta_group::1
//    .kind::f16 (M = 128, N = 256) that share the B tile, and commits each
//    stage to the raw slot's and the B slot's "empty" barriers.
//  * epilogue: warps 2..9 read their 32-lane quarter and column half of each
//    accumulator with tcgen05.ld, convert to f16 (or silu(g)*u for
//    interleaved gate/up rows) and store.
// The raw ring is deep (4 to 6 stages) because a refill can only be issued
// once the tensor core has finished with a slot, and the copy latency under
// load is several stages' worth of MMA time; the B ring needs only two slots
// (dequantize stage k+1 while the tensor core consumes stage k).
// Every mbarrier wait is bounded; on expiry the kernel records
// ZQ4_DEVERR_WAIT_TIMEOUT, lets its issued copies and MMAs complete, frees
// its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "zq4_async.cuh"
#include "zq4_common.cuh"
#include "zq4_internal.h"

namespace zq4 {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Set (OR) by this file's kernels when an internal wait gives up; read and
// cleared by read_prefill_error().
__device__ unsigned g_prefill_error = 0;

namespace pf {

constexpr int kBM = 128;                          // tokens per MMA (M)
constexpr int kBN = 256;                          // weight rows per tile (MMA N)
constexpr int kBK = 64;                           // K per stage (one 128-byte swizzle row of f16)
constexpr int kABytes = kBM * kBK * 2;            // 16 KB per 128-token block
constexpr int kBBytes = kBN * kBK * 2;            // 32 KB
constexpr int kWBytes = kBN * kBK / 2;            // 8 KB packed
constexpr int kBSlots = 2;
constexpr int kDqWarps = 8;                       // dequant / epilogue warps
constexpr int kThreads = 64 + 32 * kDqWarps;

static_assert(32 * kDqWarps == kBN, "one dequant thread per weight row of the tile");

template <int MB> struct Cfg {
    static constexpr int kRawSlots = MB == 1 ? 6 : 4;
    static constexpr int kRawBytes = MB * kABytes + kWBytes;
    static constexpr int kRawOff = 0;
    static constexpr int kBOff = kRawSlots * kRawBytes;
    static constexpr int kBarOff = kBOff + kBSlots * kBBytes;
    // mbarriers: full/empty per raw slot, full/empty per B slot, accumulator
    static constexpr int kNumBars = 2 * kRawSlots + 2 * kBSlots + 1;
    static constexpr int kSmem = 1024 + kBarOff + 8 * kNumBars + 16;
    static constexpr int kTmemCols = 256 * MB;
    static_assert(kRawBytes % 1024 == 0 && kBBytes % 1024 == 0, "1 KB swizzle alignment");
    static_assert(kSmem <= 227 * 1024, "shared memory");
};

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
    int ksplit;         // CTAs (one cluster) sharing an output tile, each a K range
    int kpart;          // K steps per part (a multiple of 4)
};

// One thread-block-cluster barrier: every thread of every CTA of the cluster
// arrives (release) and waits (acquire).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, int rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d)
{
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Receive slot of a split-K part: [owned chunk][sender][128 rows][32 floats],
// float4 j of row r stored at r*128 + 16*(j ^ (r & 7)) (bank-conflict-free).
constexpr int kRecvSlotBytes = 128 * 32 * 4;

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    return uint32_t(float_to_f16_bits(lo)) | (uint32_t(float_to_f16_bits(hi)) << 16);
}

// Convert 32 consecutive accumulator columns (weight rows n .. n+31) of
// token row m and store them: f16(acc), or f16(silu(g) * u) for interleaved
// gate/up rows (16 outputs).
__device__ __forceinline__ void store_outputs(const PrefillArgs &a, const float (&v)[32], int m, int n)
{
    const bool full = n + 32 <= a.N && a.vec_ok;
    if (!a.gate_up) {
        uint16_t *yo = a.y + size_t(m) * a.y_stride + n;
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
                if (n + i < a.N) yo[i] = float_to_f16_bits(v[i]);
        }
    } else {
        float hv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) hv[i] = silu_f32(v[2 * i]) * v[2 * i + 1];
        uint16_t *yo = a.y + size_t(m) * a.y_stride + (n >> 1);
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
                if (n + 2 * i + 1 < a.N) yo[i] = float_to_f16_bits(hv[i]);
        }
    }
}

// Scales of groups g0 .. g0+7 of one row (zero past G or for a row past N),
// as 8 f16 in a uint4; one 16-byte load when the row allows it.
__device__ __forceinline__ uint4 load_scales8(const uint16_t *srow, int g0, int G, bool row_ok, bool vec)
{
    uint4 r = make_uint4(0, 0, 0, 0);
    if (!row_ok || g0 >= G) return r;
    if (vec) return *reinterpret_cast<const uint4 *>(srow + g0);   // G % 8 == 0: aligned, in range
    uint32_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = g0 + i < G ? ldg_u16(srow + g0 + i) : 0u;
    r.x = v[0] | (v[1] << 16);
    r.y = v[2] | (v[3] << 16);
    r.z = v[4] | (v[5] << 16);
    r.w = v[6] | (v[7] << 16);
    return r;
}

__device__ __forceinline__ uint32_t pick_u32(const uint4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Dequantize four packed words (32 codes, one scale group) of a weight row
// into four 16-byte chunks of the SW128-swizzled B tile row.
__device__ __forceinline__ void dequant4(const uint4 &w4, uint32_t s2, uint8_t *brow, int chunk0, int sw)
{
    const uint32_t words[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t p[4];
        unpack_word_f16x2(words[w], p);          // (q-7) pairs (0,4),(1,5),(2,6),(3,7)
#pragma unroll
        for (int j = 0; j < 4; ++j) p[j] = hmul2(p[j], s2);
        uint4 o;                                  // natural order e0..e7
        o.x = __byte_perm(p[0], p[1], 0x5410);
        o.y = __byte_perm(p[2], p[3], 0x5410);
        o.z = __byte_perm(p[0], p[1], 0x7632);
        o.w = __byte_perm(p[2], p[3], 0x7632);
        *reinterpret_cast<uint4 *>(brow + (((chunk0 + w) ^ sw) << 4)) = o;
    }
}

template <int MB>
__global__ void __launch_bounds__(kThreads, 1) k_prefill(const __grid_constant__ CUtensorMap tm_x,
                                                         const __grid_constant__ CUtensorMap tm_w,
                                                         PrefillArgs a)
{
    using C = Cfg<MB>;
    constexpr int kRaw = C::kRawSlots;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t raw_full0 = sbase + C::kBarOff;        // producer -> dequant (tx bytes)
    const uint32_t raw_empty0 = raw_full0 + 8 * kRaw;     // MMA done -> producer
    const uint32_t b_full0 = raw_empty0 + 8 * kRaw;       // dequant -> MMA
    const uint32_t b_empty0 = b_full0 + 8 * kBSlots;      // MMA done -> dequant
    const uint32_t accum_bar = b_empty0 + 8 * kBSlots;    // all MMAs done -> epilogue
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kBarOff + 8 * C::kNumBars);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KS = a.ksplit, rank = int(blockIdx.x) % KS, tile = int(blockIdx.x) / KS;
    const int m_tile = tile % a.m_tiles, n_tile = tile / a.m_tiles;
    const int m0 = m_tile * kBM * MB, n0 = n_tile * kBN;
    const int ksteps = (a.K + kBK - 1) / kBK;
    const int k_lo = rank * a.kpart, nk = min(ksteps, k_lo + a.kpart) - k_lo;   // this CTA's K steps

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRaw; ++s) {
            mbar_init(raw_full0 + 8 * s, 1);
            mbar_init(raw_empty0 + 8 * s, 1);
        }
        for (int s = 0; s < kBSlots; ++s) {
            mbar_init(b_full0 + 8 * s, kDqWarps);
            mbar_init(b_empty0 + 8 * s, 1);
        }
        mbar_init(accum_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    bool acc_ready = false;                  // dequant/epilogue warps: the accumulator is complete

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        int issued = 0;
        if (lane == 0) {
            for (int i = 0; i < nk; ++i, ++issued) {
                const int s = i % kRaw, ks = k_lo + i;
                if (!mbar_wait(raw_empty0 + 8 * s, ((i / kRaw) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                const uint32_t st = sbase + C::kRawOff + s * C::kRawBytes;
                mbar_arrive_expect_tx(raw_full0 + 8 * s, MB * kABytes + kWBytes);
                tma_load_2d(st + MB * kABytes, &tm_w, ks * (kBK / 8), n0, raw_full0 + 8 * s);
                // the weights are constant; x may be the previous kernel's output
                if (i < kRaw) griddep_wait();
                tma_load_2d(st, &tm_x, ks * kBK, m0, raw_full0 + 8 * s);
            }
            if (!ok) atomicOr(&g_prefill_error, ZQ4_DEVERR_WAIT_TIMEOUT);
            // drain: every issued fill lands before this CTA tears down
            for (int j = std::max(0, issued - kRaw); j < issued; ++j)
                if (!mbar_wait(raw_full0 + 8 * (j % kRaw), (j / kRaw) & 1)) {
                    atomicOr(&g_prefill_error, ZQ4_DEVERR_WAIT_TIMEOUT);
                    break;
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            for (int i = 0; i < nk; ++i) {
                const int s = i % kRaw, b = i % kBSlots;
                // the B slot is filled only after its raw stage landed, so this
                // one wait covers both operands
                if (!mbar_wait(b_full0 + 8 * b, (i / kBSlots) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t at = sbase + C::kRawOff + s * C::kRawBytes;
                const uint32_t bt = sbase + C::kBOff + b * kBBytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    // K = 16 is 32 bytes along the 128-byte swizzled rows
                    const uint64_t bd = smem_desc_sw128(bt + kk * 32);
#pragma unroll
                    for (int mb = 0; mb < MB; ++mb)
                        umma_f16(tmem + uint32_t(mb * kBN), smem_desc_sw128(at + mb * kABytes + kk * 32), bd,
                                 (i | kk) != 0);
                }
                umma_commit(raw_empty0 + 8 * s);     // raw slot free once these MMAs are done
                umma_commit(b_empty0 + 8 * b);       // and the B slot
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
        const bool row_ok = n < a.N;
        const bool vec = (G & 7) == 0;
        const uint16_t *srow = a.scales + size_t(row_ok ? n : 0) * G;
        // conflict-free reads of the packed row (32 bytes): threads whose bit 2
        // is set read the second half first
        const int h0 = (nl >> 2) & 1;
        const int sw = nl & 7;
        griddep_wait();
        griddep_launch_dependents();
        // (k_lo is a multiple of 4 steps, so groups 2*(k_lo + kq) .. +7 are
        // one aligned 16-byte load)
        uint4 sc_next = load_scales8(srow, 2 * k_lo, G, row_ok, vec);
        for (int kq = 0; kq < nk && ok; kq += 4) {
            const uint4 sc_cur = sc_next;           // groups 2(k_lo+kq) .. +7
            sc_next = load_scales8(srow, 2 * (k_lo + kq) + 8, G, row_ok, vec);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = kq + u;
                if (i >= nk) break;
                const int s = i % kRaw, b = i % kBSlots;
                const uint32_t sp = pick_u32(sc_cur, u);           // (group 2ks, group 2ks+1)
                const uint32_t sg0 = __byte_perm(sp, 0, 0x1010), sg1 = __byte_perm(sp, 0, 0x3232);
                const bool got = mbar_wait(raw_full0 + 8 * s, (i / kRaw) & 1) &&
                                 mbar_wait(b_empty0 + 8 * b, ((i / kBSlots) & 1) ^ 1);
                if (!got) {
                    ok = false;
                    break;
                }
                const uint8_t *wp = smem + C::kRawOff + s * C::kRawBytes + MB * kABytes + nl * 32;
                uint8_t *brow = smem + C::kBOff + b * kBBytes + nl * 128;
                const uint4 wa = *reinterpret_cast<const uint4 *>(wp + h0 * 16);
                const uint4 wb = *reinterpret_cast<const uint4 *>(wp + (h0 ^ 1) * 16);
                dequant4(wa, h0 ? sg1 : sg0, brow, 4 * h0, sw);
                dequant4(wb, h0 ? sg0 : sg1, brow, 4 * (h0 ^ 1), sw);
                // make the generic-proxy stores visible to the tensor core, then hand over
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(b_full0 + 8 * b);
            }
        }
        if (!ok && lane == 0) atomicOr(&g_prefill_error, ZQ4_DEVERR_WAIT_TIMEOUT);

        // (tcgen05.ld is warp-collective: the decision to read must be warp-uniform)
        const bool acc_got = mbar_wait(accum_bar, 0);
        acc_ready = __all_sync(0xffffffffu, acc_got && ok);
        if (!acc_ready && lane == 0) atomicOr(&g_prefill_error, ZQ4_DEVERR_WAIT_TIMEOUT);
        tc_fence_after();
    }

    // ---- epilogue: warp w (2..9) reads TMEM lanes 32*(w%4) .. +31 (its 32
    // tokens of each 128-token block) and the column half (w-2)/4, in 32-column
    // chunks. With a K split, chunk c's owner is CTA c % KS of the cluster:
    // the others send their parts into the owner's shared memory (free once
    // every CTA of the cluster has passed the first cluster barrier), and the
    // owner sums the parts in rank order after the second.
    const bool epi = warp >= 2;
    const int q = warp & 3;
    const int cbase = ((warp - 2) >> 2) * (kBN / 2);
    const int row = 32 * q + lane;                           // TMEM lane = token row in the block
    auto slot_addr = [&](int cid, int sender, int owner) {   // in the owner's shared memory
        const int compact = sender < owner ? sender : sender - 1;
        return sbase + uint32_t(((cid / KS) * (KS - 1) + compact) * kRecvSlotBytes + row * 128);
    };
    if (KS > 1) {
        cluster_sync();                                      // every ring of the cluster is idle
        if (epi && acc_ready) {
#pragma unroll 1
            for (int mb = 0; mb < MB; ++mb)
#pragma unroll 1
                for (int c0 = cbase; c0 < cbase + kBN / 2; c0 += 32) {
                    const int cid = mb * (kBN / 32) + c0 / 32, owner = cid % KS;
                    if (owner == rank) continue;
                    float v[32];
                    tmem_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(mb * kBN + c0), v);
                    const uint32_t dst = cluster_addr(slot_addr(cid, rank, owner), owner);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_cluster_v4(dst + uint32_t((j ^ (row & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                                      v[4 * j + 3]);
                }
        }
        cluster_sync();                                      // every part has landed
    }
    if (epi && acc_ready) {
#pragma unroll 1
        for (int mb = 0; mb < MB; ++mb) {
            const int m = m0 + mb * kBM + row;
#pragma unroll 1
            for (int c0 = cbase; c0 < cbase + kBN / 2; c0 += 32) {
                const int cid = mb * (kBN / 32) + c0 / 32;
                if (cid % KS != rank) continue;
                float v[32];
                tmem_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(mb * kBN + c0), v);
                if (KS > 1) {
                    float tot[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) tot[e] = 0.f;
                    for (int sdr = 0; sdr < KS; ++sdr) {             // rank order
                        if (sdr == rank) {
#pragma unroll
                            for (int e = 0; e < 32; ++e) tot[e] += v[e];
                        } else {
                            const uint32_t src = slot_addr(cid, sdr, rank);
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint4 w = lds_v4(src + uint32_t((j ^ (row & 7)) << 4));
                                tot[4 * j] += __uint_as_float(w.x);
                                tot[4 * j + 1] += __uint_as_float(w.y);
                                tot[4 * j + 2] += __uint_as_float(w.z);
                                tot[4 * j + 3] += __uint_as_float(w.w);
                            }
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = tot[e];
                }
                if (m >= a.M || n0 + c0 >= a.N) continue;
                store_outputs(a, v, m, n0 + c0);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols)
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

#ifndef ZQ4_PF_FORCE_MB
#define ZQ4_PF_FORCE_MB 0          // 0: choose per shape; 1 or 2: always that many 128-token blocks
#endif
#ifndef ZQ4_PF_FORCE_KS
#define ZQ4_PF_FORCE_KS 0          // 0: choose per shape; 1 or 2: always split K that many ways
#endif

template <int MB>
static cudaError_t launch_mb(const CUtensorMap &tmx, const CUtensorMap &tmw, const pf::PrefillArgs &a, int n_tiles,
                             cudaStream_t s)
{
    static int smem_set[kMaxDevices] = {};
    auto kern = pf::k_prefill<MB>;
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(kern), pf::Cfg<MB>::kSmem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.m_tiles * n_tiles * a.ksplit));
    cfg.blockDim = dim3(pf::kThreads);
    cfg.dynamicSmemBytes = size_t(pf::Cfg<MB>::kSmem);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;       // the CTAs sharing a tile, adjacent in x
    attr[1].val.clusterDim.x = unsigned(a.ksplit);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.ksplit > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, tmx, tmw, a);
}

// Tile height (MB x 128 tokens) and K split (1 or 2 CTAs of a cluster per
// tile) for a shape, from a cost model fitted to measurements on GB300: a CTA
// costs a fixed ~8 us (TMEM set-up, first-copy latency, epilogue) plus its
// share of the tile's work (35 us for a 256-token tile at K = 3072, 23.3 us
// for a 128-token one: the taller tile halves the dequantization per flop)
// plus ~3 us per 128 tokens for the split's reduction through distributed
// shared memory; a launch costs its number of waves of CTAs times that.
// Splits over 3 or 4 CTAs measured slower (more reduction traffic, and
// 3-CTA clusters leave SMs idle in the GPCs). Every part keeps at least 8 K
// steps and starts on a multiple of 4.
static void choose_tiling(int M, int N, int K, int sms, int *mb_out, int *ks_out, int *kpart_out)
{
    const int n_tiles = (N + pf::kBN - 1) / pf::kBN, ksteps = (K + pf::kBK - 1) / pf::kBK;
    double best = 1e30;
    int bmb = 1, bks = 1;
    for (int mb = 2; mb >= 1; --mb) {
        if (ZQ4_PF_FORCE_MB && mb != ZQ4_PF_FORCE_MB) continue;
        const long tiles = long((M + 128 * mb - 1) / (128 * mb)) * n_tiles;
        const double work = (mb == 2 ? 35.0 : 23.3) * double(K) / 3072.0;
        for (int ks = 1; ks <= 2; ++ks) {
            if (ks > 1 && ksteps / ks < 8) break;
            if (ZQ4_PF_FORCE_KS && ks != ZQ4_PF_FORCE_KS) continue;
            const long waves = (tiles * ks + sms - 1) / sms;
            const double cost = double(waves) * (8.0 + work / ks + 3.0 * mb * (ks - 1));
            if (cost < best - 1e-9) {
                best = cost;
                bmb = mb;
                bks = ks;
            }
        }
    }
    int kpart = (ksteps + bks - 1) / bks;
    kpart = (kpart + 3) / 4 * 4;
    while (bks > 1 && (bks - 1) * kpart >= ksteps) --bks;    // no empty part
    *mb_out = bmb;
    *ks_out = bks;
    *kpart_out = bks > 1 ? kpart : ksteps;
}

cudaError_t launch_prefill(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, uint16_t *y,
                           int M, int N, int K, bool gate_up, cudaStream_t s)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const int n_tiles = (N + pf::kBN - 1) / pf::kBN;
    int MB, KS, kpart;
    choose_tiling(M, N, K, sm_count(), &MB, &KS, &kpart);
    CUtensorMap tmx, tmw;
    const cuuint32_t estr[2] = {1, 1};
    {
        const cuuint64_t dim[2] = {cuuint64_t(K), cuuint64_t(M)};
        const cuuint64_t stride[1] = {cuuint64_t(K) * 2};
        const cuuint32_t box[2] = {pf::kBK, cuuint32_t(pf::kBM * MB)};
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
    a.m_tiles = (M + pf::kBM * MB - 1) / (pf::kBM * MB);
    a.gate_up = gate_up ? 1 : 0;
    a.y_stride = gate_up ? N / 2 : N;
    a.vec_ok = (reinterpret_cast<uintptr_t>(y) & 15) == 0 && a.y_stride % 8 == 0;
    a.ksplit = KS;
    a.kpart = kpart;
    return MB == 2 ? launch_mb<2>(tmx, tmw, a, n_tiles, s) : launch_mb<1>(tmx, tmw, a, n_tiles, s);
}

}  // namespace zq4
