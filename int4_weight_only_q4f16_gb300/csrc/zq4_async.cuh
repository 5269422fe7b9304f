// zq4_async.cuh -- asynchronous-copy, mbarrier and warp-MMA helpers shared by
// the zq4 tensor-core kernels (sm_103a). Every wait here is bounded in time:
// a kernel that sees mbar_wait() return false records an error flag, stops
// issuing work, lets the copies it issued land and returns.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace zq4 {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s

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

// Wait for the phase of the given parity to complete; false once the wait
// has lasted longer than kWaitLimitNs.
__device__ __forceinline__ bool mbar_try(uint32_t addr, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    return done != 0;
}

static __device__ __noinline__ bool mbar_wait_slow(uint32_t addr, uint32_t parity)
{
    const unsigned long long t0 = globaltimer();
    for (unsigned i = 0;; ++i) {
        if (mbar_try(addr, parity)) return true;
        if ((i & 255u) == 255u && globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

// One try inline (the phase is usually complete by the time it is waited
// for), the bounded loop out of line.
__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity)
{
    return mbar_try(addr, parity) || mbar_wait_slow(addr, parity);
}

// Bring the box at (x, y) of a tensor map into L2 (no shared memory).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// 2D tensor-map TMA load of one box at (x, y) into shared memory, completion
// (transaction bytes) on the mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t mbar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar)
        : "memory");
}

// Contiguous bulk copy global -> shared (both 16-byte aligned, bytes a
// multiple of 16), completion (transaction bytes) on the mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(mbar)
        : "memory");
}

// D = A * B + C, m16n8k16, f16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                         const float (&c)[4])
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

// Four 8x8 b16 matrices from shared memory: lanes 8i..8i+7 give the row
// addresses of matrix i; lane (r = lane/4, t = lane%4) receives the 32-bit
// word t of row r of each matrix.
__device__ __forceinline__ uint4 ldmatrix_x4(uint32_t saddr)
{
    uint4 v;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(saddr));
    return v;
}

}  // namespace zq4
