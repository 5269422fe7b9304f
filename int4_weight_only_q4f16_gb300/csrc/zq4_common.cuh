// zq4_common.cuh -- device helpers shared by the zq4 kernels (sm_103a).
//
// The q4f16_1 format ("Zero TVM Documentation", section "Q4F16 quantization
// format"): 8 unsigned 4-bit codes per uint32, element i of a word in bits
// 4i..4i+3, one f16 scale per 32 weights, w = (q - 7) * s.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/zq4.h"

namespace zq4 {

// ---------------------------------------------------------------------------
// Host side: status bookkeeping and device properties
// ---------------------------------------------------------------------------
void set_last_cuda_error(cudaError_t e);
zq4_status cuda_status(cudaError_t e);     // cudaSuccess -> ZQ4_OK, else records + ZQ4_ERR_CUDA
int sm_count();                            // SMs of the current device (cached per device)
// Raise a kernel's dynamic shared memory limit once per (kernel, device).
cudaError_t ensure_smem(const void *kernel, size_t bytes, int *cache_by_device);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na && nb && x < y + nb && y < x + na;
}

// Launch with programmatic dependent launch allowed: the kernel may begin
// while the previous kernel in the stream drains; the kernel itself calls
// griddep_wait() before it touches anything that kernel produced.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// Device side
// ---------------------------------------------------------------------------

// Wait until the previous grid of the stream has completed and its writes
// are visible (no-op when the kernel was not launched early).
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next grid of the stream to start launching.
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Bring [p, p + bytes) into L2 without touching registers or shared memory.
// p must be 16-byte aligned and bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Prefetch the 16-byte-aligned interior of [lo, hi) (addresses) in chunks,
// spread over the calling threads (tid in [0, nthreads)). Never touches a
// byte outside [lo, hi).
__device__ __forceinline__ void prefetch_l2_range(const void *lo, const void *hi, int tid,
                                                  int nthreads)
{
    const uint32_t kChunk = 16384;
    uintptr_t a = (reinterpret_cast<uintptr_t>(lo) + 15) & ~uintptr_t(15);
    uintptr_t b = reinterpret_cast<uintptr_t>(hi) & ~uintptr_t(15);
    if (b <= a) return;
    uintptr_t n = (b - a + kChunk - 1) / kChunk;
    for (uintptr_t i = tid; i < n; i += nthreads) {
        uintptr_t s = a + i * kChunk;
        uintptr_t e = s + kChunk < b ? s + kChunk : b;
        prefetch_l2_bulk(reinterpret_cast<const void *>(s), uint32_t(e - s));
    }
}

// 16-byte read-only global load that does not allocate in L1 (the packed
// weights are streamed exactly once per kernel).
__device__ __forceinline__ uint4 ldg_stream_v4(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint16_t ldg_u16(const uint16_t *p)
{
    uint16_t r;
    asm("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 lds_v4(uint32_t saddr)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(saddr));
    return r;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// (a & MASK) | c in one three-input logic instruction (the compiler left to
// itself splits the two constants over two instructions).
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
    return d;
}

// Unpack one packed word into four f16x2 values holding (q - 7) exactly, as
// the element pairs (0,4), (1,5), (2,6), (3,7) (low half first).
//
// OR-ing a nibble into the mantissa of the f16 1024.0 (0x6400) gives
// 1024 + q (nibble in bits 0..3 of a half) or 1024 + 16 q (bits 4..7); one
// f16x2 subtract, or a multiply-add by 1/16, then removes the bias. Every
// intermediate is a small integer, so each step is exact in f16.
__device__ __forceinline__ void unpack_word_f16x2(uint32_t w, uint32_t p[4])
{
    const uint32_t kMagic = 0x64006400u;       // (1024, 1024)
    const uint32_t kBias = 0x64076407u;        // (1031, 1031)
    const uint32_t kSixteenth = 0x2C002C00u;   // (1/16, 1/16)
    const uint32_t kNeg71 = 0xD470D470u;       // (-71, -71): 1024/16 + 7
    uint32_t w8 = w >> 8;
    p[0] = hsub2(and_or<0x000F000Fu>(w, kMagic), kBias);                 // elements 0, 4
    p[1] = hfma2(and_or<0x00F000F0u>(w, kMagic), kSixteenth, kNeg71);    // elements 1, 5
    p[2] = hsub2(and_or<0x000F000Fu>(w8, kMagic), kBias);                // elements 2, 6
    p[3] = hfma2(and_or<0x00F000F0u>(w8, kMagic), kSixteenth, kNeg71);   // elements 3, 7
}

// Codes of the low 16 bits / high 16 bits of v (each byte holding one code
// in bits 0..3) to an f16x2 of (code / 8): read as e2m3 (sign 0, exponent
// bit = code bit 3, 3 mantissa bits), code c is c/8 exactly for c in 0..15
// (c < 8 are the subnormals c/8, c >= 8 the normals 1 + (c-8)/8). Byte 0
// of the half goes to the low f16.
__device__ __forceinline__ uint32_t e2m3x2_lo(uint32_t v)
{
    uint32_t d;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e2m3x2 %0, l;\n\t}" : "=r"(d) : "r"(v));
    return d;
}

__device__ __forceinline__ uint32_t e2m3x2_hi(uint32_t v)
{
    uint32_t d;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e2m3x2 %0, h;\n\t}" : "=r"(d) : "r"(v));
    return d;
}

// Unpack one packed word into four f16x2 values holding q/8 exactly, as the
// element pairs (0,2), (1,3), (4,6), (5,7) (low half first): one shift and
// two masks put every code alone in a byte, four conversions do the rest.
__device__ __forceinline__ void unpack_word_q8_f16x2(uint32_t w, uint32_t p[4])
{
    const uint32_t lo = w & 0x0F0F0F0Fu;          // codes 0, 2, 4, 6
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;   // codes 1, 3, 5, 7
    p[0] = e2m3x2_lo(lo);                         // elements 0, 2
    p[1] = e2m3x2_lo(hi);                         // elements 1, 3
    p[2] = e2m3x2_hi(lo);                         // elements 4, 6
    p[3] = e2m3x2_hi(hi);                         // elements 5, 7
}

// acc_lo += lo(a) * lo(b), acc_hi += hi(a) * hi(b): f16 operands, exact
// products, fp32 accumulation (one rounding per add).
__device__ __forceinline__ void fma2_f16_f32(uint32_t a, uint32_t b, float &acc_lo, float &acc_hi)
{
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\t"
        "mov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
        : "+f"(acc_lo), "+f"(acc_hi)
        : "r"(a), "r"(b));
}

__device__ __forceinline__ float f16_bits_to_float(uint16_t h)
{
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
    return f;
}

__device__ __forceinline__ uint16_t float_to_f16_bits(float f)
{
    uint16_t h;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(f));
    return h;
}

// silu(z) = z / (1 + e^-z) in fp32.
__device__ __forceinline__ float silu_f32(float z)
{
    return z / (1.0f + __expf(-z));
}

}  // namespace zq4
