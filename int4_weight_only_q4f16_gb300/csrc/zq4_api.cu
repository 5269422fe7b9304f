// zq4_api.cu -- the extern "C" entry points declared in include/zq4.h:
// host-side argument checks, then stream-ordered launches.
#include <algorithm>
#include <atomic>

#include "zq4_common.cuh"
#include "zq4_internal.h"

namespace zq4 {

static thread_local int t_last_cuda_error = 0;

void set_last_cuda_error(cudaError_t e) { t_last_cuda_error = int(e); }

zq4_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return ZQ4_OK;
    set_last_cuda_error(e);
    return ZQ4_ERR_CUDA;
}

int sm_count()
{
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        v = 152;
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

size_t smem_per_sm()
{
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 228 * 1024;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return size_t(v);
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        v <= 0)
        v = 228 * 1024;
    cache[dev].store(v, std::memory_order_relaxed);
    return size_t(v);
}

cudaError_t ensure_smem(const void *kernel, size_t bytes, int *cache_by_device)
{
    // Without the attribute a launch may use 48 KB of shared memory, static
    // and dynamic together; the kernels here have up to a few hundred bytes
    // of static arrays, so the attribute is set for anything above 32 KB.
    if (bytes <= 32 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) {
        auto *slot = reinterpret_cast<std::atomic<int> *>(&cache_by_device[dev]);
        if (size_t(slot->load(std::memory_order_relaxed)) >= bytes) return cudaSuccess;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
        if (e == cudaSuccess) {
            int cur = slot->load(std::memory_order_relaxed);
            while (size_t(cur) < bytes && !slot->compare_exchange_weak(cur, int(bytes))) {
            }
        }
        return e;
    }
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
}

}  // namespace zq4

using namespace zq4;

namespace {

// Shape checks shared by the GEMV-family calls.
zq4_status check_matrix(const void *wq, const void *scales, int N, int K)
{
    if (!wq || !scales) return ZQ4_ERR_NULL;
    if (N <= 0 || K <= 0 || (K % 32) != 0) return ZQ4_ERR_SHAPE;
    if (!aligned16(wq) || !aligned16(scales)) return ZQ4_ERR_ALIGN;
    return ZQ4_OK;
}

size_t wq_bytes(size_t N, size_t K) { return N * (K / 8) * 4; }
size_t sc_bytes(size_t N, size_t K) { return N * (K / 32) * 2; }

}  // namespace

extern "C" {

const char *zq4_status_string(int status)
{
    switch (status) {
    case ZQ4_OK: return "ZQ4_OK";
    case ZQ4_ERR_NULL: return "ZQ4_ERR_NULL: a required pointer is NULL";
    case ZQ4_ERR_SHAPE: return "ZQ4_ERR_SHAPE: a size is out of range";
    case ZQ4_ERR_ALIGN: return "ZQ4_ERR_ALIGN: a pointer is not 16-byte aligned";
    case ZQ4_ERR_FLAGS: return "ZQ4_ERR_FLAGS: unknown mode or flags";
    case ZQ4_ERR_CUDA: return "ZQ4_ERR_CUDA: a CUDA call or launch failed";
    case ZQ4_ERR_UNSUPPORTED: return "ZQ4_ERR_UNSUPPORTED: not handled by this library";
    case ZQ4_ERR_OVERLAP: return "ZQ4_ERR_OVERLAP: input and output buffers overlap";
    default: return "ZQ4: unknown status";
    }
}

int zq4_last_cuda_error(void) { return t_last_cuda_error; }

int zq4_version(void) { return 201; }

zq4_status zq4_gemv(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, uint16_t *y,
                    int M, int N, int K, void *stream)
{
    zq4_status st = check_matrix(wq, scales, N, K);
    if (st != ZQ4_OK) return st;
    if (!x || !y) return ZQ4_ERR_NULL;
    if (M <= 0) return ZQ4_ERR_SHAPE;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(y) & 1)) return ZQ4_ERR_ALIGN;
    if (!prefill_supported(M, K) && size_t(K) * 2 > decode_max_smem()) return ZQ4_ERR_UNSUPPORTED;
    size_t ybytes = size_t(M) * N * 2;
    if (overlap(y, ybytes, wq, wq_bytes(N, K)) || overlap(y, ybytes, scales, sc_bytes(N, K)) ||
        overlap(y, ybytes, x, size_t(M) * K * 2))
        return ZQ4_ERR_OVERLAP;
    if (prefill_supported(M, K))
        return cuda_status(launch_prefill(wq, scales, x, y, M, N, K, false,
                                          static_cast<cudaStream_t>(stream)));
    if (decode_tc_supported(M, K))
        return cuda_status(launch_decode_tc(wq, scales, x, y, M, N, K, false,
                                            static_cast<cudaStream_t>(stream)));
    return cuda_status(launch_decode(wq, scales, nullptr, x, y, M, N, K, false,
                                     static_cast<cudaStream_t>(stream)));
}

zq4_status zq4_qkv_rope_append(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, int M, int K, int H,
                               int H_kv, int D, double rope_base, const int32_t *pos, const int32_t *slot,
                               uint16_t *q_out, uint16_t *k_cache, uint16_t *v_cache, int n_slots,
                               int32_t *dev_status, void *stream)
{
    if (H <= 0 || H_kv <= 0 || D <= 0 || (D & 1) || M <= 0 || n_slots <= 0) return ZQ4_ERR_SHAPE;
    if (D > 512) return ZQ4_ERR_UNSUPPORTED;
    if (!(rope_base > 0.0) || !(rope_base < 1e300)) return ZQ4_ERR_SHAPE;
    const long long Nl = (long long)(H + 2LL * H_kv) * D;
    if (Nl > (1LL << 30) || (long long)n_slots * H_kv * D > (1LL << 40)) return ZQ4_ERR_UNSUPPORTED;
    const int N = int(Nl);
    zq4_status st = check_matrix(wq, scales, N, K);
    if (st != ZQ4_OK) return st;
    if (!x || !pos || !slot || !q_out || !k_cache || !v_cache) return ZQ4_ERR_NULL;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(q_out) & 1) || (reinterpret_cast<uintptr_t>(k_cache) & 1) ||
        (reinterpret_cast<uintptr_t>(v_cache) & 1) || (reinterpret_cast<uintptr_t>(pos) & 3) ||
        (reinterpret_cast<uintptr_t>(slot) & 3) || (reinterpret_cast<uintptr_t>(dev_status) & 3))
        return ZQ4_ERR_ALIGN;
    if (size_t(K) * 2 + 2048 > decode_max_smem()) return ZQ4_ERR_UNSUPPORTED;   // x beside the frequency table
    const size_t qb = size_t(M) * H * D * 2, cb = size_t(n_slots) * H_kv * D * 2;
    const void *ins[5] = {wq, scales, x, pos, slot};
    const size_t inb[5] = {wq_bytes(N, K), sc_bytes(N, K), size_t(M) * K * 2, size_t(M) * 4, size_t(M) * 4};
    const void *outs[3] = {q_out, k_cache, v_cache};
    const size_t outb[3] = {qb, cb, cb};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 5; ++i)
            if (overlap(outs[o], outb[o], ins[i], inb[i])) return ZQ4_ERR_OVERLAP;
        for (int q = o + 1; q < 3; ++q)
            if (overlap(outs[o], outb[o], outs[q], outb[q])) return ZQ4_ERR_OVERLAP;
    }
    QkvArgs a = {};
    a.wq = wq;
    a.scales = scales;
    a.x = x;
    a.pos = pos;
    a.slot = slot;
    a.q_out = q_out;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.dev_status = dev_status;
    a.base = rope_base;
    a.M = M;
    a.K = K;
    a.H = H;
    a.Hkv = H_kv;
    a.D = D;
    a.n_slots = n_slots;
    if (decode_tc_rope_supported(M, K, D))   // the tensor-core kernel, a RoPE pair in one tile (D % 16 == 0)
        return cuda_status(launch_decode_tc_rope(a, static_cast<cudaStream_t>(stream)));
    return cuda_status(launch_qkv_rope(a, static_cast<cudaStream_t>(stream)));
}

size_t zq4_add_rmsnorm_work_bytes(int M, int N)
{
    // counter, fp32 r [M][N], then 16 floats per 16-row tile (the tensor-core
    // kernel's per-CTA sums of squares)
    return M > 0 && N > 0 ? 16 + size_t(M) * N * 4 + size_t((N + 15) / 16) * 64 : 0;
}

zq4_status zq4_gemv_add_rmsnorm(const uint32_t *wq, const uint16_t *scales, const uint16_t *x,
                                const uint16_t *resid, const uint16_t *gamma, float eps, uint16_t *res_out,
                                uint16_t *out, void *work, int M, int N, int K, void *stream)
{
    zq4_status st = check_matrix(wq, scales, N, K);
    if (st != ZQ4_OK) return st;
    if (!x || !resid || !gamma || !res_out || !out || !work) return ZQ4_ERR_NULL;
    if (M <= 0 || !(eps >= 0.f) || !(eps < 3.0e38f)) return ZQ4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(work) || (reinterpret_cast<uintptr_t>(resid) & 1) ||
        (reinterpret_cast<uintptr_t>(gamma) & 1) || (reinterpret_cast<uintptr_t>(res_out) & 1) ||
        (reinterpret_cast<uintptr_t>(out) & 1))
        return ZQ4_ERR_ALIGN;
    const bool tc = decode_tc_supported(std::min(M, 16), K);
    if (!tc && size_t(K) * 2 > decode_max_smem()) return ZQ4_ERR_UNSUPPORTED;
    const size_t mn = size_t(M) * N * 2, wbytes = zq4_add_rmsnorm_work_bytes(M, N);
    const void *ins[5] = {wq, scales, x, resid, gamma};
    const size_t inb[5] = {wq_bytes(N, K), sc_bytes(N, K), size_t(M) * K * 2, mn, size_t(N) * 2};
    const void *outs[3] = {res_out, out, work};
    const size_t outb[3] = {mn, mn, wbytes};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 5; ++i)
            if (overlap(outs[o], outb[o], ins[i], inb[i])) return ZQ4_ERR_OVERLAP;
        for (int q = o + 1; q < 3; ++q)
            if (overlap(outs[o], outb[o], outs[q], outb[q])) return ZQ4_ERR_OVERLAP;
    }
    if (tc)   // the tensor-core kernel with the add + RMSNorm epilogue
        return cuda_status(launch_decode_tc_addnorm(wq, scales, x, resid, gamma, eps, res_out, out, work, M, N, K,
                                                    static_cast<cudaStream_t>(stream)));
    return cuda_status(launch_add_rmsnorm(wq, scales, x, resid, gamma, eps, res_out, out, work, M, N, K,
                                          static_cast<cudaStream_t>(stream)));
}

zq4_status zq4_gemv_argmax(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, float *y32,
                           int32_t *idx, float *maxval, uint64_t *work, int M, int N, int K, void *stream)
{
    zq4_status st = check_matrix(wq, scales, N, K);
    if (st != ZQ4_OK) return st;
    if (!x || !idx || !work) return ZQ4_ERR_NULL;
    if (M <= 0 || M > 64) return ZQ4_ERR_SHAPE;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(y32) & 3) || (reinterpret_cast<uintptr_t>(idx) & 3) ||
        (reinterpret_cast<uintptr_t>(maxval) & 3) || (reinterpret_cast<uintptr_t>(work) & 7))
        return ZQ4_ERR_ALIGN;
    if (!decode_tc_supported(std::min(M, 8), K)) return ZQ4_ERR_UNSUPPORTED;
    const size_t ybytes = y32 ? size_t(M) * N * 4 : 0, wbytes = size_t(M + 8) * 8;
    const void *outs[4] = {y32, idx, maxval, work};
    const size_t obytes[4] = {ybytes, size_t(M) * 4, maxval ? size_t(M) * 4 : 0, wbytes};
    for (int i = 0; i < 4; ++i) {
        if (!obytes[i]) continue;
        if (overlap(outs[i], obytes[i], wq, wq_bytes(N, K)) || overlap(outs[i], obytes[i], scales, sc_bytes(N, K)) ||
            overlap(outs[i], obytes[i], x, size_t(M) * K * 2))
            return ZQ4_ERR_OVERLAP;
        for (int j = 0; j < i; ++j)
            if (obytes[j] && overlap(outs[i], obytes[i], outs[j], obytes[j])) return ZQ4_ERR_OVERLAP;
    }
    return cuda_status(launch_decode_tc_argmax(wq, scales, x, y32, idx, maxval,
                                               reinterpret_cast<unsigned long long *>(work), M, N, K,
                                               static_cast<cudaStream_t>(stream)));
}

zq4_status zq4_gate_up_silu(const uint32_t *wq, const uint16_t *scales, const uint16_t *x,
                            uint16_t *h, int M, int N2, int K, void *stream)
{
    zq4_status st = check_matrix(wq, scales, N2, K);
    if (st != ZQ4_OK) return st;
    if (!x || !h) return ZQ4_ERR_NULL;
    if (M <= 0 || (N2 & 1)) return ZQ4_ERR_SHAPE;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(h) & 1)) return ZQ4_ERR_ALIGN;
    if (!prefill_supported(M, K) && size_t(K) * 2 > decode_max_smem()) return ZQ4_ERR_UNSUPPORTED;
    size_t hbytes = size_t(M) * (N2 / 2) * 2;
    if (overlap(h, hbytes, wq, wq_bytes(N2, K)) || overlap(h, hbytes, scales, sc_bytes(N2, K)) ||
        overlap(h, hbytes, x, size_t(M) * K * 2))
        return ZQ4_ERR_OVERLAP;
    if (prefill_supported(M, K))
        return cuda_status(launch_prefill(wq, scales, x, h, M, N2, K, true,
                                          static_cast<cudaStream_t>(stream)));
    if (decode_tc_supported(M, K))
        return cuda_status(launch_decode_tc(wq, scales, x, h, M, N2, K, true,
                                            static_cast<cudaStream_t>(stream)));
    return cuda_status(launch_decode(wq, scales, nullptr, x, h, M, N2, K, true,
                                     static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------------------
// MLX affine format (value = scale * code + bias, groups of 64)
// ---------------------------------------------------------------------------
namespace {

zq4_status affine_common(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases, const uint16_t *x,
                         const uint16_t *out, int M, int N, int K, size_t out_bytes)
{
    if (!wq || !scales || !biases || !x || !out) return ZQ4_ERR_NULL;
    if (M <= 0 || N <= 0 || K <= 0 || (K % 64) != 0) return ZQ4_ERR_SHAPE;
    if (!aligned16(wq) || !aligned16(x) || (reinterpret_cast<uintptr_t>(scales) & 1) ||
        (reinterpret_cast<uintptr_t>(biases) & 1) || (reinterpret_cast<uintptr_t>(out) & 1))
        return ZQ4_ERR_ALIGN;
    if (size_t(K) * 2 + size_t(K / 32) * 4 > decode_max_smem()) return ZQ4_ERR_UNSUPPORTED;
    const size_t gb = size_t(N) * (K / 64) * 2;
    if (overlap(out, out_bytes, wq, wq_bytes(N, K)) || overlap(out, out_bytes, scales, gb) ||
        overlap(out, out_bytes, biases, gb) || overlap(out, out_bytes, x, size_t(M) * K * 2))
        return ZQ4_ERR_OVERLAP;
    return ZQ4_OK;
}

}  // namespace

zq4_status zq4_gemv_affine(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases, const uint16_t *x,
                           uint16_t *y, int M, int N, int K, void *stream)
{
    const zq4_status st = affine_common(wq, scales, biases, x, y, M, N, K, size_t(M > 0 ? M : 0) * (N > 0 ? N : 0) * 2);
    if (st != ZQ4_OK) return st;
    // the tensor-core kernel reads scales and biases through tensor maps (16-byte bases)
    if (aligned16(scales) && aligned16(biases) && decode_tc_affine_supported(M, K))
        return cuda_status(launch_decode_tc_affine(wq, scales, biases, x, y, M, N, K, false,
                                                   static_cast<cudaStream_t>(stream)));
    return cuda_status(launch_decode(wq, scales, biases, x, y, M, N, K, false, static_cast<cudaStream_t>(stream)));
}

zq4_status zq4_gate_up_silu_affine(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                                   const uint16_t *x, uint16_t *h, int M, int N2, int K, void *stream)
{
    if (N2 > 0 && (N2 & 1)) return ZQ4_ERR_SHAPE;
    const zq4_status st =
        affine_common(wq, scales, biases, x, h, M, N2, K, size_t(M > 0 ? M : 0) * (N2 > 0 ? N2 / 2 : 0) * 2);
    if (st != ZQ4_OK) return st;
    if (aligned16(scales) && aligned16(biases) && decode_tc_affine_supported(M, K))
        return cuda_status(launch_decode_tc_affine(wq, scales, biases, x, h, M, N2, K, true,
                                                   static_cast<cudaStream_t>(stream)));
    return cuda_status(launch_decode(wq, scales, biases, x, h, M, N2, K, true, static_cast<cudaStream_t>(stream)));
}

namespace {

// zq4_moe_gemv and zq4_moe_gemv_affine (biases_bank != nullptr: affine banks).
zq4_status moe_common(const uint32_t *wq_bank, const uint16_t *scales_bank, const uint16_t *biases_bank,
                      int num_experts, const uint16_t *x, uint16_t *y, int T, int N, int K,
                      const int32_t *expert_ids, const float *route_w, int top_k, int mode, int32_t *dev_status,
                      void *stream)
{
    const bool aff = biases_bank != nullptr;
    if (mode != ZQ4_MOE_GATE_UP_SILU && mode != ZQ4_MOE_DOWN_COMBINE) return ZQ4_ERR_FLAGS;
    if (aff) {
        if (!wq_bank || !scales_bank) return ZQ4_ERR_NULL;
        if (N <= 0 || K <= 0 || (K % 64) != 0) return ZQ4_ERR_SHAPE;
        if (!aligned16(wq_bank) || (reinterpret_cast<uintptr_t>(scales_bank) & 1) ||
            (reinterpret_cast<uintptr_t>(biases_bank) & 1))
            return ZQ4_ERR_ALIGN;
    } else {
        zq4_status st = check_matrix(wq_bank, scales_bank, N, K);
        if (st != ZQ4_OK) return st;
    }
    if (!x || !y || !expert_ids) return ZQ4_ERR_NULL;
    if (mode == ZQ4_MOE_DOWN_COMBINE && !route_w) return ZQ4_ERR_NULL;
    if (num_experts <= 0 || T <= 0 || top_k <= 0 || top_k > 32) return ZQ4_ERR_SHAPE;
    if (mode == ZQ4_MOE_GATE_UP_SILU && (N & 1)) return ZQ4_ERR_SHAPE;
    if (T > 65535 || (mode == ZQ4_MOE_GATE_UP_SILU && size_t(T) * top_k > 65535))
        return ZQ4_ERR_UNSUPPORTED;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(y) & 1) ||
        (reinterpret_cast<uintptr_t>(expert_ids) & 3) || (reinterpret_cast<uintptr_t>(route_w) & 3) ||
        (reinterpret_cast<uintptr_t>(dev_status) & 3))
        return ZQ4_ERR_ALIGN;
    const size_t xrows = mode == ZQ4_MOE_GATE_UP_SILU ? size_t(T) : size_t(T) * top_k;
    if (moe_smem(mode, K, top_k, aff) > decode_max_smem()) return ZQ4_ERR_UNSUPPORTED;
    const size_t ybytes = mode == ZQ4_MOE_GATE_UP_SILU ? size_t(T) * top_k * (N / 2) * 2
                                                       : size_t(T) * N * 2;
    const size_t E = size_t(num_experts);
    const size_t sbytes = aff ? E * size_t(N) * (K / 64) * 2 : E * sc_bytes(N, K);
    if (overlap(y, ybytes, wq_bank, E * wq_bytes(N, K)) || overlap(y, ybytes, scales_bank, sbytes) ||
        (aff && overlap(y, ybytes, biases_bank, sbytes)) ||
        overlap(y, ybytes, x, xrows * K * 2) ||
        overlap(y, ybytes, expert_ids, size_t(T) * top_k * 4))
        return ZQ4_ERR_OVERLAP;
    MoeArgs a = {};
    a.wq = wq_bank;
    a.scales = scales_bank;
    a.biases = biases_bank;
    a.x = x;
    a.y = y;
    a.ids = expert_ids;
    a.route_w = route_w;
    a.dev_status = dev_status;
    a.num_experts = num_experts;
    a.T = T;
    a.N = N;
    a.K = K;
    a.top_k = top_k;
    return cuda_status(launch_moe(a, mode, static_cast<cudaStream_t>(stream)));
}

}  // namespace

zq4_status zq4_moe_gemv(const uint32_t *wq_bank, const uint16_t *scales_bank, int num_experts,
                        const uint16_t *x, uint16_t *y, int T, int N, int K,
                        const int32_t *expert_ids, const float *route_w, int top_k, int mode,
                        int32_t *dev_status, void *stream)
{
    return moe_common(wq_bank, scales_bank, nullptr, num_experts, x, y, T, N, K, expert_ids, route_w, top_k, mode,
                      dev_status, stream);
}

zq4_status zq4_moe_gemv_affine(const uint32_t *wq_bank, const uint16_t *scales_bank, const uint16_t *biases_bank,
                               int num_experts, const uint16_t *x, uint16_t *y, int T, int N, int K,
                               const int32_t *expert_ids, const float *route_w, int top_k, int mode,
                               int32_t *dev_status, void *stream)
{
    if (!biases_bank) return ZQ4_ERR_NULL;
    return moe_common(wq_bank, scales_bank, biases_bank, num_experts, x, y, T, N, K, expert_ids, route_w, top_k,
                      mode, dev_status, stream);
}

size_t zq4_moe_block_work_bytes(int T, int top_k, int D, int I)
{
    if (T <= 0 || top_k <= 0 || D <= 0 || I <= 0) return 0;
    return moe_block_work_layout(T, top_k, D, I, nullptr, nullptr);
}

zq4_status zq4_moe_block(const void *gu_seg, const void *dn_seg, int num_experts, const uint16_t *x, uint16_t *y,
                         int T, int D, int I, const int32_t *expert_ids, const float *route_w, int top_k, void *work,
                         size_t work_bytes, int32_t *dev_status, void *stream)
{
    if (!gu_seg || !dn_seg || !x || !y || !expert_ids || !route_w || !work) return ZQ4_ERR_NULL;
    if (num_experts <= 0 || T <= 0 || top_k <= 0 || top_k > 32 || D <= 0 || I <= 0 || D % 256 || I % 256)
        return ZQ4_ERR_SHAPE;
    if (!moe_block_supported(T, top_k, D, I)) return ZQ4_ERR_UNSUPPORTED;
    size_t h_off, z_off;
    const size_t need = moe_block_work_layout(T, top_k, D, I, &h_off, &z_off);
    if (work_bytes < need) return ZQ4_ERR_SHAPE;
    if (!aligned16(gu_seg) || !aligned16(dn_seg) || !aligned16(x) || !aligned16(work) ||
        (reinterpret_cast<uintptr_t>(y) & 1) || (reinterpret_cast<uintptr_t>(expert_ids) & 3) ||
        (reinterpret_cast<uintptr_t>(route_w) & 3) || (reinterpret_cast<uintptr_t>(dev_status) & 3))
        return ZQ4_ERR_ALIGN;
    const size_t E = size_t(num_experts), P = size_t(T) * top_k;
    const void *ins[5] = {gu_seg, dn_seg, x, expert_ids, route_w};
    const size_t inb[5] = {E * segmented_bytes(2 * I, D), E * segmented_bytes(D, I), size_t(T) * D * 2, P * 4, P * 4};
    const size_t yb = size_t(T) * D * 2;
    for (int i = 0; i < 5; ++i)
        if (overlap(y, yb, ins[i], inb[i]) || overlap(work, need, ins[i], inb[i])) return ZQ4_ERR_OVERLAP;
    if (overlap(y, yb, work, need)) return ZQ4_ERR_OVERLAP;
    return cuda_status(launch_moe_block(static_cast<const uint8_t *>(gu_seg), static_cast<const uint8_t *>(dn_seg),
                                        num_experts, x, y, T, D, I, expert_ids, route_w, top_k, work, dev_status,
                                        static_cast<cudaStream_t>(stream)));
}

zq4_status zq4_device_errors(uint32_t *flags, int clear)
{
    if (!flags) return ZQ4_ERR_NULL;
    unsigned v = 0, vp = 0, vk = 0, vs = 0;
    zq4_status st = cuda_status(read_device_error(&v, clear != 0));
    if (st == ZQ4_OK) st = cuda_status(read_prefill_error(&vp, clear != 0));
    if (st == ZQ4_OK) st = cuda_status(read_stack_error(&vk, clear != 0));
    if (st == ZQ4_OK) st = cuda_status(read_seg_error(&vs, clear != 0));
    *flags = v | vp | vk | vs;
    return st;
}

zq4_status zq4_prepare_weight(const uint32_t *wq_src, const uint16_t *scales_src,
                              uint32_t *wq_dst, uint16_t *scales_dst, int N, int K, int flags,
                              void *stream)
{
    if (flags & ~(ZQ4_PREP_CONCAT_TO_INTERLEAVED | ZQ4_PREP_SEGMENTED)) return ZQ4_ERR_FLAGS;
    zq4_status st = check_matrix(wq_src, scales_src, N, K);
    if (st != ZQ4_OK) return st;
    const bool interleave = (flags & ZQ4_PREP_CONCAT_TO_INTERLEAVED) != 0;
    if (flags & ZQ4_PREP_SEGMENTED) {
        if (!wq_dst) return ZQ4_ERR_NULL;
        if (scales_dst) return ZQ4_ERR_FLAGS;               // the scales travel inside wq_dst
        if (K % 256 != 0 || (interleave && (N & 1))) return ZQ4_ERR_SHAPE;
        if (!aligned16(wq_dst)) return ZQ4_ERR_ALIGN;
        const size_t db = segmented_bytes(N, K);
        if (overlap(wq_dst, db, wq_src, wq_bytes(N, K)) || overlap(wq_dst, db, scales_src, sc_bytes(N, K)))
            return ZQ4_ERR_OVERLAP;
        return cuda_status(launch_prepare_segmented(wq_src, scales_src, reinterpret_cast<uint8_t *>(wq_dst), N, K,
                                                    interleave, static_cast<cudaStream_t>(stream)));
    }
    if (!wq_dst || !scales_dst) return ZQ4_ERR_NULL;
    if (!aligned16(wq_dst) || !aligned16(scales_dst)) return ZQ4_ERR_ALIGN;
    if (flags == ZQ4_PREP_CONCAT_TO_INTERLEAVED && (N & 1)) return ZQ4_ERR_SHAPE;
    const size_t wb = wq_bytes(N, K), sb = sc_bytes(N, K);
    if (overlap(wq_dst, wb, wq_src, wb) || overlap(wq_dst, wb, scales_src, sb) ||
        overlap(scales_dst, sb, wq_src, wb) || overlap(scales_dst, sb, scales_src, sb) ||
        overlap(wq_dst, wb, scales_dst, sb))
        return ZQ4_ERR_OVERLAP;
    return cuda_status(launch_prepare(wq_src, scales_src, wq_dst, scales_dst, N, K, interleave,
                                      static_cast<cudaStream_t>(stream)));
}

size_t zq4_segmented_bytes(int N, int K)
{
    if (N <= 0 || K <= 0 || K % 256 != 0) return 0;
    return segmented_bytes(N, K);
}

zq4_status zq4_dequant_f32(const uint32_t *wq, const uint16_t *scales, float *w, int N, int K,
                           void *stream)
{
    zq4_status st = check_matrix(wq, scales, N, K);
    if (st != ZQ4_OK) return st;
    if (!w) return ZQ4_ERR_NULL;
    if (!aligned16(w)) return ZQ4_ERR_ALIGN;
    return cuda_status(launch_dequant_f32(wq, scales, w, N, K, static_cast<cudaStream_t>(stream)));
}

zq4_status zq4_dequant_f16(const uint32_t *wq, const uint16_t *scales, uint16_t *w, int N, int K,
                           void *stream)
{
    zq4_status st = check_matrix(wq, scales, N, K);
    if (st != ZQ4_OK) return st;
    if (!w) return ZQ4_ERR_NULL;
    if (!aligned16(w)) return ZQ4_ERR_ALIGN;
    return cuda_status(launch_dequant_f16(wq, scales, w, N, K, static_cast<cudaStream_t>(stream)));
}

static zq4_status gemv_seg_common(const uint32_t *wseg, const uint16_t *x, uint16_t *y, int M, int N, int K,
                                  bool gate_up, void *stream)
{
    if (!wseg || !x || !y) return ZQ4_ERR_NULL;
    if (M <= 0 || N <= 0 || K <= 0 || K % 256 != 0 || (gate_up && (N & 1))) return ZQ4_ERR_SHAPE;
    if (!aligned16(wseg) || !aligned16(x) || (reinterpret_cast<uintptr_t>(y) & 1)) return ZQ4_ERR_ALIGN;
    if (!seg_gemv_supported(M, K)) return ZQ4_ERR_UNSUPPORTED;
    const size_t yb = size_t(M) * (gate_up ? N / 2 : N) * 2;
    if (overlap(y, yb, wseg, segmented_bytes(N, K)) || overlap(y, yb, x, size_t(M) * K * 2)) return ZQ4_ERR_OVERLAP;
    return cuda_status(launch_gemv_seg(reinterpret_cast<const uint8_t *>(wseg), x, y, M, N, K, gate_up,
                                       static_cast<cudaStream_t>(stream)));
}

zq4_status zq4_gemv_seg(const uint32_t *wseg, const uint16_t *x, uint16_t *y, int M, int N, int K, void *stream)
{
    return gemv_seg_common(wseg, x, y, M, N, K, false, stream);
}

zq4_status zq4_gate_up_silu_seg(const uint32_t *wseg, const uint16_t *x, uint16_t *h, int M, int N2, int K,
                                void *stream)
{
    return gemv_seg_common(wseg, x, h, M, N2, K, true, stream);
}

zq4_status zq4_stack_plan_bytes(const zq4_stack_job *jobs, int n_jobs, int M, size_t *bytes)
{
    return stack_plan_bytes(jobs, n_jobs, M, bytes);
}

zq4_status zq4_stack_plan_waits(const zq4_stack_job *jobs, int n_jobs, int M, int *order, int *dep)
{
    return stack_plan_waits(jobs, n_jobs, M, order, dep);
}

zq4_status zq4_stack_plan_init(const zq4_stack_job *jobs, int n_jobs, int M, void *dev, size_t bytes,
                               zq4_stack_plan *plan, void *stream)
{
    return stack_plan_init(jobs, n_jobs, M, dev, bytes, plan, static_cast<cudaStream_t>(stream));
}

zq4_status zq4_stack_run(const zq4_stack_plan *plan, void *stream)
{
    return stack_run(plan, static_cast<cudaStream_t>(stream));
}

zq4_status zq4_stack_plan_set_wait_limit(zq4_stack_plan *plan, unsigned long long ns)
{
    if (!plan) return ZQ4_ERR_NULL;
    plan->wait_ns = ns ? ns : 2000000000ull;   // the default: 2 s
    return ZQ4_OK;
}

zq4_status zq4_stack_plan_init_static(const zq4_stack_job *jobs, int n_jobs, int M, zq4_stack_plan *plan,
                                      void *stream)
{
    return stack_plan_init_static(jobs, n_jobs, M, plan, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
