// zq4_internal.h -- declarations shared by the zq4 translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/zq4.h"

namespace zq4 {

constexpr int kMaxDevices = 64;

struct DenseArgs {
    const uint32_t *wq;
    const uint16_t *scales;
    const uint16_t *biases;   // MLX affine format only (else unused)
    const uint16_t *x;
    uint16_t *y;
    int M;              // activation rows in this launch (<= the kernel's MT)
    int K;
    int units;          // output columns: N (GEMV) or N/2 (gate_up)
    int units_per_cta;
    int y_stride;       // elements between output rows
};

// GEMV + residual add + RMSNorm (zq4_gemv_add_rmsnorm), one block of tokens.
struct RmsArgs {
    const uint32_t *wq;
    const uint16_t *scales;
    const uint16_t *x;        // [M, K]
    const uint16_t *resid;    // [M, N]
    const uint16_t *gamma;    // [N]
    uint16_t *res_out;        // [M, N] f16(r)
    uint16_t *out;            // [M, N] f16(r / rms * gamma)
    float *r32;               // [M, N] scratch: r in fp32
    unsigned *counter;        // CTAs done (the last one normalises and resets it)
    float eps;
    int M, N, K;
    int units_per_cta;
};

// QKV projection + RoPE + KV append (zq4_qkv_rope_append), one block of tokens.
struct QkvArgs {
    const uint32_t *wq;
    const uint16_t *scales;
    const uint16_t *x;        // [M, K]
    const int32_t *pos;       // [M] RoPE positions
    const int32_t *slot;      // [M] cache rows
    uint16_t *q_out;          // [M, H*D]
    uint16_t *k_cache;        // [n_slots, Hkv*D]
    uint16_t *v_cache;        // [n_slots, Hkv*D]
    int32_t *dev_status;
    double base;
    int M, K, H, Hkv, D, n_slots;
    int units, units_per_cta;
};

struct MoeArgs {
    const uint32_t *wq;
    const uint16_t *scales;
    const uint16_t *biases;   // affine banks only (else nullptr)
    const uint16_t *x;
    uint16_t *y;
    const int32_t *ids;
    const float *route_w;
    int32_t *dev_status;
    int num_experts;
    int T, N, K, top_k;
    int units_per_cta;
};

struct TcArgs {
    const uint32_t *wq;
    const uint16_t *scales;
    const uint16_t *x;
    uint16_t *y;
    int M, N, K;
    int tiles;          // 16-row tiles of W
    int y_stride;       // elements between output rows
    float *y32;                     // fp32 logits [M][y_stride] (argmax epilogue; may be null)
    unsigned long long *amax;       // [M] argmax keys (argmax epilogue; zero on entry, left zero)
    unsigned long long *done;       // CTAs finished (argmax epilogue; zero on entry, left zero)
    int32_t *idx;                   // [M] argmax rows, written by the last CTA
    float *maxval;                  // [M] argmax logits or null, written by the last CTA
    // residual add + RMSNorm epilogue (y = the new residual, f16)
    const uint16_t *resid;          // [M][N]
    const uint16_t *gamma;          // [N]
    uint16_t *out;                  // [M][N] f16(r / rms * gamma), written by the last CTA
    float *r32;                     // [M][N] r in fp32
    float *part;                    // [CTAs][16] each CTA's sum of r^2 per token
    unsigned *counter;              // CTAs done (zero on entry, left zero)
    float eps;
    // QKV + RoPE + KV append epilogue: the maps view W as [heads][2][D/2][K]
    // (a tile = pair rows i0..i0+7 of both halves of one head)
    const int32_t *pos, *slot;      // [M]
    uint16_t *q_out, *k_cache, *v_cache;
    int32_t *dev_status;
    double base;
    int H, Hkv, D, n_slots;
};

size_t smem_per_sm();      // shared memory per SM of the current device (cached)

// zq4_decode_tc.cu
bool decode_tc_supported(int M, int K);
cudaError_t launch_decode_tc(const uint32_t *wq, const uint16_t *scales, const uint16_t *x,
                             uint16_t *y, int M, int N, int K, bool gate_up, cudaStream_t s);
// fp32 logits (y32 may be null) and the per-token argmax in the same launch
// (per block of tokens): work = [M] keys then 8 counters, zero on entry and
// left zero
// GEMV + residual add + RMSNorm on the tensor-core kernel: work = 16 bytes
// of counter (zero on entry, left zero), fp32 r [M][N], then 16 floats per
// 16-row tile of W (the CTAs' partial sums of squares)
cudaError_t launch_decode_tc_addnorm(const uint32_t *wq, const uint16_t *scales, const uint16_t *x,
                                     const uint16_t *resid, const uint16_t *gamma, float eps, uint16_t *res_out,
                                     uint16_t *out, void *work, int M, int N, int K, cudaStream_t s);
// The MoE block on the step kernels' segment loop (zq4_moe_block, zq4_step.cu):
// gate_up + SiLU*mul of every (token, slot) pair into h, down into fp32 z,
// then the weighted combine; each touched expert read once per stage.
bool moe_block_supported(int T, int top_k, int D, int I);
size_t moe_block_work_layout(int T, int top_k, int D, int I, size_t *h_off, size_t *z_off);
cudaError_t launch_moe_block(const uint8_t *gu_seg, const uint8_t *dn_seg, int num_experts, const uint16_t *x,
                             uint16_t *y, int T, int D, int I, const int32_t *ids, const float *route_w, int top_k,
                             void *work, int32_t *dev_status, cudaStream_t s);
// The MLX affine format on the tensor-core kernel (zq4_gemv_affine / _gate_up_silu_affine)
bool decode_tc_affine_supported(int M, int K);
cudaError_t launch_decode_tc_affine(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                                    const uint16_t *x, uint16_t *y, int M, int N, int K, bool gate_up, cudaStream_t s);
// QKV + RoPE + KV append on the tensor-core kernel (zq4_qkv_rope_append)
bool decode_tc_rope_supported(int M, int K, int D);
cudaError_t launch_decode_tc_rope(const QkvArgs &q, cudaStream_t s);
cudaError_t launch_decode_tc_argmax(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, float *y32,
                                    int32_t *idx, float *maxval, unsigned long long *work, int M, int N, int K,
                                    cudaStream_t s);
cudaError_t read_device_error(unsigned *flags, bool clear);

// zq4_decode_seg.cu: decode GEMV / gate_up on the segmented layout, M <= 8
bool seg_gemv_supported(int M, int K);
cudaError_t launch_gemv_seg(const uint8_t *wseg, const uint16_t *x, uint16_t *y, int M, int N, int K,
                            bool gate_up, cudaStream_t s);
cudaError_t read_seg_error(unsigned *flags, bool clear);

// zq4_stack.cu: the persistent decode-step kernel
zq4_status stack_plan_bytes(const zq4_stack_job *jobs, int n_jobs, int M, size_t *bytes);
zq4_status stack_plan_waits(const zq4_stack_job *jobs, int n_jobs, int M, int *order, int *dep);
zq4_status stack_plan_init(const zq4_stack_job *jobs, int n_jobs, int M, void *dev, size_t bytes,
                           zq4_stack_plan *plan, cudaStream_t s);
zq4_status stack_run(const zq4_stack_plan *plan, cudaStream_t s);
zq4_status stack_plan_init_static(const zq4_stack_job *jobs, int n_jobs, int M, zq4_stack_plan *plan,
                                  cudaStream_t s);
cudaError_t read_stack_error(unsigned *flags, bool clear);

// zq4_prefill_tc.cu: the tensor-core GEMM for chunks of kPrefillMinRows or
// more activation rows
constexpr int kPrefillMinRows = 64;
bool prefill_supported(int M, int K);
cudaError_t launch_prefill(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, uint16_t *y,
                           int M, int N, int K, bool gate_up, cudaStream_t s);
cudaError_t read_prefill_error(unsigned *flags, bool clear);

// zq4_decode.cu
int decode_tokens_per_launch(int M, int K);
size_t decode_max_smem();
cudaError_t launch_decode(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases, const uint16_t *x,
                          uint16_t *y, int M, int N, int K, bool gate_up, cudaStream_t s);
cudaError_t launch_moe(const MoeArgs &a, int mode, cudaStream_t s);
size_t moe_smem(int mode, int K, int top_k, bool aff);
cudaError_t launch_qkv_rope(const QkvArgs &a, cudaStream_t s);
cudaError_t launch_add_rmsnorm(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, const uint16_t *resid,
                               const uint16_t *gamma, float eps, uint16_t *res_out, uint16_t *out, void *work, int M,
                               int N, int K, cudaStream_t s);
cudaError_t launch_dequant_f32(const uint32_t *wq, const uint16_t *scales, float *w, int N, int K,
                               cudaStream_t s);
cudaError_t launch_dequant_f16(const uint32_t *wq, const uint16_t *scales, uint16_t *w, int N,
                               int K, cudaStream_t s);
cudaError_t launch_prepare(const uint32_t *wq_src, const uint16_t *sc_src, uint32_t *wq_dst,
                           uint16_t *sc_dst, int N, int K, int interleave, cudaStream_t s);
cudaError_t launch_prepare_segmented(const uint32_t *wq_src, const uint16_t *sc_src, uint8_t *dst, int N, int K,
                                     int interleave, cudaStream_t s);
// bytes of one matrix in the segmented layout (16-row tiles x 256-column segments of 2304 B)
inline size_t segmented_bytes(int N, int K) { return size_t((N + 15) / 16) * size_t(K / 256) * 2304; }

}  // namespace zq4
