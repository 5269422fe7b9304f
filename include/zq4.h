/*
 * zq4.h -- C ABI of the q4f16_1 fused dequantize + NT matmul library for
 * NVIDIA GB300 (sm_103a).
 *
 * The format ("Zero TVM Documentation", section "Q4F16 quantization
 * format"): a weight matrix W of N rows and K columns (K along the reduction)
 * is stored as
 *   wq     uint32 [N, K/8]   8 unsigned 4-bit codes per word; element i of a
 *                            word (i = 0..7, least significant nibble first)
 *                            is column 8*word_index + i;
 *   scales f16    [N, K/32]  one scale per 32 consecutive columns;
 * and the weight value is w[n,k] = (q[n,k] - 7) * scales[n, k/32].
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a DEVICE pointer to memory the caller allocated
 *     and owns; the library allocates nothing and keeps no pointer after the
 *     call returns. f16 data is passed as uint16_t (IEEE binary16 bits).
 *   - Row-major, densely packed: row r of a [R, C] array starts at element
 *     r*C. No strides.
 *   - K must be a positive multiple of 32 (the group size). wq, scales and
 *     the activation input must start on a 16-byte boundary.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *     call is asynchronous and stream-ordered; none synchronises the host.
 *     Outputs are valid once the stream reaches the call.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns a negative zq4_status and launches nothing. A failed
 *     launch returns ZQ4_ERR_CUDA (zq4_last_cuda_error() gives the CUDA
 *     error code of that failure on the calling thread).
 *   - Accumulation is fp32; the output is rounded to f16 (nearest even).
 *   - Kernels are launched with programmatic dependent launch allowed: a
 *     kernel may start while the previous kernel of the stream finishes and
 *     read its WEIGHTS early, but it reads its activation input and writes
 *     its output only after that previous kernel has completed.
 *   - Threads: any entry point may be called from several host threads at
 *     once (the library's host-side caches are atomic and the last CUDA
 *     error is kept per thread). What is shared: the device error words
 *     (one set per process and device; zq4_device_errors with clear != 0
 *     clears them for every caller), the one static stack plan per device
 *     (zq4_stack_plan_init_static), and any caller scratch (work buffers,
 *     plans), which concurrent calls on different streams must not share.
 */
#ifndef ZQ4_H
#define ZQ4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ZQ4_API __attribute__((visibility("default")))
#else
#define ZQ4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum zq4_status {
    ZQ4_OK = 0,
    ZQ4_ERR_NULL = -1,        /* a required pointer is NULL */
    ZQ4_ERR_SHAPE = -2,       /* M, N, K, T, top_k or num_experts out of range */
    ZQ4_ERR_ALIGN = -3,       /* a pointer is not 16-byte aligned */
    ZQ4_ERR_FLAGS = -4,       /* unknown mode or flags */
    ZQ4_ERR_CUDA = -5,        /* a CUDA runtime call or launch failed */
    ZQ4_ERR_UNSUPPORTED = -6, /* valid arguments this library does not handle */
    ZQ4_ERR_OVERLAP = -7      /* input and output buffers overlap */
} zq4_status;

/* Human-readable name of a status (static string, never NULL). */
ZQ4_API const char *zq4_status_string(int status);

/* CUDA error code (cudaError_t as int) behind the last ZQ4_ERR_CUDA returned
 * on the calling thread; 0 if none. */
ZQ4_API int zq4_last_cuda_error(void);

/* Library version, major*10000 + minor*100 + patch. */
ZQ4_API int zq4_version(void);

/* Bits of the library's device error word. */
#define ZQ4_DEVERR_WAIT_TIMEOUT 1u   /* a kernel gave up an internal wait (2 s; stack plans: their set limit) */

/*
 * zq4_device_errors -- read (and with clear != 0, reset) the device error
 * word of the current device. Kernels never trap: an internal wait that runs
 * out sets a bit here, the kernel drains its own in-flight copies and
 * returns (its output is then undefined). SYNCHRONOUS: waits for all work
 * on the device. Errors: ZQ4_ERR_NULL, ZQ4_ERR_CUDA.
 */
ZQ4_API zq4_status zq4_device_errors(uint32_t *flags, int clear);

/*
 * zq4_gemv -- y = x * W^T, the fused dequantize + NT matmul.
 * Source: "Zero TVM Documentation", section "WGSL Kernel Roles", card 5
 * "int4 Matmul" (one output per weight row; K_groups = K/8,
 * scale_stride = K/32), and "RESEARCH.md" (Zero-TVM), section "Matmul
 * Shader Analysis" (TVM's fused_dequantize*_NT_matmul: dot product of the
 * input with (code - 7) * group scale).
 *
 *   wq     [N, K/8]  uint32, device        scales [N, K/32] f16, device
 *   x      [M, K]    f16, device           y      [M, N]    f16, device
 *   y[m,n] = f16( sum_k x[m,k] * w[n,k] )  (fp32 accumulation)
 *
 * M >= 1 (1..16 run the decode GEMV kernels; M >= 64 the tensor-core GEMM
 * that dequantizes tiles into shared memory; 17..63 the decode kernels in
 * blocks of 16 rows), N >= 1, K a multiple of 32. wq, scales and x
 * 16-byte aligned, y 2-byte aligned; y must not overlap wq, scales or x.
 * Errors: ZQ4_ERR_NULL, ZQ4_ERR_SHAPE, ZQ4_ERR_ALIGN, ZQ4_ERR_OVERLAP,
 * ZQ4_ERR_UNSUPPORTED (M < 64 and a row of x, 2K bytes, larger than the
 * decode kernels can stage in shared memory), ZQ4_ERR_CUDA.
 */
ZQ4_API zq4_status zq4_gemv(const uint32_t *wq, const uint16_t *scales, const uint16_t *x,
                    uint16_t *y, int M, int N, int K, void *stream);

/*
 * zq4_gate_up_silu -- h = silu(x * Wg^T) * (x * Wu^T) in one pass over the
 * shared gate/up matrix.
 * Source: "Zero TVM Documentation", section "WGSL Kernel Roles", card 6
 * "Fused FFN" (gate and up share one 2*I-row matrix; SiLU and the
 * multiply follow in the same dispatch) and "RESEARCH.md" (Zero-TVM),
 * section "TVM Already Fuses Elementwise Operations" (split + SiLU +
 * multiply).
 *
 *   wq     [N2, K/8]  uint32, rows INTERLEAVED: row 2j is gate j, row 2j+1
 *                     is up j (zq4_prepare_weight converts the concatenated
 *                     [gate; up] layout)
 *   scales [N2, K/32] f16          x [M, K] f16          h [M, N2/2] f16
 *   h[m,j] = f16( silu(g) * u ),  g = sum_k x[m,k] w[2j,k],
 *   u = sum_k x[m,k] w[2j+1,k],  silu(z) = z / (1 + exp(-z)), all fp32.
 *
 * N2 must be even and >= 2; M >= 1 (M >= 64 uses the tensor-core GEMM).
 * Errors as zq4_gemv.
 */
ZQ4_API zq4_status zq4_gate_up_silu(const uint32_t *wq, const uint16_t *scales, const uint16_t *x,
                            uint16_t *h, int M, int N2, int K, void *stream);

/*
 * zq4_gemv_affine / zq4_gate_up_silu_affine -- zq4_gemv and
 * zq4_gate_up_silu on weights in the MLX affine format:
 *   value w[n,k] = s[n, k/64] * q[n,k] + b[n, k/64]
 * with q the unsigned 4-bit code (packed as in q4f16_1: 8 per uint32,
 * element i of a word in bits 4i..4i+3, no zero point) and one f16 scale
 * and one f16 bias per 64 weights. Source: "Zero TVM Documentation",
 * section "Qwen3.6-35B-A3B MoE" (affine w = s*q + b, group 64, per-tensor
 * biases); "Zero-TVM benchmarks", sections "Chunked prefill for
 * plain-attention + MLX-affine specs" and "Affine wide loads" (a u32 pair
 * is a quarter of a group).
 *
 *   wq [N, K/8] uint32   scales [N, K/64] f16   biases [N, K/64] f16
 *   x [M, K] f16         y [M, N] f16 (h [M, N2/2] for gate_up, rows
 *                        interleaved as in zq4_gate_up_silu)
 * Per 64-weight group the product is s * sum(x q) + b * sum(x), fp32.
 * M >= 1, N >= 1 (N2 even), K a multiple of 64. The tensor-core kernel
 * runs when K is a multiple of 512 and scales and biases start on 16-byte
 * boundaries (blocks of up to 16 tokens per launch); other calls run the
 * CUDA-core kernel (blocks of up to 8 tokens), with the same results up to
 * fp32 summation order. wq and x 16-byte aligned, scales, biases and the
 * output 2-byte aligned; the output must not overlap any input. Device pointers,
 * caller-owned. Errors: ZQ4_ERR_NULL, ZQ4_ERR_SHAPE, ZQ4_ERR_ALIGN,
 * ZQ4_ERR_OVERLAP, ZQ4_ERR_UNSUPPORTED (x of K does not fit in shared
 * memory), ZQ4_ERR_CUDA.
 */
ZQ4_API zq4_status zq4_gemv_affine(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                                   const uint16_t *x, uint16_t *y, int M, int N, int K, void *stream);
ZQ4_API zq4_status zq4_gate_up_silu_affine(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                                           const uint16_t *x, uint16_t *h, int M, int N2, int K, void *stream);

/*
 * zq4_moe_gemv_affine -- zq4_moe_gemv on expert banks in the MLX affine
 * format (the MoE model the pages run is an MLX checkpoint: "Zero TVM
 * Documentation", section "Qwen3.6-35B-A3B MoE"). Expert e's codes start at
 * word e * N * K/8 of wq_bank, its scales and biases at e * N * K/64 of
 * scales_bank / biases_bank (f16, [num_experts * N, K/64]). Modes, shapes,
 * routing, invalid-id handling and errors as zq4_moe_gemv, with K a multiple
 * of 64, scales and biases 2-byte aligned, and ZQ4_ERR_NULL for a NULL
 * biases_bank.
 */
ZQ4_API zq4_status zq4_moe_gemv_affine(const uint32_t *wq_bank, const uint16_t *scales_bank,
                                       const uint16_t *biases_bank, int num_experts, const uint16_t *x, uint16_t *y,
                                       int T, int N, int K, const int32_t *expert_ids, const float *route_w,
                                       int top_k, int mode, int32_t *dev_status, void *stream);

/*
 * zq4_qkv_rope_append -- the attention input projection of a decode step
 * with the RoPE rotation and the KV-cache write folded in. Source: "Zero
 * TVM Documentation", section "WGSL Kernel Roles", card 3 "QKV + RoPE +
 * KV-append (fused, decode)": the int4 QKV matmul, the rotation of Q and K
 * over the pair (dim, dim + D/2) of one head, and the write of K and V into
 * the cache, in one pass, with each pair rotated where it is computed.
 *
 *   wq [(H + 2 H_kv) D, K/8] u32, scales [(H + 2 H_kv) D, K/32] f16: rows
 *   of the H query heads, then the H_kv key heads, then the H_kv value
 *   heads, D rows each (as zq4_gemv's matrix); x [M, K] f16.
 *   y = x W^T (fp32). For token m, head h and i < D/2, with
 *   theta = pos[m] * rope_base^(-2i/D) (fp64):
 *     q_out[m, h D + i]       = f16(a cos theta - b sin theta)
 *     q_out[m, h D + i + D/2] = f16(a sin theta + b cos theta)
 *   with (a, b) = y of rows (h D + i, h D + i + D/2) of the Q block; the K
 *   block alike into k_cache[slot[m], h D ..], and V unrotated into
 *   v_cache[slot[m], h D ..]. Caches [n_slots, H_kv D] f16; pos and slot
 *   int32 [M] (device). A slot outside [0, n_slots) writes nothing for that
 *   token and ORs ZQ4_DEV_BAD_SLOT into *dev_status (a device int32, may be
 *   NULL).
 *
 * D even (<= 512), H, H_kv, M, n_slots >= 1, K a multiple of 32, rope_base > 0. x
 * 16-byte aligned, outputs 2-byte, pos / slot / dev_status 4-byte aligned;
 * outputs must not overlap each other or the inputs. D % 16 == 0 and K %
 * 256 == 0: the tensor-core decode kernel (a 16-row tile holds pair rows
 * i..i+7 of both halves of one head, read through a 4-D tensor map; one
 * launch per block of up to 16 tokens; base^(-2i/D) computed on the host
 * in fp64); else the CUDA-core kernel (blocks of up to 8 tokens). Errors:
 * ZQ4_ERR_NULL, ZQ4_ERR_SHAPE, ZQ4_ERR_ALIGN, ZQ4_ERR_OVERLAP,
 * ZQ4_ERR_UNSUPPORTED (sizes), ZQ4_ERR_CUDA.
 */
ZQ4_API zq4_status zq4_qkv_rope_append(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, int M, int K,
                                       int H, int H_kv, int D, double rope_base, const int32_t *pos,
                                       const int32_t *slot, uint16_t *q_out, uint16_t *k_cache, uint16_t *v_cache,
                                       int n_slots, int32_t *dev_status, void *stream);

/*
 * zq4_gemv_add_rmsnorm -- the O or down projection with the residual add
 * and RMSNorm that follow it, folded into the GEMV as a tail reduction.
 * Source: "Zero TVM Documentation", section "WGSL Kernel Roles", card 7
 * "Fused Add + RMSNorm" (residual_out = A + B, output = RMSNorm(residual_out)
 * x gamma; A the projection's output, B the running residual), and
 * "Zero-TVM benchmarks", "Remaining levers" item 2 (fuse the add-norm into
 * the matmul that feeds it, as a reduction at its tail).
 *
 *   r[m,n]       = resid[m,n] + sum_k x[m,k] w[n,k]     (fp32, w as zq4_gemv)
 *   res_out[m,n] = f16(r[m,n])                          (the new residual)
 *   out[m,n]     = f16(r[m,n] / sqrt(mean_n r[m,n]^2 + eps) * gamma[n])
 *
 * wq [N, K/8] u32, scales [N, K/32] f16, x [M, K] f16, resid / res_out / out
 * [M, N] f16, gamma [N] f16; eps >= 0 (finite). work: caller-owned device
 * scratch of zq4_add_rmsnorm_work_bytes(M, N) = 16 + 4 M N + 64 ceil(N/16)
 * bytes, 16-byte aligned, whose first 16 bytes must be zero before the
 * first call; every call leaves them zero (the rest is overwritten); calls
 * sharing one work buffer must be ordered on one stream. K % 256 == 0: the
 * tensor-core decode kernel with the add in its epilogue, one launch per
 * block of up to 16 tokens, each CTA adding its rows' squares per token;
 * else the CUDA-core kernel, blocks of up to 8 tokens. The last CTA of each
 * launch normalises all N outputs (fixed reduction order, no
 * floating-point atomics: repeated calls give identical bits). Outputs and
 * work must not overlap each other or any input. Errors: ZQ4_ERR_NULL,
 * ZQ4_ERR_SHAPE (M, N or K, or eps), ZQ4_ERR_ALIGN, ZQ4_ERR_OVERLAP,
 * ZQ4_ERR_UNSUPPORTED (x of K does not fit in shared memory), ZQ4_ERR_CUDA.
 */
ZQ4_API size_t zq4_add_rmsnorm_work_bytes(int M, int N);
ZQ4_API zq4_status zq4_gemv_add_rmsnorm(const uint32_t *wq, const uint16_t *scales, const uint16_t *x,
                                        const uint16_t *resid, const uint16_t *gamma, float eps,
                                        uint16_t *res_out, uint16_t *out, void *work, int M, int N, int K,
                                        void *stream);

/*
 * zq4_gemv_argmax -- the LM-head step of decode: fp32 logits and, per token,
 * the index of the largest logit.
 * Source: "Zero TVM Documentation", section "WGSL Kernel Roles" (the LM-head
 * matmul writes f32 logits for a stable argmax, followed by the argmax
 * shader) and its decode loop (argmax of the last logits picks the token).
 *
 *   wq [N, K/8] uint32, scales [N, K/32] f16, x [M, K] f16  (as zq4_gemv)
 *   y32    [M, N] float, device, or NULL (logits not stored)
 *   idx    [M] int32, device: idx[m] = the n of the largest y32[m, n]; the
 *          lowest such n when several are equal (a NaN logit counts as the
 *          largest)
 *   maxval [M] float, device, or NULL: that largest logit
 *   work   [M + 8] uint64, device, caller-owned scratch: ALL ZERO before the
 *          first call (e.g. cudaMemset); every call leaves it all zero
 *          again. Calls sharing one work buffer must be ordered on one
 *          stream.
 *   y32[m, n] = sum_k x[m,k] * w[n,k] in fp32 (no f16 rounding)
 *
 * 1 <= M <= 64, 1 <= N, K a multiple of 256 (the tensor-core decode path).
 * One launch per block of up to 16 tokens: each CTA folds the largest logit
 * of every token in its tiles into an atomic maximum, and the last CTA to
 * finish writes idx / maxval and zeroes work. Errors: ZQ4_ERR_NULL, ZQ4_ERR_SHAPE,
 * ZQ4_ERR_ALIGN (x 16 B; y32, idx, maxval 4 B; work 8 B), ZQ4_ERR_OVERLAP,
 * ZQ4_ERR_UNSUPPORTED (K not a multiple of 256, or x too large for shared
 * memory), ZQ4_ERR_CUDA.
 */
ZQ4_API zq4_status zq4_gemv_argmax(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, float *y32,
                                   int32_t *idx, float *maxval, uint64_t *work, int M, int N, int K,
                                   void *stream);

/* Modes of zq4_moe_gemv. */
#define ZQ4_MOE_GATE_UP_SILU 1
#define ZQ4_MOE_DOWN_COMBINE 2

/* Bits of the device status word of zq4_moe_gemv. */
#define ZQ4_DEV_BAD_EXPERT_ID 1u
#define ZQ4_DEV_BAD_SLOT 2u          /* zq4_qkv_rope_append: a slot outside [0, n_slots) */

/*
 * zq4_moe_gemv -- expert-gather q4f16_1 GEMV of a mixture-of-experts block.
 * Source: "Zero-TVM benchmarks" (BENCH.md), section "MoE chunked prefill"
 * (routing ids and scores of shape [tokens, slots]; the expert matmul takes
 * the token in one grid dimension and the slot in another; experts never mix
 * tokens; a combine sums the slots of each token) and "Zero TVM
 * Documentation", section "Qwen3.6-35B-A3B MoE" (expert index in the grid).
 *
 * The bank holds num_experts matrices of identical shape [N, K] back to
 * back: expert e's codes start at wq_bank + e*N*(K/8) and its scales at
 * scales_bank + e*N*(K/32).
 *   expert_ids [T, top_k] int32, device; route_w [T, top_k] float32, device.
 *
 * mode ZQ4_MOE_GATE_UP_SILU: the bank holds interleaved gate/up matrices
 *   (N = 2I rows, as zq4_gate_up_silu); x is [T, K]; y is [T, top_k, I]:
 *   y[t,j,:] = silu/mul epilogue of expert expert_ids[t,j] applied to x[t].
 *   route_w is not read (may be NULL).
 * mode ZQ4_MOE_DOWN_COMBINE: x is [T, top_k, K] (one input per slot, e.g.
 *   the previous stage's y); y is [T, N]:
 *   y[t,n] = f16( sum_j route_w[t,j] * sum_k x[t,j,k] w_e[n,k] ),
 *   e = expert_ids[t,j], fp32 throughout; route_w is required.
 *
 * An expert id outside [0, num_experts) is detected on the device: that
 * slot contributes nothing (GATE_UP: its y rows are written as zero) and
 * ZQ4_DEV_BAD_EXPERT_ID is OR-ed into *dev_status (a device int32 the
 * caller clears; may be NULL). 1 <= top_k <= 32, T >= 1. Errors as
 * zq4_gemv, plus ZQ4_ERR_FLAGS for an unknown mode.
 */
ZQ4_API zq4_status zq4_moe_gemv(const uint32_t *wq_bank, const uint16_t *scales_bank, int num_experts,
                        const uint16_t *x, uint16_t *y, int T, int N, int K,
                        const int32_t *expert_ids, const float *route_w, int top_k, int mode,
                        int32_t *dev_status, void *stream);

/*
 * zq4_moe_block -- the whole MoE block of zq4_moe_gemv's two stages in one
 * call, each expert touched by the routing read once per stage: the
 * (token, slot) pairs are grouped by expert on the device (every CTA builds
 * the same grouping: touched experts in order of their first pair, each
 * expert's pairs in pair order), a work unit is (expert, block of up to 16
 * of its pairs, 16 rows of its matrix), and each warp streams its units'
 * segments through its own ring of bulk copies into the tensor-core
 * segment loop (the pairs are the MMA columns; x staged once per CTA):
 * gate_up + SiLU*mul into h, down into fp32 z, then the weighted combine
 * adds each token's slots in slot order (repeated calls give identical
 * bits). Source: "Zero-TVM benchmarks", section "MoE chunked prefill";
 * "Zero TVM Documentation", section "Qwen3.6-35B-A3B MoE".
 *
 *   gu_seg: the [E * 2I, D] gate/up bank (rows interleaved per expert, as
 *   zq4_gate_up_silu) in the segmented layout (zq4_prepare_weight with
 *   ZQ4_PREP_SEGMENTED over all E * 2I rows); dn_seg: the [E * D, I] down
 *   bank, segmented; x [T, D] f16; y [T, D] f16:
 *     y[t] = f16( sum_j route_w[t,j] * W_dn[e](h[t,j]) ),
 *     h[t,j] = f16( silu/mul epilogue of W_gu[e] x[t] ),  e = expert_ids[t,j],
 *   fp32 accumulation; an id outside [0, E) contributes nothing and sets
 *   ZQ4_DEV_BAD_EXPERT_ID in *dev_status (may be NULL).
 * work: device scratch of zq4_moe_block_work_bytes(T, top_k, D, I) bytes,
 * 16-byte aligned, caller-owned; it holds, from its start, the grouping as
 * int32: U (touched experts), V (valid pairs), the V pair indices (t top_k
 * + j) grouped by expert then P - V of -1, the U expert ids then -1, the
 * U + 1 start offsets of each expert's pairs then -1 (P = T top_k), padded
 * to 256 bytes; then h [P, I] f16 (padded to 256 bytes) and z [P, D] fp32.
 * D and I multiples of 256, P <= 256 (else ZQ4_ERR_UNSUPPORTED: the
 * per-stage zq4_moe_gemv takes any shape), 1 <= top_k <= 32. Errors:
 * ZQ4_ERR_NULL, ZQ4_ERR_SHAPE, ZQ4_ERR_ALIGN, ZQ4_ERR_OVERLAP,
 * ZQ4_ERR_UNSUPPORTED, ZQ4_ERR_CUDA.
 */
ZQ4_API size_t zq4_moe_block_work_bytes(int T, int top_k, int D, int I);
ZQ4_API zq4_status zq4_moe_block(const void *gu_seg, const void *dn_seg, int num_experts, const uint16_t *x,
                                 uint16_t *y, int T, int D, int I, const int32_t *expert_ids, const float *route_w,
                                 int top_k, void *work, size_t work_bytes, int32_t *dev_status, void *stream);

/* Flags of zq4_prepare_weight (ZQ4_PREP_SEGMENTED may be OR-ed with
 * ZQ4_PREP_CONCAT_TO_INTERLEAVED). */
#define ZQ4_PREP_COPY 0                  /* plain copy of the canonical layout */
#define ZQ4_PREP_CONCAT_TO_INTERLEAVED 1 /* [gate; up] rows -> g0,u0,g1,u1,... */
#define ZQ4_PREP_SEGMENTED 2             /* the segmented layout (below) */

/*
 * zq4_prepare_weight -- rewrite a q4f16_1 matrix into the layout the kernels
 * take. With ZQ4_PREP_COPY and ZQ4_PREP_CONCAT_TO_INTERLEAVED the row order
 * is the only thing that changes (each row's words and scales are copied bit
 * for bit); ZQ4_PREP_SEGMENTED also regroups the words and reorders the
 * codes within them (below). Dequantized values are identical either way.
 * Source: "Zero-TVM benchmarks" (BENCH.md), section "Qwen3.5 hybrid perf
 * round" (q4f16_1 matrices are concatenated row-wise by concatenating their
 * bytes) and "Zero TVM Documentation", card 6 "Fused FFN" (the gate_up
 * matrix holds all gate rows, then all up rows).
 *
 *   wq_src/scales_src [N, K/8] / [N, K/32]  ->  wq_dst/scales_dst (same shapes)
 * N even for ZQ4_PREP_CONCAT_TO_INTERLEAVED. Source and destination must
 * not overlap.
 *
 * ZQ4_PREP_SEGMENTED (K % 256 == 0; scales_dst must be NULL) writes the
 * segmented layout into wq_dst (zq4_segmented_bytes(N, K) bytes): for each
 * 16-row tile t (tile-major) and 256-column block s, 2304 contiguous bytes,
 * one 144-byte record per row i (row 16t+i) at byte 144*i: 32 code words,
 * then the row's scales 8s .. 8s+7 (16 bytes, at 144*i + 128). Record word
 * 8q + g (q = 0..3, g = 0..7) is word 32s + 4g + q of the row (word q of
 * group g), with its nibbles reordered: nibble slot j of the stored word
 * (bits 4j..4j+3) holds element (0, 2, 4, 6, 1, 3, 5, 7)[j] of the canonical
 * word. Rows past N are zero. A bijection of the canonical matrix's codes
 * and scales (same bytes count, every code and scale kept bit for bit); the
 * layout the one-launch step and zq4_gemv_seg stream with one contiguous
 * copy per segment.
 *
 * Errors: ZQ4_ERR_NULL, ZQ4_ERR_SHAPE, ZQ4_ERR_FLAGS, ZQ4_ERR_ALIGN,
 * ZQ4_ERR_OVERLAP, ZQ4_ERR_CUDA.
 */
ZQ4_API zq4_status zq4_prepare_weight(const uint32_t *wq_src, const uint16_t *scales_src,
                              uint32_t *wq_dst, uint16_t *scales_dst, int N, int K, int flags,
                              void *stream);

/* Bytes of an N x K matrix in the segmented layout (0 unless N > 0 and
 * K % 256 == 0). */
ZQ4_API size_t zq4_segmented_bytes(int N, int K);

/*
 * zq4_dequant_f32 -- w[n,k] = (q - 7) * s as float32, exact (a 4-bit integer
 * times an f16 is representable in fp32). This is the value every decode
 * kernel multiplies with. Source: "Zero TVM Documentation", section "Q4F16
 * quantization format".
 *   w [N, K] float32, device. Errors: ZQ4_ERR_NULL, ZQ4_ERR_SHAPE,
 *   ZQ4_ERR_ALIGN, ZQ4_ERR_CUDA.
 */
ZQ4_API zq4_status zq4_dequant_f32(const uint32_t *wq, const uint16_t *scales, float *w, int N, int K,
                           void *stream);

/*
 * zq4_dequant_f16 -- w[n,k] = f16((q - 7) * s), rounded once to nearest even:
 * the f16 product the docs page's dequantization formula computes (f16 of
 * (code - 7) times the f16 scale), and the operand the tensor-core GEMM
 * (M >= 64) feeds to the tensor cores. Source: "Zero TVM Documentation",
 * section "Q4F16 quantization format".
 *   w [N, K] f16, device. Errors as zq4_dequant_f32.
 */
ZQ4_API zq4_status zq4_dequant_f16(const uint32_t *wq, const uint16_t *scales, uint16_t *w, int N, int K,
                           void *stream);

/*
 * zq4_gemv_seg / zq4_gate_up_silu_seg -- zq4_gemv and zq4_gate_up_silu for
 * 1 <= M <= 8 on a matrix in the segmented layout (zq4_prepare_weight with
 * ZQ4_PREP_SEGMENTED, prepared once when the weights are loaded); the same
 * results as the canonical-layout calls up to the order of fp32 additions.
 * Source as zq4_gemv / zq4_gate_up_silu. The layout lets every weight
 * segment arrive with one contiguous copy, and the kernel is sized so that
 * two consecutive launches share the SMs (the next projection's weights
 * stream while the current one finishes).
 *   wseg: zq4_segmented_bytes(N, K) bytes, 16-byte aligned; x [M, K] f16,
 *   16-byte aligned; y [M, N] (or h [M, N2/2]) f16. K % 256 == 0; N2 even.
 * Errors: ZQ4_ERR_NULL, ZQ4_ERR_SHAPE, ZQ4_ERR_ALIGN, ZQ4_ERR_OVERLAP,
 * ZQ4_ERR_UNSUPPORTED (M > 8, or x of M rows of K does not fit in shared
 * memory), ZQ4_ERR_CUDA.
 */
ZQ4_API zq4_status zq4_gemv_seg(const uint32_t *wseg, const uint16_t *x, uint16_t *y, int M, int N, int K,
                                void *stream);
ZQ4_API zq4_status zq4_gate_up_silu_seg(const uint32_t *wseg, const uint16_t *x, uint16_t *h, int M, int N2,
                                        int K, void *stream);

/*
 * Decode step as one launch: an ordered list of projections ("jobs") run by
 * a persistent kernel, with the results of running them one after another.
 * Source: "Zero TVM Documentation", section "Decode loop" (the fixed
 * per-token sequence of dispatches) with the projections of cards 5 "int4
 * Matmul" and 6 "Fused FFN"; each job computes exactly what zq4_gemv
 * (gate_up = 0) or zq4_gate_up_silu (gate_up = 1) computes.
 *
 * Job: wq = the matrix in the segmented layout (zq4_prepare_weight with
 * ZQ4_PREP_SEGMENTED; it carries the scales, so `scales` must be NULL), x
 * [M, K] f16, y [M, N] f16 (or [M, N/2] for gate_up); device pointers,
 * caller-owned; K % 256 == 0, N even for gate_up; wq and x 16-byte aligned.
 * A job may read the y of an earlier job as its x, and may write over the x
 * or y of an earlier job. Order is kept only where buffers meet: two jobs
 * that touch the same bytes, one of them writing, run in the given order
 * (the second waiting for the first), others may run in another order or
 * at once. zq4_stack_plan_waits tells the order and the waits a plan uses.
 * The weights are only read.
 *
 * Two kernels run plans. For M = 1 or 2: every warp computes whole 16-row
 * tiles, handed out one at a time across all jobs (no barrier between
 * jobs), each job waiting for the earlier jobs it conflicts with (at most 3
 * after dropping those implied by the others; a job list that needs more
 * runs on the other kernel). Tiles of a long-K job (more than 12 segments
 * of 256 columns) that starts so late that one whole tile would outlast the
 * rest of the step are split along K into parts of at most 12 segments
 * whose fp32 sums are added in part order (the plan's device buffer holds
 * them: at most 4 MiB, else nothing is split). For M = 3..8 (and the lists
 * above): every CTA takes its share of each job in turn, a job waiting for
 * the last earlier job it conflicts with. Both give the results of the
 * given order.
 */
typedef struct zq4_stack_job {
    const uint32_t *wq;
    const uint16_t *scales;
    const uint16_t *x;
    uint16_t *y;
    int N;
    int K;
    int gate_up;
} zq4_stack_job;

/* Filled by zq4_stack_plan_init (or _init_static); pass to zq4_stack_run.
 * `dev` is the device buffer holding the plan (job table, counters);
 * `device` the CUDA device the plan was made on (it runs only there). The
 * fields after `device` are the library's own bookkeeping: leave them as
 * the init call wrote them. */
typedef struct zq4_stack_plan {
    void *dev;
    size_t bytes;
    int n_jobs;
    int M;
    int grid;
    int max_k;
    int max_tiles;
    int device;
    int engine;
    int tiles;
    int n_pub;
    int gen;
    int min_unit;
    int split_tiles;
    int part_records;
    int entries;
    unsigned long long wait_ns;   /* device-wait limit (zq4_stack_plan_set_wait_limit) */
} zq4_stack_plan;

/*
 * zq4_stack_plan_bytes -- device bytes a plan for these jobs needs on the
 * current device (1 <= M <= 8). Errors: ZQ4_ERR_NULL, ZQ4_ERR_SHAPE,
 * ZQ4_ERR_ALIGN, ZQ4_ERR_UNSUPPORTED (M >= 3 and x of the largest K does not
 * fit in shared memory).
 */
ZQ4_API zq4_status zq4_stack_plan_bytes(const zq4_stack_job *jobs, int n_jobs, int M, size_t *bytes);

/*
 * zq4_stack_plan_waits -- the run order and the waits a plan of these jobs
 * uses (host only: no device call; pointers are compared, never read). Two
 * jobs conflict when they touch the same bytes and one of them writes them
 * (y of one meets x or y of the other). Conflicting jobs keep their order;
 * within that, a job that would wait for a job run shortly before it lets
 * later jobs that conflict with nothing still to run go first, until the
 * job it waits for is followed by its own work and twice 152 x 16 of its
 * 16-row tiles' worth of other work (a constant, the same on any device); a
 * job that some later job waits for runs before up to 12 jobs just ahead of
 * it that it may pass; when some job waits, the largest job that conflicts
 * with no other job runs last.
 *   order[r] = the index (in `jobs`) of the r-th job run;
 *   dep[i]   = the last job run before job i that conflicts with it, or -1:
 *              it is finished before any part of job i starts.
 * Indices refer to `jobs`. The arrays hold n_jobs ints, caller-owned.
 * Errors: as zq4_stack_plan_bytes, and ZQ4_ERR_NULL for a NULL array.
 */
ZQ4_API zq4_status zq4_stack_plan_waits(const zq4_stack_job *jobs, int n_jobs, int M, int *order, int *dep);

/*
 * zq4_stack_plan_init -- write the plan into `dev` (256-byte aligned, at
 * least zq4_stack_plan_bytes bytes, owned by the caller and kept alive while
 * the plan is used) and fill *plan. Synchronises `stream` (it copies the job
 * table); call it outside stream capture. The job list is copied: later
 * changes to `jobs` do not affect the plan, but the buffers it points to
 * must stay allocated.
 */
ZQ4_API zq4_status zq4_stack_plan_init(const zq4_stack_job *jobs, int n_jobs, int M, void *dev, size_t bytes,
                                       zq4_stack_plan *plan, void *stream);

/*
 * zq4_stack_run -- run every job of the plan, in order, as one cooperative
 * launch on `stream` (capturable into a CUDA graph; replays reuse the plan).
 * One plan must not run on two streams at once: its counters and scratch
 * are per plan. If a device-side wait gives up (ZQ4_DEVERR_WAIT_TIMEOUT in
 * zq4_device_errors) the plan is left inconsistent and must be initialised
 * again. Errors: ZQ4_ERR_NULL, ZQ4_ERR_SHAPE (the current device is not the
 * one the plan was made on, or the plan is a static plan that a later
 * zq4_stack_plan_init_static has replaced), ZQ4_ERR_CUDA.
 */
ZQ4_API zq4_status zq4_stack_run(const zq4_stack_plan *plan, void *stream);

/*
 * zq4_stack_plan_set_wait_limit -- how long (ns) a device-side wait of the
 * plan's kernel may last before it gives up: a job waiting for the jobs it
 * depends on, a warp waiting for its x, a warp waiting for room to post a
 * finished part. The init calls set 2 s; 0 restores that. When a wait
 * gives up, the kernel sets ZQ4_DEVERR_WAIT_TIMEOUT and the plan's abort
 * flag, every other wait of the launch sees the flag (or runs out in turn),
 * each warp lets the copies it issued land, and the launch ends; the plan
 * must then be initialised again. Waits for a bulk copy of this launch to
 * land keep their own 2 s bound (such a copy always completes). Errors:
 * ZQ4_ERR_NULL.
 */
ZQ4_API zq4_status zq4_stack_plan_set_wait_limit(zq4_stack_plan *plan, unsigned long long ns);

/*
 * zq4_stack_plan_init_static -- zq4_stack_plan_init for callers that cannot
 * give the library device memory: the plan is written into a fixed array
 * inside the library (64 KiB of device memory reserved when the library
 * loads) instead of a caller buffer, and the call itself allocates nothing
 * (no device or host heap allocation; it issues one copy of the plan image
 * from a fixed host array inside the library, so calls are serialised by a
 * lock and need no stack space of the caller beyond an ordinary call).
 * Meant for a host layer that has no handle on the device
 * allocator (the memory pool belongs to another framework and is not
 * reachable from it), and for code that must not allocate once it is
 * running (an allocation can block, synchronise or fail). The method on the
 * pages has no counterpart of this call; it is a deployment variant of
 * zq4_stack_plan_init, and the plan it fills runs with zq4_stack_run.
 *
 * Jobs and M as zq4_stack_plan_init. Limit: the job table must fit in the
 * array's first 64 KiB, i.e. at most 961 entries for a plan run by the one-
 * and two-token kernel (64-byte entries; a job split along K takes one per
 * part), 333 for the 3-to-16-token kernel (64-byte entries and a 128-byte
 * tensor map each; a longer list of up to eight tokens runs on the
 * eight-token kernel instead) and 1257 jobs for the eight-token kernel
 * (48-byte entries); a longer list returns ZQ4_ERR_UNSUPPORTED and changes
 * nothing. The rest of the array
 * (4 MiB and a little more) holds the split parts' sums. What must start at
 * zero (the plan's launch counter, abort flag and per-job and split-tile
 * counters) is cleared by every call. The first call on a device
 * resolves the array's address (cudaGetSymbolAddress); every call
 * synchronises `stream`, so call it before any stream capture begins.
 *
 * There is one such plan per device: a second zq4_stack_plan_init_static
 * replaces the first, after which zq4_stack_run refuses the first one's
 * plan struct (ZQ4_ERR_SHAPE); a call that overlaps a zq4_stack_run of the
 * static plan on another stream -- or two such runs on different streams --
 * race on the same counters and give wrong results. Errors as
 * zq4_stack_plan_init.
 */
ZQ4_API zq4_status zq4_stack_plan_init_static(const zq4_stack_job *jobs, int n_jobs, int M,
                                              zq4_stack_plan *plan, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ZQ4_H */
