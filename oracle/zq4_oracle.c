/*
 * zq4_oracle.c -- plain, slow, fp64 CPU oracle for the q4f16_1 fused
 * dequantize + NT matmul.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library. The product path
 * (the CUDA library) never calls it, and the two share no code.
 *
 * Every function follows one passage of the pages it was written from:
 *
 *  [DOC-Q4]  "Zero TVM Documentation", section "Q4F16 quantization format":
 *            8 unsigned 4-bit codes per uint32, element i of a word is
 *            (word >> 4i) & 0xF, one f16 scale per 32 weights,
 *            value = (code - 7) * scale.
 *  [DOC-MM]  "Zero TVM Documentation", section "WGSL Kernel Roles", card 5
 *            "int4 Matmul": output row n is the dot product of the input
 *            vector with dequantized row n; K_groups = K/8 words per row,
 *            scale_stride = K/32 scales per row.
 *  [DOC-FFN] same page, card 6 "Fused FFN": gate and up projections share one
 *            2*I-row matrix, followed by SiLU and an elementwise multiply.
 *  [RES-TVM] "RESEARCH.md" (Zero-TVM), section "TVM Already Fuses Elementwise
 *            Operations" (fused_dequantize + NT_matmul; split + SiLU +
 *            multiply) and "Matmul Shader Analysis" (one output element is a
 *            dot product over all K of input * (code - 7) * group scale).
 *  [DOC-ARGMAX] same page, "WGSL Kernel Roles": the LM-head matmul writes
 *            f32 logits for a stable argmax (zo_argmax).
 *  [BENCH-MOE] "Zero-TVM benchmarks" (BENCH.md), section "MoE chunked
 *            prefill": per (token, slot) the expert index comes from the
 *            routing ids, experts never mix tokens, and a combine sums the
 *            slots of one token weighted by the router scores.
 *  [DOC-ADDNORM] "Zero TVM Documentation", section "WGSL Kernel Roles",
 *            card 7 "Fused Add + RMSNorm": residual_out = A + B (A the new
 *            contribution, the O or down projection's output; B the running
 *            residual), output = RMSNorm(residual_out) * gamma; "Zero-TVM
 *            benchmarks", "Remaining levers" item 2: folded into the matmul
 *            that produces A, as a reduction at its tail.
 *  [DOC-QKV] "Zero TVM Documentation", section "WGSL Kernel Roles", card 3
 *            "QKV + RoPE + KV-append (fused, decode)": the int4 QKV matmul,
 *            the RoPE rotation of Q and K over the pair (dim, dim + D/2) of
 *            one head (dim and dim+48 for D = 96), and the write of K and V
 *            into the KV cache in one pass.
 *  [DOC-AFF] "Zero TVM Documentation", section "Qwen3.6-35B-A3B MoE", and
 *            "Zero-TVM benchmarks", sections "Chunked prefill for
 *            plain-attention + MLX-affine specs" and "Affine wide loads":
 *            the MLX affine format, value = scale * code + bias with one
 *            scale and one bias per 64 weights (a pair of u32 words covers a
 *            quarter of a group, so a group is 8 words of 8 codes).
 *
 * Readings where the pages are silent (the same list is kept with the design
 * notes): SiLU(z) = z / (1 + e^-z); gate/up "interleaved" layout puts gate row
 * j at row 2j and up row j at row 2j+1, "concatenated" puts gate rows first;
 * an expert id outside [0, E) contributes nothing and is counted. Affine
 * format: the codes are packed as in q4f16_1 (LSB-first, 8 per word) and are
 * unsigned (no zero point); scales and biases are f16 arrays [N, K/64].
 * QKV rows: Q heads, then K heads, then V heads, D rows each (H, H_kv,
 * H_kv heads); RoPE angle of pair i of a token at position p: p *
 * base^(-2i/D), (a, b) -> (a cos - b sin, a sin + b cos); the KV cache as
 * rows [slot][H_kv * D] of K and of V, the slot per token given.
 * RMSNorm (named, not defined, by the pages): y / sqrt(mean(y^2) + eps) over
 * the N features of one token, eps given by the caller; in the fused form A
 * is the exact dot product, not its f16 rounding.
 *
 * Arithmetic is IEEE fp64 throughout. The dequantized weight (q-7)*s is exact
 * in fp64 (4-bit integer times an 11-bit significand). Sums are taken in
 * plain ascending k order; S = sum |x*w| is returned beside every dot product
 * because the parity tolerance is |y - y_ref| <= 2^-10 |y_ref| + 1e-4 S.
 *
 * Parallelism: when built with OpenMP, independent output elements are
 * spread over threads; no sum is split or reordered.
 *
 * Mutants: building with -DZO_MUTANT=<n> plants one deliberate mistake so
 * that the tests can show their pins catch it. The normal build has none.
 * Every mutant keeps each access inside its arrays (an index mistake wraps
 * or stays within the row), so a mutant gives wrong numbers, never a crash.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ZO_MUTANT
#define ZO_MUTANT 0
#endif

/* Upper bound of the k loops of the dot products (mutant 4 drops the last term). */
#if ZO_MUTANT == 4
#define ZO_KEND(K) ((K) - 1)
#else
#define ZO_KEND(K) (K)
#endif

/* ---------------------------------------------------------------------- */
/* IEEE 754 binary16 <-> binary64, written from the format's definition:   */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent 0 is   */
/* zero/subnormal (value = frac * 2^-24), exponent 31 is inf/NaN.           */
/* ---------------------------------------------------------------------- */

double zo_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return sign ? -v : v;
}

/* Round half to even of a non-negative double to an integer-valued double. */
static double zo_round_half_even(double r)
{
    double fl = floor(r);
    double diff = r - fl;
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

uint16_t zo_f64_to_f16_rn(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v)) return 0x7E00;
    if (isinf(a)) return sign | 0x7C00;
    if (a == 0.0) return sign;
    int E;
    frexp(a, &E);            /* a = m * 2^E, m in [0.5, 1) */
    int e = E - 1;           /* a in [2^e, 2^(e+1)) */
    if (e < -14) {           /* subnormal range: quantum 2^-24 */
        double n = zo_round_half_even(ldexp(a, 24));
        return sign | (uint16_t)n;      /* n == 1024 encodes 2^-14 exactly */
    }
    double n = zo_round_half_even(ldexp(a, 10 - e));   /* in [1024, 2048] */
    if (n == 2048.0) { n = 1024.0; e += 1; }
    if (e + 15 >= 31) return sign | 0x7C00;
    return sign | (uint16_t)(((e + 15) << 10) | ((int)n - 1024));
}

/* ---------------------------------------------------------------------- */
/* [DOC-Q4] code of element k of row n: word k/8 of the row, nibble k%8,    */
/* least significant nibble first.                                         */
/* ---------------------------------------------------------------------- */
int zo_code(const uint32_t *wq, int64_t K, int64_t n, int64_t k)
{
    uint32_t word = wq[n * (K / 8) + k / 8];
#if ZO_MUTANT == 1
    int i = 7 - (int)(k % 8);          /* mutant: most significant nibble first */
#else
    int i = (int)(k % 8);
#endif
    return (int)((word >> (4 * i)) & 0xFu);
}

/* [DOC-Q4] w[n,k] = (q[n,k] - 7) * s[n, k/32], exact in fp64. */
double zo_weight(const uint32_t *wq, const uint16_t *scales, int64_t K, int64_t n, int64_t k)
{
    int q = zo_code(wq, K, n, k);
    int64_t g = k / 32;
#if ZO_MUTANT == 3
    g = (g + 1) % (K / 32);            /* mutant: scale index off by one group */
#endif
    double s = zo_f16_to_f64(scales[n * (K / 32) + g]);
#if ZO_MUTANT == 2
    return (double)(q - 8) * s;        /* mutant: zero point 8 */
#else
    return (double)(q - 7) * s;
#endif
}

/* [DOC-AFF] w[n,k] = s[n,k/64] * q[n,k] + b[n,k/64]: exact in fp64 (a 4-bit
 * integer times an 11-bit significand, plus an f16) unless the exponents of
 * s*q and b differ by more than 38, when it is rounded once. */
double zo_weight_affine(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases, int64_t K,
                        int64_t n, int64_t k)
{
    int q = zo_code(wq, K, n, k);
#if ZO_MUTANT == 7
    int64_t g = (k / 32) % (K / 64);   /* mutant: groups of 32 */
#else
    int64_t g = k / 64;
#endif
    double s = zo_f16_to_f64(scales[n * (K / 64) + g]);
    double b = zo_f16_to_f64(biases[n * (K / 64) + g]);
#if ZO_MUTANT == 8
    (void)b;
    return s * (double)q;              /* mutant: bias dropped */
#else
    return s * (double)q + b;
#endif
}

/* [DOC-AFF] whole matrix, w[n*K + k]. */
void zo_dequant_affine(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases, int64_t N, int64_t K,
                       double *w)
{
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) w[n * K + k] = zo_weight_affine(wq, scales, biases, K, n, k);
}

/* Dequantized row n into w[0..K). */
static void zo_dequant_row(const uint32_t *wq, const uint16_t *scales, int64_t K, int64_t n, double *w)
{
    for (int64_t k = 0; k < K; ++k) w[k] = zo_weight(wq, scales, K, n, k);
}

/* [DOC-Q4] whole matrix, w[n*K + k]. */
void zo_dequant(const uint32_t *wq, const uint16_t *scales, int64_t N, int64_t K, double *w)
{
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) zo_dequant_row(wq, scales, K, n, w + n * K);
}

/* ---------------------------------------------------------------------- */
/* [DOC-MM], [RES-TVM]: y[m,n] = sum_k x[m,k] * w[n,k] (NT matmul: both     */
/* operands are stored with K innermost). Also S[m,n] = sum_k |x*w|.        */
/* rows == NULL computes every n; otherwise only the n listed in rows[0..R) */
/* (outputs are then [M, R]).                                               */
/* ---------------------------------------------------------------------- */
void zo_gemv_rows(const uint32_t *wq, const uint16_t *scales, const uint16_t *x,
                  int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t R,
                  double *y, double *S)
{
    int64_t count = rows ? R : N;
    #pragma omp parallel
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        #pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < count; ++i) {
            int64_t n = rows ? rows[i] : i;
            zo_dequant_row(wq, scales, K, n, w);
            for (int64_t m = 0; m < M; ++m) {
                double acc = 0.0, sabs = 0.0;
                for (int64_t k = 0; k < ZO_KEND(K); ++k) {
                    double p = zo_f16_to_f64(x[m * K + k]) * w[k];
                    acc += p;
                    sabs += fabs(p);
                }
                y[m * count + i] = acc;
                S[m * count + i] = sabs;
            }
        }
        free(w);
    }
}

void zo_gemv(const uint32_t *wq, const uint16_t *scales, const uint16_t *x,
             int64_t M, int64_t N, int64_t K, double *y, double *S)
{
    zo_gemv_rows(wq, scales, x, M, N, K, NULL, 0, y, S);
}

/* ---------------------------------------------------------------------- */
/* SiLU, the activation of the gated FFN ([DOC-FFN]; the pages name it but  */
/* do not define it): silu(z) = z * sigmoid(z) = z / (1 + e^-z).            */
/* ---------------------------------------------------------------------- */
double zo_silu(double z)
{
#if ZO_MUTANT == 5
    return z / (1.0 + exp(z));         /* mutant: sign error in the sigmoid */
#else
    return z / (1.0 + exp(-z));
#endif
}

/* d silu / dz = sigmoid(z) * (1 + z * (1 - sigmoid(z))), used only for the
 * first-order error propagation of the gate_up tolerance. */
double zo_silu_deriv(double z)
{
    double sg = 1.0 / (1.0 + exp(-z));
    return sg * (1.0 + z * (1.0 - sg));
}

/* Row of gate j and of up j under the two layouts of a 2*I-row matrix. */
static int64_t zo_gate_row(int64_t j, int interleaved) { return interleaved ? 2 * j : j; }
static int64_t zo_up_row(int64_t j, int64_t I, int interleaved) { return interleaved ? 2 * j + 1 : I + j; }

/* ---------------------------------------------------------------------- */
/* [DOC-FFN], [RES-TVM]: h[m,j] = silu(g[m,j]) * u[m,j] where g and u are   */
/* the GEMV outputs of gate row j and up row j of the shared N2 = 2I-row    */
/* matrix. Also returns g, u, S_g, S_u and the propagated tolerance scale   */
/* Sh = |silu'(g) u| S_g + |silu(g)| S_u.                                   */
/* Any of the optional outputs may be NULL.                                 */
/* ---------------------------------------------------------------------- */
void zo_gate_up_silu(const uint32_t *wq, const uint16_t *scales, const uint16_t *x,
                     int64_t M, int64_t N2, int64_t K, int interleaved,
                     double *h, double *Sh, double *g_out, double *u_out,
                     double *Sg_out, double *Su_out)
{
    int64_t I = N2 / 2;
    #pragma omp parallel
    {
        double *wg = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        double *wu = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        #pragma omp for schedule(dynamic, 16)
        for (int64_t j = 0; j < I; ++j) {
            zo_dequant_row(wq, scales, K, zo_gate_row(j, interleaved), wg);
            zo_dequant_row(wq, scales, K, zo_up_row(j, I, interleaved), wu);
            for (int64_t m = 0; m < M; ++m) {
                double g = 0, u = 0, sg = 0, su = 0;
                for (int64_t k = 0; k < K; ++k) {
                    double xv = zo_f16_to_f64(x[m * K + k]);
                    double pg = xv * wg[k], pu = xv * wu[k];
                    g += pg; u += pu; sg += fabs(pg); su += fabs(pu);
                }
                int64_t o = m * I + j;
                double a = zo_silu(g);
                h[o] = a * u;
#if ZO_MUTANT == 16
                if (Sh) Sh[o] = fabs(zo_silu_deriv(g)) * sg + fabs(a) * su;   /* mutant: u dropped */
#else
                if (Sh) Sh[o] = fabs(zo_silu_deriv(g) * u) * sg + fabs(a) * su;
#endif
                if (g_out) g_out[o] = g;
                if (u_out) u_out[o] = u;
                if (Sg_out) Sg_out[o] = sg;
                if (Su_out) Su_out[o] = su;
            }
        }
        free(wg);
        free(wu);
    }
}

/* ---------------------------------------------------------------------- */
/* [DOC-AFF], [DOC-MM]: y[m,n] = sum_k x[m,k] * w[n,k] with the affine       */
/* weights, and the tolerance scale of this format, Sa[m,n] = sum_k |x[m,k]| */
/* (|s| q + |b|): the sum the two halves of s * sum(x q) + b * sum(x) are    */
/* each bounded by (where w ~ 0 through s q ~ -b, |x w| is not).            */
/* rows as in zo_gemv_rows.                                                 */
/* ---------------------------------------------------------------------- */
void zo_gemv_affine_rows(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases, const uint16_t *x,
                         int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t R, double *y, double *Sa)
{
    int64_t count = rows ? R : N;
    #pragma omp parallel
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        double *wa = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        #pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < count; ++i) {
            int64_t n = rows ? rows[i] : i;
            for (int64_t k = 0; k < K; ++k) {
                w[k] = zo_weight_affine(wq, scales, biases, K, n, k);
                int64_t g = k / 64;
                wa[k] = fabs(zo_f16_to_f64(scales[n * (K / 64) + g])) * (double)zo_code(wq, K, n, k) +
                        fabs(zo_f16_to_f64(biases[n * (K / 64) + g]));
            }
            for (int64_t m = 0; m < M; ++m) {
                double acc = 0.0, sabs = 0.0;
                for (int64_t k = 0; k < ZO_KEND(K); ++k) {
                    double xv = zo_f16_to_f64(x[m * K + k]);
                    acc += xv * w[k];
                    sabs += fabs(xv) * wa[k];
                }
                y[m * count + i] = acc;
                Sa[m * count + i] = sabs;
            }
        }
        free(w);
        free(wa);
    }
}

/* [DOC-AFF], [DOC-FFN]: h[m,j] = silu(g[m,j]) * u[m,j] over interleaved      */
/* gate/up rows (gate j = row 2j, up j = row 2j+1) of affine weights, with   */
/* the propagated tolerance scale Sh = |silu'(g) u| Sa_g + |silu(g)| Sa_u.   */
/* ---------------------------------------------------------------------- */
void zo_gate_up_silu_affine(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                            const uint16_t *x, int64_t M, int64_t N2, int64_t K, double *h, double *Sh)
{
    int64_t I = N2 / 2;
    double *g = (double *)malloc(sizeof(double) * (size_t)(M * N2 > 0 ? M * N2 : 1));
    double *Sa = (double *)malloc(sizeof(double) * (size_t)(M * N2 > 0 ? M * N2 : 1));
    zo_gemv_affine_rows(wq, scales, biases, x, M, N2, K, NULL, 0, g, Sa);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < I; ++j) {
            double gv = g[m * N2 + 2 * j], uv = g[m * N2 + 2 * j + 1];
            double a = zo_silu(gv);
            h[m * I + j] = a * uv;
            Sh[m * I + j] = fabs(zo_silu_deriv(gv) * uv) * Sa[m * N2 + 2 * j] + fabs(a) * Sa[m * N2 + 2 * j + 1];
        }
    free(g);
    free(Sa);
}

/* ---------------------------------------------------------------------- */
/* [DOC-ADDNORM], [DOC-MM]: for each token m, r[m,n] = B[m,n] + sum_k       */
/* x[m,k] w[n,k] (exact dot product), rms[m] = sqrt(mean_n r[m,n]^2 + eps), */
/* out[m,n] = r[m,n] / rms[m] * gamma[n]. Also S[m,n] = sum_k |x w| (the   */
/* dot product's tolerance scale) and the first-order propagation of an    */
/* error e[m,n] = tol_r[m,n] = 2^-10 |r| + 1e-4 S + 2^-25 in r to out:      */
/* Tn[m,n] = |gamma[n]| / rms[m] * (e[m,n] + |r[m,n]| * sum_j |r_j| e_j /  */
/* (N rms[m]^2)), bounding |d out| (d rms / rms = sum_j r_j d r_j /         */
/* (N rms^2)).                                                             */
/* ---------------------------------------------------------------------- */
void zo_gemv_add_rmsnorm(const uint32_t *wq, const uint16_t *scales, const uint16_t *x,
                         const uint16_t *resid, const uint16_t *gamma, double eps, int64_t M, int64_t N,
                         int64_t K, double *r, double *out, double *S, double *Tn)
{
    zo_gemv_rows(wq, scales, x, M, N, K, NULL, 0, r, S);
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0, se = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double v = r[m * N + n] + zo_f16_to_f64(resid[m * N + n]);
            r[m * N + n] = v;
            ss += v * v;
        }
#if ZO_MUTANT == 9
        double rms = sqrt(ss / (double)N);          /* mutant: eps dropped */
#else
        double rms = sqrt(ss / (double)N + eps);
#endif
        double *e = Tn + m * N;                      /* holds e first */
        for (int64_t n = 0; n < N; ++n) {
            e[n] = ldexp(fabs(r[m * N + n]), -10) + 1e-4 * S[m * N + n] + ldexp(1.0, -25);
            se += fabs(r[m * N + n]) * e[n];
        }
        double drel = se / ((double)N * rms * rms);
        for (int64_t n = 0; n < N; ++n) {
            double g = zo_f16_to_f64(gamma[n]);
#if ZO_MUTANT == 12
            out[m * N + n] = r[m * N + n] / rms;         /* mutant: gamma dropped */
#else
            out[m * N + n] = r[m * N + n] / rms * g;
#endif
#if ZO_MUTANT == 15
            Tn[m * N + n] = fabs(g) / rms * e[n];        /* mutant: the norm's cross term dropped */
#else
            Tn[m * N + n] = fabs(g) / rms * (e[n] + fabs(r[m * N + n]) * drel);
#endif
        }
    }
}

/* ---------------------------------------------------------------------- */
/* [DOC-QKV], [DOC-MM]: y = x W^T over the (H + 2 H_kv) D rows (exact dot   */
/* products); for Q and K heads each pair (i, i + D/2), i < D/2, rotated by */
/* theta = pos[m] * base^(-2i/D): q_out[m, h D + i] = a cos - b sin,        */
/* q_out[m, h D + i + D/2] = a sin + b cos (K alike into kc, V copied into  */
/* vc), kc/vc[m, c] = the token's row of the cache (written at its slot by  */
/* the kernel). S[m, row] = sum_k |x w| of each of the two rows of a pair,  */
/* added: Sp[m, c] = S_a + S_b for both outputs of the pair (for V: the     */
/* row's own S); Ap[m, c] = |a| + |b| (V: |y|).                            */
/* ---------------------------------------------------------------------- */
void zo_qkv_rope(const uint32_t *wq, const uint16_t *scales, const uint16_t *x, int64_t M, int64_t K, int64_t H,
                 int64_t Hkv, int64_t D, double base, const int32_t *pos, double *q, double *kc, double *vc,
                 double *Sq, double *Sk, double *Sv, double *Aq, double *Ak, double *Av)
{
    int64_t N = (H + 2 * Hkv) * D, half = D / 2;
    double *y = (double *)malloc(sizeof(double) * (size_t)(M * N > 0 ? M * N : 1));
    double *S = (double *)malloc(sizeof(double) * (size_t)(M * N > 0 ? M * N : 1));
    zo_gemv_rows(wq, scales, x, M, N, K, NULL, 0, y, S);
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t hb = 0; hb < H + 2 * Hkv; ++hb) {
            for (int64_t i = 0; i < half; ++i) {
#if ZO_MUTANT == 11
                int64_t ia = 2 * i, ib = 2 * i + 1;   /* mutant: adjacent pairs */
#else
                int64_t ia = i, ib = i + half;
#endif
                int64_t ra = hb * D + ia, rb = hb * D + ib;
                double a = y[m * N + ra], b = y[m * N + rb];
                double sa = S[m * N + ra], sb = S[m * N + rb];
                if (hb < H + Hkv) {
#if ZO_MUTANT == 10
                    double th = (double)pos[m] * pow(base, -2.0 * (double)(i + 1) / (double)D); /* mutant: i+1 */
#else
                    double th = (double)pos[m] * pow(base, -2.0 * (double)i / (double)D);
#endif
                    double c = cos(th), sn = sin(th);
                    double oa = a * c - b * sn, ob = a * sn + b * c;
                    double *o = hb < H ? q + m * H * D : kc + m * Hkv * D;
                    double *so = hb < H ? Sq + m * H * D : Sk + m * Hkv * D;
                    double *ao = hb < H ? Aq + m * H * D : Ak + m * Hkv * D;
                    int64_t h = hb < H ? hb : hb - H;
                    o[h * D + ia] = oa;
                    o[h * D + ib] = ob;
#if ZO_MUTANT == 17
                    so[h * D + ia] = so[h * D + ib] = sa;        /* mutant: the partner's scale dropped */
#else
                    so[h * D + ia] = so[h * D + ib] = sa + sb;
#endif
                    ao[h * D + ia] = ao[h * D + ib] = fabs(a) + fabs(b);
                } else {
                    int64_t h = hb - H - Hkv;
                    vc[m * Hkv * D + h * D + ia] = a;
                    vc[m * Hkv * D + h * D + ib] = b;
                    Sv[m * Hkv * D + h * D + ia] = sa;
                    Sv[m * Hkv * D + h * D + ib] = sb;
                    Av[m * Hkv * D + h * D + ia] = fabs(a);
                    Av[m * Hkv * D + h * D + ib] = fabs(b);
                }
            }
        }
    }
    free(y);
    free(S);
}

/* ---------------------------------------------------------------------- */
/* [BENCH-MOE] expert gate_up stage. Expert e's matrix starts at word        */
/* e * N2 * K/8 and scale e * N2 * K/32. For token t and slot j the expert  */
/* is ids[t*top_k + j]; h[(t*top_k + j)*I + i] = silu(g) * u of that expert */
/* on x[t]. An id outside [0, E) gives h = 0, Sh = 0 and is counted in the  */
/* return value.                                                            */
/* ---------------------------------------------------------------------- */
int64_t zo_moe_gate_up(const uint32_t *wq_bank, const uint16_t *sc_bank, int64_t E,
                       const uint16_t *x, int64_t T, int64_t N2, int64_t K,
                       const int32_t *ids, int64_t top_k, int interleaved,
                       double *h, double *Sh)
{
    int64_t I = N2 / 2, bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t e = ids[t * top_k + j];
            double *ho = h + (t * top_k + j) * I;
            double *so = Sh ? Sh + (t * top_k + j) * I : NULL;
            if (e < 0 || e >= E) {
                ++bad;
                for (int64_t i = 0; i < I; ++i) { ho[i] = 0.0; if (so) so[i] = 0.0; }
                continue;
            }
            zo_gate_up_silu(wq_bank + e * N2 * (K / 8), sc_bank + e * N2 * (K / 32),
                            x + t * K, 1, N2, K, interleaved, ho, so, NULL, NULL, NULL, NULL);
        }
    }
    return bad;
}

/* ---------------------------------------------------------------------- */
/* [BENCH-MOE] expert down stage + combine: for token t,                    */
/*   y[t,n] = sum_j r[t,j] * z[t,j,n],  z[t,j,n] = sum_k h[t,j,k] w_e[n,k]  */
/* with e = ids[t,j]; S[t,n] = sum_j |r[t,j]| * sum_k |h w|. h is f16 [T,   */
/* top_k, K]; r is float32 [T, top_k]. Invalid ids contribute nothing and   */
/* are counted in the return value.                                         */
/* ---------------------------------------------------------------------- */
int64_t zo_moe_down_combine(const uint32_t *wq_bank, const uint16_t *sc_bank, int64_t E,
                            const uint16_t *h, const float *r, int64_t T, int64_t N, int64_t K,
                            const int32_t *ids, int64_t top_k, double *y, double *S)
{
    int64_t bad = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t e = ids[t * top_k + j];
            if (e < 0 || e >= E) ++bad;
        }
    #pragma omp parallel
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        #pragma omp for schedule(dynamic, 16)
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t t = 0; t < T; ++t) {
                double acc = 0.0, sabs = 0.0;
                for (int64_t j = 0; j < top_k; ++j) {
                    int64_t e = ids[t * top_k + j];
                    if (e < 0 || e >= E) continue;
                    zo_dequant_row(wq_bank + e * N * (K / 8), sc_bank + e * N * (K / 32), K, n, w);
#if ZO_MUTANT == 14
                    const uint16_t *hv = h + t * K;           /* mutant: slot's h row ignored */
#else
                    const uint16_t *hv = h + (t * top_k + j) * K;
#endif
                    double z = 0.0, sz = 0.0;
                    for (int64_t k = 0; k < K; ++k) {
                        double p = zo_f16_to_f64(hv[k]) * w[k];
                        z += p;
                        sz += fabs(p);
                    }
#if ZO_MUTANT == 13
                    double rj = 1.0;                          /* mutant: router weight dropped */
#else
                    double rj = (double)r[t * top_k + j];
#endif
                    acc += rj * z;
                    sabs += fabs(rj) * sz;
                }
                y[t * N + n] = acc;
                S[t * N + n] = sabs;
            }
        }
        free(w);
    }
    return bad;
}

/*
 * [DOC-ARGMAX] "Zero TVM Documentation", section "WGSL Kernel Roles": the
 * LM-head matmul writes f32 logits and the argmax step picks the next token
 * as the position of the largest one. Reading where the pages are silent:
 * ties go to the lowest index, and a NaN counts as larger than any number
 * (the first NaN wins). idx[m] = that position in row m of y [M][N].
 */
/* ---------------------------------------------------------------------- */
/* [BENCH-MOE] with [DOC-AFF] weights (the MoE model the pages run in the    */
/* affine format): the expert stages of zo_moe_gate_up (interleaved rows)   */
/* and zo_moe_down_combine on affine banks. Expert e's codes start at word  */
/* e * N * K/8, its scales and biases at e * N * K/64. Tolerance scales as  */
/* in zo_gemv_affine_rows (Sa), propagated through SiLU and the combine.    */
/* ---------------------------------------------------------------------- */
int64_t zo_moe_gate_up_affine(const uint32_t *wq_bank, const uint16_t *sc_bank, const uint16_t *bi_bank,
                              int64_t E, const uint16_t *x, int64_t T, int64_t N2, int64_t K,
                              const int32_t *ids, int64_t top_k, double *h, double *Sh)
{
    int64_t I = N2 / 2, bad = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t e = ids[t * top_k + j];
            double *ho = h + (t * top_k + j) * I, *so = Sh + (t * top_k + j) * I;
            if (e < 0 || e >= E) {
                ++bad;
                for (int64_t i = 0; i < I; ++i) ho[i] = so[i] = 0.0;
                continue;
            }
#if ZO_MUTANT == 18
            zo_gate_up_silu_affine(wq_bank + e * N2 * (K / 8), sc_bank + e * N2 * (K / 64),
                                   bi_bank, x + t * K, 1, N2, K, ho, so);  /* mutant: bias bank not offset */
#else
            zo_gate_up_silu_affine(wq_bank + e * N2 * (K / 8), sc_bank + e * N2 * (K / 64),
                                   bi_bank + e * N2 * (K / 64), x + t * K, 1, N2, K, ho, so);
#endif
        }
    return bad;
}

int64_t zo_moe_down_combine_affine(const uint32_t *wq_bank, const uint16_t *sc_bank, const uint16_t *bi_bank,
                                   int64_t E, const uint16_t *h, const float *r, int64_t T, int64_t N, int64_t K,
                                   const int32_t *ids, int64_t top_k, double *y, double *Sa)
{
    int64_t bad = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t e = ids[t * top_k + j];
            if (e < 0 || e >= E) ++bad;
        }
    double *z = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double *sz = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t n = 0; n < N; ++n) y[t * N + n] = Sa[t * N + n] = 0.0;
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t e = ids[t * top_k + j];
            if (e < 0 || e >= E) continue;
            zo_gemv_affine_rows(wq_bank + e * N * (K / 8), sc_bank + e * N * (K / 64), bi_bank + e * N * (K / 64),
                                h + (t * top_k + j) * K, 1, N, K, NULL, 0, z, sz);
            double rj = (double)r[t * top_k + j];
            for (int64_t n = 0; n < N; ++n) {
                y[t * N + n] += rj * z[n];
                Sa[t * N + n] += fabs(rj) * sz[n];
            }
        }
    }
    free(z);
    free(sz);
    return bad;
}

void zo_argmax(const double *y, int64_t M, int64_t N, int32_t *idx)
{
    for (int64_t m = 0; m < M; ++m) {
        const double *row = y + m * N;
        int64_t best = 0;
        for (int64_t n = 1; n < N; ++n) {
            const double v = row[n], b = row[best];
            if (isnan(b)) break;                 /* a NaN already holds the place */
#if ZO_MUTANT == 6
            if (isnan(v) || v >= b) best = n;    /* mutant: ties to the highest index */
#else
            if (isnan(v) || v > b) best = n;
#endif
        }
        idx[m] = (int32_t)best;
    }
}

/* Threads the OpenMP regions above use (1 without OpenMP). */
int zo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Use n threads in the OpenMP regions from now on (timing only; the
 * results do not depend on it). Returns the count in effect. */
int zo_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

int zo_mutant(void) { return ZO_MUTANT; }
