// zq4_moe_group.cuh -- the expert grouping of a mixture-of-experts block's
// (token, slot) pairs, built on the device by every CTA the same way (no
// atomics, no order dependence): the touched experts in order of their
// first pair, each expert's pairs in pair order ("Zero-TVM benchmarks",
// section "MoE chunked prefill": routing ids [tokens, slots]; the pairs of
// one expert share its weights).
#pragma once

#include <stdint.h>

#include "../../include/zq4.h"

namespace zq4 {

// Shared-memory ints the grouping of P pairs needs.
__host__ __device__ inline int moe_group_smem_ints(int P) { return 12 * (P + 2); }
// Ints of the published copy: U, V, order [P], experts [P], starts [P + 1].
__host__ __device__ inline int moe_group_pub_ints(int P) { return 3 * P + 3; }

struct MoeGroup {
    const int *order;    // [V] pairs grouped by expert
    const int *ustart;   // [U + 1] where each touched expert's pairs start in order
    const int *uexp;     // [U] expert id of each touched expert
    const int *jt;       // [J] blocks of up to 16 pairs: (touched expert << 8) | block
    int U, J;
};

// Called by every thread of the CTA (nthr threads, index tid); sm holds
// moe_group_smem_ints(P) ints. Ids outside [0, E) are left out (and, when
// report, OR ZQ4_DEV_BAD_EXPERT_ID into *dev_status). Ends with a barrier.
__device__ inline MoeGroup moe_group(const int32_t *ids, int P, int E, int *sm, int32_t *dev_status, bool report,
                                     int tid, int nthr)
{
    int *pe = sm, *rank = pe + P, *first = rank + P, *ueidx = first + P, *ucnt = ueidx + P;
    int *ustart = ucnt + P, *uexp = ustart + P + 1, *jstart = uexp + P, *order = jstart + P + 1;
    int *jt = order + P, *misc = jt + P;
    for (int p = tid; p < P; p += nthr) {
        const int e = ids[p];
        const bool v = e >= 0 && e < E;
        pe[p] = v ? e : -1;
        if (!v && report && dev_status) atomicOr(dev_status, int32_t(ZQ4_DEV_BAD_EXPERT_ID));
    }
    __syncthreads();
    for (int p = tid; p < P; p += nthr) {              // rank among the expert's pairs, and its first pair
        const int e = pe[p];
        int r = 0, f = p;
        if (e >= 0)
            for (int q = p - 1; q >= 0; --q)
                if (pe[q] == e) {
                    ++r;
                    f = q;
                }
        rank[p] = r;
        first[p] = f;
    }
    __syncthreads();
    for (int p = tid; p < P; p += nthr) {              // first pairs: the touched experts
        if (pe[p] < 0 || first[p] != p) continue;
        int u = 0, c = 0;
        for (int q = 0; q < p; ++q) u += pe[q] >= 0 && first[q] == q;
        for (int q = p; q < P; ++q) c += pe[q] == pe[p];
        ueidx[p] = u;
        ucnt[u] = c;
        uexp[u] = pe[p];
    }
    if (tid == 0) {
        int U = 0;
        for (int p = 0; p < P; ++p) U += pe[p] >= 0 && first[p] == p;
        misc[0] = U;
    }
    __syncthreads();
    const int U = misc[0];
    for (int u = tid; u <= U; u += nthr) {             // where each touched expert's pairs and blocks start
        int st = 0, jb = 0;
        for (int v = 0; v < u; ++v) {
            st += ucnt[v];
            jb += (ucnt[v] + 15) >> 4;
        }
        ustart[u] = st;
        jstart[u] = jb;
    }
    __syncthreads();
    for (int p = tid; p < P; p += nthr)
        if (pe[p] >= 0) order[ustart[ueidx[first[p]]] + rank[p]] = p;
    for (int u = tid; u < U; u += nthr)
        for (int b = 0; b < ((ucnt[u] + 15) >> 4); ++b) jt[jstart[u] + b] = (u << 8) | b;
    __syncthreads();
    MoeGroup g;
    g.order = order;
    g.ustart = ustart;
    g.uexp = uexp;
    g.jt = jt;
    g.U = U;
    g.J = jstart[U];
    return g;
}

// The published copy (one CTA): U, V, order then -1, experts then -1,
// starts then -1.
__device__ inline void moe_group_publish(const MoeGroup &g, int P, int32_t *out, int tid, int nthr)
{
    const int V = g.ustart[g.U];
    if (tid == 0) {
        out[0] = g.U;
        out[1] = V;
    }
    for (int i = tid; i < P; i += nthr) {
        out[2 + i] = i < V ? g.order[i] : -1;
        out[2 + P + i] = i < g.U ? g.uexp[i] : -1;
    }
    for (int i = tid; i <= P; i += nthr) out[2 + 2 * P + i] = i <= g.U ? g.ustart[i] : -1;
}

}  // namespace zq4
