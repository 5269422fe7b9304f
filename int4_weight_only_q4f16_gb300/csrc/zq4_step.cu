// zq4_step.cu -- a decode step (an ordered list of q4f16_1 projections) as
// one persistent launch for one or two tokens: whole 16-row tiles per warp,
// tiles handed out one at a time from a counter, no barrier between jobs.
//
// What it computes: for every job j, y_j = x_j * W_j^T, or the fused gate_up
// + SiLU*mul output for interleaved gate/up rows ("Zero TVM Documentation",
// section "Q4F16 quantization format", cards 5 "int4 Matmul" and 6 "Fused
// FFN"; the per-token dispatch sequence of its "Decode loop" section), with
// the results of running the jobs one after another in the given order.
//
// How:
//  * Work unit = a tile (16 weight rows x all K columns); the jobs' tiles
//    form one sequence in run order, and each compute warp takes the next
//    tile from a device counter (one atomic add per tile, half a tile
//    ahead of need). A warp computes a whole tile, so no partial sum ever leaves
//    its registers and no warp waits for another at a job boundary; a slow
//    SM simply takes fewer tiles.
//  * Each compute warp streams its segments (16 rows x 256 columns of the
//    segmented layout, 2304 contiguous bytes) through its own ring of
//    shared-memory slots: right after computing a segment it refills that
//    slot with the next one (one bulk copy, issued by lane 0 behind the same
//    control flow as every other lane), so the copies keep pace with the
//    warp without a hand-off; the slot's descriptor (job, tile, first/last)
//    travels with it.
//  * x of every job is brought into shared memory once per CTA, by a stager
//    warp, into a byte ring (the window): bytes taken in job order, one bulk
//    copy per token, issued once the job's waits are met; a job whose waits
//    are not met yet keeps its bytes and the stager goes on with the jobs
//    after it. Bytes come back once no compute warp of the CTA can still
//    read them (each warp publishes the job it is reading and a lower bound
//    of the jobs it will read after it, so a warp busy with a long tile
//    holds one job's bytes, not the window).
//  * Long-K jobs near the end of the step (where one whole tile would
//    outlast the rest of the work) are split along K into parts of at most
//    12 segments, each an entry of the job table; a part's warp leaves its
//    fp32 sums in the plan's workspace and posts the tile to the CTA's
//    finisher warp, which counts the arrival and, for the last part of a
//    tile, adds the parts in part order and writes the tile.
//  * Inner loop, one token (the MMA's 8 columns would otherwise hold 1
//    useful token): column c of the m16n8k16 accumulator collects group c
//    of the segment (a block-diagonal B: lanes of column c read x of group
//    c, all others a zero row), so the 16 MMAs of a segment leave the eight
//    group sums of rows r, r+8 in two chains (even and odd groups) and the
//    group scales are applied once per segment (4 fp32 FMAs per lane instead
//    of 32). Two tokens: columns = (token, 4 groups), two passes. The codes
//    are unpacked to exact f16 (q - 7) (magic-number OR, one f16x2 subtract
//    or multiply-add), the products are exact and accumulate in fp32.
//  * A job that reads or overwrites another's buffers waits for that job (on
//    the host's list of waits: every earlier conflicting job not already
//    implied by another wait) before its x is staged and so before any of
//    its tiles is computed: each warp counts its finished tiles of a
//    waited-for job in shared memory, and a publisher warp per CTA makes
//    them visible GPU-wide in batches (one GPU-scope fence per batch, off the
//    compute warps) by adding to the job's global counter; the stager polls
//    that counter (acquire), then fences the async proxy before its bulk
//    copy reads the data.
//  * Counters grow monotonically across launches (targets scale with the
//    launch index); the last CTA to finish resets the tile counter and
//    advances the launch index.
//  * Every wait is bounded (the plan's limit, 2 s unless the caller set
//    another; a wait for a bulk copy to land: 2 s). A timeout sets ZQ4_DEVERR_WAIT_TIMEOUT and
//    the plan's abort flag, which every waiter checks; each warp lets the
//    copies it issued land before it exits; the plan must then be
//    initialised again.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "zq4_async.cuh"
#include "zq4_common.cuh"
#include "zq4_internal.h"
#include "zq4_moe_group.cuh"
#include "zq4_segment.cuh"
#include "zq4_step.h"

namespace zq4 {

__device__ unsigned g_step_error = 0;

namespace sp {

using segk::kSegBytes;
using segk::group_word;

constexpr int kWarps = kStepWarps;         // compute warps, one ring each
constexpr int kStagerWarp = kWarps;
constexpr int kPubWarp = kWarps + 1;
constexpr int kThreads = kWarps * 32 + 64;

struct Params {
    StepHeader *hdr;
    const StepJob *jobs;
    unsigned *job_done;      // [n_jobs]: units finished (monotone across launches)
    unsigned *arrive;        // split tiles: parts finished (monotone across launches)
    float *work;             // split tiles: the parts' sums
    int n_jobs, total_tiles, M, slots, wbytes, cached, n_pub;
    int fine;                // every work unit is at least `slots` segments long
    int split;               // some job is split into parts
    unsigned long long wait_ns;   // how long a wait on another warp or CTA may last
    const CUtensorMap *tmaps;     // k_wide: per entry, x[M][K] in boxes of [M][256]
    int slot_bytes;               // k_wide: one segment and its x
};

// Finished tiles of split parts, posted by each compute warp to the
// finisher (the publisher warp): a ring of kPosts (entry, tile) pairs per
// warp, with the counts posted and taken.
constexpr int kPosts = 4;

// x window entries: job j's x is described by entry j % kEntries (barrier,
// published tag, and the stager's record of the bytes it took)
constexpr int kEntries = 32;
// tag word of an entry: job << 12 | (offset / 128) << 1 | parity of the fill
constexpr int kTagJobShift = 12;

// Shared-memory layout (bytes from a 128-byte aligned base).
struct Smem {
    uint32_t ring, bars, desc, xbar, xtag, xstart, xtotal, wcur, wlb, posted, taken, posts, misc, zero, xwin, cta_done,
        cta_pub, cta_snap,
        jobs, total;
    __host__ __device__ Smem(int slots, int wbytes, int n_pub, int cached)
    {
        ring = 0;
        bars = ring + uint32_t(kWarps * slots) * kSegBytes;
        desc = bars + uint32_t(kWarps * slots) * 8;
        xbar = desc + uint32_t(kWarps * slots) * 16;
        xtag = xbar + kEntries * 8;
        xstart = xtag + kEntries * 4;
        xtotal = xstart + kEntries * 4;
        wcur = xtotal + kEntries * 4;
        wlb = wcur + kWarps * 4;
        posted = wlb + kWarps * 4;
        taken = posted + kWarps * 4;
        posts = taken + kWarps * 4;
        misc = posts + kWarps * kPosts * 8;
        zero = (misc + 64 + 127) / 128 * 128;
        xwin = zero + 128;
        cta_done = xwin + uint32_t(wbytes);
        cta_pub = cta_done + uint32_t(n_pub) * 4;
        cta_snap = cta_pub + uint32_t(n_pub) * 4;
        jobs = (cta_snap + uint32_t(n_pub) * 4 + 15) / 16 * 16;
        total = jobs + uint32_t(cached) * uint32_t(sizeof(StepJob));
    }
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p)
{
    unsigned r;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(r) : "l"(p) : "memory");
    return r;
}
__device__ __forceinline__ int ld_acquire_cta_s32(uint32_t saddr)
{
    int r;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(r) : "r"(saddr) : "memory");
    return r;
}
__device__ __forceinline__ void st_release_cta_s32(uint32_t saddr, int v)
{
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(saddr), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_cta(uint32_t saddr, unsigned v)
{
    asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(saddr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t saddr)
{
    uint32_t r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(saddr));
    return r;
}
__device__ __forceinline__ int4 lds_s4(uint32_t saddr)
{
    int4 v;
    asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr));
    return v;
}
__device__ __forceinline__ int2 lds_s2(uint32_t saddr)
{
    int2 v;
    asm volatile("ld.shared.v2.s32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(saddr));
    return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu_() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// a counter that grows across launches has reached `target` (wrap-safe)
__device__ __forceinline__ bool reached(unsigned v, unsigned target) { return int(v - target) >= 0; }
// units a waited-for job finishes per launch (its tiles times its parts), from its part 0 entry
__device__ __forceinline__ unsigned unit_count(const StepJob &j)
{
    return unsigned((j.N + 15) >> 4) * unsigned(((j.flags >> kStepSplitShift) & 63) + 1);
}
__device__ __forceinline__ float lo_f32(uint32_t w) { return f16_bits_to_float(uint16_t(w)); }
__device__ __forceinline__ float hi_f32(uint32_t w) { return f16_bits_to_float(uint16_t(w >> 16)); }
// a value the compiler must keep in a register (not recompute in the loop)
__device__ __forceinline__ uint32_t opaque(uint32_t v)
{
    uint32_t r;
    asm volatile("mov.b32 %0, %1;" : "=r"(r) : "r"(v));
    return r;
}

// One segment into the lane's accumulators. MT tokens per pass: the 8 MMA
// columns are (token, group) pairs, GP = 8 / MT groups per pass; lane (r, t)
// supplies column r, i.e. x of token r / GP at group (pass, r % GP), or
// zeros (mk[g] = 0). `E` = the segment's x in the window for this lane's
// token minus the even zero row; the x address of group g is
// mk[g] * E + ka[g]. The lane accumulates groups (pass, (2t mod GP) + {0, 1})
// of rows r, r+8.
template <int MT>
__device__ __forceinline__ void segment(uint32_t cb, uint32_t aoff, uint32_t soff, uint32_t E,
                                        const uint32_t (&mk)[8], const uint32_t (&ka)[8], float (&acc)[4])
{
    constexpr int GP = 8 / MT;
    const uint4 c0 = lds_v4(cb + aoff), c1 = lds_v4(cb + aoff + 16);            // row r: groups 0-3, 4-7
    const uint4 c8 = lds_v4(cb + aoff + 1152), c9 = lds_v4(cb + aoff + 1168);   // row r+8
#pragma unroll
    for (int p = 0; p < MT; ++p) {
        float de[4] = {0.f, 0.f, 0.f, 0.f}, dd[4] = {0.f, 0.f, 0.f, 0.f};   // even / odd groups
#pragma unroll
        for (int gg = 0; gg < GP; ++gg) {
            const int g = p * GP + gg;
            uint32_t pa[4], pb[4];
            unpack_word_f16x2(group_word(c0, c1, g), pa);
            unpack_word_f16x2(group_word(c8, c9, g), pb);
            const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
            const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
            const uint4 xv = lds_v4(mk[g] * E + ka[g]);
            if (gg & 1) {
                mma16816(dd, a0, xv.x, xv.y, dd);
                mma16816(dd, a1, xv.z, xv.w, dd);
            } else {
                mma16816(de, a0, xv.x, xv.y, de);
                mma16816(de, a1, xv.z, xv.w, de);
            }
        }
        // columns 2t (an even group) and 2t+1 (the odd group after it)
        const uint32_t sr = lds_u32(cb + soff + 2 * p * GP), sr8 = lds_u32(cb + soff + 1152 + 2 * p * GP);
        acc[0] = fmaf(lo_f32(sr), de[0], acc[0]);
        acc[1] = fmaf(hi_f32(sr), dd[1], acc[1]);
        acc[2] = fmaf(lo_f32(sr8), de[2], acc[2]);
        acc[3] = fmaf(hi_f32(sr8), dd[3], acc[3]);
    }
}

// Rows r, r+8 of a finished unit: the lane's groups summed, then over the
// lanes of the same token (fixed order). The sums are whole in the holder
// lanes (token tok).
template <int MT>
__device__ __forceinline__ void tile_sums(const float (&acc)[4], float &v0, float &v1)
{
    v0 = acc[0] + acc[1];
    v1 = acc[2] + acc[3];
    v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
    v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
    if (MT == 1) {
        v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
    }
}
template <int MT>
__device__ __forceinline__ bool holder_lane(int lane, int M)
{
    const int t = lane & 3;
    return MT == 1 ? (t == 0) : ((t & 1) == 0 && (t >> 1) < M);
}

// Rows row0 + r, row0 + r + 8 of each token from the holder lanes' sums
// (gate_up: silu(gate) * up of the row pairs).
template <int MT>
__device__ __forceinline__ void write_rows(float v0, float v1, const StepJob &jb, int row0, int lane, int M)
{
    const int r = lane >> 2, t = lane & 3;
    const int tok = MT == 1 ? 0 : (t >> 1);
    const bool writer = holder_lane<MT>(lane, M);
    const int y_stride = (jb.flags & kStepGateUp) ? (jb.N >> 1) : jb.N;
    uint16_t *y = jb.y + size_t(tok) * y_stride;
    if (!(jb.flags & kStepGateUp)) {
        if (writer) {
            if (row0 + r < jb.N) y[row0 + r] = float_to_f16_bits(v0);
            if (row0 + r + 8 < jb.N) y[row0 + r + 8] = float_to_f16_bits(v1);
        }
    } else {
        const float u0 = __shfl_down_sync(0xffffffffu, v0, 4), u1 = __shfl_down_sync(0xffffffffu, v1, 4);
        if (writer && (r & 1) == 0) {
            if (row0 + r + 1 < jb.N) y[(row0 + r) >> 1] = float_to_f16_bits(silu_f32(v0) * u0);
            if (row0 + r + 9 < jb.N) y[(row0 + r + 8) >> 1] = float_to_f16_bits(silu_f32(v1) * u1);
        }
    }
}

// A finished unit of an unsplit job: the whole tile.
template <int MT>
__device__ __forceinline__ void finish_tile(const float (&acc)[4], const StepJob &jb, int row0, int lane, int M)
{
    float v0, v1;
    tile_sums<MT>(acc, v0, v1);
    write_rows<MT>(v0, v1, jb, row0, lane, M);
}

// Where part c of tile rt of a split job keeps its sums: 16 fp32 rows per
// token (parts part_floats apart).
__device__ __forceinline__ size_t part_floats(const StepJob &jb, int M) { return size_t((jb.N + 15) >> 4) * size_t(M) * 16; }
__device__ __forceinline__ float *part_record(const Params &p, const StepJob &jb, int rt, int c, int M)
{
    return p.work + (size_t(jb.pbase) + size_t(rt)) * size_t(M) * 16 + part_floats(jb, M) * size_t(c);
}

// Lane 0 posts (entry, tile) to the finisher once the warp's ring of posts
// has room; false (every lane) if the finisher never made room (a bounded
// wait). The caller's writes of the part's sums come before (__syncwarp).
__device__ __forceinline__ bool post_tile(int entry, int rt, int lane, uint32_t posted, uint32_t taken,
                                          uint32_t posts, volatile int *s_abort, unsigned long long limit)
{
    int ok = 1;
    if (lane == 0) {
        const int n = int(lds_u32(posted));
        const unsigned long long t0 = globaltimer();
        while (n - ld_acquire_cta_s32(taken) >= kPosts) {
            if (*s_abort || globaltimer() - t0 > limit) {
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
        if (ok) {
            asm volatile("st.shared.v2.s32 [%0], {%1, %2};" ::"r"(posts + 8u * uint32_t(n % kPosts)), "r"(entry), "r"(rt)
                         : "memory");
            st_release_cta_s32(posted, n + 1);   // the record (global) and the pair before the count
        }
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// A compute warp's finished tile rt of one part of a split job (one or two
// tokens): its sums into the part's record, then a post to the finisher.
template <int MT>
__device__ __forceinline__ bool post_part(const float (&acc)[4], const StepJob &jb, int entry, int rt, int lane, int M,
                                          const Params &p, uint32_t posted, uint32_t taken, uint32_t posts,
                                          volatile int *s_abort)
{
    float v0, v1;
    tile_sums<MT>(acc, v0, v1);
    const int r = lane >> 2, tok = MT == 1 ? 0 : ((lane & 3) >> 1);
    float *rec = part_record(p, jb, rt, (jb.flags >> kStepPartShift) & 63, M) + size_t(tok) * 16 + r;
    if (holder_lane<MT>(lane, M)) {
        rec[0] = v0;
        rec[8] = v1;
    }
    __syncwarp();
    return post_tile(entry, rt, lane, posted, taken, posts, s_abort, p.wait_ns);
}

// A tile of a split job whose parts have all arrived (the whole warp, after
// the arrival that completed it and an acquire fence): every part's sums
// read back and added in part order (the same order whichever part arrived
// last), the tile's rows written, lane = token * 16 + row.
__device__ __forceinline__ void complete_part(const Params &p, const StepJob &jb, int rt, int lane, int M)
{
    const int C = ((jb.flags >> kStepSplitShift) & 63) + 1;
    const int row = lane & 15, n = rt * 16 + row;
    const size_t step = part_floats(jb, M);
    for (int t0 = 0; t0 < M; t0 += 2) {                  // two tokens per pass
        const int tok = t0 + (lane >> 4);
        float v = 0.f;
        if (tok < M) {
            const float *rec = part_record(p, jb, rt, 0, M) + size_t(tok) * 16 + row;
            for (int c = 0; c < C; ++c) v += __ldcg(rec + step * size_t(c));
        }
        if (!(jb.flags & kStepGateUp)) {
            if (tok < M && n < jb.N) jb.y[size_t(tok) * jb.N + n] = float_to_f16_bits(v);
        } else {
            const float u = __shfl_down_sync(0xffffffffu, v, 1);
            if (tok < M && (row & 1) == 0 && n + 1 < jb.N)
                jb.y[size_t(tok) * (jb.N >> 1) + (n >> 1)] = float_to_f16_bits(silu_f32(v) * u);
        }
    }
}

__device__ __forceinline__ void fail(const Params &p, volatile int *s_abort)
{
    atomicOr(&g_step_error, ZQ4_DEVERR_WAIT_TIMEOUT);
    atomicOr(&p.hdr->abort, 1u);
    *s_abort = 1;
}

// The finisher and publisher warp of a CTA with nw compute warps (k_wide;
// k_step keeps the same steps written out in its body: measured, the call
// form cost the one-token step 15 us, 402.8 against 387.2).
// Finisher (split jobs): takes the compute warps' posted part tiles (one per
// warp at a time, lane w for warp w): a GPU-scope fence and an arrival on
// the tile's counter each; the lane whose arrival completes a tile fences
// (acquire), and the warp adds the parts and writes the tile. Each taken
// tile then counts for publishing. Publisher: makes this CTA's finished
// units of the waited-for jobs visible to every SM: snapshot the shared
// counters (acquire: the units were counted after their outputs were
// written), one GPU-scope fence for the whole batch, then one add per
// changed job. Runs until every compute warp is done (or the CTA aborts).
template <class JobFn>
__device__ __forceinline__ void publisher_loop(const Params &p, uint32_t sbase, uint32_t a_posted, uint32_t a_taken,
                                               uint32_t a_posts, uint32_t a_cta_done, unsigned *cta_pub,
                                               unsigned *cta_snap, uint32_t s_warps_done, volatile int *s_abort,
                                               int nw, int n, int M, unsigned done_mul, int lane, JobFn job)
{
    (void)sbase;
    if (p.n_pub == 0 && !p.split) return;
    int taken_l = 0;                                      // lane w < nw: posts of warp w taken
    for (;;) {
        const bool last = __shfl_sync(0xffffffffu, ld_acquire_cta_s32(s_warps_done) == nw || *s_abort, 0);
        while (p.split) {
            int have = 0, e = 0, rt = 0, done = 0;
            if (lane < nw && ld_acquire_cta_s32(a_posted + 4 * lane) != taken_l) {
                const int2 pr = lds_s2(a_posts + 8 * (lane * kPosts + taken_l % kPosts));
                have = 1;
                e = pr.x;
                rt = pr.y;
                const StepJob &jb = job(e);
                fence_acq_rel_gpu_();
                const unsigned old = atomicAdd(&p.arrive[jb.sbase + rt], 1u);
                done = reached(old + 1u, done_mul * unsigned(((jb.flags >> kStepSplitShift) & 63) + 1));
                if (done) fence_acq_rel_gpu_();
            }
            if (!__any_sync(0xffffffffu, have)) break;
            __syncwarp();
            for (unsigned m = __ballot_sync(0xffffffffu, done); m; m &= m - 1) {
                const int w = __ffs(m) - 1;
                const int ew = __shfl_sync(0xffffffffu, e, w), rw = __shfl_sync(0xffffffffu, rt, w);
                complete_part(p, job(ew), rw, lane, M);
            }
            __syncwarp();                                 // the rows written before the units count
            if (have) {
                const StepJob &jb = job(e);
                if (jb.flags & kStepPublish) red_release_cta(a_cta_done + 4 * (jb.flags >> kStepPubShift), 1u);
                st_release_cta_s32(a_taken + 4 * lane, ++taken_l);
            }
        }
        bool any = false;
        for (int i = lane; i < p.n_pub; i += 32) {
            const unsigned c = unsigned(ld_acquire_cta_s32(a_cta_done + 4 * i));
            cta_snap[i] = c;
            any |= c != cta_pub[i];
        }
        __syncwarp();                                     // the snapshot before the adds read it
        if (__any_sync(0xffffffffu, any)) {
            fence_acq_rel_gpu_();
            for (int j = lane; j < n; j += 32) {
                const StepJob &jb = job(j);
                // every part counts into the job's slot; part 0's entry holds the counter
                if (!(jb.flags & kStepPublish) || (jb.flags & (63 << kStepPartShift))) continue;
                const int i = jb.flags >> kStepPubShift;
                const unsigned c = cta_snap[i];
                if (c != cta_pub[i]) {
                    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(&p.job_done[j]), "r"(c - cta_pub[i])
                                 : "memory");
                    cta_pub[i] = c;
                }
            }
        }
        if (last) break;
        __nanosleep(p.split ? 128 : 500);
    }
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1) k_step(Params p)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128 - (smem_addr(smem_raw) & 127)) & 127);
    const uint32_t sbase = smem_addr(smem);
    const Smem L(p.slots, p.wbytes, p.n_pub, p.cached);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = p.n_jobs, M = p.M, slots = p.slots;
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L.misc);
    const uint32_t s_warps_done = sbase + L.misc + 4;
    unsigned *cta_done = reinterpret_cast<unsigned *>(smem + L.cta_done);
    unsigned *cta_pub = reinterpret_cast<unsigned *>(smem + L.cta_pub);
    unsigned *cta_snap = reinterpret_cast<unsigned *>(smem + L.cta_snap);
    StepJob *sjobs = reinterpret_cast<StepJob *>(smem + L.jobs);
    const unsigned launch = *reinterpret_cast<volatile unsigned *>(&p.hdr->epoch);

    for (int i = threadIdx.x; i < 32; i += kThreads) reinterpret_cast<uint32_t *>(smem + L.zero)[i] = 0;
    for (int i = threadIdx.x; i < p.n_pub; i += kThreads) cta_done[i] = cta_pub[i] = 0;
    for (int i = threadIdx.x; i < kWarps; i += kThreads) {
        reinterpret_cast<int *>(smem + L.wcur)[i] = -1;      // no job being read yet
        reinterpret_cast<int *>(smem + L.wlb)[i] = 0;        // every job may still be read
        reinterpret_cast<int *>(smem + L.posted)[i] = 0;
        reinterpret_cast<int *>(smem + L.taken)[i] = 0;
    }
    for (int i = threadIdx.x; i < kEntries; i += kThreads) reinterpret_cast<int *>(smem + L.xtag)[i] = -1;
    if (threadIdx.x == 0) {
        *s_abort = 0;
        *reinterpret_cast<int *>(smem + L.misc + 4) = 0;
    }
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.jobs);
        uint4 *dst = reinterpret_cast<uint4 *>(sjobs);
        const int words = p.cached * int(sizeof(StepJob) / 16);
        for (int i = threadIdx.x; i < words; i += kThreads) dst[i] = src[i];
    }
    if (warp < kWarps && lane == 0) {
        for (int j = 0; j < slots; ++j) mbar_init(sbase + L.bars + 8 * (warp * slots + j), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kStagerWarp && lane == 0) {
        for (int b = 0; b < kEntries; ++b) mbar_init(sbase + L.xbar + 8 * b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    auto job = [&](int j) -> const StepJob & { return j < p.cached ? sjobs[j] : p.jobs[j]; };
    const unsigned done_mul = launch + 1u;

    if (warp == kStagerWarp) {
        // ---------------- the x stager ----------------
        // x of every job into a byte ring (the window), bytes taken in job
        // order: job j takes M * K_j * 2 bytes (128-byte aligned) at the
        // ring's head, and the oldest jobs give their bytes back once no
        // compute warp of this CTA can still read them (warp w reads its
        // current job cur[w] and, after it, only jobs >= lb[w]). A job's x
        // is copied once its waits are met (the data it reads is final): at
        // once when they are met when its bytes are taken, else the job is
        // pending (bit j - oldest of `pend`) and the stager goes on taking
        // bytes for the jobs after it, copying theirs, and polls the pending
        // ones; a pending job keeps its bytes (and every later job's). Entry
        // j % kEntries holds the job's barrier and tag (job, offset, parity
        // of the fill), published when the copy is issued; readers wait on
        // the barrier. The ring state (head, tail, bytes used, pend) is the
        // same in every lane.
        const uint32_t lb0 = sbase + L.wlb;
        const uint32_t W = uint32_t(p.wbytes);
        int *xtag = reinterpret_cast<int *>(smem + L.xtag);
        uint32_t *xstart = reinterpret_cast<uint32_t *>(smem + L.xstart);
        uint32_t *xtotal = reinterpret_cast<uint32_t *>(smem + L.xtotal);
        uint32_t head = 0, tail = 0, used = 0;
        int oldest = 0;                                      // the oldest job still holding bytes
        int j = 0;                                           // the next job to take bytes
        unsigned pend = 0;
        // are job k's waits met (acquire loads, no waiting)
        auto ready = [&](int k) {
            const StepJob &jk = job(k);
            bool r = true;
            const int nw = (jk.flags >> kStepWaitShift) & 3;
            for (int w = 0; r && w < nw; ++w) {
                const int d = jk.wait[w];
                r = reached(ld_acquire_gpu(&p.job_done[d]), done_mul * unit_count(job(d)));
            }
            return r;
        };
        // lane 0: the copy of job k's x into its bytes; false on a timeout
        auto issue = [&](int k) -> bool {
            const StepJob &jk = job(k);
            const int e = k % kEntries;
            const uint32_t off = xstart[e] + xtotal[e] > W ? 0u : xstart[e];    // wrapped: at 0
            // the entry's previous fill has landed before its barrier is
            // armed again (no compute warp of this CTA may have waited for
            // it: the CTA can have had no tile of that job)
            const bool used_e = xtag[e] >= 0;
            if (used_e && !mbar_wait(sbase + L.xbar + 8 * e, uint32_t(xtag[e] & 1))) return false;
            // the window's last readers (generic proxy) and the data's
            // writers are ordered before the copy (async proxy)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const uint32_t bar = sbase + L.xbar + 8 * e, dst = sbase + L.xwin + off;
            const int par = used_e ? ((xtag[e] & 1) ^ 1) : 0;   // the phase this fill completes
            mbar_arrive_expect_tx(bar, uint32_t(M * jk.K * 2));
            for (int m = 0; m < M; ++m)
                bulk_load(dst + uint32_t(m * jk.K * 2), jk.x + size_t(m) * size_t(jk.tstride) * 256, uint32_t(jk.K * 2), bar);
            // job, offset and parity in one word: a reader that sees the job
            // waits for that phase on the barrier, which orders the data
            *reinterpret_cast<volatile int *>(xtag + e) = (k << kTagJobShift) | int((off >> 7) << 1) | par;
            return true;
        };
        unsigned long long t0 = globaltimer();               // the last progress
        int ok = 1;
        while (j < n || pend) {
            if (__shfl_sync(0xffffffffu, *s_abort, 0)) break;
            bool progress = false;
            // give back the bytes of the oldest jobs nobody reads any more
            // (never a pending job's): the bound first (acquire), then the
            // current job (a warp stores its current job before it raises
            // its bound)
            int wl = lane < kWarps ? ld_acquire_cta_s32(lb0 + 4 * lane) : 0x7fffffff;
            const int wc = lane < kWarps ? *reinterpret_cast<volatile int *>(smem + L.wcur + 4 * lane) : -1;
#pragma unroll
            for (int o = 16; o; o >>= 1) wl = min(wl, __shfl_xor_sync(0xffffffffu, wl, o));
            while (oldest < j && oldest < wl && !(pend & 1u) &&
                   !__any_sync(0xffffffffu, lane < kWarps && wc == oldest)) {
                const int oe = oldest % kEntries;
                used -= xtotal[oe];
                tail = xstart[oe] + xtotal[oe];
                if (tail >= W) tail -= W;
                ++oldest;
                pend >>= 1;
                progress = true;
            }
            if (used == 0) head = tail = 0;
            // pending jobs whose waits are now met (each lane polls one; lane
            // 0 checks again with its own acquire loads before the copy)
            if (pend) {
                const bool mine = (pend >> lane) & 1u;
                unsigned rdy = __ballot_sync(0xffffffffu, mine && ready(oldest + lane));
                while (rdy) {
                    const int b = __ffs(rdy) - 1;
                    rdy &= rdy - 1;
                    int r = 1;
                    if (lane == 0) r = ready(oldest + b) ? (issue(oldest + b) ? 1 : -1) : 0;
                    r = __shfl_sync(0xffffffffu, r, 0);
                    if (r < 0) {
                        ok = 0;
                        break;
                    }
                    if (r > 0) {
                        pend &= ~(1u << b);
                        progress = true;
                    }
                }
                if (!ok) break;
            }
            // bytes for job j: room at the head (wrapping to 0 wastes the end
            // of the ring), and the entry's previous job has given its bytes back
            if (j < n && j - oldest < kEntries) {
                const StepJob &jb = job(j);
                const uint32_t size = (uint32_t(M * jb.K * 2) + 127u) & ~127u;
                bool room = false;
                uint32_t off = 0, total = size;
                if (used == 0) {                             // empty (head = tail = 0)
                    room = size <= W;
                } else if (tail < head) {                    // data in [tail, head)
                    if (head + size <= W) {
                        room = true;
                        off = head;
                    } else if (size <= tail) {
                        room = true;
                        total = W - head + size;
                    }
                } else if (head + size <= tail) {            // data in [tail, W) and [0, head); full if equal
                    room = true;
                    off = head;
                }
                if (room) {
                    const int e = j % kEntries;
                    xstart[e] = head;                        // every lane writes the same values
                    xtotal[e] = total;
                    used += total;
                    head = off + size;
                    if (head >= W) head = 0;
                    __syncwarp();
                    int r = 0;
                    if (lane == 0) r = ready(j) ? (issue(j) ? 1 : -1) : 0;
                    r = __shfl_sync(0xffffffffu, r, 0);
                    if (r < 0) {
                        ok = 0;
                        break;
                    }
                    if (r == 0) pend |= 1u << (j - oldest);
                    ++j;
                    progress = true;
                }
            }
            if (progress) {
                t0 = globaltimer();
            } else {
                int stop = 0;
                if (lane == 0)
                    stop = *reinterpret_cast<volatile unsigned *>(&p.hdr->abort) || globaltimer() - t0 > p.wait_ns;
                if (__shfl_sync(0xffffffffu, stop, 0)) {
                    ok = 0;
                    break;
                }
                __nanosleep(128);
            }
        }
        if (!ok && lane == 0) fail(p, s_abort);
        __syncwarp();
        // the last fill of every entry has landed before the CTA may exit
        if (lane == 0)
            for (int c = 0; c < kEntries; ++c)
                if (xtag[c] >= 0 && !mbar_wait(sbase + L.xbar + 8 * c, uint32_t(xtag[c] & 1))) break;
    } else if (warp == kPubWarp) {
        // ---------------- the finisher and publisher ----------------
        // Finisher (split jobs): takes the compute warps' posted part tiles
        // (one per warp at a time, lane w for warp w): a GPU-scope fence and
        // an arrival on the tile's counter each; the lane whose arrival
        // completes a tile fences (acquire), and the warp adds the parts and
        // writes the tile. Each taken tile then counts for publishing.
        // Publisher: makes this CTA's finished units of the waited-for jobs
        // visible to every SM: snapshot the shared counters (acquire: the
        // units were counted after their outputs were written), one
        // GPU-scope fence for the whole batch, then one add per changed job.
        if (p.n_pub > 0 || p.split) {
            int taken_l = 0;                              // lane w < kWarps: posts of warp w taken
            for (;;) {
                const bool last = __shfl_sync(0xffffffffu, ld_acquire_cta_s32(s_warps_done) == kWarps || *s_abort, 0);
                while (p.split) {
                    int have = 0, e = 0, rt = 0, done = 0;
                    if (lane < kWarps && ld_acquire_cta_s32(sbase + L.posted + 4 * lane) != taken_l) {
                        const int2 pr = *reinterpret_cast<const int2 *>(smem + L.posts +
                                                                         8 * (lane * kPosts + taken_l % kPosts));
                        have = 1;
                        e = pr.x;
                        rt = pr.y;
                        const StepJob &jb = job(e);
                        fence_acq_rel_gpu_();
                        const unsigned old = atomicAdd(&p.arrive[jb.sbase + rt], 1u);
                        done = reached(old + 1u, done_mul * unsigned(((jb.flags >> kStepSplitShift) & 63) + 1));
                        if (done) fence_acq_rel_gpu_();
                    }
                    if (!__any_sync(0xffffffffu, have)) break;
                    __syncwarp();
                    for (unsigned m = __ballot_sync(0xffffffffu, done); m; m &= m - 1) {
                        const int w = __ffs(m) - 1;
                        const int ew = __shfl_sync(0xffffffffu, e, w), rw = __shfl_sync(0xffffffffu, rt, w);
                        complete_part(p, job(ew), rw, lane, M);
                    }
                    __syncwarp();                         // the rows written before the units count
                    if (have) {
                        const StepJob &jb = job(e);
                        if (jb.flags & kStepPublish) red_release_cta(sbase + L.cta_done + 4 * (jb.flags >> kStepPubShift), 1u);
                        st_release_cta_s32(sbase + L.taken + 4 * lane, ++taken_l);
                    }
                }
                bool any = false;
                for (int i = lane; i < p.n_pub; i += 32) {
                    const unsigned c = unsigned(ld_acquire_cta_s32(sbase + L.cta_done + 4 * i));
                    cta_snap[i] = c;
                    any |= c != cta_pub[i];
                }
                __syncwarp();                             // the snapshot before the adds read it
                if (__any_sync(0xffffffffu, any)) {
                    fence_acq_rel_gpu_();
                    for (int j = lane; j < n; j += 32) {
                        const StepJob &jb = job(j);
                        // every part counts into the job's slot; part 0's entry holds the counter
                        if (!(jb.flags & kStepPublish) || (jb.flags & (63 << kStepPartShift))) continue;
                        const int i = jb.flags >> kStepPubShift;
                        const unsigned c = cta_snap[i];
                        if (c != cta_pub[i]) {
                            asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(&p.job_done[j]),
                                         "r"(c - cta_pub[i])
                                         : "memory");
                            cta_pub[i] = c;
                        }
                    }
                }
                if (last) break;
                __nanosleep(p.split ? 128 : 500);
            }
        }
    } else {
        // ---------------- compute warps ----------------
        const int r = lane >> 2, t = lane & 3;
        constexpr int GP = 8 / MT;
        const bool leader = lane == 0;
        const uint32_t ring = sbase + L.ring + uint32_t(warp * slots) * kSegBytes;
        const uint32_t bars = sbase + L.bars + uint32_t(8 * warp * slots);
        const uint32_t descs = sbase + L.desc + uint32_t(16 * warp * slots);
        const uint32_t my_cur = sbase + L.wcur + 4 * warp, my_lb = sbase + L.wlb + 4 * warp;
        const uint32_t my_posted = sbase + L.posted + 4 * warp, my_taken = sbase + L.taken + 4 * warp;
        const uint32_t my_posts = sbase + L.posts + uint32_t(8 * kPosts * warp);
        const uint32_t aoff = opaque(segk::lane_code_offset(lane));
        const uint32_t soff = opaque(uint32_t(r * 144 + 128 + 2 * ((2 * t) % GP)));
        // x addresses: lane column r is token r / GP, group slot r % GP; the
        // zero rows are two 64-byte rows placed so that the active and the
        // idle lanes of one load never share a bank (even groups: z0, odd: z1)
        const int mtok = r / GP;
        const uint32_t z1 = sbase + L.zero, z0 = z1 + 64;
        uint32_t mk[8], ka[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const bool act = (r % GP) == (g % GP) && mtok < M;
            const uint32_t z = (g & 1) ? z1 : z0;
            mk[g] = opaque(act ? 1u : 0u);
            ka[g] = opaque(z + 16 * t + (act ? uint32_t(64 * g) + z0 - z : 0u));
        }
        const uint32_t ex = opaque(sbase + L.xwin - z0);   // + the job's offset + token * K * 2 + 512 sg

        // The issue cursor, the same in every lane: the tile whose segments
        // are being copied (job ijob, tile itile, next segment isg of iS) and
        // the tile reserved after it (its index only in lane 0's `nt`, read
        // when it is needed, so that the atomic's latency is never waited on).
        // Lane 0's copies and atomics are predicated, not branched around.
        const uint32_t lead = leader ? 1u : 0u;
        int fj = 0, ijob = 0, itile = 0, isg = 0, iS = 1, islot = 0;
        const uint8_t *iptr = nullptr;
        bool ihave = false, iend = false, reserved = false;
        unsigned nt = 0;
        unsigned *const ctr = &p.hdr->next_tile;
        auto reserve = [&](uint32_t pred) {          // lane 0 (when pred): nt = next tile index
            asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t@p atom.global.add.u32 %0, [%2], 1;\n\t}"
                         : "+r"(nt)
                         : "r"(pred), "l"(ctr)
                         : "memory");
        };
        auto next_tile = [&]() {                      // the next tile into the cursor, or the end
            if (!reserved) reserve(lead);
            reserved = false;
            const unsigned g = __shfl_sync(0xffffffffu, nt, 0);
            if (g >= unsigned(p.total_tiles)) {
                iend = true;
                return;
            }
            while (int(g) >= job(fj).tile0 + ((job(fj).N + 15) >> 4)) ++fj;
            ijob = fj;
            itile = int(g) - job(fj).tile0;
            isg = 0;
            iS = job(fj).K >> 8;
            iptr = job(fj).seg + size_t(itile) * size_t(job(fj).tstride) * kSegBytes;
            ihave = true;
            // every job the warp reads after its current one is >= this one's
            // (valid when every job's tile is at least a ring long: the tile
            // issued before this one has started to be read)
            if (p.fine && leader) st_release_cta_s32(my_lb, ijob);
        };
        // copy the cursor's next segment into slot islot; the descriptor
        // (job, tile, segment, segments in the tile) tells the consumer where
        // a tile starts and ends. False when no tile is left.
        auto issue_next = [&]() -> bool {
            if (!ihave) {
                if (iend) return false;
                next_tile();
                if (iend) return false;
            }
            const bool res = !reserved && isg == (iS >> 1);     // the tile after this one, half a tile ahead
            reserve(res ? lead : 0u);
            reserved |= res;
            const uint32_t bar = bars + 8 * islot;
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "setp.ne.u32 p, %0, 0;\n\t"
                "@p st.shared.v4.s32 [%1], {%2, %3, %4, %5};\n\t"
                "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%6], %7;\n\t"
                "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%8], [%9], %7, [%6];\n\t"
                "}" ::"r"(lead),
                "r"(descs + 16 * islot), "r"(ijob), "r"(itile), "r"(isg), "r"(iS), "r"(bar),
                "r"(uint32_t(kSegBytes)), "r"(ring + uint32_t(islot) * kSegBytes), "l"(iptr)
                : "memory");
            iptr += kSegBytes;
            ihave = ++isg < iS;
            islot = islot + 1 == slots ? 0 : islot + 1;
            return true;
        };

        int in_flight = 0;
        while (in_flight < slots && issue_next()) ++in_flight;

        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        int cslot = 0, cjob = -1, cbuf = 0;
        uint32_t cphase = 0, E = 0;
        bool ok = true;
        while (in_flight > 0) {
            if (!__all_sync(0xffffffffu, mbar_wait(bars + 8 * cslot, cphase))) {
                ok = false;
                break;
            }
            const int4 d = lds_s4(descs + 16 * cslot);     // job, tile, segment, segments
            if (d.z == 0) {
                // a tile starts: its job's x in the window (staged once per CTA)
                if (d.x != cjob) {
                    if (leader) {
                        *reinterpret_cast<volatile int *>(smem + L.wcur + 4 * warp) = d.x;
                        if (!p.fine) st_release_cta_s32(my_lb, d.x);
                    }
                    const unsigned long long t0 = globaltimer();
                    const int e = d.x % kEntries;
                    int v = -1;
                    for (;;) {
                        v = *reinterpret_cast<volatile int *>(smem + L.xtag + 4 * e);
                        if (v >= 0 && (v >> kTagJobShift) == d.x) break;
                        if (*s_abort || globaltimer() - t0 > p.wait_ns) {
                            v = -1;
                            break;
                        }
                        __nanosleep(32);
                    }
                    if (!__all_sync(0xffffffffu, v >= 0 && mbar_wait(sbase + L.xbar + 8 * e, uint32_t(v & 1)))) {
                        ok = false;
                        break;
                    }
                    cjob = d.x;
                    cbuf = int(((uint32_t(v) >> 1) & 2047u) << 7) + mtok * job(d.x).K * 2;
                }
                E = ex + uint32_t(cbuf);
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = 0.f;
            }
            segment<MT>(ring + uint32_t(cslot) * kSegBytes, aoff, soff, E, mk, ka, acc);
            E += 512;
            // every lane's reads of the slot (generic proxy) are done before
            // lane 0's copy (async proxy) refills it
            __syncwarp();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (!issue_next()) --in_flight;
            if (d.z == d.w - 1) {
                const StepJob &jb = job(d.x);
                if (!(jb.flags & (63 << kStepSplitShift))) {
                    finish_tile<MT>(acc, jb, d.y * 16, lane, M);
                    if (jb.flags & kStepPublish) {
                        __syncwarp();
                        if (leader) red_release_cta(sbase + L.cta_done + 4 * (jb.flags >> kStepPubShift), 1u);
                    }
                } else if (!post_part<MT>(acc, jb, d.x, d.y, lane, M, p, my_posted, my_taken, my_posts, s_abort)) {
                    ok = false;      // (the finisher counts a posted tile: it is published once written)
                }
            }
            if (++cslot == slots) {
                cslot = 0;
                cphase ^= 1u;
            }
            if (!ok) break;
        }
        if (!ok && leader) fail(p, s_abort);
        // after a failed wait: the copies still in flight land before the CTA exits
        if (!ok && leader)
            for (int c = 0; c < in_flight; ++c) {
                const int s = (cslot + c) % slots;
                if (!mbar_wait(bars + 8 * s, cphase ^ (cslot + c >= slots ? 1u : 0u))) break;
            }
        __syncwarp();
        if (leader) {
            st_release_cta_s32(my_cur, 0x7fffffff);             // reads no more x
            st_release_cta_s32(my_lb, 0x7fffffff);
            red_release_cta(s_warps_done, 1u);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (*s_abort) {
            atomicOr(&g_step_error, ZQ4_DEVERR_WAIT_TIMEOUT);
        } else {
            __threadfence();
            const unsigned target = (launch + 1u) * gridDim.x;
            const unsigned d = atomicAdd(&p.hdr->done, 1u);
            if (d == target - 1u) {                       // the last CTA of this launch
                p.hdr->next_tile = 0;
                __threadfence();
                atomicAdd(&p.hdr->epoch, 1u);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Three to sixteen tokens (k_wide)
// ---------------------------------------------------------------------------
// Same plan, units, counter, waits, split parts and finisher/publisher warp
// as k_step; what differs: column n of the m16n8k16 accumulator is token n
// (a block of 8 tokens; 16 tokens: two blocks from one unpack), the group
// scales are applied per group (fp32, after the group's two MMAs), and x
// comes with each segment: every ring slot holds the 2304-byte segment and
// x[M][256] of its 256 columns, brought by one 2D tensor copy from the job
// entry's tensor map (no x window). A warp checks the waits of a job when
// its cursor first reaches it; if they are not met it consumes what it has
// in flight and waits only once its ring is empty (a unit of an earlier job
// may still be in its ring).
template <int MT>
struct Wide {
    static constexpr int kGroup = MT <= 8 ? 1 : 2;     // 16-row tiles per unit (they share x)
    static constexpr int kWarps = MT <= 8 ? 16 : 8;    // compute warps
    static constexpr int kThreads = (kWarps + 1) * 32; // + the finisher/publisher warp
};
static_assert(Wide<16>::kGroup == kWideGroup16, "host and kernel agree on the unit size");

struct WSmem {
    uint32_t ring, bars, desc, posted, taken, posts, misc, cta_done, cta_pub, cta_snap, jobs, total;
    __host__ __device__ WSmem(int nw, int slots, int slot_bytes, int n_pub, int cached)
    {
        ring = 0;
        bars = ring + uint32_t(nw * slots) * uint32_t(slot_bytes);
        desc = bars + uint32_t(nw * slots) * 8;
        posted = desc + uint32_t(nw * slots) * 16;
        taken = posted + uint32_t(nw) * 4;
        posts = taken + uint32_t(nw) * 4;
        misc = posts + uint32_t(nw * kPosts) * 8;
        cta_done = misc + 64;
        cta_pub = cta_done + uint32_t(n_pub) * 4;
        cta_snap = cta_pub + uint32_t(n_pub) * 4;
        jobs = (cta_snap + uint32_t(n_pub) * 4 + 15) / 16 * 16;
        total = jobs + uint32_t(cached) * uint32_t(sizeof(StepJob));
    }
};

__device__ __forceinline__ float scale_of(const uint4 &s, int g)
{
    const uint32_t w = g < 2 ? s.x : g < 4 ? s.y : g < 6 ? s.z : s.w;
    return (g & 1) ? hi_f32(w) : lo_f32(w);
}

// One segment of G tiles (at cb + 2304 i) into the lane's accumulators:
// acc[i][4 b + j] = tile i, block b of 8 tokens (rows r, r + 8 x tokens
// 8b + 2t, 8b + 2t + 1). x of the lane's token of block b: 16 bytes at
// xr[b] + 64 g (columns 32 g + 8 t ..), shared by the G tiles.
template <int MT, int G>
__device__ __forceinline__ void segment_wide(uint32_t cb, uint32_t aoff, uint32_t srow, const uint32_t (&xr)[MT / 8],
                                             float (&acc)[G][MT / 2])
{
    uint4 c0[G], c1[G], c8[G], c9[G], s0[G], s8[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
        const uint32_t tb = cb + uint32_t(i * kSegBytes);
        c0[i] = lds_v4(tb + aoff);                       // row r: groups 0-3, 4-7
        c1[i] = lds_v4(tb + aoff + 16);
        c8[i] = lds_v4(tb + aoff + 1152);                // row r+8
        c9[i] = lds_v4(tb + aoff + 1168);
        s0[i] = lds_v4(tb + srow);                       // their 8 group scales
        s8[i] = lds_v4(tb + srow + 1152);
    }
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        uint4 xv[MT / 8];
#pragma unroll
        for (int b = 0; b < MT / 8; ++b) xv[b] = lds_v4(xr[b] + 64 * g);
#pragma unroll
        for (int i = 0; i < G; ++i) {
            uint32_t pa[4], pb[4];
            unpack_word_f16x2(group_word(c0[i], c1[i], g), pa);
            unpack_word_f16x2(group_word(c8[i], c9[i], g), pb);
            const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
            const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
            const float sr = scale_of(s0[i], g), sr8 = scale_of(s8[i], g);
#pragma unroll
            for (int b = 0; b < MT / 8; ++b) {
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma16816(d, a0, xv[b].x, xv[b].y, d);
                mma16816(d, a1, xv[b].z, xv[b].w, d);
                acc[i][4 * b + 0] = fmaf(sr, d[0], acc[i][4 * b + 0]);
                acc[i][4 * b + 1] = fmaf(sr, d[1], acc[i][4 * b + 1]);
                acc[i][4 * b + 2] = fmaf(sr8, d[2], acc[i][4 * b + 2]);
                acc[i][4 * b + 3] = fmaf(sr8, d[3], acc[i][4 * b + 3]);
            }
        }
    }
}

// A finished whole tile: rows row0 + r, row0 + r + 8 of tokens 8b + 2t and
// 8b + 2t + 1 (gate_up: silu(gate) * up of the row pairs, up from the lane
// of row r + 1).
template <int MT>
__device__ __forceinline__ void finish_wide(const float (&acc)[MT / 2], const StepJob &jb, int row0, int lane, int M)
{
    const int r = lane >> 2, t = lane & 3;
    const bool gu = jb.flags & kStepGateUp;
    const int ys = gu ? (jb.N >> 1) : jb.N;
#pragma unroll
    for (int b = 0; b < MT / 8; ++b) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {                    // rows r (h = 0), r + 8 (h = 1)
            const int row = row0 + r + 8 * h;
#pragma unroll
            for (int q = 0; q < 2; ++q) {                // tokens 8b + 2t + q
                const int tok = 8 * b + 2 * t + q;
                const float v = acc[4 * b + 2 * h + q];
                if (!gu) {
                    if (tok < M && row < jb.N) jb.y[size_t(tok) * ys + row] = float_to_f16_bits(v);
                } else {
                    const float u = __shfl_down_sync(0xffffffffu, v, 4);
                    if (tok < M && (r & 1) == 0 && row + 1 < jb.N)
                        jb.y[size_t(tok) * ys + (row >> 1)] = float_to_f16_bits(silu_f32(v) * u);
                }
            }
        }
    }
}

// A finished tile rt of one part of a split job: its sums into the part's
// record (16 rows per token), then a post to the finisher.
template <int MT>
__device__ __forceinline__ bool post_part_wide(const float (&acc)[MT / 2], const StepJob &jb, int entry, int rt,
                                               int lane, int M, const Params &p, uint32_t posted, uint32_t taken,
                                               uint32_t posts, volatile int *s_abort)
{
    const int r = lane >> 2, t = lane & 3;
    float *rec = part_record(p, jb, rt, (jb.flags >> kStepPartShift) & 63, M) + r;
#pragma unroll
    for (int b = 0; b < MT / 8; ++b)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int tok = 8 * b + 2 * t + q;
                if (tok < M) rec[size_t(tok) * 16 + 8 * h] = acc[4 * b + 2 * h + q];
            }
    __syncwarp();
    return post_tile(entry, rt, lane, posted, taken, posts, s_abort, p.wait_ns);
}

template <int MT>
__global__ void __launch_bounds__(Wide<MT>::kThreads, 1) k_wide(Params p)
{
    constexpr int NW = Wide<MT>::kWarps, G = Wide<MT>::kGroup;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128 - (smem_addr(smem_raw) & 127)) & 127);
    const uint32_t sbase = smem_addr(smem);
    const int slots = p.slots, slot_bytes = p.slot_bytes;
    const WSmem L(NW, slots, slot_bytes, p.n_pub, p.cached);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = p.n_jobs, M = p.M;
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L.misc);
    const uint32_t s_warps_done = sbase + L.misc + 4;
    unsigned *cta_done = reinterpret_cast<unsigned *>(smem + L.cta_done);
    unsigned *cta_pub = reinterpret_cast<unsigned *>(smem + L.cta_pub);
    unsigned *cta_snap = reinterpret_cast<unsigned *>(smem + L.cta_snap);
    StepJob *sjobs = reinterpret_cast<StepJob *>(smem + L.jobs);
    const unsigned launch = *reinterpret_cast<volatile unsigned *>(&p.hdr->epoch);

    for (int i = threadIdx.x; i < p.n_pub; i += blockDim.x) cta_done[i] = cta_pub[i] = 0;
    for (int i = threadIdx.x; i < NW; i += blockDim.x) {
        reinterpret_cast<int *>(smem + L.posted)[i] = 0;
        reinterpret_cast<int *>(smem + L.taken)[i] = 0;
    }
    if (threadIdx.x == 0) {
        *s_abort = 0;
        *reinterpret_cast<int *>(smem + L.misc + 4) = 0;
    }
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.jobs);
        uint4 *dst = reinterpret_cast<uint4 *>(sjobs);
        const int words = p.cached * int(sizeof(StepJob) / 16);
        for (int i = threadIdx.x; i < words; i += blockDim.x) dst[i] = src[i];
    }
    if (warp < NW && lane == 0) {
        for (int j = 0; j < slots; ++j) mbar_init(sbase + L.bars + 8 * (warp * slots + j), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    auto job = [&](int j) -> const StepJob & { return j < p.cached ? sjobs[j] : p.jobs[j]; };
    auto units_of = [&](const StepJob &e) { return (((e.N + 15) >> 4) + G - 1) / G; };
    const unsigned done_mul = launch + 1u;

    if (warp == NW) {
        publisher_loop(p, sbase, sbase + L.posted, sbase + L.taken, sbase + L.posts, sbase + L.cta_done, cta_pub,
                       cta_snap, s_warps_done, s_abort, NW, n, M, done_mul, lane, job);
    } else {
        const int r = lane >> 2, t = lane & 3;
        const bool leader = lane == 0;
        const uint32_t ring = sbase + L.ring + uint32_t(warp * slots) * uint32_t(slot_bytes);
        const uint32_t bars = sbase + L.bars + uint32_t(8 * warp * slots);
        const uint32_t descs = sbase + L.desc + uint32_t(16 * warp * slots);
        const uint32_t my_posted = sbase + L.posted + 4 * warp, my_taken = sbase + L.taken + 4 * warp;
        const uint32_t my_posts = sbase + L.posts + uint32_t(8 * kPosts * warp);
        const uint32_t aoff = segk::lane_code_offset(lane);
        const uint32_t srow = uint32_t(r * 144 + 128);
        // x of the lane's token in a slot (tokens past M read token M - 1: their columns are dropped)
        uint32_t xoff[MT / 8];
#pragma unroll
        for (int b = 0; b < MT / 8; ++b) xoff[b] = uint32_t(G * kSegBytes + min(8 * b + r, M - 1) * 512 + 16 * t);

        const uint32_t lead = leader ? 1u : 0u;
        int fj = 0, ijob = 0, itile = 0, isg = 0, iS = 1, islot = 0, checked = -1, ivalid = 1;
        const uint8_t *iptr = nullptr;
        size_t istride = 0;                                   // bytes from one tile's segment to the next tile's
        bool ihave = false, iend = false, reserved = false;
        unsigned nt = 0;
        unsigned *const ctr = &p.hdr->next_tile;
        auto reserve = [&](uint32_t pred) {
            asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t@p atom.global.add.u32 %0, [%2], 1;\n\t}"
                         : "+r"(nt)
                         : "r"(pred), "l"(ctr)
                         : "memory");
        };
        auto next_tile = [&]() {
            if (!reserved) reserve(lead);
            reserved = false;
            const unsigned g = __shfl_sync(0xffffffffu, nt, 0);
            if (g >= unsigned(p.total_tiles)) {
                iend = true;
                return;
            }
            while (int(g) >= job(fj).tile0 + units_of(job(fj))) ++fj;
            ijob = fj;
            itile = int(g) - job(fj).tile0;                   // unit: tiles G itile ..
            isg = 0;
            iS = job(fj).K >> 8;
            istride = size_t(job(fj).tstride) * kSegBytes;
            iptr = job(fj).seg + size_t(G * itile) * istride;
            ivalid = min(G, ((job(fj).N + 15) >> 4) - G * itile);
            ihave = true;
        };
        // are the waits of entry e met (lane 0's acquire loads, broadcast)
        auto ready = [&](int e) -> bool {
            int ok = 1;
            if (leader) {
                const StepJob &jk = job(e);
                const int nw = (jk.flags >> kStepWaitShift) & 3;
                for (int w = 0; ok && w < nw; ++w) {
                    const int d = jk.wait[w];
                    ok = reached(ld_acquire_gpu(&p.job_done[d]), done_mul * unit_count(job(d)));
                }
                // the data the waits guard is read by the tensor copies (async proxy)
                if (ok && nw) asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            return __shfl_sync(0xffffffffu, ok, 0) != 0;
        };
        // copy the cursor's next segment and its x into slot islot: 1 issued,
        // 0 no unit left, -1 the cursor's job waits for jobs not done yet
        auto issue_next = [&]() -> int {
            if (!ihave) {
                if (iend) return 0;
                next_tile();
                if (iend) return 0;
            }
            if (ijob != checked) {
                if (!ready(ijob)) return -1;
                checked = ijob;
            }
            const bool res = !reserved && isg == (iS >> 1);
            reserve(res ? lead : 0u);
            reserved |= res;
            const uint32_t bar = bars + 8 * islot, dst = ring + uint32_t(islot) * uint32_t(slot_bytes);
            const uint32_t tx = uint32_t(ivalid * kSegBytes + M * 512);   // bytes this slot receives
            const CUtensorMap *tm = p.tmaps + ijob;
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "setp.ne.u32 p, %0, 0;\n\t"
                "@p st.shared.v4.s32 [%1], {%2, %3, %4, %5};\n\t"
                "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%6], %7;\n\t"
                "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%8], [%9], %10, [%6];\n\t"
                "@p cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%11], [%12, {%13, %14}], [%6];\n\t"
                "}" ::"r"(lead),
                "r"(descs + 16 * islot), "r"(ijob), "r"(itile), "r"(isg), "r"(iS), "r"(bar), "r"(tx), "r"(dst),
                "l"(iptr), "r"(uint32_t(kSegBytes)), "r"(dst + uint32_t(G * kSegBytes)),
                "l"(reinterpret_cast<uint64_t>(tm)), "r"(isg * 256), "r"(0)
                : "memory");
#pragma unroll
            for (int k = 1; k < G; ++k)                       // the unit's other tiles (when they exist)
                asm volatile(
                    "{\n\t.reg .pred p;\n\t"
                    "setp.ne.u32 p, %0, 0;\n\t"
                    "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%1], [%2], %3, [%4];\n\t"
                    "}" ::"r"(k < ivalid ? lead : 0u),
                    "r"(dst + uint32_t(k * kSegBytes)), "l"(iptr + size_t(k) * istride), "r"(uint32_t(kSegBytes)),
                    "r"(bar)
                    : "memory");
            iptr += kSegBytes;
            ihave = ++isg < iS;
            islot = islot + 1 == slots ? 0 : islot + 1;
            return 1;
        };

        int in_flight = 0;
        bool blocked = false, ok = true;
        for (;;) {
            const int rv = issue_next();
            if (rv <= 0) {
                blocked = rv < 0;
                break;
            }
            if (++in_flight == slots) break;
        }
        float acc[G][MT / 2];
#pragma unroll
        for (int k = 0; k < G; ++k)
#pragma unroll
            for (int i = 0; i < MT / 2; ++i) acc[k][i] = 0.f;
        int cslot = 0;
        uint32_t cphase = 0;
        while (in_flight > 0 || blocked) {
            if (in_flight == 0) {
                // nothing in flight: every unit this warp took is finished; wait for the job's waits
                const unsigned long long t0 = globaltimer();
                int rv = -1;
                while ((rv = issue_next()) < 0) {
                    if (*s_abort || *reinterpret_cast<volatile unsigned *>(&p.hdr->abort) ||
                        globaltimer() - t0 > p.wait_ns) {
                        ok = false;
                        break;
                    }
                    __nanosleep(256);
                }
                if (!ok) break;
                blocked = false;
                if (rv == 0) break;
                ++in_flight;
                continue;
            }
            if (!__all_sync(0xffffffffu, mbar_wait(bars + 8 * cslot, cphase))) {
                ok = false;
                break;
            }
            const uint32_t cb = ring + uint32_t(cslot) * uint32_t(slot_bytes);
            const int4 d = lds_s4(descs + 16 * cslot);
            if (d.z == 0) {
#pragma unroll
                for (int k = 0; k < G; ++k)
#pragma unroll
                    for (int i = 0; i < MT / 2; ++i) acc[k][i] = 0.f;
            }
            uint32_t xr[MT / 8];
#pragma unroll
            for (int b = 0; b < MT / 8; ++b) xr[b] = cb + xoff[b];
            segment_wide<MT, G>(cb, aoff, srow, xr, acc);
            // every lane's reads of the slot are done before lane 0's copies refill it
            __syncwarp();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            --in_flight;
            if (!blocked) {
                const int rv = issue_next();
                if (rv > 0) ++in_flight;
                blocked = rv < 0;
            } else if (issue_next() > 0) {
                ++in_flight;
                blocked = false;
            }
            if (d.z == d.w - 1) {
                const StepJob &jb = job(d.x);
                const int tiles = (jb.N + 15) >> 4;
#pragma unroll
                for (int k = 0; k < G; ++k) {
                    const int rt = G * d.y + k;
                    if (rt >= tiles) break;
                    if (!(jb.flags & (63 << kStepSplitShift))) {
                        finish_wide<MT>(acc[k], jb, rt * 16, lane, M);
                        if (jb.flags & kStepPublish) {
                            __syncwarp();
                            if (leader) red_release_cta(sbase + L.cta_done + 4 * (jb.flags >> kStepPubShift), 1u);
                        }
                    } else if (!post_part_wide<MT>(acc[k], jb, d.x, rt, lane, M, p, my_posted, my_taken, my_posts,
                                                   s_abort)) {
                        ok = false;
                        break;
                    }
                }
            }
            if (++cslot == slots) {
                cslot = 0;
                cphase ^= 1u;
            }
            if (!ok) break;
        }
        if (!ok && leader) fail(p, s_abort);
        // after a failed wait: the copies still in flight land before the CTA exits
        if (!ok && leader)
            for (int c = 0; c < in_flight; ++c) {
                const int sl = (cslot + c) % slots;
                if (!mbar_wait(bars + 8 * sl, cphase ^ (cslot + c >= slots ? 1u : 0u))) break;
            }
        __syncwarp();
        if (leader) red_release_cta(s_warps_done, 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (*s_abort) {
            atomicOr(&g_step_error, ZQ4_DEVERR_WAIT_TIMEOUT);
        } else {
            __threadfence();
            const unsigned target = (launch + 1u) * gridDim.x;
            const unsigned dn = atomicAdd(&p.hdr->done, 1u);
            if (dn == target - 1u) {
                p.hdr->next_tile = 0;
                __threadfence();
                atomicAdd(&p.hdr->epoch, 1u);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// The MoE block's expert stages (k_moe)
// ---------------------------------------------------------------------------
// A stage of zq4_moe_block: MODE 1 gate_up + SiLU*mul (x = the T tokens,
// output h per (token, slot) pair), MODE 2 down (x = h of the P pairs,
// output fp32 z per pair). Every CTA stages all of x once and builds the
// expert grouping; a work unit is (touched expert, block of up to 16 of its
// pairs, 16-row tile of its matrix), dealt round-robin to the warps of the
// grid; each warp streams its units' segments (the bank in the segmented
// layout) through its own ring of bulk copies, the next unit's copies in
// flight while it finishes the current one. Column m of the accumulator is
// the block's pair m (two blocks of 8 when it has more than 8 pairs).
constexpr int kMoeWarps = 12;

struct MoeParams {
    const uint8_t *seg;       // the bank, segmented ([E * N rows] x K)
    const uint16_t *x;        // [rows][K]
    const int32_t *ids;       // [T][top_k]
    int32_t *dev_status;      // may be null
    int32_t *group;           // the published grouping (MODE 1), may be null
    uint16_t *h;              // MODE 1: [P][N / 2]
    float *z;                 // MODE 2: [P][N]
    int T, top_k, E, N, K, rows, slots, xpitch;
};

// MoE shared memory: staged x, the grouping, the rings and their barriers.
struct MSmem {
    uint32_t xs, grp, ring, bars, xbar, total;
    __host__ __device__ MSmem(int rows, int xpitch, int P, int slots)
    {
        xs = 0;
        grp = (uint32_t(rows) * uint32_t(xpitch) + 127) / 128 * 128;
        ring = (grp + uint32_t(moe_group_smem_ints(P)) * 4 + 127) / 128 * 128;
        bars = ring + uint32_t(kMoeWarps * slots) * kSegBytes;
        xbar = bars + uint32_t(kMoeWarps * slots) * 8;
        total = xbar + 8;
    }
};

// One segment into acc[0 .. MT/2) (MT = 8: one block of 8 pair columns, 16:
// two); x of the lane's column of block b at xr[b] + 64 g.
template <int MT>
__device__ __forceinline__ void segment_moe(uint32_t cb, uint32_t aoff, uint32_t srow, const uint32_t (&xr)[2],
                                            float (&acc)[8])
{
    const uint4 c0 = lds_v4(cb + aoff), c1 = lds_v4(cb + aoff + 16);
    const uint4 c8 = lds_v4(cb + aoff + 1152), c9 = lds_v4(cb + aoff + 1168);
    const uint4 s0 = lds_v4(cb + srow), s8 = lds_v4(cb + srow + 1152);
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        uint32_t pa[4], pb[4];
        unpack_word_f16x2(group_word(c0, c1, g), pa);
        unpack_word_f16x2(group_word(c8, c9, g), pb);
        const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
        const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
        const float sr = scale_of(s0, g), sr8 = scale_of(s8, g);
#pragma unroll
        for (int b = 0; b < MT / 8; ++b) {
            const uint4 xv = lds_v4(xr[b] + 64 * g);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(d, a0, xv.x, xv.y, d);
            mma16816(d, a1, xv.z, xv.w, d);
            acc[4 * b + 0] = fmaf(sr, d[0], acc[4 * b + 0]);
            acc[4 * b + 1] = fmaf(sr, d[1], acc[4 * b + 1]);
            acc[4 * b + 2] = fmaf(sr8, d[2], acc[4 * b + 2]);
            acc[4 * b + 3] = fmaf(sr8, d[3], acc[4 * b + 3]);
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(kMoeWarps * 32, 1) k_moe(MoeParams p)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128 - (smem_addr(smem_raw) & 127)) & 127);
    const uint32_t sbase = smem_addr(smem);
    const int P = p.T * p.top_k, slots = p.slots, K = p.K, N = p.N, S = K >> 8, tpe = N >> 4;
    const MSmem L(p.rows, p.xpitch, P, slots);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x, nthr = blockDim.x;

    griddep_wait();                                       // routing and x may come from the previous kernel
    const uint32_t xbar = sbase + L.xbar;
    if (lane == 0)
        for (int j = 0; j < slots; ++j) mbar_init(sbase + L.bars + 8 * (warp * slots + j), 1);
    if (tid == 0) {
        mbar_init(xbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_expect_tx(xbar, uint32_t(p.rows) * uint32_t(K * 2));   // every x row, one bulk copy each
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const MoeGroup g = moe_group(p.ids, P, p.E, reinterpret_cast<int *>(smem + L.grp), p.dev_status,
                                 MODE == 1 && blockIdx.x == 0, tid, nthr);   // ends with a barrier
    if (blockIdx.x == 0 && MODE == 1) {
        if (p.group) moe_group_publish(g, P, p.group, tid, nthr);
        // h rows of a pair with a bad expert id are zero
        const int half = N >> 1;
        for (int i = tid; i < P * half; i += nthr) {
            const int e = p.ids[i / half];
            if (e < 0 || e >= p.E) p.h[i] = 0;
        }
    }
    griddep_launch_dependents();
    const int n_units = g.J * tpe, stride = int(gridDim.x) * kMoeWarps;
    const uint32_t ring = sbase + L.ring + uint32_t(warp * slots) * kSegBytes;
    const uint32_t bars = sbase + L.bars + uint32_t(8 * warp * slots);
    const uint32_t aoff = segk::lane_code_offset(lane);
    const int r = lane >> 2, t = lane & 3;
    const uint32_t srow = uint32_t(r * 144 + 128);
    const bool leader = lane == 0;

    // issue cursor: unit iu (of this warp's), segment is
    int iu = int(blockIdx.x) * kMoeWarps + warp, is = 0, islot = 0;
    auto unit_seg = [&](int u) -> const uint8_t * {       // first segment of unit u in the bank
        const int j = u / tpe, tl = u - j * tpe;
        return p.seg + size_t(g.uexp[g.jt[j] >> 8] * tpe + tl) * size_t(S) * kSegBytes;
    };
    const uint8_t *iptr = iu < n_units ? unit_seg(iu) : nullptr;
    auto issue = [&]() -> bool {
        if (iu >= n_units) return false;
        if (leader) {
            const uint32_t bar = bars + 8 * islot;
            mbar_arrive_expect_tx(bar, uint32_t(kSegBytes));
            bulk_load(ring + uint32_t(islot) * kSegBytes, iptr + size_t(is) * kSegBytes, uint32_t(kSegBytes), bar);
        }
        if (++is == S) {
            is = 0;
            iu += stride;
            if (iu < n_units) iptr = unit_seg(iu);
        }
        islot = islot + 1 == slots ? 0 : islot + 1;
        return true;
    };
    int in_flight = 0;
    while (in_flight < slots && issue()) ++in_flight;
    // x rows into shared memory (rows padded to xpitch bytes), behind the weights' first copies
    for (int m = tid; m < p.rows; m += nthr)
        bulk_load(sbase + L.xs + uint32_t(m) * uint32_t(p.xpitch), p.x + size_t(m) * K, uint32_t(K * 2), xbar);
    bool ok = __all_sync(0xffffffffu, mbar_wait(xbar, 0));

    // consume cursor: unit cu, segment cs
    int cu = int(blockIdx.x) * kMoeWarps + warp, cs = 0, cslot = 0, ucols = 0, ubase = 0, tl = 0;
    uint32_t cphase = 0;
    uint32_t xr[2] = {0, 0};
    float acc[8];
    while (ok && in_flight > 0) {
        if (cs == 0) {
            // a unit starts: its pairs and the x rows its columns read
            const int j = cu / tpe;
            tl = cu - j * tpe;
            const int ue = g.jt[j] >> 8, blk = g.jt[j] & 255;
            ubase = g.ustart[ue] + 16 * blk;
            ucols = min(16, g.ustart[ue + 1] - ubase);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int m = min(8 * b + r, ucols - 1);   // columns past the block's pairs repeat its last pair
                const int q = g.order[ubase + m];
                const int row = MODE == 1 ? q / p.top_k : q;
                xr[b] = sbase + L.xs + uint32_t(row * p.xpitch + 16 * t);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(bars + 8 * cslot, cphase))) {
            ok = false;
            break;
        }
        const uint32_t cb = ring + uint32_t(cslot) * kSegBytes;
        const uint32_t xs_seg[2] = {xr[0] + uint32_t(cs * 512), xr[1] + uint32_t(cs * 512)};
        if (ucols > 8)
            segment_moe<16>(cb, aoff, srow, xs_seg, acc);
        else
            segment_moe<8>(cb, aoff, srow, xs_seg, acc);
        __syncwarp();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (!issue()) --in_flight;
        if (++cslot == slots) {
            cslot = 0;
            cphase ^= 1u;
        }
        if (++cs == S) {
            // the unit's outputs: rows 16 tl + r + 8 h of the block's pairs
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int qq = 0; qq < 2; ++qq) {
                        const int m = 8 * b + 2 * t + qq, row = 16 * tl + r + 8 * hh;
                        const float v = acc[4 * b + 2 * hh + qq];
                        if (MODE == 1) {
                            const float u = __shfl_down_sync(0xffffffffu, v, 4);
                            if (m < ucols && (r & 1) == 0)
                                p.h[size_t(g.order[ubase + m]) * (N >> 1) + (row >> 1)] =
                                    float_to_f16_bits(silu_f32(v) * u);
                        } else if (m < ucols) {
                            p.z[size_t(g.order[ubase + m]) * N + row] = v;
                        }
                    }
            cs = 0;
            cu += stride;
        }
    }
    if (!ok && leader) {
        atomicOr(&g_step_error, ZQ4_DEVERR_WAIT_TIMEOUT);
        for (int c = 0; c < in_flight; ++c) {
            const int sl = (cslot + c) % slots;
            if (!mbar_wait(bars + 8 * sl, cphase ^ (cslot + c >= slots ? 1u : 0u))) break;
        }
    }
}

// The weighted combine of the MoE block: y[t, n] = f16(sum_j w[t, j] z[t top_k + j, n])
// over the slots with a valid expert id, in slot order; one thread per 4 outputs.
__global__ void __launch_bounds__(256) k_moe_combine(const float *z, const int32_t *ids, const float *w,
                                                     uint16_t *y, int T, int D, int top_k, int num_experts)
{
    griddep_wait();
    const int per = D >> 2;
    const int q = int(blockIdx.x) * 256 + int(threadIdx.x);
    if (q >= T * per) return;
    const int t = q / per, n = (q - t * per) * 4;
    float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
    for (int j0 = 0; j0 < top_k; j0 += 8) {            // eight slots' loads in flight, then their sums in order
        float wj[8];
        float4 v[8];
        bool use[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int j = j0 + b;
            int e = -1;
            if (j < top_k) e = ids[t * top_k + j];
            use[b] = e >= 0 && e < num_experts;      // a bad id contributes nothing
            wj[b] = use[b] ? w[t * top_k + j] : 0.f;
            v[b] = use[b] ? *reinterpret_cast<const float4 *>(z + (size_t(t) * top_k + j) * D + n)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            if (!use[b]) continue;
            r0 = fmaf(wj[b], v[b].x, r0);
            r1 = fmaf(wj[b], v[b].y, r1);
            r2 = fmaf(wj[b], v[b].z, r2);
            r3 = fmaf(wj[b], v[b].w, r3);
        }
    }
    uint16_t *yo = y + size_t(t) * D + n;
    yo[0] = float_to_f16_bits(r0);
    yo[1] = float_to_f16_bits(r1);
    yo[2] = float_to_f16_bits(r2);
    yo[3] = float_to_f16_bits(r3);
}

}  // namespace sp

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

int step_smem_set[kMaxDevices] = {};
int step_smem_set2[kMaxDevices] = {};

const void *step_kernel(int M)
{
    return M == 1 ? reinterpret_cast<const void *>(sp::k_step<1>) : reinterpret_cast<const void *>(sp::k_step<2>);
}

}  // namespace

// Ring slots, x window and cached jobs of a launch: two slots per compute
// warp (measured: a larger x window pays more than deeper rings), the job
// table cached while it leaves the window room for eight of the largest jobs'
// x, and the window every byte that is left (at most 256 KiB: the tag word
// holds the offset in 128-byte units).
bool step_launch_shape(int M, int max_k, int n_jobs, int n_pub, StepShape *sh)
{
    const size_t cap = size_t(227) * 1024 - 128;
    const size_t big = (size_t(M) * size_t(max_k) * 2 + 127) / 128 * 128;
    const int slots = 2;
    int cached = std::min(n_jobs, 256);
    for (;;) {
        const size_t fixed = sp::Smem(slots, 0, n_pub, cached).total;
        size_t w = fixed < cap ? (cap - fixed) / 128 * 128 : 0;
        w = std::min<size_t>(w, size_t(256) * 1024 - 128);
        if (w >= 8 * big || cached == 0) {
            if (w < big) return false;                  // one job's x would not fit
            sh->slots = slots;
            sh->wbytes = int(w);
            sh->cached = cached;
            sh->smem = sp::Smem(slots, int(w), n_pub, cached).total + 128;
            return true;
        }
        cached = cached > 32 ? cached / 2 : 0;
    }
}

zq4_status step_run(const zq4_stack_plan *plan, cudaStream_t s)
{
    const StepLayout l(plan->entries, plan->split_tiles, plan->part_records);
    uint8_t *base = static_cast<uint8_t *>(plan->dev);
    sp::Params p;
    p.hdr = reinterpret_cast<StepHeader *>(base + l.hdr);
    p.jobs = reinterpret_cast<const StepJob *>(base + l.jobs);
    p.job_done = reinterpret_cast<unsigned *>(base + l.job_done);
    p.arrive = reinterpret_cast<unsigned *>(base + l.arrive);
    p.work = reinterpret_cast<float *>(base + l.work);
    p.n_jobs = plan->entries;
    p.total_tiles = plan->tiles;
    p.M = plan->M;
    p.n_pub = plan->n_pub;
    StepShape sh;
    if (!step_launch_shape(p.M, plan->max_k, p.n_jobs, p.n_pub, &sh)) return ZQ4_ERR_UNSUPPORTED;
    p.slots = sh.slots;
    p.wbytes = sh.wbytes;
    p.cached = sh.cached;
    p.fine = plan->min_unit >= sh.slots ? 1 : 0;
    p.split = plan->split_tiles > 0 ? 1 : 0;
    p.wait_ns = plan->wait_ns ? plan->wait_ns : kWaitLimitNs;
    const void *kern = step_kernel(p.M);
    cudaError_t e = ensure_smem(kern, sh.smem, p.M == 1 ? step_smem_set : step_smem_set2);
    if (e != cudaSuccess) return cuda_status(e);
    void *args[] = {&p};
    return cuda_status(cudaLaunchCooperativeKernel(kern, dim3(plan->grid), dim3(sp::kThreads), args, sh.smem, s));
}

zq4_status step_check_resident(int M, int max_k, int n_jobs, int n_pub)
{
    StepShape sh;
    if (!step_launch_shape(M, max_k, n_jobs, n_pub, &sh)) return ZQ4_ERR_UNSUPPORTED;
    const void *kern = step_kernel(M);
    cudaError_t e = ensure_smem(kern, sh.smem, M == 1 ? step_smem_set : step_smem_set2);
    if (e != cudaSuccess) return cuda_status(e);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, sp::kThreads, sh.smem);
    if (e != cudaSuccess) return cuda_status(e);
    return per_sm < 1 ? ZQ4_ERR_UNSUPPORTED : ZQ4_OK;
}

// ---------------------------------------------------------------------------
// k_wide host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

namespace {

int wide_smem_set8[kMaxDevices] = {};
int wide_smem_set16[kMaxDevices] = {};

struct WideShape {
    int slots, slot_bytes, cached;
    size_t smem;
};

// Ring slots (as many as fit, 2 to 4), slot size (one segment and x[M][256])
// and cached jobs (up to 256, while they leave the slots room).
bool wide_launch_shape(int M, int n_jobs, int n_pub, WideShape *sh)
{
    const size_t cap = size_t(227) * 1024 - 128;
    const int nw = M <= 8 ? sp::Wide<8>::kWarps : sp::Wide<16>::kWarps;
    const int slot_bytes = wide_group(M) * sp::kSegBytes + M * 512;
    for (int slots = 4; slots >= 2; --slots) {
        for (int cached = std::min(n_jobs, 256);; cached = cached > 16 ? cached / 2 : 0) {
            const size_t need = sp::WSmem(nw, slots, slot_bytes, n_pub, cached).total;
            if (need <= cap && (cached == std::min(n_jobs, 256) || slots == 2)) {
                sh->slots = slots;
                sh->slot_bytes = slot_bytes;
                sh->cached = cached;
                sh->smem = need + 128;
                return true;
            }
            if (cached == 0 || slots > 2) break;
        }
    }
    return false;
}

const void *wide_kernel(int M)
{
    return M <= 8 ? reinterpret_cast<const void *>(sp::k_wide<8>) : reinterpret_cast<const void *>(sp::k_wide<16>);
}
int wide_threads(int M) { return M <= 8 ? sp::Wide<8>::kThreads : sp::Wide<16>::kThreads; }

}  // namespace

bool wide_x_map(void *map128, const uint16_t *x, int M, int K, long long ld)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dim[2] = {cuuint64_t(K), cuuint64_t(M)};
    const cuuint64_t stride[1] = {cuuint64_t(ld) * 2};
    const cuuint32_t box[2] = {256, cuuint32_t(M)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(static_cast<CUtensorMap *>(map128), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(x), dim,
               stride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

zq4_status wide_run(const zq4_stack_plan *plan, cudaStream_t s)
{
    const StepLayout l(plan->entries, plan->split_tiles, plan->part_records, true);
    uint8_t *base = static_cast<uint8_t *>(plan->dev);
    sp::Params p;
    memset(&p, 0, sizeof(p));
    p.hdr = reinterpret_cast<StepHeader *>(base + l.hdr);
    p.jobs = reinterpret_cast<const StepJob *>(base + l.jobs);
    p.job_done = reinterpret_cast<unsigned *>(base + l.job_done);
    p.arrive = reinterpret_cast<unsigned *>(base + l.arrive);
    p.work = reinterpret_cast<float *>(base + l.work);
    p.tmaps = reinterpret_cast<const CUtensorMap *>(base + l.tmaps);
    p.n_jobs = plan->entries;
    p.total_tiles = plan->tiles;
    p.M = plan->M;
    p.n_pub = plan->n_pub;
    WideShape sh;
    if (!wide_launch_shape(p.M, p.n_jobs, p.n_pub, &sh)) return ZQ4_ERR_UNSUPPORTED;
    p.slots = sh.slots;
    p.slot_bytes = sh.slot_bytes;
    p.cached = sh.cached;
    p.split = plan->split_tiles > 0 ? 1 : 0;
    p.wait_ns = plan->wait_ns ? plan->wait_ns : kWaitLimitNs;
    const void *kern = wide_kernel(p.M);
    cudaError_t e = ensure_smem(kern, sh.smem, p.M <= 8 ? wide_smem_set8 : wide_smem_set16);
    if (e != cudaSuccess) return cuda_status(e);
    void *args[] = {&p};
    return cuda_status(
        cudaLaunchCooperativeKernel(kern, dim3(plan->grid), dim3(wide_threads(p.M)), args, sh.smem, s));
}

zq4_status wide_check_resident(int M, int n_jobs, int n_pub)
{
    WideShape sh;
    if (!wide_launch_shape(M, n_jobs, n_pub, &sh)) return ZQ4_ERR_UNSUPPORTED;
    if (!tensor_map_encoder()) return ZQ4_ERR_UNSUPPORTED;
    const void *kern = wide_kernel(M);
    cudaError_t e = ensure_smem(kern, sh.smem, M <= 8 ? wide_smem_set8 : wide_smem_set16);
    if (e != cudaSuccess) return cuda_status(e);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, wide_threads(M), sh.smem);
    if (e != cudaSuccess) return cuda_status(e);
    return per_sm < 1 ? ZQ4_ERR_UNSUPPORTED : ZQ4_OK;
}

// ---------------------------------------------------------------------------
// zq4_moe_block host side
// ---------------------------------------------------------------------------
namespace {

int moe_smem_set1[kMaxDevices] = {};
int moe_smem_set2[kMaxDevices] = {};

// Ring slots (4 down to 2) next to x [rows][K] (rows padded by 16 bytes) and the grouping.
bool moe_shape(int rows, int K, int P, int *slots, int *xpitch, size_t *smem)
{
    const size_t cap = size_t(227) * 1024 - 128;
    *xpitch = K * 2 + 16;
    for (int sl = 4; sl >= 2; --sl) {
        const size_t need = sp::MSmem(rows, *xpitch, P, sl).total;
        if (need <= cap) {
            *slots = sl;
            *smem = need + 128;
            return true;
        }
    }
    return false;
}

template <int MODE>
cudaError_t launch_moe_stage(const sp::MoeParams &p, size_t smem, cudaStream_t s)
{
    auto kern = sp::k_moe<MODE>;
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(kern), smem, MODE == 1 ? moe_smem_set1 : moe_smem_set2);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(sm_count()), dim3(sp::kMoeWarps * 32), smem, s, p);
}

}  // namespace

size_t moe_block_work_layout(int T, int top_k, int D, int I, size_t *h_off, size_t *z_off)
{
    const size_t P = size_t(T) * top_k;
    const size_t g = (size_t(moe_group_pub_ints(int(P))) * 4 + 255) / 256 * 256;
    const size_t h = (P * I * 2 + 255) / 256 * 256;
    if (h_off) *h_off = g;
    if (z_off) *z_off = g + h;
    return g + h + P * D * 4;
}

bool moe_block_supported(int T, int top_k, int D, int I)
{
    const int P = T * top_k;
    int sl, xp;
    size_t sm;
    return P <= 256 && D % 256 == 0 && I % 256 == 0 && moe_shape(T, D, P, &sl, &xp, &sm) &&
           moe_shape(P, I, P, &sl, &xp, &sm);
}

cudaError_t launch_moe_block(const uint8_t *gu_seg, const uint8_t *dn_seg, int num_experts, const uint16_t *x,
                             uint16_t *y, int T, int D, int I, const int32_t *ids, const float *route_w, int top_k,
                             void *work, int32_t *dev_status, cudaStream_t s)
{
    size_t h_off, z_off;
    moe_block_work_layout(T, top_k, D, I, &h_off, &z_off);
    uint8_t *wb = static_cast<uint8_t *>(work);
    const int P = T * top_k;
    sp::MoeParams p;
    memset(&p, 0, sizeof(p));
    p.ids = ids;
    p.T = T;
    p.top_k = top_k;
    p.E = num_experts;
    p.h = reinterpret_cast<uint16_t *>(wb + h_off);
    p.z = reinterpret_cast<float *>(wb + z_off);
    size_t smem;
    // gate_up + SiLU*mul: x [T, D] -> h [P, I]; this stage publishes the grouping and reports bad ids
    p.seg = gu_seg;
    p.x = x;
    p.group = reinterpret_cast<int32_t *>(wb);
    p.dev_status = dev_status;
    p.N = 2 * I;
    p.K = D;
    p.rows = T;
    if (!moe_shape(T, D, P, &p.slots, &p.xpitch, &smem)) return cudaErrorInvalidValue;
    cudaError_t e = launch_moe_stage<1>(p, smem, s);
    if (e != cudaSuccess) return e;
    // down: h [P, I] -> z [P, D] fp32
    p.seg = dn_seg;
    p.x = p.h;
    p.group = nullptr;
    p.dev_status = nullptr;
    p.N = D;
    p.K = I;
    p.rows = P;
    if (!moe_shape(P, I, P, &p.slots, &p.xpitch, &smem)) return cudaErrorInvalidValue;
    e = launch_moe_stage<2>(p, smem, s);
    if (e != cudaSuccess) return e;
    const int n4 = T * (D / 4);
    return launch_pdl(sp::k_moe_combine, dim3((n4 + 255) / 256), dim3(256), 0, s, static_cast<const float *>(p.z),
                      ids, route_w, y, T, D, top_k, num_experts);
}

cudaError_t read_step_error(unsigned *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_step_error, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_step_error, &zero, sizeof(unsigned));
}

}  // namespace zq4
