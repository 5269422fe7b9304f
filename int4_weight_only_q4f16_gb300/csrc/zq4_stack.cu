// zq4_stack.cu -- a whole decode step (an ordered list of q4f16_1
// projections, each reading an activation the previous ones may have
// written) as one persistent cooperative kernel.
//
// What it computes: for every job j in order, y_j = x_j * W_j^T, or the fused
// gate_up + SiLU*mul output for interleaved gate/up rows ("Zero TVM
// Documentation", section "Q4F16 quantization format", cards 5 "int4 Matmul"
// and 6 "Fused FFN"; the per-token dispatch sequence of its "Decode loop"
// section). Every job starts only after the previous job's outputs are all
// written, as in a decode step where each projection consumes the one
// before it.
//
// Why one kernel: with one launch per projection, every projection pays the
// kernel boundary (drain, launch, first-copy latency) and the small ones
// (few 16-row tiles) leave most SMs idle. Here each SM keeps streaming
// weights across job boundaries: its warps request the next jobs' segments
// into their shared-memory rings and L2 while the grid waits for the
// current job's last outputs; only the activation dependency synchronizes.
//
// How:
//  * Grid = one CTA per SM (cooperative launch, so all CTAs are resident
//    and may wait on one another): 12 compute warps and one copy warp. Work
//    unit = a segment, 16 weight rows x 256 columns.
//  * The weights are in the segmented layout (zq4_prepare_weight,
//    ZQ4_PREP_SEGMENTED): each segment is 2304 contiguous bytes (swizzled
//    codes, then scales), so one bulk copy fills a shared-memory slot and no
//    tensor map is involved. Each compute warp has its own ring of segment
//    slots; lane w of the copy warp refills ring w as soon as compute warp w
//    releases a slot (an mbarrier per slot each way), across job
//    boundaries, so the compute warps never spend issue slots on copies.
//    Per 32-column group, lane (r, t) (r = lane/4, t = lane%4) takes word t
//    of rows r and r+8 (ldmatrix.x4 fetches two groups, conflict-free on the
//    swizzle),
//    unpacks exact f16 (q - 7) pairs as the A fragments of two chained
//    m16n8k16 MMAs against the matching pair-permuted x chunk, and adds the
//    fp32 result times the fp32 group scale to its accumulator.
//  * CTA c takes the whole 16-row tiles [c*T/G, (c+1)*T/G) of every job and
//    splits their segments evenly over its warps. A tile that lies in one
//    warp's range is written by that warp; a warp holding part of a tile
//    parks the part in shared memory, and at the end of the job all threads
//    of the CTA sum the parked parts of every split tile in warp order
//    (bit-reproducible) and write them. Tiles never span CTAs, so no partial
//    sum goes through global memory.
//  * Job boundary: CTA barrier, split tiles summed, one release-add per CTA
//    on the job's counter, acquire-poll until every CTA has arrived, CTA
//    barrier. x of the next job is staged into shared memory with L2 reads
//    (it may have been written by other SMs during this kernel): after the
//    poll, or, when no earlier job of the plan writes any byte of it (decided
//    when the plan is made), already before the split-tile sums, so that its
//    latency hides behind them and the poll.
//  * The job table (as much of it as fits next to the rings) is copied to
//    shared memory once per launch; each warp's copy iterator and tile
//    position advance incrementally (no division per segment).
//  * Counters grow monotonically: a launch waits for (launch index + 1) x
//    grid arrivals, the launch index being read from the plan at start and
//    advanced by the last CTA to finish.
//  * Every wait is bounded. A timeout sets ZQ4_DEVERR_WAIT_TIMEOUT and the
//    plan's abort flag, which every waiter checks, so the whole grid leaves
//    promptly; the plan must then be initialised again.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <vector>

#include "zq4_async.cuh"
#include "zq4_common.cuh"
#include "zq4_internal.h"
#include "zq4_segment.cuh"

namespace zq4 {

__device__ unsigned g_stack_error = 0;

namespace st {

constexpr int kWarps = 12;                  // compute warps, one ring each
constexpr int kCompute = kWarps * 32;
constexpr int kThreads = kCompute + 32;      // + the copy warp
constexpr int kSlots = 5;
constexpr int kEarly = 2;   // x chunks (16 B) per thread read before the job barrier
using namespace segk;       // segment layout, inner loop, split-tile sums

struct Header {
    unsigned epoch;     // launches completed
    unsigned done;      // CTA arrivals at launch end (monotone)
    unsigned abort;     // set by any wait that gave up
    unsigned pad[29];
};

constexpr int kJobGateUp = 1;   // rows are interleaved gate/up pairs: silu(g) * u output
constexpr int kJobXEarly = 2;   // x is not written by an earlier job: it may be read at any time

struct alignas(16) Job {
    const uint8_t *seg; // the matrix in the segmented layout
    const uint16_t *x;  // [M][K]
    uint16_t *y;        // [M][y_stride]
    int N, K, T, S;
    int flags, y_stride;
};

struct Params {
    Header *hdr;
    const Job *jobs;
    unsigned *job_cnt;   // [n_jobs]
    int n_jobs, M, max_k;
    int cached;          // jobs [0, cached) are copied to shared memory at start
};

constexpr size_t kRingOff = 0;
constexpr size_t kBarOff = kRingOff + size_t(kWarps) * kSlots * kSegBytes;
constexpr size_t kMiscOff = kBarOff + 2 * size_t(kWarps) * kSlots * 8;   // full, then empty barriers
// Warp partials: slot [kWarps*2], each [kTokCols][kParkRow] floats (token
// major, rows padded to 17 so that the 16 rows of one token, read by 16
// lanes, fall in distinct banks).
constexpr int kParkRow = 17;
constexpr int kParkSlot = kTokCols * kParkRow;
constexpr size_t kParkOff = kMiscOff + 128;
constexpr size_t kTabOff = kParkOff + (size_t(kWarps) * 2 * kParkSlot * 4 + 15) / 16 * 16;   // warp range tables, two jobs
constexpr int kTabInts = 2 * (kWarps + 1) + 2;                       // one job: range starts, first tiles, CTA tiles
constexpr size_t kXsOff = kTabOff + (2 * kTabInts * 4 + 15) / 16 * 16;
__host__ __device__ inline size_t xs_bytes(int M, int max_k) { return (size_t(M) * xs_row_bytes(max_k) + 15) / 16 * 16; }
__host__ __device__ inline size_t smem_bytes(int M, int max_k) { return 1024 + kXsOff + xs_bytes(M, max_k); }
// jobs that fit in shared memory next to everything else (the rest are read from the plan)
inline int cached_jobs(int n, int M, int max_k)
{
    const size_t left = size_t(227) * 1024 - smem_bytes(M, max_k);
    return int(std::min<size_t>(size_t(n), left / sizeof(Job)));
}

// Has the phase of this parity completed? (never waits)
__device__ __forceinline__ bool mbar_test(uint32_t addr, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    return done != 0;
}

// barrier among the compute warps only (the copy warp runs on its own)
__device__ __forceinline__ void compute_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p)
{
    unsigned r;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(r) : "l"(p) : "memory");
    return r;
}

// After a barrier of the compute warps: the tiles [tb, tb + nt) of a job
// that were split between warps get the parked parts of their warps summed
// in warp order (bit-reproducible) and written. One output per thread and
// pass; `shift` = log2 of the outputs per tile rounded up to a power of
// two, so no division. `wtab` = the warp range starts (kWarps + 1 entries)
// then each warp's first tile.
__device__ __forceinline__ void sum_split_tiles(int tb, int nt, int S, int gate_up, int M, int N, int y_stride,
                                                uint16_t *y, const float *wpark, const int *wtab)
{
    const int per_tok = gate_up ? 8 : 16, tok_shift = gate_up ? 3 : 4;
    const int outs = per_tok * M;
    int shift = 3;
    while ((1 << shift) < outs) ++shift;
    int wb[kWarps + 1], wf[kWarps];
#pragma unroll
    for (int w = 0; w <= kWarps; ++w) wb[w] = wtab[w];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) wf[w] = wtab[kWarps + 1 + w];
    for (int it = threadIdx.x; it < (nt << shift); it += kCompute) {
        const int o = it & ((1 << shift) - 1);
        if (o >= outs) continue;
        const int tt = tb + (it >> shift), lo = tt * S, hi = lo + S;
        const int m = o >> tok_shift, i = o & (per_tok - 1), ra = gate_up ? 2 * i : i;
        // every warp's parked value is read (all loads in flight at once);
        // those of warps not holding part of tile tt are added as +0, which
        // leaves the warp-order sum bit-identical
        float p0[kWarps], p1[kWarps];
        bool in[kWarps];
        int parts = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            in[w] = wb[w] < wb[w + 1] && wb[w] < hi && wb[w + 1] > lo;
            parts += in[w];
            const float *qk = wpark + (w * 2 + (tt == wf[w] ? 0 : 1)) * kParkSlot + m * kParkRow + ra;
            p0[w] = qk[0];
            p1[w] = gate_up ? qk[1] : 0.f;
        }
        if (parts < 2) continue;                 // one warp held the whole tile and wrote it
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            v0 += in[w] ? p0[w] : 0.f;
            v1 += in[w] ? p1[w] : 0.f;
        }
        const int row0 = tt * 16;
        if (!gate_up) {
            if (row0 + i < N) y[size_t(m) * y_stride + row0 + i] = float_to_f16_bits(v0);
        } else if (row0 + 2 * i + 1 < N) {
            y[size_t(m) * y_stride + (row0 >> 1) + i] = float_to_f16_bits(silu_f32(v0) * v1);
        }
    }
}

// x chunk i of M*K/8 (16 bytes of token i / (K/8)) into its staged place,
// pair-permuted as the unpack produces: (x0,x4),(x1,x5),(x2,x6),(x3,x7)
__device__ __forceinline__ void put_x(uint8_t *xs, uint32_t xrow, int words, int i, uint4 v)
{
    const int m = i / words, cw = i - m * words;
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);
    o.y = __byte_perm(v.x, v.z, 0x7632);
    o.z = __byte_perm(v.y, v.w, 0x5410);
    o.w = __byte_perm(v.y, v.w, 0x7632);
    *reinterpret_cast<uint4 *>(xs + size_t(m) * xrow + size_t(cw) * 16) = o;
}

__global__ void __launch_bounds__(kThreads, 1) k_stack(Params p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_addr(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, t = lane & 3;
    const int G = gridDim.x, cta = blockIdx.x;
    const uint32_t full0 = sbase + uint32_t(kBarOff), empty0 = full0 + uint32_t(kWarps * kSlots * 8);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + kMiscOff);
    float *wpark = reinterpret_cast<float *>(smem + kParkOff);
    int *wtab = reinterpret_cast<int *>(smem + kTabOff);
    uint8_t *xs = smem + kXsOff;
    Job *sjobs = reinterpret_cast<Job *>(smem + kXsOff + xs_bytes(p.M, p.max_k));
    const uint32_t xrow = uint32_t(xs_row_bytes(p.max_k));
    const int n = p.n_jobs, M = p.M;
    const unsigned launch = *reinterpret_cast<volatile unsigned *>(&p.hdr->epoch);
    const unsigned target = (launch + 1u) * unsigned(G);

    if (threadIdx.x == 0) *s_abort = 0;
    if (warp < kWarps && lane == 0) {
        for (int j = 0; j < kSlots; ++j) {
            mbar_init(full0 + 8 * (warp * kSlots + j), 1);    // the copy's bytes
            mbar_init(empty0 + 8 * (warp * kSlots + j), 1);   // the consuming warp is done
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    {
        // the job table (or its first p.cached entries) into shared memory
        const uint4 *src = reinterpret_cast<const uint4 *>(p.jobs);
        uint4 *dst = reinterpret_cast<uint4 *>(sjobs);
        const int words = p.cached * int(sizeof(Job) / 16);
        for (int i = threadIdx.x; i < words; i += kThreads) dst[i] = src[i];
    }
    __syncthreads();
    auto job = [&](int j) -> const Job & { return j < p.cached ? sjobs[j] : p.jobs[j]; };

    // compute warp w's segment range of a job: CTA part of the job, then
    // warp part (CTA ranges are whole tiles, so a tile never spans two CTAs)
    auto warp_range = [&](int T, int S, int w, int &ub, int &ue) {
        int tb, te;
        split(0, T, cta, G, tb, te);
        split(tb * S, te * S, w, kWarps, ub, ue);
    };

    if (warp == kWarps) {
        // ---------------- the copy warp ----------------
        // Lane w keeps ring w full: it walks compute warp w's (job, segment)
        // sequence (segment u of a job, tile major, is at byte u * kSegBytes
        // of its matrix) and refills a slot as soon as that warp has released
        // it, across job boundaries: the weights never depend on earlier jobs.
        const int w = lane;
        const uint32_t ring = sbase + uint32_t(kRingOff) + uint32_t(w * kSlots * kSegBytes);
        int it_j = n, it_u = 0, it_e = 0, issued = 0;
        const uint8_t *it_seg = nullptr;
        auto seek = [&](int j) {
            for (; j < n; ++j) {
                const Job &jb = job(j);
                int ub, ue;
                warp_range(jb.T, jb.S, w, ub, ue);
                if (ub < ue) {
                    it_j = j;
                    it_u = ub;
                    it_e = ue;
                    it_seg = jb.seg;
                    return;
                }
            }
            it_j = n;
        };
        if (w < kWarps) seek(0);
        unsigned long long t0 = globaltimer();
        bool timed_out = false;
        for (;;) {
            const bool more = w < kWarps && it_j < n && !*s_abort;
            bool did = false;
            if (more) {
                const int slot = issued % kSlots, f = issued / kSlots;
                const uint32_t full = full0 + 8 * (w * kSlots + slot);
                if (f == 0 || mbar_test(empty0 + 8 * (w * kSlots + slot), (f - 1) & 1)) {
                    mbar_arrive_expect_tx(full, kSegBytes);
                    bulk_load(ring + slot * kSegBytes, it_seg + size_t(it_u) * kSegBytes, kSegBytes, full);
                    ++issued;
                    did = true;
                    if (++it_u >= it_e) seek(it_j + 1);
                }
            }
            if (!__any_sync(0xffffffffu, more)) break;
            if (__any_sync(0xffffffffu, did)) {
                t0 = globaltimer();
            } else {
                // no slot free: the compute warps are busy or between jobs
                if (globaltimer() - t0 > kWaitLimitNs) {
                    timed_out = true;
                    break;
                }
                __nanosleep(100);
            }
        }
        if (timed_out && lane == 0) {
            atomicOr(&g_stack_error, ZQ4_DEVERR_WAIT_TIMEOUT);
            atomicOr(&p.hdr->abort, 1u);
            *s_abort = 1;
        }
        // every copy this lane issued has landed before the CTA may exit (the
        // last fill of each slot; earlier fills were consumed before a refill)
        if (w < kWarps)
            for (int c = max(0, issued - kSlots); c < issued; ++c)
                if (!mbar_wait(full0 + 8 * (w * kSlots + c % kSlots), (c / kSlots) & 1)) break;
    } else {
        // ---------------- compute warps ----------------
        const uint32_t ring0 = sbase + uint32_t(kRingOff) + uint32_t(warp * kSlots * kSegBytes);
        const uint32_t bfull = full0 + uint32_t(8 * warp * kSlots), bempty = empty0 + uint32_t(8 * warp * kSlots);
        uint32_t ldm_off[4];
        ldm_offsets(lane, ldm_off);
        const uint8_t *xr = xs + size_t(min(r, M - 1)) * xrow + 16 * t;

        // stage x of a job synchronously (compute threads; caller barriers)
        auto stage_now = [&](const Job &jb, int from) {
            const int words = jb.K >> 3, total = M * words;
            for (int i0 = from + int(threadIdx.x); i0 < total; i0 += 2 * kCompute) {
                uint4 v0, v1;
                const int i1 = i0 + kCompute;
                v0 = __ldcg(reinterpret_cast<const uint4 *>(jb.x) + i0);
                if (i1 < total) v1 = __ldcg(reinterpret_cast<const uint4 *>(jb.x) + i1);
                put_x(xs, xrow, words, i0, v0);
                if (i1 < total) put_x(xs, xrow, words, i1, v1);
            }
        };
        // the warp range table of job j (one of two buffers, so that the table
        // of the next job can be made while the sums of the last one read theirs):
        // lanes 0..kWarps of warp `tw`
        auto set_wtab = [&](const Job &jb, int j, int tw) {
            const int q = int(threadIdx.x) - 32 * tw;
            if (q >= 0 && q <= kWarps) {
                int tb0, te0;
                split(0, jb.T, cta, G, tb0, te0);
                const int b = part_begin(tb0 * jb.S, te0 * jb.S, q, kWarps);
                int *tab = wtab + (j & 1) * kTabInts;
                tab[q] = b;
                tab[kWarps + 1 + q] = b / jb.S;
                if (q == 0) {
                    tab[2 * (kWarps + 1)] = tb0;      // this CTA's tiles of the job
                    tab[2 * (kWarps + 1) + 1] = te0;
                }
            }
        };

        bool ok = true;
        int slot = 0;             // ring position of the next segment and the parity of its fill
        uint32_t phase = 0;
        for (int j = 0; j < n; ++j) {
            const Job &jb = job(j);
            if (j == 0) {
                set_wtab(jb, 0, 0);
                stage_now(jb, 0);
                compute_sync();
            } else {
                // every compute warp of this CTA is done with job j-1 (x
                // buffer free, partial tiles parked)
                compute_sync();
                const bool early = (jb.flags & kJobXEarly) != 0 && !*s_abort;
                const int words = jb.K >> 3, total = M * words;
                uint4 xv[kEarly];
                const Job &pj = job(j - 1);
                if (!*s_abort) {
                    const int *ptab = wtab + ((j - 1) & 1) * kTabInts;
                    const int ptb = ptab[2 * (kWarps + 1)], pte = ptab[2 * (kWarps + 1) + 1];
                    sum_split_tiles(ptb, pte - ptb, pj.S, pj.flags & kJobGateUp, M, pj.N, pj.y_stride, pj.y, wpark,
                                    ptab);
                }
                compute_sync();      // finalize writes before the release below
                set_wtab(jb, j, 1);  // warp 1, while thread 0 waits at the grid barrier
                if (threadIdx.x == 0 && !*s_abort) {
                    // release: this CTA's outputs of job j-1 become visible with the increment
                    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&p.job_cnt[j - 1]) : "memory");
                }
                if (early) {
                    // read now (thread 0 after its release, which would otherwise wait
                    // for these loads), stored after the grid barrier: the latency hides
                    // behind it
#pragma unroll
                    for (int e = 0; e < kEarly; ++e) {
                        const int i = int(threadIdx.x) + e * kCompute;
                        if (i < total) xv[e] = __ldcg(reinterpret_cast<const uint4 *>(jb.x) + i);
                    }
                }
                if (threadIdx.x == 0 && !*s_abort) {
                    const unsigned long long t0 = globaltimer();
                    for (;;) {
                        if (ld_acquire(&p.job_cnt[j - 1]) >= target) break;
                        if (*reinterpret_cast<volatile unsigned *>(&p.hdr->abort) ||
                            globaltimer() - t0 > kWaitLimitNs) {
                            atomicOr(&p.hdr->abort, 1u);
                            *s_abort = 1;
                            break;
                        }
                    }
                }
                if (early) {
                    // the loads were issued before the poll: stored only now
#pragma unroll
                    for (int e = 0; e < kEarly; ++e) {
                        const int i = int(threadIdx.x) + e * kCompute;
                        if (i < total) put_x(xs, xrow, words, i, xv[e]);
                    }
                    if (total > kEarly * kCompute) stage_now(jb, kEarly * kCompute);
                }
                compute_sync();
                if (*s_abort) {
                    ok = false;
                    break;
                }
                if (!early) {
                    stage_now(jb, 0);
                    compute_sync();
                }
            }

            const int S = jb.S, gate_up = jb.flags & kJobGateUp;
            const int *tab = wtab + (j & 1) * kTabInts;
            const int ub = tab[warp], ue = tab[warp + 1], first_tile = tab[kWarps + 1 + warp];
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            int cur_tile = -1;
            auto flush = [&](int tt) {
                if (tt * S >= ub && (tt + 1) * S <= ue)
                    write_tile(acc, tt * 16, lane, gate_up, M, jb.N, jb.y_stride, jb.y);
                else        // part of a tile shared with other warps: summed at job end
                {
                    // lane (r, t) holds rows r, r+8 of tokens 2t, 2t+1
                    float *pk = wpark + (warp * 2 + (tt == first_tile ? 0 : 1)) * kParkSlot;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int c = 0; c < 2; ++c) pk[(2 * t + c) * kParkRow + r + 8 * h] = acc[2 * h + c];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = 0.f;
            };

            int tt = first_tile, sg = ub - first_tile * S;
            for (int u = ub; u < ue; ++u) {
                if (!__all_sync(0xffffffffu, mbar_wait(bfull + 8 * slot, phase))) {
                    ok = false;
                    break;
                }
                if (tt != cur_tile) {
                    if (cur_tile >= 0) flush(cur_tile);
                    cur_tile = tt;
                }
                accumulate(ring0 + slot * kSegBytes, ldm_off, xr + sg * 32 * 16, r, acc);
                // every lane's reads of the slot (their values are in registers)
                // are done before the copy warp may overwrite it
                __syncwarp();
                if (lane == 0) mbar_arrive(bempty + 8 * slot);
                if (++slot == kSlots) {
                    slot = 0;
                    phase ^= 1u;
                }
                if (++sg == S) {
                    sg = 0;
                    ++tt;
                }
            }
            if (!ok) {
                // leave together at the next job boundary: every compute warp
                // must still take part in the barriers there
                *s_abort = 1;
                continue;
            }
            if (cur_tile >= 0) flush(cur_tile);
        }

        if (!ok) {
            if (lane == 0) {
                atomicOr(&g_stack_error, ZQ4_DEVERR_WAIT_TIMEOUT);
                atomicOr(&p.hdr->abort, 1u);
            }
            *s_abort = 1;
        }
        compute_sync();
        if (threadIdx.x == 0 && *s_abort) atomicOr(&g_stack_error, ZQ4_DEVERR_WAIT_TIMEOUT);
        if (!*s_abort && n > 0) {                            // the last job's split tiles
            const Job &lj = job(n - 1);
            const int *ltab = wtab + ((n - 1) & 1) * kTabInts;
            sum_split_tiles(ltab[2 * (kWarps + 1)], ltab[2 * (kWarps + 1) + 1] - ltab[2 * (kWarps + 1)], lj.S,
                            lj.flags & kJobGateUp, M, lj.N, lj.y_stride, lj.y, wpark, ltab);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && !*s_abort) {
        __threadfence();
        const unsigned d = atomicAdd(&p.hdr->done, 1u);
        if (d == target - 1u) atomicAdd(&p.hdr->epoch, 1u);   // last CTA of this launch
    }
}

}  // namespace st

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Largest dynamic shared memory k_stack has been allowed per device: one
// record for every caller, so the limit only ever grows.
int stack_smem_set[kMaxDevices] = {};

struct Layout {
    size_t hdr, jobs, job_cnt, total;
};

Layout layout_for(int n_jobs)
{
    Layout l;
    l.hdr = 0;
    l.jobs = align_up(sizeof(st::Header), 128);
    l.job_cnt = l.jobs + size_t(n_jobs) * sizeof(st::Job);
    l.total = align_up(l.job_cnt + size_t(n_jobs) * 4, 256);
    return l;
}

zq4_status check_jobs(const zq4_stack_job *jobs, int n_jobs, int M, int grid, int *max_k, int *max_tiles)
{
    if (!jobs) return ZQ4_ERR_NULL;
    if (n_jobs <= 0 || M < 1 || M > st::kTokCols) return ZQ4_ERR_SHAPE;
    int mk = 0, mt = 0;
    for (int j = 0; j < n_jobs; ++j) {
        const zq4_stack_job &b = jobs[j];
        if (!b.wq || !b.x || !b.y) return ZQ4_ERR_NULL;
        if (b.scales) return ZQ4_ERR_FLAGS;     // the segmented layout carries the scales
        if (b.N <= 0 || b.K <= 0 || b.K % st::kSegCols != 0 || (b.gate_up && (b.N & 1))) return ZQ4_ERR_SHAPE;
        if (!aligned16(b.wq) || !aligned16(b.x) ||
            (reinterpret_cast<uintptr_t>(b.y) & 1))
            return ZQ4_ERR_ALIGN;
        mk = std::max(mk, b.K);
        mt = std::max(mt, (b.N + 15) / 16);
        // 32-bit part math
        const long long T = (b.N + 15) / 16, U = T * (b.K / st::kSegCols);
        if (U * std::max(grid, st::kWarps) >= (1ll << 31)) return ZQ4_ERR_UNSUPPORTED;
    }
    if (st::smem_bytes(M, mk) > size_t(227) * 1024) return ZQ4_ERR_UNSUPPORTED;
    *max_k = mk;
    *max_tiles = mt;
    return ZQ4_OK;
}

// Device entry of job j. kJobXEarly: no earlier job's output overlaps x_j,
// so the kernel may read x_j before the previous job has finished.
st::Job make_job(const zq4_stack_job *jobs, int j, int M)
{
    const zq4_stack_job &b = jobs[j];
    st::Job jb;
    memset(&jb, 0, sizeof(jb));
    jb.seg = reinterpret_cast<const uint8_t *>(b.wq);
    jb.x = b.x;
    jb.y = b.y;
    jb.N = b.N;
    jb.K = b.K;
    jb.T = (b.N + 15) / 16;
    jb.S = b.K / st::kSegCols;
    jb.y_stride = b.gate_up ? b.N / 2 : b.N;
    jb.flags = b.gate_up ? st::kJobGateUp : 0;
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(b.x), x1 = x0 + size_t(M) * size_t(b.K) * 2;
    bool early = true;
    for (int k = 0; k < j && early; ++k) {
        const zq4_stack_job &q = jobs[k];
        const size_t ys = q.gate_up ? size_t(q.N / 2) : size_t(q.N);
        const uintptr_t y0 = reinterpret_cast<uintptr_t>(q.y), y1 = y0 + size_t(M) * ys * 2;
        if (y0 < x1 && x0 < y1) early = false;
    }
    if (early) jb.flags |= st::kJobXEarly;
    return jb;
}

// Dynamic shared memory of a launch: the fixed part plus the cached jobs.
size_t launch_smem(int n_jobs, int M, int max_k)
{
    return st::smem_bytes(M, max_k) + size_t(st::cached_jobs(n_jobs, M, max_k)) * sizeof(st::Job);
}

}  // namespace

zq4_status stack_plan_bytes(const zq4_stack_job *jobs, int n_jobs, int M, size_t *bytes)
{
    if (!bytes) return ZQ4_ERR_NULL;
    int mk, mt;
    zq4_status s = check_jobs(jobs, n_jobs, M, sm_count(), &mk, &mt);
    if (s != ZQ4_OK) return s;
    *bytes = layout_for(n_jobs).total;
    return ZQ4_OK;
}

zq4_status stack_plan_init(const zq4_stack_job *jobs, int n_jobs, int M, void *dev, size_t bytes,
                           zq4_stack_plan *plan, cudaStream_t s)
{
    if (!dev || !plan) return ZQ4_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(dev) & 255) return ZQ4_ERR_ALIGN;
    int mk, mt;
    zq4_status stt = check_jobs(jobs, n_jobs, M, sm_count(), &mk, &mt);
    if (stt != ZQ4_OK) return stt;
    const int grid = sm_count();
    const Layout l = layout_for(n_jobs);
    if (bytes < l.total) return ZQ4_ERR_SHAPE;
    // the kernel needs every CTA resident at once
    const size_t smem = launch_smem(n_jobs, M, mk);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(st::k_stack), smem, stack_smem_set);
    if (e != cudaSuccess) return cuda_status(e);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, st::k_stack, st::kThreads, smem);
    if (e != cudaSuccess) return cuda_status(e);
    if (per_sm < 1) return ZQ4_ERR_UNSUPPORTED;

    std::vector<uint8_t> host(l.total, 0);
    uint8_t *hjobs = host.data() + l.jobs;
    for (int j = 0; j < n_jobs; ++j) {
        const st::Job jb = make_job(jobs, j, M);
        memcpy(hjobs + size_t(j) * sizeof(st::Job), &jb, sizeof(jb));
    }
    e = cudaMemcpyAsync(dev, host.data(), host.size(), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    plan->dev = dev;
    plan->bytes = l.total;
    plan->n_jobs = n_jobs;
    plan->M = M;
    plan->grid = grid;
    plan->max_k = mk;
    plan->max_tiles = mt;
    return ZQ4_OK;
}

zq4_status stack_run(const zq4_stack_plan *plan, cudaStream_t s)
{
    if (!plan || !plan->dev) return ZQ4_ERR_NULL;
    if (plan->grid != sm_count()) return ZQ4_ERR_SHAPE;   // initialised for another device
    const Layout l = layout_for(plan->n_jobs);
    uint8_t *base = static_cast<uint8_t *>(plan->dev);
    st::Params p;
    p.hdr = reinterpret_cast<st::Header *>(base + l.hdr);
    p.jobs = reinterpret_cast<const st::Job *>(base + l.jobs);
    p.job_cnt = reinterpret_cast<unsigned *>(base + l.job_cnt);
    p.n_jobs = plan->n_jobs;
    p.M = plan->M;
    p.max_k = plan->max_k;
    p.cached = st::cached_jobs(p.n_jobs, p.M, p.max_k);
    void *args[] = {&p};
    return cuda_status(cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(st::k_stack), dim3(plan->grid),
                                                   dim3(st::kThreads), args,
                                                   launch_smem(p.n_jobs, p.M, p.max_k), s));
}

// ---------------------------------------------------------------------------
// A plan without a caller buffer: the library's own fixed-size device array
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticPlanBytes = 64 * 1024;     // 1257 jobs
static_assert(sizeof(st::Job) == 48, "the documented job limit assumes 48-byte job entries");

// The plan lives here when the caller has no device memory to give. Header
// and counters are cleared by every zq4_stack_plan_init_static.
static __device__ __align__(256) uint8_t g_static_plan[kStaticPlanBytes];

// Device address of g_static_plan on the current device, resolved once per
// device.
cudaError_t static_plan_address(void **ptr)
{
    static std::atomic<void *> cache[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *p = cache[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_static_plan);
        if (e != cudaSuccess) return e;
        cache[dev].store(p, std::memory_order_release);
    }
    *ptr = p;
    return cudaSuccess;
}

}  // namespace

zq4_status stack_plan_init_static(const zq4_stack_job *jobs, int n_jobs, int M, zq4_stack_plan *plan,
                                  cudaStream_t s)
{
    if (!plan) return ZQ4_ERR_NULL;
    int mk, mt;
    zq4_status stt = check_jobs(jobs, n_jobs, M, sm_count(), &mk, &mt);
    if (stt != ZQ4_OK) return stt;
    const Layout l = layout_for(n_jobs);
    if (l.total > kStaticPlanBytes) return ZQ4_ERR_UNSUPPORTED;   // more jobs than the static plan holds
    const size_t smem = launch_smem(n_jobs, M, mk);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(st::k_stack), smem, stack_smem_set);
    if (e != cudaSuccess) return cuda_status(e);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, st::k_stack, st::kThreads, smem);
    if (e != cudaSuccess) return cuda_status(e);
    if (per_sm < 1) return ZQ4_ERR_UNSUPPORTED;
    void *dev = nullptr;
    e = static_plan_address(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    uint8_t *base = static_cast<uint8_t *>(dev);
    // header and counters start at zero; the job table is written after
    e = cudaMemsetAsync(base, 0, l.total, s);
    for (int j = 0; j < n_jobs && e == cudaSuccess; ++j) {
        const st::Job jb = make_job(jobs, j, M);
        // from pageable memory: the entry is staged before the call returns
        e = cudaMemcpyAsync(base + l.jobs + size_t(j) * sizeof(st::Job), &jb, sizeof(jb), cudaMemcpyHostToDevice, s);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    plan->dev = dev;
    plan->bytes = l.total;
    plan->n_jobs = n_jobs;
    plan->M = M;
    plan->grid = sm_count();
    plan->max_k = mk;
    plan->max_tiles = mt;
    return ZQ4_OK;
}

cudaError_t read_stack_error(unsigned *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_stack_error, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_stack_error, &zero, sizeof(unsigned));
}

}  // namespace zq4
