// zq4_stack.cu -- a whole decode step (a list of q4f16_1 projections, some
// reading activations that earlier ones write) as one persistent
// cooperative kernel.
//
// What it computes: for every job j, y_j = x_j * W_j^T, or the fused gate_up
// + SiLU*mul output for interleaved gate/up rows ("Zero TVM Documentation",
// section "Q4F16 quantization format", cards 5 "int4 Matmul" and 6 "Fused
// FFN"; the per-token dispatch sequence of its "Decode loop" section), with
// the results of running the jobs one after another in the given order.
//
// Why one kernel: with one launch per projection, every projection pays the
// kernel boundary (drain, launch, first-copy latency) and the small ones
// (few 16-row tiles) leave most SMs idle. Here each SM keeps streaming
// weights across job boundaries, and a job waits only where its buffers
// meet an earlier job's.
//
// How:
//  * Grid = one CTA per SM (cooperative launch, so all CTAs are resident
//    and may wait on one another): 12 compute warps, a copy warp, an x warp
//    and a release warp. Work unit = a segment, 16 weight rows x 256
//    columns.
//  * The weights are in the segmented layout (zq4_prepare_weight,
//    ZQ4_PREP_SEGMENTED): each segment is 2304 contiguous bytes (swizzled
//    codes, then scales), so one bulk copy fills a shared-memory slot and no
//    tensor map is involved. Each compute warp has its own ring of segment
//    slots; lane w of the copy warp refills ring w as soon as compute warp w
//    releases a slot (an mbarrier per slot each way), across job
//    boundaries, so the compute warps never spend issue slots on copies.
//    Per 32-column group, lane (r, t) (r = lane/4, t = lane%4) takes word t
//    of rows r and r+8 (four 16-byte shared loads fetch its words of all
//    eight groups, conflict-free in the row-record layout), unpacks exact f16
//    (q - 7) pairs as the A fragments of two chained m16n8k16 MMAs against
//    the matching x chunk (as stored), and adds the fp32 result times the
//    fp32 group scale to its accumulator.
//  * Tiles (16 output rows) are dealt round-robin over the CTAs, the jobs'
//    tiles as one sequence (Job::off), so per-CTA work over a run of jobs
//    is even to within one tile. A CTA splits the segments of its tiles
//    evenly over its compute warps; a tile that lies in one warp's range is
//    written by that warp, a warp holding part of a tile parks the part in
//    shared memory, and after a CTA barrier all compute threads sum the
//    parked parts of every split tile in warp order (bit-reproducible).
//    Tiles never span CTAs, so no partial sum goes through global memory.
//  * Order (decided on the host from the buffers' byte ranges): a job waits
//    only for the last earlier job it conflicts with (one of them writes
//    bytes the other reads or writes), until every CTA has added itself to
//    that job's counter; conflicting jobs keep their order, others may be
//    run earlier (see schedule()).
//  * x: the x warp stages x of jobs that wait for nothing into up to four
//    shared buffers ahead of the compute warps (monotone per-chunk counters
//    tell them what is there); x of a job that waits is staged by the
//    compute threads after the wait, in one round trip, and so is every x
//    when only one buffer fits.
//  * After a job's sums, the release warp makes the CTA's outputs visible
//    (one GPU-scope fence) and adds the CTA to the job's counter, off the
//    compute warps' path.
//  * The job table (as much of it as fits) is copied to shared memory once
//    per launch; each warp's copy iterator and tile position advance
//    incrementally (no division per segment).
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
#include <mutex>
#include <vector>

#include "zq4_async.cuh"
#include "zq4_common.cuh"
#include "zq4_internal.h"
#include "zq4_segment.cuh"
#include "zq4_step.h"

namespace zq4 {

__device__ unsigned g_stack_error = 0;

namespace st {

constexpr int kWarps = 12;                  // compute warps, one ring each
constexpr int kCompute = kWarps * 32;
constexpr int kCopyWarp = kWarps, kXWarp = kWarps + 1, kRelWarp = kWarps + 2;
constexpr int kThreads = kCompute + 96;      // + the copy warp, the x warp and the release warp
constexpr int kMaxChunks = 64;               // 256-column chunks of x: K <= 16384
constexpr int kXBatch = 12;                 // x rows in flight per lane of the x warp
constexpr int kSlots = 5;
using namespace segk;       // segment layout, inner loop, split-tile sums

struct Header {
    unsigned epoch;     // launches completed
    unsigned done;      // CTA arrivals at launch end (monotone)
    unsigned abort;     // set by any wait that gave up
    unsigned pad[29];
};

// Job::flags: bit 0 gate_up (rows are interleaved gate/up pairs, silu(g) * u
// output); bits 8.. the earlier job d + 1 that every CTA must be done with
// before x of this job is staged (0: none).
constexpr int kJobGateUp = 1;
constexpr int kDepShift = 8;

// Tile t of a job (16 output rows) is CTA (t + off) mod G's: the tiles of
// consecutive jobs are dealt round the CTAs as one sequence (off = the tiles
// of the earlier jobs, mod G), so a CTA that drew a tile more in one job draws
// its next only after every other CTA has, and the work of a run of jobs is
// even to within one tile across the CTAs whatever the sizes of the jobs.
struct alignas(16) Job {
    const uint8_t *seg; // the matrix in the segmented layout
    const uint16_t *x;  // [M][K]
    uint16_t *y;        // [M][N] ([M][N / 2] for gate_up)
    int N, K, T, off;
    int flags;
    int y_stride;       // N, or N / 2 for gate_up
};
__host__ __device__ inline int y_stride(const Job &jb) { return jb.y_stride; }

// This CTA's tiles of a job: t0, t0 + G, .. (nt of them).
__device__ __forceinline__ void cta_tiles(const Job &jb, int cta, int G, int &t0, int &nt)
{
    int d = cta - jb.off;
    if (d < 0) d += G;
    t0 = d;
    nt = d < jb.T ? (jb.T - 1 - d) / G + 1 : 0;
}

struct Params {
    Header *hdr;
    const Job *jobs;
    unsigned *job_cnt;            // [n_jobs]: CTAs done with each job (monotone)
    int n_jobs, M, max_k;
    int x_bufs;          // x buffers in shared memory (1 .. kMaxXBufs)
    int cached;          // jobs [0, cached) are copied to shared memory at start
    unsigned long long wait_ns;   // how long a wait on another warp or CTA may last
};

constexpr size_t kRingOff = 0;
constexpr size_t kBarOff = kRingOff + size_t(kWarps) * kSlots * kSegBytes;
constexpr size_t kXCntOff = kBarOff + 2 * size_t(kWarps) * kSlots * 8;  // full, then empty barriers
constexpr size_t kMiscOff = kXCntOff + (kMaxChunks + 4) * 4;            // chunk counters, then "x free"
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
// (+128: the base is aligned up to 128 bytes in the kernel)
__host__ __device__ inline size_t smem_bytes(int M, int max_k) { return 128 + kXsOff + xs_bytes(M, max_k); }
// x buffers: as many as fit (up to kMaxXBufs) next to room for 64 cached
// jobs, so that x of the next jobs is staged while this one computes
constexpr int kMaxXBufs = 4;
inline int x_buffers(int M, int max_k)
{
    int nb = 1;
    while (nb < kMaxXBufs && smem_bytes(M, max_k) + nb * xs_bytes(M, max_k) + 64 * sizeof(Job) <= size_t(227) * 1024)
        ++nb;
    return nb;
}
inline size_t smem_fixed(int M, int max_k) { return smem_bytes(M, max_k) + (x_buffers(M, max_k) - 1) * xs_bytes(M, max_k); }
// jobs that fit in shared memory next to everything else (the rest are read from the plan)
inline int cached_jobs(int n, int M, int max_k)
{
    const size_t left = size_t(227) * 1024 - smem_fixed(M, max_k);
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
__device__ __forceinline__ void sum_split_tiles(int t0, int G, int nt, int S, int gate_up, int M, int N, int y_stride,
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
        const int tt = it >> shift, lo = tt * S, hi = lo + S;      // local tile tt is tile t0 + tt G
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
        const int row0 = (t0 + tt * G) * 16;
        if (!gate_up) {
            if (row0 + i < N) y[size_t(m) * y_stride + row0 + i] = float_to_f16_bits(v0);
        } else if (row0 + 2 * i + 1 < N) {
            y[size_t(m) * y_stride + (row0 >> 1) + i] = float_to_f16_bits(silu_f32(v0) * v1);
        }
    }
}

// Monotone counters in shared memory between the x warp and the compute
// warps (release / acquire at CTA scope).
__device__ __forceinline__ void st_release_cta(int *p, int v)
{
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const int *p)
{
    int v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}
// Wait (bounded) until *p >= v; false once the wait has lasted longer than
// `limit` ns. Between polls the warp sleeps, leaving its issue slots to the
// warps that do the work.
__device__ __forceinline__ bool wait_at_least(const int *p, int v, unsigned long long limit)
{
    if (ld_acquire_cta(p) >= v) return true;
    const unsigned long long t0 = globaltimer();
    for (unsigned i = 0;; ++i) {
        __nanosleep(32);
        if (ld_acquire_cta(p) >= v) return true;
        if ((i & 15u) == 15u && globaltimer() - t0 > limit) return false;
    }
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1) k_stack(Params p)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128 - (smem_addr(smem_raw) & 127)) & 127);
    const uint32_t sbase = smem_addr(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, t = lane & 3;
    const int G = gridDim.x, cta = blockIdx.x;
    const uint32_t full0 = sbase + uint32_t(kBarOff), empty0 = full0 + uint32_t(kWarps * kSlots * 8);
    // s_chunk[c]: jobs whose x chunk c is staged; s_xfree: jobs the compute
    // warps are done with (so x of the next one may be staged)
    int *s_chunk = reinterpret_cast<int *>(smem + kXCntOff);
    int *s_xfree = s_chunk + kMaxChunks;
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + kMiscOff);
    // the compute warps' copy of the abort flag, written by thread 0 before a
    // compute barrier and read by all of them after it: the other warps may set
    // s_abort at any time, and every compute warp must take the same branch
    volatile int *s_cbrk = s_abort + 1;
    // jobs whose outputs this CTA has written (compute thread 0, after the
    // sums); the release warp publishes them. s_rstop: the compute warps
    // stopped early (abort), nothing more to publish
    int *s_rdone = const_cast<int *>(s_abort + 2);
    volatile int *s_rstop = s_abort + 3;
    // s_xprog: the x warp is done with every job before this one (staged or
    // skipped); x of a dependent job is staged by the compute threads only
    // then, so that they never share a buffer with the x warp's staging of an
    // earlier job (CTAs without tiles in a run of jobs can get far ahead of it)
    int *s_xprog = const_cast<int *>(s_abort + 4);
    float *wpark = reinterpret_cast<float *>(smem + kParkOff);
    int *wtab = reinterpret_cast<int *>(smem + kTabOff);
    uint8_t *xs = smem + kXsOff;                       // x of job j: xs + (j % x_bufs) * xs_size
    const int xs_size = int(xs_bytes(p.M, p.max_k));
    Job *sjobs = reinterpret_cast<Job *>(smem + kXsOff + p.x_bufs * xs_bytes(p.M, p.max_k));
    const uint32_t xrow = uint32_t(xs_row_bytes(p.max_k));
    const int n = p.n_jobs, M = p.M;
    const unsigned launch = *reinterpret_cast<volatile unsigned *>(&p.hdr->epoch);
    const unsigned target = (launch + 1u) * unsigned(G);

    if (threadIdx.x == 0) {
        *s_abort = 0;
        *s_cbrk = 0;
        *s_rdone = 0;
        *s_rstop = 0;
        *s_xprog = p.x_bufs > 1 ? 0 : p.n_jobs;
        for (int c = 0; c < kMaxChunks; ++c) s_chunk[c] = 0;
        *s_xfree = 0;
    }
    if (warp < kWarps && lane == 0) {
        for (int j = 0; j < kSlots; ++j) {
            mbar_init(full0 + 8 * (warp * kSlots + j), 1);    // the copy's bytes
            mbar_init(empty0 + 8 * (warp * kSlots + j), 1);   // the consuming warp is done
        }
    }
    if (lane == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    {
        // the job table (or its first p.cached entries) into shared memory
        const uint4 *src = reinterpret_cast<const uint4 *>(p.jobs);
        uint4 *dst = reinterpret_cast<uint4 *>(sjobs);
        const int words = p.cached * int(sizeof(Job) / 16);
        for (int i = threadIdx.x; i < words; i += kThreads) dst[i] = src[i];
    }
    __syncthreads();
    auto job = [&](int j) -> const Job & { return j < p.cached ? sjobs[j] : p.jobs[j]; };

    // compute warp w's part of this CTA's segments of a job, numbered tile
    // major over the CTA's tiles (local segment u: tile t0 + (u / S) G,
    // column segment u % S); a tile never spans two CTAs
    auto warp_range = [&](const Job &jb, int w, int &ub, int &ue, int &t0) {
        int nt;
        cta_tiles(jb, cta, G, t0, nt);
        split(0, nt * (jb.K >> 8), w, kWarps, ub, ue);
    };

    if (warp == kCopyWarp) {
        // ---------------- the copy warp ----------------
        // Lane w keeps ring w full: it walks compute warp w's (job, segment)
        // sequence (segment sg of tile t of a job is at byte (t S + sg) *
        // kSegBytes of its matrix) and refills a slot as soon as that warp
        // has released it, across job boundaries: the weights never depend on
        // earlier jobs.
        const int w = lane;
        const uint32_t ring = sbase + uint32_t(kRingOff) + uint32_t(w * kSlots * kSegBytes);
        int it_j = n, it_left = 0, it_S = 1, it_sg = 0, issued = 0;
        const uint8_t *it_ptr = nullptr;          // the next segment
        auto seek = [&](int j) {
            for (; j < n; ++j) {
                const Job &jb = job(j);
                int ub, ue, t0;
                warp_range(jb, w, ub, ue, t0);
                if (ub < ue) {
                    const int S = jb.K >> 8, k = ub / S;
                    it_j = j;
                    it_left = ue - ub;
                    it_S = S;
                    it_sg = ub - k * S;
                    it_ptr = jb.seg + (size_t(t0 + k * G) * S + it_sg) * kSegBytes;
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
                    bulk_load(ring + slot * kSegBytes, it_ptr, kSegBytes, full);
                    ++issued;
                    did = true;
                    if (--it_left == 0) {
                        seek(it_j + 1);
                    } else if (++it_sg == it_S) {       // next tile of this CTA: G tiles on
                        it_sg = 0;
                        it_ptr += (size_t(G - 1) * it_S + 1) * kSegBytes;
                    } else {
                        it_ptr += kSegBytes;
                    }
                }
            }
            if (!__any_sync(0xffffffffu, more)) break;
            if (__any_sync(0xffffffffu, did)) {
                t0 = globaltimer();
            } else {
                // no slot free: the compute warps are busy or between jobs
                if (globaltimer() - t0 > p.wait_ns) {
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
    } else if (warp == kRelWarp) {
        // ---------------- the release warp ----------------
        // Publishes "this CTA is done with job j" (an add on the job's
        // counter) once the compute warps have written the CTA's outputs of
        // job j: one GPU-scope fence, then the add. The fence
        // waits for the CTA's writes to reach the whole GPU (about a
        // microsecond under a full memory stream); here it holds up no
        // compute warp. The release is cumulative: the outputs were written
        // before compute thread 0's CTA-scope release of s_rdone, which this
        // lane acquires first.
        if (lane == 0) {
            for (int j = 0; j < n; ++j) {
                if (!wait_at_least(s_rdone, j + 1, p.wait_ns)) {
                    atomicOr(&g_stack_error, ZQ4_DEVERR_WAIT_TIMEOUT);
                    atomicOr(&p.hdr->abort, 1u);
                    *s_abort = 1;
                    break;
                }
                if (*s_rstop) break;
                fence_acq_rel_gpu();
                asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(&p.job_cnt[j]) : "memory");
            }
        }
    } else if (warp == kXWarp) {
        // ---------------- the x warp ----------------
        // Stages x of every job that depends on no earlier job (decided on
        // the host from the buffers: Job::flags) into shared memory ahead of
        // the compute warps, kXBatch 512-byte rows of 256-column chunks in
        // flight at a time (lane l moves bytes 16l.. of each row), into
        // buffer j % x_bufs once the compute warps are past the job that used
        // it last. s_chunk[c] = j + 1 once chunk c of job j is staged
        // (monotone, so a fast compute warp can never mistake an earlier
        // job's chunk for this one's). x of a job that does depend on an
        // earlier one is staged by the compute warps after their wait, and so
        // is every x when there is one buffer only (nothing to stage ahead
        // into; the compute threads move it in one round trip).
        bool stop = false;
        for (int j = 0; j < n && !stop && p.x_bufs > 1; ++j) {
            const Job &jb = job(j);
            if (lane == 0) st_release_cta(s_xprog, j);       // every earlier job's x is in place
            if ((jb.flags >> kDepShift) != 0) continue;
            if (j >= p.x_bufs && !wait_at_least(s_xfree, j + 1 - p.x_bufs, p.wait_ns)) {
                stop = true;
                break;
            }
            if (*s_abort) {
                stop = true;
                break;
            }
            uint8_t *xsj = xs + (j % p.x_bufs) * xs_size;
            const int nch = jb.K >> 8, words = jb.K >> 3;
            const unsigned long long all = nch >= 64 ? ~0ull : ((1ull << nch) - 1ull);
            unsigned long long rem = all;
            int ck = __ffsll(rem) - 1, cm = 0;
            const uint4 *xg = reinterpret_cast<const uint4 *>(jb.x) + lane;
            while (rem) {
                int qc[kXBatch];                  // chunk | token << 8, or -1
#pragma unroll
                for (int q = 0; q < kXBatch; ++q) {
                    qc[q] = -1;
                    if (rem) {
                        qc[q] = ck | (cm << 8);
                        if (++cm == M) {
                            cm = 0;
                            rem &= rem - 1;
                            ck = __ffsll(rem) - 1;
                        }
                    }
                }
                uint4 v[kXBatch];
#pragma unroll
                for (int q = 0; q < kXBatch; ++q)
                    if (qc[q] >= 0) v[q] = __ldcg(xg + (qc[q] >> 8) * words + (qc[q] & 255) * 32);
#pragma unroll
                for (int q = 0; q < kXBatch; ++q)
                    if (qc[q] >= 0)
                        *reinterpret_cast<uint4 *>(xsj + (qc[q] >> 8) * int(xrow) + ((qc[q] & 255) * 32 + lane) * 16) =
                            v[q];
            }
            __syncwarp();
            // lane l publishes chunks l and l + 32
            if ((all >> lane) & 1ull) st_release_cta(s_chunk + lane, j + 1);
            if ((all >> (lane + 32)) & 1ull) st_release_cta(s_chunk + lane + 32, j + 1);
        }
        if (lane == 0) st_release_cta(s_xprog, stop ? (1 << 30) : n);
        if (stop) {
            // release every chunk, so that no compute warp waits on one (the results are void)
            if (lane == 0)
                for (int kc = 0; kc < kMaxChunks; ++kc) st_release_cta(s_chunk + kc, 1 << 30);
            if (lane == 0 && !*s_abort) {
                atomicOr(&g_stack_error, ZQ4_DEVERR_WAIT_TIMEOUT);
                atomicOr(&p.hdr->abort, 1u);
                *s_abort = 1;
            }
        }
    } else {
        // ---------------- compute warps ----------------
        const uint32_t ring0 = sbase + uint32_t(kRingOff) + uint32_t(warp * kSlots * kSegBytes);
        const uint32_t bfull = full0 + uint32_t(8 * warp * kSlots), bempty = empty0 + uint32_t(8 * warp * kSlots);
        const uint32_t aoff = lane_code_offset(lane);
        const uint8_t *xr = xs + size_t(min(r, M - 1)) * xrow + 16 * t;

        // the warp range table of job j (one of two buffers, so that the table
        // of the next job can be made while the sums of the last one read theirs):
        // lanes 0..kWarps of warp `tw`
        auto set_wtab = [&](const Job &jb, int j, int tw) {
            const int q = int(threadIdx.x) - 32 * tw;
            if (q >= 0 && q <= kWarps) {
                int t0, nt;
                cta_tiles(jb, cta, G, t0, nt);
                const int S = jb.K >> 8;
                const int b = part_begin(0, nt * S, q, kWarps);
                int *tab = wtab + (j & 1) * kTabInts;
                tab[q] = b;                           // local segments, tile major
                tab[kWarps + 1 + q] = b / S;          // local tile
                if (q == 0) {
                    tab[2 * (kWarps + 1)] = t0;       // this CTA's tiles of the job: t0, t0 + G, ..
                    tab[2 * (kWarps + 1) + 1] = nt;
                }
            }
        };

        bool ok = true;
        int slot = 0;             // ring position of the next segment and the parity of its fill
        uint32_t phase = 0;
        set_wtab(job(0), 0, 0);
        compute_sync();
        for (int j = 0; j < n; ++j) {
            const Job &jb = job(j);
            const int S = jb.K >> 8, gate_up = jb.flags & kJobGateUp;
            const int *tab = wtab + (j & 1) * kTabInts;
            const int ub = tab[warp], ue = tab[warp + 1], first_tile = tab[kWarps + 1 + warp];
            const int ct0 = tab[2 * (kWarps + 1)];   // local tile k is tile ct0 + k G
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            int cur_tile = -1;
            auto flush = [&](int tt) {
                if (tt * S >= ub && (tt + 1) * S <= ue)
                    write_tile(acc, (ct0 + tt * G) * 16, lane, gate_up, M, jb.N, y_stride(jb), jb.y);
                else {
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
            const uint8_t *xrj = xr + (j % p.x_bufs) * xs_size;
            unsigned long long seen = 0;          // x chunks of this job known to be staged
            const int dep = (jb.flags >> kDepShift) - 1;
            if (dep >= 0 || p.x_bufs == 1) {
                // x depends on earlier jobs (every CTA must be done with job
                // dep: thread 0 waits, the barrier passes its acquire on) or
                // there is no buffer to stage ahead into: the compute threads
                // stage x, all loads in one round trip
                if (threadIdx.x == 0 && !wait_at_least(s_xprog, j, p.wait_ns)) {
                    atomicOr(&g_stack_error, ZQ4_DEVERR_WAIT_TIMEOUT);
                    atomicOr(&p.hdr->abort, 1u);
                    *s_abort = 1;
                }
                if (threadIdx.x == 0 && dep >= 0) {
                    const unsigned long long t0 = globaltimer();
                    while (int(ld_acquire(&p.job_cnt[dep]) - target) < 0) {   // wrap-safe: counters grow across launches
                        if (*s_abort || *reinterpret_cast<volatile unsigned *>(&p.hdr->abort) ||
                            globaltimer() - t0 > p.wait_ns) {
                            atomicOr(&g_stack_error, ZQ4_DEVERR_WAIT_TIMEOUT);
                            atomicOr(&p.hdr->abort, 1u);
                            *s_abort = 1;
                            break;
                        }
                    }
                }
                compute_sync();
                uint8_t *xsj = xs + (j % p.x_bufs) * xs_size;
                const int words = jb.K >> 3, total = M * words;
                const uint4 *xg = reinterpret_cast<const uint4 *>(jb.x);
                for (int i0 = int(threadIdx.x); i0 < total; i0 += 4 * kCompute) {
                    uint4 v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (i0 + q * kCompute < total) v[q] = __ldcg(xg + i0 + q * kCompute);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int i = i0 + q * kCompute;
                        if (i < total) {
                            const int m = i / words;
                            *reinterpret_cast<uint4 *>(xsj + m * int(xrow) + (i - m * words) * 16) = v[q];
                        }
                    }
                }
                compute_sync();
                seen = ~0ull;
            }
            for (int u = ub; u < ue && ok; ++u) {
                // x chunk sg of this job (segment sg of a tile covers columns 256 sg ..)
                if (!((seen >> sg) & 1ull)) {
                    if (!__all_sync(0xffffffffu, wait_at_least(s_chunk + sg, j + 1, p.wait_ns))) {
                        ok = false;
                        break;
                    }
                    seen |= 1ull << sg;
                }
                if (!__all_sync(0xffffffffu, mbar_wait(bfull + 8 * slot, phase))) {
                    ok = false;
                    break;
                }
                if (tt != cur_tile) {
                    if (cur_tile >= 0) flush(cur_tile);
                    cur_tile = tt;
                }
                accumulate(ring0 + slot * kSegBytes, aoff, xrj + sg * 32 * 16, r, acc);
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
            if (ok && cur_tile >= 0) flush(cur_tile);
            if (!ok) *s_abort = 1;
            compute_sync();                       // every compute warp is done with x and its segments
            if (threadIdx.x == 0) st_release_cta(s_xfree, j + 1);
            if (j + 1 < n) set_wtab(job(j + 1), j + 1, 1);
            if (!*s_abort) {
                const int *ptab = wtab + (j & 1) * kTabInts;
                sum_split_tiles(ptab[2 * (kWarps + 1)], G, ptab[2 * (kWarps + 1) + 1], S, gate_up, M, jb.N, y_stride(jb),
                                jb.y, wpark, ptab);
            }
            if (threadIdx.x == 0) *s_cbrk = *s_abort;
            compute_sync();                       // the split-tile sums before the release below
            const bool brk = *s_cbrk != 0;
            if (threadIdx.x == 0) {
                // the release warp publishes this CTA's outputs of job j
                if (brk) *s_rstop = 1;
                st_release_cta(s_rdone, brk ? (1 << 30) : j + 1);
            }
            if (brk) break;
        }
        if (!ok && lane == 0) {
            atomicOr(&g_stack_error, ZQ4_DEVERR_WAIT_TIMEOUT);
            atomicOr(&p.hdr->abort, 1u);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && *s_abort) atomicOr(&g_stack_error, ZQ4_DEVERR_WAIT_TIMEOUT);
    if (threadIdx.x == 0 && !*s_abort) {
        __threadfence();
        const unsigned d = atomicAdd(&p.hdr->done, 1u);
        if (d == target - 1u) atomicAdd(&p.hdr->epoch, 1u);   // last CTA of this launch
    }
}

}  // namespace st

// ---------------------------------------------------------------------------
// Host side: the plan API shared by both engines (this file's k_stack for 3..8
// tokens, zq4_step.cu's k_step for 1 or 2)
// ---------------------------------------------------------------------------
namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

enum Engine { kEngineStack = 0, kEngineStep = 1, kEngineWide = 2 };
// engines that run the step plan (job entries, split parts, finisher)
inline bool step_like(int engine) { return engine == kEngineStep || engine == kEngineWide; }

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

// Work (segments) to place between a job and a job that waits for it, beyond
// the job's own work: two tiles per compute warp of a full GB300 (152 SMs x
// 16 warps), so that in the step engine, where each warp takes tiles one at
// a time, the last tiles of the job are done before the first tiles of the
// waiting job are handed out. A constant, so the order does not depend on
// the device (a smaller GPU only gets more room than it needs).
constexpr long long kSlackTiles = 2ll * 152 * kStepWarps;

// Parts per tile of the job run at position r of a step-engine plan: its
// tiles are split along K (step_split) only when they start so late that a
// whole tile would outlast the rest of the step, i.e. when the work from the
// job's start to the end (segments) is less than kSlackTiles tiles of its
// length (every compute warp of a full GB300 taking two such tiles); earlier
// tiles run whole, with no workspace traffic. f(r, C) for every position.
template <class F>
void for_each_split(const zq4_stack_job *jobs, int n, const int *order, F f)
{
    long long rest = 0;
    for (int r = 0; r < n; ++r) rest += (long long)((jobs[order[r]].N + 15) / 16) * (jobs[order[r]].K / st::kSegCols);
    for (int r = 0; r < n; ++r) {
        const zq4_stack_job &b = jobs[order[r]];
        const long long S = b.K / st::kSegCols;
        f(r, rest < kSlackTiles * S ? step_split(b.K) : 1);
        rest -= (long long)((b.N + 15) / 16) * S;
    }
}

// The split workspace of a step-engine plan: tiles split along K and their
// 16-float part records, over all jobs; none at all when the records would
// take more than kStepMaxWorkBytes.
struct SplitTotals {
    long long tiles = 0, records = 0;
    int entries = 0;          // job-table entries (a split job has one per part)
    bool on = false;
};
SplitTotals split_totals(const zq4_stack_job *jobs, int n, int M, const int *order)
{
    SplitTotals t;
    long long entries = 0;
    for_each_split(jobs, n, order, [&](int r, int C) {
        entries += C;
        if (C == 1) return;
        const long long rows = (jobs[order[r]].N + 15) / 16;
        t.tiles += rows;
        t.records += rows * C * M;
    });
    t.on = t.records > 0 && t.records * 64 <= (long long)kStepMaxWorkBytes && entries < (1 << 20);
    if (!t.on) t.tiles = t.records = 0;
    t.entries = t.on ? int(entries) : n;
    return t;
}

// Device bytes of a plan, and the part of them the host image covers (the
// rest: the split counters, cleared by a memset, and the part records, which
// need no initial value).
size_t plan_bytes_for(int engine, const zq4_stack_job *jobs, int n, int M, const int *order)
{
    if (!step_like(engine)) return layout_for(n).total;
    const SplitTotals t = split_totals(jobs, n, M, order);
    return StepLayout(t.entries, t.tiles, t.records, engine == kEngineWide).total;
}
// `entries`: job-table entries (the step engine), else jobs
size_t image_bytes_for(int engine, int entries)
{
    return step_like(engine) ? StepLayout(entries, 0, 0, engine == kEngineWide).arrive : layout_for(entries).total;
}
int entries_for(int engine, const zq4_stack_job *jobs, int n, int M, const int *order)
{
    return step_like(engine) ? split_totals(jobs, n, M, order).entries : n;
}

zq4_status check_jobs(const zq4_stack_job *jobs, int n_jobs, int M, int grid, int *max_k, int *max_tiles)
{
    if (!jobs) return ZQ4_ERR_NULL;
    if (n_jobs <= 0 || M < 1 || M > kWideMaxM) return ZQ4_ERR_SHAPE;
    int mk = 0, mt = 0;
    long long tiles = 0;
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
        tiles += T;
    }
    if (tiles >= (1ll << 31)) return ZQ4_ERR_UNSUPPORTED;
    *max_k = mk;
    *max_tiles = mt;
    return ZQ4_OK;
}

// What only the stack engine (k_stack) requires.
zq4_status stack_engine_fits(int M, int max_k)
{
    if (M > st::kTokCols) return ZQ4_ERR_UNSUPPORTED;                       // eight tokens at most
    if (max_k > st::kMaxChunks * st::kSegCols) return ZQ4_ERR_UNSUPPORTED;   // x staged in at most 64 chunks
    if (st::smem_bytes(M, max_k) > size_t(227) * 1024) return ZQ4_ERR_UNSUPPORTED;
    return ZQ4_OK;
}

// Byte ranges of a job's x and y.
struct Span {
    uintptr_t lo, hi;
    bool meets(const Span &o) const { return lo < o.hi && o.lo < hi; }
};
inline Span x_span(const zq4_stack_job &b, int M)
{
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(b.x);
    return {x0, x0 + size_t(M) * size_t(b.K) * 2};
}
inline Span y_span(const zq4_stack_job &b, int M)
{
    const uintptr_t y0 = reinterpret_cast<uintptr_t>(b.y);
    return {y0, y0 + size_t(M) * size_t(b.gate_up ? b.N / 2 : b.N) * 2};
}

// Do jobs a and b touch the same bytes, one of them writing?
bool conflict(const zq4_stack_job &a, const zq4_stack_job &b, int M)
{
    const Span xa = x_span(a, M), ya = y_span(a, M), xb = x_span(b, M), yb = y_span(b, M);
    return ya.meets(xb) || ya.meets(yb) || xa.meets(yb);
}

constexpr int kLookAhead = 32;   // jobs a waiting job may be passed by
constexpr int kProducerAhead = 12; // jobs a job that others wait for may pass (three layers of four projections)


// Scratch for the host scheduling (n entries each; anc: n bitsets of
// `words` 64-bit words), from the caller so that the static-plan path
// allocates nothing.
struct SchedScratch {
    long long *work, *need, *at;
    char *placed, *prod;
    int *nwait;
    int *first;                  // step engine: the job-table entry of each position's part 0
    int (*waits)[kStepMaxWaits];
    uint64_t *anc;
    int words;
};

// The order the kernel runs the jobs in and the wait before each. The
// results are those of the given order: two jobs that conflict keep their
// order. Within that, a job that would wait for a job placed shortly before
// it lets later jobs that conflict with no job still to place (it included)
// and wait for nothing recent go first, until the job it waits for is
// followed by at least its own work and kSlackTiles of its tiles' segments:
// the SMs that finish the first job early work on those meanwhile instead of
// waiting for the last ones.
//
// dep[r] (positions in run order) = the last job before r that conflicts
// with it (-1: none).
void schedule(const zq4_stack_job *jobs, int n, int M, int *order, int *dep, const SchedScratch &sc)
{
    long long *work = sc.work, *need = sc.need, *at = sc.at;
    char *placed = sc.placed;
    for (int i = 0; i < n; ++i) {
        const long long S = jobs[i].K / st::kSegCols;
        work[i] = (long long)((jobs[i].N + 15) / 16) * S;
        need[i] = std::max(work[i], kSlackTiles * S);
        at[i] = -1;
        placed[i] = 0;
        sc.prod[i] = 0;
        for (int j = i + 1; j < n && !sc.prod[i]; ++j)
            if (conflict(jobs[i], jobs[j], M)) sc.prod[i] = 1;
    }
    int n_placed = 0;
    long long total = 0;
    // how much more work must be placed before job j runs without a wait on a recent job
    auto short_by = [&](int j) {
        long long sh = 0;
        for (int i = 0; i < n; ++i)
            if (placed[i] && conflict(jobs[i], jobs[j], M)) sh = std::max(sh, need[i] - (total - at[i]));
        return sh;
    };
    // the largest job that touches no other job's bytes runs last: whatever
    // it waits for, it can fill the end of the step with its tiles while the
    // last waiting jobs finish
    // (only when some job waits at all)
    int last = -1;
    bool any_wait = false;
    for (int j = 0; j < n; ++j) {
        bool alone = true;
        for (int i = 0; i < n && alone; ++i)
            if (i != j && conflict(jobs[i], jobs[j], M)) alone = false;
        any_wait |= !alone;
        if (alone && (last < 0 || work[j] > work[last])) last = j;
    }
    if (!any_wait) last = -1;
    if (n > 1 && last >= 0) placed[last] = 1;
    int first = 0;
    while (n_placed < n - (n > 1 && last >= 0 ? 1 : 0)) {
        while (placed[first]) ++first;
        // may job k run next: no unplaced job before it conflicts with it,
        // and whatever it waits for has had its room
        auto may_run = [&](int k) {
            if (placed[k]) return false;
            for (int i = first; i < k; ++i)
                if (!placed[i] && conflict(jobs[i], jobs[k], M)) return false;
            return short_by(k) <= 0;
        };
        int pick = first;
        if (short_by(first) > 0)
            for (int k = first + 1; k < n && k <= first + kLookAhead; ++k)
                if (may_run(k)) {
                    pick = k;
                    break;
                }
        // a job some later job waits for goes before the independent jobs
        // just after the pick, so that the job waiting for it gets more room
        if (!sc.prod[pick])
            for (int k = pick + 1; k < n && k <= pick + kProducerAhead; ++k)
                if (sc.prod[k] && may_run(k)) {
                    pick = k;
                    break;
                }
        placed[pick] = 1;
        total += work[pick];
        at[pick] = total;
        order[n_placed++] = pick;
    }
    if (n_placed < n) {
        total += work[last];
        at[last] = total;
        order[n_placed++] = last;
    }
    for (int r = 0; r < n; ++r) {
        int q = r - 1;
        while (q >= 0 && !conflict(jobs[order[q]], jobs[order[r]], M)) --q;
        dep[r] = q;
    }
}

// The step engine's waits (positions in run order): every earlier job that
// conflicts with job r, except those already complete when another of its
// waits is (a job's tiles start only after its own waits are complete).
// False if some job would need more than kStepMaxWaits.
bool wait_lists(const zq4_stack_job *jobs, int n, int M, const int *order, const SchedScratch &sc)
{
    const int W = sc.words;
    for (int r = 0; r < n; ++r) {
        uint64_t *ar = sc.anc + size_t(r) * W;
        for (int w = 0; w < W; ++w) ar[w] = 0;
        sc.nwait[r] = 0;
        for (int q = r - 1; q >= 0; --q) {
            if ((ar[q >> 6] >> (q & 63)) & 1u) continue;               // implied by a later wait
            if (!conflict(jobs[order[q]], jobs[order[r]], M)) continue;
            if (sc.nwait[r] == kStepMaxWaits) return false;
            sc.waits[r][sc.nwait[r]++] = q;
            const uint64_t *aq = sc.anc + size_t(q) * W;
            for (int w = 0; w < W; ++w) ar[w] |= aq[w];
            ar[q >> 6] |= uint64_t(1) << (q & 63);
        }
    }
    return true;
}

// Device entry of the job run at position r (stack engine).
st::Job make_job(const zq4_stack_job &b, int off, int dep)
{
    st::Job jb;
    memset(&jb, 0, sizeof(jb));
    jb.seg = reinterpret_cast<const uint8_t *>(b.wq);
    jb.x = b.x;
    jb.y = b.y;
    jb.N = b.N;
    jb.K = b.K;
    jb.T = (b.N + 15) / 16;
    jb.off = off;
    jb.y_stride = b.gate_up ? b.N / 2 : b.N;
    jb.flags = (b.gate_up ? st::kJobGateUp : 0) | ((dep + 1) << st::kDepShift);
    return jb;
}

// Heap scratch for the calls that may allocate.
struct SchedBuffers {
    std::vector<int> order, dep, nwait, first;
    std::vector<long long> work, need, at;
    std::vector<char> placed, prod;
    std::vector<int> waits;
    std::vector<uint64_t> anc;
    int words;
    explicit SchedBuffers(int n)
        : order(n), dep(n), nwait(n), first(n), work(n), need(n), at(n), placed(n), prod(n), waits(size_t(n) * kStepMaxWaits),
          anc(size_t(n) * ((n + 63) / 64)), words((n + 63) / 64) {}
    SchedScratch scratch()
    {
        return {work.data(), need.data(), at.data(), placed.data(), prod.data(), nwait.data(), first.data(),
                reinterpret_cast<int(*)[kStepMaxWaits]>(waits.data()), anc.data(), words};
    }
};

// Jobs that wait for a job placed with less than half its room before them
// (a chain of projections, each reading the one before, has nothing to put
// in between).
int tight_waits(int n, const int *order, const int *dep, const SchedScratch &sc)
{
    int tight = 0;
    for (int r = 0; r < n; ++r) {
        if (dep[r] < 0) continue;
        const int j = order[r], d = order[dep[r]];
        if (2 * ((sc.at[j] - sc.work[j]) - sc.at[d]) < sc.need[d]) ++tight;
    }
    return tight;
}

// The engine a plan of these jobs runs on: k_step for one or two tokens
// when every job needs at most kStepMaxWaits waits and at most one job in
// eight waits for a job placed shortly before it (k_step computes a whole
// tile per warp: a job's last tiles take a tile's time, which a waiting job
// pays in full, where k_stack splits every tile of a job over a CTA's warps);
// else k_stack. Three to sixteen tokens: k_wide under the same rule (for
// nine tokens and more whatever the waits, as long as each job needs at most
// kStepMaxWaits: k_stack holds eight).
int choose_engine(const zq4_stack_job *jobs, int n, int M, const int *order, const int *dep, const SchedScratch &sc)
{
    if (n >= kStepMaxPub) return kEngineStack;
    const bool loose = 8 * tight_waits(n, order, dep, sc) <= n;
    if (M <= kStepMaxM && loose && wait_lists(jobs, n, M, order, sc)) return kEngineStep;
    if (M > kStepMaxM && (loose || M > st::kTokCols) && wait_lists(jobs, n, M, order, sc)) return kEngineWide;
    return kEngineStack;
}

// What write_image reports besides the image.
struct ImageInfo {
    bool ok = true;           // false: a tensor map could not be encoded
    long long tiles = 0;      // work units of the launch
    int entries = 0;          // job-table entries (step engine: a split job has one per part)
    int n_pub = 0;            // jobs another job waits for (step engine)
    int min_unit = 0;         // segments of the shortest work unit
    long long split_tiles = 0, part_records = 0;
};

// The plan's device image (header zero, job table, counters zero) into `host`
// (image_bytes_for(engine, entries) bytes), for G CTAs. The schedule must
// have been computed into sc / order / dep (and the wait lists for the step
// engine).
void write_image(int engine, const zq4_stack_job *jobs, int n, int M, const int *order, const int *dep,
                 const SchedScratch &sc, int G, uint8_t *host, ImageInfo *info)
{
    *info = ImageInfo();
    if (!step_like(engine)) {
        memset(host, 0, image_bytes_for(engine, n));
        info->entries = n;
        st::Job *t = reinterpret_cast<st::Job *>(host + layout_for(n).jobs);
        for (int r = 0, off = 0; r < n; ++r) {
            t[r] = make_job(jobs[order[r]], off, dep[r]);
            off = int((off + (long long)t[r].T) % G);
        }
        info->min_unit = 1 << 30;
        for (int j = 0; j < n; ++j) info->min_unit = std::min(info->min_unit, jobs[j].K / st::kSegCols);
        return;
    }
    const SplitTotals split = split_totals(jobs, n, M, order);
    memset(host, 0, image_bytes_for(engine, split.entries));
    const StepLayout lay(split.entries, 0, 0, engine == kEngineWide);
    StepJob *t = reinterpret_cast<StepJob *>(host + lay.jobs);
    // the entry of part 0 of each position
    int e = 0;
    for_each_split(jobs, n, order, [&](int r, int Cr) {
        sc.first[r] = e;
        e += split.on ? Cr : 1;
    });
    long long tile0 = 0, sbase = 0, pbase = 0;
    int min_unit = 1 << 30, n_pub = 0;
    for_each_split(jobs, n, order, [&](int r, int Cr) {
        const zq4_stack_job &b = jobs[order[r]];
        const int rows = (b.N + 15) / 16, S = b.K / st::kSegCols;
        const int C = split.on ? Cr : 1;
        // jobs some later job waits for count their units for it
        bool waited = false;
        for (int q = r + 1; q < n && !waited; ++q)
            for (int w = 0; w < sc.nwait[q]; ++w) waited |= sc.waits[q][w] == r;
        const int pub = waited ? n_pub++ : 0;
        for (int c = 0; c < C; ++c) {
            const int c0 = c * S / C, len = (c + 1) * S / C - c0;
            StepJob &jb = t[sc.first[r] + c];
            jb.seg = reinterpret_cast<const uint8_t *>(b.wq) + size_t(c0) * st::kSegBytes;
            jb.x = b.x + size_t(c0) * st::kSegCols;
            jb.y = b.y;
            jb.N = b.N;
            jb.K = len * st::kSegCols;
            jb.tstride = S;
            jb.tile0 = int(tile0);
            jb.flags = (b.gate_up ? kStepGateUp : 0) | (sc.nwait[r] << kStepWaitShift) |
                       ((C - 1) << kStepSplitShift) | (c << kStepPartShift) |
                       (waited ? kStepPublish | (pub << kStepPubShift) : 0);
            jb.sbase = C > 1 ? int(sbase) : 0;
            jb.pbase = C > 1 ? int(pbase) : 0;
            for (int w = 0; w < kStepMaxWaits; ++w) jb.wait[w] = w < sc.nwait[r] ? sc.first[sc.waits[r][w]] : 0;
            // k_wide: the entry's x columns as a tensor map of [M][256] boxes
            if (engine == kEngineWide &&
                !wide_x_map(host + lay.tmaps + size_t(sc.first[r] + c) * 128, jb.x, M, jb.K, b.K))
                info->ok = false;
            // work units: tiles, or groups of wide_group(M) tiles for k_wide
            const int G = engine == kEngineWide ? wide_group(M) : 1;
            tile0 += (rows + G - 1) / G;
            min_unit = std::min(min_unit, len);
        }
        if (C > 1) {
            sbase += rows;
            pbase += (long long)rows * C;
        }
    });
    info->tiles = tile0;
    info->entries = split.entries;
    info->n_pub = n_pub;
    info->min_unit = min_unit;
    info->split_tiles = sbase;
    info->part_records = pbase * M;
}

// The image, then the split counters cleared, on stream s (synchronised).
zq4_status upload_plan(void *dev, const uint8_t *image, int engine, const ImageInfo &info, cudaStream_t s)
{
    cudaError_t e = cudaMemcpyAsync(dev, image, image_bytes_for(engine, info.entries), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && step_like(engine) && info.split_tiles > 0) {
        const StepLayout l(info.entries, info.split_tiles, info.part_records, engine == kEngineWide);
        e = cudaMemsetAsync(static_cast<uint8_t *>(dev) + l.arrive, 0, l.work - l.arrive, s);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? ZQ4_OK : cuda_status(e);
}

// Kernel attributes and residency for a launch of this plan shape.
zq4_status check_resident(int engine, int n_jobs, int M, int max_k, int n_pub);

// Dynamic shared memory of a stack-engine launch: the fixed part plus the cached jobs.
size_t launch_smem(int n_jobs, int M, int max_k)
{
    return st::smem_fixed(M, max_k) + size_t(st::cached_jobs(n_jobs, M, max_k)) * sizeof(st::Job);
}

zq4_status check_resident(int engine, int n_jobs, int M, int max_k, int n_pub)
{
    if (engine == kEngineStep) return step_check_resident(M, max_k, n_jobs, n_pub);
    if (engine == kEngineWide) return wide_check_resident(M, n_jobs, n_pub);
    const size_t smem = launch_smem(n_jobs, M, max_k);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(st::k_stack), smem, stack_smem_set);
    if (e != cudaSuccess) return cuda_status(e);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, st::k_stack, st::kThreads, smem);
    if (e != cudaSuccess) return cuda_status(e);
    return per_sm < 1 ? ZQ4_ERR_UNSUPPORTED : ZQ4_OK;
}

// Checks, schedule and engine choice shared by every entry point.
zq4_status plan_common(const zq4_stack_job *jobs, int n_jobs, int M, int grid, int *order, int *dep,
                       const SchedScratch &sc, int *engine, int *max_k, int *max_tiles)
{
    zq4_status st = check_jobs(jobs, n_jobs, M, grid, max_k, max_tiles);
    if (st != ZQ4_OK) return st;
    schedule(jobs, n_jobs, M, order, dep, sc);
    *engine = choose_engine(jobs, n_jobs, M, order, dep, sc);
    if (*engine == kEngineStack) return stack_engine_fits(M, *max_k);
    return ZQ4_OK;
}

int current_device()
{
    int d = -1;
    return cudaGetDevice(&d) == cudaSuccess ? d : -1;
}

}  // namespace

zq4_status stack_plan_waits(const zq4_stack_job *jobs, int n_jobs, int M, int *order, int *dep)
{
    if (!order || !dep) return ZQ4_ERR_NULL;
    if (!jobs) return ZQ4_ERR_NULL;
    if (n_jobs <= 0) return ZQ4_ERR_SHAPE;
    SchedBuffers b(n_jobs);
    int engine, mk, mt;
    const zq4_status st = plan_common(jobs, n_jobs, M, 1, b.order.data(), b.dep.data(), b.scratch(), &engine, &mk, &mt);
    if (st != ZQ4_OK) return st;
    for (int r = 0; r < n_jobs; ++r) {
        const int *o = b.order.data();
        order[r] = o[r];
        dep[o[r]] = b.dep[r] >= 0 ? o[b.dep[r]] : -1;      // as indices of the given list
    }
    return ZQ4_OK;
}

zq4_status stack_plan_bytes(const zq4_stack_job *jobs, int n_jobs, int M, size_t *bytes)
{
    if (!bytes) return ZQ4_ERR_NULL;
    if (!jobs) return ZQ4_ERR_NULL;
    if (n_jobs <= 0) return ZQ4_ERR_SHAPE;
    SchedBuffers b(n_jobs);
    int engine, mk, mt;
    const zq4_status s = plan_common(jobs, n_jobs, M, sm_count(), b.order.data(), b.dep.data(), b.scratch(), &engine,
                                     &mk, &mt);
    if (s != ZQ4_OK) return s;
    *bytes = plan_bytes_for(engine, jobs, n_jobs, M, b.order.data());
    return ZQ4_OK;
}

namespace {

void fill_plan(zq4_stack_plan *plan, const zq4_stack_job *jobs, const int *order, void *dev, int engine, int n_jobs,
               int M, int grid, int mk, int mt, const ImageInfo &info, int gen)
{
    plan->min_unit = info.min_unit;
    plan->entries = info.entries;
    plan->split_tiles = int(info.split_tiles);
    plan->part_records = int(info.part_records);
    plan->dev = dev;
    plan->bytes = plan_bytes_for(engine, jobs, n_jobs, M, order);
    plan->n_jobs = n_jobs;
    plan->M = M;
    plan->grid = grid;
    plan->max_k = mk;
    plan->max_tiles = mt;
    plan->device = current_device();
    plan->engine = engine;
    plan->tiles = int(info.tiles);
    plan->n_pub = info.n_pub;
    plan->gen = gen;
    plan->wait_ns = kWaitLimitNs;
}

}  // namespace

zq4_status stack_plan_init(const zq4_stack_job *jobs, int n_jobs, int M, void *dev, size_t bytes,
                           zq4_stack_plan *plan, cudaStream_t s)
{
    if (!dev || !plan || !jobs) return ZQ4_ERR_NULL;
    if (n_jobs <= 0) return ZQ4_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(dev) & 255) return ZQ4_ERR_ALIGN;
    const int grid = sm_count();
    SchedBuffers b(n_jobs);
    int engine, mk, mt;
    zq4_status stt = plan_common(jobs, n_jobs, M, grid, b.order.data(), b.dep.data(), b.scratch(), &engine, &mk, &mt);
    if (stt != ZQ4_OK) return stt;
    if (bytes < plan_bytes_for(engine, jobs, n_jobs, M, b.order.data())) return ZQ4_ERR_SHAPE;
    std::vector<uint8_t> host(image_bytes_for(engine, entries_for(engine, jobs, n_jobs, M, b.order.data())));
    ImageInfo info;
    write_image(engine, jobs, n_jobs, M, b.order.data(), b.dep.data(), b.scratch(), grid, host.data(), &info);
    if (!info.ok) return ZQ4_ERR_UNSUPPORTED;
    // the kernel needs every CTA resident at once
    stt = check_resident(engine, info.entries, M, mk, info.n_pub);
    if (stt != ZQ4_OK) return stt;
    stt = upload_plan(dev, host.data(), engine, info, s);
    if (stt != ZQ4_OK) return stt;
    fill_plan(plan, jobs, b.order.data(), dev, engine, n_jobs, M, grid, mk, mt, info, 0);
    return ZQ4_OK;
}

// ---------------------------------------------------------------------------
// A plan without a caller buffer: the library's own fixed-size device array
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticPlanBytes = 64 * 1024;   // header, job table, counters
// ... then the split workspace: counters (at most one per two part records)
// and part records
constexpr size_t kStaticDevBytes = kStaticPlanBytes + (kStepMaxWorkBytes / 32 + 256) + kStepMaxWorkBytes;
constexpr int kStaticMaxJobs = 1257;          // stack engine: 128 + 52 n bytes (rounded to 256) fit
constexpr int kStaticMaxJobsStep = 961;       // step engine: 128 + 68 n bytes (rounded to 256) fit
static_assert(sizeof(st::Job) == 48, "the documented job limit assumes 48-byte job entries");

// The plan lives here when the caller has no device memory to give. Header
// and counters are cleared by every zq4_stack_plan_init_static.
static __device__ __align__(256) uint8_t g_static_plan[kStaticDevBytes];

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

// The generation of the static plan each device holds: every
// zq4_stack_plan_init_static advances it, and a plan struct filled by an
// earlier call no longer runs.
std::atomic<int> g_static_gen[kMaxDevices];

// Host scratch of zq4_stack_plan_init_static: file-scope arrays (not the
// caller's stack, not the heap), one call at a time.
std::mutex g_static_mutex;
uint8_t g_static_image[kStaticPlanBytes];
int g_static_order[kStaticMaxJobs], g_static_dep[kStaticMaxJobs], g_static_nwait[kStaticMaxJobs],
    g_static_first[kStaticMaxJobs];
int g_static_waits[kStaticMaxJobs][kStepMaxWaits];
long long g_static_work[kStaticMaxJobs], g_static_need[kStaticMaxJobs], g_static_at[kStaticMaxJobs];
char g_static_placed[kStaticMaxJobs], g_static_prod[kStaticMaxJobs];
constexpr int kStaticWords = (kStaticMaxJobs + 63) / 64;
uint64_t g_static_anc[size_t(kStaticMaxJobs) * kStaticWords];

}  // namespace

zq4_status stack_plan_init_static(const zq4_stack_job *jobs, int n_jobs, int M, zq4_stack_plan *plan,
                                  cudaStream_t s)
{
    if (!plan || !jobs) return ZQ4_ERR_NULL;
    if (n_jobs <= 0) return ZQ4_ERR_SHAPE;
    if (n_jobs > kStaticMaxJobs) return ZQ4_ERR_UNSUPPORTED;   // more jobs than the static plan holds
    std::lock_guard<std::mutex> lock(g_static_mutex);
    const int words = (n_jobs + 63) / 64;
    const SchedScratch sc = {g_static_work, g_static_need, g_static_at, g_static_placed, g_static_prod, g_static_nwait,
                             g_static_first,
                             g_static_waits, g_static_anc, words};
    const int grid = sm_count();
    int engine, mk, mt;
    zq4_status stt = plan_common(jobs, n_jobs, M, grid, g_static_order, g_static_dep, sc, &engine, &mk, &mt);
    if (stt != ZQ4_OK) return stt;
    auto fits = [&](int eng) {
        return !(step_like(eng) && n_jobs > kStaticMaxJobsStep) &&
               image_bytes_for(eng, entries_for(eng, jobs, n_jobs, M, g_static_order)) <= kStaticPlanBytes &&
               plan_bytes_for(eng, jobs, n_jobs, M, g_static_order) <= kStaticDevBytes;
    };
    // a wide-kernel table (a tensor map per entry) too long for the array: k_stack, up to eight tokens
    if (engine == kEngineWide && !fits(engine) && M <= st::kTokCols && stack_engine_fits(M, mk) == ZQ4_OK)
        engine = kEngineStack;
    if (!fits(engine)) return ZQ4_ERR_UNSUPPORTED;
    ImageInfo info;
    write_image(engine, jobs, n_jobs, M, g_static_order, g_static_dep, sc, grid, g_static_image, &info);
    if (!info.ok) return ZQ4_ERR_UNSUPPORTED;
    stt = check_resident(engine, info.entries, M, mk, info.n_pub);
    if (stt != ZQ4_OK) return stt;
    void *dev = nullptr;
    cudaError_t e = static_plan_address(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) return ZQ4_ERR_CUDA;
    // from pageable memory: the image is staged before the call returns
    stt = upload_plan(dev, g_static_image, engine, info, s);
    if (stt != ZQ4_OK) return stt;
    const int gen = g_static_gen[d].fetch_add(1) + 1;
    fill_plan(plan, jobs, g_static_order, dev, engine, n_jobs, M, grid, mk, mt, info, gen);
    return ZQ4_OK;
}

zq4_status stack_run(const zq4_stack_plan *plan, cudaStream_t s)
{
    if (!plan || !plan->dev) return ZQ4_ERR_NULL;
    const int d = current_device();
    if (d != plan->device || plan->grid != sm_count()) return ZQ4_ERR_SHAPE;   // made on another device
    if (plan->gen != 0) {
        // a static plan: only the latest one of this device is still in the array
        void *p = nullptr;
        if (static_plan_address(&p) != cudaSuccess || p != plan->dev || d < 0 || d >= kMaxDevices ||
            plan->gen != g_static_gen[d].load())
            return ZQ4_ERR_SHAPE;
    }
    if (plan->engine == kEngineStep) return step_run(plan, s);
    if (plan->engine == kEngineWide) return wide_run(plan, s);
    if (plan->engine != kEngineStack) return ZQ4_ERR_SHAPE;
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
    p.wait_ns = plan->wait_ns ? plan->wait_ns : kWaitLimitNs;
    p.x_bufs = st::x_buffers(p.M, p.max_k);
    void *args[] = {&p};
    return cuda_status(cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(st::k_stack), dim3(plan->grid),
                                                   dim3(st::kThreads), args,
                                                   launch_smem(p.n_jobs, p.M, p.max_k), s));
}

cudaError_t read_stack_error(unsigned *flags, bool clear)
{
    unsigned a = 0, b = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&a, g_stack_error, sizeof(unsigned));
    if (e == cudaSuccess) e = read_step_error(&b, clear);
    if (e != cudaSuccess) return e;
    *flags = a | b;
    if (!clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_stack_error, &zero, sizeof(unsigned));
}

}  // namespace zq4
