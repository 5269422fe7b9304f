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
//    and may wait on one another), 16 warps each. Work unit = a segment, 16
//    weight rows x 256 columns.
//  * The weights are in the segmented layout (zq4_prepare_weight,
//    ZQ4_PREP_SEGMENTED): each segment is 2304 contiguous bytes (swizzled
//    codes, then scales), so one bulk copy fills a shared-memory slot and no
//    tensor map is involved. Each warp runs its own ring of segment slots
//    across job boundaries, with a look-ahead of L2 prefetches. Per 32-column
//    group, lane (r, t) (r = lane/4, t = lane%4) takes word t of rows r and
//    r+8 (ldmatrix.x4 fetches two groups, conflict-free on the swizzle),
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
//    barrier, then x of the next job is staged into shared memory (L2 reads:
//    it may have been written by other SMs during this kernel).
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

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 4;
constexpr int kPrefetch = 8;
using namespace segk;   // segment layout, inner loop, split-tile sums

struct Header {
    unsigned epoch;     // launches completed
    unsigned done;      // CTA arrivals at launch end (monotone)
    unsigned abort;     // set by any wait that gave up
    unsigned pad[29];
};

struct alignas(16) Job {
    const uint8_t *seg; // the matrix in the segmented layout
    const uint16_t *x;  // [M][K]
    uint16_t *y;        // [M][y_stride]
    int N, K, T, S;
    int gate_up, y_stride;
};

struct Params {
    Header *hdr;
    const Job *jobs;
    unsigned *job_cnt;   // [n_jobs]
    int n_jobs, M, max_k;
};

constexpr size_t kRingOff = 0;
constexpr size_t kBarOff = kRingOff + size_t(kWarps) * kSlots * kSegBytes;
constexpr size_t kMiscOff = kBarOff + size_t(kWarps) * kSlots * 8;
constexpr size_t kParkOff = kMiscOff + 128;                          // warp partials [kWarps*2][16][kTokCols]
constexpr size_t kTabOff = kParkOff + size_t(kWarps) * 2 * 16 * kTokCols * 4;   // warp range table [2][kWarps + 1]
constexpr size_t kXsOff = kTabOff + 2 * 4 * (kWarps + 1 + 15) / 16 * 16;
__host__ __device__ inline size_t smem_bytes(int M, int max_k) { return 1024 + kXsOff + size_t(M) * xs_row_bytes(max_k); }

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p)
{
    unsigned r;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(r) : "l"(p) : "memory");
    return r;
}

// Position in one warp's sequence of (job, segment) pairs.
struct SegIt {
    int j, u, e;
};

__global__ void __launch_bounds__(kThreads, 1) k_stack(Params p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_addr(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, t = lane & 3;
    const int G = gridDim.x, cta = blockIdx.x;
    const uint32_t ring0 = sbase + uint32_t(kRingOff) + uint32_t(warp * kSlots * kSegBytes);
    const uint32_t bar0 = sbase + uint32_t(kBarOff) + uint32_t(warp * kSlots * 8);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + kMiscOff);
    float *wpark = reinterpret_cast<float *>(smem + kParkOff);
    int *wtab = reinterpret_cast<int *>(smem + kTabOff);
    uint8_t *xs = smem + kXsOff;
    const uint32_t xrow = uint32_t(xs_row_bytes(p.max_k));
    const int n = p.n_jobs;
    const unsigned launch = *reinterpret_cast<volatile unsigned *>(&p.hdr->epoch);
    const unsigned target = (launch + 1u) * unsigned(G);

    if (threadIdx.x == 0) *s_abort = 0;
    if (lane == 0) {
        for (int j = 0; j < kSlots; ++j) mbar_init(bar0 + 8 * j, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();

    // this warp's segment range of a job: CTA part of the job, then warp part
    // (CTA ranges are whole tiles, so a tile never spans two CTAs)
    auto warp_range = [&](int T, int S, int &ub, int &ue) {
        int tb, te;
        split(0, T, cta, G, tb, te);
        split(tb * S, te * S, warp, kWarps, ub, ue);
    };
    auto seek = [&](SegIt &it, int j) {
        for (; j < n; ++j) {
            const Job &jb = p.jobs[j];
            int ub, ue;
            warp_range(jb.T, jb.S, ub, ue);
            if (ub < ue) {
                it.j = j;
                it.u = ub;
                it.e = ue;
                return;
            }
        }
        it.j = n;
    };
    auto next = [&](SegIt &it) {
        if (++it.u >= it.e) seek(it, it.j + 1);
    };
    // segment u of a job (tile-major) is at byte u * kSegBytes of its matrix
    auto issue = [&](const SegIt &it, int slot) {       // lane 0
        const uint32_t bar = bar0 + 8 * slot;
        mbar_arrive_expect_tx(bar, kSegBytes);
        bulk_load(ring0 + slot * kSegBytes, p.jobs[it.j].seg + size_t(it.u) * kSegBytes, kSegBytes, bar);
    };
    auto prefetch = [&](const SegIt &it) {              // lane 0
        prefetch_l2_bulk(p.jobs[it.j].seg + size_t(it.u) * kSegBytes, kSegBytes);
    };

    // ---- first copies of this warp's sequence, and the L2 look-ahead
    SegIt iss, pf;
    seek(iss, 0);
    if (lane == 0) {
        for (int q = 0; q < kSlots && iss.j < n; ++q, next(iss)) issue(iss, q);
        pf = iss;
        for (int q = 0; q < kPrefetch && pf.j < n; ++q, next(pf)) prefetch(pf);
    }

    uint32_t ldm_off[4];
    ldm_offsets(lane, ldm_off);
    const uint8_t *xr = xs + size_t(min(r, p.M - 1)) * xrow + 16 * t;

    bool ok = true;
    int consumed = 0;
    for (int j = 0; j < n; ++j) {
        const Job &jb = p.jobs[j];
        // ---- wait until every CTA has finished job j-1, then stage x_j
        if (j > 0) {
            __syncthreads();
            if (!*s_abort) {
                const Job &pj = p.jobs[j - 1];
                int ptb, pte;
                split(0, pj.T, cta, G, ptb, pte);
                finalize_split<kWarps, kThreads>(ptb, pte, pj.S, pj.gate_up, p.M, pj.N, pj.y_stride, pj.y, wpark, wtab);
            }
            __syncthreads();
            if (threadIdx.x == 0 && !*s_abort) {
                // release: this CTA's outputs of job j-1 (ordered before by
                // the barrier) become visible with the increment
                asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&p.job_cnt[j - 1]) : "memory");
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
            __syncthreads();
            if (*s_abort) {
                ok = false;
                break;
            }
        }
        {
            // this job's warp range boundaries and each warp's first tile
            if (threadIdx.x <= kWarps) {
                int tb0, te0;
                split(0, jb.T, cta, G, tb0, te0);
                const int b = part_begin(tb0 * jb.S, te0 * jb.S, threadIdx.x, kWarps);
                wtab[threadIdx.x] = b;
                wtab[kWarps + 1 + threadIdx.x] = b / jb.S;
            }
            stage_x<2>(xs, xrow, jb.x, p.M, jb.K, threadIdx.x, kThreads);
        }
        __syncthreads();

        const int S = jb.S, gate_up = jb.gate_up;
        int tb, te, ub, ue;
        split(0, jb.T, cta, G, tb, te);
        const int cb = tb * S, ce = te * S;
        split(cb, ce, warp, kWarps, ub, ue);
        const int first_tile = ub / S;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        int cur_tile = -1;

        auto flush = [&](int tt) {
            if (tt * S >= ub && (tt + 1) * S <= ue)
                write_tile(acc, tt * 16, lane, gate_up, p.M, jb.N, jb.y_stride, jb.y);
            else        // part of a tile shared with other warps: summed at job end
                park(acc, wpark, warp, tt == first_tile ? 0 : 1, lane);
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = 0.f;
        };

        for (int u = ub; u < ue; ++u, ++consumed) {
            const int slot = consumed % kSlots;
            if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * slot, (consumed / kSlots) & 1))) {
                ok = false;
                break;
            }
            const int tt = u / S, seg = u - tt * S;
            if (tt != cur_tile) {
                if (cur_tile >= 0) flush(cur_tile);
                cur_tile = tt;
            }
            accumulate(ring0 + slot * kSegBytes, ldm_off, xr + seg * 32 * 16, r, acc);
            __syncwarp();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (lane == 0 && iss.j < n) {
                issue(iss, slot);
                next(iss);
                if (pf.j < n) {
                    prefetch(pf);
                    next(pf);
                }
            }
        }
        if (!ok) {
            // leave together at the next job boundary: every warp must still
            // take part in the CTA barriers there
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
    __syncthreads();
    if (threadIdx.x == 0 && *s_abort) atomicOr(&g_stack_error, ZQ4_DEVERR_WAIT_TIMEOUT);
    if (!*s_abort && n > 0) {                            // the last job's split tiles
        const Job &lj = p.jobs[n - 1];
        int ltb, lte;
        split(0, lj.T, cta, G, ltb, lte);
        st::finalize_split<st::kWarps, st::kThreads>(ltb, lte, lj.S, lj.gate_up, p.M, lj.N, lj.y_stride, lj.y, wpark, wtab);
    }
    // let every copy this warp issued land before the CTA exits
    {
        int outstanding = 0;
        if (lane == 0) {
            // copies issued = min(kSlots, total) initially + one per consumed segment while any remained
            SegIt probe;
            seek(probe, 0);
            int total = 0;
            for (; probe.j < n; next(probe)) ++total;
            outstanding = std::min(total, consumed + kSlots) - consumed;
        }
        outstanding = __shfl_sync(0xffffffffu, outstanding, 0);
        for (int c = consumed; c < consumed + outstanding; ++c)
            if (!mbar_wait(bar0 + 8 * (c % kSlots), (c / kSlots) & 1)) break;
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
    const size_t smem = st::smem_bytes(M, mk);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(st::k_stack), smem, stack_smem_set);
    if (e != cudaSuccess) return cuda_status(e);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, st::k_stack, st::kThreads, smem);
    if (e != cudaSuccess) return cuda_status(e);
    if (per_sm < 1) return ZQ4_ERR_UNSUPPORTED;

    std::vector<uint8_t> host(l.total, 0);
    uint8_t *hjobs = host.data() + l.jobs;
    for (int j = 0; j < n_jobs; ++j) {
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
        jb.gate_up = b.gate_up ? 1 : 0;
        jb.y_stride = b.gate_up ? b.N / 2 : b.N;
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
    void *args[] = {&p};
    return cuda_status(cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(st::k_stack), dim3(plan->grid),
                                                   dim3(st::kThreads), args, st::smem_bytes(p.M, p.max_k), s));
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
    const size_t smem = st::smem_bytes(M, mk);
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
        jb.gate_up = b.gate_up ? 1 : 0;
        jb.y_stride = b.gate_up ? b.N / 2 : b.N;
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
