// zq4_step.h -- the device plan of the one-launch decode step for one or two
// tokens (zq4_step.cu), shared by its kernel and the host code that builds
// the plan (zq4_stack.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/zq4.h"

namespace zq4 {

constexpr int kStepMaxM = 2;          // tokens the step engine handles
constexpr int kWideMaxM = 16;         // tokens the wide step engine handles (3 ..)
constexpr int kWideGroup16 = 2;       // k_wide above 8 tokens: 16-row tiles per work unit
// 16-row tiles per work unit of the wide step engine at M tokens
inline int wide_group(int M) { return M > 8 ? kWideGroup16 : 1; }
constexpr int kStepWarps = 16;        // compute warps per CTA
constexpr int kStepMaxWaits = 3;      // jobs one job may wait for

// Work units: a 16-row tile of a job whose K is longer than kStepUnitSegs
// segments of 256 columns, and which runs so late that a whole tile would
// outlast the rest of the step, is split along K into C parts of at most
// that many segments (C = ceil(S / kStepUnitSegs), part c = segments
// [c S / C, (c + 1) S / C)). Each part is an entry of its own in the job
// table (its columns of the weights and of x); the parts' fp32 sums meet in
// a workspace and the last part of a tile to finish adds them in part order
// and writes the tile.
constexpr int kStepUnitSegs = 12;
constexpr int kStepMaxSplit = 64;
constexpr size_t kStepMaxWorkBytes = size_t(4) << 20;   // larger: no job is split

// StepJob::flags
constexpr int kStepGateUp = 1;        // interleaved gate/up rows, silu(g) * u output
constexpr int kStepPublish = 2;       // a later job waits for this one: count its finished units
constexpr int kStepWaitShift = 2;     // bits 2..3: number of waits
constexpr int kStepSplitShift = 4;    // bits 4..9: C - 1 (parts of the job)
constexpr int kStepPartShift = 10;    // bits 10..15: c (this entry's part)
constexpr int kStepPubShift = 16;     // bits 16..: index of the job among the waited-for ones
constexpr int kStepMaxPub = 1 << 15;

// Parts per tile of a job with K columns, when it is split.
inline int step_split(int K)
{
    const int S = K / 256;
    return S <= kStepUnitSegs ? 1 : std::min((S + kStepUnitSegs - 1) / kStepUnitSegs, kStepMaxSplit);
}

struct StepHeader {
    unsigned epoch;       // launches completed
    unsigned done;        // CTA arrivals at launch end (monotone)
    unsigned abort;       // set by any wait that gave up
    unsigned next_tile;   // the next tile to hand out (reset by the last CTA of a launch)
    unsigned pad[28];
};

// One entry of the job table: a job in run order, or one part of a split
// job (its parts are consecutive entries, part 0 first). Its tiles are
// [tile0, tile0 + (N + 15) / 16) of the launch's unit sequence; tile t's
// segment s is at seg + (t * tstride + s) * 2304, s < K / 256 (a part's seg,
// x and K are those of its columns; tstride = the whole job's K / 256, also
// the row stride of x in units of 256 columns). Split jobs: tile t counts
// its finished parts in arrive[sbase + t] and keeps part c of token m in
// work[((pbase + c * tiles + t) * M + m) * 16 ...] (16 rows, fp32). The waits
// name the entries of part 0 of the waited-for jobs.
struct alignas(16) StepJob {
    const uint8_t *seg;   // the matrix in the segmented layout
    const uint16_t *x;    // [M][tstride * 256]
    uint16_t *y;          // [M][N] (gate_up: [M][N / 2])
    int N, K, tstride, tile0;
    int flags;
    int sbase, pbase;     // split jobs: first arrival counter, first 16-float part record
    int wait[kStepMaxWaits];   // entries of the jobs to wait for
};
static_assert(sizeof(StepJob) == 64, "step jobs are 64 bytes");

// Device plan: header, job table, per-entry finished-unit counters, for
// k_wide a tensor map per entry (x[M][K] in boxes of [M][256], 128 bytes
// each), then the split workspace: per split tile an arrival counter, and
// the parts' sums.
struct StepLayout {
    size_t hdr, jobs, job_done, tmaps, arrive, work, total;
    StepLayout(int n_entries, long long split_tiles, long long part_records, bool wide = false)
    {
        hdr = 0;
        jobs = 128;
        job_done = jobs + size_t(n_entries) * sizeof(StepJob);
        tmaps = (job_done + size_t(n_entries) * 4 + 127) / 128 * 128;
        arrive = (tmaps + (wide ? size_t(n_entries) * 128 : 0) + 255) / 256 * 256;
        work = (arrive + size_t(split_tiles) * 4 + 255) / 256 * 256;
        total = work + size_t(part_records) * 64;
    }
};

// zq4_step.cu
struct StepShape {
    int slots, wbytes, cached;
    size_t smem;
};
bool step_launch_shape(int M, int max_k, int n_jobs, int n_pub, StepShape *sh);
zq4_status step_check_resident(int M, int max_k, int n_jobs, int n_pub);
zq4_status step_run(const zq4_stack_plan *plan, cudaStream_t s);
zq4_status wide_check_resident(int M, int n_jobs, int n_pub);
zq4_status wide_run(const zq4_stack_plan *plan, cudaStream_t s);
// x[M][K] f16 of an entry (row stride ld elements) as a tensor map of [M][256] boxes
bool wide_x_map(void *map128, const uint16_t *x, int M, int K, long long ld);
cudaError_t read_step_error(unsigned *flags, bool clear);

}  // namespace zq4
