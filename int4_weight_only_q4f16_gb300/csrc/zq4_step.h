// zq4_step.h -- the device plan of the one-launch decode step for one or two
// tokens (zq4_step.cu), shared by its kernel and the host code that builds
// the plan (zq4_stack.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/zq4.h"

namespace zq4 {

constexpr int kStepMaxM = 2;          // tokens the step engine handles
constexpr int kStepWarps = 16;        // compute warps per CTA
constexpr int kStepMaxWaits = 3;      // jobs one job may wait for

// StepJob::flags
constexpr int kStepGateUp = 1;        // interleaved gate/up rows, silu(g) * u output
constexpr int kStepPublish = 2;       // a later job waits for this one: count its finished tiles
constexpr int kStepPubShift = 8;      // bits 8..: index of the job among the waited-for ones

struct StepHeader {
    unsigned epoch;       // launches completed
    unsigned done;        // CTA arrivals at launch end (monotone)
    unsigned abort;       // set by any wait that gave up
    unsigned next_tile;   // the next tile to hand out (reset by the last CTA of a launch)
    unsigned pad[28];
};

// One job in run order. Its tiles are [tile0, tile0 + T) of the launch's tile
// sequence; tile t's segment s is at seg + (t * (K / 256) + s) * 2304.
struct alignas(16) StepJob {
    const uint8_t *seg;   // the matrix in the segmented layout
    const uint16_t *x;    // [M][K]
    uint16_t *y;          // [M][y_stride]
    int N, K, T, tile0;
    int flags;
    int y_stride;         // N, or N / 2 for gate_up
    int nwait;
    int wait[kStepMaxWaits];   // positions (in run order) of the jobs to wait for
};
static_assert(sizeof(StepJob) == 64, "step jobs are 64 bytes");

// Device plan: header, job table, per-job finished-tile counters.
struct StepLayout {
    size_t hdr, jobs, job_done, total;
    explicit StepLayout(int n_jobs)
    {
        hdr = 0;
        jobs = 128;
        job_done = jobs + size_t(n_jobs) * sizeof(StepJob);
        total = (job_done + size_t(n_jobs) * 4 + 255) / 256 * 256;
    }
};

// zq4_step.cu
struct StepShape {
    int slots, wbytes, cached;
    size_t smem;
};
size_t step_plan_layout_bytes(int n_jobs);
bool step_launch_shape(int M, int max_k, int n_jobs, int n_pub, StepShape *sh);
zq4_status step_check_resident(int M, int max_k, int n_jobs, int n_pub);
zq4_status step_run(const zq4_stack_plan *plan, cudaStream_t s);
cudaError_t read_step_error(unsigned *flags, bool clear);

}  // namespace zq4
