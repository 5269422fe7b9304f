"""The run order and waits of the one-launch decode step
(zq4_stack_plan_waits), on plain addresses: host logic only, no device call
(nothing is read at the addresses). Hand-derived cases, plus a check on
seeded random job lists that conflicting jobs (touching the same bytes, one
of them writing) keep their order and that every job waits for the last
conflicting job run before it."""
import numpy as np
import pytest

W = 1 << 44                      # a weight address (only compared)


def buf(i, off=0):
    """Address of buffer i (buffers 4 GiB apart) plus a byte offset."""
    return (i + 1) << 32 | off


@pytest.fixture(scope="module")
def zq4():
    from int4_weight_only_q4f16_gb300 import build
    build.build()
    from int4_weight_only_q4f16_gb300 import zq4 as z
    return z


def spans(job, M):
    _, x, y, N, K, gu = job
    return (x, x + M * K * 2), (y, y + M * (N // 2 if gu else N) * 2)


def meets(a, b):
    return a[0] < b[1] and b[0] < a[1]


def conflict(a, b, M):
    (xa, ya), (xb, yb) = spans(a, M), spans(b, M)
    return meets(ya, xb) or meets(ya, yb) or meets(xa, yb)


def check_valid(jobs, M, order, dep):
    n = len(jobs)
    assert sorted(order) == list(range(n))
    pos = {j: r for r, j in enumerate(order)}
    for j in range(n):
        for i in range(j):
            if conflict(jobs[i], jobs[j], M):
                assert pos[i] < pos[j], f"jobs {i} and {j} conflict but run out of order"
        before = sorted((pos[i], i) for i in range(n) if pos[i] < pos[j] and conflict(jobs[i], jobs[j], M))
        assert dep[j] == (before[-1][1] if before else -1), j


def test_mixed_job_list(zq4):
    M = 2
    jobs = [
        (W, buf(0), buf(1), 768, 512, 0),         # 0 touches nothing earlier
        (W, buf(1), buf(2), 1024, 768, 1),        # 1 x == y0: waits for 0
        (W, buf(2), buf(3), 256, 512, 0),         # 2 x == y1 (gate_up output)
        (W, buf(1, 512), buf(4), 256, 512, 0),    # 3 x inside y0 at an offset: whole job 0
        (W, buf(5), buf(1), 768, 256, 0),         # 4 y over y0 / x1 / x3: whole job 3
        (W, buf(1), buf(6), 512, 768, 0),         # 5 x == y4 (and y0, older)
        (W, buf(6), buf(2), 512, 512, 0),         # 6 x == y5; y over y1 / x2
        (W, buf(7), buf(6), 256, 512, 0),         # 7 y over y5 / x6
    ]
    order, dep = zq4.stack_plan_waits(jobs, M)
    # every job here is small next to the room a waited-for job gets (its own
    # work and 2 x 152 x 16 of its tiles' segments), so each wait is on a
    # recent job for every job after it; the only job free of the jobs still
    # to place (3) itself waits for job 0: nothing moves forward
    assert order == list(range(8))
    assert dep == [-1, 0, 1, 0, 3, 4, 5, 6]
    check_valid(jobs, M, order, dep)


def test_an_independent_job_passes_a_waiting_one(zq4):
    # job 1 reads job 0's output; jobs 2 and 3 touch no other job: the
    # largest of those (3) runs last, the other runs between 0 and 1
    jobs = [(W, buf(0), buf(1), 16384, 3072, 0), (W, buf(1), buf(2), 3072, 16384, 0),
            (W, buf(3), buf(4), 3072, 3072, 0), (W, buf(5), buf(6), 32064, 3072, 0)]
    for M in (1, 2):
        assert zq4.stack_plan_waits(jobs, M) == ([0, 2, 1, 3], [-1, 0, -1, -1])


def test_decode_layers_run_down_after_the_next_layers_projections(zq4):
    # qkv, o and gate_up on fresh inputs, down on gate_up's output; a head
    jobs = []
    for l in range(3):
        b = 10 * l
        jobs += [(W, buf(b), buf(b + 1), 9216, 3072, 0), (W, buf(b + 2), buf(b + 3), 3072, 3072, 0),
                 (W, buf(b + 4), buf(b + 5), 16384, 3072, 1), (W, buf(b + 5), buf(b + 6), 3072, 8192, 0)]
    jobs.append((W, buf(99), buf(98), 32064, 3072, 0))
    order, dep = zq4.stack_plan_waits(jobs, 1)
    # down of layer l waits for its gate_up. A job some later job waits for
    # (each gate_up) goes before up to 12 independent jobs ahead of it, so
    # the three gate_ups run first; each down is put after at least
    # 2 x 152 x 16 tiles' worth of its gate_up's segments (58,368) where
    # there is that much work. The head, which touches no other job's bytes
    # and is the largest such job, runs last
    assert order == [2, 6, 10, 0, 1, 4, 5, 8, 9, 3, 7, 11, 12]
    assert dep == [-1, -1, -1, 2, -1, -1, -1, 6, -1, -1, -1, 10, -1]
    check_valid(jobs, 1, order, dep)


def test_a_chain_keeps_its_order(zq4):
    # every job reads the one before: nothing may move
    jobs = [(W, buf(i), buf(i + 1), 256, 256, 0) for i in range(6)]
    order, dep = zq4.stack_plan_waits(jobs, 3)
    assert order == list(range(6))
    assert dep == [-1, 0, 1, 2, 3, 4]


def test_exact_address_but_other_stride_waits_for_the_whole_job(zq4):
    # y0 is [M, 512]; x1 starts at y0 but is read as [M, 256] rows
    jobs = [(W, buf(0), buf(1), 512, 256, 0), (W, buf(1), buf(2), 64, 256, 0)]
    for M in (1, 2):
        assert zq4.stack_plan_waits(jobs, M) == ([0, 1], [-1, 0])


def test_exact_input_but_output_over_the_previous_input(zq4):
    # x1 == y0, but y1 overwrites x0: job 1 waits for all of job 0
    jobs = [(W, buf(0), buf(1), 256, 256, 0), (W, buf(1), buf(0), 256, 256, 0)]
    assert zq4.stack_plan_waits(jobs, 1) == ([0, 1], [-1, 0])


def test_meeting_depends_on_M(zq4):
    # x1 starts 1024 bytes after y0: y0 spans M * 256 * 2 bytes
    jobs = [(W, buf(0), buf(1), 256, 256, 0), (W, buf(1, 1024), buf(2), 64, 256, 0)]
    assert zq4.stack_plan_waits(jobs, 2) == ([0, 1], [-1, -1])      # y0 ends at 1024
    assert zq4.stack_plan_waits(jobs, 3) == ([0, 1], [-1, 0])       # y0 ends at 1536


def test_reads_of_the_same_buffer_do_not_order(zq4):
    jobs = [(W, buf(0), buf(1), 256, 256, 0), (W, buf(0), buf(2), 256, 256, 0), (W, buf(0), buf(3), 256, 256, 0)]
    assert zq4.stack_plan_waits(jobs, 4) == ([0, 1, 2], [-1] * 3)


def _random_jobs(seed):
    rng = np.random.default_rng(seed)
    M = int(rng.integers(1, 5))
    jobs = []
    for _ in range(40):
        K = 256 * int(rng.integers(1, 4))
        gu = int(rng.integers(0, 2))
        N = 2 * 16 * int(rng.integers(1, 40))
        xb, yb = int(rng.integers(0, 10)), int(rng.integers(0, 10))
        xo = 16 * int(rng.integers(0, 3)) * (1 if rng.random() < 0.3 else 0)
        if jobs and rng.random() < 0.4:         # read the previous output exactly
            p = jobs[-1]
            xb_addr, K = p[2], (p[3] // 2 if p[5] else p[3])
            if K % 256:
                K = 256
                xb_addr = buf(xb, xo)
        else:
            xb_addr = buf(xb, xo)
        jobs.append((W, xb_addr, buf(yb), N, K, gu))
    return jobs, M


@pytest.mark.parametrize("seed", range(6))
def test_random_job_lists_keep_conflicting_jobs_in_order(zq4, seed):
    jobs, M = _random_jobs(seed)
    order, dep = zq4.stack_plan_waits(jobs, M)
    check_valid(jobs, M, order, dep)


def test_concurrent_calls_from_host_threads_agree_with_sequential_ones(zq4):
    """The scheduler runs on the host in caller-owned scratch: calls from
    several threads at once (ctypes releases the GIL) give what one thread
    gets, and a rejected call on one thread leaves the others unaffected."""
    from concurrent.futures import ThreadPoolExecutor
    cases = [_random_jobs(seed) for seed in range(8)]
    want = [zq4.stack_plan_waits(jobs, M) for jobs, M in cases]

    def work(i):
        jobs, M = cases[i % len(cases)]
        if i % 5 == 4:
            with pytest.raises(zq4.Zq4Error, match="ALIGN"):
                zq4.stack_plan_waits([(W, buf(0, 8), buf(1), 256, 256, 0)], 1)
        return i, zq4.stack_plan_waits(jobs, M)

    with ThreadPoolExecutor(max_workers=8) as ex:
        for i, got in ex.map(work, range(200)):
            assert got == want[i % len(cases)], i


def test_waits_reject_bad_jobs(zq4):
    with pytest.raises(zq4.Zq4Error, match="SHAPE"):
        zq4.stack_plan_waits([(W, buf(0), buf(1), 256, 100, 0)], 1)
    with pytest.raises(zq4.Zq4Error, match="ALIGN"):
        zq4.stack_plan_waits([(W, buf(0, 8), buf(1), 256, 256, 0)], 1)
