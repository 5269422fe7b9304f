"""zq4_stack_plan_init_static (the plan in the library's fixed device array,
no allocation) against zq4_stack_plan_init (the plan in a caller buffer):
the same jobs give bit-identical outputs, on two runs in a row of each, and
either order of the two plans. Collected last on purpose; it also passes
alone."""
import numpy as np
import pytest
import torch

from int4_weight_only_q4f16_gb300 import stack as stk
from helpers import host_f16

pytestmark = pytest.mark.gpu

LAYER = (("qkv", 200, 512), ("o", 64, 768), ("gate_up", 512, 512), ("down", 72, 256))
HEAD = ("lm_head", 333, 512)


def _outputs(jobs):
    torch.cuda.synchronize()
    return [host_f16(j[2]).view(np.uint16).copy() for j in jobs]


@pytest.mark.parametrize("M", [1, 4])
def test_static_plan_matches_caller_buffer_plan(M):
    from int4_weight_only_q4f16_gb300 import zq4
    s = stk.DecodeStack(LAYER, 2, HEAD, M=M, mode="calls")
    jobs = []
    for wq, sc, x, y, N, K, gate_up in s.jobs():
        seg, _ = zq4.prepare_weight(wq, sc, N, K, zq4.PREP_SEGMENTED)
        jobs.append((seg, x, y, N, K, gate_up))

    ref_plan = zq4.StackPlan(jobs, M)
    ref_plan.run()
    ref = _outputs(jobs)
    ref_plan.run()
    assert all(np.array_equal(a, b) for a, b in zip(ref, _outputs(jobs)))

    static_plan = zq4.StaticStackPlan(jobs, M)
    for _ in range(2):                        # two calls in a row
        for j in jobs:
            j[2].zero_()
        static_plan.run()
        got = _outputs(jobs)
        for i, (a, b) in enumerate(zip(ref, got)):
            assert np.array_equal(a, b), f"job {i} differs"

    # and the caller-buffer plan still gives the same after the static one ran
    for j in jobs:
        j[2].zero_()
    ref_plan.run()
    assert all(np.array_equal(a, b) for a, b in zip(ref, _outputs(jobs)))
    assert zq4.device_errors(clear=True) == 0


def _jobs(M, count):
    """`count` projections of one matrix on one input, each writing its own
    output (a view into one buffer): no job waits for another."""
    from int4_weight_only_q4f16_gb300 import zq4
    s = stk.DecodeStack((("qkv", 64, 512),), 1, None, M=M, mode="calls")
    wq, sc, x, y, N, K, gu = s.jobs()[0]
    seg, _ = zq4.prepare_weight(wq, sc, N, K, zq4.PREP_SEGMENTED)
    ys = torch.empty((count, M, N), dtype=torch.float16, device="cuda")
    return [(seg, x, ys[i], N, K, gu) for i in range(count)]


@pytest.mark.parametrize("M,limit", [(1, 961), (3, 1257), (12, 333)])
def test_static_plan_rejects_more_jobs_than_it_holds(M, limit):
    """The 64 KiB array holds 961 job entries of the one- and two-token
    kernel (64 bytes each), 1257 of the eight-token kernel (48 bytes each;
    three tokens: a list too long for the wide kernel's table runs there)
    and 333 of the wide kernel (64 bytes and a 128-byte tensor map each)."""
    from int4_weight_only_q4f16_gb300 import zq4
    jobs = _jobs(M, limit + 1)
    with pytest.raises(zq4.Zq4Error, match="UNSUPPORTED"):
        zq4.StaticStackPlan(jobs, M)
    plan = zq4.StaticStackPlan(jobs[:limit], M)     # the documented limit fits
    assert plan.plan.engine == {1: 1, 3: 0, 12: 2}[M]


def test_static_plan_wide_table_falls_back_to_the_eight_token_kernel():
    from int4_weight_only_q4f16_gb300 import zq4
    jobs = _jobs(3, 334)
    assert zq4.StaticStackPlan(jobs[:333], 3).plan.engine == 2
    assert zq4.StaticStackPlan(jobs, 3).plan.engine == 0


def test_static_plan_allocates_no_device_memory():
    """Making and running a static plan leaves the device's allocations as
    they were (after one warm-up plan, so that lazy module loading and the
    context are not counted)."""
    from int4_weight_only_q4f16_gb300 import zq4
    s = stk.DecodeStack(LAYER, 2, HEAD, M=1, mode="calls")
    jobs = []
    for wq, sc, x, y, N, K, gate_up in s.jobs():
        seg, _ = zq4.prepare_weight(wq, sc, N, K, zq4.PREP_SEGMENTED)
        jobs.append((seg, x, y, N, K, gate_up))
    zq4.StaticStackPlan(jobs, 1).run()
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    plan = zq4.StaticStackPlan(jobs, 1)
    plan.run()
    plan.run()
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    assert zq4.device_errors(clear=True) == 0


@pytest.mark.parametrize("M", [1, 3])
def test_an_older_static_plan_no_longer_runs(M):
    """A second zq4_stack_plan_init_static replaces the array's contents: the
    plan struct of the first (here with fewer jobs) is refused by
    zq4_stack_run, and the newest one runs."""
    from int4_weight_only_q4f16_gb300 import zq4
    jobs = _jobs(M, 5)
    old = zq4.StaticStackPlan(jobs[:2], M)
    new = zq4.StaticStackPlan(jobs, M)
    with pytest.raises(zq4.Zq4Error, match="SHAPE"):
        old.run()
    new.run()
    torch.cuda.synchronize()
    assert zq4.device_errors(clear=True) == 0
