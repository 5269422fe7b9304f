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


def test_static_plan_rejects_more_jobs_than_it_holds():
    from int4_weight_only_q4f16_gb300 import zq4
    s = stk.DecodeStack((("qkv", 64, 512),), 1, None, M=1, mode="calls")
    wq, sc, x, y, N, K, gu = s.jobs()[0]
    seg, _ = zq4.prepare_weight(wq, sc, N, K, zq4.PREP_SEGMENTED)
    with pytest.raises(zq4.Zq4Error, match="UNSUPPORTED"):
        zq4.StaticStackPlan([(seg, x, y, N, K, gu)] * 1258, 1)
    zq4.StaticStackPlan([(seg, x, y, N, K, gu)] * 1257, 1)     # the documented limit fits
