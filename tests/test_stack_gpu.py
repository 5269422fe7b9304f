"""GPU parity of the one-launch decode step (zq4_stack_run) against the CPU
oracle.

Every job's output is compared with the oracle on the same inputs the GPU
job read: the seeded activations for the independent projections and, for
the down projection, the GPU's own f16 gate_up output (each chained stage
is checked on its own input). Also: repeated runs and CUDA-graph replays are
bit-identical (the plan's counters advance across launches), and the full
Phi-3-mini-shaped 32-layer step, exactly as the benchmark runs it, matches
on sampled rows of every fourth layer and of the LM head."""
import numpy as np
import pytest
import torch

from int4_weight_only_q4f16_gb300 import synth
from int4_weight_only_q4f16_gb300 import stack as stk
from helpers import assert_within, dev, host_f16

pytestmark = pytest.mark.gpu

SMALL_LAYER = (("qkv", 200, 512), ("o", 64, 768), ("gate_up", 512, 512), ("down", 72, 256))
SMALL_HEAD = ("lm_head", 333, 512)


def _check_job(oracle, job, what, rows=None):
    wq, sc, x, y, N, K, gate_up = job
    wq_h = wq.cpu().numpy().view(np.uint32)
    sc_h = sc.cpu().numpy().view(np.float16)
    x_h = host_f16(x)
    y_h = host_f16(y)
    if gate_up:
        if rows is None:
            js = np.arange(N // 2)
        else:
            js = np.unique(np.clip(rows // 2, 0, N // 2 - 1))
        r2 = np.stack([2 * js, 2 * js + 1], 1).ravel()
        h_ref, Sh = oracle.gate_up_silu(wq_h[r2], sc_h[r2], x_h, len(r2), K, interleaved=True)
        assert_within(y_h[:, js], h_ref, Sh, what)
    else:
        y_ref, S = oracle.gemv(wq_h, sc_h, x_h, N, K, rows=rows)
        assert_within(y_h if rows is None else y_h[:, rows], y_ref, S, what)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
def test_small_stack_matches_oracle(oracle, M):
    """Three runs of one plan, each checked: the plan runs the three down
    projections last, after a run of small jobs most SMs have no tile of (a
    CTA with nothing to do in them reaches the dependent jobs early; their
    inputs must still be the finished gate_up outputs)."""
    s = stk.DecodeStack(SMALL_LAYER, 3, SMALL_HEAD, M=M, mode="plan")
    names = [n for n, _, _ in SMALL_LAYER]
    for run in range(3):
        for j in s.jobs():
            j[3].fill_(float("nan"))
        s.launch_step()
        torch.cuda.synchronize()
        for i, job in enumerate(s.jobs()):
            l, name = divmod(i, len(names))
            what = f"M={M} run {run} job {i} " + ("lm_head" if l == 3 else f"layer {l} {names[name]}")
            _check_job(oracle, job, what)


@pytest.mark.parametrize("M", [1, 2, 5, 8, 16])
def test_step_engine_split_tiles_match_oracle(oracle, M):
    """Tiles of long-K jobs split along K (K = 9728: 4 parts of 9, 10, 9, 10
    segments; 3328: 6 + 7; 4096 and 4608: 8 + 8 and 9 + 9), a split gate_up
    and a split job that waits for it included: every part's sums meet in
    the plan's workspace and the last part adds them in part order, so three
    runs (counters advancing across launches) give the same bits, each
    matching the oracle."""
    from int4_weight_only_q4f16_gb300 import zq4
    rng = synth.rng_for("step_split", M)
    spec = [(200, 9728, False), (72, 3328, False), (9216, 4096, True)] + [(256, 3072, False)] * 6 + \
        [(88, 4608, False), (333, 3072, False)]
    jobs, mats = [], []
    for i, (N, K, gu) in enumerate(spec):
        wq_h, sc_h = synth.weight("step_split_w", N, K, i)
        seg = zq4.prepare_weight(dev(wq_h), dev(sc_h), N, K, zq4.PREP_SEGMENTED)[0]
        x = jobs[2][2] if i == 9 else dev(synth.activations(rng, M, K))      # job 9 reads job 2's output
        y = torch.full((M, N // 2 if gu else N), float("nan"), dtype=torch.float16, device="cuda")
        jobs.append((seg, x, y, N, K, gu))
        mats.append((wq_h, sc_h))
    plan = zq4.StackPlan(jobs, M)
    assert plan.plan.engine == (1 if M <= 2 else 2) and plan.plan.split_tiles > 0
    first = None
    for run in range(3):
        for j in jobs:
            j[2].fill_(float("nan"))
        plan.run()
        torch.cuda.synchronize()
        assert zq4.device_errors(clear=True) == 0
        bits = [host_f16(j[2]).view(np.uint16).copy() for j in jobs]
        if first is None:
            first = bits
            for i, ((seg, x, y, N, K, gu), (wq_h, sc_h)) in enumerate(zip(jobs, mats)):
                _check_job(oracle, (dev(wq_h), dev(sc_h), x, y, N, K, gu), f"M={M} split job {i}")
        else:
            for i, (a, b) in enumerate(zip(first, bits)):
                assert np.array_equal(a, b), f"M={M} run {run} job {i} differs from run 0"


CHAIN_LAYER = (("qkv", 768, 256), ("o", 256, 512), ("gate_up", 1024, 256), ("down", 256, 512))
CHAIN_HEAD = ("lm_head", 333, 256)


@pytest.mark.parametrize("M", [1, 3])
def test_chained_stack_matches_oracle(oracle, M):
    """Every projection reads the previous one's output (o a view over
    qkv's): each job waits for the one before, and matches
    the oracle on the values its x holds after the step (each buffer is
    written once)."""
    from int4_weight_only_q4f16_gb300 import zq4
    s = stk.DecodeStack(CHAIN_LAYER, 3, CHAIN_HEAD, M=M, mode="plan", chain=True)
    s.launch_step()
    torch.cuda.synchronize()
    assert zq4.device_errors(clear=True) == 0
    jobs = s.jobs()
    _, dep = zq4.stack_plan_waits([(j[0].data_ptr(), j[2].data_ptr(), j[3].data_ptr(), j[4], j[5], j[6])
                                   for j in jobs], M)
    assert dep[1:5] == [0, 1, 2, 3]
    names = [n for n, _, _ in CHAIN_LAYER]
    for i, job in enumerate(jobs):
        l, name = divmod(i, len(names))
        _check_job(oracle, job, f"M={M} job {i} " + ("lm_head" if l == 3 else f"layer {l} {names[name]}"))


def test_stack_runs_and_graph_replays_are_bit_identical():
    s = stk.DecodeStack(SMALL_LAYER, 3, SMALL_HEAD, M=2, mode="plan")
    strm = torch.cuda.Stream()
    with torch.cuda.stream(strm):
        s.launch_step(strm)
    torch.cuda.synchronize()
    ref = [host_f16(j[3]).view(np.uint16).copy() for j in s.jobs()]
    with torch.cuda.stream(strm):
        s.launch_step(strm)
    torch.cuda.synchronize()
    for a, j in zip(ref, s.jobs()):
        assert np.array_equal(a, host_f16(j[3]).view(np.uint16))
    g = s.capture(strm)
    for _ in range(3):
        for j in s.jobs():
            j[3].zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, j in zip(ref, s.jobs()):
            assert np.array_equal(a, host_f16(j[3]).view(np.uint16))


def test_stack_plan_rejects_bad_jobs():
    from int4_weight_only_q4f16_gb300 import zq4
    s = stk.DecodeStack((("qkv", 64, 512),), 1, None, M=1, mode="calls")
    wq, sc, x, y, N, K, gu = s.jobs()[0]
    seg, _ = zq4.prepare_weight(wq, sc, N, K, zq4.PREP_SEGMENTED)
    x9 = torch.zeros((17, K), dtype=torch.float16, device="cuda")
    y9 = torch.empty((17, N), dtype=torch.float16, device="cuda")
    with pytest.raises(zq4.Zq4Error, match="SHAPE"):
        zq4.StackPlan([(seg, x9, y9, N, K, gu)], 17)                   # M > 16
    with pytest.raises(zq4.Zq4Error, match="SHAPE"):
        zq4.StackPlan([(seg, x, y, N, 480, gu)], 1)                    # K % 256 != 0
    with pytest.raises(zq4.Zq4Error, match="FLAGS"):
        zq4.prepare_weight(wq, sc, N, K, 4)                            # unknown flag


def test_phi3_full_step_sampled(oracle):
    s = stk.phi3_stack(mode="plan")
    strm = torch.cuda.Stream()
    with torch.cuda.stream(strm):
        s.launch_step(strm)
        s.launch_step(strm)            # the second run is the one checked
    torch.cuda.synchronize()
    jobs = s.jobs()
    per_layer = len(synth.PHI3_LAYER)
    rng = np.random.default_rng(5)
    for l in range(0, synth.PHI3_LAYERS, 4):
        for i, (name, N, K) in enumerate(synth.PHI3_LAYER):
            job = jobs[l * per_layer + i]
            rows = np.unique(np.concatenate([t * 16 + rng.integers(0, 16, 1) for t in range(0, N // 16, 3)]
                                            + [[0, N - 1]]))
            _check_job(oracle, job, f"phi3 layer {l} {name}", rows=rows)
    head = jobs[-1]
    N = head[4]
    rows = np.unique(np.concatenate([np.arange(0, N, 7), [N - 1]]))
    _check_job(oracle, head, "phi3 lm_head", rows=rows)


def test_stack_no_device_errors():
    from int4_weight_only_q4f16_gb300 import zq4
    assert zq4.device_errors(clear=True) == 0


def _plan_outputs(jobs, M):
    """Run `jobs` [(wq, sc, x, N, K, gate_up)] as one plan on segmented
    copies; returns the host f16 outputs."""
    from int4_weight_only_q4f16_gb300 import zq4
    pj, ys = [], []
    for wq, sc, x, N, K, gate_up in jobs:
        seg, _ = zq4.prepare_weight(wq, sc, N, K, zq4.PREP_SEGMENTED)
        y = torch.full((M, N // 2 if gate_up else N), float("nan"), dtype=torch.float16, device="cuda")
        pj.append((seg, x, y, N, K, gate_up))
        ys.append(y)
    zq4.StackPlan(pj, M).run()
    torch.cuda.synchronize()
    assert zq4.device_errors(clear=True) == 0
    return [host_f16(y) for y in ys]


@pytest.mark.parametrize("K", [256, 3072, 8192])
def test_stack_all_zero_point_codes_give_exact_zero(K):
    """Codes all 7 make every weight exactly 0 (S = 0): the one-launch step,
    tiles split between warps included, must give exactly 0 for large
    activations too, in both epilogues."""
    M, N = 3, 400
    rng = synth.rng_for("stack_zp7", K)
    x = dev((rng.standard_normal((M, K)) * 300).astype(np.float16))
    wq = dev(np.full((N, K // 8), 0x77777777, np.uint32))
    sc = dev(synth.group_scales(rng, N, K))
    y, h = _plan_outputs([(wq, sc, x, N, K, False), (wq, sc, x, N, K, True)], M)
    assert np.all(y == 0) and np.all(h == 0)


def test_stack_one_hot_bit_exact(oracle):
    """x = e_k returns f16(w[:, k]) exactly through the one-launch step
    (one non-zero product per output, whichever warp or split tile holds it)."""
    N, K = 640, 3072
    wq_h, sc_h = synth.weight("stack_onehot", N, K, 0)
    w = oracle.dequant(wq_h, sc_h, N, K)
    ks = (0, 1, 7, 8, 255, 256, 1029, 3071)
    xs = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        xs[i, k] = 1.0
    wq, sc = dev(wq_h), dev(sc_h)
    jobs = [(wq, sc, dev(xs[i:i + 1]), N, K, False) for i in range(len(ks))]
    outs = _plan_outputs(jobs, 1)
    for i, k in enumerate(ks):
        want = oracle.round_f16(w[:, k])
        assert np.array_equal(outs[i][0].view(np.uint16), want.view(np.uint16)), k


@pytest.mark.parametrize("M", [1, 3])
def test_stack_orders_jobs_that_share_buffers(oracle, M):
    """Jobs that read an earlier output, exactly or through an offset view,
    and that write over an earlier job's input
    or output (the plan may also run them in another order where they do not
    conflict): the final buffers equal a sequential host replay of the jobs
    in the given order with the oracle, each job on the f16 values its x
    holds at its turn.
    Buffers start as NaN, so a read before its write shows as NaN. The bound
    is wider than one job's (2^-6 S): the replay's inputs are the oracle's
    f16 outputs, the GPU's its own; a read out of order is off by O(S)."""
    from int4_weight_only_q4f16_gb300 import zq4
    width = 1024
    pool = torch.full((8, M * width), float("nan"), dtype=torch.float16, device="cuda")
    host = np.full((8, M * width), np.nan, np.float64)
    for b in (0, 5, 7):                                   # fresh inputs
        a = synth.activations(synth.rng_for("stack_order_x", b, M), M, width).ravel()
        pool[b] = dev(a)
        host[b] = a.astype(np.float64)

    def view(b, cols, off):
        return pool[b][off:off + M * cols].view(M, cols)

    # (N, K, gate_up, (x buffer, x offset), (y buffer, y offset)); offsets in elements
    spec = [(768, 512, False, (0, 0), (1, 0)),
            (1024, 768, True, (1, 0), (2, 0)),          # x == y0: chunk-wise
            (256, 512, False, (2, 0), (3, 0)),          # x == y1 (gate_up output)
            (256, 512, False, (1, 256), (4, 0)),        # x inside y0 at an offset
            (768, 256, False, (5, 0), (1, 0)),          # y over y0 / x1 / x3
            (512, 768, False, (1, 0), (6, 0)),          # x == y4
            (512, 512, False, (6, 0), (2, 0)),          # x == y5; y over y1 / x2
            (256, 512, False, (7, 0), (6, 0))]          # y over y5 / x6
    jobs, mats = [], []
    for i, (N, K, gu, (xb, xo), (yb, yo)) in enumerate(spec):
        wq_h, sc_h = synth.weight("stack_order_w", N, K, i)
        seg, _ = zq4.prepare_weight(dev(wq_h), dev(sc_h), N, K, zq4.PREP_SEGMENTED)
        cols = N // 2 if gu else N
        jobs.append((seg, view(xb, K, xo), view(yb, cols, yo), N, K, gu))
        mats.append((wq_h, sc_h))
    order, dep = zq4.stack_plan_waits(
        [(j[0].data_ptr(), j[1].data_ptr(), j[2].data_ptr(), j[3], j[4], j[5]) for j in jobs], M)
    assert dep == [-1, 0, 1, 0, 3, 4, 5, 6]
    zq4.StackPlan(jobs, M).run()
    torch.cuda.synchronize()
    assert zq4.device_errors(clear=True) == 0

    S_img = np.zeros_like(host)
    for i, (N, K, gu, (xb, xo), (yb, yo)) in enumerate(spec):
        x_h = host[xb][xo:xo + M * K].reshape(M, K).astype(np.float16)
        assert np.all(np.isfinite(x_h)), f"replay reads job {i}'s x before it is written"
        wq_h, sc_h = mats[i]
        if gu:
            y, S = oracle.gate_up_silu(wq_h, sc_h, x_h, N, K, interleaved=True)
        else:
            y, S = oracle.gemv(wq_h, sc_h, x_h, N, K)
        cols = y.shape[1]
        host[yb][yo:yo + M * cols] = oracle.round_f16(y).astype(np.float64).ravel()
        S_img[yb][yo:yo + M * cols] = S.ravel()
    got = host_f16(pool).astype(np.float64)
    written = np.isfinite(host)
    assert np.array_equal(np.isfinite(got), written), "a buffer written or left unwritten out of order"
    err = np.abs(got[written] - host[written])
    bound = 2.0 ** -6 * S_img[written] + 2.0 ** -10 * np.abs(host[written]) + 2.0 ** -24
    assert np.all(err <= bound), f"{int((err > bound).sum())} values off; worst {float((err - bound).max())}"


def test_stack_with_one_x_buffer(oracle):
    """M = 4 and K = 8192 leave room for one x buffer only: the compute
    threads stage x of every job (independent ones and the one that reads
    an earlier output); each job matches the oracle on its input."""
    from int4_weight_only_q4f16_gb300 import zq4
    M, K = 4, 8192
    rng = synth.rng_for("stack_onebuf", M)
    x0 = dev(synth.activations(rng, M, K))
    x2 = dev(synth.activations(rng, M, K))
    spec = [(8192, False, x0), (1024, True, None), (256, False, x2)]   # job 1 reads job 0's output
    jobs, mats, ys = [], [], []
    for i, (N, gu, x) in enumerate(spec):
        # unit-gain scales: a gate_up on a 8192-wide output of |N(0, 0.02)|
        # scales would overflow f16
        wq_h, sc_h = synth.weight("stack_onebuf_w", N, K, i, sigma=synth.unit_gain_sigma(K, gu), signed=True)
        seg, _ = zq4.prepare_weight(dev(wq_h), dev(sc_h), N, K, zq4.PREP_SEGMENTED)
        y = torch.full((M, N // 2 if gu else N), float("nan"), dtype=torch.float16, device="cuda")
        jobs.append((seg, ys[0] if x is None else x, y, N, K, gu))
        mats.append((dev(wq_h), dev(sc_h)))
        ys.append(y)
    zq4.StackPlan(jobs, M).run()
    torch.cuda.synchronize()
    assert zq4.device_errors(clear=True) == 0
    for i, ((seg, x, y, N, K_, gu), (wq, sc)) in enumerate(zip(jobs, mats)):
        _check_job(oracle, (wq, sc, x, y, N, K_, gu), f"one-buffer job {i}")


def test_step_engine_job_that_waits_for_two_jobs(oracle):
    """One- and two-token plans run on the tile-per-warp kernel, whose waits
    are lists: job C reads job A's output and overwrites job B's, so it waits
    for both (neither implies the other); independent jobs around them keep
    the waits from being tight. The final buffers equal the given order."""
    from int4_weight_only_q4f16_gb300 import zq4
    M, N, K = 1, 256, 512
    rng = synth.rng_for("step_two_waits")
    mats = [synth.weight("step_two_waits_w", N, K, i) for i in range(16)]
    segs = [zq4.prepare_weight(dev(w), dev(s), N, K, zq4.PREP_SEGMENTED)[0] for w, s in mats]
    xs = [dev(synth.activations(rng, M, K)) for _ in range(16)]
    bufA = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    bufB = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    fill = [torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda") for _ in range(13)]
    jobs = [(segs[0], xs[0], bufA, N, K, False),                     # A: writes bufA
            (segs[1], xs[1], bufB, N, K, False)]              # B: writes bufB
    jobs += [(segs[3 + i], xs[3 + i], fill[i], N, K, False) for i in range(6)]
    # C reads A's output (K = N) and overwrites B's
    wc, sc_ = synth.weight("step_two_waits_c", N, N, 0)
    segC = zq4.prepare_weight(dev(wc), dev(sc_), N, N, zq4.PREP_SEGMENTED)[0]
    jobs.append((segC, bufA, bufB, N, N, False))              # C: reads A, overwrites B
    jobs += [(segs[9 + i], xs[9 + i], fill[6 + i], N, K, False) for i in range(7)]
    plan = zq4.StackPlan(jobs, M)
    assert plan.plan.engine == 1
    plan.run()
    torch.cuda.synchronize()
    assert zq4.device_errors(clear=True) == 0
    order, dep = zq4.stack_plan_waits([(j[0].data_ptr(), j[1].data_ptr(), j[2].data_ptr(), j[3], j[4], j[5])
                                       for j in jobs], M)
    assert order.index(8) > order.index(0) and order.index(8) > order.index(1)
    a = host_f16(bufA)
    a_ref, Sa = oracle.gemv(*mats[0], host_f16(xs[0]), N, K)
    assert_within(a, a_ref, Sa, "job A")
    c_ref, Sc = oracle.gemv(wc, sc_, a, N, N)
    assert_within(host_f16(bufB), c_ref, Sc, "job C after A and over B")
    for i in range(13):
        w, s = mats[3 + i] if i < 6 else mats[9 + i - 6]
        x = xs[3 + i] if i < 6 else xs[9 + i - 6]
        y_ref, S = oracle.gemv(w, s, host_f16(x), N, K)
        assert_within(host_f16(fill[i]), y_ref, S, f"independent job {i}")


def test_step_wait_runs_out_then_a_new_plan_runs(oracle):
    """The bounded-wait recovery path, with host-built data only: the last
    entry of a one-token plan's job table is made to wait for itself (a
    counter nothing ever adds to: it is no waited-for job). With a 5 ms
    limit the launch gives up, reports ZQ4_DEVERR_WAIT_TIMEOUT and ends (no
    kernel left waiting); a plan initialised again over the same jobs then
    runs and matches the oracle."""
    import time
    from int4_weight_only_q4f16_gb300 import zq4
    M, N, K = 1, 256, 512
    rng = synth.rng_for("step_timeout")
    mats = [synth.weight("step_timeout_w", N, K, i) for i in range(10)]
    jobs = []
    for wq_h, sc_h in mats:
        seg = zq4.prepare_weight(dev(wq_h), dev(sc_h), N, K, zq4.PREP_SEGMENTED)[0]
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        jobs.append((seg, dev(synth.activations(rng, M, K)), y, N, K, False))
    plan = zq4.StackPlan(jobs, M)
    assert plan.plan.engine == 1 and plan.plan.entries == len(jobs)
    # job-table entry e: 64 bytes at 128 + 64 e; int32 word 10 = flags (bits
    # 2-3: number of waits, bit 1: waited for), word 13 = its first wait
    e = plan.plan.entries - 1
    img = plan.buffer.cpu()
    words = img[128 + 64 * e:128 + 64 * (e + 1)].view(torch.int32)
    flags = int(words[10])
    assert (flags >> 2) & 3 == 0 and not flags & 2
    words[10] = flags | (1 << 2)
    words[13] = e
    plan.buffer.copy_(img)
    torch.cuda.synchronize()
    assert zq4.device_errors(clear=True) == 0
    plan.set_wait_limit(5_000_000)
    t0 = time.perf_counter()
    plan.run()
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert zq4.device_errors(clear=True) & zq4.DEVERR_WAIT_TIMEOUT
    assert took < 1.0, f"the launch took {took:.3f} s: it should give up after the 5 ms limit"
    again = zq4.StackPlan(jobs, M)
    again.run()
    torch.cuda.synchronize()
    assert zq4.device_errors(clear=True) == 0
    for i, ((seg, x, y, N_, K_, gu), (wq_h, sc_h)) in enumerate(zip(jobs, mats)):
        y_ref, S = oracle.gemv(wq_h, sc_h, host_f16(x), N_, K_)
        assert_within(host_f16(y), y_ref, S, f"job {i} after the re-initialised plan")


@pytest.mark.parametrize("M", [3, 4, 7, 8, 9, 13, 16])
def test_wide_engine_matches_oracle(oracle, M):
    """Three to sixteen tokens on the wide step kernel (x brought with every
    segment by a tensor copy, one MMA column per token): ragged N, K from
    one to 38 segments (split parts included), gate_up, and a job that reads
    a gate_up's output; three runs, bit-identical, each matching the oracle."""
    from int4_weight_only_q4f16_gb300 import zq4
    rng = synth.rng_for("step_wide", M)
    spec = [(200, 256, False), (72, 2560, False), (4096, 3072, True), (336, 768, False), (48, 9728, False)] + \
        [(256, 1024, False)] * 6 + [(120, 2048, False), (333, 512, False)]
    jobs, mats = [], []
    for i, (N, K, gu) in enumerate(spec):
        wq_h, sc_h = synth.weight("step_wide_w", N, K, i)
        seg = zq4.prepare_weight(dev(wq_h), dev(sc_h), N, K, zq4.PREP_SEGMENTED)[0]
        x = jobs[2][2] if i == 11 else dev(synth.activations(rng, M, K))   # job 11 reads job 2's output
        y = torch.full((M, N // 2 if gu else N), float("nan"), dtype=torch.float16, device="cuda")
        jobs.append((seg, x, y, N, K, gu))
        mats.append((wq_h, sc_h))
    plan = zq4.StackPlan(jobs, M)
    assert plan.plan.engine == 2
    first = None
    for run in range(3):
        for j in jobs:
            j[2].fill_(float("nan"))
        plan.run()
        torch.cuda.synchronize()
        assert zq4.device_errors(clear=True) == 0
        bits = [host_f16(j[2]).view(np.uint16).copy() for j in jobs]
        if first is None:
            first = bits
            for i, ((seg, x, y, N, K, gu), (wq_h, sc_h)) in enumerate(zip(jobs, mats)):
                _check_job(oracle, (dev(wq_h), dev(sc_h), x, y, N, K, gu), f"M={M} wide job {i}")
        else:
            for i, (a, b) in enumerate(zip(first, bits)):
                assert np.array_equal(a, b), f"M={M} run {run} job {i} differs from run 0"


@pytest.fixture(scope="module")
def qwen3_16():
    """The Qwen3-4B-shaped stack (36 layers of qkv, o, gate_up, down) with
    16 tokens of seeded input; plans for fewer tokens use its first rows."""
    s = stk.qwen3_4b_stack(M=16, mode="plan")
    return s, s.segmented()


@pytest.mark.slow
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_qwen3_full_step_sampled(oracle, qwen3_16, M):
    """The whole Qwen3-4B-shaped step as one plan at M tokens (the first M
    rows of the 16-token inputs and outputs; down reads gate_up's output),
    run twice; sampled rows of every fourth layer match the oracle."""
    from int4_weight_only_q4f16_gb300 import zq4
    s, segs = qwen3_16
    full = s.jobs()
    views = {}

    def rows(t):
        if t.data_ptr() not in views:
            views[t.data_ptr()] = t[:M]
        return views[t.data_ptr()]
    pj = [(seg, rows(x), rows(y), N, K, gu) for seg, (wq, sc, x, y, N, K, gu) in zip(segs, full)]
    plan = zq4.StackPlan(pj, M)
    assert plan.plan.engine == (1 if M <= 2 else 2)
    plan.run()
    plan.run()
    torch.cuda.synchronize()
    assert zq4.device_errors(clear=True) == 0
    per_layer = len(synth.QWEN3_4B_LAYER)
    rng = np.random.default_rng(7 + M)
    for l in range(0, synth.QWEN3_4B_LAYERS, 4):
        for i, (name, N, K) in enumerate(synth.QWEN3_4B_LAYER):
            wq, sc, x, y, N_, K_, gu = full[l * per_layer + i]
            r = np.unique(np.concatenate([t * 16 + rng.integers(0, 16, 1) for t in range(0, N // 16, 3)]
                                         + [[0, N - 1]]))
            _check_job(oracle, (wq, sc, rows(x), rows(y), N, K, gu), f"qwen3 M={M} layer {l} {name}", rows=r)
