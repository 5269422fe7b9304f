"""GPU parity of zq4_gemv_seg / zq4_gate_up_silu_seg (weights in the
segmented layout, M <= 8) against the CPU oracle: ragged shapes spanning many
tiles and CTAs, every Phi-3 projection at full size on sampled rows, a
chained gate_up -> down, reproducibility, and rejection of bad arguments."""
import numpy as np
import pytest
import torch

from int4_weight_only_q4f16_gb300 import synth
from int4_weight_only_q4f16_gb300 import stack as stk
from helpers import assert_within, dev, host_f16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zq4():
    from int4_weight_only_q4f16_gb300 import zq4 as m
    return m


def _case(tag, M, N, K):
    rng = synth.rng_for(tag, M, N, K)
    return synth.packed_codes(rng, N, K), synth.group_scales(rng, N, K), synth.activations(rng, M, K)


SHAPES = [(1, 1, 256), (1, 17, 512), (1, 333, 3072), (2, 130, 1024), (3, 77, 3072), (4, 2560, 2560),
          (5, 33, 768), (8, 64, 4096), (8, 3072, 8192), (1, 40, 9728), (1, 5000, 256), (7, 16, 256)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemv_seg_parity(zq4, oracle, M, N, K):
    wq, sc, x = _case("seg", M, N, K)
    seg, _ = zq4.prepare_weight(dev(wq), dev(sc), N, K, zq4.PREP_SEGMENTED)
    y = host_f16(zq4.gemv_seg(seg, dev(x), N, K))
    y_ref, S = oracle.gemv(wq, sc, x, N, K)
    assert_within(y, y_ref, S, f"gemv_seg M={M} N={N} K={K}")


@pytest.mark.parametrize("M,I,K", [(1, 8, 256), (1, 8192, 3072), (2, 50, 2560), (8, 64, 512), (3, 9728, 2560)])
def test_gate_up_silu_seg_parity(zq4, oracle, M, I, K):
    wq, sc, x = _case("seg_gu", M, 2 * I, K)
    seg, _ = zq4.prepare_weight(dev(wq), dev(sc), 2 * I, K, zq4.PREP_SEGMENTED)
    h = host_f16(zq4.gate_up_silu_seg(seg, dev(x), 2 * I, K))
    if I > 512:
        js = np.unique(np.concatenate([np.arange(0, I, 37), [I - 1]]))
        rows = np.stack([2 * js, 2 * js + 1], 1).ravel()
        h_ref, Sh = oracle.gate_up_silu(wq[rows], sc[rows], x, len(rows), K, interleaved=True)
        assert_within(h[:, js], h_ref, Sh, f"gate_up_seg M={M} I={I} K={K}")
    else:
        h_ref, Sh = oracle.gate_up_silu(wq, sc, x, 2 * I, K, interleaved=True)
        assert_within(h, h_ref, Sh, f"gate_up_seg M={M} I={I} K={K}")


def test_seg_matches_canonical_calls_and_is_reproducible(zq4):
    """Same matrix, segmented and canonical: within the tolerance of each
    other (different fp32 addition order), and the segmented call repeats
    bit for bit."""
    M, N, K = 2, 3072, 8192
    wq, sc, x = _case("seg_vs", M, N, K)
    W, Sd, X = dev(wq), dev(sc), dev(x)
    seg, _ = zq4.prepare_weight(W, Sd, N, K, zq4.PREP_SEGMENTED)
    a = host_f16(zq4.gemv_seg(seg, X, N, K))
    b = host_f16(zq4.gemv_seg(seg, X, N, K))
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    c = host_f16(zq4.gemv(W, Sd, X, N, K)).astype(np.float64)
    assert np.max(np.abs(a.astype(np.float64) - c)) <= 2.0 ** -8 * np.max(np.abs(c))


def test_phi3_step_in_seg_mode_sampled(oracle):
    """The Phi-3 step as the benchmark runs it in seg mode: every projection
    of layers 0, 13, 31 and the LM head on sampled rows (down on the GPU's own
    gate_up output)."""
    s = stk.phi3_stack(mode="seg")
    strm = torch.cuda.Stream()
    with torch.cuda.stream(strm):
        s.launch_step(strm)
        s.launch_step(strm)
    torch.cuda.synchronize()
    jobs = s.jobs()
    per = len(synth.PHI3_LAYER)
    check = [l * per + i for l in (0, 13, 31) for i in range(per)] + [len(jobs) - 1]
    rng = np.random.default_rng(9)
    for j in check:
        wq, sc, x, y, N, K, gate_up = jobs[j]
        wq_h, sc_h, x_h, y_h = wq.cpu().numpy().view(np.uint32), sc.cpu().numpy().view(np.float16), host_f16(x), host_f16(y)
        if gate_up:
            js = np.unique(np.concatenate([rng.integers(0, N // 2, 150), [0, N // 2 - 1]]))
            rows = np.stack([2 * js, 2 * js + 1], 1).ravel()
            h_ref, Sh = oracle.gate_up_silu(wq_h[rows], sc_h[rows], x_h, len(rows), K, interleaved=True)
            assert_within(y_h[:, js], h_ref, Sh, f"job {j} gate_up")
        else:
            rows = np.unique(np.concatenate([rng.integers(0, N, 200), [0, N - 1]]))
            y_ref, S = oracle.gemv(wq_h, sc_h, x_h, N, K, rows=rows)
            assert_within(y_h[:, rows], y_ref, S, f"job {j}")


def test_seg_rejects_bad_arguments(zq4):
    wq, sc, x = _case("seg_bad", 1, 64, 512)
    seg, _ = zq4.prepare_weight(dev(wq), dev(sc), 64, 512, zq4.PREP_SEGMENTED)
    x9 = torch.zeros((9, 512), dtype=torch.float16, device="cuda")
    with pytest.raises(zq4.Zq4Error, match="UNSUPPORTED"):
        zq4.gemv_seg(seg, x9, 64, 512)                       # M = 9
    with pytest.raises(zq4.Zq4Error, match="SHAPE"):
        zq4.gemv_seg(seg, dev(x)[:, :480].contiguous(), 64, 480)   # K % 256
    assert zq4.device_errors(clear=True) == 0
