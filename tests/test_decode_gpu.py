"""GPU parity of zq4_gemv / zq4_gate_up_silu / zq4_dequant_* against the CPU
oracle, element by element, on small and ragged shapes that still span
several tiles. Bar: |y - y_ref| <= 2^-10 |y_ref| + 1e-4 sum|x*w|; dequantized
weights bit-exact."""
import numpy as np
import pytest
import torch

from int4_weight_only_q4f16_gb300 import synth
from helpers import assert_within, dev, host_f16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zq4():
    from int4_weight_only_q4f16_gb300 import zq4 as m
    return m


def _case(tag, M, N, K):
    rng = synth.rng_for(tag, M, N, K)
    return synth.packed_codes(rng, N, K), synth.group_scales(rng, N, K), synth.activations(rng, M, K)


SHAPES = [  # (M, N, K): ragged N, K spanning <1, 1 and many 32-lane strides
    (1, 1, 32), (1, 7, 64), (1, 64, 96), (1, 200, 2560), (1, 333, 3072), (1, 96, 8192),
    (1, 40, 9728), (1, 256, 512), (2, 130, 1024), (3, 77, 3072), (4, 128, 2560),
    (5, 33, 416), (8, 64, 4096), (9, 65, 2048), (16, 100, 3072), (17, 31, 1024),
    (31, 20, 512), (63, 17, 256), (64, 40, 512), (65, 24, 640),
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemv_parity(zq4, oracle, M, N, K):
    wq, sc, x = _case("gemv", M, N, K)
    y = zq4.gemv(dev(wq), dev(sc), dev(x), N, K)
    y_ref, S = oracle.gemv(wq, sc, x, N, K)
    assert_within(host_f16(y), y_ref, S, f"gemv M={M} N={N} K={K}")


def test_gemv_one_hot_bit_exact(zq4, oracle):
    """x = e_k returns f16(w[:, k]) exactly (one non-zero product)."""
    N, K = 48, 256
    wq, sc, _ = _case("onehot", 1, N, K)
    w = oracle.dequant(wq, sc, N, K)
    for k in (0, 1, 7, 8, 31, 32, 33, 100, 255):
        x = np.zeros((1, K), np.float16)
        x[0, k] = 1.0
        y = host_f16(zq4.gemv(dev(wq), dev(sc), dev(x), N, K))
        want = oracle.round_f16(w[:, k])
        assert np.array_equal(y[0].view(np.uint16), want.view(np.uint16)), k


def test_gemv_constant_codes_closed_form(zq4, oracle):
    N, K = 64, 1024
    rng = synth.rng_for("const", N, K)
    x = synth.activations(rng, 2, K)
    sx = x.astype(np.float64).sum(axis=1)
    for c in (0, 7, 15):
        wq = np.full((N, K // 8), c * 0x11111111, np.uint32)
        sc = np.full((N, K // 32), 0.0137, np.float16)
        y = host_f16(zq4.gemv(dev(wq), dev(sc), dev(x), N, K)).astype(np.float64)
        want = (c - 7) * float(sc[0, 0]) * sx
        S = np.abs(x.astype(np.float64)).sum(axis=1) * abs(c - 7) * float(sc[0, 0])
        assert_within(y, np.repeat(want[:, None], N, 1), np.repeat(S[:, None], N, 1), f"c={c}")
        if c == 7:
            assert np.all(y == 0)


@pytest.mark.parametrize("K", [256, 3072, 8192])
def test_all_zero_point_codes_give_exact_zero(zq4, K):
    """Codes all 7 make every weight exactly 0: S = 0, so the output must be
    exactly 0 even for large activations (no bias-cancellation residue)."""
    N, M = 48, 3
    rng = synth.rng_for("zp7", K)
    x = (rng.standard_normal((M, K)) * 300).astype(np.float16)
    wq = np.full((N, K // 8), 0x77777777, np.uint32)
    sc = synth.group_scales(rng, N, K)
    y = host_f16(zq4.gemv(dev(wq), dev(sc), dev(x), N, K))
    assert np.all(y == 0)
    h = host_f16(zq4.gate_up_silu(dev(wq), dev(sc), dev(x), N, K))
    assert np.all(h == 0)


def test_gemv_reproducible_and_linear(zq4):
    M, N, K = 3, 257, 3072
    wq, sc, x = _case("repro", M, N, K)
    W, Sd = dev(wq), dev(sc)
    y1 = host_f16(zq4.gemv(W, Sd, dev(x), N, K))
    y2 = host_f16(zq4.gemv(W, Sd, dev(x), N, K))
    assert np.array_equal(y1.view(np.uint16), y2.view(np.uint16))
    x2 = (x.astype(np.float32) * 4).astype(np.float16)
    y4 = host_f16(zq4.gemv(W, Sd, dev(x2), N, K))
    assert np.array_equal(y4.astype(np.float64), 4 * y1.astype(np.float64))


def test_gemv_guard_band_and_nonzero(zq4):
    M, N, K = 2, 300, 2560
    wq, sc, x = _case("guard", M, N, K)
    buf = torch.full((M * N + 4096,), float("nan"), dtype=torch.float16, device="cuda")
    y = buf[: M * N].view(M, N)
    zq4.gemv(dev(wq), dev(sc), dev(x), N, K, y=y)
    torch.cuda.synchronize()
    assert torch.isnan(buf[M * N:]).all(), "kernel wrote past its output"
    assert torch.isfinite(y).all() and (y != 0).any()


def test_gemv_in_cuda_graph(zq4, oracle):
    M, N, K = 1, 512, 3072
    wq, sc, x = _case("graph", M, N, K)
    W, Sd, X = dev(wq), dev(sc), dev(x)
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        zq4.gemv(W, Sd, X, N, K, y=y)       # warm (kernel attributes set outside capture)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            zq4.gemv(W, Sd, X, N, K, y=y)
    y.zero_()
    g.replay()
    y_ref, S = oracle.gemv(wq, sc, x, N, K)
    assert_within(host_f16(y), y_ref, S, "graph replay")


@pytest.mark.parametrize("M,I,K", [(1, 1, 32), (1, 96, 3072), (2, 50, 2560), (4, 64, 512),
                                   (7, 33, 1024), (16, 40, 2048), (1, 17, 8192), (20, 8, 96)])
def test_gate_up_silu_parity(zq4, oracle, M, I, K):
    wq, sc, x = _case("gateup", M, 2 * I, K)
    h = zq4.gate_up_silu(dev(wq), dev(sc), dev(x), 2 * I, K)
    h_ref, Sh = oracle.gate_up_silu(wq, sc, x, 2 * I, K, interleaved=True)
    assert_within(host_f16(h), h_ref, Sh, f"gate_up M={M} I={I} K={K}")


def test_prepare_concat_to_interleaved(zq4, oracle):
    I, K, M = 40, 512, 3
    wq, sc, x = _case("prep", M, 2 * I, K)        # concatenated [gate; up]
    wq_i, sc_i = zq4.prepare_weight(dev(wq), dev(sc), 2 * I, K, zq4.PREP_CONCAT_TO_INTERLEAVED)
    torch.cuda.synchronize()
    order = np.empty(2 * I, np.int64)
    order[0::2] = np.arange(I)
    order[1::2] = I + np.arange(I)
    assert np.array_equal(wq_i.cpu().numpy().view(np.uint32), wq[order])
    assert np.array_equal(sc_i.cpu().numpy().view(np.uint16), sc[order].view(np.uint16))
    h = zq4.gate_up_silu(wq_i, sc_i, dev(x), 2 * I, K)
    h_ref, Sh = oracle.gate_up_silu(wq, sc, x, 2 * I, K, interleaved=False)
    assert_within(host_f16(h), h_ref, Sh, "prepared gate_up")
    wc, scc = zq4.prepare_weight(dev(wq), dev(sc), 2 * I, K, zq4.PREP_COPY)
    assert np.array_equal(wc.cpu().numpy().view(np.uint32), wq)


def _segmented_reference(wq, sc, N, K):
    """The segmented layout, built from its definition in the C header:
    tile-major 2304-byte segments of 16 row records of 144 bytes (record
    word 8q + g = word q of group g with nibble slot j holding element
    (0, 2, 4, 6, 1, 3, 5, 7)[j], then the row's 8 scales); rows past N zero."""
    T, S = (N + 15) // 16, K // 256
    elem_of_slot = (0, 2, 4, 6, 1, 3, 5, 7)
    out = np.zeros(T * S * 576, np.uint32)
    scw = np.ascontiguousarray(sc).view(np.uint32).reshape(N, K // 64)   # scale pairs
    for t in range(T):
        for s_ in range(S):
            for i in range(16):
                n = 16 * t + i
                if n >= N:
                    continue
                base = (t * S + s_) * 576 + 36 * i
                for q in range(4):
                    for g in range(8):
                        w = int(wq[n, 32 * s_ + 4 * g + q])
                        v = 0
                        for j in range(8):
                            v |= ((w >> (4 * elem_of_slot[j])) & 0xF) << (4 * j)
                        out[base + 8 * q + g] = v
                out[base + 32: base + 36] = scw[n, 4 * s_: 4 * s_ + 4]
    return out.view(np.uint8)


@pytest.mark.parametrize("N,K,interleave", [(37, 512, False), (16, 256, False), (40, 768, True)])
def test_prepare_segmented_layout_bytes(zq4, N, K, interleave):
    wq, sc, _ = _case("segl", 1, N, K)
    flags = zq4.PREP_SEGMENTED | (zq4.PREP_CONCAT_TO_INTERLEAVED if interleave else 0)
    seg, none = zq4.prepare_weight(dev(wq), dev(sc), N, K, flags)
    assert none is None and seg.numel() == zq4.segmented_bytes(N, K)
    if interleave:
        order = np.empty(N, np.int64)
        order[0::2] = np.arange(N // 2)
        order[1::2] = N // 2 + np.arange(N // 2)
        wq, sc = wq[order], sc[order]
    assert np.array_equal(seg.cpu().numpy(), _segmented_reference(wq, sc, N, K))


@pytest.mark.parametrize("N,K", [(1, 32), (13, 96), (64, 3072), (5, 9728)])
def test_dequant_bit_exact(zq4, oracle, N, K):
    wq, sc, _ = _case("deq", 1, N, K)
    w = oracle.dequant(wq, sc, N, K)
    w32 = zq4.dequant_f32(dev(wq), dev(sc), N, K).cpu().numpy()
    assert np.array_equal(w32.view(np.uint32), w.astype(np.float32).view(np.uint32))
    assert np.array_equal(w32.astype(np.float64), w)       # (q-7)*s is exact in fp32
    w16 = zq4.dequant_f16(dev(wq), dev(sc), N, K).cpu().numpy()
    want16 = oracle.round_f16(w.ravel()).reshape(N, K)
    assert np.array_equal(w16.view(np.uint16), want16.view(np.uint16))


def test_subnormal_and_zero_scales(zq4, oracle):
    N, K = 32, 256
    wq, _, x = _case("subn", 1, N, K)
    bits = np.random.default_rng(0).integers(0, 0x400, (N, K // 32)).astype(np.uint16)
    bits[0] = 0
    sc = bits.view(np.float16)                      # zero and subnormal scales only
    w = oracle.dequant(wq, sc, N, K)
    w32 = zq4.dequant_f32(dev(wq), dev(sc), N, K).cpu().numpy()
    assert np.array_equal(w32.astype(np.float64), w)
    y = zq4.gemv(dev(wq), dev(sc), dev(x), N, K)
    y_ref, S = oracle.gemv(wq, sc, x, N, K)
    assert_within(host_f16(y), y_ref, S, "subnormal scales")


def test_no_device_errors_recorded(zq4):
    """No kernel run so far gave up an internal wait."""
    assert zq4.device_errors(clear=True) == 0
