"""GPU parity of the MLX affine format (zq4_gemv_affine,
zq4_gate_up_silu_affine: value = s * q + b, one f16 scale and bias per 64
weights) against the CPU oracle. The tolerance is the format's:
|y - y_ref| <= 2^-10 |y_ref| + 1e-4 Sa with Sa = sum_k |x_k| (|s| q_k + |b|),
the size of each of the two sums (s * sum(x q), b * sum(x)) the kernel adds."""
import numpy as np
import pytest
import torch

from int4_weight_only_q4f16_gb300 import synth
from helpers import assert_within, dev, host_f16

pytestmark = pytest.mark.gpu


def _affine_weight(tag, N, K, i=0):
    rng = synth.rng_for(tag, N, K, i)
    wq = synth.packed_codes(rng, N, K)
    sc = np.abs(rng.standard_normal((N, K // 64)) * 0.02).astype(np.float16)
    # biases near -8 s (codes centred, as quantizers choose them) plus noise
    bi = (-8.0 * sc.astype(np.float32) + rng.standard_normal((N, K // 64)).astype(np.float32) * 0.01).astype(np.float16)
    return wq, sc, bi


@pytest.mark.parametrize("M,N,K", [(1, 3072, 2560), (3, 333, 192), (8, 1000, 9728), (16, 256, 640),
                                   (5, 64, 64), (1, 2560, 9728), (16, 1000, 1536), (13, 77, 3072)])
def test_affine_gemv_matches_oracle(oracle, M, N, K):
    from int4_weight_only_q4f16_gb300 import zq4
    wq, sc, bi = _affine_weight("aff_gemv", N, K)
    x = synth.activations(synth.rng_for("aff_x", M, K), M, K)
    y = zq4.gemv_affine(dev(wq), dev(sc), dev(bi), dev(x), N, K)
    y_ref, Sa = oracle.gemv_affine(wq, sc, bi, x, N, K)
    assert_within(host_f16(y), y_ref, Sa, f"affine gemv M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N2,K", [(1, 2048, 2560), (4, 66, 192), (9, 512, 1024)])
def test_affine_gate_up_matches_oracle(oracle, M, N2, K):
    from int4_weight_only_q4f16_gb300 import zq4
    wq, sc, bi = _affine_weight("aff_gu", N2, K)
    x = synth.activations(synth.rng_for("aff_gux", M, K), M, K)
    h = zq4.gate_up_silu_affine(dev(wq), dev(sc), dev(bi), dev(x), N2, K)
    h_ref, Sh = oracle.gate_up_silu_affine(wq, sc, bi, x, N2, K)
    assert_within(host_f16(h), h_ref, Sh, f"affine gate_up M={M} N2={N2} K={K}")


def _offset_by_one(a):
    """a copy of f16 array a on the device whose first element sits 2 bytes
    past an allocation's (16-byte aligned) start"""
    buf = torch.zeros(a.size + 1, dtype=torch.float16, device="cuda")
    buf[1:] = torch.from_numpy(np.ascontiguousarray(a).reshape(-1)).cuda()
    return buf[1:]


@pytest.mark.parametrize("gate_up", [False, True])
def test_affine_scales_on_2_byte_boundaries(oracle, gate_up):
    """Scales and biases need only 2-byte alignment: at K = 1024 (a shape the
    tensor-core kernel takes when they are 16-byte aligned) the call runs the
    CUDA-core kernel and still matches the oracle."""
    from int4_weight_only_q4f16_gb300 import zq4
    M, N, K = 3, 160, 1024
    wq, sc, bi = _affine_weight("aff_odd", N, K)
    x = synth.activations(synth.rng_for("aff_oddx", M, K), M, K)
    s2, b2 = _offset_by_one(sc), _offset_by_one(bi)
    assert s2.data_ptr() % 16 == 2 and b2.data_ptr() % 16 == 2
    if gate_up:
        out = zq4.gate_up_silu_affine(dev(wq), s2, b2, dev(x), N, K)
        ref, S = oracle.gate_up_silu_affine(wq, sc, bi, x, N, K)
    else:
        out = zq4.gemv_affine(dev(wq), s2, b2, dev(x), N, K)
        ref, S = oracle.gemv_affine(wq, sc, bi, x, N, K)
    assert_within(host_f16(out), ref, S, f"affine, 2-byte aligned scales, gate_up={gate_up}")
    assert zq4.device_errors(clear=True) == 0


@pytest.mark.parametrize("K", [256, 1024])
def test_affine_one_hot_bit_exact(oracle, K):
    """x = e_k returns f16(s q + b) exactly: scales and biases are multiples
    of 2^-8 below 1, so s q + b is exact in fp32 and f16 rounds it once
    (K = 256: the CUDA-core kernel; K = 1024: the tensor-core kernel, whose
    64-column group sums x q and x exactly when x is one-hot)."""
    N = 96
    rng = synth.rng_for("aff_onehot", K)
    wq = synth.packed_codes(rng, N, K)
    sc = (rng.integers(1, 64, (N, K // 64)) / 256.0).astype(np.float16)
    bi = (rng.integers(-255, 256, (N, K // 64)) / 256.0).astype(np.float16)
    w = oracle.dequant_affine(wq, sc, bi, N, K)
    from int4_weight_only_q4f16_gb300 import zq4
    for k in (0, 7, 63, 64, 130, 255, K - 1):
        x = np.zeros((1, K), np.float16)
        x[0, k] = 1.0
        y = host_f16(zq4.gemv_affine(dev(wq), dev(sc), dev(bi), dev(x), N, K))
        assert np.array_equal(y[0].view(np.uint16), oracle.round_f16(w[:, k]).view(np.uint16)), k


def test_affine_zero_weights_give_exact_zero():
    """Scales and biases all 0 (any codes), and codes all 0 with biases 0:
    every weight is exactly 0, so y is exactly 0 for large activations too."""
    from int4_weight_only_q4f16_gb300 import zq4
    M, N, K = 4, 200, 512
    rng = synth.rng_for("aff_zero")
    x = dev((rng.standard_normal((M, K)) * 300).astype(np.float16))
    wq = dev(synth.packed_codes(rng, N, K))
    z = dev(np.zeros((N, K // 64), np.float16))
    assert torch.all(zq4.gemv_affine(wq, z, z, x, N, K) == 0)
    sc = dev(np.abs(rng.standard_normal((N, K // 64)) * 0.02).astype(np.float16))
    w0 = dev(np.zeros((N, K // 8), np.uint32))
    assert torch.all(zq4.gemv_affine(w0, sc, z, x, N, K) == 0)
    assert zq4.device_errors(clear=True) == 0


def _affine_bank(tag, E, N, K):
    rng = synth.rng_for(tag, E, N, K)
    wq = synth.packed_codes(rng, E * N, K)
    sc = np.abs(rng.standard_normal((E * N, K // 64)) * 0.02).astype(np.float16)
    bi = (-8.0 * sc.astype(np.float32) + rng.standard_normal((E * N, K // 64)).astype(np.float32) * 0.01).astype(np.float16)
    return wq, sc, bi


@pytest.mark.parametrize("E,T,top_k,I,D", [(8, 1, 2, 64, 128), (16, 4, 8, 128, 256), (128, 3, 8, 512, 2048),
                                           (5, 6, 5, 192, 64)])
def test_affine_moe_two_stage_parity(oracle, E, T, top_k, I, D):
    """Both expert stages on affine banks; the down stage is checked on the
    GPU's own f16 intermediate, so each call's error is isolated."""
    from int4_weight_only_q4f16_gb300 import zq4
    gq, gs, gb = _affine_bank("aff_moe_gu", E, 2 * I, D)     # gate_up: [2I, D] per expert
    dq, ds, db = _affine_bank("aff_moe_dn", E, D, I)         # down:    [D, I]  per expert
    rng = synth.rng_for("aff_moe_x", E, T)
    x = synth.activations(rng, T, D)
    ids, r = synth.routing(rng, T, E, top_k)
    ids[0, 0] = E + 3                                         # one invalid id: reported, contributes nothing
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    h = zq4.moe_gemv_affine(dev(gq), dev(gs), dev(gb), E, dev(x), 2 * I, D, dev(ids), zq4.MOE_GATE_UP_SILU,
                            dev_status=status)
    h_ref, Sh, bad = oracle.moe_gate_up_affine(gq, gs, gb, E, x, 2 * I, D, ids)
    h_gpu = host_f16(h)
    assert_within(h_gpu, h_ref, Sh, "affine moe gate_up")
    y = zq4.moe_gemv_affine(dev(dq), dev(ds), dev(db), E, h, D, I, dev(ids), zq4.MOE_DOWN_COMBINE,
                            route_w=dev(r), dev_status=status)
    y_ref, S, bad2 = oracle.moe_down_combine_affine(dq, ds, db, E, h_gpu, r, D, I, ids)
    assert_within(host_f16(y), y_ref, S, "affine moe down+combine")
    assert bad == bad2 == 1 and int(status.item()) != 0
    assert zq4.device_errors(clear=True) == 0
