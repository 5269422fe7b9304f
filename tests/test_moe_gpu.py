"""GPU parity of zq4_moe_gemv (expert-gather GEMV) against the CPU oracle:
the GATE_UP_SILU stage, the DOWN_COMBINE stage (checked on the GPU's own f16
intermediate, so each call's error is isolated), routing exactness, and the
device-side report of invalid expert ids."""
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


def _bank(tag, E, N, K):
    rng = synth.rng_for(tag, E, N, K)
    return synth.packed_codes(rng, E * N, K), synth.group_scales(rng, E * N, K)


@pytest.mark.parametrize("E,T,top_k,I,D", [(8, 1, 2, 32, 64), (16, 4, 8, 64, 128),
                                           (128, 3, 8, 96, 64), (5, 6, 5, 96, 96),
                                           (4, 2, 1, 32, 32)])
def test_moe_two_stage_parity(zq4, oracle, E, T, top_k, I, D):
    gq, gs = _bank("moe_gu", E, 2 * I, D)     # gate_up: [2I, D] per expert
    dq, ds = _bank("moe_dn", E, D, I)         # down:    [D, I]  per expert
    rng = synth.rng_for("moe_x", E, T)
    x = synth.activations(rng, T, D)
    ids, r = synth.routing(rng, T, E, top_k)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    h = zq4.moe_gemv(dev(gq), dev(gs), E, dev(x), 2 * I, D, dev(ids), zq4.MOE_GATE_UP_SILU,
                     dev_status=status)
    h_ref, Sh, bad = oracle.moe_gate_up(gq, gs, E, x, 2 * I, D, ids)
    h_gpu = host_f16(h)
    assert_within(h_gpu, h_ref, Sh, "moe gate_up")
    y = zq4.moe_gemv(dev(dq), dev(ds), E, h, D, I, dev(ids), zq4.MOE_DOWN_COMBINE,
                     route_w=dev(r), dev_status=status)
    y_ref, S, bad2 = oracle.moe_down_combine(dq, ds, E, h_gpu, r, D, I, ids)
    assert_within(host_f16(y), y_ref, S, "moe down+combine")
    assert bad == bad2 == 0 and int(status.item()) == 0


def test_moe_routing_exact(zq4, oracle):
    """Each expert's down matrix is constant code c_e with scale 1, so z_e =
    (c_e - 7) * sum(x) identifies exactly which expert served each slot."""
    E, T, top_k, K, N = 15, 5, 4, 64, 32
    c = np.arange(E) + (np.arange(E) >= 7)                  # distinct codes 0..15 except 7
    wq = np.repeat((c * 0x11111111).astype(np.uint32), N)[:, None].repeat(K // 8, 1)
    sc = np.ones((E * N, K // 32), np.float16)
    rng = synth.rng_for("route", E)
    ids, _ = synth.routing(rng, T, E, top_k)
    x = np.zeros((T, top_k, K), np.float16)
    for t in range(T):
        for j in range(top_k):
            x[t, j, j] = 1.0                                # slot j reads column j only
    onehot = np.eye(top_k, dtype=np.float32)
    for j in range(top_k):
        r = np.tile(onehot[j], (T, 1))
        y = host_f16(zq4.moe_gemv(dev(wq), dev(sc), E, dev(x), N, K, dev(ids),
                                  zq4.MOE_DOWN_COMBINE, route_w=dev(r)))
        want = (c[ids[:, j]] - 7).astype(np.float64)
        assert np.array_equal(y.astype(np.float64), np.repeat(want[:, None], N, 1))


def test_moe_invalid_ids_report_and_contribute_nothing(zq4, oracle):
    E, T, top_k, I, D = 6, 3, 3, 32, 64
    gq, gs = _bank("bad_gu", E, 2 * I, D)
    dq, ds = _bank("bad_dn", E, D, I)
    x = synth.activations(synth.rng_for("bad_x"), T, D)
    ids = np.array([[0, 9, 2], [-3, 1, 5], [4, 4, 6]], np.int32)
    r = np.full((T, top_k), 1.0 / 3, np.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    h = zq4.moe_gemv(dev(gq), dev(gs), E, dev(x), 2 * I, D, dev(ids), zq4.MOE_GATE_UP_SILU,
                     dev_status=status)
    h_gpu = host_f16(h)
    assert int(status.item()) & zq4.DEV_BAD_EXPERT_ID
    for t, j in [(0, 1), (1, 0), (2, 2)]:
        assert np.all(h_gpu[t, j] == 0)
    h_ref, Sh, bad = oracle.moe_gate_up(gq, gs, E, x, 2 * I, D, ids)
    assert bad == 3
    assert_within(h_gpu, h_ref, Sh, "gate_up with bad ids")
    status.zero_()
    y = zq4.moe_gemv(dev(dq), dev(ds), E, h, D, I, dev(ids), zq4.MOE_DOWN_COMBINE,
                     route_w=dev(r), dev_status=status)
    y_ref, S, bad = oracle.moe_down_combine(dq, ds, E, h_gpu, r, D, I, ids)
    assert bad == 3 and int(status.item()) & zq4.DEV_BAD_EXPERT_ID
    assert_within(host_f16(y), y_ref, S, "down with bad ids")


@pytest.mark.slow
@pytest.mark.parametrize("T", [1, 4, 16])
def test_moe_full_size_parity(zq4, oracle, T):
    """The MoE block at its full size: 128 experts, gate_up 1024 x 2048
    (interleaved, SiLU*mul -> 512) and down 2048 x 512, top-8 routing, T
    tokens -- bank 0 of the benchmark's MoE workload, both stages exactly as
    it runs them. Every output is compared with the oracle; the down stage
    reads the GPU's own f16 h, as in the small cases."""
    E, top_k = synth.MOE_EXPERTS, synth.MOE_TOP_K
    (N2, D), (Dn, I) = synth.MOE_GATE_UP, synth.MOE_DOWN
    gq, gs = synth.weight("moe_gu", E * N2, D, 0)
    dq, ds = synth.weight("moe_dn", E * Dn, I, 0)
    rng = synth.rng_for("moe_route", 0, T)
    ids, r = synth.routing(rng, T, E, top_k)
    x = synth.activations(rng, T, D)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    h = zq4.moe_gemv(dev(gq), dev(gs), E, dev(x), N2, D, dev(ids), zq4.MOE_GATE_UP_SILU, dev_status=status)
    h_gpu = host_f16(h)
    h_ref, Sh, bad = oracle.moe_gate_up(gq, gs, E, x, N2, D, ids)
    assert h_gpu.shape == (T, top_k, N2 // 2)
    assert_within(h_gpu, h_ref, Sh, f"moe gate_up T={T}")
    y = zq4.moe_gemv(dev(dq), dev(ds), E, h, Dn, I, dev(ids), zq4.MOE_DOWN_COMBINE, route_w=dev(r),
                     dev_status=status)
    y_ref, S, bad2 = oracle.moe_down_combine(dq, ds, E, h_gpu, r, Dn, I, ids)
    assert_within(host_f16(y), y_ref, S, f"moe down+combine T={T}")
    assert bad == bad2 == 0 and int(status.item()) == 0


def test_moe_routing_exact_128_experts(zq4):
    """Routing at the full bank size: expert e's down matrix (2048 x 512,
    the MoE workload's shape) has every code 8 and every scale 1 + e/1024
    (distinct, exact in f16), so with slot j reading a one-hot input and a
    one-hot router weight on slot j, every output of token t is exactly
    1 + ids[t, j]/1024: the expert that served each (token, slot) is read
    back bit for bit, for all 16 tokens of the largest case."""
    E, T, top_k = synth.MOE_EXPERTS, 16, synth.MOE_TOP_K
    Dn, I = synth.MOE_DOWN
    wq = np.full((E * Dn, I // 8), 0x88888888, np.uint32)
    sc = np.repeat((1.0 + np.arange(E) / 1024.0).astype(np.float16), Dn)[:, None].repeat(I // 32, 1)
    ids, _ = synth.routing(synth.rng_for("route128", T), T, E, top_k)
    x = np.zeros((T, top_k, I), np.float16)
    for j in range(top_k):
        x[:, j, 5 + 3 * j] = 1.0                                 # slot j reads one column of its own
    for j in range(top_k):
        r = np.zeros((T, top_k), np.float32)
        r[:, j] = 1.0
        y = host_f16(zq4.moe_gemv(dev(wq), dev(sc), E, dev(x), Dn, I, dev(ids), zq4.MOE_DOWN_COMBINE,
                                  route_w=dev(r)))
        want = (1.0 + ids[:, j] / 1024.0).astype(np.float16)
        assert np.array_equal(y, np.repeat(want[:, None], Dn, 1)), f"slot {j}"
