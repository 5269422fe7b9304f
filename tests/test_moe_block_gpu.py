"""GPU parity of zq4_moe_block (the MoE block in one call, each touched
expert read once per stage) against the CPU oracle: the full-size bank of
the MoE workload (128 experts, gate_up 1024 x 2048, down 2048 x 512, top-8)
at T = 1, 4, 16; the device grouping compared bit-exactly with a host
grouping of the same routing; repeated calls bit-identical; invalid expert
ids; and the CUDA-core path of shapes the tensor-core one does not take."""
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


def host_grouping(ids, E):
    """The grouping the block documents: touched experts in order of their
    first (token, slot) pair, each expert's pairs in pair order."""
    flat = [int(e) for e in np.asarray(ids).ravel()]
    experts = []
    for e in flat:
        if 0 <= e < E and e not in experts:
            experts.append(e)
    order, starts = [], [0]
    for e in experts:
        order += [p for p, f in enumerate(flat) if f == e]
        starts.append(len(order))
    return len(experts), len(order), order, experts, starts


def check_group(group, ids, E):
    P = np.asarray(ids).size
    g = group.cpu().numpy()
    U, V, order, experts, starts = host_grouping(ids, E)
    assert g[0] == U and g[1] == V
    assert list(g[2:2 + V]) == order and all(g[2 + V:2 + P] == -1)
    assert list(g[2 + P:2 + P + U]) == experts and all(g[2 + P + U:2 + 2 * P] == -1)
    assert list(g[2 + 2 * P:2 + 2 * P + U + 1]) == starts


def _banks(zq4, gq, gs, dq, ds, E, D, I):
    gu = zq4.prepare_weight(dev(gq), dev(gs), E * 2 * I, D, zq4.PREP_SEGMENTED)[0]
    dn = zq4.prepare_weight(dev(dq), dev(ds), E * D, I, zq4.PREP_SEGMENTED)[0]
    return gu, dn


def _run(zq4, oracle, gq, gs, dq, ds, E, x, ids, r, D, I, status=None):
    T, top_k = ids.shape
    gu, dn = _banks(zq4, gq, gs, dq, ds, E, D, I)
    y, work = zq4.moe_block(gu, dn, E, dev(x), D, I, dev(ids), dev(r), dev_status=status)
    torch.cuda.synchronize()
    group, h, z = zq4.moe_block_views(work, T, top_k, D, I)
    h_gpu = host_f16(h)
    h_ref, Sh, bad = oracle.moe_gate_up(gq, gs, E, x, 2 * I, D, ids)
    assert_within(h_gpu, h_ref, Sh, f"moe block gate_up T={T}")
    y_ref, S, bad2 = oracle.moe_down_combine(dq, ds, E, h_gpu, r, D, I, ids)
    assert_within(host_f16(y), y_ref, S, f"moe block down+combine T={T}")
    assert bad == bad2
    return y, work, group, bad


@pytest.mark.slow
@pytest.mark.parametrize("T", [1, 4, 16])
def test_moe_block_full_size(zq4, oracle, T):
    E, top_k = synth.MOE_EXPERTS, synth.MOE_TOP_K
    (N2, D), (Dn, I) = synth.MOE_GATE_UP, synth.MOE_DOWN
    assert N2 == 2 * I and Dn == D
    gq, gs = synth.weight("moe_gu", E * N2, D, 0)
    dq, ds = synth.weight("moe_dn", E * Dn, I, 0)
    rng = synth.rng_for("moe_route", 0, T)
    ids, r = synth.routing(rng, T, E, top_k)
    x = synth.activations(rng, T, D)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y, work, group, bad = _run(zq4, oracle, gq, gs, dq, ds, E, x, ids, r, D, I, status)
    assert bad == 0 and int(status.item()) == 0
    check_group(group, ids, E)
    first = host_f16(y).view(np.uint16).copy()
    gu, dn = _banks(zq4, gq, gs, dq, ds, E, D, I)
    y2, _ = zq4.moe_block(gu, dn, E, dev(x), D, I, dev(ids), dev(r))
    torch.cuda.synchronize()
    assert np.array_equal(first, host_f16(y2).view(np.uint16))


def test_moe_block_bad_ids_and_repeats(zq4, oracle):
    """Two slots with ids outside [0, E): flagged, their h rows zero, no
    contribution to the combine; an expert routed from several tokens (more
    than 16 pairs: two blocks of pairs)."""
    E, T, top_k, D, I = 16, 6, 4, 256, 256
    gq, gs = synth.weight("moeb_gu", E * 2 * I, D, 0)
    dq, ds = synth.weight("moeb_dn", E * D, I, 0)
    rng = synth.rng_for("moeb_route", T)
    ids, r = synth.routing(rng, T, E, top_k)
    ids = np.array(ids)
    ids[1, 2] = E
    ids[4, 0] = -3
    x = synth.activations(rng, T, D)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y, work, group, bad = _run(zq4, oracle, gq, gs, dq, ds, E, x, ids.astype(np.int32), r, D, I, status)
    assert bad == 2 and int(status.item()) & 1
    check_group(group, ids, E)
    _, h, _ = zq4.moe_block_views(work, T, top_k, D, I)
    assert torch.all(h[1, 2] == 0) and torch.all(h[4, 0] == 0)
    # one expert for every slot of every token: 24 pairs, two blocks
    ids2 = np.full((T, top_k), 5, np.int32)
    ids2[:, 1] = 7
    _run(zq4, oracle, gq, gs, dq, ds, E, x, ids2, r, D, I)


def test_moe_block_refuses_other_shapes(zq4):
    """D or I not a multiple of 256, or more than 256 (token, slot) pairs:
    ZQ4_ERR_SHAPE / ZQ4_ERR_UNSUPPORTED, nothing launched (the per-stage
    zq4_moe_gemv takes those shapes)."""
    E, D, I = 4, 256, 256
    gu = torch.zeros(E * 2 * I * D * 9 // 16, dtype=torch.uint8, device="cuda")
    dn = torch.zeros(E * D * I * 9 // 16, dtype=torch.uint8, device="cuda")
    x = torch.zeros((40, D), dtype=torch.float16, device="cuda")
    ids = torch.zeros((40, 8), dtype=torch.int32, device="cuda")
    r = torch.zeros((40, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(zq4.Zq4Error, match="UNSUPPORTED"):
        zq4.moe_block(gu, dn, E, x, D, I, ids, r)                       # 320 pairs
    with pytest.raises(zq4.Zq4Error, match="SHAPE"):
        zq4.moe_block(gu, dn, E, x[:2, :96].contiguous(), 96, I, ids[:2], r[:2])
