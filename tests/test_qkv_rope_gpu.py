"""GPU parity of zq4_qkv_rope_append (QKV projection, RoPE over the
(i, i + D/2) pairs of each Q / K head, K and V written to the cache rows of
each token's slot) against the CPU oracle. Bound per output:
2^-10 A + 1e-4 S + 2^-25 with A = |a| + |b| and S = S_a + S_b of its RoPE
pair (|y| and the row's own S for V): the GEMV bar of the two dot products
carried through the rotation (|cos|, |sin| <= 1); f16 rounding of the
output is within 2^-11 A."""
import numpy as np
import pytest
import torch

from int4_weight_only_q4f16_gb300 import synth
from helpers import assert_within, dev, host_f16

pytestmark = pytest.mark.gpu


def _case(H, Hkv, D, K, M, seed):
    rng = synth.rng_for("qkv_rope", H, Hkv, D, K, M, seed)
    N = (H + 2 * Hkv) * D
    return rng, synth.packed_codes(rng, N, K), synth.group_scales(rng, N, K), synth.activations(rng, M, K)


@pytest.mark.parametrize("H,Hkv,D,K,M", [(32, 32, 96, 3072, 1), (8, 2, 64, 512, 3), (2, 1, 8, 64, 9),
                                         (4, 4, 128, 2560, 2), (8, 2, 64, 1024, 16), (4, 2, 96, 768, 17)])
def test_qkv_rope_append_matches_oracle(oracle, H, Hkv, D, K, M):
    from int4_weight_only_q4f16_gb300 import zq4
    rng, wq, sc, x = _case(H, Hkv, D, K, M, 0)
    n_slots = M + 7
    pos = rng.integers(0, 4096, M).astype(np.int32)
    pos[0] = 4095
    slot = rng.permutation(n_slots)[:M].astype(np.int32)
    kc = torch.full((n_slots, Hkv * D), float("nan"), dtype=torch.float16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = zq4.qkv_rope_append(dev(wq), dev(sc), dev(x), K, H, Hkv, D, 10000.0, dev(pos), dev(slot), kc, vc,
                            dev_status=status)
    o = oracle.qkv_rope(wq, sc, x, K, H, Hkv, D, 10000.0, pos)
    for name, got in (("q", host_f16(q)), ("k", host_f16(kc)[slot]), ("v", host_f16(vc)[slot])):
        bound = np.ldexp(o["A_" + name], -10) + 1e-4 * o["S_" + name] + 2.0 ** -25
        assert_within(got, o[name], o["S_" + name], f"{name} H={H} Hkv={Hkv} D={D} K={K} M={M}", bound=bound)
    untouched = np.setdiff1d(np.arange(n_slots), slot)
    assert np.all(np.isnan(host_f16(kc)[untouched])) and np.all(np.isnan(host_f16(vc)[untouched]))
    assert int(status.item()) == 0


@pytest.mark.parametrize("D,K", [(16, 128), (32, 256)])      # CUDA-core and tensor-core kernels
def test_qkv_rope_bad_slot_is_reported_and_skipped(oracle, D, K):
    from int4_weight_only_q4f16_gb300 import zq4
    H, Hkv, M = 4, 2, 3
    rng, wq, sc, x = _case(H, Hkv, D, K, M, 1)
    n_slots = 4
    pos = np.array([1, 2, 3], np.int32)
    slot = np.array([2, n_slots, 0], np.int32)                 # token 1's slot is out of range
    kc = torch.zeros((n_slots, Hkv * D), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    zq4.qkv_rope_append(dev(wq), dev(sc), dev(x), K, H, Hkv, D, 10000.0, dev(pos), dev(slot), kc, vc,
                        dev_status=status)
    assert int(status.item()) & zq4.DEV_BAD_SLOT
    o = oracle.qkv_rope(wq, sc, x, K, H, Hkv, D, 10000.0, pos)
    got = host_f16(kc)
    for m, sl in ((0, 2), (2, 0)):
        bound = np.ldexp(o["A_k"][m], -10) + 1e-4 * o["S_k"][m] + 2.0 ** -25
        assert_within(got[sl][None], o["k"][m][None], o["S_k"][m][None], "k", bound=bound[None])
    assert np.all(got[[1, 3]] == 0)                            # rows no token wrote
