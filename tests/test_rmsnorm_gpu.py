"""GPU parity of zq4_gemv_add_rmsnorm (the O / down projection with the
residual add and RMSNorm folded in as a tail reduction) against the CPU
oracle. r = resid + x W^T is held to the GEMV bar |r - r_ref| <= 2^-10 |r_ref|
+ 1e-4 S + 2^-25; the normalised output to 2^-10 |out_ref| + Tn + 2^-25, Tn
the oracle's first-order propagation of r's bar through the norm."""
import numpy as np
import pytest
import torch

from int4_weight_only_q4f16_gb300 import synth
from helpers import assert_within, dev, host_f16

pytestmark = pytest.mark.gpu


def _case(tag, M, N, K):
    rng = synth.rng_for(tag, M, N, K)
    wq, sc = synth.packed_codes(rng, N, K), synth.group_scales(rng, N, K)
    x = synth.activations(rng, M, K)
    res = synth.activations(rng, M, N)
    gam = (1.0 + 0.1 * rng.standard_normal(N)).astype(np.float16)
    return wq, sc, x, res, gam


@pytest.mark.parametrize("M,N,K", [(1, 3072, 3072), (1, 3072, 8192), (3, 333, 256), (8, 1000, 512),
                                   (16, 2000, 1024), (17, 3072, 3072), (11, 64, 96)])
def test_add_rmsnorm_matches_oracle(oracle, M, N, K):
    from int4_weight_only_q4f16_gb300 import zq4
    wq, sc, x, res, gam = _case("addnorm", M, N, K)
    eps = 1e-5
    res_out, out = zq4.gemv_add_rmsnorm(dev(wq), dev(sc), dev(x), dev(res), dev(gam), eps, N, K)
    r_ref, o_ref, S, Tn = oracle.gemv_add_rmsnorm(wq, sc, x, res, gam, eps, N, K)
    assert_within(host_f16(res_out), r_ref, S, f"residual M={M} N={N} K={K}")
    bound = np.ldexp(np.abs(o_ref), -10) + Tn + 2.0 ** -25
    assert_within(host_f16(out), o_ref, S, f"normalised M={M} N={N} K={K}", bound=bound)


def test_add_rmsnorm_repeated_calls_identical_and_work_left_zero():
    from int4_weight_only_q4f16_gb300 import zq4
    M, N, K = 9, 3072, 3072
    wq, sc, x, res, gam = (dev(a) for a in _case("addnorm_rep", M, N, K))
    work = torch.zeros(zq4.add_rmsnorm_work_bytes(M, N), dtype=torch.uint8, device="cuda")
    a1, b1 = zq4.gemv_add_rmsnorm(wq, sc, x, res, gam, 1e-6, N, K, work=work)
    a1, b1 = a1.clone(), b1.clone()
    for _ in range(3):
        a2, b2 = zq4.gemv_add_rmsnorm(wq, sc, x, res, gam, 1e-6, N, K, work=work)
        assert torch.equal(a1.view(torch.int16), a2.view(torch.int16))
        assert torch.equal(b1.view(torch.int16), b2.view(torch.int16))
    torch.cuda.synchronize()
    assert int(work[:16].view(torch.int32).abs().sum()) == 0


def test_add_rmsnorm_zero_weights_pass_the_residual_exactly(oracle):
    """All codes 7: r is the residual, so the new residual is it bit for bit."""
    from int4_weight_only_q4f16_gb300 import zq4
    M, N, K = 2, 500, 256
    _, sc, x, res, gam = _case("addnorm_zero", M, N, K)
    wq = np.full((N, K // 8), 0x77777777, np.uint32)
    res_out, out = zq4.gemv_add_rmsnorm(dev(wq), dev(sc), dev(x), dev(res), dev(gam), 0.5, N, K)
    assert np.array_equal(host_f16(res_out).view(np.uint16), res.view(np.uint16))
    r_ref, o_ref, S, Tn = oracle.gemv_add_rmsnorm(wq, sc, x, res, gam, 0.5, N, K)
    bound = np.ldexp(np.abs(o_ref), -10) + Tn + 2.0 ** -25
    assert_within(host_f16(out), o_ref, S, "normalised, W = 0", bound=bound)
