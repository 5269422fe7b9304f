"""The LM-head step (zq4_gemv_argmax): fp32 logits against the CPU oracle,
and the argmax decided in the kernel's own precision: it must be exactly
the oracle's argmax (lowest index on ties) of the logits the kernel
returned, and that logit must be within the parity bound of the true
maximum. Also: ties, a planted maximum in every tile position, several
tokens, the shape of the Phi-3 LM head at full size, and argument checks."""
import numpy as np
import pytest
import torch

from int4_weight_only_q4f16_gb300 import synth
from helpers import assert_within, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zq4():
    from int4_weight_only_q4f16_gb300 import zq4 as m
    return m


def _run(zq4, wq, sc, x, N, K, logits=True, work=None):
    idx, mx, y32 = zq4.gemv_argmax(dev(wq), dev(sc), dev(x), N, K, logits=logits, work=work)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), mx.cpu().numpy(), (y32.cpu().numpy() if y32 is not None else None)


@pytest.mark.parametrize("M,N,K", [(1, 333, 512), (3, 1000, 768), (8, 2049, 1024), (13, 517, 256),
                                   (40, 300, 512)])
def test_logits_and_argmax_match_oracle(zq4, oracle, M, N, K):
    wq, sc = synth.weight("lmh", N, K, M)
    x = synth.activations(synth.rng_for("lmh_x", M, N, K), M, K)
    idx, mx, y32 = _run(zq4, wq, sc, x, N, K)
    y_ref, S = oracle.gemv(wq, sc, x, N, K)
    assert_within(y32, y_ref, S, f"logits M={M} N={N} K={K}")
    assert np.array_equal(idx, oracle.argmax(y32.astype(np.float64)))
    assert np.array_equal(mx, y32[np.arange(M), idx])
    # the chosen logit is a true maximum within the bound
    tol = np.ldexp(np.abs(y_ref), -10) + 1e-4 * S
    for m in range(M):
        assert y_ref[m, idx[m]] + tol[m, idx[m]] >= (y_ref[m] - tol[m]).max()


def test_argmax_without_logits_and_planted_maxima(zq4, oracle):
    """One row made clearly largest for each token, in every position of a
    16-row tile and in the ragged last tile; the logits are not stored, and
    one work buffer serves every call (each call leaves it zero)."""
    N, K = 16 * 9 + 5, 512
    wq, sc = synth.weight("lmh_plant", N, K, 0)
    rows = [0, 1, 7, 8, 15, 16, 31, 100, N - 1]
    M = len(rows)
    x = np.zeros((M, K), np.float16)
    x[:, 0] = 1.0                               # y[m, n] = w[n, 0]
    wq2 = wq.copy()
    sc2 = sc.copy()
    sc2[:, 0] = np.float16(0.001)
    for n in range(N):                          # codes of column 0: 7 (zero) everywhere ...
        wq2[n, 0] = (wq2[n, 0] & ~np.uint32(0xF)) | np.uint32(7)
    idx_all = []
    work = torch.zeros(9, dtype=torch.int64, device="cuda")
    for m, r in enumerate(rows):
        w = wq2.copy()
        w[r, 0] = (w[r, 0] & ~np.uint32(0xF)) | np.uint32(15)   # ... but row r: +8 * scale
        idx, mx, y32 = _run(zq4, w, sc2, x[m:m + 1], N, K, logits=False, work=work)
        assert y32 is None
        assert idx[0] == r, (r, idx)
        assert mx[0] == np.float32(8 * float(np.float16(0.001)))
        idx_all.append(idx[0])
    assert idx_all == rows
    assert torch.count_nonzero(work).item() == 0


def test_argmax_ties_go_to_lowest_index(zq4):
    """Every logit equal (all codes 7 -> all logits exactly 0): index 0."""
    N, K, M = 1000, 256, 4
    rng = synth.rng_for("lmh_tie")
    wq = np.full((N, K // 8), 0x77777777, np.uint32)
    sc = synth.group_scales(rng, N, K)
    x = synth.activations(rng, M, K)
    idx, mx, y32 = _run(zq4, wq, sc, x, N, K)
    assert np.all(y32 == 0) and np.all(idx == 0) and np.all(mx == 0)


def test_phi3_lm_head_full_size(zq4, oracle):
    """32064 x 3072 at M = 1 and 2: sampled logits against the oracle and the
    argmax against the oracle's argmax of all returned logits."""
    N, K = synth.PHI3_LM_HEAD[1], synth.PHI3_LM_HEAD[2]
    wq, sc = synth.weight("lm_head", N, K, 0)
    for M in (1, 2):
        x = synth.activations(synth.rng_for("lmh_full", M), M, K)
        idx, mx, y32 = _run(zq4, wq, sc, x, N, K)
        rows = np.unique(np.concatenate([np.arange(0, N, 997), idx]))
        y_ref, S = oracle.gemv(wq, sc, x, N, K, rows=rows)
        assert_within(y32[:, rows], y_ref, S, f"LM head M={M}")
        assert np.array_equal(idx, oracle.argmax(y32.astype(np.float64)))


def test_argmax_rejects_bad_arguments(zq4):
    N, K = 64, 256
    wq, sc = synth.weight("lmh_bad", N, K, 0)
    W, S = dev(wq), dev(sc)
    x = dev(synth.activations(synth.rng_for("lmh_bad_x"), 1, K))
    with pytest.raises(zq4.Zq4Error, match="UNSUPPORTED"):      # K not a multiple of 256
        wq3, sc3 = synth.weight("lmh_bad3", N, 288, 0)
        zq4.gemv_argmax(dev(wq3), dev(sc3), dev(synth.activations(synth.rng_for("b3"), 1, 288)), N, 288)
    x65 = dev(synth.activations(synth.rng_for("lmh_65"), 65, K))
    with pytest.raises(zq4.Zq4Error, match="SHAPE"):             # M > 64
        zq4.gemv_argmax(W, S, x65, N, K)
    y32 = torch.empty((1, N), dtype=torch.float32, device="cuda")
    with pytest.raises(zq4.Zq4Error, match="OVERLAP"):           # logits over the work buffer
        zq4.gemv_argmax(W, S, x, N, K, y32=y32, work=y32.view(torch.int64)[:9])
    assert zq4.device_errors(clear=True) == 0
