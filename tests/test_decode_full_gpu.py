"""Full-size decode parity: every projection shape of the single-GEMV, Phi-3
and Qwen3-4B workloads, run through the C ABI exactly as the benchmark runs
it (same call, same M, same weights layout), compared with the CPU oracle on
sampled output rows (all of them for the single 3072 x 3072 GEMV).

Rows are sampled two per 16-row tile at random plus the first and last row,
so every tile and every CTA of the launch is checked; the gate_up rows are
sampled as (gate, up) pairs."""
import numpy as np
import pytest

from int4_weight_only_q4f16_gb300 import synth
from helpers import assert_within, dev, host_f16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zq4():
    from int4_weight_only_q4f16_gb300 import zq4 as m
    return m


def _sample_tiles(N, seed, per_tile=2):
    rng = np.random.default_rng(seed)
    T = (N + 15) // 16
    rows = [t * 16 + rng.integers(0, min(16, N - t * 16), per_tile) for t in range(T)]
    return np.unique(np.concatenate(rows + [[0, N - 1]]))


def test_single_gemv_3072_all_outputs(zq4, oracle):
    """The single GEMV workload, M = 1, N = K = 3072: every output."""
    N = K = 3072
    wq, sc = synth.weight("gemv3072", N, K, 0)
    x = synth.activations(synth.rng_for("x_gemv3072", 0), 1, K)
    y = host_f16(zq4.gemv(dev(wq), dev(sc), dev(x), N, K))
    y_ref, S = oracle.gemv(wq, sc, x, N, K)
    assert_within(y, y_ref, S, "gemv 3072")


PHI3 = [(name, N, K) for name, N, K in synth.PHI3_LAYER] + [synth.PHI3_LM_HEAD]
QWEN = [(name, N, K) for name, N, K in synth.QWEN3_4B_LAYER]


def _projection(zq4, oracle, name, N, K, M, tag):
    wq, sc = synth.weight(tag + name, N, K, 0)
    x = synth.activations(synth.rng_for("x_" + tag + name, M), M, K)
    W, Sd, X = dev(wq), dev(sc), dev(x)
    if name == "gate_up":
        h = host_f16(zq4.gate_up_silu(W, Sd, X, N, K))
        js = _sample_tiles(N // 2, N + M) // 1
        js = np.unique(np.clip(js, 0, N // 2 - 1))
        rows = np.stack([2 * js, 2 * js + 1], 1).ravel()
        h_ref, Sh = oracle.gate_up_silu(wq[rows], sc[rows], x, len(rows), K, interleaved=True)
        assert_within(h[:, js], h_ref, Sh, f"{tag}{name} M={M}")
    else:
        y = host_f16(zq4.gemv(W, Sd, X, N, K))
        rows = _sample_tiles(N, N + K + M)
        y_ref, S = oracle.gemv(wq, sc, x, N, K, rows=rows)
        assert_within(y[:, rows], y_ref, S, f"{tag}{name} M={M}")


@pytest.mark.parametrize("name,N,K", PHI3)
def test_phi3_projection_full_size(zq4, oracle, name, N, K):
    _projection(zq4, oracle, name, N, K, 1, "phi3_")


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("name,N,K", QWEN)
def test_qwen3_projection_full_size(zq4, oracle, name, N, K, M):
    _projection(zq4, oracle, name, N, K, M, "qwen3_")


def test_full_size_no_device_errors(zq4):
    assert zq4.device_errors(clear=True) == 0
