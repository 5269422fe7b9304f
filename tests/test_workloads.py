"""The workload shapes and byte counts the benchmark uses, pinned to the
Phi-3-mini weight table of the Zero TVM docs page (CPU only)."""
import os

import numpy as np

from int4_weight_only_q4f16_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _table():
    rows, extra = {}, {}
    with open(os.path.join(GOLDEN, "phi3_weight_shapes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if len(line) == 5:
                rows[line[0]] = tuple(int(v) for v in line[1:])
            elif len(line) == 2:
                extra[line[0]] = float(line[1])
    return rows, extra


def test_phi3_shapes_match_weight_table():
    rows, extra = _table()
    for name, N, K in synth.PHI3_LAYER + (synth.PHI3_LM_HEAD,):
        n, words, scales, per_layer = rows[name]
        assert (N, K // 8, K // 32) == (n, words, scales)
        assert per_layer == (0 if name == "lm_head" else 1)
    assert synth.PHI3_LAYERS == int(extra["layers"])


def test_phi3_bytes_per_token_about_2_09_gb():
    rows, extra = _table()
    total = 0
    for name, (n, words, scales, per_layer) in rows.items():
        b = n * (4 * words + 2 * scales)
        total += b * (int(extra["layers"]) if per_layer else 1)
    assert total == 2_093_838_336
    assert abs(total / 1e9 - extra["approx_total_gb"]) < 0.005


def test_generator_shapes_and_ranges():
    rng = synth.rng_for("t", 1)
    wq = synth.packed_codes(rng, 7, 96)
    sc = synth.group_scales(rng, 7, 96)
    x = synth.activations(rng, 3, 96)
    assert wq.shape == (7, 12) and wq.dtype == np.uint32
    assert sc.shape == (7, 3) and sc.dtype == np.float16 and np.all(sc >= 0)
    assert x.shape == (3, 96) and x.dtype == np.float16
    ids, r = synth.routing(rng, 5, 128, 8)
    assert ids.shape == (5, 8) and r.shape == (5, 8)
    for t in range(5):
        assert len(set(ids[t])) == 8 and ids[t].min() >= 0 and ids[t].max() < 128
    assert np.allclose(r.sum(axis=1), 1.0, atol=1e-6) and np.all(r > 0)
    # streams are reproducible and independent of each other
    a = synth.packed_codes(synth.rng_for("w", 3), 4, 64)
    b = synth.packed_codes(synth.rng_for("w", 3), 4, 64)
    c = synth.packed_codes(synth.rng_for("w", 4), 4, 64)
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_chained_stack_wiring_and_bytes():
    """DecodeStack(chain=True): every projection reads the previous output
    (o a view over the first M*K values of qkv's), only the first input is
    seeded, and the algorithmic bytes count each projection's input and
    output once, as for the unchained stack."""
    import torch
    from int4_weight_only_q4f16_gb300 import stack as st
    layer = (("qkv", 96, 64), ("o", 32, 64), ("gate_up", 128, 32), ("down", 64, 64))
    for M in (1, 3):
        s = st.DecodeStack(layer, 2, ("lm_head", 40, 64), M=M, device="cpu", chain=True)
        assert s.fresh == [(0, "qkv")]
        prev = None
        for l in range(2):
            for name, N, K in layer:
                x = s.input_for(l, name)
                assert tuple(x.shape) == (M, K)
                if prev is not None:
                    assert x.data_ptr() == s.y[prev].data_ptr()
                prev = (l, name)
        assert s.x[("head",)].data_ptr() == s.y[(1, "down")].data_ptr()
        plain = st.DecodeStack(layer, 2, ("lm_head", 40, 64), M=M, device="cpu")
        assert s.bytes_per_step() == plain.bytes_per_step()
        assert len(plain.fresh) == 2 * 3 + 1                       # qkv, o, gate_up per layer + head


def test_generator_distributions():
    """The input recipe: every nibble a uniform code 0..15, scales
    |N(0, 0.02)| (mean 0.02 sqrt(2/pi)), activations N(0, 1)."""
    rng = synth.rng_for("dist", 0)
    wq = synth.packed_codes(rng, 256, 256)
    for i in range(8):
        counts = np.bincount(((wq >> (4 * i)) & 0xF).ravel(), minlength=16)
        assert counts.size == 16 and np.all(np.abs(counts / counts.mean() - 1) < 0.15), (i, counts)
    sc = synth.group_scales(rng, 4096, 256).astype(np.float64)
    assert abs(sc.mean() / (0.02 * np.sqrt(2 / np.pi)) - 1) < 0.02
    x = synth.activations(rng, 64, 4096).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01


def test_unit_gain_scales_keep_the_activation_size():
    """Signed scales N(0, unit_gain_sigma(K)) keep the root mean square of a
    projection's output near that of its N(0, 1) input (E[(q - 7)^2] = 21.5
    for uniform codes), and the gate_up sigma does the same for silu(g) u."""
    import oracle
    o = oracle.get()
    K, N = 3072, 512
    x = synth.activations(synth.rng_for("ug_x"), 4, K)
    assert np.mean([(q - 7) ** 2 for q in range(16)]) == 21.5
    wq, sc = synth.weight("ug", N, K, 0, sigma=synth.unit_gain_sigma(K), signed=True)
    y, _ = o.gemv(wq, sc, x, N, K)
    assert abs(np.sqrt(np.mean(y * y)) - 1) < 0.1
    wq, sc = synth.weight("ug_gu", 2 * N, K, 0, sigma=synth.unit_gain_sigma(K, gate_up=True), signed=True)
    h, _ = o.gate_up_silu(wq, sc, x, 2 * N, K)
    assert abs(np.sqrt(np.mean(h * h)) - 1) < 0.15


def _definition_bytes(layer, layers, head, M):
    """Per projection: codes N K/2, scales N K/16, x read M K 2, y written
    M N_out 2 (N_out = N/2 for gate_up)."""
    def one(name, N, K):
        n_out = N // 2 if name == "gate_up" else N
        return N * K // 2 + N * K // 16 + M * K * 2 + M * n_out * 2
    return layers * sum(one(*p) for p in layer) + (one(*head) if head else 0)


def test_stack_bytes_follow_the_definition():
    """DecodeStack.bytes_per_step (the roofline numerator of the bench) is
    the algorithmic byte count, and the Phi-3 step at M = 1 moves
    2,096,530,048 bytes (2,093,838,336 of them packed weights)."""
    from int4_weight_only_q4f16_gb300 import stack as st
    layer = (("qkv", 96, 64), ("o", 32, 64), ("gate_up", 128, 32), ("down", 64, 64))
    head = ("lm_head", 40, 64)
    for M in (1, 4):
        s = st.DecodeStack(layer, 3, head, M=M, device="cpu")
        assert s.bytes_per_step() == _definition_bytes(layer, 3, head, M)
    phi3 = _definition_bytes(synth.PHI3_LAYER, synth.PHI3_LAYERS, synth.PHI3_LM_HEAD, 1)
    assert phi3 == 2_096_530_048
    assert _definition_bytes(synth.PHI3_LAYER, synth.PHI3_LAYERS, synth.PHI3_LM_HEAD, 0) == 2_093_838_336
    gate_up = [p for p in synth.PHI3_LAYER if p[0] == "gate_up"]
    assert _definition_bytes(gate_up, 1, None, 1) == 28_334_080      # the per-call roofline's launch
