"""Decode-step driver: a transformer-shaped stack of q4f16_1 projections.

One step runs, for every layer, the four projections of token-by-token
decode in stream order -- QKV GEMV, O GEMV, the fused gate_up + SiLU*mul,
and the down GEMV that consumes the gate_up output -- then the LM-head GEMV,
as in the decode loop of the Zero TVM docs page (section "Decode loop";
layer dispatch list in "RESEARCH.md", section "TVM's Per-Token Execution
Profile"). Attention, norms and the residual stream are not part of this
path: the QKV, O and gate_up inputs are independent seeded activations, the
down input is the gate_up output.

The step is issued through the zq4 C ABI on one CUDA stream and is captured
once into a CUDA graph; replaying the graph runs the step with no host work.
Every matrix of every layer is distinct, so a step streams the whole stack
from HBM (2.09 GB for the Phi-3-mini shapes, far above the L2 size).
"""
from __future__ import annotations

import numpy as np
import torch

from . import synth
from . import zq4


def _dev(a: np.ndarray, device) -> torch.Tensor:
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class Projection:
    """One q4f16_1 matrix on the device (+ optional host copy)."""

    def __init__(self, name, N, K, layer, device, keep_host, seed, sigma=0.02, signed=False):
        self.name, self.N, self.K, self.layer = name, N, K, layer
        wq, sc = synth.weight(name, N, K, layer, seed=seed, sigma=sigma, signed=signed)
        self.wq, self.sc = _dev(wq, device), _dev(sc, device)
        self.host = (wq, sc) if keep_host else None

    @property
    def nbytes(self) -> int:
        return self.N * (self.K // 8) * 4 + self.N * (self.K // 32) * 2


class DecodeStack:
    """Layer stack with per-layer shapes ``layer_shapes`` = ((name, N, K), ...)
    in execution order; the projection named "gate_up" runs the fused SiLU*mul
    epilogue and the one named "down" reads its output."""

    def __init__(self, layer_shapes, n_layers, head=None, M=1, device="cuda",
                 keep_host=False, seed=synth.MASTER_SEED, mode="calls", chain=False):
        """mode "calls": one zq4_gemv / zq4_gate_up_silu per projection on
        the canonical matrices; "seg": one zq4_gemv_seg / zq4_gate_up_silu_seg
        per projection on segmented copies made once; "plan": the whole step
        as one persistent launch (zq4_stack_run) on segmented copies.

        chain=False: every projection reads a fresh seeded x except "down",
        which reads its layer's gate_up output. chain=True: the dependencies
        of a decode step without its attention and norms -- each projection
        reads the output of the one before it (the first qkv a seeded x);
        where the widths differ (o after qkv) x is a view over the first
        M * K values of that output, standing in for attention, which reads
        all of it. Chained stacks draw signed scales N(0, sigma) with sigma =
        synth.unit_gain_sigma(K) instead of |N(0, 0.02)| (a stand-in for the
        norms between projections: activations stay O(1) through the
        layers)."""
        self.chain = chain
        self.M, self.device, self.n_layers = M, torch.device(device), n_layers
        self.mode = mode
        self.plan = None
        self.layers = []
        for l in range(n_layers):
            self.layers.append({name: Projection(name, N, K, l, self.device, keep_host, seed,
                                                 synth.unit_gain_sigma(K, name == "gate_up") if chain else 0.02,
                                                 signed=chain)
                                for name, N, K in layer_shapes})
        self.order = [name for name, _, _ in layer_shapes]
        self.head = Projection(head[0], head[1], head[2], 0, self.device, keep_host, seed,
                               synth.unit_gain_sigma(head[2]) if chain else 0.02, signed=chain) if head else None
        # activations: a fresh seeded input for every projection that does
        # not read another projection's output
        self.x, self.y = {}, {}
        self.fresh = []                               # keys of the seeded inputs (the rest are outputs)
        prev = None                                   # key of the previous output
        for l, layer in enumerate(self.layers):
            for name in self.order:
                p = layer[name]
                if chain and prev is not None:
                    y_prev = self.y[prev]
                    if y_prev.shape[1] != p.K and y_prev.numel() < M * p.K:
                        raise ValueError(f"chain: {name} reads {M * p.K} values, the previous output "
                                         f"holds {y_prev.numel()}")
                    self.x[(l, name)] = y_prev if y_prev.shape[1] == p.K else \
                        y_prev.view(-1)[:M * p.K].view(M, p.K)
                elif name != "down" or chain:
                    xa = synth.activations(synth.rng_for("x_" + name, l, M, seed=seed), M, p.K)
                    self.x[(l, name)] = _dev(xa, self.device)
                    self.fresh.append((l, name))
                cols = p.N // 2 if name == "gate_up" else p.N
                self.y[(l, name)] = torch.empty((M, cols), dtype=torch.float16, device=self.device)
                prev = (l, name)
        if self.head:
            if chain and prev is not None and self.y[prev].shape[1] == self.head.K:
                self.x[("head",)] = self.y[prev]
            else:
                xa = synth.activations(synth.rng_for("x_head", 0, M, seed=seed), M, self.head.K)
                self.x[("head",)] = _dev(xa, self.device)
                self.fresh.append(("head",))
            self.y[("head",)] = torch.empty((M, self.head.N), dtype=torch.float16, device=self.device)
        self.graph = None

    # --- accounting ----------------------------------------------------------
    def weight_bytes(self) -> int:
        b = sum(p.nbytes for layer in self.layers for p in layer.values())
        return b + (self.head.nbytes if self.head else 0)

    def activation_bytes(self) -> int:
        """Every projection's x read once and y written once."""
        return sum(self.input_for(k[0], k[1]).numel() * 2 if len(k) == 2 else self.x[k].numel() * 2
                   for k in self.y) + sum(t.numel() * 2 for t in self.y.values())

    def bytes_per_step(self) -> int:
        """Algorithmic bytes: every packed weight and scale once, every
        activation read and every output written once."""
        return self.weight_bytes() + self.activation_bytes()

    def launches_per_step(self) -> int:
        if self.mode == "plan":
            return 1
        if self.mode == "seg":
            return len(self.jobs())
        per_layer = 0
        for name in self.order:
            p = self.layers[0][name]
            per_layer += -(-self.M // zq4_tokens_per_launch(self.M, p.K))
        head = -(-self.M // zq4_tokens_per_launch(self.M, self.head.K)) if self.head else 0
        return per_layer * self.n_layers + head

    # --- execution -----------------------------------------------------------
    def input_for(self, l, name):
        if (l, name) in self.x:
            return self.x[(l, name)]
        return self.y[(l, "gate_up")]                  # down, unchained

    def jobs(self):
        """(wq, scales, x, y, N, K, gate_up) of every projection in step order."""
        out = []
        for l, layer in enumerate(self.layers):
            for name in self.order:
                p = layer[name]
                out.append((p.wq, p.sc, self.input_for(l, name), self.y[(l, name)], p.N, p.K,
                            name == "gate_up"))
        if self.head:
            out.append((self.head.wq, self.head.sc, self.x[("head",)], self.y[("head",)],
                        self.head.N, self.head.K, False))
        return out

    def build_plan(self, stream=None):
        """Segmented copies of every matrix (kept on the projections) and the
        one-launch plan over them."""
        pjobs = [(seg, x, y, N, K, gate_up)
                 for seg, (wq, sc, x, y, N, K, gate_up) in zip(self.segmented(stream), self.jobs())]
        self.plan = zq4.StackPlan(pjobs, self.M, stream=stream)
        return self.plan

    def segmented(self, stream=None):
        """Segmented copies of every matrix, in step order (made once)."""
        if getattr(self, "_seg", None) is None:
            self._seg = [zq4.prepare_weight(wq, sc, N, K, zq4.PREP_SEGMENTED, stream=stream)[0]
                         for wq, sc, x, y, N, K, gate_up in self.jobs()]
        return self._seg

    def launch_step(self, stream=None):
        if self.mode == "plan":
            if self.plan is None:
                self.build_plan(stream)
            self.plan.run(stream)
            return
        if self.mode == "seg":
            for seg, (wq, sc, x, y, N, K, gate_up) in zip(self.segmented(stream), self.jobs()):
                if gate_up:
                    zq4.gate_up_silu_seg(seg, x, N, K, h=y, stream=stream)
                else:
                    zq4.gemv_seg(seg, x, N, K, y=y, stream=stream)
            return
        for l, layer in enumerate(self.layers):
            for name in self.order:
                p = layer[name]
                x, y = self.input_for(l, name), self.y[(l, name)]
                if name == "gate_up":
                    zq4.gate_up_silu(p.wq, p.sc, x, p.N, p.K, h=y, stream=stream)
                else:
                    zq4.gemv(p.wq, p.sc, x, p.N, p.K, y=y, stream=stream)
        if self.head:
            zq4.gemv(self.head.wq, self.head.sc, self.x[("head",)], self.head.N, self.head.K,
                     y=self.y[("head",)], stream=stream)

    def capture(self, stream: torch.cuda.Stream):
        """Capture one step into a CUDA graph on ``stream`` (call after one
        eager step so that kernel attributes are already set)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.launch_step(stream)
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()


def zq4_tokens_per_launch(M: int, K: int) -> int:
    """Activation rows one decode launch handles (mirrors the library's
    choice, used only to count launches)."""
    mt = 8
    while mt > 1 and (mt > M or mt * K * 2 > 227 * 1024):
        mt //= 2
    return mt


def phi3_stack(**kw) -> DecodeStack:
    return DecodeStack(synth.PHI3_LAYER, synth.PHI3_LAYERS, synth.PHI3_LM_HEAD, **kw)


def qwen3_4b_stack(M=1, **kw) -> DecodeStack:
    return DecodeStack(synth.QWEN3_4B_LAYER, synth.QWEN3_4B_LAYERS, None, M=M, **kw)
