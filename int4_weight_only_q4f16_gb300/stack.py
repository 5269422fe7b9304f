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

    def __init__(self, name, N, K, layer, device, keep_host, seed):
        self.name, self.N, self.K, self.layer = name, N, K, layer
        wq, sc = synth.weight(name, N, K, layer, seed=seed)
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
                 keep_host=False, seed=synth.MASTER_SEED, mode="calls"):
        """mode "calls": one zq4_gemv / zq4_gate_up_silu per projection on
        the canonical matrices; "seg": one zq4_gemv_seg / zq4_gate_up_silu_seg
        per projection on segmented copies made once; "plan": the whole step
        as one persistent launch (zq4_stack_run) on segmented copies."""
        self.M, self.device, self.n_layers = M, torch.device(device), n_layers
        self.mode = mode
        self.plan = None
        self.layers = []
        for l in range(n_layers):
            self.layers.append({name: Projection(name, N, K, l, self.device, keep_host, seed)
                                for name, N, K in layer_shapes})
        self.order = [name for name, _, _ in layer_shapes]
        self.head = Projection(head[0], head[1], head[2], 0, self.device, keep_host, seed) if head else None
        # activations: a fresh seeded input for every projection that does
        # not read another projection's output
        self.x, self.y = {}, {}
        for l, layer in enumerate(self.layers):
            for name in self.order:
                p = layer[name]
                if name != "down":
                    xa = synth.activations(synth.rng_for("x_" + name, l, M, seed=seed), M, p.K)
                    self.x[(l, name)] = _dev(xa, self.device)
                cols = p.N // 2 if name == "gate_up" else p.N
                self.y[(l, name)] = torch.empty((M, cols), dtype=torch.float16, device=self.device)
        if self.head:
            xa = synth.activations(synth.rng_for("x_head", 0, M, seed=seed), M, self.head.K)
            self.x[("head",)] = _dev(xa, self.device)
            self.y[("head",)] = torch.empty((M, self.head.N), dtype=torch.float16, device=self.device)
        self.graph = None

    # --- accounting ----------------------------------------------------------
    def weight_bytes(self) -> int:
        b = sum(p.nbytes for layer in self.layers for p in layer.values())
        return b + (self.head.nbytes if self.head else 0)

    def activation_bytes(self) -> int:
        return sum(t.numel() * 2 for t in self.x.values()) + \
            sum(t.numel() * 2 for t in self.y.values()) + \
            sum(self.y[(l, "gate_up")].numel() * 2 for l in range(self.n_layers)
                if (l, "gate_up") in self.y and "down" in self.order)

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
        return self.y[(l, "gate_up")] if name == "down" else self.x[(l, name)]

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
