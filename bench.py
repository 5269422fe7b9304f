#!/usr/bin/env python
"""Benchmark of the q4f16_1 dequant-GEMV decode path on GB300.

Default workload: the Phi-3-mini-shaped decode layer stack at M = 1
(32 layers x {QKV 9216x3072, O 3072x3072, gate_up 16384x3072 -> SiLU*mul
8192, down 3072x8192} + LM head 32064x3072, every matrix distinct, seeded
synthetic weights; 2.09 GB of packed weights per token). One step = one
decode token through the whole stack: by default one cooperative launch of
the persistent step kernel over a plan of the 129 projections
(--stack-mode plan); --stack-mode calls issues one launch per projection.
The step is replayed from a CUDA graph. Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl zq4|reference]
                  [--workload phi3|gemv3072|qwen3|moe] [--m M] [--t T]

--impl reference times the CPU oracle (fp64, host cores) on a bounded
sample of the same workload and prints the same line with "impl":
"reference". Multi-GPU runs (torchrun) are independent replicas: every rank
runs its own stack; value = tokens of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "W4A16 dequant-GEMV achieved HBM GB/s (% of peak); Phi-3-shape decode tok/s"
L2_BYTES = 126 * 1024 * 1024
# the arithmetic of the GPU path: 4-bit weights dequantized exactly to f16,
# f16 activations, f16 x f16 products accumulated in fp32, f16 outputs
DTYPE = "w4a16: f16*f16 products, fp32 accumulate"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="zq4", choices=["zq4", "reference"])
    ap.add_argument("--workload", default="phi3",
                    choices=["phi3", "gemv3072", "qwen3", "moe", "kernel", "prefill", "lmhead", "oracle-table"])
    ap.add_argument("--stack-mode", default="plan", choices=["calls", "seg", "plan"],
                    help="phi3/qwen3: one launch per projection, or the whole step as one launch")
    ap.add_argument("--n", type=int, default=16384, help="rows of W (kernel workload)")
    ap.add_argument("--k", type=int, default=3072, help="columns of W (kernel workload)")
    ap.add_argument("--gate-up", action="store_true", help="kernel workload: fused gate_up + SiLU*mul")
    ap.add_argument("--qkv-rope", action="store_true",
                    help="kernel workload: the Phi-3 QKV projection (32 + 2 x 32 heads of 96) with RoPE and the "
                         "KV-cache write folded in (--n is taken as 9216)")
    ap.add_argument("--add-rmsnorm", action="store_true",
                    help="kernel workload: the GEMV with the residual add and RMSNorm folded in")
    ap.add_argument("--affine", action="store_true",
                    help="kernel workload: the MLX affine format (w = s q + b, groups of 64)")
    ap.add_argument("--copies", type=int, default=8, help="distinct weight copies (kernel workload)")
    ap.add_argument("--eager", action="store_true", help="kernel workload: plain launches, no graph")
    ap.add_argument("--m", type=int, default=1, help="tokens per step (qwen3 workload)")
    ap.add_argument("--chain", action="store_true",
                    help="phi3: every projection reads the previous one's output (a decode step's "
                         "dependencies without attention and norms) instead of a fresh seeded x")
    ap.add_argument("--layers", type=int, default=32,
                    help="layers of the Phi-3 stack (32 is the workload; fewer only for profiling)")
    ap.add_argument("--t", type=int, default=16, help="tokens per step (moe workload)")
    ap.add_argument("--moe-stages", action="store_true",
                    help="moe workload: the two per-stage zq4_moe_gemv calls instead of zq4_moe_block")
    ap.add_argument("--moe-block", action="store_true",
                    help="moe workload: zq4_moe_block at any T (the default uses it from 16 tokens)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="CPU time budget of the oracle sample")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only: barrier and max-of-times, no data path)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
            self.t0 = time.time()
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 10:
                continue
            if self.uuid and f[1] != self.uuid:
                continue
            rows.append(f)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2])]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(num(r[3]) or 0 for r in rows),
                "power_w_max": max(num(r[4]) or 0 for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# the source files that define each profiled kernel (its traffic figure is
# dropped as soon as one of them changes)
KERNEL_SOURCES = {
    "gate_up_phi3_M1": ("zq4_decode_tc.cu", "zq4_async.cuh", "zq4_common.cuh"),
    "stack_phi3_M1": ("zq4_stack.cu", "zq4_segment.cuh", "zq4_async.cuh", "zq4_common.cuh"),
    "step_phi3_M1": ("zq4_step.cu", "zq4_step.h", "zq4_segment.cuh", "zq4_async.cuh", "zq4_common.cuh"),
    "prefill_gate_up_M1024": ("zq4_prefill_tc.cu", "zq4_async.cuh", "zq4_common.cuh"),
}


def kernel_source_hash(tag: str):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "int4_weight_only_q4f16_gb300", "csrc")
    for name in KERNEL_SOURCES[tag]:
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel,
    or None when the kernel sources changed since that capture."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            v = v.strip()
            if v.startswith("`"):
                v = v[1:].split("`", 1)[0]
            vals[k.strip()] = v
    if vals.get("kernel_source_sha256_16") != kernel_source_hash(kernel_tag):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# CPU oracle baseline (test infrastructure; timed, never used for results)
# ---------------------------------------------------------------------------
def oracle_sample_rate(projs, budget_s: float, M: int = 1):
    """Run the fp64 oracle over row blocks of the given projections
    ((name, N, K, layer) in step order) until budget_s seconds of wall time;
    return (weight bytes covered per second, threads, description)."""
    import oracle
    from int4_weight_only_q4f16_gb300 import synth
    o = oracle.get()
    covered = 0
    spent = 0.0
    done = []
    for name, N, K, layer in projs:
        wq, sc = synth.weight(name, N, K, layer)
        x = synth.activations(synth.rng_for("cpu_x", layer), M, K)
        rows_per_call = max(1, min(N, 256))
        for r0 in range(0, N, rows_per_call):
            rows = np.arange(r0, min(N, r0 + rows_per_call))
            t0 = time.perf_counter()
            o.gemv(wq, sc, x, N, K, rows=rows)
            spent += time.perf_counter() - t0
            covered += rows.size * (K // 8 * 4 + K // 32 * 2)
            if spent >= budget_s:
                done.append(f"{name}[layer {layer}] rows 0..{rows[-1]}")
                return covered / spent, o.num_threads(), _sample_desc(done)
        done.append(f"{name}[layer {layer}]")
    return covered / max(spent, 1e-9), o.num_threads(), _sample_desc(done)


def _sample_desc(done):
    if len(done) <= 4:
        return "; ".join(done)
    return f"{len(done)} projections in step order ({done[0]} ... {done[-1]})"


def phi3_projs():
    from int4_weight_only_q4f16_gb300 import synth
    out = []
    for l in range(synth.PHI3_LAYERS):
        for name, N, K in synth.PHI3_LAYER:
            out.append((name, N, K, l))
        if l == 0:
            out.append((synth.PHI3_LM_HEAD[0],) + synth.PHI3_LM_HEAD[1:] + (0,))
    return out


# ---------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------
def time_replays(torch, fn, steps, stream):
    """Seconds for `steps` calls of fn issued on `stream`, CUDA events on
    that stream, synchronised on both sides."""
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            fn()
        stop.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(stop) / 1e3


def replay_on(torch, g, stream, n):
    with torch.cuda.stream(stream):
        for _ in range(n):
            g.replay()
    torch.cuda.synchronize()


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def run_phi3(args, torch, dist, peaks, peak_kind):
    from int4_weight_only_q4f16_gb300 import stack as stack_mod, synth, zq4
    dev = torch.device("cuda", dist.local)
    st = stack_mod.DecodeStack(synth.PHI3_LAYER, args.layers, synth.PHI3_LM_HEAD, M=1, device=dev,
                               mode=args.stack_mode, chain=args.chain)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        st.launch_step(stream)                         # eager step: sets kernel attributes
    torch.cuda.synchronize()
    head = st.y[("head",)].float()
    # (chained stacks: values shrink through the un-normed SiLU*mul of every layer and may reach 0;
    # the timing does not depend on them, and their parity is tested on a 3-layer chain)
    assert torch.isfinite(head).all() and (args.chain or head.abs().sum() > 0), "stack output is zero/non-finite"
    g = st.capture(stream)
    replay_on(torch, g, stream, args.warmup)

    sampler = ClockSampler(gpu_uuid(torch, dev) if dist.rank == 0 else None)
    if dist.rank == 0:
        sampler.start()
        time.sleep(0.3)
    dist.barrier()
    elapsed = time_replays(torch, g.replay, args.steps, stream)
    dist.barrier()
    clocks = sampler.stop() if dist.rank == 0 else None
    elapsed = dist.max(elapsed)
    step_s = elapsed / args.steps
    bytes_step = st.bytes_per_step()
    tok_s = dist.world * st.M / step_s

    if args.stack_mode == "plan":
        # the whole step is one launch of the step kernel: it is the dominant kernel
        achieved = bytes_step / step_s / 1e9
        kname, ktag = (("k_step<1> (whole decode step, one cooperative launch)", "step_phi3_M1")
                       if st.plan.plan.engine == 1 else
                       ("k_stack (whole decode step, one cooperative launch)", "stack_phi3_M1"))
        roofline = {"bound": "hbm", "kernel": kname,
                    "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)",
                    "traffic": profiled_traffic(ktag) if args.layers == 32 else None,
                    "bytes_per_launch": bytes_step, "avg_launch_us": round(step_s * 1e6, 3),
                    "launches_timed": args.steps}
    else:
        # dominant kernel: gate_up + SiLU*mul over the stack's distinct matrices
        gu = [st.layers[l]["gate_up"] for l in range(st.n_layers)]

        def gate_up_chain():
            for l, p in enumerate(gu):
                zq4.gate_up_silu(p.wq, p.sc, st.x[(l, "gate_up")], p.N, p.K, h=st.y[(l, "gate_up")],
                                 stream=stream)
        gg = capture(torch, gate_up_chain, stream)
        replay_on(torch, gg, stream, 3)
        reps = max(10, min(200, args.steps // 10))
        gu_s = time_replays(torch, gg.replay, reps, stream) / (reps * len(gu))
        p0 = gu[0]
        gu_bytes = p0.nbytes + st.M * p0.K * 2 + st.M * (p0.N // 2) * 2
        achieved = gu_bytes / gu_s / 1e9
        roofline = {"bound": "hbm", "kernel": "k_decode_tc<1,2> (gate_up + SiLU*mul, 16384x3072)",
                    "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)",
                    "traffic": profiled_traffic("gate_up_phi3_M1"),
                    "bytes_per_launch": gu_bytes, "avg_launch_us": round(gu_s * 1e6, 3),
                    "launches_timed": reps * len(gu)}

    e2e = None
    if not args.no_e2e:
        e2e = phi3_e2e(args, torch, st, stream, dist)

    cpu = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        rate, threads, desc = oracle_sample_rate(phi3_projs(), args.cpu_seconds)
        cpu = {"value": round(rate / st.weight_bytes(), 4), "unit": "tok/s", "cores": threads,
               "kind": "oracle",
               "sample": f"fp64 oracle GEMV over {desc} (~{args.cpu_seconds:.0f} s), scaled by "
                         f"weight bytes to one 2.09 GB token"}

    launches = st.launches_per_step() * args.steps
    line = {
        "metric": METRIC, "value": round(tok_s, 2), "unit": "tok/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "hbm_gbs": round(bytes_step / step_s / 1e9, 1),
        "hbm_frac_of_measured": round(bytes_step / step_s / 1e9 / peaks["hbm_gbs"], 4),
        "hbm_frac_of_8tbs": round(bytes_step / step_s / 8e12, 4),
        "config": {"workload": f"phi3-mini decode layer stack, M=1 ({args.layers} layers + LM head)",
                   "M": 1, "layers": args.layers, "launches_per_step": st.launches_per_step(),
                   "bytes_per_step": bytes_step, "weight_bytes_per_step": st.weight_bytes(),
                   "l2": f"inputs larger than L2: {st.weight_bytes() / 1e9:.2f} GB of distinct "
                         f"weights per step vs {L2_BYTES >> 20} MiB L2",
                   "parallelism": f"replicas x{dist.world}", "graph": "one CUDA graph per step",
                   "step": {"calls": "one launch per projection (zq4_gemv / zq4_gate_up_silu)",
                            "seg": "one launch per projection on segmented weights (zq4_gemv_seg / _gate_up_silu_seg)",
                            "plan": "whole step as one persistent launch (zq4_stack_run)"}[args.stack_mode],
                   "inputs": ("chained: each projection reads the previous one's output (o: a view over "
                              "qkv's output)" if args.chain else
                              "a fresh seeded x per projection, except down, which reads its layer's gate_up "
                              "output"),
                   "dependencies": ("stream order: every launch starts after the previous one completes"
                                    if args.stack_mode != "plan" else
                                    "ordered only where buffers meet: every projection waits for all of the one "
                                    "before it" if args.chain else
                                    "ordered only where buffers meet: down waits for all of its gate_up and runs "
                                    "after the next layer's qkv, o and gate_up, which touch none of its buffers"),
                   "arith": "int4 codes -> exact f16 (q-7); f16*f16 products, fp32 accumulate; "
                            "f16 out"},
        "clocks": clocks, "e2e": e2e, "gpu_launches": launches, "roofline": roofline,
        "cpu_baseline": cpu,
    }
    return line


def phi3_e2e(args, torch, st, stream, dist):
    """Same metric through the public API with host buffers: per step, copy
    every fresh activation from pinned host memory, replay, read the logits
    back to pinned host memory."""
    keys = list(st.fresh)                 # the seeded inputs; the rest are outputs of the step
    sizes = [st.x[k].numel() for k in keys]
    host_in = torch.empty(sum(sizes), dtype=torch.float16, pin_memory=True)
    off = 0
    for k, n in zip(keys, sizes):
        host_in[off:off + n].copy_(st.x[k].flatten().cpu())
        off += n
    dev_in = torch.empty_like(host_in, device=st.device)
    views, off = [], 0
    for k, n in zip(keys, sizes):
        views.append((st.x[k], dev_in[off:off + n].view_as(st.x[k])))
        off += n
    out = st.y[("head",)]
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    # the step's inputs are read from dev_in: rebind the stack's inputs to it
    saved, saved_plan = dict(st.x), st.plan
    for (k, _), (_, v) in zip(zip(keys, sizes), views):
        st.x[k] = v
    st.plan = None                     # plan mode: the job table must point at the rebound inputs
    with torch.cuda.stream(stream):
        st.launch_step(stream)
    torch.cuda.synchronize()
    g = st.capture(stream)
    steps = max(3, min(args.steps, 500))

    def one():
        with torch.cuda.stream(stream):
            dev_in.copy_(host_in, non_blocking=True)
            g.replay()
            host_out.copy_(out, non_blocking=True)
    for _ in range(3):
        one()
    torch.cuda.synchronize()
    dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    el = dist.max(time.perf_counter() - t0)
    st.x.update(saved)
    st.plan = saved_plan
    return {"value": round(dist.world * st.M * steps / el, 2), "unit": "tok/s",
            "h2d_bytes_per_step": int(host_in.numel() * 2),
            "d2h_bytes_per_step": int(host_out.numel() * 2), "steps": steps,
            "timer": "host wall clock around copies + replay, synchronised"}


def run_gemv3072(args, torch, dist, peaks, peak_kind):
    """Single 3072x3072 GEMV, M=1, rotating over distinct weight copies that
    together exceed 4x L2 (so every call reads HBM)."""
    from int4_weight_only_q4f16_gb300 import synth, zq4
    N = K = 3072
    copies = 128
    wq, sc = synth.weight("cfg0", N, K, 0)
    W = torch.from_numpy(wq.view(np.int32)).cuda().repeat(copies, 1).view(copies, N, K // 8)
    S = torch.from_numpy(sc).cuda().repeat(copies, 1).view(copies, N, K // 32)
    x = torch.from_numpy(synth.activations(synth.rng_for("cfg0x"), 1, K)).cuda()
    y = torch.empty((copies, 1, N), dtype=torch.float16, device="cuda")
    stream = torch.cuda.Stream()

    def chain():
        for c in range(copies):
            zq4.gemv(W[c], S[c], x, N, K, y=y[c], stream=stream)
    with torch.cuda.stream(stream):
        chain()
    g = capture(torch, chain, stream)
    replay_on(torch, g, stream, max(3, args.warmup))
    reps = max(5, min(args.steps // copies, 100))
    el = time_replays(torch, g.replay, reps, stream)
    per = el / (reps * copies)
    b = N * (K // 8) * 4 + N * (K // 32) * 2 + K * 2 + N * 2
    gbs = b / per / 1e9
    return {"metric": "single GEMV 3072x3072 M=1 achieved HBM GB/s", "value": round(gbs, 1),
            "unit": "GB/s", "us_per_call": round(per * 1e6, 3), "bytes_per_call": b,
            "frac_of_measured": round(gbs / peaks["hbm_gbs"], 4),
            "config": {"workload": "gemv 3072x3072 M=1", "copies": copies,
                       "l2": f"{copies} distinct copies ({copies * b / 1e6:.0f} MB) > 4x L2"}}


def run_lmhead(args, torch, dist, peaks, peak_kind):
    """The LM-head step of decode: Phi-3 LM head 32064x3072 at M = 1 with
    fp32 logits and the fused argmax (zq4_gemv_argmax), over rotating weight
    copies that together exceed 4x L2; the plain f16 GEMV of the same shape
    is timed beside it."""
    from int4_weight_only_q4f16_gb300 import synth, zq4
    _, N, K = synth.PHI3_LM_HEAD
    copies = 10
    wq, sc = synth.weight("lm_head", N, K, 0)
    W = torch.from_numpy(wq.view(np.int32)).cuda().repeat(copies, 1).view(copies, N, K // 8)
    S = torch.from_numpy(sc).cuda().repeat(copies, 1).view(copies, N, K // 32)
    x = torch.from_numpy(synth.activations(synth.rng_for("lmhead_x"), 1, K)).cuda()
    y32 = torch.empty((copies, 1, N), dtype=torch.float32, device="cuda")
    y16 = torch.empty((copies, 1, N), dtype=torch.float16, device="cuda")
    idx = torch.empty((copies, 1), dtype=torch.int32, device="cuda")
    mx = torch.empty((copies, 1), dtype=torch.float32, device="cuda")
    work = torch.zeros((copies, 9), dtype=torch.int64, device="cuda")
    stream = torch.cuda.Stream()

    def chain_argmax():
        for c in range(copies):
            zq4.gemv_argmax(W[c], S[c], x, N, K, y32=y32[c], idx=idx[c], maxval=mx[c], work=work[c],
                            stream=stream)

    def chain_plain():
        for c in range(copies):
            zq4.gemv(W[c], S[c], x, N, K, y=y16[c], stream=stream)
    res = {}
    for name, fn in (("argmax", chain_argmax), ("plain", chain_plain)):
        with torch.cuda.stream(stream):
            fn()
        g = capture(torch, fn, stream)
        replay_on(torch, g, stream, max(3, args.warmup))
        reps = max(5, min(args.steps // copies, 200))
        res[name] = time_replays(torch, g.replay, reps, stream) / (reps * copies)
    torch.cuda.synchronize()
    b = N * (K // 8) * 4 + N * (K // 32) * 2 + K * 2
    gbs = (b + N * 4) / res["argmax"] / 1e9
    return {"metric": "LM-head GEMV 32064x3072 M=1 with fp32 logits + fused argmax, achieved HBM GB/s",
            "value": round(gbs, 1), "unit": "GB/s", "us_per_call": round(res["argmax"] * 1e6, 3),
            "frac_of_measured": round(gbs / peaks["hbm_gbs"], 4),
            "plain_f16_gemv_us": round(res["plain"] * 1e6, 3),
            "argmax_token": int(idx[0, 0].item()),
            "config": {"workload": "Phi-3 LM head 32064x3072, M=1, argmax", "copies": copies,
                       "l2": f"{copies} distinct copies ({copies * b / 1e6:.0f} MB) > 4x L2"}}


def run_qwen3(args, torch, dist, peaks, peak_kind):
    from int4_weight_only_q4f16_gb300 import stack as stack_mod, zq4
    st = stack_mod.qwen3_4b_stack(M=args.m, mode=args.stack_mode)
    stream = torch.cuda.Stream()
    if st.mode == "plan":
        try:
            st.build_plan(stream)
        except zq4.Zq4Error as e:     # a plan the library cannot run as one launch
            if "UNSUPPORTED" not in str(e):
                raise
            st.mode = "calls"
    engine = {0: "k_stack", 1: "k_step", 2: "k_wide"}.get(st.plan.plan.engine) if st.mode == "plan" else None
    with torch.cuda.stream(stream):
        st.launch_step(stream)
    g = st.capture(stream)
    replay_on(torch, g, stream, max(3, args.warmup))
    steps = max(5, min(args.steps, 1000))
    el = time_replays(torch, g.replay, steps, stream)
    step = el / steps
    b = st.bytes_per_step()
    return {"metric": "Qwen3-4B-shape projection stack tokens/s", "value": round(st.M / step, 1),
            "unit": "tok/s", "M": st.M, "ms_per_step": round(step * 1e3, 4),
            "hbm_gbs": round(b / step / 1e9, 1), "frac_of_measured": round(b / step / 1e9 / peaks["hbm_gbs"], 4),
            "launches_per_step": st.launches_per_step(),
            "config": {"workload": f"qwen3-4b 36-layer projection stack, M={st.M}",
                       "bytes_per_step": b, "stack_mode": st.mode, "engine": engine}}


def run_moe(args, torch, dist, peaks, peak_kind):
    """MoE expert GEMV (gate_up+SiLU, down+combine), 128 experts, top-8,
    rotating over 4 distinct banks (> 4x L2 in total)."""
    from int4_weight_only_q4f16_gb300 import synth, zq4
    E, top_k, T = synth.MOE_EXPERTS, synth.MOE_TOP_K, args.t
    (N2, D), (Dn, I) = synth.MOE_GATE_UP, synth.MOE_DOWN
    banks = 4
    gq, gs, gbi, dq, ds, dbi, xs, ids, rs, hs, ys = [], [], [], [], [], [], [], [], [], [], []
    uniq_bytes = []
    aff = args.affine                            # MLX affine banks: a scale and a bias per 64 weights
    per_scale = 64 if aff else 32

    def to_dev(a, s):
        if aff:
            s = s[:, ::2].copy()
            return (torch.from_numpy(a.view(np.int32)).cuda(), torch.from_numpy(s).cuda(),
                    torch.from_numpy((-8.0 * s.astype(np.float32)).astype(np.float16)).cuda())
        return torch.from_numpy(a.view(np.int32)).cuda(), torch.from_numpy(s).cuda(), None
    for b in range(banks):
        w_, s_, b_ = to_dev(*synth.weight("moe_gu", E * N2, D, b))
        gq.append(w_)
        gs.append(s_)
        gbi.append(b_)
        w_, s_, b_ = to_dev(*synth.weight("moe_dn", E * Dn, I, b))
        dq.append(w_)
        ds.append(s_)
        dbi.append(b_)
        rng = synth.rng_for("moe_route", b, T)
        i_, r_ = synth.routing(rng, T, E, top_k)
        xs.append(torch.from_numpy(synth.activations(rng, T, D)).cuda())
        ids.append(torch.from_numpy(i_).cuda())
        rs.append(torch.from_numpy(r_).cuda())
        hs.append(torch.empty((T, top_k, N2 // 2), dtype=torch.float16, device="cuda"))
        ys.append(torch.empty((T, Dn), dtype=torch.float16, device="cuda"))
        nu = len(np.unique(i_))
        sb = (4 if aff else 2)                  # scale (+ bias) bytes per group
        uniq_bytes.append(nu * (N2 * (D // 8) * 4 + N2 * (D // per_scale) * sb + Dn * (I // 8) * 4 +
                                Dn * (I // per_scale) * sb))
    stream = torch.cuda.Stream()
    # the q4f16_1 block as one call (each touched expert read once per stage)
    # where it measured faster than the two per-stage calls (16 tokens: 30% of
    # HBM against 25%; at 1 and 4 tokens its three launches' fixed cost loses)
    block = not aff and not args.moe_stages and (T >= 16 or args.moe_block)
    works = [torch.zeros(zq4.moe_block_work_bytes(T, top_k, D, I), dtype=torch.uint8, device="cuda")
             for _ in range(banks)] if block else []
    # the block reads the banks in the segmented layout (same bytes, permuted; made once)
    gsegs = [zq4.prepare_weight(gq[b], gs[b], E * N2, D, zq4.PREP_SEGMENTED)[0] for b in range(banks)] if block else []
    dsegs = [zq4.prepare_weight(dq[b], ds[b], E * Dn, I, zq4.PREP_SEGMENTED)[0] for b in range(banks)] if block else []

    def chain():
        for b in range(banks):
            if block:
                zq4.moe_block(gsegs[b], dsegs[b], E, xs[b], D, I, ids[b], rs[b], y=ys[b], work=works[b],
                              stream=stream)
            elif aff:
                zq4.moe_gemv_affine(gq[b], gs[b], gbi[b], E, xs[b], N2, D, ids[b], zq4.MOE_GATE_UP_SILU, y=hs[b],
                                    stream=stream)
                zq4.moe_gemv_affine(dq[b], ds[b], dbi[b], E, hs[b], Dn, I, ids[b], zq4.MOE_DOWN_COMBINE,
                                    route_w=rs[b], y=ys[b], stream=stream)
            else:
                zq4.moe_gemv(gq[b], gs[b], E, xs[b], N2, D, ids[b], zq4.MOE_GATE_UP_SILU, y=hs[b],
                             stream=stream)
                zq4.moe_gemv(dq[b], ds[b], E, hs[b], Dn, I, ids[b], zq4.MOE_DOWN_COMBINE,
                             route_w=rs[b], y=ys[b], stream=stream)
    with torch.cuda.stream(stream):
        chain()
    g = capture(torch, chain, stream)
    replay_on(torch, g, stream, max(3, args.warmup))
    reps = max(5, min(args.steps, 500))
    el = time_replays(torch, g.replay, reps, stream)
    per = el / (reps * banks)
    ub = sum(uniq_bytes) / banks
    return {"metric": ("MLX affine " if aff else "") +
                      "MoE expert GEMV block (gate_up+SiLU, down+combine) GB/s over unique experts",
            "value": round(ub / per / 1e9, 1), "unit": "GB/s", "T": T, "us_per_block": round(per * 1e6, 3),
            "unique_expert_bytes": ub, "frac_of_measured": round(ub / per / 1e9 / peaks["hbm_gbs"], 4),
            "config": {"workload": f"MoE 128 experts top-8, T={T}", "banks": banks,
                       "path": "zq4_moe_block" if block else "zq4_moe_gemv stages"}}


def run_kernel(args, torch, dist, peaks, peak_kind):
    """One projection shape: `copies` distinct matrices called in turn (a CUDA
    graph of them, or plain launches with --eager, e.g. under a profiler)."""
    from int4_weight_only_q4f16_gb300 import synth, zq4
    N, K, M, C = args.n, args.k, args.m, args.copies
    gs = 64 if args.affine else 32                  # weights per scale
    wq, sc = synth.weight("kernel", N, K, 0)
    if args.affine:                                 # one scale and one bias per 64 weights
        sc = sc[:, ::2].copy()
        bi = (-8.0 * sc.astype(np.float32)).astype(np.float16)
        B = torch.from_numpy(bi).cuda().repeat(C, 1).view(C, N, K // gs)
    W = torch.from_numpy(wq.view(np.int32)).cuda().repeat(C, 1).view(C, N, K // 8)
    S = torch.from_numpy(sc).cuda().repeat(C, 1).view(C, N, K // gs)
    x = torch.from_numpy(synth.activations(synth.rng_for("kernel_x"), M, K)).cuda()
    cols = N // 2 if args.gate_up else N
    y = torch.empty((C, M, cols), dtype=torch.float16, device="cuda")
    stream = torch.cuda.Stream()
    if args.qkv_rope:
        Hh, Hk, Dh = 32, 32, 96
        assert N == (Hh + 2 * Hk) * Dh, "--qkv-rope takes --n 9216"
        n_slots = 4096
        kcs = [torch.zeros((n_slots, Hk * Dh), dtype=torch.float16, device="cuda") for _ in range(C)]
        vcs = [torch.zeros_like(kcs[0]) for _ in range(C)]
        posd = torch.full((M,), 1000, dtype=torch.int32, device="cuda")
        slotd = torch.arange(M, dtype=torch.int32, device="cuda")
        qo = torch.empty((C, M, Hh * Dh), dtype=torch.float16, device="cuda")

        def chain():
            for c in range(C):
                zq4.qkv_rope_append(W[c], S[c], x, K, Hh, Hk, Dh, 10000.0, posd, slotd, kcs[c], vcs[c], q_out=qo[c],
                                    stream=stream)
    elif args.add_rmsnorm:
        resid = torch.from_numpy(synth.activations(synth.rng_for("kernel_res"), M, N)).cuda()
        gam = torch.ones(N, dtype=torch.float16, device="cuda")
        y2 = torch.empty_like(y)
        works = [torch.zeros(zq4.add_rmsnorm_work_bytes(M, N), dtype=torch.uint8, device="cuda") for _ in range(C)]

        def chain():
            for c in range(C):
                zq4.gemv_add_rmsnorm(W[c], S[c], x, resid, gam, 1e-5, N, K, res_out=y[c], out=y2[c], work=works[c],
                                     stream=stream)
    elif args.affine:
        fa = zq4.gate_up_silu_affine if args.gate_up else zq4.gemv_affine

        def chain():
            for c in range(C):
                fa(W[c], S[c], B[c], x, N, K, y[c], stream=stream)
    else:
        f = zq4.gate_up_silu if args.gate_up else zq4.gemv

        def chain():
            for c in range(C):
                f(W[c], S[c], x, N, K, y[c], stream=stream)
    reps = max(1, args.steps // C)
    if args.eager:
        with torch.cuda.stream(stream):
            for _ in range(max(1, args.warmup)):
                chain()
        el = time_replays(torch, chain, reps, stream)
    else:
        with torch.cuda.stream(stream):
            chain()
        g = capture(torch, chain, stream)
        replay_on(torch, g, stream, max(3, args.warmup))
        el = time_replays(torch, g.replay, reps, stream)
    torch.cuda.synchronize()
    out_chk = qo if args.qkv_rope else y
    assert torch.isfinite(out_chk).all() and (out_chk != 0).any(), "kernel output zero/non-finite"
    per = el / (reps * C)
    b = N * (K // 8) * 4 + N * (K // gs) * 2 * (2 if args.affine else 1) + M * K * 2 + M * cols * 2
    if args.add_rmsnorm:
        b += M * N * 2 * 2 + N * 2              # + residual in, normalised out, gamma
    if args.qkv_rope:
        b += M * 8                              # + pos, slot (the outputs are the N columns already counted)
    kind = ("MLX affine " if args.affine else "") + ("gate_up+SiLU" if args.gate_up else "GEMV") + \
        (" + add + RMSNorm" if args.add_rmsnorm else "") + (" + RoPE + KV append" if args.qkv_rope else "")
    return {"metric": f"{kind} {N}x{K} M={M} achieved HBM GB/s",
            "value": round(b / per / 1e9, 1), "unit": "GB/s", "us_per_call": round(per * 1e6, 3),
            "bytes_per_call": b, "frac_of_measured": round(b / per / 1e9 / peaks["hbm_gbs"], 4),
            "config": {"workload": f"kernel {N}x{K} M={M}", "copies": C, "graph": not args.eager,
                       "l2": f"{C} distinct copies, {C * b / 1e6:.0f} MB"}}


def run_prefill(args, torch, dist, peaks, peak_kind):
    """The prefill-chunk GEMM workloads: 1024 tokens through the Phi-3 gate_up
    shape (16384 x 3072) and the down shape (3072 x 8192), each timed over
    distinct weight copies that together exceed L2. Reports TFLOP/s of the
    pair (2*M*N*K per GEMM) against the measured dense bf16 peak (f16 has the
    same nominal tensor rate)."""
    from int4_weight_only_q4f16_gb300 import synth, zq4
    M = 1024
    shapes = [("gate_up shape", 16384, 3072), ("down shape", 3072, 8192)]
    stream = torch.cuda.Stream()
    per_shape, tot_flop, tot_s = [], 0, 0.0
    for name, N, K in shapes:
        wbytes = N * (K // 8) * 4 + N * (K // 32) * 2
        copies = max(2, int(4 * L2_BYTES // wbytes) + 1)
        wq, sc = synth.weight("prefill_" + name, N, K, 0)
        W = torch.from_numpy(wq.view(np.int32)).cuda().repeat(copies, 1).view(copies, N, K // 8)
        S = torch.from_numpy(sc).cuda().repeat(copies, 1).view(copies, N, K // 32)
        x = torch.from_numpy(synth.activations(synth.rng_for("prefill_x", N, K), M, K)).cuda()
        y = torch.empty((copies, M, N), dtype=torch.float16, device="cuda")

        def chain():
            for c in range(copies):
                zq4.gemv(W[c], S[c], x, N, K, y=y[c], stream=stream)
        with torch.cuda.stream(stream):
            chain()
        g = capture(torch, chain, stream)
        replay_on(torch, g, stream, max(3, args.warmup))
        reps = max(3, min(args.steps // copies, 50))
        el = time_replays(torch, g.replay, reps, stream)
        torch.cuda.synchronize()
        assert torch.isfinite(y).all() and (y != 0).any(), "prefill output zero/non-finite"
        per = el / (reps * copies)
        flop = 2 * M * N * K
        per_shape.append({"shape": f"{M}x{N}x{K}", "name": name, "us_per_gemm": round(per * 1e6, 2),
                          "tflops": round(flop / per / 1e12, 1), "copies": copies,
                          "frac_of_measured_bf16": round(flop / per / 1e12 / peaks["bf16_tflops"], 4)})
        tot_flop += flop
        tot_s += per
        del W, S, y, g
        torch.cuda.empty_cache()
    tf = tot_flop / tot_s / 1e12
    best = max(per_shape, key=lambda d: d["tflops"])
    return {"metric": "prefill-chunk dequant GEMM TFLOP/s (M=1024, gate_up and down shapes)",
            "value": round(tf, 1), "unit": "TFLOP/s", "n_gpus": dist.world, "higher_is_better": True,
            "dtype": "f16 x f16 -> fp32", "data": "synthetic", "shapes": per_shape,
            "roofline": {"bound": "tensor", "kernel": "k_prefill (tcgen05 kind::f16, dequant into SMEM)",
                         "achieved": round(tf, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(tf / peaks["bf16_tflops"], 4),
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json bf16_tflops burst; f16 nominal = bf16)",
                         "traffic": profiled_traffic("prefill_gate_up_M1024"),
                         "traffic_note": "DRAM bytes of one gate_up-shape launch (ncu)",
                         "best_shape": best["shape"]},
            "config": {"workload": "prefill chunk, 1024 tokens, Phi-3 gate_up 16384x3072 and down 3072x8192",
                       "l2": "distinct weight copies per shape exceed 4x L2"}}


def run_reference(args, dist):
    """The CPU oracle on the host cores, timed on a bounded sample of the
    Phi-3 stack; each step covers the same row sample."""
    if dist.rank != 0:
        return None
    import oracle
    from int4_weight_only_q4f16_gb300 import synth
    o = oracle.get()
    # sample: 256 rows of each projection of layer 0 and of the LM head
    projs = [(n, N, K) for n, N, K in synth.PHI3_LAYER] + [synth.PHI3_LM_HEAD]
    data = []
    rows = 256
    for name, N, K in projs:
        wq, sc = synth.weight(name, N, K, 0)
        x = synth.activations(synth.rng_for("ref_x"), 1, K)
        data.append((wq, sc, x, N, K, np.arange(rows)))
    sample_bytes = sum(rows * (K // 8 * 4 + K // 32 * 2) for _, _, _, _, K, _ in data)
    token_bytes = sum(N * (K // 8 * 4 + K // 32 * 2) for _, N, K in synth.PHI3_LAYER) * synth.PHI3_LAYERS + \
        synth.PHI3_LM_HEAD[1] * (synth.PHI3_LM_HEAD[2] // 8 * 4 + synth.PHI3_LM_HEAD[2] // 32 * 2)

    def step():
        for wq, sc, x, N, K, r in data:
            o.gemv(wq, sc, x, N, K, rows=r)
    t0 = time.perf_counter()
    step()
    one = time.perf_counter() - t0
    budget = 150.0
    steps = args.steps
    scale = 1
    if one * (steps + args.warmup) > budget:       # keep the whole run within a few minutes
        steps = max(1, int(budget / one) - args.warmup)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    el = time.perf_counter() - t0
    per_step = el / steps
    tok_s = sample_bytes / per_step / token_bytes
    desc = (f"256 rows of each layer-0 projection (QKV, O, gate_up, down) and of the LM head "
            f"({sample_bytes / 1e6:.2f} MB of packed weights per step), scaled by weight bytes "
            f"to one {token_bytes / 1e9:.2f} GB token")
    return {"impl": "reference", "metric": METRIC, "value": round(tok_s, 5), "unit": "tok/s",
            "n_gpus": dist.world, "steps": steps, "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_step * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "phi3-mini decode layer stack, M=1 (32 layers + LM head)",
                       "M": 1, "layers": 32},
            "cpu_baseline": {"value": round(tok_s, 5), "unit": "tok/s", "cores": o.num_threads(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(tok_s, 5), "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_oracle_table(args):
    """The fp64 oracle timed on every workload, on one host thread and on all
    of them (a reported baseline; host CPU only, no GPU). Each cell runs a
    bounded sample and is scaled by weight bytes (GEMV stacks) or flops
    (prefill) to the workload's unit."""
    import oracle
    from int4_weight_only_q4f16_gb300 import synth
    o = oracle.get()
    all_threads = o.num_threads()
    budget = max(0.5, args.cpu_seconds / 10)

    def timed(fn, min_s):
        n, t = 0, 0.0
        while t < min_s or n == 0:
            t0 = time.perf_counter()
            fn()
            t += time.perf_counter() - t0
            n += 1
        return t / n

    def qwen_projs(M):
        return [(name, N, K, 0) for name, N, K in synth.QWEN3_4B_LAYER]

    cells = []
    for threads in (1, all_threads):
        used = o.set_num_threads(threads)
        # config 0: one 3072 x 3072 GEMV, M = 1
        wq, sc = synth.weight("gemv3072", 3072, 3072, 0)
        x = synth.activations(synth.rng_for("ot_x0"), 1, 3072)
        t = timed(lambda: o.gemv(wq, sc, x, 3072, 3072), budget)
        cells.append({"config": 0, "threads": used, "value": round(t * 1e6, 1), "unit": "us per call",
                      "sample": "whole call"})
        # config 1: the Phi-3 stack, M = 1 (rows of the projections in step order)
        rate, _, desc = oracle_sample_rate(phi3_projs(), 2 * budget)
        wb = sum(N * (K // 8 * 4 + K // 32 * 2) for _, N, K, _ in phi3_projs()[:4]) * synth.PHI3_LAYERS + \
            synth.PHI3_LM_HEAD[1] * (synth.PHI3_LM_HEAD[2] // 8 * 4 + synth.PHI3_LM_HEAD[2] // 32 * 2)
        cells.append({"config": 1, "threads": used, "value": round(wb / rate, 3), "unit": "s per token",
                      "sample": desc + ", scaled by weight bytes"})
        # config 2: the Qwen3-4B stack at M tokens (layer-0 rows, scaled to 36 layers)
        qb = sum(N * (K // 8 * 4 + K // 32 * 2) for _, N, K in synth.QWEN3_4B_LAYER) * synth.QWEN3_4B_LAYERS
        for M in (1, 2, 4, 8, 16):
            rate, _, desc = oracle_sample_rate(qwen_projs(M), budget, M=M)
            cells.append({"config": 2, "M": M, "threads": used, "value": round(qb / rate, 3),
                          "unit": "s per step", "tok_s": round(M * rate / qb, 4),
                          "sample": desc + ", scaled by weight bytes"})
        # config 3: the MoE block (gate_up + SiLU*mul, down + combine), T tokens, bank 0
        E, top_k = synth.MOE_EXPERTS, synth.MOE_TOP_K
        (N2, D), (Dn, I) = synth.MOE_GATE_UP, synth.MOE_DOWN
        gq, gs = synth.weight("moe_gu", E * N2, D, 0)
        dq, ds = synth.weight("moe_dn", E * Dn, I, 0)
        for T in (1, 4, 16):
            rng = synth.rng_for("moe_route", 0, T)
            ids, r = synth.routing(rng, T, E, top_k)
            xm = synth.activations(rng, T, D)

            def block():
                h, _, _ = o.moe_gate_up(gq, gs, E, xm, N2, D, ids)
                o.moe_down_combine(dq, ds, E, o.round_f16(h.ravel()).reshape(h.shape), r, Dn, I, ids)
            t = timed(block, budget)
            cells.append({"config": 3, "T": T, "threads": used, "value": round(t * 1e6, 1),
                          "unit": "us per block", "sample": "whole block"})
        # config 4: prefill GEMMs at M = 1024 (8 token rows, scaled by flops)
        for N, K in ((16384, 3072), (3072, 8192)):
            wq, sc = synth.weight("ot_prefill", N, K, 0)
            xs = synth.activations(synth.rng_for("ot_xp", N), 8, K)
            t = timed(lambda: o.gemv(wq, sc, xs, N, K), budget / 2) * (1024 / 8)
            cells.append({"config": 4, "shape": f"1024x{N}x{K}", "threads": used, "value": round(t, 2),
                          "unit": "s per call", "tflops": round(2 * 1024 * N * K / t / 1e12, 6),
                          "sample": "8 of the 1024 token rows, scaled by flops"})
    o.set_num_threads(all_threads)
    return {"impl": "oracle", "metric": "fp64 oracle time per workload unit (host CPU)",
            "cores": all_threads, "cells": cells}


def main():
    args = parse_args()
    dist = Dist()
    if args.workload == "oracle-table":
        print(json.dumps(run_oracle_table(args)), flush=True)
        return 0
    if args.impl == "reference":
        line = run_reference(args, dist)
        if line is not None:
            print(json.dumps(line), flush=True)
        dist.close()
        return 0
    import torch
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(dist.local)
    peaks, kind = measured_peaks()
    fn = {"phi3": run_phi3, "gemv3072": run_gemv3072, "qwen3": run_qwen3, "moe": run_moe,
          "kernel": run_kernel, "prefill": run_prefill, "lmhead": run_lmhead}[args.workload]
    line = fn(args, torch, dist, peaks, kind)
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
