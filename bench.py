"""Benchmark: INT4 weight-only MatMulNBits decode step on GB300.

Workload: one batch-1 decode step of Qwen3-4B's projections (M = 1, bf16
activations ~ N(0,1), block size 128, no zero points (8), bf16 scales
U[0.002, 0.01]): q 2560->4096, k/v 2560->1024, o 4096->2560, gate/up
2560->9728, down 9728->2560, for 36 layers, plus lm_head 2560->151936 —
253 weights and 2.08 GB of algorithmic bytes per step, each weight with its
own seeded codes and scales, all resident in HBM before timing.

The step follows the model's data flow: q, k and v read one activation row
and run as one fused-N call (mnb_matmul_grouped); gate and up run as one
gated-MLP call that stores SiLU(gate) * up (mnb_matmul_gate_up); o, down
and lm_head each read their own row. That is 4 calls per layer and 145 per
step, recorded once by the library as one CUDA graph (mnb_graph_build) and
run with one mnb_graph_run per step; `e2e` runs it with
mnb_graph_run_from_host, which copies the step's activation rows in from
pinned host memory and its outputs back every step. The step's bytes exceed
the 129 MB L2 many times over, so no flush is needed.

Also measured after the headline's timed region, each with its roofline,
an oracle baseline and a clock record: the prefill GEMM at M = 2048 and
M = 512 over the seven Qwen3-4B projection shapes (TFLOP/s), the Qwen3-0.6B
decode step (fp32 activations, bs 32, zero points), the single
1024 x 3072 GEMV (cold and hot L2) and a condensed GEMV / tensor-core
crossover; and the same step as one persistent chain launch.

`--impl reference` times the CPU oracle on a bounded sample of the same
workload instead (there is no runnable reference implementation of this
operator; the oracle is the reference arm).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT4 decode GEMV GB/s and % HBM peak (M=1); prefill TFLOP/s (M=2048)"
WORKLOAD = "Qwen3-4B decode step projections, M=1, bf16 A, bs 128, no zp"


# DRAM traffic of the decode kernel relative to its algorithmic bytes, from
# an ncu capture of three launches of the Qwen3-4B gate projection (9728 x
# 2560, bs 128; dram__bytes_read.sum + dram__bytes_write.sum, median
# 12,930,048 B for 12,865,536 algorithmic), scaled to the step's mean launch;
# valid only for the decode-kernel sources it was measured on.
STEP_TRAFFIC = {
    "ratio": 12930048 / 12865536,
    "sources": ("gemv.cu", "mnb_common.cuh", "mnb_launch.h"),
    "sha256": "7e836f0e9ac4775f9e39585695f7020438442d61cdb344768b0f8165343b6d30",
}


def step_traffic(algo_bytes_per_launch):
    import hashlib
    h = hashlib.sha256()
    for f in STEP_TRAFFIC["sources"]:
        with open(os.path.join(ROOT, "int4_weight_only_matmulnbits_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != STEP_TRAFFIC["sha256"]:
        return None
    return round(STEP_TRAFFIC["ratio"] * algo_bytes_per_launch)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_path: str | None = None):
        import tempfile
        self.gpu = gpu_index
        self.proc = None
        # The raw samples go to the caller's file (--clock-log) or a private
        # temporary file; only their summary enters the JSON line.
        self.out = log_path or os.path.join(tempfile.mkdtemp(prefix="mnb_clocks_"),
                                            f"clocks_gpu{gpu_index}.csv")

    def start(self):
        try:
            self.f = open(self.out, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.out) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for name, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# CPU oracle leg
# ----------------------------------------------------------------------------

def oracle_sample(budget_s: float, seed_base: int = 3000, spec=None):
    """Times the oracle (single thread) over a decode step's projections in
    order until about budget_s seconds of CPU work; returns (bytes, seconds,
    description). spec: the step (default: the Qwen3-4B step)."""
    import torch

    import oracle
    from int4_weight_only_matmulnbits_gb300 import workloads
    spec = spec or STEP_4B
    model = getattr(workloads, spec["model"])
    adt = torch.float32 if spec["a_dtype"] == "f32" else torch.bfloat16
    oracle.load()
    projs = [(l, p) for l in range(model["layers"]) for p in model["projections"]]
    done_bytes, spent, names = 0, 0.0, []
    for i, (layer, p) in enumerate(projs):
        prob = workloads.make_problem(1, p.N, p.K, spec["bs"], dtype=adt, zero_points=spec["zp"],
                                      seed=seed_base + i, scale_range=spec["scale_range"])
        if spec["scale_dtype"] == "f32":
            prob.scales = prob.scales.float()
        t0 = time.perf_counter()
        oracle.matmulnbits(prob.A, prob.B, prob.scales, prob.zero_points, None, N=p.N, K=p.K,
                           block_size=spec["bs"])
        spent += time.perf_counter() - t0
        done_bytes += prob.algorithmic_bytes()
        names.append(f"L{layer}.{p.name}")
        if spent >= budget_s:
            break
    desc = (f"first {len(names)} projections of the {spec['model']} decode step "
            f"({names[0]}..{names[-1]}, {done_bytes / 1e6:.1f} MB algorithmic), "
            f"oracle single-threaded")
    return done_bytes, spent, desc


def cpu_leg(budget_s, spec=None, seed_base=3000):
    nbytes, secs, desc = oracle_sample(budget_s, seed_base, spec)
    return {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": 1, "cpu": cpu_model(),
            "kind": "oracle", "sample": desc}


def run_reference(args, rank, world):
    if rank != 0:
        return
    desc = ""
    for _ in range(args.warmup):
        oracle_sample(args.ref_budget / 8)
    nbytes_total, t_total = 0, 0.0
    for _ in range(args.steps):
        nbytes, t, desc = oracle_sample(args.ref_budget)
        nbytes_total += nbytes
        t_total += t
    gbs = nbytes_total / t_total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t_total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD + " (bounded sample per step)", "M": 1,
                   "block_size": 128, "a_dtype": "bf16"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# GPU leg
# ----------------------------------------------------------------------------

STEP_4B = dict(model="QWEN3_4B", a_dtype="bf16", bs=128, zp=False, scale_dtype="bf16",
               scale_range=(0.002, 0.01))
STEP_0P6B = dict(model="QWEN3_0P6B", a_dtype="f32", bs=32, zp=True, scale_dtype="f32",
                 scale_range=(0.005, 0.02))


def build_decode_step(dev, seed_base=5000, keep=None, spec=STEP_4B):
    """Prepacked weights, activations and outputs of one decode step, all
    resident on dev, as a list of launches: (name, weights, activation row,
    outputs). Per layer: q/k/v on one row (one fused-N launch), o, the gated
    gate/up pair, down; then lm_head. Weights are drawn on the device from a
    seeded generator (2 GB would take minutes on the host). `keep`: names of
    launches whose raw inputs (activation row, and per weight its codes and
    scales) are also returned as host tensors in a fifth element, for parity
    checks (steps without zero points)."""
    import torch

    import int4_weight_only_matmulnbits_gb300 as mnb
    from int4_weight_only_matmulnbits_gb300 import workloads
    model = getattr(workloads, spec["model"])
    adt = torch.float32 if spec["a_dtype"] == "f32" else torch.bfloat16
    sdt = torch.float32 if spec["scale_dtype"] == "f32" else torch.bfloat16
    bs, zp = spec["bs"], spec["zp"]
    lo, hi = spec["scale_range"]
    P = {p.name: p for p in model["projections"]}
    groups = [("qkv", [P["q"], P["k"], P["v"]]), ("o", [P["o"]]),
              ("gate_up", [P["gate"], P["up"]]), ("down", [P["down"]])]
    plan = [(f"L{l}.{name}", ps) for l in range(model["layers"]) for name, ps in groups]
    plan.append(("lm_head", [model["lm_head"]]))
    g = torch.Generator(device=dev)
    a_total = sum(ps[0].K for _, ps in plan)
    # The gated-MLP launch writes one output for its two weights.
    y_total = sum(ps[0].N if name.endswith("gate_up") else sum(p.N for p in ps)
                  for name, ps in plan)
    A_all = torch.empty(a_total, dtype=adt, device=dev)
    Y_all = torch.empty(y_total, dtype=adt, device=dev)
    es = A_all.element_size()
    ao = yo = 0
    algo_bytes = 0
    launches = []
    kept = {}
    seed = seed_base
    for name, ps in plan:
        K = ps[0].K
        nb = -(-K // bs)
        A = A_all[ao:ao + K].view(1, K)
        g.manual_seed(seed)
        A.copy_(torch.randn(1, K, device=dev, generator=g).to(adt))
        ao += K
        algo_bytes += K * es
        ws, Ys = [], []
        paired = name.endswith("gate_up")
        for i, p in enumerate(ps):
            seed += 1
            g.manual_seed(seed)
            B = torch.randint(0, 256, (p.N, nb, bs // 2), dtype=torch.uint8, device=dev,
                              generator=g)
            S = (torch.rand(p.N, nb, device=dev, generator=g) * (hi - lo) + lo).to(sdt)
            Z = (torch.randint(0, 256, (p.N, (nb + 1) // 2), dtype=torch.uint8, device=dev,
                               generator=g) if zp else None)
            ws.append(mnb.mnb_prepack(B, S, Z, p.N, K, bs))
            if keep and name in keep:
                kept.setdefault(name, {"A": A.cpu(), "weights": []})["weights"].append(
                    (B.cpu(), S.cpu(), p.N, K))
            del B, S, Z
            algo_bytes += p.N * nb * bs // 2 + p.N * nb * S_bytes(sdt)
            algo_bytes += p.N * ((nb + 1) // 2) if zp else 0
            if not paired or i == 0:
                Ys.append(Y_all[yo:yo + p.N].view(1, p.N))
                yo += p.N
                algo_bytes += p.N * es
        launches.append((name, ws, A, Ys))
        seed += 1
    torch.cuda.synchronize()
    if keep is not None:
        return launches, A_all, Y_all, algo_bytes, kept
    return launches, A_all, Y_all, algo_bytes


def S_bytes(dt):
    import torch
    return 4 if dt == torch.float32 else 2


def step_ops(mnb, launches):
    """The launches of a decode step as op descriptors for mnb_graph_build:
    q, k and v share their activation row (one fused-N call), gate and up
    form a gated pair; array order is launch order."""
    ops = []
    for name, ws, A, Ys in launches:
        if name.endswith("gate_up"):
            ops.append(mnb.ChainOp(A, ws[0], Ys[0], up=ws[1]))
        else:
            for w, Y in zip(ws, Ys):
                ops.append(mnb.ChainOp(A, w, Y))
    return ops


def build_decode_chain(mnb, launches):
    """The decode step as one chain (mnb_chain_build): the same weights,
    activations and outputs as `launches`, with the decoder's dependencies:
    q, k, v after the previous layer's down projection, o after q, k and v,
    the gated-MLP pair after o, down after the pair, lm_head after the last
    down. Each op still reads its own activation row."""
    ops = []
    prev_down = qkv = o_idx = gu_idx = None
    for name, ws, A, Ys in launches:
        kind = name.split(".")[-1]
        if kind == "qkv":
            deps = () if prev_down is None else (prev_down,)
            first = len(ops)
            for w, Y in zip(ws, Ys):
                ops.append(mnb.ChainOp(A, w, Y, deps=deps))
            qkv = tuple(range(first, len(ops)))
        elif kind == "o":
            ops.append(mnb.ChainOp(A, ws[0], Ys[0], deps=qkv))
            o_idx = len(ops) - 1
        elif kind == "gate_up":
            ops.append(mnb.ChainOp(A, ws[0], Ys[0], up=ws[1], deps=(o_idx,)))
            gu_idx = len(ops) - 1
        elif kind == "down":
            ops.append(mnb.ChainOp(A, ws[0], Ys[0], deps=(gu_idx,)))
            prev_down = len(ops) - 1
        else:
            ops.append(mnb.ChainOp(A, ws[0], Ys[0], deps=(prev_down,)))
    return mnb.mnb_chain_build(ops)


def run_launch(mnb, name, ws, A, Ys):
    """One launch of the decode step."""
    if name.endswith("gate_up"):
        mnb.mnb_matmul_gate_up(A, ws[0], ws[1], out=Ys[0])
    elif len(ws) == 1:
        mnb.mnb_matmul(A, ws[0], None, out=Ys[0])
    else:
        mnb.mnb_matmul_grouped(A, ws, outs=Ys)


def time_region(fn, steps, stream):
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3


def time_steps(fn, steps, stream):
    """Device time of each of `steps` calls of fn (CUDA events around each, on
    `stream`); returns (total seconds, per-call seconds)."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(steps):
        fn()
        ev[i + 1].record(stream)
    ev[-1].synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(steps)]
    return ev[0].elapsed_time(ev[-1]) / 1e3, per


def pct(xs, q):
    xs = sorted(xs)
    if not xs:
        return None
    k = (len(xs) - 1) * q / 100.0
    i = int(k)
    return xs[i] if i + 1 >= len(xs) else xs[i] + (xs[i + 1] - xs[i]) * (k - i)


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def lm_head_fusions(mnb, lm_launch, dev, steps=50):
    """The step's lm_head launch alone and with the fused final RMSNorm and
    greedy ArgMax (mnb_matmul_rmsnorm), us per call on the same stream;
    the weight (200 MB) exceeds L2, so every call streams it from HBM."""
    import torch
    _, ws, A, Ys = lm_launch
    w, Y = ws[0], Ys[0]
    g = torch.Generator(device=dev)
    g.manual_seed(4321)
    gamma = torch.rand(w.K, device=dev, generator=g) + 0.5
    stream = torch.cuda.current_stream()
    out = {}
    for name, fn in (("lm_head", lambda: mnb.mnb_matmul(A, w, None, out=Y)),
                     ("rmsnorm_lm_head", lambda: mnb.mnb_matmul_rmsnorm(A, w, gamma=gamma, out=Y)),
                     ("rmsnorm_lm_head_argmax",
                      lambda: mnb.mnb_matmul_rmsnorm(A, w, gamma=gamma, logits=False,
                                                     argmax=True))):
        for _ in range(3):
            fn()
        out[name + "_us"] = time_region(fn, steps, stream) * 1e6 / steps
    return out


def prefill_measure(dev, steps=10, warmup=3, M=2048, repeats=5, path="gemm"):
    """TFLOP/s of the tensor-core path at M rows over the seven Qwen3-4B
    projection shapes (bf16 A, bs 128, zero points, bias), each timed alone
    as the median of `repeats` regions of `steps` back-to-back launches;
    None when the path is not available."""
    import torch

    import int4_weight_only_matmulnbits_gb300 as mnb
    from int4_weight_only_matmulnbits_gb300.workloads import QWEN3_4B
    bs = 128
    g = torch.Generator(device=dev)
    total_flops, total_s, per = 0, 0.0, {}
    stream = torch.cuda.current_stream()
    for i, p in enumerate(QWEN3_4B["projections"]):
        g.manual_seed(9000 + i)
        nb = -(-p.K // bs)
        B = torch.randint(0, 256, (p.N, nb, bs // 2), dtype=torch.uint8, device=dev, generator=g)
        S = (torch.rand(p.N, nb, device=dev, generator=g) * 0.008 + 0.002).to(torch.bfloat16)
        Z = torch.randint(0, 256, (p.N, (nb + 1) // 2), dtype=torch.uint8, device=dev,
                          generator=g)
        bias = torch.randn(p.N, device=dev, generator=g) * 0.02
        A = torch.randn(M, p.K, device=dev, generator=g).to(torch.bfloat16)
        w = mnb.mnb_prepack(B, S, Z, p.N, p.K, bs)
        Y = torch.empty(M, p.N, dtype=torch.bfloat16, device=dev)
        try:
            mnb.mnb_matmul(A, w, bias, out=Y, path=path)
        except mnb.MnbError as e:
            if e.status == -8:
                return None
            raise
        for _ in range(warmup):
            mnb.mnb_matmul(A, w, bias, out=Y, path=path)
        ts = sorted(time_region(lambda: mnb.mnb_matmul(A, w, bias, out=Y, path=path), steps,
                                stream) for _ in range(repeats))
        t = ts[len(ts) // 2]
        flops = 2 * M * p.N * p.K * steps
        per[p.name] = flops / t / 1e12
        total_flops += flops
        total_s += t
    return {"value": total_flops / total_s / 1e12, "unit": "TFLOP/s", "M": M,
            "per_projection_tflops": per}


def measure_step(mnb, dev, spec, steps, warmup, seed_base=5000, local=0, clock_log=None,
                 dist=None):
    """One decode step recorded as a CUDA graph through the C ABI
    (mnb_graph_build) and timed: device only (mnb_graph_run, clocks sampled
    during the timed region) and end to end (mnb_graph_run_from_host: the
    step's activation rows copied in from pinned host memory, its outputs
    copied back, every step)."""
    import torch
    launches, A_all, Y_all, algo_bytes = build_decode_step(dev, seed_base, spec=spec)
    graph = mnb.mnb_graph_build(step_ops(mnb, launches))
    assert graph.calls == len(launches), (graph.calls, len(launches))
    stream = torch.cuda.current_stream()
    for _ in range(max(warmup, 3)):
        graph.run()
    torch.cuda.synchronize()
    sampler = ClockSampler(local, clock_log)
    if dist:
        dist.barrier()
    sampler.start()
    time.sleep(0.3)
    t, per = time_steps(graph.run, steps, stream)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    A_host = torch.empty(A_all.shape, dtype=A_all.dtype).pin_memory()
    A_host.copy_(A_all.cpu())
    Y_host = torch.empty(Y_all.shape, dtype=Y_all.dtype).pin_memory()
    e2e_step = lambda: graph.run_from_host(A_host, A_all, Y_all, Y_host)
    for _ in range(3):
        e2e_step()
    t_e2e, _ = time_steps(e2e_step, steps, stream)
    return dict(launches=launches, A_all=A_all, Y_all=Y_all, algo_bytes=algo_bytes,
                graph=graph, t=t, per=per, t_e2e=t_e2e, clocks=clocks,
                h2d=A_all.numel() * A_all.element_size(),
                d2h=Y_all.numel() * Y_all.element_size())


def clocked(local, fn):
    """fn() with the SM clocks sampled while it runs: (result, clocks)."""
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    try:
        out = fn()
    finally:
        clocks = sampler.stop()
    return out, clocks


def single_gemv(mnb, dev, reps=30):
    """The single GEMV workload (A fp32 [1, 1024], B [3072, 1024] bs 32, fp32
    scales, no zero points, no bias): device time per launch with L2 flushed
    before each launch (cold) and back to back with the 1.98 MB weight left in
    L2 (hot)."""
    import torch
    from int4_weight_only_matmulnbits_gb300.workloads import make_problem
    prob = make_problem(1, 3072, 1024, 32, dtype=torch.float32, seed=0)
    w = mnb.mnb_prepack(prob.B.to(dev), prob.scales.to(dev), None, 3072, 1024, 32)
    A = prob.A.to(dev)
    Y = torch.empty(1, 3072, dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
    fn = lambda: mnb.mnb_matmul(A, w, None, out=Y, workspace=None)
    cold = _cold_launch_us(fn, reps, flush)
    # Hot: 20 back-to-back launches replayed from one CUDA graph, so that no
    # host gap sits between them.
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(20):
            fn()
    for _ in range(3):
        g.replay()
    t, per = time_steps(g.replay, reps, torch.cuda.current_stream())
    hot = statistics.median(per) * 1e6 / 20
    return prob, {"cold_us": cold, "hot_us": hot, "algorithmic_bytes": prob.algorithmic_bytes()}


def bnb4_prefill(mnb, dev, M=2048, N=9728, K=2560, bs=64, reps=10):
    """The bitsandbytes-style 4-bit matrix at prefill size on the tensor-core
    kernel's code-book mode: gate-sized weight (9728 x 2560, bs 64, bf16
    absmax and activations, a 16-value code book), L2 flushed before each
    launch, median of reps."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    B = torch.randint(0, 256, (N * K // 2,), dtype=torch.uint8, device=dev, generator=g)
    absmax = (torch.rand(N * K // bs, device=dev, generator=g) * 0.04 + 0.01).to(torch.bfloat16)
    code = torch.linspace(-1.0, 1.0, 16, device=dev)
    w = mnb.mnb_prepack_bnb4(B, absmax, N, K, bs)
    A = torch.randn(M, K, device=dev, generator=g).to(torch.bfloat16)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
    us = _cold_launch_us(lambda: mnb.mnb_matmul_bnb4(A, w, code, out=Y), reps, flush)
    return {"workload": f"MatMulBnb4 {N}x{K}, bs {bs}, bf16 absmax and A, M={M}, L2 flushed",
            "us": us, "value": 2 * M * N * K / us / 1e6, "unit": "TFLOP/s"}


def crossover(mnb, dev, flush):
    """Condensed GEMV / tensor-core crossover: device time per launch (L2
    flushed, median of 5) of both kernels and of the dispatch, on gate
    2560->9728 and down 9728->2560, bf16 A, bs 128, no zero points."""
    import torch
    rows = []
    for name, N, K in (("gate", 9728, 2560), ("down", 2560, 9728)):
        w, _ = _weights(dev, N, K, 128, torch.bfloat16, False, 21)
        for M in (1, 8, 16, 32, 64, 256):
            A = torch.randn(M, K, device=dev).to(torch.bfloat16)
            Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            row = {"shape": name, "M": M}
            for path in ("gemv", "gemm", "auto"):
                try:
                    mnb.mnb_matmul(A, w, None, out=Y, path=path, workspace=None)
                except mnb.MnbError:
                    continue
                row[path + "_us"] = round(_cold_launch_us(
                    lambda: mnb.mnb_matmul(A, w, None, out=Y, path=path, workspace=None), 5,
                    flush), 2)
            rows.append(row)
    return rows


def max_over_ranks(values, dist, device=None):
    """Element-wise maximum of a list of floats over all ranks (the slowest
    rank's times); the list itself at N = 1."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_step, steps, world, seconds):
    """Units per second processed by all ranks together (weak scaling: every
    rank runs the same step), over the slowest rank's time, in units / 1e9."""
    return units_per_step * steps * world / seconds / 1e9


def run_gpu(args, rank, world, dist):
    import torch

    import int4_weight_only_matmulnbits_gb300 as mnb
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mnb.build_library()
    mnb.load()
    hbm_peak, bf16_peak, _, peak_kind = peaks()

    m = measure_step(mnb, dev, STEP_4B, args.steps, args.warmup, local=local,
                     clock_log=args.clock_log, dist=dist)
    launches, algo_bytes, graph = m["launches"], m["algo_bytes"], m["graph"]
    cur = torch.cuda.current_stream()

    # The same step as one persistent launch (mnb_chain_run), for comparison;
    # not the headline: the graph of launches is faster on this workload.
    chain = build_decode_chain(mnb, launches)
    for _ in range(3):
        chain.run()
    t_chain = time_region(chain.run, args.steps, cur)

    t, t_e2e, t_chain = max_over_ranks([m["t"], m["t_e2e"], t_chain], dist, device=dev)

    if rank != 0:
        return
    value = whole_job_rate(algo_bytes, args.steps, world, t)
    e2e = whole_job_rate(algo_bytes, args.steps, world, t_e2e)
    per_gpu = whole_job_rate(algo_bytes, args.steps, 1, t)
    per = [x * 1e3 for x in m["per"]]
    warmup = max(args.warmup, 3)
    extras = world == 1 and not args.skip_extras
    cpu = None
    if world == 1 and not args.skip_cpu:
        cpu = cpu_leg(args.cpu_budget)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": warmup,
        "ms_per_step": 1e3 * t / args.steps,
        "ms_per_step_p10": pct(per, 10), "ms_per_step_p50": pct(per, 50),
        "ms_per_step_p90": pct(per, 90), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "block_size": 128, "a_dtype": "bf16",
                   "weights_per_step": sum(len(ws) for _, ws, _, _ in launches),
                   "launches_per_step": len(launches),
                   "algorithmic_bytes_per_step": algo_bytes,
                   "l2": "inputs larger than L2 (2.08 GB per step vs 129 MB)",
                   "launch": "one CUDA graph per step recorded by the library "
                             "(mnb_graph_build, run with mnb_graph_run): per layer fused "
                             "qkv, o, gated-MLP gate+up (SiLU(gate)*up), down, then lm_head "
                             f"({graph.calls} calls, {graph.kernels} kernels), programmatic "
                             "dependent launch",
                   "parallelism": f"replicas x{world}"},
        "hbm_fraction": per_gpu / hbm_peak,
        "roofline": {"bound": "hbm", "achieved": per_gpu, "peak": hbm_peak,
                     "unit": "GB/s", "frac": per_gpu / hbm_peak,
                     "traffic": step_traffic(algo_bytes / len(launches)),
                     "peak_kind": peak_kind,
                     "kernel": "gemv_kernel (every launch of the step)",
                     "achieved_basis": "algorithmic bytes of the step / device time of the "
                                       "step (= bytes per launch / mean launch time)",
                     "algorithmic_bytes_per_launch": algo_bytes / len(launches),
                     "traffic_basis": "ncu dram read+write of the decode kernel on the "
                                      "gate shape (3 launches, 1.0050 x algorithmic), "
                                      "scaled to the step's mean launch; null if the "
                                      "kernel changed"},
        "e2e": {"value": e2e, "unit": "GB/s", "h2d_bytes_per_step": m["h2d"],
                "d2h_bytes_per_step": m["d2h"],
                "api": "mnb_graph_run_from_host (C ABI): pinned host activations in, the "
                       "step, outputs back to pinned host memory, on one stream"},
        "gpu_launches": graph.kernels * args.steps,
        "clocks": m["clocks"],
        "cpu_baseline": cpu,
        "decode_chain": {"value": algo_bytes * args.steps / t_chain / 1e9, "unit": "GB/s",
                         "ms_per_step": 1e3 * t_chain / args.steps, "launches_per_step": 1,
                         "note": "the same step and dependencies as one persistent "
                                 "cooperative launch (mnb_chain_run)"},
    }
    if extras:
        line["lm_head_fusions"] = lm_head_fusions(mnb, launches[-1], dev)
        del chain, m, launches, graph
        torch.cuda.empty_cache()
        flops_peak = {"bound": "tensor", "peak": bf16_peak, "unit": "TFLOP/s",
                      "peak_kind": peak_kind + " bf16 burst (cuBLAS)"}
        for key, M in (("prefill", 2048), ("prefill_m512", 512)):
            pf, clk = clocked(local, lambda: prefill_measure(dev, M=M))
            if pf is not None:
                pf["roofline"] = dict(flops_peak, achieved=pf["value"],
                                      frac=pf["value"] / bf16_peak, traffic=None,
                                      kernel="gemm_kernel / gemm_sk_kernel (7 shapes)")
                pf["clocks"] = clk
                pf["workload"] = (f"Qwen3-4B prefill projections, M={M}, bf16 A, bs 128, "
                                  "zero points, fp32 bias, each shape timed alone")
                pf["cpu_baseline"] = None if args.skip_cpu else dict(
                    cpu_leg(3.0, seed_base=3500),
                    note="the oracle's GB/s on decode-step projections; its prefill rate "
                         "is the same dot products (not run again at M rows)")
            line[key] = pf
        # The persistent CTA-pair kernel (forced path; the dispatch keeps the
        # tile-per-CTA kernel, which is faster on these shapes).
        pp, clk = clocked(local, lambda: prefill_measure(dev, M=2048, path="gemm_pair"))
        if pp is not None:
            pp["roofline"] = dict(flops_peak, achieved=pp["value"],
                                  frac=pp["value"] / bf16_peak, traffic=None,
                                  kernel="gemm_pair_kernel (7 shapes)")
            pp["clocks"] = clk
            pp["workload"] = ("Qwen3-4B prefill projections, M=2048, as 'prefill', through "
                              "mnb_matmul_path(..., MNB_PATH_GEMM_PAIR)")
            line["prefill_cta_pair"] = pp
        m6 = measure_step(mnb, dev, STEP_0P6B, args.steps, warmup, seed_base=7000,
                          local=local)
        b6 = m6["algo_bytes"]
        g6 = b6 * args.steps / m6["t"] / 1e9
        line["decode_step_qwen3_0p6b"] = {
            "workload": "Qwen3-0.6B decode step projections, M=1, fp32 A, bs 32, uint4 zero "
                        "points, fp32 scales (28 layers + lm_head)",
            "value": g6, "unit": "GB/s", "ms_per_step": 1e3 * m6["t"] / args.steps,
            "ms_per_step_p10": pct([x * 1e3 for x in m6["per"]], 10),
            "ms_per_step_p90": pct([x * 1e3 for x in m6["per"]], 90),
            "algorithmic_bytes_per_step": b6, "launches_per_step": len(m6["launches"]),
            "e2e": {"value": b6 * args.steps / m6["t_e2e"] / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": m6["h2d"], "d2h_bytes_per_step": m6["d2h"]},
            "roofline": {"bound": "hbm", "achieved": g6, "peak": hbm_peak, "unit": "GB/s",
                         "frac": g6 / hbm_peak, "traffic": None, "peak_kind": peak_kind},
            "clocks": m6["clocks"],
            "cpu_baseline": None if args.skip_cpu else cpu_leg(3.0, STEP_0P6B, 3700),
        }
        del m6
        torch.cuda.empty_cache()
        prob1, s1 = single_gemv(mnb, dev)
        nb1 = s1["algorithmic_bytes"]
        cold_gbs = nb1 / s1["cold_us"] / 1e3
        t0 = time.perf_counter()
        import oracle
        oracle.load()
        reps = 0
        while time.perf_counter() - t0 < 2.0:
            oracle.matmulnbits(prob1.A, prob1.B, prob1.scales, None, None, N=3072, K=1024,
                               block_size=32)
            reps += 1
        o_s = (time.perf_counter() - t0) / reps
        line["single_gemv"] = {
            "workload": "single MatMulNBits GEMV, A fp32 [1,1024], B [3072,1024] bs 32, fp32 "
                        "scales, no zero points, no bias, seed 0",
            "cold_us": s1["cold_us"], "hot_us": s1["hot_us"], "algorithmic_bytes": nb1,
            "value": cold_gbs, "unit": "GB/s (cold L2)", "hot_GBps": nb1 / s1["hot_us"] / 1e3,
            "roofline": {"bound": "hbm", "achieved": cold_gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": cold_gbs / hbm_peak, "traffic": None,
                         "peak_kind": peak_kind,
                         "note": "cold: L2 flushed before every launch; hot (weight in L2) "
                                 "is not bounded by HBM"},
            "cpu_baseline": {"value": nb1 / o_s / 1e9, "unit": "GB/s", "cores": 1,
                             "cpu": cpu_model(), "kind": "oracle",
                             "sample": f"the whole GEMV, {reps} runs"},
        }
        bb, clk = clocked(local, lambda: bnb4_prefill(mnb, dev))
        bb["roofline"] = dict(flops_peak, achieved=bb["value"], frac=bb["value"] / bf16_peak,
                              traffic=None, kernel="gemm_kernel, code-book instantiation")
        bb["clocks"] = clk
        line["bnb4_prefill"] = bb
        flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
        cross, clk = clocked(local, lambda: crossover(mnb, dev, flush))
        line["crossover"] = {"unit": "us per launch, L2 flushed, median of 5", "rows": cross,
                             "clocks": clk}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# single-kernel cases (for profiler captures) and the GEMV/GEMM crossover sweep
# ----------------------------------------------------------------------------

def _weights(dev, N, K, bs, sdtype, zp, seed):
    import torch

    import int4_weight_only_matmulnbits_gb300 as mnb
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    nb = -(-K // bs)
    B = torch.randint(0, 256, (N, nb, bs // 2), dtype=torch.uint8, device=dev, generator=g)
    S = (torch.rand(N, nb, device=dev, generator=g) * 0.008 + 0.002).to(sdtype)
    Z = (torch.randint(0, 256, (N, (nb + 1) // 2), dtype=torch.uint8, device=dev, generator=g)
         if zp else None)
    w = mnb.mnb_prepack(B, S, Z, N, K, bs)
    nbytes = N * nb * bs // 2 + N * nb * S.element_size() + (N * ((nb + 1) // 2) if zp else 0)
    return w, nbytes


def _cold_launch_us(fn, reps, flush):
    """Median device time of fn, each launch after an L2 flush."""
    import torch
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(ts)


CASES = {
    # name: (M, N, K, bs, A dtype, zero points, bias, path)
    "single": (1, 3072, 1024, 32, "f32", False, False, "auto"),
    "gemv_gate": (1, 9728, 2560, 128, "bf16", False, False, "auto"),
    "gemv_lm_head": (1, 151936, 2560, 128, "bf16", False, False, "auto"),
    "gemm_gate": (2048, 9728, 2560, 128, "bf16", True, True, "gemm"),
    "gemm_gate_f32": (2048, 9728, 2560, 128, "f32", True, True, "gemm"),
    "gemm_pair_gate": (2048, 9728, 2560, 128, "bf16", True, True, "gemm_pair"),
}


def run_case(args):
    """One kernel shape, --steps cold launches (L2 flushed before each); or one
    eager decode step per --steps ("step"); or the crossover sweep."""
    import torch

    import int4_weight_only_matmulnbits_gb300 as mnb
    dev = torch.device("cuda", 0)
    mnb.build_library()
    mnb.load()
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
    if args.case == "step":
        launches, _, _, algo_bytes = build_decode_step(dev)
        for _ in range(args.steps):
            for name, ws, A, Ys in launches:
                run_launch(mnb, name, ws, A, Ys)
        torch.cuda.synchronize()
        print(json.dumps({"case": "step", "launches": len(launches) * args.steps,
                          "algorithmic_bytes_per_step": algo_bytes}))
        return
    if args.case == "sweep":
        return run_sweep(dev, flush)
    M, N, K, bs, adt, zp, bias, path = CASES[args.case]
    dt = torch.float32 if adt == "f32" else torch.bfloat16
    w, wbytes = _weights(dev, N, K, bs, dt, zp, 11)
    g = torch.Generator(device=dev)
    g.manual_seed(12)
    A = torch.randn(M, K, device=dev, generator=g).to(dt)
    b = torch.randn(N, device=dev, generator=g) * 0.02 if bias else None
    Y = torch.empty(M, N, dtype=dt, device=dev)
    us = _cold_launch_us(lambda: mnb.mnb_matmul(A, w, b, out=Y, path=path), args.steps, flush)
    nbytes = wbytes + A.numel() * A.element_size() + Y.numel() * Y.element_size() + (
        4 * N if bias else 0)
    print(json.dumps({"case": args.case, "M": M, "N": N, "K": K, "block_size": bs,
                      "us_per_launch_cold": us, "algorithmic_bytes": nbytes,
                      "GB_s": nbytes / us / 1e3, "TFLOP_s": 2 * M * N * K / us / 1e6}))


def run_sweep(dev, flush):
    """GEMV and tensor-core GEMM device time per M on the gate and down shapes,
    per block size, activation dtype and zero points (cold L2, median of 7)."""
    import torch

    import int4_weight_only_matmulnbits_gb300 as mnb
    Ms = (1, 2, 4, 8, 16, 32, 64, 256)
    rows = []
    for name, N, K in (("gate", 9728, 2560), ("down", 2560, 9728)):
        for bs in (32, 64, 128):
            for adt in ("f32", "bf16"):
                dt = torch.float32 if adt == "f32" else torch.bfloat16
                for zp in (False, True):
                    w, _ = _weights(dev, N, K, bs, dt, zp, 21)
                    for M in Ms:
                        A = torch.randn(M, K, device=dev).to(dt)
                        Y = torch.empty(M, N, dtype=dt, device=dev)
                        t = {}
                        for path in ("gemv", "gemm", "auto"):
                            try:
                                mnb.mnb_matmul(A, w, None, out=Y, path=path)
                            except mnb.MnbError:
                                continue
                            t[path] = _cold_launch_us(
                                lambda: mnb.mnb_matmul(A, w, None, out=Y, path=path), 7, flush)
                        rows.append({"shape": name, "bs": bs, "a": adt, "zp": zp, "M": M, **t})
                        print(json.dumps(rows[-1]), flush=True)
                    del w
                    torch.cuda.empty_cache()
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-budget", type=float, default=8.0)
    ap.add_argument("--clock-log", default=None,
                    help="file for the raw nvidia-smi clock samples of the timed region "
                         "(default: a private temporary file)")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-extras", action="store_true",
                    help="only the headline decode step (no prefill, Qwen3-0.6B step, single "
                         "GEMV or crossover keys)")
    ap.add_argument("--case", default=None, choices=sorted(CASES) + ["step", "sweep"],
                    help="run one kernel shape (or one eager decode step per --steps, or "
                         "the GEMV/GEMM crossover sweep) instead of the benchmark")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return

    world = int(os.environ.get("WORLD_SIZE", 1))
    rank = int(os.environ.get("RANK", 0))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group(backend)
        dist = tdist
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, dist)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
