"""Benchmark: INT4 weight-only MatMulNBits decode step on GB300.

Workload: one batch-1 decode step of Qwen3-4B's projections (M = 1, bf16
activations ~ N(0,1), block size 128, no zero points (8), bf16 scales
U[0.002, 0.01]): q 2560->4096, k/v 2560->1024, o 4096->2560, gate/up
2560->9728, down 9728->2560, for 36 layers, plus lm_head 2560->151936 —
253 weights and 2.08 GB of algorithmic bytes per step, each weight with its
own seeded codes and scales, all resident in HBM before timing.

The step follows the model's data flow: q, k and v read one activation row
and run as one fused-N launch (mnb_matmul_grouped); gate and up run as one
gated-MLP launch that stores SiLU(gate) * up (mnb_matmul_gate_up); o, down
and lm_head each read their own row. That is 4 launches per layer and 145
per step, replayed as one CUDA graph. The step's bytes exceed the 129 MB L2
many times over, so no flush is needed.

Also measured, outside the timed region of the headline number: the prefill
GEMM at M = 2048 over the seven Qwen3-4B projection shapes (TFLOP/s), when
the tensor-core path is available.

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


# DRAM read + write per decode-kernel launch of one decode step, from one ncu
# capture of the 145 launches (dram__bytes_read.sum + dram__bytes_write.sum),
# valid only for the decode-kernel sources it was measured on.
STEP_TRAFFIC = {
    "bytes_per_launch": 14399640,
    "sources": ("gemv.cu", "mnb_common.cuh", "mnb_launch.h"),
    "sha256": "604251cb1579c44863bc26c95029890d02f40b0237f20ce896671d5979cb1d64",
}


def step_traffic():
    import hashlib
    h = hashlib.sha256()
    for f in STEP_TRAFFIC["sources"]:
        with open(os.path.join(ROOT, "int4_weight_only_matmulnbits_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return STEP_TRAFFIC["bytes_per_launch"] if h.hexdigest() == STEP_TRAFFIC["sha256"] else None


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
                 "--format=csv,noheader,nounits", "-lms", "200"],
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

def oracle_sample(budget_s: float, seed_base: int = 3000):
    """Times the oracle (single thread) over the decode step's projections in
    order until about budget_s seconds of CPU work; returns (bytes, seconds,
    description)."""
    import torch

    import oracle
    from int4_weight_only_matmulnbits_gb300.workloads import QWEN3_4B, make_problem
    oracle.load()
    projs = [(l, p) for l in range(QWEN3_4B["layers"]) for p in QWEN3_4B["projections"]]
    done_bytes, spent, names = 0, 0.0, []
    for i, (layer, p) in enumerate(projs):
        prob = make_problem(1, p.N, p.K, 128, dtype=torch.bfloat16, seed=seed_base + i,
                            scale_range=(0.002, 0.01))
        t0 = time.perf_counter()
        oracle.matmulnbits(prob.A, prob.B, prob.scales, None, None, N=p.N, K=p.K,
                           block_size=128)
        spent += time.perf_counter() - t0
        done_bytes += prob.algorithmic_bytes()
        names.append(f"L{layer}.{p.name}")
        if spent >= budget_s:
            break
    desc = (f"first {len(names)} projections of the decode step ({names[0]}..{names[-1]}, "
            f"{done_bytes / 1e6:.1f} MB algorithmic), oracle single-threaded")
    return done_bytes, spent, desc


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

def build_decode_step(dev, seed_base=5000, keep=None):
    """Prepacked weights, activations and outputs of one decode step, all
    resident on dev, as a list of launches: (weights, activation row,
    outputs). Weights are drawn on the device from a seeded generator
    (2 GB would take minutes on the host). `keep`: names of launches whose
    raw inputs (activation row, and per weight its codes and scales) are
    also returned as host tensors in a fifth element, for parity checks."""
    import torch

    import int4_weight_only_matmulnbits_gb300 as mnb
    from int4_weight_only_matmulnbits_gb300.workloads import QWEN3_4B
    P = {p.name: p for p in QWEN3_4B["projections"]}
    groups = [("qkv", [P["q"], P["k"], P["v"]]), ("o", [P["o"]]),
              ("gate_up", [P["gate"], P["up"]]), ("down", [P["down"]])]
    plan = [(f"L{l}.{name}", ps) for l in range(QWEN3_4B["layers"]) for name, ps in groups]
    plan.append(("lm_head", [QWEN3_4B["lm_head"]]))
    bs = 128
    g = torch.Generator(device=dev)
    a_total = sum(ps[0].K for _, ps in plan)
    # The gated-MLP launch writes one output for its two weights.
    y_total = sum(ps[0].N if name.endswith("gate_up") else sum(p.N for p in ps)
                  for name, ps in plan)
    A_all = torch.empty(a_total, dtype=torch.bfloat16, device=dev)
    Y_all = torch.empty(y_total, dtype=torch.bfloat16, device=dev)
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
        A.copy_(torch.randn(1, K, device=dev, generator=g).to(torch.bfloat16))
        ao += K
        algo_bytes += K * 2
        ws, Ys = [], []
        paired = name.endswith("gate_up")
        for i, p in enumerate(ps):
            seed += 1
            g.manual_seed(seed)
            B = torch.randint(0, 256, (p.N, nb, bs // 2), dtype=torch.uint8, device=dev,
                              generator=g)
            S = (torch.rand(p.N, nb, device=dev, generator=g) * 0.008 + 0.002).to(torch.bfloat16)
            ws.append(mnb.mnb_prepack(B, S, None, p.N, K, bs))
            if keep and name in keep:
                kept.setdefault(name, {"A": A.cpu(), "weights": []})["weights"].append(
                    (B.cpu(), S.cpu(), p.N, K))
            del B, S
            algo_bytes += p.N * nb * bs // 2 + p.N * nb * 2
            if not paired or i == 0:
                Ys.append(Y_all[yo:yo + p.N].view(1, p.N))
                yo += p.N
                algo_bytes += p.N * 2
        launches.append((name, ws, A, Ys))
        seed += 1
    torch.cuda.synchronize()
    if keep is not None:
        return launches, A_all, Y_all, algo_bytes, kept
    return launches, A_all, Y_all, algo_bytes


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


def prefill_measure(dev, steps=5, warmup=3):
    """TFLOP/s of the tensor-core path at M=2048 over the seven Qwen3-4B
    projection shapes (bf16 A, bs 128, zero points, bias), each timed alone;
    None when the path is not available."""
    import torch

    import int4_weight_only_matmulnbits_gb300 as mnb
    from int4_weight_only_matmulnbits_gb300.workloads import QWEN3_4B
    M, bs = 2048, 128
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
            mnb.mnb_matmul(A, w, bias, out=Y, path="gemm")
        except mnb.MnbError as e:
            if e.status == -8:
                return None
            raise
        for _ in range(warmup):
            mnb.mnb_matmul(A, w, bias, out=Y, path="gemm")
        t = time_region(lambda: mnb.mnb_matmul(A, w, bias, out=Y, path="gemm"), steps, stream)
        flops = 2 * M * p.N * p.K * steps
        per[p.name] = flops / t / 1e12
        total_flops += flops
        total_s += t
    return {"value": total_flops / total_s / 1e12, "unit": "TFLOP/s", "M": M,
            "per_projection_tflops": per}


def run_gpu(args, rank, world, dist):
    import torch

    import int4_weight_only_matmulnbits_gb300 as mnb
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mnb.build_library()
    mnb.load()
    hbm_peak, _, _, peak_kind = peaks()

    launches, A_all, Y_all, algo_bytes = build_decode_step(dev)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def step_eager():
        for name, ws, A, Ys in launches:
            run_launch(mnb, name, ws, A, Ys)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step_eager()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step_eager()
    torch.cuda.synchronize()
    launches_per_step = len(launches)

    warmup = max(args.warmup, 3)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local, args.clock_log)
    if dist:
        dist.barrier()
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t = time_region(graph.replay, args.steps, torch.cuda.current_stream())
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()

    # end to end: host activations in, host results out, every step
    A_host = torch.empty(A_all.shape, dtype=A_all.dtype).pin_memory()
    A_host.copy_(A_all.cpu())
    Y_host = torch.empty(Y_all.shape, dtype=Y_all.dtype).pin_memory()
    cur = torch.cuda.current_stream()

    def step_e2e():
        A_all.copy_(A_host, non_blocking=True)
        graph.replay()
        Y_host.copy_(Y_all, non_blocking=True)

    for _ in range(3):
        step_e2e()
    t_e2e = time_region(step_e2e, args.steps, cur)

    # The same step as one persistent launch (mnb_chain_run), for comparison;
    # not the headline: the graph of launches is faster on this workload.
    chain = build_decode_chain(mnb, launches)
    for _ in range(3):
        chain.run()
    t_chain = time_region(chain.run, args.steps, cur)

    ts = torch.tensor([t, t_e2e, t_chain], device=dev, dtype=torch.float64)
    if dist:
        dist.all_reduce(ts, op=dist.ReduceOp.MAX)
    t, t_e2e, t_chain = ts.tolist()

    if rank != 0:
        return
    value = algo_bytes * args.steps * world / t / 1e9
    e2e = algo_bytes * args.steps * world / t_e2e / 1e9
    per_gpu = algo_bytes * args.steps / t / 1e9

    prefill = None if args.skip_prefill else prefill_measure(dev)
    fusions = lm_head_fusions(mnb, launches[-1], dev)
    cpu = None
    if world == 1 and not args.skip_cpu:
        nbytes, secs, desc = oracle_sample(args.cpu_budget)
        cpu = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": desc}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": warmup,
        "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "block_size": 128, "a_dtype": "bf16",
                   "weights_per_step": sum(len(ws) for _, ws, _, _ in launches),
                   "launches_per_step": launches_per_step,
                   "algorithmic_bytes_per_step": algo_bytes,
                   "l2": "inputs larger than L2 (2.08 GB per step vs 129 MB)",
                   "launch": "one CUDA graph per step: per layer fused qkv, o, gated-MLP "
                             "gate+up (SiLU(gate)*up), down, then lm_head (145 launches), "
                             "programmatic dependent launch",
                   "parallelism": f"replicas x{world}"},
        "hbm_fraction": per_gpu / hbm_peak,
        "roofline": {"bound": "hbm", "achieved": per_gpu, "peak": hbm_peak,
                     "unit": "GB/s", "frac": per_gpu / hbm_peak, "traffic": step_traffic(),
                     "peak_kind": peak_kind,
                     "kernel": "gemv_kernel (every launch of the step)",
                     "achieved_basis": "algorithmic bytes of the step / device time of the "
                                       "step (= bytes per launch / mean launch time)",
                     "algorithmic_bytes_per_launch": algo_bytes / launches_per_step,
                     "traffic_basis": "ncu dram read+write per launch, mean over the "
                                      "step's 145 launches; null if the kernel changed"},
        "e2e": {"value": e2e, "unit": "GB/s",
                "h2d_bytes_per_step": A_all.numel() * A_all.element_size(),
                "d2h_bytes_per_step": Y_all.numel() * Y_all.element_size()},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "prefill": prefill,
        "lm_head_fusions": fusions,
        "decode_chain": {"value": algo_bytes * args.steps / t_chain / 1e9, "unit": "GB/s",
                         "ms_per_step": 1e3 * t_chain / args.steps, "launches_per_step": 1,
                         "note": "the same step and dependencies as one persistent "
                                 "cooperative launch (mnb_chain_run)"},
        "cpu_baseline": cpu,
    }
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
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--clock-log", default=None,
                    help="file for the raw nvidia-smi clock samples of the timed region "
                         "(default: a private temporary file)")
    ap.add_argument("--skip-cpu", action="store_true")
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
