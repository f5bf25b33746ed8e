"""Parity of the decode step exactly as the benchmark times it: the Qwen3-4B
batch-1 step (M = 1, bf16, bs 128, no zero points; 253 weights, 2.08 GB)
recorded by the library as one CUDA graph of 145 programmatically dependent
calls (mnb_graph_build: fused q/k/v, o, the gated-MLP pair, down, then
lm_head), run with mnb_graph_run, and checked against the oracle on the raw
inputs of selected launches (drawn by the same seeded device generator as
the benchmark, copied to the host). Small projections are checked in full,
lm_head on seeded columns. The run framed by host copies
(mnb_graph_run_from_host, the benchmark's end-to-end form) returns the same
outputs."""
import numpy as np
import pytest
import torch

import bench
import int4_weight_only_matmulnbits_gb300 as mnb
import oracle
from tests.tolerance import check

pytestmark = pytest.mark.gpu

KEEP = ("L0.qkv", "L0.o", "L0.gate_up", "L0.down", "L17.down", "L35.gate_up", "lm_head")


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def test_decode_step_graph_matches_oracle(dev):
    launches, A_all, Y_all, _, kept = bench.build_decode_step(dev, keep=KEEP)
    graph = mnb.mnb_graph_build(bench.step_ops(mnb, launches))
    assert (graph.calls, graph.kernels) == (145, 145)
    Y_all.fill_(float("nan"))
    graph.run()
    torch.cuda.synchronize()
    Y_first = Y_all.clone()
    A_host = A_all.cpu().pin_memory()
    Y_host = torch.full(Y_all.shape, float("nan"), dtype=Y_all.dtype).pin_memory()
    Y_all.fill_(float("nan"))
    graph.run_from_host(A_host, A_all, Y_all, Y_host)
    torch.cuda.synchronize()
    assert torch.equal(Y_host, Y_first.cpu())
    outs = {name: Ys for name, _, _, Ys in launches}
    rng = np.random.default_rng(5)
    for name in KEEP:
        rec = kept[name]
        A = rec["A"]
        if name.endswith("gate_up"):
            (Bg, Sg, N, K), (Bu, Su, _, _) = rec["weights"]
            cols = np.sort(rng.choice(N, 512, replace=False))
            R, gv, uv, mg, mu = oracle.gate_up(A, (Bg, Sg, None, None), (Bu, Su, None, None),
                                               N=N, K=K, block_size=128, cols=cols)
            Y = outs[name][0][:, cols].float().cpu().double().numpy()
            eg, eu = 2e-3 * mg + 1e-5, 2e-3 * mu + 1e-5
            silu = gv / (1 + np.exp(-gv))
            b = (1.1 * eg * (np.abs(uv) + eu) + (np.abs(silu) + 1.1 * eg) * eu
                 + 2.0 ** -8 * np.abs(R) + 1e-6 * (np.abs(R) + 1))
            assert np.all(np.isfinite(Y)), name
            assert np.all(np.abs(Y - R) <= b), (name, float(np.max(np.abs(Y - R) / b)))
            continue
        for (B, S, N, K), Y in zip(rec["weights"], outs[name]):
            cols = None if N <= 4096 else np.sort(rng.choice(N, 1024, replace=False))
            R, mag = oracle.matmulnbits(A, B, S, None, None, N=N, K=K, block_size=128,
                                        cols=cols)
            check(Y if cols is None else Y[:, cols], R, mag, f"{name} N{N}")
    assert mnb.mnb_fault_status() == 0
